"""ssd_chunk_scan_fwd (Mamba-2 SSD layer) on the GPU, through the C ABI, against the fp64
oracle's recurrence.

Shapes cover one chunk exactly (128 tokens), ragged last chunks, a single token, seqlen 0, two
groups of B/C, an initial state, every optional input absent, fp32 and bf16 outputs; at the
Mamba-2 2.7B layer shape (4 x 2048 tokens, 80 heads) sampled heads are compared in full, and a
sequence split in two calls (the second starting from the first's final state) must match one
call. Bound: 2e-3 with the RMS floor, as for the bf16 scan.
"""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_110_b300 import SelscanError, ssd_chunk_scan_fwd
from tests.parity import TOL, assert_close
from workloads import SsdConfig, make_ssd_inputs, ssd_config

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_BF16 = TOL[torch.bfloat16]


def _gpu(x, **kw):
    return ssd_chunk_scan_fwd(x["x"], x["dt"], x["A"], x["B"], x["C"], x["D"], x["z"],
                              x["dt_bias"], x["dt_softplus"], **kw)


def _oracle(x, h0=None):
    return oracle.ssd_fwd(x["x"], x["dt"], x["A"], x["B"], x["C"], x["D"], x["z"], x["dt_bias"],
                          x["dt_softplus"], h0)


def _inputs(batch, seqlen, nheads, ngroups, seed, **kw):
    return make_ssd_inputs(SsdConfig("t", batch, seqlen, nheads, 64, ngroups, 128, seed, **kw), DEV)


def test_tiny_config_full():
    x = make_ssd_inputs(ssd_config("ssd0"), DEV)
    y, fin = _gpu(x, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ry, rf = _oracle(x)
    assert_close(y, ry, TOL_BF16, "ssd0 y")
    assert_close(fin, rf, TOL_BF16, "ssd0 final state")


SHAPES = [
    # (batch, seqlen, nheads, ngroups, with initial state, out dtype)
    (1, 128, 2, 1, False, torch.float32),   # exactly one chunk
    (2, 300, 4, 2, True, torch.float32),    # ragged last chunk, two groups, initial state
    (1, 129, 3, 1, True, torch.float32),    # one token into the second chunk
    (2, 1, 2, 2, True, torch.float32),      # a single token
    (1, 700, 2, 1, False, torch.bfloat16),  # bf16 output
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}x{s[2]}g{s[3]}-h0{int(s[4])}-{str(s[5])[6:]}")
def test_shapes(shape):
    b, L, H, G, with_h0, odt = shape
    x = _inputs(b, L, H, G, 50 + L + H)
    h0 = None
    if with_h0:
        h0 = torch.randn(b, H, 64, 128, device=DEV, generator=torch.Generator(DEV).manual_seed(L))
    y, fin = _gpu(x, out_dtype=odt, initial_state=h0)
    torch.cuda.synchronize()
    ry, rf = _oracle(x, h0)
    assert_close(y, ry, TOL_BF16, "y")
    assert_close(fin, rf, TOL_BF16, "final state")


def test_no_optional_inputs():
    x = _inputs(2, 260, 3, 1, 61, has_z=False, has_D=False)
    x["dt_bias"] = None
    x["dt_softplus"] = False
    x["dt"] = (x["dt"].float().abs() * 0.05 + 0.01).to(torch.bfloat16)  # Delta = dt, positive
    y, fin = _gpu(x, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ry, rf = _oracle(x)
    assert_close(y, ry, TOL_BF16, "y")
    assert_close(fin, rf, TOL_BF16, "final state")


def test_empty_sequence_keeps_the_state():
    x = _inputs(2, 0, 2, 1, 5)
    h0 = torch.randn(2, 2, 64, 128, device=DEV)
    _, fin = _gpu(x, out_dtype=torch.float32, initial_state=h0)
    _, fin0 = _gpu(x, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(fin, h0)
    assert torch.count_nonzero(fin0) == 0


def test_rejects_unsupported_shapes():
    x = _inputs(1, 64, 2, 1, 7)
    with pytest.raises(SelscanError, match="UNSUPPORTED"):
        ssd_chunk_scan_fwd(x["x"][..., :32].contiguous(), x["dt"], x["A"], x["B"], x["C"])
    with pytest.raises(SelscanError, match="UNSUPPORTED"):
        ssd_chunk_scan_fwd(x["x"], x["dt"], x["A"], x["B"][..., :64].contiguous(),
                           x["C"][..., :64].contiguous())


def _heads(x, idx):
    y = dict(x)
    for k in ("x", "z"):
        y[k] = None if x[k] is None else x[k][:, :, idx].contiguous()
    y["dt"] = x["dt"][:, :, idx].contiguous()
    for k in ("A", "D", "dt_bias"):
        y[k] = None if x[k] is None else x[k][idx].contiguous()
    return y


def test_mamba2_layer_sampled_heads():
    """Full Mamba-2 2.7B layer shape in one launch; three heads checked against the oracle over
    every batch and token, with the final states."""
    cfg = ssd_config("ssd1")
    x = make_ssd_inputs(cfg, DEV)
    y, fin = _gpu(x, out_dtype=torch.float32)
    torch.cuda.synchronize()
    idx = torch.tensor([0, 37, 79], device=DEV)
    ry, rf = _oracle(_heads(x, idx))
    assert_close(y[:, :, idx], ry, TOL_BF16, "sampled heads y")
    assert_close(fin[:, idx], rf, TOL_BF16, "sampled heads final state")


def test_split_sequence_equals_one_call():
    """Prefill in two calls (the second from the first's final state) equals one call: the
    state passed between calls is the state passed between chunks."""
    cfg = ssd_config("ssd1").replace(batch=2, nheads=16)
    x = make_ssd_inputs(cfg, DEV)
    y, fin = _gpu(x, out_dtype=torch.float32)
    cut = 1000  # not a multiple of the chunk length
    first = {k: (v[:, :cut].contiguous() if k in ("x", "dt", "z", "B", "C") and v is not None else v)
             for k, v in x.items()}
    second = {k: (v[:, cut:].contiguous() if k in ("x", "dt", "z", "B", "C") and v is not None else v)
              for k, v in x.items()}
    y1, f1 = _gpu(first, out_dtype=torch.float32)
    y2, f2 = _gpu(second, out_dtype=torch.float32, initial_state=f1)
    torch.cuda.synchronize()
    assert_close(torch.cat([y1, y2], dim=1), y.double(), TOL_BF16, "split y")
    assert_close(f2, fin.double(), TOL_BF16, "split final state")


@pytest.mark.parametrize("dt_range", [(0.2, 0.5), (5.0, 8.0)], ids=["mixed", "strong"])
def test_strong_decay(dt_range):
    """Steps large enough that the decay factor over 16 tokens falls below 2^-64 in many heads
    (steps of 0.2-0.5: some 16-token pieces of a head on each side of that line; steps of 5-8:
    the state all but forgotten from one token to the next). M's decays are then taken both
    ways, as a row factor times a column factor within a piece and per element where a piece
    decays further; they underflow for distant tokens with no overflow or NaN on the way."""
    cfg = SsdConfig("decay", 2, 500, 8, 64, 1, 128, 77, dt_min=dt_range[0], dt_max=dt_range[1])
    x = make_ssd_inputs(cfg, DEV)
    y, fin = _gpu(x, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ry, rf = _oracle(x)
    assert_close(y, ry, TOL_BF16, "y")
    assert_close(fin, rf, TOL_BF16, "final state")


@pytest.mark.parametrize("seqlen,dt_range", [(1024, None), (1000, (0.2, 0.5))],
                         ids=["1024-tokens", "1000-tokens-mixed-decay"])
def test_balanced_launch(seqlen, dt_range):
    """160 chains (2 x 80 heads) on 148 SMs: the last 12 chains (batch 1, heads 68-79) are cut
    into time segments (their local end states from a first pass, folded into each segment's
    initial state). Sampled heads on both sides of the cut, with an initial state, against the
    oracle; every output against the unsplit launch; and a workspace too small for the plan
    runs unsplit, bit for bit."""
    from selective_state_space_110_b300 import ssd_workspace_size
    kw = {} if dt_range is None else dict(dt_min=dt_range[0], dt_max=dt_range[1])
    cfg = SsdConfig("bal", 2, seqlen, 80, 64, 1, 128, 91 + seqlen, **kw)
    need = ssd_workspace_size(2, seqlen, 80)
    assert need > 0, "the plan should cut the last wave's chains on this device"
    x = make_ssd_inputs(cfg, DEV)
    h0 = torch.randn(2, 80, 64, 128, device=DEV, generator=torch.Generator(DEV).manual_seed(5))
    y, fin = _gpu(x, out_dtype=torch.float32, initial_state=h0)
    y0, fin0 = _gpu(x, out_dtype=torch.float32, initial_state=h0, balance=False)
    small = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    y1, fin1 = _gpu(x, out_dtype=torch.float32, initial_state=h0, workspace=small)
    torch.cuda.synchronize()
    assert torch.equal(y1, y0) and torch.equal(fin1, fin0)
    assert_close(y, y0.double(), TOL_BF16, "balanced y vs unsplit")
    assert_close(fin, fin0.double(), TOL_BF16, "balanced final state vs unsplit")
    idx = torch.tensor([3, 67, 68, 74, 79], device=DEV)
    ry, rf = _oracle(_heads(x, idx), h0[:, idx].contiguous())
    assert_close(y[:, :, idx], ry, TOL_BF16, "sampled heads y")
    assert_close(fin[:, idx], rf, TOL_BF16, "sampled heads final state")


def test_balanced_launch_groups_no_gate_bf16_out():
    """300 chains (3 x 100 heads) on 148 SMs leave 4 chains to cut; 700 tokens end in a
    part-filled chunk; two groups of B / C, no z, bf16 output."""
    from selective_state_space_110_b300 import ssd_workspace_size
    cfg = SsdConfig("bal2", 3, 700, 100, 64, 2, 128, 97, has_z=False)
    assert ssd_workspace_size(3, 700, 100) > 0
    x = make_ssd_inputs(cfg, DEV)
    y, fin = _gpu(x, out_dtype=torch.bfloat16)
    # the unsplit reference in fp32: two bf16 roundings of nearly equal values can differ by a
    # whole ulp, more than the allowance of a bf16 output against an exact value
    y0, fin0 = _gpu(x, out_dtype=torch.float32, balance=False)
    torch.cuda.synchronize()
    assert_close(y, y0.double(), TOL_BF16, "balanced y vs unsplit")
    assert_close(fin, fin0.double(), TOL_BF16, "balanced final state vs unsplit")
    # heads 96-99 of batch 2 are cut; two heads of each group, so that the 4-head subset keeps
    # every head's group of B / C (group = head // (heads / 2))
    idx = torch.tensor([0, 49, 96, 99], device=DEV)
    ry, rf = _oracle(_heads(x, idx))
    assert_close(y[:, :, idx], ry, TOL_BF16, "sampled heads y")
    assert_close(fin[:, idx], rf, TOL_BF16, "sampled heads final state")
