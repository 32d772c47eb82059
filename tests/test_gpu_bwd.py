"""ssm_scan_bwd on the GPU, through the C ABI, against the fp64 oracle's reverse-mode backward.

Every gradient is compared element by element: du, ddelta, dz (per token), dA, dD, ddelta_bias
(per channel, summed over batches and tokens), dB, dC (per token, summed over channels) and the
gradient of the initial state. A, D and the bias are drawn per channel so that a wrong channel
index shows. Shapes cover ragged channel blocks (dim % 32 != 0), ragged chunks (seqlen % 16 != 0),
a single token, seqlen = 0, and every optional input present or absent. At the Mamba-2.8B layer
shape the full batch-0 slice and a sample of channels are checked.
"""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_110_b300 import SelscanError, ssm_scan_bwd
from tests.parity import TOL, assert_close
from workloads import ScanConfig, make_scan_inputs, scan_config

pytestmark = pytest.mark.gpu
DEV = "cuda"
KEYS = ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias", "dinitial_state")


def _problem(b, d, L, dt, seed, grad_dt=None, h0=True, dfinal=True, **kw):
    cfg = ScanConfig("bwd", b, d, 16, L, dt, dt, 1e-3, 1e-1, seed, **kw)
    x = make_scan_inputs(cfg, DEV)
    g = torch.Generator(DEV).manual_seed(seed + 1)
    x["A"] = (x["A"] * (0.5 + torch.rand(d, 1, generator=g, device=DEV))).contiguous()
    if x["D"] is not None:
        x["D"] = torch.randn(d, generator=g, device=DEV)
    gdt = x["u"].dtype if grad_dt is None else grad_dt
    x["dout"] = torch.randn(b, d, L, generator=g, device=DEV).to(gdt)
    x["initial_state"] = torch.randn(b, d, 16, generator=g, device=DEV) if h0 else None
    x["dfinal_state"] = torch.randn(b, d, 16, generator=g, device=DEV) if dfinal else None
    return x


def _gpu(x, **kw):
    return ssm_scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                        x["delta_bias"], x["delta_softplus"], initial_state=x["initial_state"],
                        dout=x["dout"], dfinal_state=x["dfinal_state"], **kw)


def _oracle(x):
    return oracle.scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                           x["delta_bias"], x["delta_softplus"], x["initial_state"], x["dout"],
                           x["dfinal_state"])


def _compare(got, ref, tol, label):
    for k in KEYS:
        if ref[k] is None:
            assert got[k] is None, k
            continue
        assert got[k] is not None, k
        if ref[k].size == 0:
            continue
        assert_close(got[k], ref[k], tol, f"{label} {k}")


SHAPES = [
    # (batch, dim, seqlen, in dtype, grad dtype)
    (1, 32, 16, "f32", torch.float32),      # one chunk, one CTA
    (2, 64, 100, "f32", torch.float32),     # ragged last chunk
    (3, 40, 257, "bf16", torch.float32),    # ragged channel block and chunk
    (2, 96, 1000, "bf16", torch.bfloat16),  # bf16 gradients
    (1, 33, 77, "f32", torch.bfloat16),
    (1, 1, 1, "bf16", torch.float32),
    (2, 128, 2048, "bf16", torch.float32),  # several channel blocks and 128 chunks
    (1, 49, 300, "bf16", torch.float32),    # one full 48-channel CTA and one row beyond it
    # more than 2 CTAs per SM of 148: the build for 3 per SM (per-token shuffle sums of dB | dC)
    (4, 3600, 64, "bf16", torch.float32),   # 4 x 75 CTAs
    (3, 4801, 40, "f32", torch.float32),    # 3 x 101 CTAs, the last of each batch one row
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}x{s[2]}-{s[3]}-{str(s[4])[6:]}")
def test_bwd_matches_oracle(shape):
    b, d, L, dt, gdt = shape
    x = _problem(b, d, L, dt, 300 + b * d + L, grad_dt=gdt)
    got = _gpu(x)
    torch.cuda.synchronize()
    _compare(got, _oracle(x), TOL[x["u"].dtype], f"{b}x{d}x{L}")


@pytest.mark.parametrize("variant", ["no_optional", "no_softplus", "no_z", "no_state_grads"])
def test_bwd_optional_inputs(variant):
    kw = {}
    h0 = dfinal = True
    if variant == "no_optional":
        kw = dict(has_z=False, has_D=False, has_bias=False)
        h0 = dfinal = False
    elif variant == "no_softplus":
        kw = dict(delta_softplus=False, delta_std=0.05)
    elif variant == "no_z":
        kw = dict(has_z=False)
    else:
        h0, dfinal = True, False
    x = _problem(2, 48, 130, "f32", 41, h0=h0, dfinal=dfinal, **kw)
    if variant == "no_softplus":  # Delta = delta + bias is used as is: keep it in (0, 0.2)
        x["delta"] = x["delta"].abs().contiguous()
        x["delta_bias"] = torch.linspace(0.01, 0.1, 48, device=DEV)
    got = _gpu(x)
    torch.cuda.synchronize()
    _compare(got, _oracle(x), TOL[torch.float32], variant)


def test_bwd_empty_sequence():
    """seqlen = 0: the final state is the initial state, so dinitial = dfinal; the rest is 0."""
    x = _problem(2, 40, 0, "f32", 5)
    got = _gpu(x)
    torch.cuda.synchronize()
    assert torch.equal(got["dinitial_state"], x["dfinal_state"])
    for k in ("dA", "dD", "ddelta_bias"):
        assert torch.count_nonzero(got[k]) == 0, k


@pytest.mark.parametrize("shape", [(2, 96, 600), (4, 5120, 64)], ids=["2x96x600", "4x5120x64"])
def test_bwd_is_deterministic(shape):
    """Bit-identical gradients on a repeat call: in the CTA instantiation built for 2 per SM
    (per-chunk contractions for dB | dC) and in the one built for 3 (the 428 CTAs of a
    5120-channel, 4-batch grid; per-token shuffle reduce-scatter)."""
    x = _problem(*shape, "bf16", 77)
    a = _gpu(x)
    b = _gpu(x)
    torch.cuda.synchronize()
    for k in KEYS:
        assert torch.equal(a[k], b[k]), k


def test_bwd_rejects_zoh_through_the_abi():
    from selective_state_space_110_b300 import _lib
    x = _problem(1, 32, 32, "f32", 9)
    g = _gpu(x)  # valid outputs to reuse as buffers
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
    st = _lib.lib().ssm_scan_bwd(
        x["u"].data_ptr(), x["delta"].data_ptr(), x["A"].data_ptr(), x["B"].data_ptr(),
        x["C"].data_ptr(), None, None, None, _lib.FLAG_SOFTPLUS | _lib.FLAG_ZOH, None,
        x["dout"].data_ptr(), None, g["du"].data_ptr(), g["ddelta"].data_ptr(),
        g["dA"].data_ptr(), g["dB"].data_ptr(), g["dC"].data_ptr(), None, None, None, None,
        1, 32, 16, 32, _lib.F32, _lib.F32, None, ws.data_ptr(), ws.numel(), None)
    with pytest.raises(SelscanError, match="UNSUPPORTED"):
        _lib.check("ssm_scan_bwd", st)


def _slice(x, bsl, dsl):
    """The sub-problem of batches bsl and channels dsl (per-channel inputs sliced too)."""
    y = {}
    for k in ("u", "delta", "z", "dout"):
        y[k] = None if x[k] is None else x[k][bsl, dsl].contiguous()
    for k in ("initial_state", "dfinal_state"):
        y[k] = None if x[k] is None else x[k][bsl, dsl].contiguous()
    for k in ("B", "C"):
        y[k] = x[k][bsl].contiguous()
    y["A"] = x["A"][dsl].contiguous()
    for k in ("D", "delta_bias"):
        y[k] = None if x[k] is None else x[k][dsl].contiguous()
    y["delta_softplus"] = x["delta_softplus"]
    return y


def test_bwd_mamba2p8b_layer_sampled():
    """Full Mamba-2.8B layer shape (4 x 5120 x 2048, bf16) in one launch. Checked against the
    oracle: every gradient of batch 0 (dB, dC of batch 0 sum over all 5120 channels of that
    batch alone), and dA, dD, ddelta_bias of 64 sampled channels over all 4 batches."""
    cfg = scan_config("c2")
    b, d, L = cfg.batch, cfg.dim, cfg.seqlen
    x = _problem(b, d, L, cfg.in_dtype, cfg.seed, grad_dt=torch.bfloat16)
    got = _gpu(x)
    torch.cuda.synchronize()
    tol = TOL[torch.bfloat16]
    r0 = _oracle(_slice(x, slice(0, 1), slice(None)))
    for k in ("du", "ddelta", "dz", "dB", "dC", "dinitial_state"):
        assert_close(got[k][0:1], r0[k], tol, f"batch 0 {k}")
    idx = torch.randperm(d, generator=torch.Generator().manual_seed(11))[:64].sort().values
    rs = _oracle(_slice(x, slice(None), idx.to(DEV)))
    assert_close(got["dA"][idx.to(DEV)], rs["dA"], tol, "sampled dA")
    assert_close(got["dD"][idx.to(DEV)], rs["dD"], tol, "sampled dD")
    assert_close(got["ddelta_bias"][idx.to(DEV)], rs["ddelta_bias"], tol, "sampled ddelta_bias")


def _unsplit_workspace_bytes(b, d, L):
    """Workspace of the backward without time segments (mirrors its layout: CTAs of 48 channels,
    256-byte parts)."""
    up = lambda x: (x + 63) // 64 * 64
    rows, chunks, blocks = b * d, (L + 15) // 16, (d + 47) // 48
    return 4 * (up(rows * chunks * 16) + up(blocks * b * L * 32) + up(rows * 16) + 2 * up(rows))


SEG_SHAPES = [
    # few rows and long sequences: the backward cuts them into time segments
    (1, 32, 40000, "bf16", torch.float32),
    (1, 40, 20001, "f32", torch.float32),    # ragged length (scalar loads), fp32
    (2, 16, 16384, "bf16", torch.bfloat16),
    (2, 768, 8192, "bf16", torch.float32),   # 16 blocks per batch, each cut in two segments
]


@pytest.mark.parametrize("shape", SEG_SHAPES, ids=lambda s: f"{s[0]}x{s[1]}x{s[2]}-{s[3]}-{str(s[4])[6:]}")
def test_bwd_time_segments(shape):
    from selective_state_space_110_b300 import bwd_workspace_size
    b, d, L, dt, gdt = shape
    assert bwd_workspace_size(b, d, 16, L) > _unsplit_workspace_bytes(b, d, L), "not split"
    x = _problem(b, d, L, dt, 500 + L, grad_dt=gdt)
    got = _gpu(x)
    torch.cuda.synchronize()
    _compare(got, _oracle(x), TOL[x["u"].dtype], f"{b}x{d}x{L} segments")


def test_bwd_rejects_a_small_workspace():
    from selective_state_space_110_b300 import bwd_workspace_size
    x = _problem(1, 32, 40000, "bf16", 3)
    need = bwd_workspace_size(1, 32, 16, 40000)
    with pytest.raises(SelscanError, match="WORKSPACE"):
        _gpu(x, workspace=torch.empty(need - 256, dtype=torch.uint8, device=DEV))


@pytest.mark.parametrize("shape", [(2, 64, 300, "f32"), (3, 40, 1000, "bf16"), (1, 32, 40000, "bf16")],
                         ids=lambda s: f"{s[0]}x{s[1]}x{s[2]}-{s[3]}")
def test_bwd_with_forward_checkpoints(shape):
    """ssm_scan_fwd_ckpt saves the state before every 16th token; ssm_scan_bwd given those
    checkpoints skips its own forward pass and must give the same gradients."""
    from selective_state_space_110_b300 import ssm_scan_fwd_ckpt
    b, d, L, dt = shape
    x = _problem(b, d, L, dt, 800 + L)
    _, fin, ck = ssm_scan_fwd_ckpt(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                                   x["delta_bias"], x["delta_softplus"],
                                   initial_state=x["initial_state"], out_dtype=torch.float32)
    got = _gpu(x, checkpoints=ck)
    torch.cuda.synchronize()
    tol = TOL[x["u"].dtype]
    assert torch.equal(ck[:, :, 0], x["initial_state"])
    # checkpoint c is the state after the first 16c tokens: the oracle's final state there
    for c in (1, (L - 1) // 16):
        pre = {k: (v[..., :16 * c].contiguous() if k in ("u", "delta", "z", "B", "C") and v is not None else v)
               for k, v in x.items()}
        _, rf = oracle.scan_fwd(pre["u"], pre["delta"], pre["A"], pre["B"], pre["C"], pre["D"],
                                pre["z"], pre["delta_bias"], pre["delta_softplus"], pre["initial_state"])
        assert_close(ck[:, :, c], rf, tol, f"checkpoint {c}")
    _compare(got, _oracle(x), tol, f"{b}x{d}x{L} with checkpoints")


@pytest.mark.parametrize("shape", [(2, 64, 300, "f32"), (3, 40, 1000, "bf16"), (4, 5120, 256, "bf16"),
                                   (1, 32, 40000, "bf16")],
                         ids=lambda s: f"{s[0]}x{s[1]}x{s[2]}-{s[3]}")
def test_forward_with_checkpoints_gives_the_same_outputs(shape):
    """The checkpoint-storing forward only adds stores: y and the final state are the plain
    forward's, bit for bit (one and two rows per lane, and time segments)."""
    from selective_state_space_110_b300 import ssm_scan_fwd, ssm_scan_fwd_ckpt
    b, d, L, dt = shape
    x = _problem(b, d, L, dt, 900 + L)
    args = (x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"],
            x["delta_softplus"])
    y0, f0 = ssm_scan_fwd(*args, initial_state=x["initial_state"], out_dtype=torch.float32)
    y1, f1, _ = ssm_scan_fwd_ckpt(*args, initial_state=x["initial_state"], out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1) and torch.equal(f0, f1)


@pytest.mark.parametrize("shape", [(4, 5120, 2048), (1, 1536, 1 << 20), (1, 32, 40000)],
                         ids=lambda s: f"{s[0]}x{s[1]}x{s[2]}")
def test_bwd_plan_on_the_device_matches_the_workspace(shape):
    """ssm_scan_bwd_plan for the current device reports the workspace ssm_scan_bwd_workspace_size
    gives, and the plan for the device's own SM count."""
    from selective_state_space_110_b300 import bwd_plan, bwd_workspace_size
    b, d, L = shape
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for ck in (False, True):
        p = bwd_plan(b, d, 16, L, checkpoints=ck)
        assert p == bwd_plan(b, d, 16, L, checkpoints=ck, sms=sms)
        assert p["workspace_bytes"] == bwd_workspace_size(b, d, 16, L, ck)


def test_bwd_parity_shapes_reach_both_builds():
    """The parity shapes above run both CTA builds on this GPU: the 3-per-SM one (shuffle sums)
    for grids of more than 2 CTAs per SM, the 2-per-SM one (contractions) otherwise."""
    from selective_state_space_110_b300 import bwd_plan
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for b, d, L in [(4, 3600, 64), (3, 4801, 40)]:
        p = bwd_plan(b, d, 16, L)
        assert p["ctas"] > 2 * sms and p["ctas_per_sm"] == 3, (b, d, L, p)
    for b, d, L in [(1, 49, 300), (2, 128, 2048)]:
        assert bwd_plan(b, d, 16, L)["ctas_per_sm"] == 2
