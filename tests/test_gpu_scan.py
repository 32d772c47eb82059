"""ssm_scan_fwd on the GPU, through the C ABI, against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_110_b300 import ssm_scan_fwd, workspace_size
from tests.parity import TOL, assert_close, rel_err
from workloads import ScanConfig, make_scan_inputs, scan_config

pytestmark = pytest.mark.gpu

DEV = "cuda"


def run_gpu(x, out_dtype=None, initial_state=None, **kw):
    return ssm_scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                        x["delta_bias"], x["delta_softplus"], out_dtype=out_dtype,
                        initial_state=initial_state, **kw)


def run_oracle(x, initial_state=None):
    return oracle.scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                           x["delta_bias"], x["delta_softplus"], initial_state)


def small_cfg(batch, dim, seqlen, dt, seed, **kw):
    return ScanConfig("t", batch, dim, 16, seqlen, dt, dt, 1e-3, 1e-1, seed, **kw)


def test_config0_tiny_fp32_full():
    cfg = scan_config("c0")
    x = make_scan_inputs(cfg, DEV)
    out, fin = run_gpu(x)
    torch.cuda.synchronize()
    ref, rfin = run_oracle(x)
    assert_close(out, ref, TOL[torch.float32], "c0 y")
    assert_close(fin, rfin, TOL[torch.float32], "c0 final state")


SHAPES = [
    # (batch, dim, seqlen, in dtype, out dtype): ragged channels / tokens, both load paths
    (2, 40, 100, "bf16", torch.float32),   # dim % 32 != 0, seqlen % 8 != 0 (scalar path)
    (2, 64, 256, "bf16", torch.float32),
    (3, 96, 1000, "bf16", torch.bfloat16),  # partial last chunk, bf16 output
    (1, 33, 77, "f32", torch.float32),
    (2, 64, 1024, "f32", torch.bfloat16),
    (1, 1, 1, "bf16", torch.float32),
    (4, 7, 33, "f32", torch.float32),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}x{s[2]}-{s[3]}-{str(s[4])[6:]}")
def test_small_shapes(shape):
    b, d, L, dt, odt = shape
    cfg = small_cfg(b, d, L, dt, 7 + b * d + L)
    x = make_scan_inputs(cfg, DEV)
    out, fin = run_gpu(x, out_dtype=odt)
    ref, rfin = run_oracle(x)
    tol = TOL[x["u"].dtype]
    assert_close(out, ref, tol, "y")
    assert_close(fin, rfin, tol, "final state")


OPTIONS = {
    "no_z": dict(has_z=False),
    "no_D": dict(has_D=False),
    "no_bias": dict(has_bias=False),
    "softplus_off": dict(delta_softplus=False, has_bias=False),
}


@pytest.mark.parametrize("opt", sorted(OPTIONS))
@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_optional_arguments(opt, dt):
    cfg = small_cfg(2, 64, 200, dt, 99, **OPTIONS[opt])
    x = make_scan_inputs(cfg, DEV)
    if opt == "softplus_off":  # keep Delta positive without softplus
        x["delta"] = x["delta"].abs() * 0.1 + 0.01
    out, fin = run_gpu(x, out_dtype=torch.float32)
    ref, rfin = run_oracle(x)
    tol = TOL[x["u"].dtype]
    assert_close(out, ref, tol, "y")
    assert_close(fin, rfin, tol, "final state")


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_initial_state(dt):
    cfg = small_cfg(2, 48, 300, dt, 5)
    x = make_scan_inputs(cfg, DEV)
    h0 = torch.randn(2, 48, 16, device=DEV, generator=torch.Generator(DEV).manual_seed(3))
    out, fin = run_gpu(x, out_dtype=torch.float32, initial_state=h0)
    ref, rfin = run_oracle(x, initial_state=h0)
    tol = TOL[x["u"].dtype]
    assert_close(out, ref, tol, "y")
    assert_close(fin, rfin, tol, "final state")


# Two rows per lane (taken from 16,384 rows on, bf16 with seqlen % 8 == 0), every element
# checked: a ragged channel count leaves the last CTA partly inactive.
TWO_ROWS = [
    (8, 2048, 256, torch.float32, False),
    (2, 8200, 96, torch.bfloat16, True),
]


@pytest.mark.parametrize("case", TWO_ROWS, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-{str(c[3])[6:]}-h0{int(c[4])}")
def test_two_rows_per_lane_full_check(case):
    b, d, L, odt, with_h0 = case
    assert b * d >= 16384 and workspace_size(b, d, 16, L) == 0
    cfg = small_cfg(b, d, L, "bf16", 40 + d)
    x = make_scan_inputs(cfg, DEV)
    h0 = torch.randn(b, d, 16, device=DEV, generator=torch.Generator(DEV).manual_seed(6)) if with_h0 else None
    out, fin = run_gpu(x, out_dtype=odt, initial_state=h0)
    ref, rfin = run_oracle(x, initial_state=h0)
    assert_close(out, ref, TOL[torch.bfloat16], "y")
    assert_close(fin, rfin, TOL[torch.bfloat16], "final state")


SEGMENTED = [
    # few rows, long sequences: the time split (local-end pass + folding) is taken
    (1, 64, 40960, "bf16", False),
    (2, 16, 20000, "bf16", True),
    (1, 8, 16392, "f32", True),
    (1, 24, 30001, "bf16", False),  # seqlen % 8 != 0: scalar path with segments
]


@pytest.mark.parametrize("case", SEGMENTED, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-{c[3]}-h0{int(c[4])}")
def test_time_segments(case):
    b, d, L, dt, with_h0 = case
    assert workspace_size(b, d, 16, L) > 0, "this shape is meant to take the segmented path"
    cfg = small_cfg(b, d, L, dt, 17 + L)
    x = make_scan_inputs(cfg, DEV)
    h0 = torch.randn(b, d, 16, device=DEV) if with_h0 else None
    out, fin = run_gpu(x, out_dtype=torch.float32, initial_state=h0)
    ref, rfin = run_oracle(x, initial_state=h0)
    tol = TOL[x["u"].dtype]
    assert_close(out, ref, tol, "y")
    assert_close(fin, rfin, tol, "final state")


def test_zero_length_sequence_returns_initial_state():
    cfg = small_cfg(2, 40, 0, "bf16", 1)
    x = make_scan_inputs(cfg, DEV)
    h0 = torch.randn(2, 40, 16, device=DEV)
    out, fin = run_gpu(x, initial_state=h0)
    torch.cuda.synchronize()
    assert out.numel() == 0 and torch.equal(fin, h0)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_delta_zero_keeps_state_bit_exact(dt):
    """'Chosen by the Token': a small Delta keeps the state. Delta = 0 exactly must leave it
    bit-identical, and y = (C . h0 + D u) silu(z)."""
    cfg = small_cfg(2, 64, 128, dt, 8, delta_softplus=False, has_bias=False)
    x = make_scan_inputs(cfg, DEV)
    x["delta"] = torch.zeros_like(x["delta"])
    h0 = torch.randn(2, 64, 16, device=DEV)
    out, fin = run_gpu(x, out_dtype=torch.float32, initial_state=h0)
    torch.cuda.synchronize()
    assert torch.equal(fin, h0)
    ref, _ = run_oracle(x, initial_state=h0)
    assert_close(out, ref, TOL[x["u"].dtype], "y")


def test_deterministic_and_guard_bands():
    cfg = small_cfg(3, 80, 520, "bf16", 12)
    x = make_scan_inputs(cfg, DEV)
    pad = 64
    sentinel = -12345.0
    big_out = torch.full((3 * 80 * 520 + 2 * pad,), sentinel, dtype=torch.float32, device=DEV)
    big_fin = torch.full((3 * 80 * 16 + 2 * pad,), sentinel, dtype=torch.float32, device=DEV)
    out = big_out[pad:-pad].view(3, 80, 520)
    fin = big_fin[pad:-pad].view(3, 80, 16)
    run_gpu(x, out=out, final_state=fin)
    o2, f2 = run_gpu(x, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.all(big_out[:pad] == sentinel) and torch.all(big_out[-pad:] == sentinel)
    assert torch.all(big_fin[:pad] == sentinel) and torch.all(big_fin[-pad:] == sentinel)
    assert torch.equal(out, o2) and torch.equal(fin, f2)


def _sample_rows(batch, dim, k, seed):
    r = np.random.default_rng(seed)
    R = batch * dim
    edge = [0, dim - 1, R - 1, R - dim, 31 % dim, min(32, dim - 1)]
    rows = np.unique(np.concatenate([edge, r.choice(R, size=min(k, R), replace=False)]))
    return rows


@pytest.mark.parametrize("name,k", [("c1", 48), ("c2", 48), ("c3", 12)])
def test_full_size_config_sampled_rows(name, k):
    """Full-size workload, in the launch configuration the benchmark times; the oracle
    recomputes a sample of rows (all tokens of each) and every output must be finite."""
    cfg = scan_config(name)
    x = make_scan_inputs(cfg, DEV)
    out, fin = run_gpu(x, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all() and torch.isfinite(fin).all()
    rows = _sample_rows(cfg.batch, cfg.dim, k, 5)
    flat = lambda t: t.view(cfg.batch * cfg.dim, -1)[torch.as_tensor(rows, device=DEV)]
    ref, rfin = oracle.scan_fwd_rows(rows, flat(x["u"]), flat(x["delta"]), x["A"], x["B"], x["C"],
                                     x["D"], flat(x["z"]), x["delta_bias"], True)
    tol = TOL[torch.bfloat16]
    assert_close(flat(out), ref, tol, f"{name} y (sampled rows)")
    assert_close(flat(fin), rfin, tol, f"{name} final state (sampled rows)")


# More blocks of 128 channels than SMs (bf16 fast path): the balanced plan runs one whole
# block per SM in wide CTAs and cuts the remainder blocks into time segments (local-end
# pass + fold) that fill the last wave. Every element checked, with the plan asserted, and the
# same call with too small a workspace (the unsplit launch) checked too.
BALANCED = [
    (5, 4096, 512, "bf16", torch.float32, True),
    (5, 4096, 520, "bf16", torch.bfloat16, False),  # seqlen % 16 != 0, last segment ragged
    (3, 6840, 512, "bf16", torch.float32, True),    # dim % 128 != 0: a cut block part-empty
]


@pytest.mark.parametrize("case", BALANCED, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-{c[3]}-h0{int(c[5])}")
def test_balanced_plan_full_check(case):
    from selective_state_space_110_b300 import scan_plan
    b, d, L, dt, odt, with_h0 = case
    in_dt = torch.bfloat16 if dt == "bf16" else torch.float32
    plan = scan_plan(b, d, 16, L, in_dtype=in_dt)
    assert plan["split_blocks"] > 0 and plan["whole_blocks"] > 0 and plan["segments"] > 1, plan
    assert plan["required_workspace_bytes"] == 0 and plan["channels_per_block"] == 128, plan
    cfg = small_cfg(b, d, L, dt, 60 + d + L)
    x = make_scan_inputs(cfg, DEV)
    h0 = torch.randn(b, d, 16, device=DEV, generator=torch.Generator(DEV).manual_seed(9)) if with_h0 else None
    out, fin = run_gpu(x, out_dtype=odt, initial_state=h0)
    ref, rfin = run_oracle(x, initial_state=h0)
    tol = TOL[x["u"].dtype]
    assert_close(out, ref, tol, "balanced y")
    assert_close(fin, rfin, tol, "balanced final state")
    # Without room for the split: the unsplit launch, same results to rounding.
    tiny = torch.empty(16, dtype=torch.uint8, device=DEV)
    assert scan_plan(b, d, 16, L, 16, in_dtype=in_dt)["split_blocks"] == 0
    out2, fin2 = run_gpu(x, out_dtype=odt, initial_state=h0, workspace=tiny)
    assert_close(out2, ref, tol, "unsplit y")
    assert_close(fin2, rfin, tol, "unsplit final state")
