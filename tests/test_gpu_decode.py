"""ssm_state_update on the GPU, through the C ABI, against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_110_b300 import ssm_scan_fwd, ssm_state_update
from tests.parity import TOL, assert_close
from workloads import (DECODE_CONFIG, ScanConfig, make_decode_layer_params, make_decode_state,
                       make_decode_tokens, make_scan_inputs)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("batch", [1, 16, 64])
def test_decode_steps_full_rows(batch):
    """A few steps of one layer at the decode sweep's shape, every row checked."""
    cfg = DECODE_CONFIG
    p = make_decode_layer_params(cfg, DEV)
    st = make_decode_state(cfg, batch, 0, DEV)
    ref_state = st.clone()
    for step in range(3):
        tok = make_decode_tokens(cfg, batch, 0, step, DEV)
        out = ssm_state_update(st, tok["x"], tok["dt"], p["A"], tok["B"], tok["C"], p["D"],
                               tok["z"], dt_bias=p["dt_bias"], out_dtype=torch.float32)
        ref_state, ref = oracle.state_update(ref_state, tok["x"], tok["dt"], p["A"], tok["B"],
                                             tok["C"], p["D"], tok["z"], p["dt_bias"], True)
        assert_close(out, ref, TOL[torch.bfloat16], f"step {step} y")
        assert_close(st, ref_state, TOL[torch.bfloat16], f"step {step} state")


def test_decode_1024_steps_sampled_channels():
    """The sweep's 1,024 generated tokens at batch 64 on the GPU; the oracle follows a sample
    of channels (rows are independent) through all steps, with the ring of 8 token sets."""
    cfg = DECODE_CONFIG
    batch = 64
    p = make_decode_layer_params(cfg, DEV)
    st = make_decode_state(cfg, batch, 0, DEV)
    toks = [make_decode_tokens(cfg, batch, 0, s, DEV) for s in range(cfg.ring)]
    ch = torch.as_tensor(np.unique(np.r_[0, 1, 31, 32, 4095, 5119,
                                         np.random.default_rng(2).choice(5120, 20, replace=False)]),
                         device=DEV)
    sub = lambda t: t[:, ch].contiguous()
    ref_state = sub(st).clone()
    pA, pD, pb = p["A"][ch], p["D"][ch], p["dt_bias"][ch]
    outs = torch.empty(cfg.steps, batch, 5120, dtype=torch.float32, device=DEV)
    for s in range(cfg.steps):
        t = toks[s % cfg.ring]
        ssm_state_update(st, t["x"], t["dt"], p["A"], t["B"], t["C"], p["D"], t["z"],
                         out=outs[s], dt_bias=p["dt_bias"])
    torch.cuda.synchronize()
    for s in range(cfg.steps):
        t = toks[s % cfg.ring]
        ref_state, ref = oracle.state_update(ref_state, sub(t["x"]), sub(t["dt"]), pA, t["B"],
                                             t["C"], pD, sub(t["z"]), pb, True)
        if s % 32 == 31 or s < 4:
            assert_close(outs[s][:, ch], ref, TOL[torch.bfloat16], f"step {s} y")
    assert_close(st[:, ch], ref_state, TOL[torch.bfloat16], "state after 1024 steps")


def test_scan_equals_repeated_updates():
    """The scan and the decode step are the same recurrence: L state updates from h0 give
    the scan's outputs and final state (both GPU paths, fp32 out)."""
    cfg = ScanConfig("t", 2, 64, 16, 40, "bf16", "f32", 1e-3, 1e-1, 4)
    x = make_scan_inputs(cfg, DEV)
    h0 = torch.randn(2, 64, 16, device=DEV)
    out, fin = ssm_scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                            x["delta_bias"], True, out_dtype=torch.float32, initial_state=h0)
    st = h0.clone()
    ys = []
    for t in range(40):
        ys.append(ssm_state_update(st, x["u"][:, :, t].contiguous(), x["delta"][:, :, t].contiguous(),
                                   x["A"], x["B"][:, :, t].contiguous(), x["C"][:, :, t].contiguous(),
                                   x["D"], x["z"][:, :, t].contiguous(), dt_bias=x["delta_bias"],
                                   out_dtype=torch.float32))
    y = torch.stack(ys, dim=2)
    assert_close(y, out.double(), 1e-4, "updates vs scan y")
    assert_close(st, fin.double(), 1e-4, "updates vs scan state")


def test_update_bf16_output_and_no_gate():
    cfg = DECODE_CONFIG
    p = make_decode_layer_params(cfg, DEV)
    st = make_decode_state(cfg, 16, 1, DEV)
    ref_state = st.clone()
    tok = make_decode_tokens(cfg, 16, 1, 0, DEV)
    out = ssm_state_update(st, tok["x"], tok["dt"], p["A"], tok["B"], tok["C"], None, None,
                           dt_bias=p["dt_bias"])
    ref_state, ref = oracle.state_update(ref_state, tok["x"], tok["dt"], p["A"], tok["B"],
                                         tok["C"], None, None, p["dt_bias"], True)
    assert out.dtype == torch.bfloat16
    assert_close(out, ref, TOL[torch.bfloat16], "y")
    assert_close(st, ref_state, TOL[torch.bfloat16], "state")


def test_ragged_channels_larger_batch():
    """1,000 channels (the last block of 64 part-empty) at batch 40: every row checked over
    three steps."""
    cfg = DECODE_CONFIG.replace(dim=1000)
    batch = 40
    p = make_decode_layer_params(cfg, DEV)
    st = make_decode_state(cfg, batch, 0, DEV)
    ref_state = st.clone()
    for step in range(3):
        tok = make_decode_tokens(cfg, batch, 0, step, DEV)
        out = ssm_state_update(st, tok["x"], tok["dt"], p["A"], tok["B"], tok["C"], p["D"],
                               tok["z"], dt_bias=p["dt_bias"], out_dtype=torch.float32)
        ref_state, ref = oracle.state_update(ref_state, tok["x"], tok["dt"], p["A"], tok["B"],
                                             tok["C"], p["D"], tok["z"], p["dt_bias"], True)
        assert_close(out, ref, TOL[torch.bfloat16], f"step {step} y")
        assert_close(st, ref_state, TOL[torch.bfloat16], f"step {step} state")


@pytest.mark.parametrize("dim", [5000, 5120])
def test_two_rows_per_quad_back_to_back(dim):
    """Batch 16: one row per lane quad would need a second wave of CTAs, so each quad takes two
    rows and the next launch is let in early. dim 5,000 leaves the last CTA 8 of its 128 rows.
    Three steps on the same state run back to back on one stream (each launch's state prefetch
    comes before the previous step has written that state); every row is checked."""
    cfg = DECODE_CONFIG.replace(dim=dim)
    batch = 16
    p = make_decode_layer_params(cfg, DEV)
    st = make_decode_state(cfg, batch, 0, DEV)
    ref_state = st.clone()
    toks = [make_decode_tokens(cfg, batch, 0, step, DEV) for step in range(3)]
    outs = []
    for tok in toks:
        outs.append(ssm_state_update(st, tok["x"], tok["dt"], p["A"], tok["B"], tok["C"], p["D"],
                                     tok["z"], dt_bias=p["dt_bias"]))
    torch.cuda.synchronize()
    for step, tok in enumerate(toks):
        ref_state, ref = oracle.state_update(ref_state, tok["x"], tok["dt"], p["A"], tok["B"],
                                             tok["C"], p["D"], tok["z"], p["dt_bias"], True)
        assert_close(outs[step], ref, TOL[torch.bfloat16], f"step {step} y")
    assert_close(st, ref_state, TOL[torch.bfloat16], "state after three steps")
