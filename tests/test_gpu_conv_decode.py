"""The fused decode step of a layer (short convolution + state update) on the GPU, through the
C ABI, against the fp64 oracle ('A State of Fixed Size': 16 state numbers per channel plus a
short convolution that holds the last 4 inputs)."""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_110_b300 import ssm_conv_state_update
from tests.parity import TOL, assert_close
from workloads import DECODE_CONFIG, make_decode_layer_params, make_decode_state, make_decode_tokens

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _conv_params(dim, seed):
    g = torch.Generator(DEV).manual_seed(seed)
    w = torch.randn(dim, 4, generator=g, device=DEV) * 0.5
    bias = torch.randn(dim, generator=g, device=DEV) * 0.1
    return w, bias


@pytest.mark.parametrize("batch", [1, 16, 64])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_fused_conv_and_update_steps(batch, dt):
    cfg = DECODE_CONFIG
    p = make_decode_layer_params(cfg, DEV)
    st = make_decode_state(cfg, batch, 0, DEV)
    w, cb = _conv_params(cfg.dim, batch)
    g = torch.Generator(DEV).manual_seed(100 + batch)
    cs = torch.randn(batch, cfg.dim, 4, generator=g, device=DEV).to(dt)
    ref_cs, ref_st = cs.double().cpu().numpy(), st.double().cpu().numpy()
    for step in range(4):
        tok = {k: v.to(dt) for k, v in make_decode_tokens(cfg, batch, 0, step, DEV).items()}
        out, u = ssm_conv_state_update(cs, tok["x"], w, cb, True, st, tok["dt"], p["A"], tok["B"],
                                       tok["C"], p["D"], tok["z"], dt_bias=p["dt_bias"],
                                       out_dtype=torch.float32, return_conv_out=True)
        ref_cs, ref_st, ref_u, ref_out = oracle.conv_state_update(
            ref_cs, tok["x"], w, cb, True, ref_st, tok["dt"], p["A"], tok["B"], tok["C"], p["D"],
            tok["z"], p["dt_bias"], True)
        tol = TOL[dt]
        assert_close(out, ref_out, tol, f"step {step} y")
        assert_close(u, ref_u, tol, f"step {step} conv output")
        assert torch.equal(cs.double().cpu(), torch.from_numpy(ref_cs)), "window is a copy of inputs"
        assert_close(st, ref_st, tol, f"step {step} state")


@pytest.mark.parametrize("silu", [True, False])
def test_conv_step_alone(silu):
    batch, dim = 8, 1000  # ragged channel count
    w, cb = _conv_params(dim, 7)
    g = torch.Generator(DEV).manual_seed(9)
    cs = torch.zeros(batch, dim, 4, device=DEV, dtype=torch.bfloat16)
    xs = torch.randn(6, batch, dim, generator=g, device=DEV).to(torch.bfloat16)
    ref_cs = cs.double().cpu().numpy()
    for t in range(6):
        _, u = ssm_conv_state_update(cs, xs[t], w, None if t % 2 else cb, silu)
        ref_cs, ru = oracle.conv_step(ref_cs, xs[t], w, None if t % 2 else cb, silu)
        assert_close(u, ru, TOL[torch.bfloat16], f"conv output step {t}")
    assert torch.equal(cs.double().cpu(), torch.from_numpy(ref_cs))


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_fused_steps_ragged_channels_larger_batch(dt):
    """The fused step with 1,000 channels (the last block of 64 part-empty) at batch 40."""
    cfg = DECODE_CONFIG.replace(dim=1000)
    batch = 40
    p = make_decode_layer_params(cfg, DEV)
    st = make_decode_state(cfg, batch, 0, DEV)
    w, cb = _conv_params(cfg.dim, 3)
    g = torch.Generator(DEV).manual_seed(303)
    cs = torch.randn(batch, cfg.dim, 4, generator=g, device=DEV).to(dt)
    ref_cs, ref_st = cs.double().cpu().numpy(), st.double().cpu().numpy()
    for step in range(3):
        tok = {k: v.to(dt) for k, v in make_decode_tokens(cfg, batch, 0, step, DEV).items()}
        out, u = ssm_conv_state_update(cs, tok["x"], w, cb, True, st, tok["dt"], p["A"], tok["B"],
                                       tok["C"], p["D"], tok["z"], dt_bias=p["dt_bias"],
                                       out_dtype=torch.float32, return_conv_out=True)
        ref_cs, ref_st, ref_u, ref_out = oracle.conv_state_update(
            ref_cs, tok["x"], w, cb, True, ref_st, tok["dt"], p["A"], tok["B"], tok["C"], p["D"],
            tok["z"], p["dt_bias"], True)
        tol = TOL[dt]
        assert_close(out, ref_out, tol, f"step {step} y")
        assert_close(u, ref_u, tol, f"step {step} conv output")
        assert torch.equal(cs.double().cpu(), torch.from_numpy(ref_cs)), "window is a copy of inputs"
        assert_close(st, ref_st, tol, f"step {step} state")
