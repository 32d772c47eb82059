"""Zero-order-hold discretisation on the GPU (SELSCAN_FLAG_ZOH), through the C ABI.

'Chosen by the Token' (world.lapla.si): with a state of a single number the selective update is
exactly a recurrent gate h <- (1 - g) h + g x. Under the zero-order hold with A = -1, B = C = 1
and Delta = softplus(delta + bias), g = sigmoid(delta + bias). The first tests run that case on
the GPU (state 0 only: B and C are zero for the other 15 states) and compare with the gate
recursion evaluated with the logistic function, not with the oracle. The others compare random
problems with the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_110_b300 import ssm_scan_fwd, ssm_state_update
from tests.oracle_pins import gate_reference
from tests.parity import TOL, assert_close
from workloads import ScanConfig, make_scan_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _gate_problem(dtype, batch=2, dim=48, L=200, seed=3):
    g = torch.Generator(DEV).manual_seed(seed)
    delta = (torch.randn(batch, dim, L, generator=g, device=DEV) * 1.5).to(dtype)
    u = torch.randn(batch, dim, L, generator=g, device=DEV).to(dtype)
    bias = torch.rand(dim, generator=g, device=DEV) * 5.0 - 3.0
    A = -torch.ones(dim, 16, device=DEV)
    B = torch.zeros(batch, 16, L, device=DEV, dtype=dtype)
    B[:, 0, :] = 1.0
    C = B.clone()
    h0 = torch.zeros(batch, dim, 16, device=DEV)
    h0[:, :, 0] = torch.randn(batch, dim, generator=g, device=DEV)
    return delta, u, bias, A, B, C, h0


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_theorem1_gate_scan(dtype):
    delta, u, bias, A, B, C, h0 = _gate_problem(dtype)
    out, fin = ssm_scan_fwd(u, delta, A, B, C, None, None, bias, True, initial_state=h0,
                            out_dtype=torch.float32, zoh=True)
    torch.cuda.synchronize()
    x = delta.double().cpu().numpy() + bias.double().cpu().numpy()[None, :, None]
    ref = gate_reference(x, u.double().cpu().numpy(), h0[:, :, 0].double().cpu().numpy())
    assert_close(out, ref, TOL[dtype], "y = gated state")
    assert_close(fin[:, :, 0], ref[..., -1], TOL[dtype], "final state")
    assert torch.count_nonzero(fin[:, :, 1:]) == 0  # states without input stay zero


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_theorem1_gate_decode(dtype):
    delta, u, bias, A, B, C, h0 = _gate_problem(dtype, L=50)
    st = h0.clone()
    ys = []
    for t in range(u.shape[-1]):
        ys.append(ssm_state_update(st, u[:, :, t].contiguous(), delta[:, :, t].contiguous(), A,
                                   B[:, :, t].contiguous(), C[:, :, t].contiguous(), None, None,
                                   dt_bias=bias, out_dtype=torch.float32, zoh=True))
    torch.cuda.synchronize()
    x = delta.double().cpu().numpy() + bias.double().cpu().numpy()[None, :, None]
    ref = gate_reference(x, u.double().cpu().numpy(), h0[:, :, 0].double().cpu().numpy())
    assert_close(torch.stack(ys, dim=2), ref, TOL[dtype], "decode y = gated state")


CASES = [
    # (batch, dim, seqlen, in dtype, out dtype)
    (2, 64, 256, "bf16", torch.float32),
    (3, 40, 100, "bf16", torch.bfloat16),  # ragged channels and tokens (scalar path)
    (2, 48, 300, "f32", torch.float32),
    (1, 64, 40960, "bf16", torch.float32),  # time segments
    (1, 24, 16392, "f32", torch.float32),   # time segments, fp32
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-{c[3]}-{str(c[4])[6:]}")
def test_zoh_scan_matches_oracle(case):
    b, d, L, dt, odt = case
    cfg = ScanConfig("z", b, d, 16, L, dt, dt, 1e-3, 1e-1, 90 + L)
    x = make_scan_inputs(cfg, DEV)
    h0 = torch.randn(b, d, 16, device=DEV, generator=torch.Generator(DEV).manual_seed(1))
    out, fin = ssm_scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                            x["delta_bias"], True, initial_state=h0, out_dtype=odt, zoh=True)
    ref, rfin = oracle.scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                                x["delta_bias"], True, h0, zoh=True)
    tol = TOL[x["u"].dtype]
    assert_close(out, ref, tol, "zoh y")
    assert_close(fin, rfin, tol, "zoh final state")


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_zoh_decode_matches_oracle(dt):
    cfg = ScanConfig("z", 16, 320, 16, 6, dt, dt, 1e-3, 1e-1, 77)
    x = make_scan_inputs(cfg, DEV)
    st = torch.randn(16, 320, 16, device=DEV, generator=torch.Generator(DEV).manual_seed(2))
    ref_state = st.double().cpu().numpy()
    for t in range(6):
        tok = {k: x[k][:, :, t].contiguous() for k in ("u", "delta", "z", "B", "C")}
        y = ssm_state_update(st, tok["u"], tok["delta"], x["A"], tok["B"], tok["C"], x["D"], tok["z"],
                             dt_bias=x["delta_bias"], out_dtype=torch.float32, zoh=True)
        ref_state, ry = oracle.state_update(ref_state, tok["u"], tok["delta"], x["A"], tok["B"],
                                            tok["C"], x["D"], tok["z"], x["delta_bias"], True, zoh=True)
        assert_close(y, ry, TOL[x["u"].dtype], f"step {t} y")
    assert_close(st, ref_state, TOL[x["u"].dtype], "state")
