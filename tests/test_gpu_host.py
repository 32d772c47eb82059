"""ssm_scan_fwd_host (host buffers, copies pipelined with the scan) on the GPU, against the fp64
oracle and against ssm_scan_fwd on device copies of the same inputs."""
import pytest
import torch

import oracle
from selective_state_space_110_b300 import ssm_scan_fwd, ssm_scan_fwd_host
from tests.parity import TOL, assert_close
from workloads import ScanConfig, make_scan_inputs

pytestmark = pytest.mark.gpu

NAMES = ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")


def _host(x, pinned=True):
    return {k: (None if x[k] is None else (x[k].cpu().pin_memory() if pinned else x[k].cpu()))
            for k in NAMES}


@pytest.mark.parametrize("shape", [(3, 64, 256, "bf16"), (1, 40, 100, "f32"), (4, 96, 1000, "bf16")],
                         ids=lambda s: f"{s[0]}x{s[1]}x{s[2]}-{s[3]}")
def test_host_scan_matches_oracle(shape):
    b, d, L, dt = shape
    cfg = ScanConfig("h", b, d, 16, L, dt, "f32", 1e-3, 1e-1, 70 + L)
    x = make_scan_inputs(cfg, "cpu")
    h0 = torch.randn(b, d, 16).pin_memory()
    hx = _host(x)
    out, fin = ssm_scan_fwd_host(hx["u"], hx["delta"], hx["A"], hx["B"], hx["C"], hx["D"], hx["z"],
                                 hx["delta_bias"], True, initial_state=h0, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref, rfin = oracle.scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                                x["delta_bias"], True, h0)
    tol = TOL[x["u"].dtype]
    assert_close(out, ref, tol, "y")
    assert_close(fin, rfin, tol, "final state")


def test_host_scan_equals_device_scan_and_accepts_pageable_memory():
    cfg = ScanConfig("h", 4, 128, 16, 2048, "bf16", "bf16", 1e-3, 1e-1, 81)
    x = make_scan_inputs(cfg, "cuda")
    ref, rfin = ssm_scan_fwd(*[x[k] for k in NAMES], True)
    for pinned in (True, False):
        hx = _host(x, pinned)
        out, fin = ssm_scan_fwd_host(*[hx[k] for k in NAMES], True)
        torch.cuda.synchronize()
        assert_close(out, ref.double().cpu(), TOL[torch.bfloat16], "y")
        assert_close(fin, rfin.double().cpu(), TOL[torch.bfloat16], "final state")
