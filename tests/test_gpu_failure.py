"""Failure detection on the GPU without a fault: a bounded device wait that runs out.

The scan kernels wait (bounded, about two seconds) for TMA copies of B and C to land in shared
memory. The self-test hook launches one CTA that waits on an mbarrier nothing arrives at, with a
short limit; it must give up, set the device flag, exit normally and leave the context usable.
"""
import pytest
import torch

from selective_state_space_110_b300 import _lib, ssm_scan_fwd
from tests.parity import TOL, assert_close
from workloads import ScanConfig, make_scan_inputs
import oracle

pytestmark = pytest.mark.gpu

OK, INVALID, TIMEOUT = 0, 1, 7


def test_bounded_wait_reports_timeout_and_context_survives():
    lib = _lib.lib()
    s = torch.cuda.current_stream().cuda_stream
    assert lib.selscan_device_status(1, s) == OK  # clear anything earlier
    assert lib.selscan_selftest_wait_timeout(200_000, s) == OK  # ~0.1 ms of SM clock
    assert lib.selscan_device_status(0, s) == TIMEOUT
    assert lib.selscan_device_status(1, s) == TIMEOUT  # read and clear
    assert lib.selscan_device_status(0, s) == OK
    assert lib.selscan_selftest_wait_timeout(0, s) == INVALID
    # The context still runs the scan correctly, and a normal scan raises no flag.
    cfg = ScanConfig("f", 2, 64, 16, 256, "bf16", "f32", 1e-3, 1e-1, 77)
    x = make_scan_inputs(cfg, "cuda")
    out, fin = ssm_scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                            x["delta_bias"], True, out_dtype=torch.float32)
    assert lib.selscan_device_status(0, s) == OK
    ref, rfin = oracle.scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                                x["delta_bias"], True)
    assert_close(out, ref, TOL[torch.bfloat16], "y after a timed-out wait")
    assert_close(fin, rfin, TOL[torch.bfloat16], "final state after a timed-out wait")


def test_device_flag_is_shared_by_streams():
    """The error word is one per device: a timeout raised by a launch on one stream is reported
    by a query on another stream, and a reset from there clears it for both."""
    lib = _lib.lib()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    assert lib.selscan_device_status(1, s1.cuda_stream) == OK
    assert lib.selscan_selftest_wait_timeout(200_000, s1.cuda_stream) == OK
    s1.synchronize()
    assert lib.selscan_device_status(0, s2.cuda_stream) == TIMEOUT
    assert lib.selscan_device_status(1, s2.cuda_stream) == TIMEOUT
    assert lib.selscan_device_status(0, s1.cuda_stream) == OK
