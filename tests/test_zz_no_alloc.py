"""ssm_scan_fwd_no_alloc against ssm_scan_fwd on the GPU, through the C ABI.

The no-alloc entry point serves callers that cannot allocate device memory (code under a host
framework that owns every device allocation, or a loop that must not call cudaMalloc because
it can synchronise the device). It takes the time-split scratch from the library's own fixed
device array instead of a caller workspace. These tests use shapes that do take the time-split
path, so the fixed array is really used, and check two calls in a row (different inputs, the
second reusing whatever the first left in the array) against the workspace entry point.

This file is named so that pytest collects it last.
"""
import pytest
import torch

from selective_state_space_110_b300 import (SelscanError, ssm_scan_fwd, ssm_scan_fwd_no_alloc,
                                            workspace_size)
from selective_state_space_110_b300 import _lib
from tests.parity import TOL, assert_close
from workloads import ScanConfig, make_scan_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"

# Two different segmented shapes, run back to back.
CALLS = [(1, 64, 40960, 21), (2, 16, 20000, 22)]


def _args(x):
    return (x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"],
            x["delta_softplus"])


def test_no_alloc_matches_workspace_entry_point_on_two_calls():
    for batch, dim, seqlen, seed in CALLS:
        need = workspace_size(batch, dim, 16, seqlen)
        assert 0 < need <= _lib.NO_ALLOC_SCRATCH_BYTES, need
    results = []
    for batch, dim, seqlen, seed in CALLS:
        cfg = ScanConfig("na", batch, dim, 16, seqlen, "bf16", "f32", 1e-3, 1e-1, seed)
        x = make_scan_inputs(cfg, DEV)
        h0 = torch.randn(batch, dim, 16, device=DEV,
                         generator=torch.Generator(DEV).manual_seed(seed))
        got = ssm_scan_fwd_no_alloc(*_args(x), out_dtype=torch.float32, initial_state=h0)
        results.append((x, h0, got))
    torch.cuda.synchronize()
    for x, h0, (out, fin) in results:
        ref, rfin = ssm_scan_fwd(*_args(x), out_dtype=torch.float32, initial_state=h0)
        torch.cuda.synchronize()
        assert_close(out, ref.double(), TOL[torch.bfloat16], "no-alloc y vs ssm_scan_fwd")
        assert_close(fin, rfin.double(), TOL[torch.bfloat16], "no-alloc final state vs ssm_scan_fwd")


def test_no_alloc_without_time_split():
    """A shape that needs no scratch at all goes through unchanged."""
    cfg = ScanConfig("na", 2, 96, 16, 512, "bf16", "f32", 1e-3, 1e-1, 23)
    assert workspace_size(2, 96, 16, 512) == 0
    x = make_scan_inputs(cfg, DEV)
    out, fin = ssm_scan_fwd_no_alloc(*_args(x), out_dtype=torch.float32)
    ref, rfin = ssm_scan_fwd(*_args(x), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert_close(out, ref.double(), TOL[torch.bfloat16], "y")
    assert_close(fin, rfin.double(), TOL[torch.bfloat16], "final state")


def test_no_alloc_rejects_shapes_beyond_the_fixed_scratch():
    """Shapes needing more scratch than the fixed array are refused before any launch. The
    pointers are fake, 16-byte aligned addresses: the size check comes first and nothing is
    dereferenced."""
    shapes = [(1, 1536, 1 << 20), (1, 3072, 1 << 21), (2, 4096, 1 << 22)]
    big = [s for s in shapes if workspace_size(s[0], s[1], 16, s[2]) > _lib.NO_ALLOC_SCRATCH_BYTES]
    assert big, "no candidate shape exceeds the fixed scratch on this device"
    b, d, L = big[0]
    fake = [(1 << 40) + i * (1 << 38) for i in range(11)]
    lib = _lib.lib()
    st = lib.ssm_scan_fwd_no_alloc(fake[0], fake[1], fake[2], fake[3], fake[4], fake[5], fake[6],
                                   fake[7], 1, fake[8], fake[9], b, d, 16, L, _lib.BF16,
                                   _lib.BF16, None, None)
    assert st == 6
    assert b"SCRATCH_LIMIT" in lib.selscan_status_string(st)
    with pytest.raises(SelscanError, match="SCRATCH_LIMIT"):
        _lib.check("ssm_scan_fwd_no_alloc", st)


def test_no_alloc_segmented_against_the_oracle():
    """The fixed-scratch path checked directly against the fp64 oracle (not only through
    ssm_scan_fwd), on a time-split shape, with an initial state and bf16 output."""
    import oracle
    batch, dim, seqlen = 2, 24, 24576
    assert 0 < workspace_size(batch, dim, 16, seqlen) <= _lib.NO_ALLOC_SCRATCH_BYTES
    cfg = ScanConfig("na", batch, dim, 16, seqlen, "bf16", "bf16", 1e-3, 1e-1, 24)
    x = make_scan_inputs(cfg, DEV)
    h0 = torch.randn(batch, dim, 16, device=DEV, generator=torch.Generator(DEV).manual_seed(25))
    for _ in range(2):  # the second call finds the first call's values in the array
        out, fin = ssm_scan_fwd_no_alloc(*_args(x), initial_state=h0)
        torch.cuda.synchronize()
        ref, rfin = oracle.scan_fwd(*_args(x), initial_state=h0)
        assert_close(out, ref, TOL[torch.bfloat16], "no-alloc y vs oracle")
        assert_close(fin, rfin, TOL[torch.bfloat16], "no-alloc final state vs oracle")
