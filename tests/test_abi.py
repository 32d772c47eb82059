"""The C ABI without a GPU: the library loads, exports every declared symbol, and rejects
bad arguments with the documented status before touching any device (no compute here)."""
import ctypes
import os
import re

import pytest

from selective_state_space_110_b300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "selscan.h")

OK, INVALID, UNSUP, ALIGN, WS, CUDA = 0, 1, 2, 3, 4, 5


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)) - {"defined"})


@pytest.fixture(scope="module")
def lib():
    return _lib.lib()


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(_lib.EXPORTS), names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code, name in _lib.STATUS.items():
        assert lib.selscan_status_string(code).decode().startswith(name)
    assert b"UNKNOWN" in lib.selscan_status_string(99)


# Fake, 16-byte aligned, non-overlapping addresses: validation never dereferences them.
BASE = 1 << 40
GAP = 1 << 36


def fake(i):
    return BASE + i * GAP


def scan_args(**kw):
    a = dict(u=fake(0), delta=fake(1), A=fake(2), B=fake(3), C=fake(4), D=fake(5), z=fake(6),
             delta_bias=fake(7), softplus=1, out=fake(8), final_state=fake(9), batch=2, dim=64,
             dstate=16, seqlen=128, in_dtype=_lib.BF16, out_dtype=_lib.BF16, initial_state=None,
             workspace=None, ws_bytes=0, stream=None)
    a.update(kw)
    return a


def call_scan(lib, **kw):
    a = scan_args(**kw)
    return lib.ssm_scan_fwd(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"],
                            a["delta_bias"], a["softplus"], a["out"], a["final_state"], a["batch"],
                            a["dim"], a["dstate"], a["seqlen"], a["in_dtype"], a["out_dtype"],
                            a["initial_state"], a["workspace"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(dstate=8), UNSUP),
    (dict(dstate=32), UNSUP),
    (dict(in_dtype=7), UNSUP),
    (dict(out_dtype=-1), UNSUP),
    (dict(batch=0), INVALID),
    (dict(dim=0), INVALID),
    (dict(seqlen=-1), INVALID),
    (dict(batch=70000), INVALID),
    (dict(u=None), INVALID),
    (dict(delta=None), INVALID),
    (dict(A=None), INVALID),
    (dict(B=None), INVALID),
    (dict(C=None), INVALID),
    (dict(out=None), INVALID),
    (dict(u=fake(0) + 2), ALIGN),
    (dict(z=fake(6) + 8), ALIGN),
    (dict(final_state=fake(9) + 4), ALIGN),
    (dict(out=fake(0) + 64), INVALID),          # out inside u
    (dict(final_state=fake(8) + 16), INVALID),  # final_state inside out
    (dict(out=fake(5)), INVALID),               # out over D
    (dict(initial_state=fake(9)), INVALID),     # final_state over initial_state
    (dict(softplus=4), INVALID),                # unknown flag bit
    (dict(softplus=-1), INVALID),
])
def test_scan_rejects(lib, kw, expect):
    assert call_scan(lib, **kw) == expect


def test_scan_valid_args_reach_the_device_check(lib):
    """Valid arguments pass every host check; on a machine without a CUDA device the call
    then stops at the device query with SELSCAN_ERR_CUDA (nothing is launched)."""
    import torch
    st = call_scan(lib)
    if torch.cuda.is_available():
        pytest.skip("device present: covered by the GPU tests")
    assert st == CUDA
    # seqlen = 0 needs no activation pointers
    assert call_scan(lib, seqlen=0, u=None, delta=None, B=None, C=None, out=None) == CUDA
    assert lib.ssm_scan_workspace_size(1, 1536, 16, 1 << 20) == 0
    assert lib.ssm_scan_workspace_size(1, 1536, 8, 1 << 20) == 0


def call_update(lib, **kw):
    a = dict(state=fake(0), x=fake(1), dt=fake(2), A=fake(3), B=fake(4), C=fake(5), D=fake(6),
             z=fake(7), out=fake(8), dt_bias=fake(9), softplus=1, batch=4, dim=5120, dstate=16,
             in_dtype=_lib.BF16, out_dtype=_lib.BF16, stream=None)
    a.update(kw)
    return lib.ssm_state_update(a["state"], a["x"], a["dt"], a["A"], a["B"], a["C"], a["D"],
                                a["z"], a["out"], a["dt_bias"], a["softplus"], a["batch"],
                                a["dim"], a["dstate"], a["in_dtype"], a["out_dtype"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(dstate=4), UNSUP),
    (dict(in_dtype=3), UNSUP),
    (dict(batch=0), INVALID),
    (dict(state=None), INVALID),
    (dict(x=None), INVALID),
    (dict(out=None), INVALID),
    (dict(B=fake(4) + 2), ALIGN),
    (dict(out=fake(0) + 32), INVALID),   # out inside state
    (dict(state=fake(1)), INVALID),      # state over x
    (dict(softplus=8), INVALID),         # unknown flag bit
])
def test_update_rejects(lib, kw, expect):
    assert call_update(lib, **kw) == expect


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        _lib.load()


def test_no_alloc_scratch_size_matches_header():
    text = open(HEADER).read()
    m = re.search(r"#define SELSCAN_NO_ALLOC_SCRATCH_BYTES \(\(size_t\)(\d+)\)", text)
    assert m and int(m.group(1)) == _lib.NO_ALLOC_SCRATCH_BYTES


def call_conv(lib, **kw):
    a = dict(conv_state=fake(0), x=fake(1), w=fake(2), cb=fake(3), silu=1, width=4, conv_out=fake(4),
             state=fake(5), dt=fake(6), A=fake(7), B=fake(8), C=fake(9), D=fake(10), z=fake(11),
             out=fake(12), dt_bias=fake(13), flags=1, batch=4, dim=512, dstate=16,
             in_dtype=_lib.BF16, out_dtype=_lib.BF16, stream=None)
    a.update(kw)
    return lib.ssm_conv_state_update(a["conv_state"], a["x"], a["w"], a["cb"], a["silu"], a["width"],
                                     a["conv_out"], a["state"], a["dt"], a["A"], a["B"], a["C"], a["D"],
                                     a["z"], a["out"], a["dt_bias"], a["flags"], a["batch"], a["dim"],
                                     a["dstate"], a["in_dtype"], a["out_dtype"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(width=3), UNSUP),
    (dict(dstate=8), UNSUP),
    (dict(conv_state=None), INVALID),
    (dict(x=None), INVALID),
    (dict(w=None), INVALID),
    (dict(dt=None), INVALID),                  # needed when state is given
    (dict(state=None, conv_out=None), INVALID),  # conv step alone must write conv_out
    (dict(flags=4), INVALID),
    (dict(x=fake(1) + 2), ALIGN),
    (dict(conv_out=fake(0) + 16), INVALID),    # conv_out inside conv_state
    (dict(out=fake(5) + 64), INVALID),         # out inside state
    (dict(conv_state=fake(2)), INVALID),       # conv_state over the weights
])
def test_conv_update_rejects(lib, kw, expect):
    assert call_conv(lib, **kw) == expect


def test_conv_update_valid_args_reach_the_device_check(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("device present: covered by the GPU tests")
    assert call_conv(lib) == CUDA
    assert call_conv(lib, state=None, dt=None, A=None, B=None, C=None, out=None) == CUDA


def call_bwd(lib, **kw):
    a = dict(u=fake(0), delta=fake(1), A=fake(2), B=fake(3), C=fake(4), D=fake(5), z=fake(6),
             delta_bias=fake(7), flags=1, h0=fake(8), dout=fake(9), dfinal=fake(10), du=fake(11),
             ddelta=fake(12), dA=fake(13), dB=fake(14), dC=fake(15), dD=fake(16), dz=fake(17),
             dbias=fake(18), dh0=fake(19), batch=2, dim=64, dstate=16, seqlen=128,
             in_dtype=_lib.BF16, g_dtype=_lib.BF16, ws=fake(20), ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return lib.ssm_scan_bwd(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"],
                            a["delta_bias"], a["flags"], a["h0"], a["dout"], a["dfinal"], a["du"],
                            a["ddelta"], a["dA"], a["dB"], a["dC"], a["dD"], a["dz"], a["dbias"],
                            a["dh0"], a["batch"], a["dim"], a["dstate"], a["seqlen"],
                            a["in_dtype"], a["g_dtype"], a.get("ckpt"), a["ws"], a["ws_bytes"],
                            a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(dstate=8), UNSUP),
    (dict(g_dtype=5), UNSUP),
    (dict(flags=3), UNSUP),                   # zero-order hold has no backward
    (dict(flags=4), INVALID),
    (dict(batch=0), INVALID),
    (dict(dout=None), INVALID),
    (dict(du=None), INVALID),
    (dict(dA=None), INVALID),
    (dict(dB=None), INVALID),
    (dict(dz=None), INVALID),                 # z given without dz
    (dict(z=None), INVALID),                  # dz given without z
    (dict(dC=fake(14) + 64), INVALID),        # dC inside dB
    (dict(du=fake(0) + 32), INVALID),         # du inside u
    (dict(ws=None, ws_bytes=0), WS),
    (dict(ws_bytes=0), WS),
    (dict(dout=fake(9) + 8), ALIGN),
    (dict(ckpt=fake(21) + 4), ALIGN),
    (dict(ckpt=fake(11) + 64), INVALID),      # checkpoints (an input) inside du (an output)
])
def test_bwd_rejects(lib, kw, expect):
    assert call_bwd(lib, **kw) == expect


def test_bwd_valid_args_reach_the_device_check(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("device present: covered by the GPU tests")
    assert call_bwd(lib) == CUDA
    assert call_bwd(lib, z=None, dz=None, D=None, dD=None, h0=None, dh0=None, dfinal=None) == CUDA
    # The workspace size depends on the device (time segments); without one it is 0.
    assert lib.ssm_scan_bwd_workspace_size(2, 64, 16, 128, 0) == 0
    assert lib.ssm_scan_bwd_workspace_size(2, 64, 8, 128, 1) == 0


def call_ssd(lib, **kw):
    a = dict(x=fake(0), dt=fake(1), A=fake(2), B=fake(3), C=fake(4), D=fake(5), z=fake(6),
             dt_bias=fake(7), flags=1, y=fake(8), fin=fake(9), h0=None, batch=2, seqlen=256,
             nheads=8, headdim=64, ngroups=1, dstate=128, in_dtype=_lib.BF16, out_dtype=_lib.BF16,
             ws=None, ws_bytes=0, stream=None)
    a.update(kw)
    return lib.ssd_chunk_scan_fwd(a["x"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["z"],
                                  a["dt_bias"], a["flags"], a["y"], a["fin"], a["h0"], a["batch"],
                                  a["seqlen"], a["nheads"], a["headdim"], a["ngroups"],
                                  a["dstate"], a["in_dtype"], a["out_dtype"], a["ws"],
                                  a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(headdim=128), UNSUP),
    (dict(dstate=64), UNSUP),
    (dict(in_dtype=_lib.F32), UNSUP),
    (dict(out_dtype=9), UNSUP),
    (dict(ngroups=3), INVALID),              # 8 heads do not split into 3 groups
    (dict(flags=2), INVALID),                # zero-order hold is not an SSD option
    (dict(batch=0), INVALID),
    (dict(x=None), INVALID),
    (dict(A=None), INVALID),
    (dict(y=None), INVALID),
    (dict(y=fake(0) + 64), INVALID),         # y inside x
    (dict(fin=fake(8) + 16), INVALID),       # final state inside y
    (dict(h0=fake(9)), INVALID),             # final state over the initial state
    (dict(B=fake(3) + 8), ALIGN),
    (dict(ws=fake(10) + 8, ws_bytes=1 << 20), ALIGN),
])
def test_ssd_rejects(lib, kw, expect):
    assert call_ssd(lib, **kw) == expect


def test_ssd_valid_args_reach_the_device_check(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("device present: covered by the GPU tests")
    assert call_ssd(lib) == CUDA
    assert call_ssd(lib, seqlen=0, x=None, dt=None, B=None, C=None, y=None) == CUDA
    assert call_ssd(lib, ws=fake(10), ws_bytes=1 << 30) == CUDA
    # The balanced plan depends on the device's SM count; without a device it is 0 bytes.
    assert lib.ssd_chunk_scan_workspace_size(4, 2048, 80) == 0


def call_host(lib, **kw):
    a = dict(u=fake(0), delta=fake(1), A=fake(2), B=fake(3), C=fake(4), D=fake(5), z=fake(6),
             delta_bias=fake(7), flags=1, out=fake(8), fin=fake(9), batch=2, dim=64, dstate=16,
             seqlen=128, in_dtype=_lib.BF16, out_dtype=_lib.BF16, h0=None, ws=fake(10),
             ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return lib.ssm_scan_fwd_host(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"],
                                 a["delta_bias"], a["flags"], a["out"], a["fin"], a["batch"],
                                 a["dim"], a["dstate"], a["seqlen"], a["in_dtype"], a["out_dtype"],
                                 a["h0"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(dstate=8), UNSUP),
    (dict(in_dtype=4), UNSUP),
    (dict(batch=0), INVALID),
    (dict(u=None), INVALID),
    (dict(A=None), INVALID),
    (dict(ws=None), WS),
    (dict(ws_bytes=4096), WS),
    (dict(ws=fake(10) + 16), ALIGN),       # the workspace must be 256-byte aligned
])
def test_host_scan_rejects(lib, kw, expect):
    assert call_host(lib, **kw) == expect


def test_host_workspace_size(lib):
    n = lib.ssm_scan_fwd_host_workspace_size(2, 64, 16, 128, _lib.BF16, _lib.F32)
    # two slots of (u, delta, z, B, C, y, final and initial state) plus A, D, bias
    assert n >= 2 * (3 * 64 * 128 * 2 + 2 * 16 * 128 * 2 + 64 * 128 * 4 + 2 * 64 * 16 * 4)
    assert lib.ssm_scan_fwd_host_workspace_size(2, 64, 8, 128, _lib.BF16, _lib.F32) == 0


def test_fwd_ckpt_rejects(lib):
    a = scan_args()
    base = [a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"], a["delta_bias"]]
    tail = [a["out"], a["final_state"], a["batch"], a["dim"], a["dstate"], a["seqlen"],
            a["in_dtype"], a["out_dtype"], None, None, 0]
    assert lib.ssm_scan_fwd_ckpt(*base, 1, *tail, None, None) == INVALID          # no checkpoints
    assert lib.ssm_scan_fwd_ckpt(*base, 3, *tail, fake(12), None) == UNSUP        # zero-order hold
    assert lib.ssm_scan_fwd_ckpt(*base, 1, *tail, fake(12) + 8, None) == ALIGN
    assert lib.ssm_scan_fwd_ckpt(*base, 1, *tail, fake(8) + 16, None) == INVALID  # inside out


def test_plan_entry_points_reject_bad_arguments(lib):
    import ctypes
    info = (ctypes.c_int64 * 8)()
    assert lib.ssm_scan_plan(4, 5120, 16, 2048, _lib.BF16, 1, 0, -1, info) == INVALID
    assert lib.ssm_scan_plan(4, 5120, 16, 2048, _lib.BF16, 1, 0, 5000, info) == INVALID
    assert lib.ssm_scan_plan(4, 5120, 16, 2048, _lib.BF16, 1, 0, 148, None) == INVALID
    assert lib.ssm_scan_plan(4, 5120, 8, 2048, _lib.BF16, 1, 0, 148, info) == UNSUP
    assert lib.ssm_scan_plan(4, 5120, 16, 2048, _lib.BF16, 1, 0, 148, info) == 0
    assert lib.ssd_chunk_scan_plan(4, 2048, 80, 148, None) == INVALID
    assert lib.ssd_chunk_scan_plan(0, 2048, 80, 148, info) == INVALID
    assert lib.ssd_chunk_scan_plan(4, 2048, 80, -3, info) == INVALID
    assert lib.ssd_chunk_scan_plan(4, 2048, 80, 148, info) == 0 and info[1] == 24
