"""Torch-facing wrappers of the libselscan entry points.

torch provides device memory and the current stream; the library does all of the work.
Shapes and layouts follow include/selscan.h:
  u, delta, z, out (batch, dim, seqlen); B, C (batch, 16, seqlen); A (dim, 16) fp32;
  D, delta_bias (dim) fp32; states (batch, dim, 16) fp32.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib

_DT = {torch.float32: _lib.F32, torch.bfloat16: _lib.BF16}


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check_dev(name, t, dtype=None, shape=None, device=None):
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _stream_handle(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def workspace_size(batch: int, dim: int, dstate: int, seqlen: int) -> int:
    """Bytes of workspace ssm_scan_fwd needs on the current device (0 = none)."""
    return int(_lib.lib().ssm_scan_workspace_size(batch, dim, dstate, seqlen))


def scan_plan(batch: int, dim: int, dstate: int, seqlen: int, workspace_bytes: int | None = None,
              in_dtype=torch.bfloat16, softplus: bool = True, zoh: bool = False,
              sms: int = 0) -> dict:
    """How ssm_scan_fwd launches this shape (ssm_scan_plan) on the current device, or with sms > 0
    on a GPU of that many SMs (no device needed). With workspace_bytes None, the plan for a
    workspace large enough for it (what workspace_size() returns on that GPU)."""
    if workspace_bytes is None:
        workspace_bytes = 1 << 62
    info = (ctypes.c_int64 * 8)()
    st = _lib.lib().ssm_scan_plan(batch, dim, dstate, seqlen, _DT[in_dtype], _flags(softplus, zoh),
                                  workspace_bytes, sms, info)
    _lib.check("ssm_scan_plan", st)
    keys = ("rows_per_lane", "whole_blocks", "split_blocks", "segments", "segment_tokens",
            "channels_per_block", "workspace_bytes", "required_workspace_bytes")
    return dict(zip(keys, (int(v) for v in info)))


def ssd_plan(batch: int, seqlen: int, nheads: int, sms: int = 0) -> dict:
    """The balanced launch of ssd_chunk_scan_fwd (ssd_chunk_scan_plan) on the current device, or
    with sms > 0 on a GPU of that many SMs (no device needed)."""
    info = (ctypes.c_int64 * 5)()
    st = _lib.lib().ssd_chunk_scan_plan(batch, seqlen, nheads, sms, info)
    _lib.check("ssd_chunk_scan_plan", st)
    keys = ("whole_chains", "cut_chains", "segments", "segment_chunks", "workspace_bytes")
    return dict(zip(keys, (int(v) for v in info)))


def bwd_plan(batch: int, dim: int, dstate: int, seqlen: int, checkpoints: bool = False,
             sms: int = 0) -> dict:
    """How ssm_scan_bwd launches this shape (ssm_scan_bwd_plan) on the current device, or with
    sms > 0 on a GPU of that many SMs (no device needed)."""
    info = (ctypes.c_int64 * 6)()
    st = _lib.lib().ssm_scan_bwd_plan(batch, dim, dstate, seqlen, int(checkpoints), sms, info)
    _lib.check("ssm_scan_bwd_plan", st)
    keys = ("segments", "segment_tokens", "channels_per_cta", "ctas", "ctas_per_sm",
            "workspace_bytes")
    return dict(zip(keys, (int(v) for v in info)))


def _flags(softplus, zoh):
    return (_lib.FLAG_SOFTPLUS if softplus else 0) | (_lib.FLAG_ZOH if zoh else 0)


def ssm_scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                 out=None, final_state=None, initial_state=None, workspace=None,
                 out_dtype=None, return_final_state=True, stream=None, zoh=False):
    """Selective scan over whole sequences. Returns (out, final_state or None).
    zoh: zero-order-hold discretisation of B instead of Euler."""
    if u.dim() != 3:
        raise ValueError("u must be (batch, dim, seqlen)")
    batch, dim, seqlen = u.shape
    dstate = A.shape[-1]
    in_dt = u.dtype
    if in_dt not in _DT:
        raise ValueError(f"unsupported input dtype {in_dt}")
    dev = u.device
    _check_dev("u", u, in_dt, (batch, dim, seqlen), dev)
    _check_dev("delta", delta, in_dt, (batch, dim, seqlen), dev)
    _check_dev("A", A, torch.float32, (dim, dstate), dev)
    _check_dev("B", B, in_dt, (batch, dstate, seqlen), dev)
    _check_dev("C", C, in_dt, (batch, dstate, seqlen), dev)
    _check_dev("D", D, torch.float32, (dim,), dev)
    _check_dev("z", z, in_dt, (batch, dim, seqlen), dev)
    _check_dev("delta_bias", delta_bias, torch.float32, (dim,), dev)
    _check_dev("initial_state", initial_state, torch.float32, (batch, dim, dstate), dev)
    if out is None:
        out = torch.empty((batch, dim, seqlen), dtype=out_dtype or in_dt, device=dev)
    if out.dtype not in _DT:
        raise ValueError(f"unsupported output dtype {out.dtype}")
    _check_dev("out", out, None, (batch, dim, seqlen), dev)
    if final_state is None and return_final_state:
        final_state = torch.empty((batch, dim, dstate), dtype=torch.float32, device=dev)
    _check_dev("final_state", final_state, torch.float32, (batch, dim, dstate), dev)
    with torch.cuda.device(dev):
        need = workspace_size(batch, dim, dstate, seqlen)
        if need and workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        _check_dev("workspace", workspace, None, None, dev)
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        st = _lib.lib().ssm_scan_fwd(
            _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
            _flags(delta_softplus, zoh), _ptr(out), _ptr(final_state), batch, dim, dstate, seqlen,
            _DT[in_dt], _DT[out.dtype], _ptr(initial_state), _ptr(workspace), ws_bytes,
            _stream_handle(stream))
    _lib.check("ssm_scan_fwd", st)
    return out, final_state


def ssm_state_update(state, x, dt, A, B, C, D=None, z=None, out=None, dt_bias=None,
                     dt_softplus=True, out_dtype=None, stream=None, zoh=False):
    """One token: updates `state` in place and returns out (batch, dim)."""
    batch, dim, dstate = state.shape
    in_dt = x.dtype
    if in_dt not in _DT:
        raise ValueError(f"unsupported input dtype {in_dt}")
    dev = state.device
    _check_dev("state", state, torch.float32, (batch, dim, dstate), dev)
    _check_dev("x", x, in_dt, (batch, dim), dev)
    _check_dev("dt", dt, in_dt, (batch, dim), dev)
    _check_dev("A", A, torch.float32, (dim, dstate), dev)
    _check_dev("B", B, in_dt, (batch, dstate), dev)
    _check_dev("C", C, in_dt, (batch, dstate), dev)
    _check_dev("D", D, torch.float32, (dim,), dev)
    _check_dev("z", z, in_dt, (batch, dim), dev)
    _check_dev("dt_bias", dt_bias, torch.float32, (dim,), dev)
    if out is None:
        out = torch.empty((batch, dim), dtype=out_dtype or in_dt, device=dev)
    if out.dtype not in _DT:
        raise ValueError(f"unsupported output dtype {out.dtype}")
    _check_dev("out", out, None, (batch, dim), dev)
    with torch.cuda.device(dev):
        st = _lib.lib().ssm_state_update(
            _ptr(state), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
            _ptr(out), _ptr(dt_bias), _flags(dt_softplus, zoh), batch, dim, dstate, _DT[in_dt],
            _DT[out.dtype], _stream_handle(stream))
    _lib.check("ssm_state_update", st)
    return out


def ssm_scan_fwd_no_alloc(u, delta, A, B, C, D=None, z=None, delta_bias=None,
                          delta_softplus=True, out=None, final_state=None, initial_state=None,
                          out_dtype=None, return_final_state=True, stream=None, zoh=False):
    """ssm_scan_fwd without a workspace, for callers that cannot allocate device scratch.

    The library's time-split scratch comes from its own fixed device array
    (NO_ALLOC_SCRATCH_BYTES per GPU), shared by every call: calls that overlap on the GPU race.
    Shapes that need more scratch raise SelscanError (SELSCAN_ERR_SCRATCH_LIMIT). The first
    call on a device should come before any stream capture on it. `out` and `final_state` are
    allocated here only when not given.
    """
    if u.dim() != 3:
        raise ValueError("u must be (batch, dim, seqlen)")
    batch, dim, seqlen = u.shape
    dstate = A.shape[-1]
    in_dt = u.dtype
    if in_dt not in _DT:
        raise ValueError(f"unsupported input dtype {in_dt}")
    dev = u.device
    _check_dev("u", u, in_dt, (batch, dim, seqlen), dev)
    _check_dev("delta", delta, in_dt, (batch, dim, seqlen), dev)
    _check_dev("A", A, torch.float32, (dim, dstate), dev)
    _check_dev("B", B, in_dt, (batch, dstate, seqlen), dev)
    _check_dev("C", C, in_dt, (batch, dstate, seqlen), dev)
    _check_dev("D", D, torch.float32, (dim,), dev)
    _check_dev("z", z, in_dt, (batch, dim, seqlen), dev)
    _check_dev("delta_bias", delta_bias, torch.float32, (dim,), dev)
    _check_dev("initial_state", initial_state, torch.float32, (batch, dim, dstate), dev)
    if out is None:
        out = torch.empty((batch, dim, seqlen), dtype=out_dtype or in_dt, device=dev)
    if out.dtype not in _DT:
        raise ValueError(f"unsupported output dtype {out.dtype}")
    _check_dev("out", out, None, (batch, dim, seqlen), dev)
    if final_state is None and return_final_state:
        final_state = torch.empty((batch, dim, dstate), dtype=torch.float32, device=dev)
    _check_dev("final_state", final_state, torch.float32, (batch, dim, dstate), dev)
    with torch.cuda.device(dev):
        st = _lib.lib().ssm_scan_fwd_no_alloc(
            _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
            _flags(delta_softplus, zoh), _ptr(out), _ptr(final_state), batch, dim, dstate, seqlen,
            _DT[in_dt], _DT[out.dtype], _ptr(initial_state), _stream_handle(stream))
    _lib.check("ssm_scan_fwd_no_alloc", st)
    return out, final_state


def ssm_conv_state_update(conv_state, x, conv_weight, conv_bias=None, conv_silu=True,
                          state=None, dt=None, A=None, B=None, C=None, D=None, z=None, out=None,
                          dt_bias=None, dt_softplus=True, out_dtype=None, conv_out=None,
                          return_conv_out=False, stream=None, zoh=False):
    """Decode step of the short convolution (conv_state (batch, dim, 4) rolled in place) and,
    when `state` is given, of the selective state with the convolution output as its input.
    Returns (out or None, conv_out or None)."""
    batch, dim, width = conv_state.shape
    in_dt = x.dtype
    if in_dt not in _DT:
        raise ValueError(f"unsupported input dtype {in_dt}")
    dev = conv_state.device
    _check_dev("conv_state", conv_state, in_dt, (batch, dim, width), dev)
    _check_dev("x", x, in_dt, (batch, dim), dev)
    _check_dev("conv_weight", conv_weight, torch.float32, (dim, width), dev)
    _check_dev("conv_bias", conv_bias, torch.float32, (dim,), dev)
    if conv_out is None and (return_conv_out or state is None):
        conv_out = torch.empty((batch, dim), dtype=in_dt, device=dev)
    _check_dev("conv_out", conv_out, in_dt, (batch, dim), dev)
    dstate = 16
    if state is not None:
        dstate = state.shape[-1]
        _check_dev("state", state, torch.float32, (batch, dim, dstate), dev)
        _check_dev("dt", dt, in_dt, (batch, dim), dev)
        _check_dev("A", A, torch.float32, (dim, dstate), dev)
        _check_dev("B", B, in_dt, (batch, dstate), dev)
        _check_dev("C", C, in_dt, (batch, dstate), dev)
        _check_dev("D", D, torch.float32, (dim,), dev)
        _check_dev("z", z, in_dt, (batch, dim), dev)
        _check_dev("dt_bias", dt_bias, torch.float32, (dim,), dev)
        if out is None:
            out = torch.empty((batch, dim), dtype=out_dtype or in_dt, device=dev)
        _check_dev("out", out, None, (batch, dim), dev)
    odt = _DT[out.dtype] if out is not None else _DT[in_dt]
    with torch.cuda.device(dev):
        st = _lib.lib().ssm_conv_state_update(
            _ptr(conv_state), _ptr(x), _ptr(conv_weight), _ptr(conv_bias), int(bool(conv_silu)),
            width, _ptr(conv_out), _ptr(state), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
            _ptr(z), _ptr(out), _ptr(dt_bias), _flags(dt_softplus, zoh), batch, dim, dstate,
            _DT[in_dt], odt, _stream_handle(stream))
    _lib.check("ssm_conv_state_update", st)
    return out, conv_out


def bwd_workspace_size(batch: int, dim: int, dstate: int, seqlen: int,
                       checkpoints_given: bool = False) -> int:
    """Bytes of workspace ssm_scan_bwd needs on the current device."""
    return int(_lib.lib().ssm_scan_bwd_workspace_size(batch, dim, dstate, seqlen,
                                                      int(bool(checkpoints_given))))


def ssm_scan_fwd_ckpt(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                      out=None, final_state=None, initial_state=None, workspace=None,
                      out_dtype=None, checkpoints=None, stream=None):
    """ssm_scan_fwd that also returns the state before every 16th token
    (batch, dim, ceil(seqlen/16), 16) fp32, for ssm_scan_bwd(..., checkpoints=...).
    Returns (out, final_state, checkpoints)."""
    batch, dim, seqlen = u.shape
    dstate = A.shape[-1]
    dev = u.device
    if checkpoints is None:
        checkpoints = torch.empty((batch, dim, (seqlen + 15) // 16, dstate), dtype=torch.float32,
                                  device=dev)
    _check_dev("checkpoints", checkpoints, torch.float32, (batch, dim, (seqlen + 15) // 16, dstate), dev)
    if out is None:
        out = torch.empty((batch, dim, seqlen), dtype=out_dtype or u.dtype, device=dev)
    if final_state is None:
        final_state = torch.empty((batch, dim, dstate), dtype=torch.float32, device=dev)
    for name, t in (("u", u), ("delta", delta), ("A", A), ("B", B), ("C", C), ("D", D), ("z", z),
                    ("delta_bias", delta_bias), ("initial_state", initial_state), ("out", out),
                    ("final_state", final_state)):
        _check_dev(name, t, None, None, dev)
    with torch.cuda.device(dev):
        need = workspace_size(batch, dim, dstate, seqlen)
        if need and workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        st = _lib.lib().ssm_scan_fwd_ckpt(
            _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
            _flags(delta_softplus, False), _ptr(out), _ptr(final_state), batch, dim, dstate, seqlen,
            _DT[u.dtype], _DT[out.dtype], _ptr(initial_state), _ptr(workspace), ws_bytes,
            _ptr(checkpoints), _stream_handle(stream))
    _lib.check("ssm_scan_fwd_ckpt", st)
    return out, final_state, checkpoints


def ssm_scan_bwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                 initial_state=None, dout=None, dfinal_state=None, workspace=None, stream=None,
                 checkpoints=None):
    """Gradients of sum(dout*out) + sum(dfinal_state*final_state) of ssm_scan_fwd (Euler) with
    respect to its inputs. dout (batch, dim, seqlen) sets the dtype of du, ddelta and dz; the
    other gradients are fp32. checkpoints: the states ssm_scan_fwd_ckpt saved (skips the
    backward's own forward pass). Returns a dict with keys du, ddelta, dA, dB, dC, dD, dz,
    ddelta_bias, dinitial_state (None where the matching input is None)."""
    if u.dim() != 3:
        raise ValueError("u must be (batch, dim, seqlen)")
    batch, dim, seqlen = u.shape
    dstate = A.shape[-1]
    in_dt = u.dtype
    if in_dt not in _DT:
        raise ValueError(f"unsupported input dtype {in_dt}")
    if dout is None:
        raise ValueError("dout is required")
    g_dt = dout.dtype
    if g_dt not in _DT:
        raise ValueError(f"unsupported gradient dtype {g_dt}")
    dev = u.device
    act = (batch, dim, seqlen)
    _check_dev("u", u, in_dt, act, dev)
    _check_dev("delta", delta, in_dt, act, dev)
    _check_dev("A", A, torch.float32, (dim, dstate), dev)
    _check_dev("B", B, in_dt, (batch, dstate, seqlen), dev)
    _check_dev("C", C, in_dt, (batch, dstate, seqlen), dev)
    _check_dev("D", D, torch.float32, (dim,), dev)
    _check_dev("z", z, in_dt, act, dev)
    _check_dev("delta_bias", delta_bias, torch.float32, (dim,), dev)
    _check_dev("initial_state", initial_state, torch.float32, (batch, dim, dstate), dev)
    _check_dev("dout", dout, g_dt, act, dev)
    _check_dev("dfinal_state", dfinal_state, torch.float32, (batch, dim, dstate), dev)
    f32 = torch.float32
    g = {
        "du": torch.empty(act, dtype=g_dt, device=dev),
        "ddelta": torch.empty(act, dtype=g_dt, device=dev),
        "dA": torch.empty((dim, dstate), dtype=f32, device=dev),
        "dB": torch.empty((batch, dstate, seqlen), dtype=f32, device=dev),
        "dC": torch.empty((batch, dstate, seqlen), dtype=f32, device=dev),
        "dD": None if D is None else torch.empty(dim, dtype=f32, device=dev),
        "dz": None if z is None else torch.empty(act, dtype=g_dt, device=dev),
        "ddelta_bias": None if delta_bias is None else torch.empty(dim, dtype=f32, device=dev),
        "dinitial_state": (None if initial_state is None
                           else torch.empty((batch, dim, dstate), dtype=f32, device=dev)),
    }
    _check_dev("checkpoints", checkpoints, torch.float32, (batch, dim, (seqlen + 15) // 16, dstate), dev)
    with torch.cuda.device(dev):
        need = bwd_workspace_size(batch, dim, dstate, seqlen, checkpoints is not None)
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        _check_dev("workspace", workspace, None, None, dev)
        st = _lib.lib().ssm_scan_bwd(
            _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
            _flags(delta_softplus, False), _ptr(initial_state), _ptr(dout), _ptr(dfinal_state),
            _ptr(g["du"]), _ptr(g["ddelta"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]),
            _ptr(g["dD"]), _ptr(g["dz"]), _ptr(g["ddelta_bias"]), _ptr(g["dinitial_state"]),
            batch, dim, dstate, seqlen, _DT[in_dt], _DT[g_dt], _ptr(checkpoints), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _lib.check("ssm_scan_bwd", st)
    return g


def ssd_workspace_size(batch: int, seqlen: int, nheads: int) -> int:
    """Bytes of workspace ssd_chunk_scan_fwd uses on the current device to balance the last wave
    of (batch x nheads) chains (0 = it runs them unsplit)."""
    return int(_lib.lib().ssd_chunk_scan_workspace_size(batch, seqlen, nheads))


def ssd_chunk_scan_fwd(x, dt, A, B, C, D=None, z=None, dt_bias=None, dt_softplus=True,
                       initial_state=None, out_dtype=None, y=None, final_state=None,
                       return_final_state=True, workspace=None, balance=True, stream=None):
    """Mamba-2 SSD layer. x (batch, seqlen, nheads, 64) bf16, dt (batch, seqlen, nheads) bf16,
    A (nheads) fp32, B/C (batch, seqlen, ngroups, 128) bf16. Returns (y, final_state or None).
    With balance (the default) and no workspace given, one of ssd_workspace_size() bytes is
    allocated, so that the last wave of chains is cut into time segments; balance=False runs
    every chain unsplit."""
    if x.dim() != 4:
        raise ValueError("x must be (batch, seqlen, nheads, headdim)")
    batch, seqlen, nheads, headdim = x.shape
    if B.dim() != 4:
        raise ValueError("B must be (batch, seqlen, ngroups, dstate)")
    ngroups, dstate = B.shape[2], B.shape[3]
    in_dt = x.dtype
    if in_dt not in _DT:
        raise ValueError(f"unsupported input dtype {in_dt}")
    dev = x.device
    _check_dev("x", x, in_dt, (batch, seqlen, nheads, headdim), dev)
    _check_dev("dt", dt, in_dt, (batch, seqlen, nheads), dev)
    _check_dev("A", A, torch.float32, (nheads,), dev)
    _check_dev("B", B, in_dt, (batch, seqlen, ngroups, dstate), dev)
    _check_dev("C", C, in_dt, (batch, seqlen, ngroups, dstate), dev)
    _check_dev("D", D, torch.float32, (nheads,), dev)
    _check_dev("z", z, in_dt, (batch, seqlen, nheads, headdim), dev)
    _check_dev("dt_bias", dt_bias, torch.float32, (nheads,), dev)
    _check_dev("initial_state", initial_state, torch.float32, (batch, nheads, headdim, dstate), dev)
    if y is None:
        y = torch.empty((batch, seqlen, nheads, headdim), dtype=out_dtype or in_dt, device=dev)
    if y.dtype not in _DT:
        raise ValueError(f"unsupported output dtype {y.dtype}")
    _check_dev("y", y, None, (batch, seqlen, nheads, headdim), dev)
    if final_state is None and return_final_state:
        final_state = torch.empty((batch, nheads, headdim, dstate), dtype=torch.float32, device=dev)
    _check_dev("final_state", final_state, torch.float32, (batch, nheads, headdim, dstate), dev)
    with torch.cuda.device(dev):
        if balance and workspace is None:
            need = ssd_workspace_size(batch, seqlen, nheads)
            if need:
                workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        if not balance:
            workspace = None
        _check_dev("workspace", workspace, None, None, dev)
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        st = _lib.lib().ssd_chunk_scan_fwd(
            _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(dt_bias),
            _flags(dt_softplus, False), _ptr(y), _ptr(final_state), _ptr(initial_state), batch,
            seqlen, nheads, headdim, ngroups, dstate, _DT[in_dt], _DT[y.dtype], _ptr(workspace),
            ws_bytes, _stream_handle(stream))
    _lib.check("ssd_chunk_scan_fwd", st)
    return y, final_state


def _check_host(name, t, dtype=None, shape=None):
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def host_workspace_size(batch, dim, dstate, seqlen, in_dtype, out_dtype) -> int:
    """Device workspace bytes ssm_scan_fwd_host needs."""
    return int(_lib.lib().ssm_scan_fwd_host_workspace_size(batch, dim, dstate, seqlen,
                                                           _DT[in_dtype], _DT[out_dtype]))


def ssm_scan_fwd_host(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                      out=None, final_state=None, initial_state=None, workspace=None,
                      out_dtype=None, return_final_state=True, device=None, stream=None):
    """ssm_scan_fwd on host (CPU) tensors, pinned for overlap: the library uploads, scans and
    downloads slice by slice. Returns (out, final_state or None) as host tensors; they are valid
    after the stream (default: the current stream of `device`) has been synchronised."""
    if u.dim() != 3:
        raise ValueError("u must be (batch, dim, seqlen)")
    batch, dim, seqlen = u.shape
    dstate = A.shape[-1]
    in_dt = u.dtype
    if in_dt not in _DT:
        raise ValueError(f"unsupported input dtype {in_dt}")
    _check_host("u", u, in_dt, (batch, dim, seqlen))
    _check_host("delta", delta, in_dt, (batch, dim, seqlen))
    _check_host("A", A, torch.float32, (dim, dstate))
    _check_host("B", B, in_dt, (batch, dstate, seqlen))
    _check_host("C", C, in_dt, (batch, dstate, seqlen))
    _check_host("D", D, torch.float32, (dim,))
    _check_host("z", z, in_dt, (batch, dim, seqlen))
    _check_host("delta_bias", delta_bias, torch.float32, (dim,))
    _check_host("initial_state", initial_state, torch.float32, (batch, dim, dstate))
    odt = out_dtype or in_dt
    if out is None:
        out = torch.empty((batch, dim, seqlen), dtype=odt).pin_memory()
    _check_host("out", out, None, (batch, dim, seqlen))
    if final_state is None and return_final_state:
        final_state = torch.empty((batch, dim, dstate), dtype=torch.float32).pin_memory()
    _check_host("final_state", final_state, torch.float32, (batch, dim, dstate))
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        need = host_workspace_size(batch, dim, dstate, seqlen, in_dt, out.dtype)
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        _check_dev("workspace", workspace, None, None, dev)
        st = _lib.lib().ssm_scan_fwd_host(
            _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
            _flags(delta_softplus, False), _ptr(out), _ptr(final_state), batch, dim, dstate,
            seqlen, _DT[in_dt], _DT[out.dtype], _ptr(initial_state), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _lib.check("ssm_scan_fwd_host", st)
    return out, final_state
