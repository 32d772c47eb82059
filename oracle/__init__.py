"""fp64 CPU oracle for the selective-SSM (S6) scan and the single-token state update.

TEST INFRASTRUCTURE ONLY: the plain, slow, sequential definition the CUDA path is checked
against. Only the tests, the smoke check and the benchmark's CPU-baseline leg use it; the
product path never imports it. It shares no code with the CUDA library.

The arithmetic lives in selscan_oracle.c (double precision, sequential in t, OpenMP over
independent (batch, channel) rows). Definition, from "Mamba and State Space Models"
(world.lapla.si): section "A State of Fixed Size" (h <- Abar*h + Bbar*x, then y = C*h),
section "Chosen by the Token" (Delta, B, C per token, A fixed, Abar = exp(Delta*A)) and
section "A Scan on the Chip" (discretise, then recur). Readings where the pages are silent:
Delta = softplus(delta + delta_bias); Euler Bbar*x = Delta*B*u (zero-order hold
((exp(Delta*A) - 1)/A)*B*u as an option); y = C*h + D*u, then times silu(z); zero initial state
unless one is given.

Every function here is pinned by tests/test_oracle_pins.py (LTI convolution, solved form of
the recurrence, Delta -> 0, large Delta, hand-worked N = 1 sequences, linearity in u).
"""
from __future__ import annotations

import ctypes

import numpy as np

from .build import build as _build, LIB as _LIB_PATH

_DP = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.c_int64


def _f64(a):
    """Contiguous float64 numpy copy of a numpy array or torch tensor (None passes through)."""
    if a is None:
        return None
    if hasattr(a, "detach"):
        import torch

        a = a.detach().to("cpu").to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a):
    return a.ctypes.data_as(_DP) if a is not None else None


class Oracle:
    """ctypes front end of one compiled copy of selscan_oracle.c."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.oracle_scan_fwd.restype = None
        lib.oracle_scan_fwd.argtypes = [_DP] * 8 + [ctypes.c_int, ctypes.c_int, _DP, _DP, _DP] + [_I64] * 4
        lib.oracle_scan_fwd_rows.restype = None
        lib.oracle_scan_fwd_rows.argtypes = ([_DP] * 8 + [ctypes.c_int, ctypes.c_int, _DP, _DP, _DP,
                                             ctypes.POINTER(ctypes.c_int64)] + [_I64] * 4)
        lib.oracle_state_update.restype = None
        lib.oracle_state_update.argtypes = [_DP] * 9 + [ctypes.c_int, ctypes.c_int, _DP] + [_I64] * 3
        lib.oracle_scan_bwd.restype = None
        lib.oracle_scan_bwd.argtypes = [_DP] * 8 + [ctypes.c_int] + [_DP] * 12 + [_I64] * 4
        lib.oracle_conv_step.restype = None
        lib.oracle_conv_step.argtypes = [_DP] * 4 + [ctypes.c_int, _DP] + [_I64] * 3
        lib.oracle_ssd_fwd.restype = None
        lib.oracle_ssd_fwd.argtypes = [_DP] * 8 + [ctypes.c_int, _DP, _DP, _DP] + [_I64] * 6
        lib.oracle_max_threads.restype = ctypes.c_int
        self._lib = lib
        self.path = path

    def max_threads(self) -> int:
        return int(self._lib.oracle_max_threads())

    def scan_fwd(self, u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                 initial_state=None, zoh=False):
        """Returns (out (batch, dim, seqlen), final_state (batch, dim, dstate)), float64.
        zoh: zero-order-hold discretisation of B instead of Euler."""
        u, delta, A, B, C = map(_f64, (u, delta, A, B, C))
        D, z, delta_bias, initial_state = map(_f64, (D, z, delta_bias, initial_state))
        batch, dim, seqlen = u.shape
        dstate = A.shape[1]
        assert delta.shape == u.shape and A.shape == (dim, dstate)
        assert B.shape == (batch, dstate, seqlen) and C.shape == B.shape
        assert z is None or z.shape == u.shape
        assert D is None or D.shape == (dim,)
        assert delta_bias is None or delta_bias.shape == (dim,)
        assert initial_state is None or initial_state.shape == (batch, dim, dstate)
        out = np.empty((batch, dim, seqlen), dtype=np.float64)
        fin = np.empty((batch, dim, dstate), dtype=np.float64)
        self._lib.oracle_scan_fwd(_p(u), _p(delta), _p(A), _p(B), _p(C), _p(D), _p(z),
                                  _p(delta_bias), int(bool(delta_softplus)), int(bool(zoh)),
                                  _p(initial_state),
                                  _p(out), _p(fin), batch, dim, dstate, seqlen)
        return out, fin

    def scan_fwd_rows(self, rows, u_rows, delta_rows, A, B, C, D=None, z_rows=None,
                      delta_bias=None, delta_softplus=True, initial_state_rows=None, zoh=False):
        """Scan of selected rows (flat indices b*dim + d) only.

        u_rows, delta_rows, z_rows: (nrows, seqlen) slices of the full tensors for those rows;
        A, D, delta_bias: full per-channel tensors; B, C: full (batch, dstate, seqlen).
        Returns (out (nrows, seqlen), final_state (nrows, dstate)).
        """
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        u_rows, delta_rows, A, B, C = map(_f64, (u_rows, delta_rows, A, B, C))
        D, z_rows, delta_bias, initial_state_rows = map(
            _f64, (D, z_rows, delta_bias, initial_state_rows))
        nrows, seqlen = u_rows.shape
        dim, dstate = A.shape
        assert rows.shape == (nrows,) and B.shape[1:] == (dstate, seqlen)
        assert rows.min(initial=0) >= 0 and rows.max(initial=0) < B.shape[0] * dim
        out = np.empty((nrows, seqlen), dtype=np.float64)
        fin = np.empty((nrows, dstate), dtype=np.float64)
        self._lib.oracle_scan_fwd_rows(
            _p(u_rows), _p(delta_rows), _p(A), _p(B), _p(C), _p(D), _p(z_rows), _p(delta_bias),
            int(bool(delta_softplus)), int(bool(zoh)), _p(initial_state_rows), _p(out), _p(fin),
            rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), nrows, dim, dstate, seqlen)
        return out, fin

    def state_update(self, state, x, dt, A, B, C, D=None, z=None, dt_bias=None, dt_softplus=True,
                     zoh=False):
        """One token. Returns (new_state (batch, dim, dstate), out (batch, dim)); inputs untouched."""
        st = _f64(state).copy()
        x, dt, A, B, C = map(_f64, (x, dt, A, B, C))
        D, z, dt_bias = map(_f64, (D, z, dt_bias))
        batch, dim, dstate = st.shape
        assert x.shape == (batch, dim) and dt.shape == x.shape and A.shape == (dim, dstate)
        assert B.shape == (batch, dstate) and C.shape == B.shape
        out = np.empty((batch, dim), dtype=np.float64)
        self._lib.oracle_state_update(_p(st), _p(x), _p(dt), _p(A), _p(B), _p(C), _p(D), _p(z),
                                      _p(dt_bias), int(bool(dt_softplus)), int(bool(zoh)), _p(out),
                                      batch, dim,
                                      dstate)
        return st, out


    def scan_bwd(self, u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                 initial_state=None, dout=None, dfinal=None):
        """Gradients of sum(dout*out) + sum(dfinal*final_state) with respect to every input of
        scan_fwd (Euler). Returns a dict of float64 arrays: du, ddelta, dA, dB, dC, dD, dz,
        ddelta_bias, dinitial_state (dD / dz / ddelta_bias / dinitial_state None when the
        corresponding input is None)."""
        u, delta, A, B, C = map(_f64, (u, delta, A, B, C))
        D, z, delta_bias, initial_state, dout, dfinal = map(
            _f64, (D, z, delta_bias, initial_state, dout, dfinal))
        batch, dim, seqlen = u.shape
        dstate = A.shape[1]
        assert dout is not None and dout.shape == u.shape
        g = {k: np.zeros(u.shape) for k in ("du", "ddelta")}
        g["dA"] = np.zeros(A.shape)
        g["dB"] = np.zeros(B.shape)
        g["dC"] = np.zeros(C.shape)
        g["dD"] = np.zeros(dim) if D is not None else None
        g["dz"] = np.zeros(u.shape) if z is not None else None
        g["ddelta_bias"] = np.zeros(dim) if delta_bias is not None else None
        g["dinitial_state"] = np.zeros((batch, dim, dstate)) if initial_state is not None else None
        self._lib.oracle_scan_bwd(
            _p(u), _p(delta), _p(A), _p(B), _p(C), _p(D), _p(z), _p(delta_bias),
            int(bool(delta_softplus)), _p(initial_state), _p(dout), _p(dfinal), _p(g["du"]),
            _p(g["ddelta"]), _p(g["dA"]), _p(g["dB"]), _p(g["dC"]), _p(g["dD"]), _p(g["dz"]),
            _p(g["ddelta_bias"]), _p(g["dinitial_state"]), batch, dim, dstate, seqlen)
        return g

    def ssd_fwd(self, x, dt, A, B, C, D=None, z=None, dt_bias=None, dt_softplus=True,
                initial_state=None):
        """Mamba-2 SSD layer by its recurrence. x (batch, seqlen, nheads, headdim), dt
        (batch, seqlen, nheads), A (nheads), B/C (batch, seqlen, ngroups, dstate). Returns
        (y like x, final_state (batch, nheads, headdim, dstate)) as float64."""
        x, dt, A, B, C = map(_f64, (x, dt, A, B, C))
        D, z, dt_bias, initial_state = map(_f64, (D, z, dt_bias, initial_state))
        batch, seqlen, nheads, headdim = x.shape
        ngroups, dstate = B.shape[2], B.shape[3]
        assert nheads % ngroups == 0 and C.shape == B.shape and dt.shape == x.shape[:3]
        y = np.empty(x.shape, dtype=np.float64)
        fin = np.empty((batch, nheads, headdim, dstate), dtype=np.float64)
        self._lib.oracle_ssd_fwd(_p(x), _p(dt), _p(A), _p(B), _p(C), _p(D), _p(z), _p(dt_bias),
                                 int(bool(dt_softplus)), _p(initial_state), _p(y), _p(fin),
                                 batch, seqlen, nheads, headdim, ngroups, dstate)
        return y, fin

    def conv_step(self, conv_state, x, weight, bias=None, silu=True):
        """One step of the short causal convolution. Returns (new_conv_state (batch, dim,
        width), u (batch, dim)); inputs untouched."""
        st = _f64(conv_state).copy()
        x, weight, bias = map(_f64, (x, weight, bias))
        batch, dim, width = st.shape
        assert x.shape == (batch, dim) and weight.shape == (dim, width)
        assert bias is None or bias.shape == (dim,)
        u = np.empty((batch, dim), dtype=np.float64)
        self._lib.oracle_conv_step(_p(st), _p(x), _p(weight), _p(bias), int(bool(silu)), _p(u),
                                   batch, dim, width)
        return st, u

    def conv_state_update(self, conv_state, x, weight, conv_bias, conv_silu, state, dt, A, B, C,
                          D=None, z=None, dt_bias=None, dt_softplus=True, zoh=False):
        """The decode step of a layer: the convolution step, then the state update with the
        convolution output as the input x. Returns (conv_state, state, u, out)."""
        cst, u = self.conv_step(conv_state, x, weight, conv_bias, conv_silu)
        st, out = self.state_update(state, u, dt, A, B, C, D, z, dt_bias, dt_softplus, zoh=zoh)
        return cst, st, u, out


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(_build())
    return _default


def max_threads() -> int:
    return default().max_threads()


def scan_fwd(*a, **k):
    return default().scan_fwd(*a, **k)


def scan_fwd_rows(*a, **k):
    return default().scan_fwd_rows(*a, **k)


def state_update(*a, **k):
    return default().state_update(*a, **k)


def conv_step(*a, **k):
    return default().conv_step(*a, **k)


def scan_bwd(*a, **k):
    return default().scan_bwd(*a, **k)


def conv_state_update(*a, **k):
    return default().conv_state_update(*a, **k)


def ssd_fwd(*a, **k):
    return default().ssd_fwd(*a, **k)
