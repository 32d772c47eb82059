"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each pin takes an oracle object (a compiled copy of oracle/selscan_oracle.c) and returns
the largest error it saw; the caller compares it with the pin's bound. The expected values
are computed here by other routes: the convolution form of a time-invariant system, the
solved (non-recursive) form of the recurrence, limits of Delta, hand-worked closed forms and
linearity. Helper functions below use formulas different from the oracle's
(logaddexp for softplus, the tanh form of the logistic function for silu).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def softplus_ref(x):
    return np.logaddexp(0.0, x)


def silu_ref(z):
    return z * 0.5 * (1.0 + np.tanh(0.5 * z))


def relerr(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = max(float(np.sqrt(np.mean(ref * ref))), 1e-300)
    return float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), scale)))


def _rng(seed):
    return np.random.default_rng(seed)


def _random_problem(seed, batch=2, dim=3, dstate=5, seqlen=40, lti=False):
    r = _rng(seed)
    A = -r.uniform(0.3, 3.0, size=(dim, dstate))
    D = r.standard_normal(dim)
    bias = r.uniform(-3.0, 0.5, size=dim)
    u = r.standard_normal((batch, dim, seqlen))
    z = r.standard_normal((batch, dim, seqlen))
    h0 = r.standard_normal((batch, dim, dstate))
    if lti:
        delta = np.repeat(r.normal(0.0, 0.5, size=(batch, dim, 1)), seqlen, axis=2)
        B = np.repeat(r.standard_normal((batch, dstate, 1)), seqlen, axis=2)
        C = np.repeat(r.standard_normal((batch, dstate, 1)), seqlen, axis=2)
    else:
        delta = r.normal(0.0, 0.5, size=(batch, dim, seqlen))
        B = r.standard_normal((batch, dstate, seqlen))
        C = r.standard_normal((batch, dstate, seqlen))
    return dict(u=u, delta=delta, A=A, B=B, C=C, D=D, z=z, delta_bias=bias, h0=h0)


def _bbar_ref(dlt, An, zoh):
    """Factor of B*u per state: Delta (Euler) or (exp(Delta*A) - 1)/A (zero-order hold),
    written with numpy's expm1 independently of the oracle."""
    return np.expm1(dlt * An) / An if zoh else dlt * np.ones_like(An)


def pin_lti_convolution(orc, seed=11, with_state=True, zoh=False):
    """'Every Step the Same' (world.lapla.si): with the same Delta, A, B, C at every token the
    output is the input convolved with one fixed kernel K_k = sum_n C[n] Abar[n]^k Bbar[n],
    computed here in closed form with exp(k*Delta*A) and an O(L^2) sum."""
    p = _random_problem(seed, lti=True)
    batch, dim, L = p["u"].shape
    N = p["A"].shape[1]
    h0 = p["h0"] if with_state else None
    out, fin = orc.scan_fwd(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"],
                            p["delta_bias"], True, h0, zoh=zoh)
    ref = np.zeros_like(out)
    ref_fin = np.zeros_like(fin)
    k = np.arange(L)
    for b in range(batch):
        for d in range(dim):
            dlt = softplus_ref(p["delta"][b, d, 0] + p["delta_bias"][d])
            Bn, Cn, An = p["B"][b, :, 0], p["C"][b, :, 0], p["A"][d]
            decay = np.exp(np.outer(k, dlt * An))  # (L, N): Abar^k
            bb = _bbar_ref(dlt, An, zoh) * Bn  # Bbar
            K = decay @ (Cn * bb)  # kernel K_k
            u = p["u"][b, d]
            y = np.array([np.dot(K[: t + 1], u[t::-1]) for t in range(L)])
            if h0 is not None:
                y = y + np.exp(np.outer(k + 1, dlt * An)) @ (Cn * h0[b, d])
            y = (y + p["D"][d] * u) * silu_ref(p["z"][b, d])
            ref[b, d] = y
            hf = (decay[::-1] * bb[None, :] * u[:, None]).sum(axis=0)
            if h0 is not None:
                hf = hf + np.exp(L * dlt * An) * h0[b, d]
            ref_fin[b, d] = hf
    return max(relerr(out, ref), relerr(fin, ref_fin))


def pin_solved_form(orc, seed=12, softplus=True, with_state=True, zoh=False):
    """The recurrence h_t = exp(Delta_t*A) h_{t-1} + Delta_t*B_t*u_t has the solution
    h_t = exp(A*S_t) h_init + sum_{s<=t} exp(A*(S_t - S_s)) Delta_s B_s u_s with
    S_t = Delta_0 + ... + Delta_t. This evaluates that sum directly (no recursion) for
    time-varying Delta, B, C and reads y_t = C_t . h_t + D u_t, gated by silu(z_t)."""
    p = _random_problem(seed, batch=2, dim=3, dstate=5, seqlen=32)
    batch, dim, L = p["u"].shape
    h0 = p["h0"] if with_state else None
    out, fin = orc.scan_fwd(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"],
                            p["delta_bias"], softplus, h0, zoh=zoh)
    ref = np.zeros_like(out)
    ref_fin = np.zeros_like(fin)
    for b in range(batch):
        for d in range(dim):
            x = p["delta"][b, d] + p["delta_bias"][d]
            dlt = softplus_ref(x) if softplus else x
            S = np.cumsum(dlt)
            An = p["A"][d]
            fac = np.stack([_bbar_ref(dl, An, zoh) for dl in dlt])  # (L, N)
            src = fac * p["B"][b].T * p["u"][b, d][:, None]  # (L, N)
            for t in range(L):
                w = np.exp(An[None, :] * (S[t] - S[: t + 1])[:, None])  # (t+1, N)
                h = (w * src[: t + 1]).sum(axis=0)
                if h0 is not None:
                    h = h + np.exp(An * S[t]) * h0[b, d]
                y = np.dot(p["C"][b][:, t], h) + p["D"][d] * p["u"][b, d, t]
                ref[b, d, t] = y * silu_ref(p["z"][b, d, t])
                if t == L - 1:
                    ref_fin[b, d] = h
    return max(relerr(out, ref), relerr(fin, ref_fin))


def pin_delta_zero(orc, seed=13):
    """'Chosen by the Token': a small Delta keeps the state and ignores the input. At Delta = 0
    exactly (softplus off, delta = bias = 0) Abar = 1 and Bbar*x = 0, so the state must come
    out bit-identical and y_t = (C_t . h0 + D u_t) silu(z_t)."""
    p = _random_problem(seed)
    zeros = np.zeros_like(p["delta"])
    out, fin = orc.scan_fwd(p["u"], zeros, p["A"], p["B"], p["C"], p["D"], p["z"], None, False,
                            p["h0"])
    bit_err = float(np.max(np.abs(fin - p["h0"])))
    ref = (np.einsum("bnt,bdn->bdt", p["C"], p["h0"]) + p["D"][None, :, None] * p["u"]) * silu_ref(p["z"])
    return max(bit_err * 1e300, relerr(out, ref))  # any state change at all fails the pin


def pin_large_delta(orc, seed=14):
    """'Chosen by the Token': a large Delta resets the state and takes in the current token.
    With Delta = 50 and A <= -1 the old state is multiplied by at most e^-50, so
    h_t = 50 B_t u_t and y_t = C_t . h_t + D u_t up to ~1e-21 relative."""
    p = _random_problem(seed)
    A = -np.abs(p["A"]) - 1.0
    big = np.full_like(p["delta"], 50.0)
    out, fin = orc.scan_fwd(p["u"], big, A, p["B"], p["C"], p["D"], None, None, False, p["h0"])
    h = 50.0 * p["B"][:, None, :, :] * p["u"][:, :, None, :]  # (b, d, n, t)
    ref = np.einsum("bnt,bdnt->bdt", p["C"], h) + p["D"][None, :, None] * p["u"]
    return max(relerr(out, ref), relerr(fin, h[..., -1]))


def pin_linearity(orc, seed=15):
    """Without the gate and from a zero state, y is linear in u (Delta depends on delta only)."""
    p = _random_problem(seed)
    r = _rng(seed + 1)
    u1, u2 = p["u"], r.standard_normal(p["u"].shape)
    a, c = 0.75, -1.25
    args = lambda u: (u, p["delta"], p["A"], p["B"], p["C"], p["D"], None, p["delta_bias"], True, None)
    y1, f1 = orc.scan_fwd(*args(u1))
    y2, f2 = orc.scan_fwd(*args(u2))
    y3, f3 = orc.scan_fwd(*args(a * u1 + c * u2))
    return max(relerr(y3, a * y1 + c * y2), relerr(f3, a * f1 + c * f2))


def load_hand_worked():
    with open(os.path.join(GOLDEN, "hand_worked_n1.json")) as f:
        return json.load(f)


def _zval(zspec, L):
    if zspec is None:
        return None
    if zspec == "ln3":
        return np.full((1, 1, L), math.log(3.0))
    return np.asarray(zspec, dtype=np.float64).reshape(1, 1, L)


def pin_hand_worked_scan(orc):
    g = load_hand_worked()
    worst = 0.0
    for c in g["scan_cases"]:
        L = len(c["u"])
        u = np.asarray(c["u"], dtype=np.float64).reshape(1, 1, L)
        delta = np.asarray(c["delta"], dtype=np.float64).reshape(1, 1, L)
        B = np.full((1, 1, L), c["B"])
        C = np.full((1, 1, L), c["C"])
        h0 = None if c["h0"] is None else np.full((1, 1, 1), c["h0"])
        out, fin = orc.scan_fwd(u, delta, np.array([[c["A"]]]), B, C, np.array([c["D"]]),
                                _zval(c["z"], L), np.array([c["bias"]]), c["softplus"], h0)
        e = np.asarray(c["expected"])
        worst = max(worst, float(np.max(np.abs(out[0, 0] - e) / np.maximum(np.abs(e), 1e-300)))
                    if np.any(e != 0) else float(np.max(np.abs(out[0, 0]))) * 1e300)
        worst = max(worst, abs(fin[0, 0, 0] - c["final"]) / abs(c["final"]))
    return worst


def pin_hand_worked_update(orc):
    g = load_hand_worked()
    worst = 0.0
    for c in g["update_cases"]:
        st, out = orc.state_update(np.full((1, 1, 1), c["state"]), np.array([[c["x"]]]),
                                   np.array([[c["dt"]]]), np.array([[c["A"]]]),
                                   np.array([[c["B"]]]), np.array([[c["C"]]]),
                                   np.array([c["D"]]),
                                   None if c["z"] is None else np.array([[math.log(3.0)]]),
                                   np.array([c["bias"]]), c["softplus"])
        worst = max(worst, abs(st[0, 0, 0] - c["state_expected"]) / abs(c["state_expected"]),
                    abs(out[0, 0] - c["out_expected"]) / abs(c["out_expected"]))
    return worst


def pin_update_is_one_scan_step(orc, seed=16, zoh=False):
    """The generation step is the scan's update applied once ('Taken Apart': one token read,
    the state moves once): state_update == a length-1 scan from that state, and L updates in a
    row == the length-L scan. The scan side is pinned by the pins above."""
    p = _random_problem(seed, batch=3, dim=4, dstate=5, seqlen=12)
    batch, dim, L = p["u"].shape
    st = p["h0"].copy()
    ys = np.zeros((batch, dim, L))
    for t in range(L):
        st, ys[:, :, t] = orc.state_update(st, p["u"][:, :, t], p["delta"][:, :, t], p["A"],
                                           p["B"][:, :, t], p["C"][:, :, t], p["D"],
                                           p["z"][:, :, t], p["delta_bias"], True, zoh=zoh)
    out, fin = orc.scan_fwd(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"],
                            p["delta_bias"], True, p["h0"], zoh=zoh)
    return max(relerr(ys, out), relerr(st, fin))


def gate_reference(x, u, h0):
    """The recurrent gate of 'Chosen by the Token' (the paper's Theorem 1):
    h_t = (1 - g_t) h_{t-1} + g_t u_t with g_t = sigmoid(x_t), evaluated with the logistic
    function. x, u: (..., L); h0: (...). Returns the sequence h (..., L)."""
    g = 1.0 / (1.0 + np.exp(-x))
    h = np.array(h0, dtype=np.float64)
    out = np.empty_like(u)
    for t in range(u.shape[-1]):
        h = (1.0 - g[..., t]) * h + g[..., t] * u[..., t]
        out[..., t] = h
    return out


def pin_theorem1_gate(orc, seed=17):
    """'Chosen by the Token': with a state of a single number the selective update is exactly
    a recurrent network's gate h <- (1 - g) h + g x. That holds for the zero-order hold with
    A = -1, B = C = 1, D = 0 and Delta = softplus(x): then Abar = exp(-Delta) = 1 - sigmoid(x)
    and Bbar = 1 - exp(-Delta) = sigmoid(x). Checked for the scan and for L state updates."""
    r = _rng(seed)
    batch, dim, L = 2, 3, 60
    delta = r.normal(0.0, 1.5, size=(batch, dim, L))
    bias = r.uniform(-3.0, 2.0, size=dim)
    u = r.standard_normal((batch, dim, L))
    h0 = r.standard_normal((batch, dim, 1))
    A = -np.ones((dim, 1))
    ones = np.ones((batch, 1, L))
    out, fin = orc.scan_fwd(u, delta, A, ones, ones, np.zeros(dim), None, bias, True, h0, zoh=True)
    ref = gate_reference(delta + bias[None, :, None], u, h0[..., 0])
    st = h0.copy()
    ys = np.empty_like(u)
    for t in range(L):
        st, ys[:, :, t] = orc.state_update(st, u[:, :, t], delta[:, :, t], A, ones[:, :, t],
                                           ones[:, :, t], None, None, bias, True, zoh=True)
    return max(relerr(out, ref), relerr(fin[..., 0], ref[..., -1]), relerr(ys, ref))


def pin_conv_step_is_causal_convolution(orc, seed=18):
    """'A State of Fixed Size': the block's short convolution holds the last 4 inputs. Run
    step by step from a zero window, its outputs must be the causal depthwise convolution of
    the input sequence with the 4 taps, evaluated here with numpy.convolve (then silu)."""
    r = _rng(seed)
    batch, dim, width, L = 2, 5, 4, 23
    x = r.standard_normal((batch, dim, L))
    w = r.standard_normal((dim, width))
    bias = r.standard_normal(dim)
    st = np.zeros((batch, dim, width))
    got = np.empty((batch, dim, L))
    for t in range(L):
        st, got[:, :, t] = orc.conv_step(st, x[:, :, t], w, bias, True)
    ref = np.empty_like(got)
    for b in range(batch):
        for d in range(dim):
            # window oldest-first: u_t = sum_k w[k] x[t - (width-1) + k]
            full = np.convolve(x[b, d], w[d][::-1])[:L] + bias[d]
            ref[b, d] = silu_ref(full)
    last = x[:, :, L - width:]
    return max(relerr(got, ref), float(np.max(np.abs(st - last))) * 1e300)


def pin_backward_finite_differences(orc, seed=19, softplus=True, full=True):
    """The backward pass (the training half of 'A Scan on the Chip') against central finite
    differences of the forward: for loss = sum(dout*out) + sum(dfinal*final_state), each
    gradient entry sampled below must equal (loss(x+eps) - loss(x-eps)) / (2 eps) of the
    oracle's own forward. Every input is probed: u, delta, A, B, C, D, z, delta_bias, h0."""
    r = _rng(seed)
    p = _random_problem(seed, batch=2, dim=3, dstate=4, seqlen=14)
    if not full:
        p["z"], p["D"], p["delta_bias"], p["h0"] = None, None, None, None
    if not softplus:  # keep Delta positive without softplus
        p["delta"] = np.abs(p["delta"]) * 0.3 + 0.05
        if p["delta_bias"] is not None:
            p["delta_bias"] = np.abs(p["delta_bias"]) * 0.1
    dout = r.standard_normal(p["u"].shape)
    dfin = r.standard_normal((2, 3, 4))
    keys = ["u", "delta", "A", "B", "C", "D", "z", "delta_bias", "h0"]

    def loss(q):
        out, fin = orc.scan_fwd(q["u"], q["delta"], q["A"], q["B"], q["C"], q["D"], q["z"],
                                q["delta_bias"], softplus, q["h0"])
        return float(np.sum(out * dout) + np.sum(fin * dfin))

    g = orc.scan_bwd(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"], p["delta_bias"],
                     softplus, p["h0"], dout, dfin)
    names = {"u": "du", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD", "z": "dz",
             "delta_bias": "ddelta_bias", "h0": "dinitial_state"}
    worst, eps = 0.0, 1e-5
    for k in keys:
        if p[k] is None:
            continue
        flat = p[k].reshape(-1)
        for i in r.choice(flat.size, size=min(6, flat.size), replace=False):
            q = {kk: (None if v is None else v.copy()) for kk, v in p.items()}
            q[k].reshape(-1)[i] += eps
            lp = loss(q)
            q[k].reshape(-1)[i] -= 2 * eps
            lm = loss(q)
            fd = (lp - lm) / (2 * eps)
            an = g[names[k]].reshape(-1)[i]
            worst = max(worst, abs(an - fd) / max(abs(fd), 1e-2))
    return worst


def _ssd_problem(seed, batch=2, seqlen=23, nheads=4, headdim=3, ngroups=2, dstate=5,
                 full=True):
    r = _rng(seed)
    q = {
        "x": r.standard_normal((batch, seqlen, nheads, headdim)),
        "dt": r.standard_normal((batch, seqlen, nheads)) * 0.7,
        "A": -r.uniform(0.5, 4.0, nheads),
        "B": r.standard_normal((batch, seqlen, ngroups, dstate)),
        "C": r.standard_normal((batch, seqlen, ngroups, dstate)),
        "D": r.standard_normal(nheads) if full else None,
        "z": r.standard_normal((batch, seqlen, nheads, headdim)) if full else None,
        "dt_bias": r.standard_normal(nheads) * 0.5 if full else None,
        "h0": r.standard_normal((batch, nheads, headdim, dstate)) if full else None,
    }
    return q


def ssd_matrix_form(q, softplus=True):
    """'Mamba-2' (world.lapla.si): the layer as one lower-triangular matrix per head, entry
    (i, j) = C_i . B_j times all the decay in between, applied to the Delta-scaled input; plus
    the initial state carried to every step and read by C_i. The decay from step j to step i
    is exp(A * (S_i - S_j)) with S the running sum of Delta: closed form, no repeated product."""
    x, dt, A, B, C = q["x"], q["dt"], q["A"], q["B"], q["C"]
    batch, L, H, P = x.shape
    G = B.shape[2]
    bias = q["dt_bias"] if q["dt_bias"] is not None else np.zeros(H)
    pre = dt + bias[None, None, :]
    dl = softplus_ref(pre) if softplus else pre
    y = np.zeros_like(x)
    fin = np.zeros((batch, H, P, B.shape[3]))
    for b in range(batch):
        for h in range(H):
            g = h // (H // G)
            S = np.cumsum(dl[b, :, h])
            CB = C[b, :, g, :] @ B[b, :, g, :].T                      # (L, L): C_i . B_j
            dec = np.exp(A[h] * (S[:, None] - S[None, :]))
            M = np.tril(CB * dec) * dl[b, None, :, h]                  # times Delta_j
            yy = M @ x[b, :, h, :]                                     # (L, P)
            w = np.exp(A[h] * (S[-1] - S)) * dl[b, :, h]               # step j to the end
            fin[b, h] = (x[b, :, h, :] * w[:, None]).T @ B[b, :, g, :]
            if q["h0"] is not None:
                carry = np.exp(A[h] * S)                               # from the start to i
                yy += carry[:, None] * (C[b, :, g, :] @ q["h0"][b, h].T)
                fin[b, h] += np.exp(A[h] * S[-1]) * q["h0"][b, h]
            if q["D"] is not None:
                yy += q["D"][h] * x[b, :, h, :]
            if q["z"] is not None:
                yy *= silu_ref(q["z"][b, :, h, :])
            y[b, :, h, :] = yy
    return y, fin


def pin_ssd_matrix_form(orc, seed=41, full=True, softplus=True):
    q = _ssd_problem(seed, full=full)
    y, fin = orc.ssd_fwd(q["x"], q["dt"], q["A"], q["B"], q["C"], q["D"], q["z"], q["dt_bias"],
                         softplus, q["h0"])
    ry, rf = ssd_matrix_form(q, softplus)
    return max(relerr(y, ry), relerr(fin, rf))


def pin_ssd_is_s6_with_scalar_A(orc, seed=42):
    """With A[d, n] = A_h for every state and B, C shared by all heads (one group), each of the
    headdim channels of a head is one S6 channel: the SSD recurrence must equal the selective
    scan (itself pinned above) run on dim = nheads * headdim channels."""
    q = _ssd_problem(seed, batch=2, seqlen=19, nheads=3, headdim=2, ngroups=1, dstate=16)
    y, fin = orc.ssd_fwd(q["x"], q["dt"], q["A"], q["B"], q["C"], q["D"], q["z"], q["dt_bias"],
                         True, q["h0"])
    batch, L, H, P = q["x"].shape
    to_bdl = lambda a: np.ascontiguousarray(a.reshape(batch, L, H * P).transpose(0, 2, 1))
    u = to_bdl(q["x"])
    z = to_bdl(q["z"])
    delta = np.ascontiguousarray(np.repeat(q["dt"], P, axis=2).transpose(0, 2, 1))
    A = np.repeat(q["A"], P)[:, None] * np.ones((1, 16))
    Bs = np.ascontiguousarray(q["B"][:, :, 0, :].transpose(0, 2, 1))
    Cs = np.ascontiguousarray(q["C"][:, :, 0, :].transpose(0, 2, 1))
    out, sfin = orc.scan_fwd(u, delta, A, Bs, Cs, np.repeat(q["D"], P), z,
                             np.repeat(q["dt_bias"], P), True, q["h0"].reshape(batch, H * P, 16))
    return max(relerr(y, out.transpose(0, 2, 1).reshape(batch, L, H, P)),
               relerr(fin, sfin.reshape(batch, H, P, 16)))


def pin_ssd_no_decay_is_running_sum(orc, seed=43):
    """A = 0: nothing decays, so the state is the running sum of Delta_j x_j B_j^T and
    y_i = C_i . H_i (no gate, no skip) -- evaluated with numpy's cumulative sum."""
    q = _ssd_problem(seed, full=False)
    q["A"] = np.zeros_like(q["A"])
    y, fin = orc.ssd_fwd(q["x"], q["dt"], q["A"], q["B"], q["C"], None, None, None, True, None)
    batch, L, H, P = q["x"].shape
    G = q["B"].shape[2]
    dl = softplus_ref(q["dt"])
    worst = 0.0
    for b in range(batch):
        for h in range(H):
            g = h // (H // G)
            outer = (dl[b, :, h, None, None] * q["x"][b, :, h, :, None] *
                     q["B"][b, :, g, None, :])                      # (L, P, N)
            Hs = np.cumsum(outer, axis=0)
            ry = np.einsum("tpn,tn->tp", Hs, q["C"][b, :, g, :])
            worst = max(worst, relerr(y[b, :, h, :], ry), relerr(fin[b, h], Hs[-1]))
    return worst


# (pin function, bound) pairs used by the pin tests and the mutation tests.
ALL_PINS = [
    (pin_lti_convolution, 1e-11),
    (lambda o: pin_lti_convolution(o, seed=21, with_state=False), 1e-11),
    (pin_solved_form, 1e-11),
    (lambda o: pin_solved_form(o, seed=22, softplus=False, with_state=False), 1e-11),
    (pin_delta_zero, 1e-13),
    (pin_large_delta, 1e-12),
    (pin_linearity, 1e-11),
    (pin_hand_worked_scan, 1e-14),
    (pin_hand_worked_update, 1e-14),
    (pin_update_is_one_scan_step, 1e-12),
    (pin_theorem1_gate, 1e-12),
    (lambda o: pin_lti_convolution(o, seed=23, zoh=True), 1e-11),
    (lambda o: pin_solved_form(o, seed=24, zoh=True), 1e-11),
    (lambda o: pin_update_is_one_scan_step(o, seed=25, zoh=True), 1e-12),
    (pin_conv_step_is_causal_convolution, 1e-13),
    (pin_backward_finite_differences, 1e-5),
    (lambda o: pin_backward_finite_differences(o, seed=26, softplus=False, full=False), 1e-5),
    (pin_ssd_matrix_form, 1e-11),
    (lambda o: pin_ssd_matrix_form(o, seed=44, full=False, softplus=False), 1e-11),
    (pin_ssd_is_s6_with_scalar_A, 1e-12),
    (pin_ssd_no_decay_is_running_sum, 1e-12),
]
