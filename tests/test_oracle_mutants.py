"""Each plausible mistake, planted in a copy of the oracle's C source, must fail a pin.

The mistakes are planted in temporary copies compiled on the CPU; the real oracle is
untouched. This shows the pins in oracle_pins.py constrain every term of the definition.
"""
import os
import subprocess

import numpy as np
import pytest

from oracle import Oracle
from oracle.build import SRC
from tests import oracle_pins as P

_ROW_UPDATE = """            h[n] = abar * h[n] + bbar_x;
        }
        double y = 0.0;
        for (int64_t n = 0; n < dstate; ++n) y += Cb[n * seqlen + t] * h[n];"""

MUTANTS = {
    "drop_D_skip": ("y += D_d * u[t];", ""),
    "exp_sign": ("double abar = exp(dlt * A_d[n]);", "double abar = exp(-dlt * A_d[n]);"),
    "zoh_instead_of_euler": ("if (!zoh || a == 0.0) return dlt;", "if (a == 0.0) return dlt;"),
    "euler_instead_of_zoh": ("return expm1(dlt * a) / a;", "return dlt;"),
    "zoh_without_divide": ("return expm1(dlt * a) / a;", "return expm1(dlt * a);"),
    "missing_delta_in_B": ("double bbar_x = bbar_factor(dlt, A_d[n], zoh) * Bb[n * seqlen + t] * u[t];",
                           "double bbar_x = Bb[n * seqlen + t] * u[t];"),
    "B_transposed": ("double bbar_x = bbar_factor(dlt, A_d[n], zoh) * Bb[n * seqlen + t] * u[t];",
                     "double bbar_x = bbar_factor(dlt, A_d[n], zoh) * Bb[t * dstate + n] * u[t];"),
    "C_is_B": ("y += Cb[n * seqlen + t] * h[n];", "y += Bb[n * seqlen + t] * h[n];"),
    "read_before_update": (_ROW_UPDATE, """            h[n] = abar * h[n] + bbar_x;
        }
        double y = 0.0;
        for (int64_t n = 0; n < dstate; ++n) y += Cb[n * seqlen + t] * (h[n] - bbar_factor(dlt, A_d[n], zoh) * Bb[n * seqlen + t] * u[t]) / exp(dlt * A_d[n]);"""),
    "bias_after_softplus": ("double x = delta[t] + bias;\n        double dlt = softplus_on ? softplus(x) : x;",
                            "double x = delta[t];\n        double dlt = (softplus_on ? softplus(x) : x) + bias;"),
    "softplus_dropped_log1p": ("return fmax(x, 0.0) + log1p(exp(-fabs(x)));", "return fmax(x, 0.0);"),
    "silu_is_sigmoid": ("return z / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(-z));"),
    "initial_state_ignored": ("h[n] = initial_state ? initial_state[r * dstate + n] : 0.0;", "h[n] = 0.0;"),
    "A_wrong_stride": ("A + d * dstate, B + b * dstate * seqlen,\n                 C + b * dstate * seqlen, D ? D[d] : 0.0, z ? z + off : NULL,",
                       "A + d, B + b * dstate * seqlen,\n                 C + b * dstate * seqlen, D ? D[d] : 0.0, z ? z + off : NULL,"),
    "update_zoh_ignored": ("double f = bbar_factor(dlt, A[d * dstate + n], zoh);",
                           "double f = dlt;"),
    "readout_skips_last_state": ("for (int64_t n = 0; n < dstate; ++n) y += Cb[n * seqlen + t] * h[n];",
                                 "for (int64_t n = 0; n + 1 < dstate; ++n) y += Cb[n * seqlen + t] * h[n];"),
    "update_drops_batch_of_B": ("h[n] = abar * h[n] + f * B[b * dstate + n] * x[r];",
                                "h[n] = abar * h[n] + f * B[n] * x[r];"),
    "update_bias_ignored": ("double xx = dt[r] + (dt_bias ? dt_bias[d] : 0.0);", "double xx = dt[r];"),
    "update_gate_dropped": ("if (z) y *= silu(z[r]);", ""),
    "bwd_dDelta_drops_input_term": ("dDelta += dk * u[off + t];", ""),
    "bwd_g_decays_before_readout": ("g[n] += ds * Cb[n * L + t];", "g[n] = g[n] * exp(dl[t] * A[d * N + n]) + ds * Cb[n * L + t];"),
    "bwd_no_softplus_derivative": ("const double dx = delta_softplus ? dDelta / (1.0 + exp(-x)) : dDelta;",
                                   "const double dx = dDelta;"),
    "bwd_dB_without_delta": ("dB[b * N * L + n * L + t] += g[n] * dl[t] * u[off + t];",
                             "dB[b * N * L + n * L + t] += g[n] * u[off + t];"),
    "bwd_dC_uses_previous_state": ("dC[b * N * L + n * L + t] += ds * hs[(t + 1) * N + n];",
                                   "dC[b * N * L + n * L + t] += ds * hs[t * N + n];"),
    "bwd_dA_without_delta": ("dA[d * N + n] += dabar * abar * dl[t];", "dA[d * N + n] += dabar * abar;"),
    "bwd_silu_derivative_wrong": ("(sig * (1.0 + zz * (1.0 - sig)))", "(sig)"),
    "conv_window_not_shifted": ("for (int64_t k = 0; k + 1 < width; ++k) s[k] = s[k + 1];", ""),
    "conv_taps_reversed": ("acc += w[d * width + k] * s[k];", "acc += w[d * width + (width - 1 - k)] * s[k];"),
    "conv_bias_dropped": ("double acc = bias ? bias[d] : 0.0;", "double acc = 0.0;"),
    "conv_silu_dropped": ("u[r] = silu_on ? silu(acc) : acc;", "u[r] = acc;"),
    "ssd_decay_sign": ("const double decay = exp(dlt * A[h]);", "const double decay = exp(-dlt * A[h]);"),
    "ssd_missing_delta": ("H[p * N + n] = decay * H[p * N + n] + dlt * xt[p] * Bt[n];",
                          "H[p * N + n] = decay * H[p * N + n] + xt[p] * Bt[n];"),
    "ssd_group_index": ("g = h / heads_per_group;", "g = h % ngroups;"),
    "ssd_readout_before_update": ("""                    H[p * N + n] = decay * H[p * N + n] + dlt * xt[p] * Bt[n];
                    acc += Ct[n] * H[p * N + n];""", """                    acc += Ct[n] * H[p * N + n];
                    H[p * N + n] = decay * H[p * N + n] + dlt * xt[p] * Bt[n];"""),
    "ssd_C_is_B": ("acc += Ct[n] * H[p * N + n];", "acc += Bt[n] * H[p * N + n];"),
    "ssd_D_dropped": ("acc += (D ? D[h] : 0.0) * xt[p];", ""),
    "ssd_gate_dropped": ("if (z) acc *= silu(z[((b * seqlen + t) * nheads + h) * P + p]);", ""),
    "ssd_bias_ignored": ("const double xr = dt[(b * seqlen + t) * nheads + h] + (dt_bias ? dt_bias[h] : 0.0);",
                         "const double xr = dt[(b * seqlen + t) * nheads + h];"),
    "ssd_initial_state_ignored": ("H[i] = initial_state ? initial_state[bh * P * N + i] : 0.0;",
                                  "H[i] = 0.0;"),
    "ssd_final_state_transposed": ("for (int64_t i = 0; i < P * N; ++i) final_state[bh * P * N + i] = H[i];",
                                   "for (int64_t i = 0; i < P * N; ++i) final_state[bh * P * N + i] = H[(i % P) * N + i / P];"),
}


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared", "-o",
                           str(lib), str(src), "-lm"])
    orc = Oracle(str(lib))
    failed = []
    for i, (fn, bound) in enumerate(P.ALL_PINS):
        with np.errstate(all="ignore"):
            err = fn(orc)
        if not (err <= bound):  # NaN counts as a failure
            failed.append(i)
    assert failed, f"mutant {name} passed every pin"
