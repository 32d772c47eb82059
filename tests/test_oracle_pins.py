"""The fp64 oracle against values fixed by the pages and by the mathematics (CPU only)."""
import json
import math
import os

import numpy as np
import pytest

import oracle
from tests import oracle_pins as P


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("i", range(len(P.ALL_PINS)))
def test_pin(orc, i):
    fn, bound = P.ALL_PINS[i]
    err = fn(orc)
    assert err <= bound, f"pin {i} error {err:.3e} > {bound:.1e}"


def test_hand_worked_fixture_matches_its_expressions():
    g = P.load_hand_worked()
    env = {"log": math.log, "exp": math.exp, "__builtins__": {}}
    for c in g["scan_cases"]:
        for t, v in enumerate(c["expected"]):
            assert v == pytest.approx(eval(c["expected_expr"], dict(env), {"t": t}), rel=1e-15, abs=0)
        assert c["final"] == pytest.approx(eval(c["final_expr"], dict(env)), rel=1e-15)


def test_rows_variant_matches_full(orc):
    p = P._random_problem(31, batch=2, dim=5, dstate=16, seqlen=50)
    out, fin = orc.scan_fwd(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"],
                            p["delta_bias"], True, p["h0"])
    rows = np.array([7, 0, 9, 3])
    batch, dim, L = p["u"].shape
    flat = lambda a: a.reshape(batch * dim, -1)[rows]
    o2, f2 = orc.scan_fwd_rows(rows, flat(p["u"]), flat(p["delta"]), p["A"], p["B"], p["C"],
                               p["D"], flat(p["z"]), p["delta_bias"], True, flat(p["h0"]))
    assert np.array_equal(o2, out.reshape(batch * dim, L)[rows])
    assert np.array_equal(f2, fin.reshape(batch * dim, -1)[rows])


def test_split_scan_equals_whole(orc):
    """Resuming from the final state: scan(L1) then scan(L2) == scan(L1 + L2)."""
    p = P._random_problem(32, batch=2, dim=3, dstate=16, seqlen=60)
    a = lambda s: (p["u"][..., s], p["delta"][..., s], p["A"], p["B"][..., s], p["C"][..., s],
                   p["D"], p["z"][..., s], p["delta_bias"], True)
    out, fin = orc.scan_fwd(*a(slice(None)), p["h0"])
    o1, f1 = orc.scan_fwd(*a(slice(0, 23)), p["h0"])
    o2, f2 = orc.scan_fwd(*a(slice(23, None)), f1)
    assert P.relerr(np.concatenate([o1, o2], axis=2), out) < 1e-13
    assert P.relerr(f2, fin) < 1e-13


def test_workload_sizes_match_pages():
    """Decode workload shape against the sizes printed in 'A State of Fixed Size' and the
    initial values of A in 'Every Step the Same'."""
    from workloads import DECODE_CONFIG, make_decode_layer_params
    with open(os.path.join(P.GOLDEN, "mamba_state_sizes.json")) as f:
        g = json.load(f)
    m = g["mamba_2p8b"]
    assert (DECODE_CONFIG.layers, DECODE_CONFIG.dim, DECODE_CONFIG.dstate) == (
        m["layers"], m["channels"], m["state_per_channel"])
    numbers = m["layers"] * m["channels"] * (m["state_per_channel"] + m["conv_inputs_per_channel"])
    assert numbers == m["numbers_per_text"]
    assert round(numbers * 2 / 1e6, 1) == m["megabytes_at_16_bit"]
    py = g["pythia_2p8b"]
    per_tok = 2 * py["layers"] * py["kv_width"] * py["bytes_per_number"]
    assert per_tok == py["bytes_per_token"]
    assert round(per_tok * py["tokens_trained"] / 1e6) == py["cache_megabytes_at_2048"]
    state_bytes = numbers * 2
    assert math.ceil(state_bytes / per_tok) == py["passes_mamba_state_at_token"]
    assert round(per_tok * py["tokens_trained"] / state_bytes) == py["times_larger_at_2048"]
    A = make_decode_layer_params(DECODE_CONFIG.replace(dim=4))["A"]
    assert A[0, 0].item() == g["A_initial_values"]["first"]
    assert A[0, -1].item() == g["A_initial_values"]["last"]
