"""The seeded input recipe (CPU): what every parity test and the benchmark draw from."""
import math

import torch

from workloads import (DECODE_CONFIG, SsdConfig, make_decode_layer_params, make_scan_inputs,
                       make_ssd_inputs, scan_config)


def _small(name, **kw):
    return scan_config(name).replace(batch=2, dim=48, seqlen=96, **kw)


def test_scan_inputs_are_deterministic_per_seed_and_differ_across_seeds():
    cfg = _small("c2_mamba2p8b")
    x, y = make_scan_inputs(cfg), make_scan_inputs(cfg)
    for k in ("u", "delta", "z", "B", "C", "A", "D", "delta_bias"):
        assert torch.equal(x[k], y[k]), k
    other = make_scan_inputs(cfg, seed=cfg.seed + 1)
    assert not torch.equal(x["u"], other["u"])


def test_scan_input_recipe():
    cfg = _small("c2_mamba2p8b")
    x = make_scan_inputs(cfg)
    # shapes and dtypes
    assert x["u"].shape == (2, 48, 96) and x["u"].dtype == torch.bfloat16
    assert x["B"].shape == (2, 16, 96) and x["C"].shape == (2, 16, 96)
    # A[d, n] = -(n + 1), D = 1
    assert torch.equal(x["A"], -torch.arange(1, 17, dtype=torch.float32).repeat(48, 1))
    assert torch.equal(x["D"], torch.ones(48))
    # softplus(delta_bias) is the per-channel dt, log-uniform in [dt_min, dt_max]
    dt = torch.nn.functional.softplus(x["delta_bias"].double())
    assert float(dt.min()) >= cfg.dt_min * (1 - 1e-5) and float(dt.max()) <= cfg.dt_max * (1 + 1e-5)
    # delta ~ N(0, 0.5^2), u ~ N(0, 1) (loose moments on 9,216 draws)
    assert abs(float(x["delta"].float().std()) - 0.5) < 0.05
    assert abs(float(x["u"].float().std()) - 1.0) < 0.1


def test_long_sequence_workload_takes_the_slower_decay():
    # the 1 M-token workload draws dt in [1e-4, 1e-2]
    cfg = scan_config("c3_long_1m")
    assert (cfg.dt_min, cfg.dt_max) == (1e-4, 1e-2)
    x = make_scan_inputs(cfg.replace(batch=1, dim=64, seqlen=8))
    dt = torch.nn.functional.softplus(x["delta_bias"].double())
    assert float(dt.max()) <= 1e-2 * (1 + 1e-5) and float(dt.min()) >= 1e-4 * (1 - 1e-5)


def test_decode_layer_parameters():
    p = make_decode_layer_params(DECODE_CONFIG)
    assert p["A"].shape == (DECODE_CONFIG.dim, 16)
    assert torch.equal(p["A"][0], -torch.arange(1, 17, dtype=torch.float32))


def test_ssd_input_recipe():
    cfg = SsdConfig("t", 2, 130, 4, 64, 2, 128, 5)
    x = make_ssd_inputs(cfg)
    assert x["x"].shape == (2, 130, 4, 64) and x["dt"].shape == (2, 130, 4)
    assert x["B"].shape == (2, 130, 2, 128) and x["C"].shape == (2, 130, 2, 128)
    # A_h = -U(1, 16) per head
    assert bool(((x["A"] <= -1.0) & (x["A"] >= -16.0)).all())
    dt = torch.nn.functional.softplus(x["dt_bias"].double())
    assert float(dt.min()) >= 1e-3 * (1 - 1e-5) and float(dt.max()) <= 1e-1 * (1 + 1e-5)
    assert not math.isnan(float(x["x"].float().sum()))
