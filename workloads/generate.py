"""Seeded generators: every tensor is drawn from a torch.Generator seeded per workload.

Recipe (one generator per workload, drawn in this order):
  dt       log-uniform in [dt_min, dt_max], one per channel; delta_bias = log(expm1(dt)),
           the inverse of softplus, so that softplus(delta_bias) = dt
  u        N(0, 1)        (batch, dim, seqlen)
  delta    N(0, 0.5^2)    (batch, dim, seqlen)
  z        N(0, 1)        (batch, dim, seqlen)
  B, C     N(0, 1)        (batch, dstate, seqlen)
  A[d, n] = -(n + 1), D[d] = 1  (fp32, not random)
Values are drawn in fp32 and rounded to nearest-even when the workload is bf16.
Large tensors are drawn in slabs of at most SLAB elements, so the sequence of draws
depends on the shape only, never on the device memory available.
"""
from __future__ import annotations

import math

import torch

from .configs import ScanConfig, DecodeConfig, SsdConfig

SLAB = 1 << 26

_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def torch_dtype(name: str) -> torch.dtype:
    return _DT[name]


def _normal(shape, std, dtype, gen, device):
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, SLAB):
        e = min(n, s + SLAB)
        tmp = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            tmp.mul_(std)
        flat[s:e].copy_(tmp)
    return out


def _bias_from_dt(dim, dt_min, dt_max, gen, device):
    r = torch.rand(dim, generator=gen, device=device, dtype=torch.float64)
    dt = torch.exp(r * (math.log(dt_max) - math.log(dt_min)) + math.log(dt_min))
    return torch.log(torch.expm1(dt)).to(torch.float32)


def make_scan_inputs(cfg: ScanConfig, device="cpu", seed: int | None = None) -> dict:
    """Inputs for one ssm_scan_fwd call of workload `cfg`, on `device`."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(cfg.seed if seed is None else seed)
    dt = _DT[cfg.in_dtype]
    bias = _bias_from_dt(cfg.dim, cfg.dt_min, cfg.dt_max, gen, device)
    shp = (cfg.batch, cfg.dim, cfg.seqlen)
    u = _normal(shp, 1.0, dt, gen, device)
    delta = _normal(shp, cfg.delta_std, dt, gen, device)
    z = _normal(shp, 1.0, dt, gen, device)
    B = _normal((cfg.batch, cfg.dstate, cfg.seqlen), 1.0, dt, gen, device)
    C = _normal((cfg.batch, cfg.dstate, cfg.seqlen), 1.0, dt, gen, device)
    A = -torch.arange(1, cfg.dstate + 1, dtype=torch.float32, device=device).repeat(cfg.dim, 1).contiguous()
    D = torch.ones(cfg.dim, dtype=torch.float32, device=device)
    return {
        "u": u,
        "delta": delta,
        "A": A,
        "B": B,
        "C": C,
        "D": D if cfg.has_D else None,
        "z": z if cfg.has_z else None,
        "delta_bias": bias if cfg.has_bias else None,
        "delta_softplus": cfg.delta_softplus,
    }


def make_decode_layer_params(cfg: DecodeConfig, device="cpu") -> dict:
    """Per-layer A (dim, dstate), D (dim), dt_bias (dim). Every layer gets the same values."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(cfg.seed)
    bias = _bias_from_dt(cfg.dim, cfg.dt_min, cfg.dt_max, gen, device)
    A = -torch.arange(1, cfg.dstate + 1, dtype=torch.float32, device=device).repeat(cfg.dim, 1).contiguous()
    D = torch.ones(cfg.dim, dtype=torch.float32, device=device)
    return {"A": A, "D": D, "dt_bias": bias}


def make_decode_state(cfg: DecodeConfig, batch: int, layer: int, device="cpu") -> torch.Tensor:
    """Initial fp32 state (batch, dim, dstate) ~ N(0, 1) of one layer."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(cfg.seed * 7919 + 104729 * batch + layer)
    return _normal((batch, cfg.dim, cfg.dstate), 1.0, torch.float32, gen, device)


def make_decode_tokens(cfg: DecodeConfig, batch: int, layer: int, slot: int, device="cpu") -> dict:
    """Per-token bf16 inputs of one layer for ring slot `slot`: x, dt, z (batch, dim); B, C (batch, dstate)."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(cfg.seed * 1000003 + 7777 * batch + 97 * layer + slot)
    bf = torch.bfloat16
    x = _normal((batch, cfg.dim), 1.0, bf, gen, device)
    dt = _normal((batch, cfg.dim), cfg.delta_std, bf, gen, device)
    z = _normal((batch, cfg.dim), 1.0, bf, gen, device)
    B = _normal((batch, cfg.dstate), 1.0, bf, gen, device)
    C = _normal((batch, cfg.dstate), 1.0, bf, gen, device)
    return {"x": x, "dt": dt, "z": z, "B": B, "C": C}


def make_ssd_inputs(cfg: SsdConfig, device="cpu") -> dict:
    """Inputs of one Mamba-2 SSD layer call, in this draw order: dt_bias from dt log-uniform in
    [dt_min, dt_max] per head (inverse softplus), A = -U(1, 16) per head (fp32), x, dt (raw,
    N(0, 0.5^2)), z, B, C (N(0, 1), bf16); D = 1 per head."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(cfg.seed)
    bf = torch.bfloat16
    bias = _bias_from_dt(cfg.nheads, cfg.dt_min, cfg.dt_max, gen, device)
    A = -(1.0 + 15.0 * torch.rand(cfg.nheads, generator=gen, device=device, dtype=torch.float32))
    act = (cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim)
    x = _normal(act, 1.0, bf, gen, device)
    dt = _normal((cfg.batch, cfg.seqlen, cfg.nheads), 0.5, bf, gen, device)
    z = _normal(act, 1.0, bf, gen, device)
    bc = (cfg.batch, cfg.seqlen, cfg.ngroups, cfg.dstate)
    B = _normal(bc, 1.0, bf, gen, device)
    C = _normal(bc, 1.0, bf, gen, device)
    D = torch.ones(cfg.nheads, dtype=torch.float32, device=device)
    return {"x": x, "dt": dt, "A": A, "B": B, "C": C, "D": D if cfg.has_D else None,
            "z": z if cfg.has_z else None, "dt_bias": bias, "dt_softplus": True}
