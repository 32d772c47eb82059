"""Workload shapes for the selective scan (S6) and its decode step.

Sizes follow the Mamba layer shapes described in "Mamba and State Space Models"
(world.lapla.si, sections "A State of Fixed Size" and "Every Step the Same"):
N = 16 state numbers per channel, A initialised to -1 ... -16, Mamba-2.8B with
64 layers of 5,120 channels. The 130M-like layer uses d_model 768 with an
expansion factor of 2 (1,536 channels).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass


@dataclass(frozen=True)
class ScanConfig:
    name: str
    batch: int
    dim: int
    dstate: int
    seqlen: int
    in_dtype: str  # "f32" or "bf16": u, delta, z, B, C
    out_dtype: str  # "f32" or "bf16": y
    dt_min: float  # delta_bias = inverse-softplus(dt), dt log-uniform in [dt_min, dt_max]
    dt_max: float
    seed: int
    has_z: bool = True
    has_D: bool = True
    has_bias: bool = True
    delta_softplus: bool = True
    delta_std: float = 0.5  # delta ~ N(0, delta_std^2)

    @property
    def elements(self) -> int:
        return self.batch * self.dim * self.seqlen

    def replace(self, **kw) -> "ScanConfig":
        return dataclasses.replace(self, **kw)


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    layers: int
    batches: tuple
    dim: int
    dstate: int
    steps: int
    ring: int  # distinct per-token input sets per layer, used as step % ring
    dt_min: float
    dt_max: float
    seed: int
    delta_std: float = 0.5

    def replace(self, **kw) -> "DecodeConfig":
        return dataclasses.replace(self, **kw)


SCAN_CONFIGS = {
    # Tiny oracle check, fp32 everywhere.
    "c0_tiny_f32": ScanConfig("c0_tiny_f32", 1, 64, 16, 256, "f32", "f32", 1e-3, 1e-1, 1000),
    # Mamba-130M-like layer (d_model 768, expand 2).
    "c1_mamba130m": ScanConfig("c1_mamba130m", 8, 1536, 16, 2048, "bf16", "bf16", 1e-3, 1e-1, 1001),
    # Mamba-2.8B-like layer.
    "c2_mamba2p8b": ScanConfig("c2_mamba2p8b", 4, 5120, 16, 2048, "bf16", "bf16", 1e-3, 1e-1, 1002),
    # Long sequence: 1,048,576 tokens, slower decay so the state carries over long spans.
    "c3_long_1m": ScanConfig("c3_long_1m", 1, 1536, 16, 1 << 20, "bf16", "bf16", 1e-4, 1e-2, 1003),
}

# Decode sweep, Mamba-2.8B shape: 64 layers x state update, 1,024 generated tokens.
DECODE_CONFIG = DecodeConfig("c4_decode_mamba2p8b", 64, (1, 16, 64), 5120, 16, 1024, 8, 1e-3, 1e-1, 1004)


@dataclass(frozen=True)
class SsdConfig:
    """Mamba-2 SSD layer: x (batch, seqlen, nheads, headdim), B/C (batch, seqlen, ngroups, dstate)."""
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    ngroups: int
    dstate: int
    seed: int
    dt_min: float = 1e-3
    dt_max: float = 1e-1
    has_z: bool = True
    has_D: bool = True

    @property
    def elements(self) -> int:  # batch * seqlen * nheads * headdim = B*L*d_inner
        return self.batch * self.seqlen * self.nheads * self.headdim

    def replace(self, **kw) -> "SsdConfig":
        return dataclasses.replace(self, **kw)


SSD_CONFIGS = {
    # Small case the oracle finishes in well under a second.
    "ssd0_tiny": SsdConfig("ssd0_tiny", 1, 256, 4, 64, 1, 128, 2000),
    # Mamba-2 2.7B-like layer: d_model 2560, expand 2 -> d_inner 5120 = 80 heads x 64, a state
    # of 128 numbers per channel ("Mamba-2": the released models keep 128 where Mamba keeps 16),
    # one group of B/C; the same batch, sequence length and d_inner as the Mamba-2.8B scan layer.
    "ssd1_mamba2_2p7b": SsdConfig("ssd1_mamba2_2p7b", 4, 2048, 80, 64, 1, 128, 2001),
}


def ssd_config(name: str) -> SsdConfig:
    for k, v in SSD_CONFIGS.items():
        if k == name or k.split("_")[0] == name:
            return v
    raise KeyError(f"unknown SSD config {name!r}; known: {sorted(SSD_CONFIGS)}")


def scan_config(name: str) -> ScanConfig:
    for k, v in SCAN_CONFIGS.items():
        if k == name or k.split("_")[0] == name:
            return v
    raise KeyError(f"unknown scan config {name!r}; known: {sorted(SCAN_CONFIGS)}")
