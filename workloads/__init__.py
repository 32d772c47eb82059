"""Seeded synthetic inputs for the selective-SSM scan and the single-token state update.

This package only draws random numbers and lays them out. It holds none of the
method's arithmetic, so both the CUDA path and the fp64 CPU oracle can take the
same tensors from it without sharing any computation.
"""
from .configs import (
    ScanConfig,
    DecodeConfig,
    SsdConfig,
    SSD_CONFIGS,
    ssd_config,
    SCAN_CONFIGS,
    DECODE_CONFIG,
    scan_config,
)
from .generate import (
    make_scan_inputs,
    make_decode_layer_params,
    make_decode_tokens,
    make_decode_state,
    make_ssd_inputs,
)

__all__ = [
    "ScanConfig",
    "DecodeConfig",
    "SCAN_CONFIGS",
    "DECODE_CONFIG",
    "scan_config",
    "make_scan_inputs",
    "make_decode_layer_params",
    "make_decode_tokens",
    "make_decode_state",
    "make_ssd_inputs",
    "SsdConfig",
    "SSD_CONFIGS",
    "ssd_config",
]
