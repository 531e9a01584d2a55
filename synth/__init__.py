"""Seeded synthetic inputs shared by the oracle tests, the CUDA parity tests and the bench.

This package only draws and encodes random inputs (normal draws, bf16 / fp8 encoding,
page tables); it holds none of the attention arithmetic.
"""
from .inputs import (  # noqa: F401
    PrefillCase,
    DecodeCase,
    make_prefill,
    make_decode,
    prefill_config,
    decode_config,
    PREFILL_CONFIGS,
    DECODE_CONFIGS,
)
