"""Seeded synthetic inputs for paged KV-cache attention.

This package only draws random numbers and lays them out the way a paged
KV-cache engine would (page pool, page table, slot map, ragged query offsets).
It holds none of the attention arithmetic, so both the CPU oracle and the CUDA
path can consume the same inputs without sharing any computation.
"""
from .workloads import (  # noqa: F401
    CONFIGS,
    share_prefix,
    PagedInputs,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    make_inputs,
    make_config,
    cu_seqlens_from_lengths,
)
