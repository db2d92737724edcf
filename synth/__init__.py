"""Seeded synthetic inputs for paged FP8 KV decode attention.

Shared by the product tests, the benchmark and the oracle checks; it generates
inputs only (random bf16 tensors, context lengths, page permutations, block
tables, slot mappings, top-k lists and the per-tensor amax-based scales) and
holds none of the attention or quantisation arithmetic.
"""
from . import gen  # noqa: F401
from .workloads import (  # noqa: F401
    MlaWorkload,
    PagedWorkload,
    workload,
    WORKLOADS,
    TINY_GQA,
    MHA_B32,
    GQA_PREFIX,
    MLA_TOPK,
    LONG_SPLITKV,
)
