"""Seeded synthetic workloads for MSA decode over an NVFP4 KV cache.

This package only draws random numbers and lays out shapes; it contains none of the
method's arithmetic (no quantisation, scoring, selection or attention).  Both the
CPU oracle and the CUDA path read their inputs from here.
"""
from .synthetic import (  # noqa: F401
    BLOCK,
    HEAD_DIM,
    INDEX_DIM,
    NUM_KV_GROUPS,
    TOP_K,
    WORKLOADS,
    Workload,
    custom,
    seq_lens,
    gen_block_fp32,
    gen_index_queries,
    gen_queries,
    layout,
)
