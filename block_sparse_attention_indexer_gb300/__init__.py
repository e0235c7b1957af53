"""MiniMax Sparse Attention (MSA) decode over an NVFP4 paged KV cache, for one GB300 (sm_103a).

The compute lives in libmsa.so (hand-written CUDA kernels behind the C ABI in include/msa.h);
this package is its thin Python binding.  Importing it requires the built library.
"""
from .binding import (  # noqa: F401
    EXPORTED,
    MSA_DEVERR_BAD_PAGE,
    MSA_DEVERR_BAD_SEQLEN,
    MSA_DEVERR_TIMEOUT,
    MSA_OP_DECODE,
    MSA_OP_INDEXER_SCORES,
    MSA_OP_SELECT_BLOCKS,
    MSA_OP_SPARSE_ATTN,
    MSA_SCORE_LSE,
    MSA_SCORE_MAX,
    Batch,
    Config,
    MsaError,
    PagedCache,
    alloc_workspace,
    default_softmax_scale,
    msa_abi_version,
    msa_clear_device_error,
    msa_dcp_local_candidates,
    msa_dcp_merge,
    msa_decode,
    msa_fp8_quantize,
    msa_indexer_scores,
    msa_noalloc_read_device_error,
    msa_nvfp4_insert,
    msa_read_device_error,
    msa_select_blocks,
    msa_sparse_attn_decode,
    msa_sparse_attn_decode_noalloc,
    msa_test_attention_stall,
    msa_test_indexer_stall,
    msa_workspace_bytes,
)
