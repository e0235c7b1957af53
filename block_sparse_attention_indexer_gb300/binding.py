"""Thin ctypes binding of libmsa.so (include/msa.h).

Argument marshalling only: every function takes torch tensors, checks dtype / device /
contiguity, passes data pointers and the current CUDA stream to the C entry point of the
same name, and raises MsaError on a non-OK status.  All compute happens in the library's
CUDA kernels; there is no Python or CPU fallback.  If libmsa.so has not been built the
import fails loudly (build with `python block_sparse_attention_indexer_gb300/build.py`).
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmsa.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python block_sparse_attention_indexer_gb300/build.py` "
        "(the MSA path has no CPU fallback)")
_lib = ctypes.CDLL(LIB_PATH)

# ---------------------------------------------------------------------------- C types
MSA_OK, MSA_ERR_INVALID_ARG, MSA_ERR_UNSUPPORTED, MSA_ERR_WORKSPACE, MSA_ERR_CUDA = range(5)
MSA_OP_INDEXER_SCORES, MSA_OP_SELECT_BLOCKS, MSA_OP_SPARSE_ATTN, MSA_OP_DECODE = range(4)
MSA_DEVERR_BAD_PAGE, MSA_DEVERR_BAD_SEQLEN, MSA_DEVERR_TIMEOUT = 0x1, 0x2, 0x4
MSA_SCORE_MAX, MSA_SCORE_LSE = 0, 1


class _Config(ctypes.Structure):
    _fields_ = [("num_kv_groups", ctypes.c_int32), ("heads_per_group", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("index_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("init_blocks", ctypes.c_int32), ("local_blocks", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float), ("score_type", ctypes.c_int32)]


class _Cache(ctypes.Structure):
    _fields_ = [("k_data", ctypes.c_void_p), ("k_scale", ctypes.c_void_p), ("v_data", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p), ("idx_data", ctypes.c_void_p), ("idx_scale", ctypes.c_void_p),
                ("num_pages", ctypes.c_int64)]


class _Batch(ctypes.Structure):
    _fields_ = [("block_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p), ("batch", ctypes.c_int32),
                ("max_blocks", ctypes.c_int32), ("q_len", ctypes.c_int32)]


_P = ctypes.c_void_p
_CP, _CC, _CB = ctypes.POINTER(_Config), ctypes.POINTER(_Cache), ctypes.POINTER(_Batch)
_SIGS = {
    "msa_abi_version": (ctypes.c_int32, []),
    "msa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "msa_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int, _CP, _CB]),
    "msa_nvfp4_insert": (ctypes.c_int, [_P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _P, _P, _P,
                                        ctypes.c_int64, ctypes.c_int32, _P]),
    "msa_fp8_quantize": (ctypes.c_int, [_P, ctypes.c_int64, _P, _P]),
    "msa_indexer_scores": (ctypes.c_int, [_CP, _CC, _CB, _P, _P, _P, ctypes.c_size_t, _P]),
    "msa_select_blocks": (ctypes.c_int, [_CP, _CB, _P, _P, _P]),
    "msa_dcp_local_candidates": (ctypes.c_int, [_CP, _CC, _CB, _P, ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P,
                                                ctypes.c_size_t, _P]),
    "msa_dcp_merge": (ctypes.c_int, [_CP, _CB, ctypes.c_int32, _P, _P, _P, _P]),
    "msa_sparse_attn_decode": (ctypes.c_int, [_CP, _CC, _CB, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "msa_decode": (ctypes.c_int, [_CP, _CC, _CB, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "msa_sparse_attn_decode_noalloc": (ctypes.c_int, [_CP, _CC, _CB, _P, _P, _P, _P, _P]),
    "msa_noalloc_read_device_error": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), _P]),
    "msa_test_indexer_stall": (ctypes.c_int, [_CP, _CC, _CB, _P, _P, _P, ctypes.c_size_t, ctypes.c_uint32, _P]),
    "msa_test_attention_stall": (ctypes.c_int, [_CP, _CC, _CB, _P, _P, _P, _P, _P, ctypes.c_size_t, ctypes.c_uint32,
                                                _P]),
    "msa_read_device_error": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_uint32), _P]),
    "msa_clear_device_error": (ctypes.c_int, [_P, _P]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

EXPORTED = tuple(_SIGS)


class MsaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {_lib.msa_status_string(status).decode()}")


def _check(fn: str, status: int):
    if status != MSA_OK:
        raise MsaError(fn, status)


def _ptr(t: Optional[torch.Tensor], dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


# ---------------------------------------------------------------------------- Python-side views
@dataclasses.dataclass
class Config:
    num_kv_groups: int = 4
    heads_per_group: int = 8
    head_dim: int = 128
    index_dim: int = 128
    block_size: int = 128
    top_k: int = 16
    init_blocks: int = 0
    local_blocks: int = 1
    softmax_scale: float = 0.0      # 0 = 1/sqrt(head_dim)
    score_type: int = 0             # MSA_SCORE_MAX (0) or MSA_SCORE_LSE (1)

    def c(self):
        return ctypes.byref(_Config(self.num_kv_groups, self.heads_per_group, self.head_dim, self.index_dim,
                                    self.block_size, self.top_k, self.init_blocks, self.local_blocks,
                                    self.softmax_scale, self.score_type))

    @property
    def num_heads(self):
        return self.num_kv_groups * self.heads_per_group


class PagedCache:
    """The six NVFP4 page pools (device tensors, uint8), allocated by torch."""

    def __init__(self, num_pages: int, groups: int = 4, dim: int = 128, index_dim: int = 128, block: int = 128,
                 device="cuda"):
        u8 = dict(dtype=torch.uint8, device=device)
        self.num_pages, self.groups, self.block = num_pages, groups, block
        self.k_data = torch.zeros(num_pages, groups, block, dim // 2, **u8)
        self.k_scale = torch.zeros(num_pages, groups, block, dim // 16, **u8)
        self.v_data = torch.zeros(num_pages, groups, block, dim // 2, **u8)
        self.v_scale = torch.zeros(num_pages, groups, block, dim // 16, **u8)
        self.idx_data = torch.zeros(num_pages, block, index_dim // 2, **u8)
        self.idx_scale = torch.zeros(num_pages, block, index_dim // 16, **u8)

    def tensors(self):
        return (self.k_data, self.k_scale, self.v_data, self.v_scale, self.idx_data, self.idx_scale)

    def c(self):
        ps = [_ptr(t, torch.uint8, "cache") for t in self.tensors()]
        return ctypes.byref(_Cache(*ps, self.num_pages))

    @property
    def nbytes(self):
        return sum(t.numel() for t in self.tensors())


@dataclasses.dataclass
class Batch:
    block_table: torch.Tensor     # int32 [B, max_blocks] on the device
    seq_lens: torch.Tensor        # int32 [B] on the device
    q_len: int = 1

    def c(self):
        B, MB = self.block_table.shape
        return ctypes.byref(_Batch(_ptr(self.block_table, torch.int32, "block_table"),
                                   _ptr(self.seq_lens, torch.int32, "seq_lens"), B, MB, self.q_len))

    @property
    def batch(self):
        return self.block_table.shape[0]

    @property
    def max_blocks(self):
        return self.block_table.shape[1]


# ---------------------------------------------------------------------------- entry points
def msa_abi_version() -> int:
    return _lib.msa_abi_version()


def msa_workspace_bytes(op: int, cfg: Config, batch: Batch) -> int:
    return int(_lib.msa_workspace_bytes(op, cfg.c(), batch.c()))


def alloc_workspace(op: int, cfg: Config, batch: Batch, device="cuda") -> torch.Tensor:
    """Zero-filled workspace of the size `op` needs (the zero fill clears the error word)."""
    n = max(msa_workspace_bytes(op, cfg, batch), 256)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def msa_nvfp4_insert(x: torch.Tensor, slots: torch.Tensor, data: torch.Tensor, scale: torch.Tensor,
                     block_size: int = 128, stream=None):
    """x float32 [n_tokens, rows_per_token, dim]; slots int64 [n_tokens]; data/scale are a
    cache pool pair ([P, rows, block, dim/2] and [P, rows, block, dim/16])."""
    n, rows, dim = x.shape
    num_pages = data.shape[0]
    _check("msa_nvfp4_insert", _lib.msa_nvfp4_insert(
        _ptr(x, torch.float32, "x"), n, rows, dim, _ptr(slots, torch.int64, "slots"),
        _ptr(data, torch.uint8, "data"), _ptr(scale, torch.uint8, "scale"), num_pages, block_size,
        _stream(stream)))


def msa_fp8_quantize(x: torch.Tensor, out: torch.Tensor, stream=None):
    _check("msa_fp8_quantize", _lib.msa_fp8_quantize(_ptr(x, torch.float32, "x"), x.numel(),
                                                     _ptr(out, torch.uint8, "out"), _stream(stream)))


def msa_indexer_scores(cfg: Config, cache: PagedCache, batch: Batch, index_q: torch.Tensor,
                       block_scores: torch.Tensor, workspace: torch.Tensor, stream=None):
    _check("msa_indexer_scores", _lib.msa_indexer_scores(
        cfg.c(), cache.c(), batch.c(), _ptr(index_q, torch.uint8, "index_q"),
        _ptr(block_scores, torch.float32, "block_scores"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def msa_select_blocks(cfg: Config, batch: Batch, block_scores: torch.Tensor, selection: torch.Tensor, stream=None):
    _check("msa_select_blocks", _lib.msa_select_blocks(
        cfg.c(), batch.c(), _ptr(block_scores, torch.float32, "block_scores"),
        _ptr(selection, torch.int32, "selection"), _stream(stream)))


def msa_dcp_local_candidates(cfg: Config, cache: PagedCache, batch: Batch, index_q: torch.Tensor, block_lo: int,
                             block_hi: int, block_scores: torch.Tensor, cand_scores: torch.Tensor,
                             cand_blocks: torch.Tensor, workspace: torch.Tensor, stream=None):
    _check("msa_dcp_local_candidates", _lib.msa_dcp_local_candidates(
        cfg.c(), cache.c(), batch.c(), _ptr(index_q, torch.uint8, "index_q"), block_lo, block_hi,
        _ptr(block_scores, torch.float32, "block_scores"), _ptr(cand_scores, torch.float32, "cand_scores"),
        _ptr(cand_blocks, torch.int32, "cand_blocks"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def msa_dcp_merge(cfg: Config, batch: Batch, cand_scores: torch.Tensor, cand_blocks: torch.Tensor,
                  selection: torch.Tensor, stream=None):
    """cand_scores / cand_blocks: [num_shards, B, T, G, 15] (the shards' outputs stacked)."""
    _check("msa_dcp_merge", _lib.msa_dcp_merge(
        cfg.c(), batch.c(), int(cand_scores.shape[0]), _ptr(cand_scores, torch.float32, "cand_scores"),
        _ptr(cand_blocks, torch.int32, "cand_blocks"), _ptr(selection, torch.int32, "selection"), _stream(stream)))


def msa_sparse_attn_decode(cfg: Config, cache: PagedCache, batch: Batch, q: torch.Tensor, selection: torch.Tensor,
                           out: torch.Tensor, lse: Optional[torch.Tensor], workspace: torch.Tensor, stream=None):
    _check("msa_sparse_attn_decode", _lib.msa_sparse_attn_decode(
        cfg.c(), cache.c(), batch.c(), _ptr(q, torch.uint8, "q"), _ptr(selection, torch.int32, "selection"),
        _ptr(out, torch.bfloat16, "out"), _ptr(lse, torch.float32, "lse"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def msa_sparse_attn_decode_noalloc(cfg: Config, cache: PagedCache, batch: Batch, q: torch.Tensor,
                                   selection: torch.Tensor, out: torch.Tensor, lse: Optional[torch.Tensor],
                                   stream=None):
    """msa_sparse_attn_decode without a workspace, for callers that cannot allocate device
    memory: the scratch is the library's own 8 MiB device array (see include/msa.h).  Calls
    that overlap on the GPU share that array and race."""
    _check("msa_sparse_attn_decode_noalloc", _lib.msa_sparse_attn_decode_noalloc(
        cfg.c(), cache.c(), batch.c(), _ptr(q, torch.uint8, "q"), _ptr(selection, torch.int32, "selection"),
        _ptr(out, torch.bfloat16, "out"), _ptr(lse, torch.float32, "lse"), _stream(stream)))


def msa_noalloc_read_device_error(stream=None) -> int:
    """The device error word of the no-allocation entry point's array (the last call's)."""
    flags = ctypes.c_uint32(0)
    _check("msa_noalloc_read_device_error", _lib.msa_noalloc_read_device_error(ctypes.byref(flags), _stream(stream)))
    return int(flags.value)


def msa_test_indexer_stall(cfg: Config, cache: PagedCache, batch: Batch, index_q: torch.Tensor,
                           block_scores: torch.Tensor, workspace: torch.Tensor, spin_limit: int, stream=None):
    """Test hook: the streaming indexer with its page copies withheld and its waits capped at
    spin_limit polls (include/msa.h)."""
    _check("msa_test_indexer_stall", _lib.msa_test_indexer_stall(
        cfg.c(), cache.c(), batch.c(), _ptr(index_q, torch.uint8, "index_q"),
        _ptr(block_scores, torch.float32, "block_scores"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), spin_limit, _stream(stream)))


def msa_test_attention_stall(cfg: Config, cache: PagedCache, batch: Batch, q: torch.Tensor, selection: torch.Tensor,
                             out: torch.Tensor, lse: Optional[torch.Tensor], workspace: torch.Tensor, spin_limit: int,
                             stream=None):
    """Test hook: the team attention with its page copies withheld and every wait capped at
    spin_limit polls (the waits run out; MSA_DEVERR_TIMEOUT is set)."""
    _check("msa_test_attention_stall", _lib.msa_test_attention_stall(
        cfg.c(), cache.c(), batch.c(), _ptr(q, torch.uint8, "q"), _ptr(selection, torch.int32, "selection"),
        _ptr(out, torch.bfloat16, "out"), _ptr(lse, torch.float32, "lse"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), spin_limit, _stream(stream)))


def msa_decode(cfg: Config, cache: PagedCache, batch: Batch, q: torch.Tensor, index_q: torch.Tensor,
               out: torch.Tensor, lse: Optional[torch.Tensor], selection_out: Optional[torch.Tensor],
               workspace: torch.Tensor, stream=None):
    _check("msa_decode", _lib.msa_decode(
        cfg.c(), cache.c(), batch.c(), _ptr(q, torch.uint8, "q"), _ptr(index_q, torch.uint8, "index_q"),
        _ptr(out, torch.bfloat16, "out"), _ptr(lse, torch.float32, "lse"),
        _ptr(selection_out, torch.int32, "selection_out"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def msa_read_device_error(workspace: torch.Tensor, stream=None) -> int:
    flags = ctypes.c_uint32(0)
    _check("msa_read_device_error", _lib.msa_read_device_error(_ptr(workspace, None, "workspace"),
                                                               ctypes.byref(flags), _stream(stream)))
    return int(flags.value)


def msa_clear_device_error(workspace: torch.Tensor, stream=None):
    _check("msa_clear_device_error", _lib.msa_clear_device_error(_ptr(workspace, None, "workspace"),
                                                                 _stream(stream)))


def default_softmax_scale(head_dim: int = 128) -> float:
    return 1.0 / math.sqrt(head_dim)
