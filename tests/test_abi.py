"""The C ABI without a GPU: libmsa.so builds for sm_103a, loads, exports every entry point
include/msa.h declares, and its host-only logic (status strings, workspace sizes, argument
validation that rejects before any CUDA call) behaves as documented."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "msa.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\*?\s*(msa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return ctypes.CDLL(os.path.join(ROOT, "block_sparse_attention_indexer_gb300", "libmsa.so"))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ["msa_indexer_scores", "msa_select_blocks", "msa_sparse_attn_decode", "msa_decode",
              "msa_workspace_bytes", "msa_nvfp4_insert", "msa_fp8_quantize"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in _declared():
        assert hasattr(lib, n), n


def test_binding_covers_the_header(lib):
    import block_sparse_attention_indexer_gb300 as msa
    assert sorted(msa.EXPORTED) == _declared()


def test_version_and_status_strings(lib):
    lib.msa_abi_version.restype = ctypes.c_int32
    ver = int(re.search(r"#define MSA_ABI_VERSION (\d+)", open(HEADER).read()).group(1))
    assert lib.msa_abi_version() == ver
    lib.msa_status_string.restype = ctypes.c_char_p
    assert [lib.msa_status_string(i).decode() for i in range(5)] == [
        "MSA_OK", "MSA_ERR_INVALID_ARG", "MSA_ERR_UNSUPPORTED", "MSA_ERR_WORKSPACE", "MSA_ERR_CUDA"]


def test_workspace_sizes(lib):
    import block_sparse_attention_indexer_gb300 as msa
    b = msa.binding
    cfg = b._Config(4, 8, 128, 128, 128, 16, 0, 1, 0.0)
    f = b._lib.msa_workspace_bytes
    # 64 sequences x 1 token x 4 groups = 256 rows; the attention's partial-state area is two
    # slots of 8 heads x 130 floats per team, 3 teams per CTA, up to 160 CTAs, whatever the batch
    bt = b._Batch(1, 1, 64, 1024, 1)
    scores = 256 * 1024 * 4
    sel = 256 * 16 * 4
    partial = 2 * 160 * 3 * 8 * 130 * 4
    assert f(b.MSA_OP_INDEXER_SCORES, ctypes.byref(cfg), ctypes.byref(bt)) == 256
    assert f(b.MSA_OP_SELECT_BLOCKS, ctypes.byref(cfg), ctypes.byref(bt)) == 0
    assert f(b.MSA_OP_SPARSE_ATTN, ctypes.byref(cfg), ctypes.byref(bt)) == 256 + partial
    # the decode step keeps the scores, the selection and the selected entries' pages
    assert f(b.MSA_OP_DECODE, ctypes.byref(cfg), ctypes.byref(bt)) == 256 + scores + 2 * sel + partial
    bt = b._Batch(1, 1, 1, 544, 63)   # 63 query tokens: still the team kernel
    assert f(b.MSA_OP_SPARSE_ATTN, ctypes.byref(cfg), ctypes.byref(bt)) == 256 + partial

    # from 64 query tokens on (chunked prefill) the attention runs block-major: CSR offsets,
    # block counts, insertion cursors and entries, (m, l) and o / l in f16 for every
    # (token, head, selection slot), and the queries in f16, each area rounded up to 256 bytes
    def al(x):
        return (x + 255) // 256 * 256

    def block_major(B, T, G, Hg, MB):
        slots = B * T * G * Hg * 16
        return (al(B * G * (MB + 1) * 4) + 2 * al(B * G * MB * 4) + al(B * G * T * 16 * 4) + al(slots * 8)
                + al(slots * 128 * 2) + al(B * T * G * Hg * 128 * 2))

    bt = b._Batch(1, 1, 1, 544, 4096)
    bm = block_major(1, 4096, 4, 8, 544)
    assert bm == 8960 + 2 * 8704 + 1048576 + 16777216 + 536870912 + 33554432
    assert f(b.MSA_OP_SPARSE_ATTN, ctypes.byref(cfg), ctypes.byref(bt)) == 256 + bm
    assert f(b.MSA_OP_DECODE, ctypes.byref(cfg), ctypes.byref(bt)) == (
        256 + al(4096 * 4 * 544 * 4) + 2 * al(4096 * 4 * 16 * 4) + bm)
    bt = b._Batch(1, 1, 2, 300, 64)
    assert f(b.MSA_OP_SPARSE_ATTN, ctypes.byref(cfg), ctypes.byref(bt)) == 256 + block_major(2, 64, 4, 8, 300)
    # unsupported configurations report 0
    bad = b._Config(4, 8, 64, 128, 128, 16, 0, 1, 0.0)
    assert f(b.MSA_OP_DECODE, ctypes.byref(bad), ctypes.byref(bt)) == 0
    bad = b._Config(4, 8, 128, 128, 128, 4, 3, 2, 0.0)      # init + local > top_k
    assert f(b.MSA_OP_DECODE, ctypes.byref(bad), ctypes.byref(bt)) == 0
    # the configuration variants are accepted: top_k 8 with init 2 and local 2, log-sum-exp
    var = b._Config(4, 8, 128, 128, 128, 8, 2, 2, 0.0, b.MSA_SCORE_LSE)
    assert f(b.MSA_OP_DECODE, ctypes.byref(var), ctypes.byref(bt)) > 0


def test_validation_rejects_before_any_cuda_call(lib):
    import block_sparse_attention_indexer_gb300 as msa
    b = msa.binding
    L = b._lib
    good = b._Config(4, 8, 128, 128, 128, 16, 0, 1, 0.0)
    cache = b._Cache(16, 16, 16, 16, 16, 16, 10)
    batch = b._Batch(16, 16, 2, 8, 1)
    ref = ctypes.byref
    # unsupported sparse configs (top_k 17, top_k 0, init + local > top_k, score type 2, 9 groups)
    for cfg in [b._Config(4, 8, 128, 128, 128, 17, 0, 1, 0.0), b._Config(4, 8, 128, 128, 128, 0, 0, 0, 0.0),
                b._Config(4, 8, 128, 128, 128, 8, 4, 5, 0.0), b._Config(4, 8, 128, 128, 128, 16, 0, 1, 0.0, 2),
                b._Config(9, 8, 128, 128, 128, 16, 0, 1, 0.0)]:
        assert L.msa_decode(ref(cfg), ref(cache), ref(batch), 16, 16, 16, None, None, 16, 1 << 30, None) == 2
    # null / misaligned pointers, bad sizes
    assert L.msa_decode(None, ref(cache), ref(batch), 16, 16, 16, None, None, 16, 1 << 30, None) == 1
    assert L.msa_decode(ref(good), ref(cache), ref(batch), 17, 16, 16, None, None, 16, 1 << 30, None) == 1
    assert L.msa_decode(ref(good), ref(b._Cache(16, 16, 16, 16, 16, 17, 10)), ref(batch), 16, 16, 16, None, None,
                        16, 1 << 30, None) == 1
    assert L.msa_indexer_scores(ref(good), ref(cache), ref(b._Batch(16, 16, 2, 8, 0)), 16, 16, 16, 256, None) == 1
    # workspace too small
    assert L.msa_decode(ref(good), ref(cache), ref(batch), 16, 16, 16, None, None, 16, 8, None) == 3
    # batch larger than the kernels support / grid limit
    assert L.msa_select_blocks(ref(good), ref(b._Batch(16, 16, 5000, 8, 1)), 16, 16, None) == 2
    assert L.msa_select_blocks(ref(good), ref(b._Batch(16, 16, 100, 8, 1000)), 16, 16, None) == 2
    # empty batch is a no-op
    assert L.msa_decode(ref(good), ref(cache), ref(b._Batch(0, 0, 0, 8, 1)), 16, 16, 16, None, None, 16, 0,
                        None) == 0
    # quantiser argument checks
    assert L.msa_nvfp4_insert(16, 4, 1, 100, 16, 16, 16, 3, 128, None) == 1      # dim not a multiple of 16
    assert L.msa_nvfp4_insert(None, 0, 1, 128, None, None, None, 3, 128, None) == 0
    assert L.msa_fp8_quantize(None, -1, None, None) == 1
