// C ABI of libmsa.so: host-side validation, workspace layout and kernel dispatch.
// The operations and their definitions are documented in include/msa.h.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "../../include/msa.h"
#include "api_internal.h"
#include "msa_kernels.h"

using namespace msa;

namespace {

constexpr size_t kWsAlign = 256;
constexpr size_t kErrBytes = 256;  // error word + padding
constexpr int kMaxDevices = 64;

size_t align_up(size_t x) { return (x + kWsAlign - 1) / kWsAlign * kWsAlign; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

msa_status_t check_config(const msa_config_t* c) {
  if (c == nullptr) return MSA_ERR_INVALID_ARG;
  if (c->num_kv_groups < 1 || c->num_kv_groups > 8 || c->heads_per_group < 1 || c->heads_per_group > 8)
    return MSA_ERR_UNSUPPORTED;
  if (c->head_dim != 128 || c->index_dim != 128 || c->block_size != 128) return MSA_ERR_UNSUPPORTED;
  if (c->top_k < 1 || c->top_k > kSelTopK || c->init_blocks < 0 || c->local_blocks < 0 ||
      c->init_blocks + c->local_blocks > c->top_k)
    return MSA_ERR_UNSUPPORTED;
  if (c->score_type != MSA_SCORE_MAX && c->score_type != MSA_SCORE_LSE) return MSA_ERR_UNSUPPORTED;
  if (!(c->softmax_scale >= 0.0f) || !std::isfinite(c->softmax_scale)) return MSA_ERR_INVALID_ARG;
  return MSA_OK;
}

msa_status_t check_batch(const msa_batch_t* b) {
  if (b == nullptr) return MSA_ERR_INVALID_ARG;
  if (b->batch < 0 || b->max_blocks < 1 || b->q_len < 1) return MSA_ERR_INVALID_ARG;
  if (b->batch > 0 && (b->block_table == nullptr || b->seq_lens == nullptr)) return MSA_ERR_INVALID_ARG;
  if (b->batch > kMaxBatchSmem) return MSA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(b->batch) * b->q_len > 65535) return MSA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(b->max_blocks) * 128 > INT32_MAX) return MSA_ERR_UNSUPPORTED;
  return MSA_OK;
}

msa_status_t check_cache(const msa_cache_t* c, bool idx, bool kv) {
  if (c == nullptr || c->num_pages < 1 || c->num_pages > INT32_MAX) return MSA_ERR_INVALID_ARG;
  if (idx && (c->idx_data == nullptr || c->idx_scale == nullptr || !aligned16(c->idx_data) ||
              !aligned16(c->idx_scale)))
    return MSA_ERR_INVALID_ARG;
  if (kv && (c->k_data == nullptr || c->k_scale == nullptr || c->v_data == nullptr || c->v_scale == nullptr ||
             !aligned16(c->k_data) || !aligned16(c->k_scale) || !aligned16(c->v_data) || !aligned16(c->v_scale)))
    return MSA_ERR_INVALID_ARG;
  return MSA_OK;
}

int num_sms_of_current_device() {
  static int cache[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
  if (dev < kMaxDevices && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return -1;
  if (dev < kMaxDevices) cache[dev] = n;
  return n;
}

int64_t rows_tg(const msa_batch_t* b, const msa_config_t* c) {
  return static_cast<int64_t>(b->batch) * b->q_len * c->num_kv_groups;
}

size_t scores_bytes(const msa_config_t* c, const msa_batch_t* b) {
  return align_up(static_cast<size_t>(rows_tg(b, c)) * b->max_blocks * sizeof(float));
}
size_t sel_bytes(const msa_config_t* c, const msa_batch_t* b) {
  return align_up(static_cast<size_t>(rows_tg(b, c)) * kSelTopK * sizeof(int32_t));
}
size_t partial_bytes() { return align_up(attn_partial_bytes()); }

// long query chunks (chunked prefill) attend block-major: their scratch is the K-to-Q plan and
// one partial state per (token, head, selection slot) instead of the team kernel's slots
bool block_major(const msa_config_t* c, const msa_batch_t* b) {
  return bm_supported(b->batch, b->q_len, c->num_kv_groups, c->heads_per_group, b->max_blocks);
}
size_t attn_scratch_bytes(const msa_config_t* c, const msa_batch_t* b) {
  return block_major(c, b)
             ? align_up(bm_workspace_bytes(b->batch, b->q_len, c->num_kv_groups, c->heads_per_group, b->max_blocks))
             : partial_bytes();
}



float scale_log2(const msa_config_t* c) {
  const float sm = c->softmax_scale > 0.0f ? c->softmax_scale : 1.0f / std::sqrt(static_cast<float>(c->head_dim));
  return sm * 1.4426950408889634f;
}

msa_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA; }

// stage 1: the streaming decode indexer (<= 8 query rows per sequence), the tcgen05 form with
// the keys as M (speculative decode, 9..63 rows) or the tcgen05 GEMM (long query chunks)
cudaError_t run_indexer(const IndexerArgs& a, int sms, cudaStream_t s) {
  const int rows = a.q_len * a.groups;
  if (rows >= kPrefillMinRows) return launch_prefill_indexer(a, s);
  if (rows > 8) return launch_spec_indexer(a, sms, s);
  return launch_indexer(a, sms, s);
}

IndexerArgs indexer_args(const msa_config_t* cfg, const msa_cache_t* cache, const msa_batch_t* batch,
                         const uint8_t* index_q, float* scores, uint32_t* err) {
  IndexerArgs a{};
  a.idx_data = cache->idx_data;
  a.idx_scale = cache->idx_scale;
  a.num_pages = cache->num_pages;
  a.block_table = batch->block_table;
  a.seq_lens = batch->seq_lens;
  a.batch = batch->batch;
  a.max_blocks = batch->max_blocks;
  a.q_len = batch->q_len;
  a.groups = cfg->num_kv_groups;
  a.index_q = index_q;
  a.block_scores = scores;
  a.err = err;
  a.lse = cfg->score_type == MSA_SCORE_LSE ? 1 : 0;
  a.spin_limit = kDefaultSpinLimit;
  a.block_lo = 0;
  a.block_hi = INT32_MAX;
  return a;
}

SelectArgs select_args(const msa_config_t* cfg, const msa_batch_t* batch, const float* scores, int32_t* sel) {
  SelectArgs a{};
  a.block_scores = scores;
  a.seq_lens = batch->seq_lens;
  a.batch = batch->batch;
  a.max_blocks = batch->max_blocks;
  a.q_len = batch->q_len;
  a.groups = cfg->num_kv_groups;
  a.selection = sel;
  a.top_k = cfg->top_k;
  a.init_blocks = cfg->init_blocks;
  a.local_blocks = cfg->local_blocks;
  return a;
}

AttnArgs attn_args(const msa_config_t* cfg, const msa_cache_t* cache, const msa_batch_t* batch, const uint8_t* q,
                   const int32_t* sel, uint16_t* out, float* lse, float* partial, uint32_t* err) {
  AttnArgs a{};
  a.k_data = cache->k_data;
  a.k_scale = cache->k_scale;
  a.v_data = cache->v_data;
  a.v_scale = cache->v_scale;
  a.num_pages = cache->num_pages;
  a.block_table = batch->block_table;
  a.seq_lens = batch->seq_lens;
  a.batch = batch->batch;
  a.max_blocks = batch->max_blocks;
  a.q_len = batch->q_len;
  a.groups = cfg->num_kv_groups;
  a.heads_per_group = cfg->heads_per_group;
  a.q = q;
  a.selection = sel;
  a.out = out;
  a.lse = lse;
  a.partial = partial;
  a.scale_log2 = scale_log2(cfg);
  a.err = err;
  a.spin_limit = kDefaultSpinLimit;
  a.top_k = cfg->top_k;
  a.init_blocks = cfg->init_blocks;
  a.local_blocks = cfg->local_blocks;
  return a;
}

// stage 3: block-major for long query chunks (when allowed), else the persistent team kernel
cudaError_t run_attention(const msa_config_t* cfg, const msa_batch_t* batch, const AttnArgs& a, uint8_t* scratch,
                          int sms, cudaStream_t s, bool block_major_ok) {
  if (block_major_ok && block_major(cfg, batch))
    return launch_block_major_attention(
        a, bm_workspace(scratch, batch->batch, batch->q_len, cfg->num_kv_groups, cfg->heads_per_group, batch->max_blocks),
        sms, s);
  return launch_attention(a, sms, s);
}

}  // namespace

size_t msa::team_attn_workspace_bytes() { return kErrBytes + partial_bytes(); }

msa_status_t msa::sparse_attn_entry(const msa_config_t* cfg, const msa_cache_t* cache, const msa_batch_t* batch,
                                    const uint8_t* q, const int32_t* selection, uint16_t* out, float* lse,
                                    void* workspace, size_t workspace_bytes, void* stream, bool block_major_ok,
                                    bool clear_error) {
  msa_status_t st;
  if ((st = check_config(cfg)) != MSA_OK || (st = check_batch(batch)) != MSA_OK ||
      (st = check_cache(cache, false, true)) != MSA_OK)
    return st;
  if (batch->batch == 0) return MSA_OK;
  if (q == nullptr || selection == nullptr || out == nullptr || !aligned16(q)) return MSA_ERR_INVALID_ARG;
  const size_t need = block_major_ok ? msa_workspace_bytes(MSA_OP_SPARSE_ATTN, cfg, batch) : team_attn_workspace_bytes();
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return MSA_ERR_WORKSPACE;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return MSA_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  AttnArgs a = attn_args(cfg, cache, batch, q, selection, out, lse, reinterpret_cast<float*>(ws + kErrBytes),
                         reinterpret_cast<uint32_t*>(ws));
  if (clear_error && cudaMemsetAsync(ws, 0, sizeof(uint32_t), static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MSA_ERR_CUDA;
  return cuda_status(run_attention(cfg, batch, a, ws + kErrBytes, sms, static_cast<cudaStream_t>(stream), block_major_ok));
}

cudaError_t msa::ensure_dynamic_smem(const void* kernel, size_t bytes) {
  static std::mutex mu;
  static std::unordered_map<uint64_t, size_t> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t key = static_cast<uint64_t>(reinterpret_cast<uintptr_t>(kernel)) * 131u + static_cast<uint64_t>(dev);
  std::lock_guard<std::mutex> lock(mu);
  auto it = done.find(key);
  if (it != done.end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess) done[key] = bytes;
  return e;
}

extern "C" {

int32_t msa_abi_version(void) { return MSA_ABI_VERSION; }

const char* msa_status_string(msa_status_t s) {
  switch (s) {
    case MSA_OK: return "MSA_OK";
    case MSA_ERR_INVALID_ARG: return "MSA_ERR_INVALID_ARG";
    case MSA_ERR_UNSUPPORTED: return "MSA_ERR_UNSUPPORTED";
    case MSA_ERR_WORKSPACE: return "MSA_ERR_WORKSPACE";
    case MSA_ERR_CUDA: return "MSA_ERR_CUDA";
  }
  return "MSA_ERR_UNKNOWN";
}

size_t msa_workspace_bytes(msa_op_t op, const msa_config_t* cfg, const msa_batch_t* batch) {
  if (check_config(cfg) != MSA_OK || check_batch(batch) != MSA_OK) return 0;
  switch (op) {
    case MSA_OP_INDEXER_SCORES: return kErrBytes;
    case MSA_OP_SELECT_BLOCKS: return 0;
    case MSA_OP_SPARSE_ATTN: return kErrBytes + attn_scratch_bytes(cfg, batch);
    case MSA_OP_DECODE:
      return kErrBytes + scores_bytes(cfg, batch) + 2 * sel_bytes(cfg, batch) + attn_scratch_bytes(cfg, batch);
  }
  return 0;
}

msa_status_t msa_nvfp4_insert(const float* x, int64_t n_tokens, int32_t rows_per_token, int32_t dim,
                              const int64_t* slots, uint8_t* data, uint8_t* scale, int64_t num_pages,
                              int32_t block_size, void* stream) {
  if (n_tokens < 0 || rows_per_token < 1 || dim < 16 || dim % 16 != 0 || num_pages < 1 || block_size < 1)
    return MSA_ERR_INVALID_ARG;
  if (n_tokens == 0) return MSA_OK;
  if (x == nullptr || slots == nullptr || data == nullptr || scale == nullptr || !aligned16(x) ||
      (reinterpret_cast<uintptr_t>(data) & 7u) != 0)
    return MSA_ERR_INVALID_ARG;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return MSA_ERR_CUDA;
  QuantArgs a{x, n_tokens, rows_per_token, dim, slots, data, scale, num_pages, block_size};
  return cuda_status(launch_nvfp4_insert(a, sms, static_cast<cudaStream_t>(stream)));
}

msa_status_t msa_fp8_quantize(const float* x, int64_t n, uint8_t* out, void* stream) {
  if (n < 0) return MSA_ERR_INVALID_ARG;
  if (n == 0) return MSA_OK;
  if (x == nullptr || out == nullptr) return MSA_ERR_INVALID_ARG;
  return cuda_status(launch_fp8_quantize(x, n, out, static_cast<cudaStream_t>(stream)));
}

msa_status_t msa_indexer_scores(const msa_config_t* cfg, const msa_cache_t* cache, const msa_batch_t* batch,
                                const uint8_t* index_q, float* block_scores, void* workspace,
                                size_t workspace_bytes, void* stream) {
  msa_status_t st;
  if ((st = check_config(cfg)) != MSA_OK || (st = check_batch(batch)) != MSA_OK ||
      (st = check_cache(cache, true, false)) != MSA_OK)
    return st;
  if (batch->batch == 0) return MSA_OK;
  if (index_q == nullptr || block_scores == nullptr || !aligned16(index_q)) return MSA_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < msa_workspace_bytes(MSA_OP_INDEXER_SCORES, cfg, batch) ||
      !aligned16(workspace))
    return MSA_ERR_WORKSPACE;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return MSA_ERR_CUDA;
  IndexerArgs a = indexer_args(cfg, cache, batch, index_q, block_scores, static_cast<uint32_t*>(workspace));
  return cuda_status(run_indexer(a, sms, static_cast<cudaStream_t>(stream)));
}

msa_status_t msa_select_blocks(const msa_config_t* cfg, const msa_batch_t* batch, const float* block_scores,
                               int32_t* selection, void* stream) {
  msa_status_t st;
  if ((st = check_config(cfg)) != MSA_OK || (st = check_batch(batch)) != MSA_OK) return st;
  if (batch->batch == 0) return MSA_OK;
  if (block_scores == nullptr || selection == nullptr) return MSA_ERR_INVALID_ARG;
  SelectArgs a = select_args(cfg, batch, block_scores, selection);
  return cuda_status(launch_select(a, static_cast<cudaStream_t>(stream)));
}

msa_status_t msa_dcp_local_candidates(const msa_config_t* cfg, const msa_cache_t* cache, const msa_batch_t* batch,
                                      const uint8_t* index_q, int32_t block_lo, int32_t block_hi, float* block_scores,
                                      float* cand_scores, int32_t* cand_blocks, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  msa_status_t st;
  if ((st = check_config(cfg)) != MSA_OK || (st = check_batch(batch)) != MSA_OK ||
      (st = check_cache(cache, true, false)) != MSA_OK)
    return st;
  if (batch->q_len * cfg->num_kv_groups > 8 || cfg->init_blocks != 0 || cfg->local_blocks != 1)
    return MSA_ERR_UNSUPPORTED;
  if (block_lo < 0 || block_hi <= block_lo) return MSA_ERR_INVALID_ARG;
  if (batch->batch == 0) return MSA_OK;
  if (index_q == nullptr || block_scores == nullptr || cand_scores == nullptr || cand_blocks == nullptr ||
      !aligned16(index_q))
    return MSA_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < msa_workspace_bytes(MSA_OP_INDEXER_SCORES, cfg, batch) ||
      !aligned16(workspace))
    return MSA_ERR_WORKSPACE;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return MSA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  IndexerArgs a = indexer_args(cfg, cache, batch, index_q, block_scores, static_cast<uint32_t*>(workspace));
  a.block_lo = block_lo;
  a.block_hi = block_hi;
  cudaError_t e = launch_indexer(a, sms, s);
  if (e == cudaSuccess)
    e = launch_dcp_local(select_args(cfg, batch, block_scores, nullptr), block_lo, block_hi, cand_scores, cand_blocks,
                         s);
  return cuda_status(e);
}

msa_status_t msa_dcp_merge(const msa_config_t* cfg, const msa_batch_t* batch, int32_t num_shards,
                           const float* cand_scores, const int32_t* cand_blocks, int32_t* selection, void* stream) {
  msa_status_t st;
  if ((st = check_config(cfg)) != MSA_OK || (st = check_batch(batch)) != MSA_OK) return st;
  if (cfg->init_blocks != 0 || cfg->local_blocks != 1 || num_shards < 1 || num_shards > kDcpShardsMax)
    return MSA_ERR_UNSUPPORTED;
  if (batch->batch == 0) return MSA_OK;
  if (cand_scores == nullptr || cand_blocks == nullptr || selection == nullptr) return MSA_ERR_INVALID_ARG;
  return cuda_status(launch_dcp_merge(select_args(cfg, batch, nullptr, selection), num_shards, cand_scores,
                                      cand_blocks, static_cast<cudaStream_t>(stream)));
}

msa_status_t msa_sparse_attn_decode(const msa_config_t* cfg, const msa_cache_t* cache, const msa_batch_t* batch,
                                    const uint8_t* q, const int32_t* selection, uint16_t* out, float* lse,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  return msa::sparse_attn_entry(cfg, cache, batch, q, selection, out, lse, workspace, workspace_bytes, stream, true,
                                false);
}

msa_status_t msa_decode(const msa_config_t* cfg, const msa_cache_t* cache, const msa_batch_t* batch,
                        const uint8_t* q, const uint8_t* index_q, uint16_t* out, float* lse,
                        int32_t* selection_out, void* workspace, size_t workspace_bytes, void* stream) {
  msa_status_t st;
  if ((st = check_config(cfg)) != MSA_OK || (st = check_batch(batch)) != MSA_OK ||
      (st = check_cache(cache, true, true)) != MSA_OK)
    return st;
  if (batch->batch == 0) return MSA_OK;
  if (q == nullptr || index_q == nullptr || out == nullptr || !aligned16(q) || !aligned16(index_q))
    return MSA_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < msa_workspace_bytes(MSA_OP_DECODE, cfg, batch) ||
      !aligned16(workspace))
    return MSA_ERR_WORKSPACE;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return MSA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* err = reinterpret_cast<uint32_t*>(ws);
  float* scores = reinterpret_cast<float*>(ws + kErrBytes);
  int32_t* sel = selection_out != nullptr
                     ? selection_out
                     : reinterpret_cast<int32_t*>(ws + kErrBytes + scores_bytes(cfg, batch));
  int32_t* pages = reinterpret_cast<int32_t*>(ws + kErrBytes + scores_bytes(cfg, batch) + sel_bytes(cfg, batch));
  uint8_t* scratch = ws + kErrBytes + scores_bytes(cfg, batch) + 2 * sel_bytes(cfg, batch);
  AttnArgs aa = attn_args(cfg, cache, batch, q, sel, out, lse, reinterpret_cast<float*>(scratch), err);
  aa.q_early = 1;  // the kernel before it is this step's selection, or its indexer
  // a small batch of short rows: the attention's producers select their rows themselves (no
  // selection launch between the indexer and the attention)
  if (!block_major(cfg, batch) && rows_tg(batch, cfg) <= kFusedSelectMaxRows &&
      batch->max_blocks <= kFusedSelectMaxBlocks) {
    aa.block_scores = scores;
    aa.sel_out = sel;
    cudaError_t e = run_indexer(indexer_args(cfg, cache, batch, index_q, scores, err), sms, s);
    if (e == cudaSuccess) e = launch_attention(aa, sms, s);
    return cuda_status(e);
  }
  // the selection looks the selected pages up for the team attention kernel; the step's
  // inputs were written before its first kernel, which waited for them
  SelectArgs sa = select_args(cfg, batch, scores, sel);
  sa.inputs_early = 1;
  if (!block_major(cfg, batch)) {
    sa.block_table = batch->block_table;
    sa.sel_pages = pages;
  }
  cudaError_t e = run_indexer(indexer_args(cfg, cache, batch, index_q, scores, err), sms, s);
  if (e == cudaSuccess) e = launch_select(sa, s);
  if (select_writes_pages(sa)) aa.sel_pages = pages;
  if (e == cudaSuccess) e = run_attention(cfg, batch, aa, scratch, sms, s, true);
  return cuda_status(e);
}

msa_status_t msa_test_indexer_stall(const msa_config_t* cfg, const msa_cache_t* cache, const msa_batch_t* batch,
                                    const uint8_t* index_q, float* block_scores, void* workspace,
                                    size_t workspace_bytes, uint32_t spin_limit, void* stream) {
  msa_status_t st;
  if ((st = check_config(cfg)) != MSA_OK || (st = check_batch(batch)) != MSA_OK ||
      (st = check_cache(cache, true, false)) != MSA_OK)
    return st;
  if (batch->batch == 0) return MSA_OK;
  if (batch->q_len * cfg->num_kv_groups > 8 || spin_limit < 1 || spin_limit > kDefaultSpinLimit)
    return MSA_ERR_UNSUPPORTED;
  if (index_q == nullptr || block_scores == nullptr || !aligned16(index_q)) return MSA_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < msa_workspace_bytes(MSA_OP_INDEXER_SCORES, cfg, batch) ||
      !aligned16(workspace))
    return MSA_ERR_WORKSPACE;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return MSA_ERR_CUDA;
  IndexerArgs a = indexer_args(cfg, cache, batch, index_q, block_scores, static_cast<uint32_t*>(workspace));
  a.spin_limit = spin_limit;
  a.test_withhold = 1;
  return cuda_status(launch_indexer(a, sms, static_cast<cudaStream_t>(stream)));
}

msa_status_t msa_test_attention_stall(const msa_config_t* cfg, const msa_cache_t* cache, const msa_batch_t* batch,
                                      const uint8_t* q, const int32_t* selection, uint16_t* out, float* lse,
                                      void* workspace, size_t workspace_bytes, uint32_t spin_limit, void* stream) {
  msa_status_t st;
  if ((st = check_config(cfg)) != MSA_OK || (st = check_batch(batch)) != MSA_OK ||
      (st = check_cache(cache, false, true)) != MSA_OK)
    return st;
  if (batch->batch == 0) return MSA_OK;
  if (spin_limit < 1 || spin_limit > kDefaultSpinLimit) return MSA_ERR_UNSUPPORTED;
  if (q == nullptr || selection == nullptr || out == nullptr || !aligned16(q)) return MSA_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < team_attn_workspace_bytes() || !aligned16(workspace))
    return MSA_ERR_WORKSPACE;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return MSA_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  AttnArgs a = attn_args(cfg, cache, batch, q, selection, out, lse, reinterpret_cast<float*>(ws + kErrBytes),
                         reinterpret_cast<uint32_t*>(ws));
  a.spin_limit = spin_limit;
  a.test_withhold = 1;
  return cuda_status(launch_attention(a, sms, static_cast<cudaStream_t>(stream)));
}

msa_status_t msa_read_device_error(const void* workspace, uint32_t* flags, void* stream) {
  if (workspace == nullptr || flags == nullptr) return MSA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(flags, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return cuda_status(e);
}

msa_status_t msa_clear_device_error(void* workspace, void* stream) {
  if (workspace == nullptr) return MSA_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(workspace, 0, sizeof(uint32_t), static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
