// Kernel argument blocks and launchers shared between the C-ABI layer (api.cu) and the
// kernel translation units.  Host-only declarations; every pointer is device memory.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace msa {

// Polls every bounded wait makes before it gives up and flags MSA_DEVERR_TIMEOUT (kernels
// whose arguments carry a spin_limit take it from there).
constexpr uint32_t kDefaultSpinLimit = 1u << 22;

struct IndexerArgs {
  const uint8_t* idx_data;     // [P][128][64]
  const uint8_t* idx_scale;    // [P][128][8]
  int64_t num_pages;
  const int32_t* block_table;  // [B][max_blocks]
  const int32_t* seq_lens;     // [B]
  int32_t batch, max_blocks, q_len, groups;
  const uint8_t* index_q;      // [B][T][G][128] E4M3
  float* block_scores;         // [B][T][G][max_blocks]
  uint32_t* err;
  int32_t lse;                 // block pooling: 0 max, 1 log-sum-exp
  uint32_t spin_limit;         // polls per bounded wait (streaming kernel)
  int32_t test_withhold;       // test hook: the streaming kernel issues no page copies
  int32_t block_lo, block_hi;  // logical blocks scored (streaming kernel; others get -inf)
};

struct SelectArgs {
  const float* block_scores;   // [B][T][G][max_blocks]
  const int32_t* seq_lens;
  int32_t batch, max_blocks, q_len, groups;
  int32_t* selection;          // [B][T][G][16]
  int32_t top_k, init_blocks, local_blocks;
  int32_t row_cap;             // candidates per row staged in shared memory (set by the launcher)
  // decode step only (else null / 0): the page of every selected entry, [B][T][G][16] (-1 where
  // the selection is -1), looked up in block_table ([B][max_blocks]); inputs_early: seq_lens
  // and block_table were written before the previous kernel on the stream started, so they
  // may be read before waiting on it
  const int32_t* block_table;
  int32_t* sel_pages;
  int32_t inputs_early;
};

struct AttnArgs {
  const uint8_t* k_data;       // [P][G][128][64]
  const uint8_t* k_scale;      // [P][G][128][8]
  const uint8_t* v_data;
  const uint8_t* v_scale;
  int64_t num_pages;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int32_t batch, max_blocks, q_len, groups, heads_per_group;
  const uint8_t* q;            // [B][T][H][128] E4M3
  const int32_t* selection;    // [B][T][G][16]
  const int32_t* sel_pages;    // null, or the page of every selected entry (written with the selection)
  uint16_t* out;               // [B][T][H][128] bf16
  float* lse;                  // [B][T][H] or null
  float* partial;              // attn_partial_bytes(): two partial-state slots per CTA
  float scale_log2;            // softmax_scale * log2(e)
  int32_t q_early;             // 1: read the first queries before waiting on the previous kernel
  uint32_t* err;
  uint32_t spin_limit;         // polls per bounded wait (team kernel)
  int32_t test_withhold;       // test hook: the producers arm each page slot's byte count but
                               // issue no copy, so the consumers' waits run out (team kernel)
  // decode step of a small batch (else null): the producers select each row's blocks from its
  // scores ([B][T][G][max_blocks]) themselves instead of reading `selection`; the team holding
  // a row's first entry writes the row's selection to sel_out
  const float* block_scores;
  int32_t* sel_out;
  int32_t top_k, init_blocks, local_blocks;
};
// the producers' own selection: at most this many rows of at most this many blocks
constexpr int kFusedSelectMaxRows = 128;
constexpr int kFusedSelectMaxBlocks = 256;

struct QuantArgs {
  const float* x;
  int64_t n_tokens;
  int32_t rows_per_token, dim;
  const int64_t* slots;
  uint8_t* data;
  uint8_t* scale;
  int64_t num_pages;
  int32_t block_size;
};

// Raises a kernel's dynamic shared-memory limit to `bytes` the first time a larger size is
// needed on the current device (later calls are a lookup, so launches stay cheap).
cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes);

// Launchers return cudaGetLastError() after enqueueing.
cudaError_t launch_nvfp4_insert(const QuantArgs& a, int num_sms, cudaStream_t s);
cudaError_t launch_fp8_quantize(const float* x, int64_t n, uint8_t* out, cudaStream_t s);
cudaError_t launch_indexer(const IndexerArgs& a, int num_sms, cudaStream_t s);
// tcgen05 GEMM form of the indexer for long query chunks (chunked prefill)
cudaError_t launch_prefill_indexer(const IndexerArgs& a, cudaStream_t s);
// tcgen05 form with the keys as M (converted in registers into tensor memory) for
// 8 < T x G < 64 query rows per sequence (speculative decode)
cudaError_t launch_spec_indexer(const IndexerArgs& a, int num_sms, cudaStream_t s);
// query rows (token x group) per sequence from which the GEMM form is used
constexpr int kPrefillMinRows = 64;
cudaError_t launch_select(const SelectArgs& a, cudaStream_t s);
// whether launch_select(a) fills a.sel_pages (the CTA-per-row form, the table row staged in
// shared memory: decode rows of at most kSelTableCap blocks)
bool select_writes_pages(const SelectArgs& a);
constexpr int kSelTableCap = 4096;
// Decode context parallelism: a shard's best top_k - 1 candidates among logical blocks [lo, hi)
// of every row ([rows][15] scores and block ids, rank order), and the owner's merge of S such
// lists ([S][rows][15] each) into the selection.
cudaError_t launch_dcp_local(const SelectArgs& a, int lo, int hi, float* cand_scores, int32_t* cand_blocks,
                             cudaStream_t s);
cudaError_t launch_dcp_merge(const SelectArgs& a, int S, const float* cand_scores, const int32_t* cand_blocks,
                             cudaStream_t s);
constexpr int kDcpShardsMax = 8;
cudaError_t launch_attention(const AttnArgs& a, int num_sms, cudaStream_t s);

// KV-block-major attention for long query chunks (chunked prefill): K-to-Q CSR plan, block
// attention writing one partial state per (token, head, selection slot), log-sum-exp merge.
struct BmWorkspace {
  int32_t* off;   // [B][G][max_blocks + 1] CSR offsets of each (sequence, group)
  int32_t* cnt;   // [B][G][max_blocks] entries per block (zeroed before each plan)
  int32_t* cur;   // [B][G][max_blocks] insertion cursors
  int32_t* ent;   // [B][G][T * 16] entries t * 16 + slot, grouped by block
  float2* pm;     // [B][T][H][16] (m in the scaled log2 domain, l) of each slot; m = -inf: empty
  __half* po;     // [B][T][H][16][128] o / l of each slot
  __half* q16;    // [B][T][H][128] the queries in f16
};
// query tokens per sequence from which the block-major form is used
constexpr int kBlockMajorMinTokens = 64;
bool bm_supported(int64_t batch, int q_len, int groups, int heads_per_group, int max_blocks);
size_t bm_workspace_bytes(int64_t batch, int q_len, int groups, int heads_per_group, int max_blocks);
BmWorkspace bm_workspace(void* base, int64_t batch, int q_len, int groups, int heads_per_group, int max_blocks);
cudaError_t launch_block_major_attention(const AttnArgs& a, const BmWorkspace& w, int num_sms, cudaStream_t s);

// Upper bound of the attention grid (one CTA per SM); the partial-state area is sized for it.
constexpr int kAttnMaxCtas = 160;
// Bytes of the attention partial-state area (independent of the batch).
size_t attn_partial_bytes();

// Kernel-side limits the host validates against.
constexpr int kMaxBatchSmem = 2048;   // sequences per call (the indexers keep a prefix table in smem)
constexpr int kSelTopK = 16;          // selection width the kernels are built for



}  // namespace msa
