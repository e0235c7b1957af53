/*
 * msa.h -- C ABI of the GB300 (sm_103a) MiniMax Sparse Attention decode library (libmsa.so).
 *
 * MSA replaces full attention with block-sparse attention.  The KV cache is split into
 * 128-token blocks; a lightweight indexer scores every key in the context with one index
 * query per GQA group against a single shared index-key head, max-pools the scores to
 * one score per block, and the main attention then runs exactly, but only over the
 * top-16 blocks, the most recent block always kept, so every query sees at most 2,048
 * keys ("vLLM liefert Day-0-Unterstützung für MiniMax-M3.1-Flash", §MSA-Grundlagen).
 * Both the main K/V cache and the index-key cache are NVFP4 (E2M1 values, one E4M3
 * scale per 16 elements); queries are FP8 E4M3 (same page, §Was ist neu in der
 * MiniMax-M3.1-Architektur and §NVIDIA-Blackwell-optimierte MSA-Kernel).
 *
 * Conventions shared by every entry point:
 *   - Every tensor pointer is DEVICE memory owned by the caller; the library allocates
 *     and frees nothing and never synchronises the device (msa_read_device_error is the
 *     one documented exception).
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL = legacy
 *     default stream) and returns immediately.
 *   - Arguments are validated on the host before anything is launched; a violation
 *     returns MSA_ERR_INVALID_ARG / MSA_ERR_UNSUPPORTED / MSA_ERR_WORKSPACE and
 *     launches nothing.  A failed launch returns MSA_ERR_CUDA.  Output contents are
 *     unspecified after a non-OK status.
 *   - Data that only the device can check (block-table entries, sequence lengths) is
 *     checked in the kernels: a bad entry sets a bit in the workspace error word, the
 *     offending page or sequence is skipped, and nothing traps.
 *   - Query position: token t (0 <= t < q_len) of sequence b sits at position
 *     pos = seq_lens[b] - q_len + t (the q_len new tokens are already in the cache);
 *     key j is visible to it iff j <= pos.  Speculative draft tokens are the q_len
 *     tokens of one request, flattened request-major ("MiniMax M3 x vLLM：百万 token 多模态
 *     推理的 Day-0 部署", §Decode Kernel 中的投机解码).
 *   - seq_lens[b] == 0 marks a padding row: its outputs are defined (scores -inf,
 *     selection -1, output 0, lse -inf) and no error is raised.
 *
 * Layouts (row-major; every pointer 16-byte aligned):
 *   index-key cache  idx_data  uint8 [num_pages][128][Di/2]   idx_scale uint8 [num_pages][128][Di/16]
 *   K (and V) cache  k_data    uint8 [num_pages][G][128][D/2] k_scale   uint8 [num_pages][G][128][D/16]
 *     byte i of a row holds element 2i in its low nibble and element 2i+1 in its high nibble;
 *     scale byte s of a row is the E4M3 scale of elements 16s..16s+15.
 *   block_table      int32 [batch][max_blocks]  logical block n of sequence b -> page
 *   seq_lens         int32 [batch]
 *   queries q        uint8 E4M3 [batch][q_len][G*Hg][D]   (head h belongs to group h / Hg)
 *   index queries    uint8 E4M3 [batch][q_len][G][Di]
 *   block_scores     float [batch][q_len][G][max_blocks]
 *   selection        int32 [batch][q_len][G][16]  ascending logical block ids, -1 padded (rows
 *                    are 16 wide, the largest top_k; entries past min(top_k, r + 1) are -1)
 *   out              bfloat16 bits (uint16) [batch][q_len][G*Hg][D]
 *   lse              float [batch][q_len][G*Hg]  natural log of the softmax denominator
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MSA_ABI_VERSION 2

typedef enum {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer */
  MSA_ERR_UNSUPPORTED = 2,  /* a configuration the library does not implement */
  MSA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than msa_workspace_bytes() */
  MSA_ERR_CUDA = 4          /* a CUDA launch or query failed */
} msa_status_t;

/* Bits of the device error word (first 4 bytes of the workspace). */
#define MSA_DEVERR_BAD_PAGE 0x1u    /* a block-table entry outside [0, num_pages) */
#define MSA_DEVERR_BAD_SEQLEN 0x2u  /* seq_len < q_len (but > 0), or > max_blocks*128 */
#define MSA_DEVERR_TIMEOUT 0x4u     /* a bounded wait inside a kernel gave up */

/* Block-score reduction over the visible keys of a block ("MiniMax M3 x vLLM：百万 token
 * 多模态推理的 Day-0 部署", §Prefill 执行 step 2: a block-level rule such as max or
 * log-sum-exp, by model configuration). */
#define MSA_SCORE_MAX 0  /* max_j s_j (the recipe) */
#define MSA_SCORE_LSE 1  /* ln sum_j e^{s_j} (natural log) */

/* Sparse configuration.  The pages' M3 recipe: block 128, top-16, init_blocks = 0,
 * local_blocks = 1, max pooling ("MiniMax M3 x vLLM：百万 token 多模态推理的 Day-0 部署",
 * §MSA 机制细节, which names init_blocks / local_blocks as configuration).
 * The library implements: num_kv_groups in 1..8, heads_per_group in 1..8,
 * head_dim = index_dim = block_size = 128, 1 <= top_k <= 16, init_blocks >= 0,
 * local_blocks >= 0 with init_blocks + local_blocks <= top_k, score_type MSA_SCORE_MAX or
 * MSA_SCORE_LSE; anything else returns MSA_ERR_UNSUPPORTED.
 * Selection of a row whose recent block is r = pos / 128: min(top_k, r + 1) blocks -- the
 * first init_blocks blocks and the last local_blocks blocks up to r (each once), and the
 * best of the other blocks up to r for the remaining places. */
typedef struct {
  int32_t num_kv_groups;    /* G */
  int32_t heads_per_group;  /* Hg */
  int32_t head_dim;         /* D */
  int32_t index_dim;        /* Di */
  int32_t block_size;       /* tokens per block and per cache page */
  int32_t top_k;            /* blocks kept per (query token, KV group), recent block included */
  int32_t init_blocks;      /* leading blocks always kept */
  int32_t local_blocks;     /* trailing (recent) blocks always kept */
  float softmax_scale;      /* logits = (q . k) * softmax_scale; 0 means 1/sqrt(head_dim) */
  int32_t score_type;       /* MSA_SCORE_MAX or MSA_SCORE_LSE */
} msa_config_t;

/* The paged NVFP4 caches (device, caller-owned, read-only for decode). */
typedef struct {
  const uint8_t* k_data;
  const uint8_t* k_scale;
  const uint8_t* v_data;
  const uint8_t* v_scale;
  const uint8_t* idx_data;
  const uint8_t* idx_scale;
  int64_t num_pages;
} msa_cache_t;

/* One decode batch (device pointers; sizes on the host). */
typedef struct {
  const int32_t* block_table;  /* [batch][max_blocks] */
  const int32_t* seq_lens;     /* [batch] */
  int32_t batch;               /* 0..2048; batch * q_len <= 65535 */
  int32_t max_blocks;          /* >= 1 */
  int32_t q_len;               /* query tokens per sequence, >= 1 */
} msa_batch_t;

typedef enum {
  MSA_OP_INDEXER_SCORES = 0,
  MSA_OP_SELECT_BLOCKS = 1,
  MSA_OP_SPARSE_ATTN = 2,
  MSA_OP_DECODE = 3
} msa_op_t;

/* ABI version of the loaded library (MSA_ABI_VERSION). */
int32_t msa_abi_version(void);

/* Human-readable name of a status code (static string). */
const char* msa_status_string(msa_status_t status);

/* Bytes of device workspace `op` needs for this configuration and batch (host-only
 * arithmetic, no device access).  The workspace must be zero-filled once when it is
 * allocated (its first 4 bytes are the device error word); after that it may be reused
 * by every call with the same or smaller sizes.  Returns 0 for invalid arguments. */
size_t msa_workspace_bytes(msa_op_t op, const msa_config_t* cfg, const msa_batch_t* batch);

/* NVFP4 quantise-and-insert of new cache rows (the cache-write step in front of decode;
 * the pages fuse it into the QKV GEMM epilogue: "vLLM liefert Day-0-Unterstützung für
 * MiniMax-M3.1-Flash", §QKV GEMM + Norm + RoPE + KV-Insert-Fusion).
 *   x        float [n_tokens][rows_per_token][dim]   (K or V: rows = G; index keys: rows = 1)
 *   slots    int64 [n_tokens]  slot = page * block_size + offset of each token
 *   data     uint8 [num_pages][rows_per_token][block_size][dim/2]   (written)
 *   scale    uint8 [num_pages][rows_per_token][block_size][dim/16]  (written)
 * For every 16 consecutive elements: scale code = E4M3(amax/6), amax/6 in float32 rounded
 * to nearest even and saturated at 448; element code = E2M1(x/scale), x/scale in float32,
 * rounded to nearest even, saturated at +-6, sign kept; a zero scale gives zero codes.
 * Slots outside [0, num_pages*block_size) set nothing and are skipped. */
msa_status_t msa_nvfp4_insert(const float* x, int64_t n_tokens, int32_t rows_per_token, int32_t dim,
                              const int64_t* slots, uint8_t* data, uint8_t* scale, int64_t num_pages,
                              int32_t block_size, void* stream);

/* FP8 E4M3 encoding of float32 values (round to nearest even, saturating at +-448, sign kept). */
msa_status_t msa_fp8_quantize(const float* x, int64_t n, uint8_t* out, void* stream);

/* Stage 1 -- indexer score + block pooling.
 * block_scores[b][t][g][n] = max (MSA_SCORE_MAX) or log-sum-exp (MSA_SCORE_LSE) over the
 * visible keys j of block n of (qi[b][t][g] . key_j), exact products (E2M1 x E4M3 x E4M3)
 * accumulated in float32 (the log-sum-exp with expf / logf); -inf where block n has no
 * visible key (n beyond the query's own block or past the sequence end).  Entries
 * n >= ceil(seq_len/128) are written -inf too.  Any q_len works: with R = q_len x groups
 * query rows per sequence, R <= 8 (decode) takes a streaming kernel, 8 < R < 64
 * (speculative decode) a tcgen05 kernel with the keys as M, R >= 64 (chunked prefill) a
 * tcgen05 GEMM with the query rows as M; all three give the same exact products and float32
 * accumulation.  Errors: MSA_ERR_CUDA also when the driver's tensor-map encoder is not
 * available (8 < R < 64) or num_pages * 128 exceeds 2^31 rows there.
 * workspace: msa_workspace_bytes(MSA_OP_INDEXER_SCORES, ...). */
msa_status_t msa_indexer_scores(const msa_config_t* cfg, const msa_cache_t* cache, const msa_batch_t* batch,
                                const uint8_t* index_q, float* block_scores, void* workspace,
                                size_t workspace_bytes, void* stream);

/* Stage 2 -- top-k block selection with forced blocks.
 * For each (b, t, g) with recent block r = pos / 128: the first init_blocks and the last
 * local_blocks blocks up to r are always selected (the recipe: r alone); the other places,
 * up to min(top_k, r + 1) in all, go to the blocks between them ranked by (score
 * descending, index ascending; NaN below -inf); the result is sorted ascending, -1 padded
 * to 16.  Bit-exact for given scores.  No workspace. */
msa_status_t msa_select_blocks(const msa_config_t* cfg, const msa_batch_t* batch, const float* block_scores,
                               int32_t* selection, void* stream);

/* Decode context parallelism, shard side ("vLLM liefert Day-0-Unterstützung für
 * MiniMax-M3.1-Flash", §NVFP4-Indexer-DCP: each GPU scores every index-query head over its
 * slice of the context, keeps a local top-16 per head and sends it to the head's owner, who
 * merges exactly).  On one GPU a shard is a range of logical blocks of every sequence.
 * Scores logical blocks [block_lo, block_hi) exactly as msa_indexer_scores does into
 * block_scores (same layout; -inf for blocks outside the range or past the sequence end),
 * then writes for every (b, t, g) row the shard's best top_k - 1 blocks among
 * [block_lo, min(block_hi, r)) -- r the row's recent block, which the owner adds -- ranked
 * as msa_select_blocks ranks (score descending, then index ascending; NaN below -inf), best
 * first, with their scores:
 *   cand_scores  float [batch][q_len][G][15]   cand_blocks  int32 [batch][q_len][G][15]
 *   (-inf / -1 past the end of a shorter list).
 * Supported: q_len x num_kv_groups <= 8 (decode) and the recipe's init_blocks == 0,
 * local_blocks == 1, else MSA_ERR_UNSUPPORTED; 0 <= block_lo < block_hi, else
 * MSA_ERR_INVALID_ARG.  workspace: msa_workspace_bytes(MSA_OP_INDEXER_SCORES, ...). */
msa_status_t msa_dcp_local_candidates(const msa_config_t* cfg, const msa_cache_t* cache, const msa_batch_t* batch,
                                      const uint8_t* index_q, int32_t block_lo, int32_t block_hi, float* block_scores,
                                      float* cand_scores, int32_t* cand_blocks, void* workspace,
                                      size_t workspace_bytes, void* stream);

/* Decode context parallelism, owner side: merges the candidate lists of num_shards shards
 * (1..8; disjoint block ranges that together cover every block of every sequence) into the
 * selection: the best top_k - 1 of all candidates plus each row's recent block, ascending, -1
 * padded to 16 (every block 0 .. r when r + 1 <= top_k).
 *   cand_scores  float [num_shards][batch][q_len][G][15], cand_blocks int32 alike (the
 *   shards' outputs, concatenated in any shard order).
 * The merge is exact: top_k - 1 of the union of each shard's top_k - 1 is the global top_k - 1
 * under one strict order, so the selection is bit-identical to msa_select_blocks on the
 * unsharded scores.  Same support rules as the shard side; no workspace. */
msa_status_t msa_dcp_merge(const msa_config_t* cfg, const msa_batch_t* batch, int32_t num_shards,
                           const float* cand_scores, const int32_t* cand_blocks, int32_t* selection, void* stream);

/* Stage 3 -- exact sparse GQA attention over the selected blocks.  Every head h of group g
 * attends, with logits (q . k) * softmax_scale, to the visible keys of selection[b][t][g][:];
 * K/V are dequantised exactly from NVFP4 in the kernel.  out is rounded to bfloat16;
 * lse may be NULL.  workspace: msa_workspace_bytes(MSA_OP_SPARSE_ATTN, ...).
 * Below 64 query tokens per sequence the selected pages of all rows are split evenly across
 * the GPU (online softmax, split rows' partial states merged).  From 64 tokens on (chunked
 * prefill) the attention is KV-block-major ("MiniMax M3 x vLLM：百万 token 多模态推理的 Day-0
 * 部署", the query-major versus KV-block-major scheduling of the sparse GQA step): the
 * selections are inverted into a per-block list of (token, slot) entries, each selected
 * block is loaded once for all the tokens that chose it, and every (token, head) merges its
 * per-block partial states by log-sum-exp; its workspace then holds B*T*H*16 partial states
 * of 264 bytes (o / l in fp16, m and l in fp32) and the queries in fp16.  Both forms give
 * the same attention within the stated tolerances, and each is bit-reproducible. */
msa_status_t msa_sparse_attn_decode(const msa_config_t* cfg, const msa_cache_t* cache, const msa_batch_t* batch,
                                    const uint8_t* q, const int32_t* selection, uint16_t* out, float* lse,
                                    void* workspace, size_t workspace_bytes, void* stream);

/* Fused decode step = stage 1 + stage 2 + stage 3 on one stream, intermediate scores and
 * selections kept in the workspace.  selection_out (may be NULL) receives the selection.
 * workspace: msa_workspace_bytes(MSA_OP_DECODE, ...): the error word, the block scores, the
 * selection, the page of every selected entry (looked up by the selection kernel for the
 * team attention kernel) and the stage-3 scratch (the stage-3 form follows the same 64-token
 * rule as msa_sparse_attn_decode).  seq_lens and block_table are read from the selection
 * kernel's start, before the indexer has finished: like q and index_q, they must be written
 * before the call's first kernel runs (any earlier stream-ordered write is).  For a small
 * batch of short rows (at most 128 (token, group) rows of at most 256 blocks, below 64 query
 * tokens) there is no selection kernel: the attention kernel's producers select their rows
 * from the block scores themselves, with the same order (the selection, written to
 * selection_out or the workspace, is the one msa_select_blocks makes). */
msa_status_t msa_decode(const msa_config_t* cfg, const msa_cache_t* cache, const msa_batch_t* batch,
                        const uint8_t* q, const uint8_t* index_q, uint16_t* out, float* lse,
                        int32_t* selection_out, void* workspace, size_t workspace_bytes, void* stream);

/* The stage-3 sparse attention of msa_sparse_attn_decode for callers that cannot allocate
 * device memory, or cannot hand the library a workspace: for example a plugin inside a host
 * application whose device memory all belongs to that application's own pool, or code that
 * must not allocate between decode steps.  The source pages have no counterpart; this is a
 * deployment convenience.
 * Same arguments and results as msa_sparse_attn_decode, minus the workspace: the scratch
 * (partial softmax states of rows shared by two CTAs, and the device error word) lives in
 * one library-owned device array of 8 MiB, which every GPU that loads the library holds
 * until the process exits.  Nothing is allocated or freed.
 *   - It always runs the query-major form (whatever the number of query tokens), whose
 *     scratch is 4.0 MB whatever the batch, so every valid call fits; a call whose scratch
 *     would exceed 8 MiB would be rejected with MSA_ERR_WORKSPACE before any launch.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress,
 *     with that device current); make that first call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents: calls that can
 *     overlap on the GPU (different streams, or different host threads, on one device) race
 *     and must be serialised by the caller.
 *   - The array's device error word (bad block-table entries, bad lengths, a wait that gave
 *     up) is zeroed on `stream` by every call that passes validation, right before its
 *     launch (a rejected call leaves it alone), and read back with
 *     msa_noalloc_read_device_error. */
msa_status_t msa_sparse_attn_decode_noalloc(const msa_config_t* cfg, const msa_cache_t* cache,
                                            const msa_batch_t* batch, const uint8_t* q, const int32_t* selection,
                                            uint16_t* out, float* lse, void* stream);

/* The device error word of the no-allocation entry point's array, as the last call on this
 * device left it (MSA_DEVERR_* bits), copied into *flags; synchronises `stream`.  Like that
 * entry point it needs no workspace, and it shares its race: a call still running on
 * another stream may change the word.  The pages have no counterpart to it either. */
msa_status_t msa_noalloc_read_device_error(uint32_t* flags, void* stream);

/* Test hook for the failure path of the bounded waits; not part of the decode path.
 * Launches the streaming indexer of msa_indexer_scores (q_len x num_kv_groups <= 8; else
 * MSA_ERR_UNSUPPORTED) with its page copies withheld and every wait capped at spin_limit
 * polls (1 .. 2^22; msa_indexer_scores uses 2^22).  Nothing then arrives on the page ring,
 * so each warp with pages to score gives up its first wait, sets MSA_DEVERR_TIMEOUT in the
 * workspace error word and returns, with no copy in flight; block_scores are unspecified
 * afterwards.  The context stays usable: the next regular call computes normally.  Same
 * arguments and workspace as msa_indexer_scores, plus spin_limit. */
msa_status_t msa_test_indexer_stall(const msa_config_t* cfg, const msa_cache_t* cache, const msa_batch_t* batch,
                                    const uint8_t* index_q, float* block_scores, void* workspace,
                                    size_t workspace_bytes, uint32_t spin_limit, void* stream);

/* Test hook for the failure path of the team attention kernel's bounded waits; not part of
 * the decode path.  Runs the query-major team attention of msa_sparse_attn_decode (whatever
 * q_len; workspace of team size: msa_workspace_bytes(MSA_OP_SPARSE_ATTN, ...) for a batch below
 * 64 query tokens) with every wait capped at spin_limit polls (1 .. 2^22) and the page copies
 * withheld: each page slot is armed for its bytes but never filled, so the consumers' first
 * waits run out, then the producers' waits for free slots.  Every wait ends, no copy is in
 * flight when a wait gives up, MSA_DEVERR_TIMEOUT is set in the workspace error word and the
 * launch returns; outputs are unspecified.  The context stays usable. */
msa_status_t msa_test_attention_stall(const msa_config_t* cfg, const msa_cache_t* cache, const msa_batch_t* batch,
                                      const uint8_t* q, const int32_t* selection, uint16_t* out, float* lse,
                                      void* workspace, size_t workspace_bytes, uint32_t spin_limit, void* stream);

/* Debug helper: copies the device error word out of `workspace` into *flags (this call
 * synchronises `stream`). */
msa_status_t msa_read_device_error(const void* workspace, uint32_t* flags, void* stream);

/* Clears the device error word (asynchronous). */
msa_status_t msa_clear_device_error(void* workspace, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H_ */
