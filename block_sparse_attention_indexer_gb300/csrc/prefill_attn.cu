// Stage 3 for long query chunks (chunked prefill): KV-block-major sparse attention.
//
// In prefill thousands of query tokens of one sequence each select 16 blocks, and many of
// them select the same block.  Walking each query's own blocks (query-major) loads a block
// once per query that chose it; the block-major order inverts the query -> block map into a
// block -> queries list (a K-to-Q CSR), loads each selected KV block once and lets every
// query that chose it attend to it, then merges each query's per-block partial outputs by
// log-sum-exp ("MiniMax M3 x vLLM：百万 token 多模态推理的 Day-0 部署", §Prefill 执行 step 4 and
// the paragraph on query-major versus KV-block-major scheduling of the sparse GQA step;
// §MiniMax 稀疏注意力后端 on the CSR form and the log-sum-exp reduction of partial outputs).
// The result is the same exact attention over the selected set as the query-major kernel.
//
// Launches, each a programmatic dependent of the one before:
//   1. the plan (K-to-Q CSR of every (sequence, KV group)): a memset of the block counters,
//      bm_count_kernel (a CTA per chunk of 128 query tokens of a (sequence, group): its
//      entries' blocks counted in a shared-memory histogram, then one atomic per block; a slot
//      without a block gets the empty state m = -inf for every head; the launch's other CTAs
//      widen the FP8 queries to f16), bm_scan_kernel (one CTA per (sequence, group): exclusive
//      prefix of the counts into offsets and insertion cursors) and bm_scatter_kernel (every
//      valid entry t * 16 + slot into its block's list, a chunk's run of each list reserved
//      with one atomic);
//   2. bm_attn_kernel, persistent, one CTA per SM, on the tcgen05 tensor cores.  A work unit
//      is one (sequence, group, block) with entries.  Loader warps copy the block's K and V
//      pages (18 KB of E2M1 + E4M3 scales, one bulk copy a unit ahead) and dequantise them
//      exactly to f16: K as a K-major 128-byte-swizzled tile (rows = keys), V transposed
//      (rows = dims, K = keys).  The unit's entries go in tiles of 128 query rows (tokens x
//      the group's heads), FP8 -> f16 (exact) into the same layout.  One thread issues
//      S = Q K^T into TMEM; a softmax warpgroup (one row per thread, TMEM lane quarter =
//      warp % 4) reads S back, masks the keys past each token's position, takes the row
//      maximum and p = 2^(s c - m), writes P as f16 into a K-major tile and the row sum; the
//      issuer runs O = P V into TMEM, and the same warpgroup writes o / l as f16 and (m, l)
//      into the slot of the row's selection entry.  Two warpgroups take alternate tiles;
//      S, P and O are double-buffered, so the tensor core works on one tile while the
//      softmax runs on the other.  Every partial covers one block, so no running rescale is
//      needed;
//   3. bm_merge_kernel, one warp per (token, head): o = sum_s w_s (o_s / l_s) / sum_s w_s with
//      w_s = l_s 2^(m_s - M), and the natural-log LSE (M + log2 sum_s w_s) ln 2.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "msa_device.cuh"
#include "msa_kernels.h"
#include "umma.cuh"

namespace msa {

constexpr int kBmThreads = 256;                             // plan and merge kernels
constexpr int kBmRows = 128;                                // query rows (token, head) per tile
constexpr int kBmPageBytes = 2 * (kPageData + kPageScale);  // K data | K scales | V data | V scales
constexpr int kPlanThreads = 1024;
constexpr float kBmLn2 = 0.69314718055994530942f;

__device__ __forceinline__ float bm_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Plan: validity of entry (t, s) of row (b, g) -- a block id in 0 .. r(t) with a valid page.
__device__ __forceinline__ int bm_entry_block(const AttnArgs& a, int b, int g, int t, int s, int L, bool ok) {
  if (!ok) return -1;
  const int n = a.selection[((static_cast<int64_t>(b) * a.q_len + t) * a.groups + g) * kTopK + s];
  const int r = (L - a.q_len + t) / kBlock;
  if (n < 0 || n > r || n >= a.max_blocks) return -1;
  const int p = a.block_table[static_cast<int64_t>(b) * a.max_blocks + n];
  if (p < 0 || p >= a.num_pages) {
    flag_error(a.err, MSA_DEVERR_BAD_PAGE);
    return -1;
  }
  return n;
}

// The plan kernels take a (sequence, group) in chunks of kPlanTokens query tokens, one CTA per
// chunk, kPlanPer entries (token, slot) per thread.  A chunk's block counts are first gathered
// in a shared-memory histogram (its 128 tokens all select their own recent block, and popular
// blocks are chosen by many), so a global counter takes one atomic per chunk instead of one
// per entry; rows of more than kPlanHistMax blocks count with global atomics directly.
constexpr int kPlanTokens = 128;
constexpr int kPlanPer = kPlanTokens * kTopK / kBmThreads;  // 8
constexpr int kPlanHistMax = 12288;                         // 48 KB of shared memory

__device__ __forceinline__ int plan_chunks(const AttnArgs& a) { return (a.q_len + kPlanTokens - 1) / kPlanTokens; }

// The block of each of this thread's entries of chunk `c` (-1: none), entry k = (token t0 +
// (threadIdx.x + k * kBmThreads) / 16, slot (threadIdx.x + k * kBmThreads) % 16).
__device__ __forceinline__ void plan_entries(const AttnArgs& a, int c, int& bg, int& t0, int (&n)[kPlanPer]) {
  const int chunks = plan_chunks(a);
  bg = c / chunks;
  t0 = (c - bg * chunks) * kPlanTokens;
  const int b = bg / a.groups, g = bg - b * a.groups;
  const int L = a.seq_lens[b];
  const bool ok = L > 0 && L >= a.q_len && L <= static_cast<int64_t>(a.max_blocks) * kBlock;
#pragma unroll
  for (int k = 0; k < kPlanPer; ++k) {
    const int e = threadIdx.x + k * kBmThreads, t = t0 + e / kTopK;
    n[k] = t < a.q_len ? bm_entry_block(a, b, g, t, e % kTopK, L, ok) : -1;
  }
}

// Plan, count (CTAs 0 .. count_ctas - 1): each chunk's block counts into the counters, and the
// empty state (m = -inf for every head of the group) for each slot without a block.  The
// CTAs after them widen the FP8 queries to f16 (exact), 16 values per thread: the block
// attention gathers query rows from this copy with asynchronous 16-byte copies straight into
// its swizzled tiles.  (The widening needs nothing of the plan; it shares the launch so that it
// runs beside the counting.)
__global__ void __launch_bounds__(kBmThreads) bm_count_kernel(const AttnArgs a, BmWorkspace w, int count_ctas) {
  extern __shared__ int32_t hist[];  // [max_blocks] when max_blocks <= kPlanHistMax
  grid_dependency_wait();  // the selection (and the zeroed counters)
  grid_dependents_launch();
  if (static_cast<int>(blockIdx.x) >= count_ctas) {
    const int64_t i = static_cast<int64_t>(blockIdx.x - count_ctas) * kBmThreads + threadIdx.x;
    const int64_t nq = static_cast<int64_t>(a.batch) * a.q_len * a.groups * a.heads_per_group * kDim / 16;
    if (i >= nq) return;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.q) + i);
    const uint32_t wq[4] = {v.x, v.y, v.z, v.w};
    uint32_t h[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      h[2 * k] = e4m3x2_to_f16x2(wq[k]);
      h[2 * k + 1] = e4m3x2_to_f16x2(wq[k] >> 16);
    }
    uint4* dst = reinterpret_cast<uint4*>(w.q16) + 2 * i;
    dst[0] = make_uint4(h[0], h[1], h[2], h[3]);
    dst[1] = make_uint4(h[4], h[5], h[6], h[7]);
    return;
  }
  const int MB = a.max_blocks, Hg = a.heads_per_group, H = a.groups * Hg;
  const bool use_hist = MB <= kPlanHistMax;
  if (use_hist) {
    for (int i = threadIdx.x; i < MB; i += kBmThreads) hist[i] = 0;
    __syncthreads();
  }
  int bg, t0, n[kPlanPer];
  plan_entries(a, blockIdx.x, bg, t0, n);
  int32_t* cnt = w.cnt + static_cast<int64_t>(bg) * MB;
  const int b = bg / a.groups, g = bg - b * a.groups;
#pragma unroll
  for (int k = 0; k < kPlanPer; ++k) {
    const int e = threadIdx.x + k * kBmThreads, t = t0 + e / kTopK;
    if (t >= a.q_len) continue;
    if (n[k] >= 0) {
      atomicAdd(use_hist ? &hist[n[k]] : &cnt[n[k]], 1);
    } else {
      for (int h = 0; h < Hg; ++h)
        w.pm[((static_cast<int64_t>(b) * a.q_len + t) * H + g * Hg + h) * kTopK + e % kTopK] =
            make_float2(-INFINITY, 0.f);
    }
  }
  if (use_hist) {
    __syncthreads();
    for (int i = threadIdx.x; i < MB; i += kBmThreads)
      if (hist[i] > 0) atomicAdd(&cnt[i], hist[i]);
  }
}

// Plan, scan: one CTA per (sequence, group), exclusive prefix of the block counts into the
// CSR offsets and the insertion cursors.
__global__ void __launch_bounds__(kPlanThreads) bm_scan_kernel(const AttnArgs a, BmWorkspace w) {
  __shared__ int32_t warp_sum[kPlanThreads / 32];
  grid_dependency_wait();
  grid_dependents_launch();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bg = blockIdx.x, MB = a.max_blocks;
  const int32_t* cnt = w.cnt + static_cast<int64_t>(bg) * MB;
  int32_t* off = w.off + static_cast<int64_t>(bg) * (MB + 1);
  int32_t* cur = w.cur + static_cast<int64_t>(bg) * MB;
  const int per = (MB + kPlanThreads - 1) / kPlanThreads;
  const int lo = min(MB, tid * per), hi = min(MB, lo + per);
  int local = 0;
  for (int n = lo; n < hi; ++n) local += cnt[n];
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  int base = 0;
  for (int i = 0; i < warp; ++i) base += warp_sum[i];
  int run = base + incl - local;
  for (int n = lo; n < hi; ++n) {
    off[n] = run;
    cur[n] = run;
    run += cnt[n];
  }
  if (tid == kPlanThreads - 1) off[MB] = base + incl;
}

// Plan, scatter: every valid entry (t * 16 + slot) to its block's list.  A chunk reserves one
// run of each block's list with one atomic on the block's cursor (its count from the
// shared-memory histogram) and hands the places inside the run out with shared atomics.
__global__ void __launch_bounds__(kBmThreads) bm_scatter_kernel(const AttnArgs a, BmWorkspace w) {
  extern __shared__ int32_t hist[];  // [max_blocks] when max_blocks <= kPlanHistMax
  grid_dependency_wait();
  grid_dependents_launch();
  const int MB = a.max_blocks;
  const bool use_hist = MB <= kPlanHistMax;
  if (use_hist) {
    for (int i = threadIdx.x; i < MB; i += kBmThreads) hist[i] = 0;
    __syncthreads();
  }
  int bg, t0, n[kPlanPer];
  plan_entries(a, blockIdx.x, bg, t0, n);
  int32_t* cur = w.cur + static_cast<int64_t>(bg) * MB;
  int32_t* ent = w.ent + static_cast<int64_t>(bg) * a.q_len * kTopK;
  if (use_hist) {
#pragma unroll
    for (int k = 0; k < kPlanPer; ++k)
      if (n[k] >= 0) atomicAdd(&hist[n[k]], 1);
    __syncthreads();
    for (int i = threadIdx.x; i < MB; i += kBmThreads)
      if (hist[i] > 0) hist[i] = atomicAdd(&cur[i], hist[i]);  // the run's first place
    __syncthreads();
  }
#pragma unroll
  for (int k = 0; k < kPlanPer; ++k) {
    if (n[k] < 0) continue;
    const int e = threadIdx.x + k * kBmThreads;
    ent[atomicAdd(use_hist ? &hist[n[k]] : &cur[n[k]], 1)] = (t0 + e / kTopK) * kTopK + e % kTopK;
  }
}

// ---- tcgen05 block attention ------------------------------------------------------------
// Warp roles of bm_attn_kernel: warps 0-7 softmax + epilogue (warpgroup w = warp / 4 owns the
// tiles of parity w and their buffers; TMEM lane quarter warp % 4), warps 8-10 loaders (the
// unit's page copy and its dequantisation, the query tiles), warp 11 the MMA issuer.
constexpr int kTcSmWarps = 8;
constexpr int kTcLdWarps = 3;  // (12 warps in all: 168 registers a thread, no spills)
constexpr int kTcMmaWarp = kTcSmWarps + kTcLdWarps;
constexpr int kTcThreads = (kTcMmaWarp + 1) * 32;
constexpr int kTcHalf = kBmRows * 128;  // [128 rows x 64 f16] K-major SW128 half tile: 16 KB
constexpr int kTcTile = 2 * kTcHalf;    // 32 KB
constexpr uint32_t kTcTmemCols = 512;   // S[2] at 0 / 128, O[2] at 256 / 384

struct TcShared {
  uint64_t raw_full, kv_full, kv_free, raw_free;
  uint64_t q_full[2], q_empty[2], s_full[2], s_empty[2], p_full[2], p_empty[2], o_full[2], o_empty[2];
  uint32_t tmem_base;
};
// K | V^T | Q[2] | P[2] | raw page | shared
constexpr size_t kTcSmem = 1024 + 6 * static_cast<size_t>(kTcTile) + kBmPageBytes + sizeof(TcShared);

// next unit of this CTA with entries, from u (units advance by gridDim.x); `units` if none
__device__ __forceinline__ int64_t tc_next_unit(const BmWorkspace& w, int64_t u, int64_t units, int MB, int& e0,
                                                int& e1) {
  for (; u < units; u += gridDim.x) {
    const int32_t* off = w.off + (u / MB) * (MB + 1) + (u % MB);
    e0 = off[0];
    e1 = off[1];
    if (e0 < e1) return u;
  }
  return units;
}

// K tile from the raw page: rows = keys, K = dims (the prefill indexer's octet mapping: an
// octet's 16-byte loads and swizzled stores hit 8 distinct bank groups)
__device__ __forceinline__ void tc_dequant_k(const uint8_t* src, uint8_t* kdst, int lt) {
#pragma unroll 2
  for (int item = lt; item < kBlock * 4; item += kTcLdWarps * 32) {
    const int i8 = item & 7, oct = item >> 3;
    const int r = 4 * (oct >> 1) + (i8 & 1) + 2 * (((i8 >> 1) & 1) ^ (oct & 1));
    const int c = i8 >> 1;  // dims 32c .. 32c+31
    const uint4 d = lds128(src + r * kRowBytes + 16 * c);
    const uint32_t sc = lds16(src + kPageData + r * kRowScales + 2 * c);
    const uint32_t s0 = e4m3_bcast_f16x2(sc, 0), s1 = e4m3_bcast_f16x2(sc, 1);
    const uint32_t wd[4] = {d.x, d.y, d.z, d.w};
    uint32_t h[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      e2m1x8_to_f16x2(wd[i], h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
#pragma unroll
      for (int j = 0; j < 4; ++j) h[4 * i + j] = hmul2(h[4 * i + j], i < 2 ? s0 : s1);
    }
    uint8_t* tdst = kdst + (c < 2 ? 0 : kTcHalf);
    const int ch = 4 * (c & 1);
    const bool rot = c >= 2;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int qq = q ^ 2;
      const uint4 v = rot ? make_uint4(h[4 * qq], h[4 * qq + 1], h[4 * qq + 2], h[4 * qq + 3])
                          : make_uint4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
      *reinterpret_cast<uint4*>(tdst + sw128(r, ch + (rot ? qq : q))) = v;
    }
  }
}

// V^T tile from the raw page: rows = dims, K = keys.  Item (dims 8o .. 8o+7; keys 8k .. 8k+7):
// the 8 keys' bytes 4o .. 4o+3 times their scales (f16 pairs of dims of one key), regrouped
// by byte permutes into one 16-byte chunk (8 keys) of each of the 8 dim rows.
__device__ __forceinline__ void tc_dequant_vt(const uint8_t* src, uint8_t* vdst, int lt) {
#pragma unroll 1
  for (int item = lt; item < (kDim / 8) * (kBlock / 8); item += kTcLdWarps * 32) {
    const int o = item & 15, kg = item >> 4;  // dim octet, key group
    uint32_t x[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int key = 8 * kg + j;
      const uint32_t wd = *reinterpret_cast<const uint32_t*>(src + key * kRowBytes + 4 * o);
      const uint32_t sc = e4m3_bcast_f16x2(lds8(src + kPageData + key * kRowScales + (o >> 1)), 0);
      e2m1x8_to_f16x2(wd, x[j][0], x[j][1], x[j][2], x[j][3]);
#pragma unroll
      for (int i = 0; i < 4; ++i) x[j][i] = hmul2(x[j][i], sc);
    }
    uint8_t* base = vdst + (kg >> 3) * kTcHalf;
    const int ch = kg & 7;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      *reinterpret_cast<uint4*>(base + sw128(8 * o + 2 * i, ch)) =
          make_uint4(__byte_perm(x[0][i], x[1][i], 0x5410), __byte_perm(x[2][i], x[3][i], 0x5410),
                     __byte_perm(x[4][i], x[5][i], 0x5410), __byte_perm(x[6][i], x[7][i], 0x5410));
      *reinterpret_cast<uint4*>(base + sw128(8 * o + 2 * i + 1, ch)) =
          make_uint4(__byte_perm(x[0][i], x[1][i], 0x7632), __byte_perm(x[2][i], x[3][i], 0x7632),
                     __byte_perm(x[4][i], x[5][i], 0x7632), __byte_perm(x[6][i], x[7][i], 0x7632));
    }
  }
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// arrives on `bar` once this thread's earlier cp.async copies have landed (counted in the
// barrier's expected arrivals)
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__global__ void __launch_bounds__(kTcThreads, 1) bm_attn_kernel(const AttnArgs a, BmWorkspace w) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base_u32 = smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024 - (base_u32 & 1023)) & 1023);  // SW128 tiles: 1024-byte aligned
  uint8_t* kt = base;
  uint8_t* vt = kt + kTcTile;
  uint8_t* qt = vt + kTcTile;            // [2]
  uint8_t* pt = qt + 2 * kTcTile;        // [2]
  uint8_t* raw = pt + 2 * kTcTile;
  TcShared* sh = reinterpret_cast<TcShared*>(raw + kBmPageBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.q_len, G = a.groups, Hg = a.heads_per_group, H = G * Hg, MB = a.max_blocks;
  const int tok_per_tile = kBmRows / Hg;
  const int E = T * kTopK;
  const int64_t units = static_cast<int64_t>(a.batch) * G * MB;
  const int slots = a.batch * T * H * kTopK;  // partial-state slots (below 2^31: checked on the host)

  if (tid == 0) {
    mbar_init(&sh->raw_full, 1);
    mbar_init(&sh->kv_full, kTcLdWarps);
    mbar_init(&sh->kv_free, 1);
    mbar_init(&sh->raw_free, kTcLdWarps);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh->q_full[b], kTcLdWarps * 32);
      mbar_init(&sh->q_empty[b], 1);
      mbar_init(&sh->s_full[b], 1);
      mbar_init(&sh->s_empty[b], 4);
      mbar_init(&sh->p_full[b], 4);
      mbar_init(&sh->p_empty[b], 1);
      mbar_init(&sh->o_full[b], 1);
      mbar_init(&sh->o_empty[b], 4);
    }
    fence_mbar_init();
  }
  if (warp == kTcMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sh->tmem_base)),
                 "r"(kTcTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  grid_dependency_wait();  // the plan
  grid_dependents_launch();
  bool failed = false;

  if (warp >= kTcSmWarps && warp < kTcMmaWarp) {
    // ---- loaders: per unit the page copy (issued a unit ahead) and its dequantisation into K
    // and V^T, then the unit's query tiles with their row metadata
    const int lt = tid - kTcSmWarps * 32;
    int e0, e1;
    int64_t u = tc_next_unit(w, blockIdx.x, units, MB, e0, e1);
    auto issue_page = [&](int64_t uu) {
      const int bg = static_cast<int>(uu / MB), n = static_cast<int>(uu % MB);
      const int64_t pg = static_cast<int64_t>(a.block_table[static_cast<int64_t>(bg / G) * MB + n]) * G + bg % G;
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&sh->raw_full, kBmPageBytes);
      bulk_g2s(raw, a.k_data + pg * kPageData, kPageData, &sh->raw_full);
      bulk_g2s(raw + kPageData, a.k_scale + pg * kPageScale, kPageScale, &sh->raw_full);
      bulk_g2s(raw + kPageData + kPageScale, a.v_data + pg * kPageData, kPageData, &sh->raw_full);
      bulk_g2s(raw + 2 * kPageData + kPageScale, a.v_scale + pg * kPageScale, kPageScale, &sh->raw_full);
    };
    if (u < units && lt == 0) issue_page(u);
    int nunit = 0, tile = 0;
    bool pending = u < units;  // a page copy is in flight
    // thread lt gathers rows lt, lt + 96, ... of every tile: (token slot r / Hg, head r % Hg)
    for (; u < units && !failed; ++nunit) {
      const int bg = static_cast<int>(u / MB), b = bg / G, g = bg % G;
      const int32_t* ent = w.ent + static_cast<int64_t>(bg) * E;
      const int nt = (e1 - e0 + tok_per_tile - 1) / tok_per_tile;
      // query tile j of the unit (global tile `tile`) with its row metadata
      auto gather = [&](int j) -> bool {
        const int bb = tile & 1, e = e0 + j * tok_per_tile;
        if (tile >= 2 && !mbar_wait(&sh->q_empty[bb], ((tile >> 1) - 1) & 1)) return false;
        const uint32_t q = smem_u32(qt + bb * kTcTile);
        for (int r = lt; r < kBmRows; r += kTcLdWarps * 32) {
          const int tl = r / Hg;  // (with 128 % Hg != 0 the last rows are unused)
          const int et = (tl < tok_per_tile && e + tl < e1) ? ent[e + tl] : -1;
          if (et >= 0) {
            const int64_t qrow = (static_cast<int64_t>(b) * T + (et >> 4)) * H + g * Hg + r % Hg;
            const __half* src = w.q16 + qrow * kDim;
#pragma unroll
            for (int c = 0; c < 16; ++c) cp_async16(q + (c >> 3) * kTcHalf + sw128(r, c & 7), src + 8 * c);
          }
        }
        cp_async_arrive(&sh->q_full[bb]);
        ++tile;
        return true;
      };
      // the unit's first two query tiles go out before the wait for K and V^T (the previous
      // unit's products), so the first product of the unit waits only on the dequantisation
      int j = 0;
      for (; j < nt && j < 2 && !failed; ++j) failed = !gather(j);
      if (failed) break;
      if (!mbar_wait_warp(&sh->raw_full, nunit & 1) || (nunit > 0 && !mbar_wait_warp(&sh->kv_free, (nunit - 1) & 1))) {
        failed = true;
        break;
      }
      pending = false;
      tc_dequant_k(raw, kt, lt);
      tc_dequant_vt(raw + kPageData + kPageScale, vt, lt);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sh->kv_full);
        mbar_arrive(&sh->raw_free);
      }
      int f0, f1;
      const int64_t un = tc_next_unit(w, u + gridDim.x, units, MB, f0, f1);
      // the next page goes into the raw area once every loader is done with it (a bounded
      // mbarrier wait, not a named barrier: a loader that gave up must not stall the rest)
      if (un < units && lt == 0) {
        if (mbar_wait(&sh->raw_free, nunit & 1))
          issue_page(un);
        else
          failed = true;
      }
      if (__any_sync(0xffffffffu, failed)) failed = true;
      pending = un < units && !failed;
      if (failed) break;
      for (; j < nt && !failed; ++j) failed = !gather(j);
      u = un;
      e0 = f0;
      e1 = f1;
    }
    if (failed) {  // the copies in flight, before the CTA leaves (bounded)
      asm volatile("cp.async.wait_all;" ::: "memory");
      if (lt == 0 && pending) mbar_wait(&sh->raw_full, nunit & 1);
    }
  } else if (warp == kTcMmaWarp) {
    // ---- MMA issuer: S = Q K^T of tile i, then O = P V of tile i - 1; at a unit boundary the
    // previous unit's last P V goes first and frees K and V^T for the next dequantisation
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_f16(kBmRows, kBlock);
      const uint32_t ka = smem_u32(kt), va = smem_u32(vt);
      int tile = 0, nunit = 0;
      bool pv_pending = false;
      auto do_pv = [&](int i) -> bool {  // O[i & 1] = P[i & 1] V
        const int bb = i & 1;
        if (!mbar_wait(&sh->p_full[bb], (i >> 1) & 1) || (i >= 2 && !mbar_wait(&sh->o_empty[bb], ((i >> 1) - 1) & 1)))
          return false;
        tc_fence_after();
        const uint32_t pa = smem_u32(pt + bb * kTcTile);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >= 4 ? kTcHalf : 0) + (kk & 3) * 32;
          umma_f16(tmem + 256 + bb * 128, umma_desc(pa + off), umma_desc(va + off), idesc, kk > 0 ? 1u : 0u);
        }
        umma_commit(&sh->o_full[bb]);
        umma_commit(&sh->p_empty[bb]);
        return true;
      };
      int e0, e1;
      for (int64_t u = tc_next_unit(w, blockIdx.x, units, MB, e0, e1); u < units && !failed;
           u = tc_next_unit(w, u + gridDim.x, units, MB, e0, e1), ++nunit) {
        if (pv_pending) {  // the previous unit's last tile
          if (!do_pv(tile - 1)) {
            failed = true;
            break;
          }
          pv_pending = false;
          umma_commit(&sh->kv_free);
        }
        if (!mbar_wait(&sh->kv_full, nunit & 1)) {
          failed = true;
          break;
        }
        for (int e = e0; e < e1; e += tok_per_tile, ++tile) {
          const int bb = tile & 1;
          if (!mbar_wait(&sh->q_full[bb], (tile >> 1) & 1) ||
              (tile >= 2 && !mbar_wait(&sh->s_empty[bb], ((tile >> 1) - 1) & 1))) {
            failed = true;
            break;
          }
          tc_fence_after();
          fence_proxy_async_smem();  // the query rows arrived by cp.async (generic proxy)
          const uint32_t qa = smem_u32(qt + bb * kTcTile);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >= 4 ? kTcHalf : 0) + (kk & 3) * 32;
            umma_f16(tmem + bb * 128, umma_desc(qa + off), umma_desc(ka + off), idesc, kk > 0 ? 1u : 0u);
          }
          umma_commit(&sh->s_full[bb]);
          umma_commit(&sh->q_empty[bb]);
          if (pv_pending && !do_pv(tile - 1)) {
            failed = true;
            break;
          }
          pv_pending = true;
        }
      }
      if (!failed && pv_pending) {
        if (do_pv(tile - 1))
          umma_commit(&sh->kv_free);
        else
          failed = true;
      }
    }
    __syncwarp();
  } else {
    // ---- softmax + epilogue: warpgroup wg takes the tiles of parity wg, one row per thread
    const int wg = warp >> 2, quarter = warp & 3, row = quarter * 32 + lane;
    const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    int tile = 0;
    int e0, e1;
    // the row of each tile: (token slot row / Hg, head row % Hg) of the unit's entries
    const int tl = row / Hg, hh = row % Hg;
    const bool has_row = tl < tok_per_tile;
    for (int64_t u = tc_next_unit(w, blockIdx.x, units, MB, e0, e1); u < units && !failed;
         u = tc_next_unit(w, u + gridDim.x, units, MB, e0, e1)) {
      const int bg = static_cast<int>(u / MB), n = static_cast<int>(u % MB), b = bg / G, g = bg % G;
      const int L = a.seq_lens[b];
      const int32_t* ent = w.ent + static_cast<int64_t>(bg) * E;
      for (int e = e0; e < e1 && !failed; e += tok_per_tile, ++tile) {
        if ((tile & 1) != wg) continue;
        const int bb = wg, k = tile >> 1;
        // the row's partial-state index (-1: no row) and last visible key, read from the CSR
        // while the product is in flight
        const int et = (has_row && e + tl < e1) ? ent[e + tl] : -1;
        int2 m = make_int2(-1, -1);
        if (et >= 0) {
          const int t = et >> 4;
          m.x = static_cast<int>(((static_cast<int64_t>(b) * T + t) * H + g * Hg + hh) * kTopK + (et & 15));
          m.y = (L - T + t) - n * kBlock;
          if (m.x >= slots) m.x = -1;  // defensive: every valid entry indexes below slots
        }
        if (!mbar_wait_warp(&sh->s_full[bb], k & 1)) {
          failed = true;
          break;
        }
        tc_fence_after();
        const int lim = m.y;
        // the row of S in registers: two 64-column loads, one wait (each TMEM wait is a full
        // round trip), each load also returning its maximum (tcgen05.ld.red); pass 1 the
        // maximum over the visible keys, pass 2 the exponentials
        uint32_t sv[2][64];
        float hmax[2];
        tmem_ld64_max(trow + bb * 128, sv[0], hmax[0]);
        tmem_ld64_max(trow + bb * 128 + 64, sv[1], hmax[1]);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        float mrow = -INFINITY;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (64 * h + 63 <= lim) {  // the whole half is visible (every half but the causal edge)
            mrow = fmaxf(mrow, hmax[h]);
          } else {
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int j = 0; j < 64; ++j)
              mx4[j & 3] = fmaxf(mx4[j & 3], 64 * h + j <= lim ? __uint_as_float(sv[h][j]) : -INFINITY);
            mrow = fmaxf(mrow, fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])));
          }
        }
        const float mscaled = lim >= 0 ? mrow * a.scale_log2 : 0.f;
        // S is read: the next tile's product may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->s_empty[bb]);
        // pass 2: p = 2^(s c - m) (0 where masked), the row sum, P as f16 (A operand of P V)
        if (k >= 1 && !mbar_wait_warp(&sh->p_empty[bb], (k - 1) & 1)) {
          failed = true;
          break;
        }
        uint8_t* prow = pt + bb * kTcTile;
        float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t* v = sv[h];
          if (64 * h + 63 <= lim) {
#pragma unroll
            for (int j = 0; j < 64; j += 2) {
              const float p0 = bm_exp2(fmaf(__uint_as_float(v[j]), a.scale_log2, -mscaled));
              const float p1 = bm_exp2(fmaf(__uint_as_float(v[j + 1]), a.scale_log2, -mscaled));
              l4[(j >> 1) & 3] += p0 + p1;
              v[j >> 1] = pack_f16x2(p0, p1);  // packed in place: pair j / 2
            }
          } else {
#pragma unroll
            for (int j = 0; j < 64; j += 2) {
              const float p0 = 64 * h + j <= lim ? bm_exp2(fmaf(__uint_as_float(v[j]), a.scale_log2, -mscaled)) : 0.f;
              const float p1 =
                  64 * h + j + 1 <= lim ? bm_exp2(fmaf(__uint_as_float(v[j + 1]), a.scale_log2, -mscaled)) : 0.f;
              l4[(j >> 1) & 3] += p0 + p1;
              v[j >> 1] = pack_f16x2(p0, p1);
            }
          }
          uint8_t* hdst = prow + h * kTcHalf;  // keys 64h .. 64h+63: SW128 half h
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<uint4*>(hdst + sw128(row, q)) = make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
        const float lrow = (l4[0] + l4[1]) + (l4[2] + l4[3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->p_full[bb]);
        // epilogue: O row / l as f16, staged in the P buffer (its product is done) at exactly the
        // bytes the P layout gives the same row -- dims 64h .. 64h+63 in half h, 128-byte swizzle
        // -- so that a warp touches only its own rows while the warpgroup's faster warps already
        // write the next tile's P; then one coalesced 256-byte store per row into the row's
        // partial slot, with (m, l)
        if (!mbar_wait_warp(&sh->o_full[bb], k & 1)) {
          failed = true;
          break;
        }
        tc_fence_after();
        const float inv = lrow > 0.f ? 1.f / lrow : 0.f;
        uint8_t* stage = pt + bb * kTcTile;
        {
          uint32_t ov[2][64];
          tmem_ld64(trow + 256 + bb * 128, ov[0]);
          tmem_ld64(trow + 256 + bb * 128 + 64, ov[1]);
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t* v = ov[h];
#pragma unroll
            for (int j = 0; j < 64; j += 2)
              v[j >> 1] = pack_f16x2(__uint_as_float(v[j]) * inv, __uint_as_float(v[j + 1]) * inv);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              *reinterpret_cast<uint4*>(stage + h * kTcHalf + sw128(row, q)) =
                  make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          }
        }
        __syncwarp();
#pragma unroll 1
        for (int r8 = 0; r8 < 32; r8 += 8) {  // 8 rows at a time: independent loads, then stores
          int px[8];
          uint2 val[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r2 = quarter * 32 + r8 + i;
            px[i] = __shfl_sync(0xffffffffu, m.x, r8 + i);
            val[i] = *reinterpret_cast<const uint2*>(stage + (lane >> 4) * kTcHalf + sw128(r2, (lane & 15) >> 1) +
                                                     8 * (lane & 1));
          }
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (px[i] >= 0) *reinterpret_cast<uint2*>(w.po + static_cast<int64_t>(px[i]) * kDim + 4 * lane) = val[i];
        }
        __syncwarp();
        if (m.x >= 0) w.pm[m.x] = make_float2(mscaled, lrow);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->o_empty[bb]);
      }
    }
  }
  if (failed && lane == 0) flag_error(a.err, MSA_DEVERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kTcMmaWarp) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcTmemCols));
}

// One warp per (token, head) row: lanes 0-15 read the 16 slots' (m, l), every lane 4 dims.
__global__ void __launch_bounds__(kBmThreads) bm_merge_kernel(const AttnArgs a, BmWorkspace w) {
  grid_dependency_wait();  // the partial states
  grid_dependents_launch();
  const int lane = threadIdx.x & 31;
  const int64_t rows = static_cast<int64_t>(a.batch) * a.q_len * a.groups * a.heads_per_group;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (kBmThreads / 32) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const float2 ml = lane < kTopK ? w.pm[row * kTopK + lane] : make_float2(-INFINITY, 0.f);
  float M = ml.x;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float wt = (ml.x == -INFINITY) ? 0.f : ml.y * bm_exp2(ml.x - M);
  float W = wt;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const __half* po = w.po + row * kTopK * kDim + 4 * lane;
#pragma unroll
  for (int s = 0; s < kTopK; ++s) {
    const float ws = __shfl_sync(0xffffffffu, wt, s);
    if (ws == 0.f) continue;  // warp-uniform
    const uint2 v = __ldcs(reinterpret_cast<const uint2*>(po + s * kDim));
    const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
    const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
    acc[0] = fmaf(ws, f0.x, acc[0]);
    acc[1] = fmaf(ws, f0.y, acc[1]);
    acc[2] = fmaf(ws, f1.x, acc[2]);
    acc[3] = fmaf(ws, f1.y, acc[3]);
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  uint16_t h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[i] * inv));
  *reinterpret_cast<uint2*>(a.out + row * kDim + 4 * lane) =
      make_uint2(static_cast<uint32_t>(h[0]) | (static_cast<uint32_t>(h[1]) << 16),
                 static_cast<uint32_t>(h[2]) | (static_cast<uint32_t>(h[3]) << 16));
  if (lane == 0 && a.lse != nullptr) a.lse[row] = W > 0.f ? (M + log2f(W)) * kBmLn2 : -INFINITY;
}

bool bm_supported(int64_t batch, int q_len, int groups, int heads_per_group, int max_blocks) {
  return q_len >= kBlockMajorMinTokens && max_blocks >= 1 && batch * groups <= 65535 && batch * q_len * groups * heads_per_group * kTopK <= INT32_MAX &&
         batch * q_len * kTopK <= INT32_MAX;
}

size_t bm_workspace_bytes(int64_t batch, int q_len, int groups, int heads_per_group, int max_blocks) {
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t bg = static_cast<size_t>(batch) * groups;
  const size_t slots = static_cast<size_t>(batch) * q_len * groups * heads_per_group * kTopK;
  return al(bg * (max_blocks + 1) * sizeof(int32_t)) + 2 * al(bg * max_blocks * sizeof(int32_t)) +
         al(bg * q_len * kTopK * sizeof(int32_t)) + al(slots * sizeof(float2)) + al(slots * kDim * sizeof(__half)) +
         al(slots / kTopK * kDim * sizeof(__half));
}

BmWorkspace bm_workspace(void* base, int64_t batch, int q_len, int groups, int heads_per_group, int max_blocks) {
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t bg = static_cast<size_t>(batch) * groups;
  const size_t slots = static_cast<size_t>(batch) * q_len * groups * heads_per_group * kTopK;
  uint8_t* p = static_cast<uint8_t*>(base);
  BmWorkspace w;
  w.off = reinterpret_cast<int32_t*>(p);
  p += al(bg * (max_blocks + 1) * sizeof(int32_t));
  w.cnt = reinterpret_cast<int32_t*>(p);
  p += al(bg * max_blocks * sizeof(int32_t));
  w.cur = reinterpret_cast<int32_t*>(p);
  p += al(bg * max_blocks * sizeof(int32_t));
  w.ent = reinterpret_cast<int32_t*>(p);
  p += al(bg * q_len * kTopK * sizeof(int32_t));
  w.pm = reinterpret_cast<float2*>(p);
  p += al(slots * sizeof(float2));
  w.po = reinterpret_cast<__half*>(p);
  p += al(slots * kDim * sizeof(__half));
  w.q16 = reinterpret_cast<__half*>(p);
  return w;
}

cudaError_t launch_block_major_attention(const AttnArgs& a, const BmWorkspace& w, int num_sms, cudaStream_t s) {
  const int64_t units = static_cast<int64_t>(a.batch) * a.groups * a.max_blocks;
  if (units == 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // 1. plan: zero the counters, count (with the queries widened to f16 beside it), scan, scatter
  const int64_t plan_ctas = static_cast<int64_t>(a.batch) * a.groups * ((a.q_len + kPlanTokens - 1) / kPlanTokens);
  const int64_t q16n = static_cast<int64_t>(a.batch) * a.q_len * a.groups * a.heads_per_group * kDim / 16;
  const size_t hist_bytes = a.max_blocks <= kPlanHistMax ? static_cast<size_t>(a.max_blocks) * sizeof(int32_t) : 0;
  cudaError_t e = cudaMemsetAsync(w.cnt, 0, static_cast<size_t>(a.batch) * a.groups * a.max_blocks * sizeof(int32_t), s);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(static_cast<unsigned>(plan_ctas + (q16n + kBmThreads - 1) / kBmThreads));
  cfg.blockDim = dim3(kBmThreads);
  cfg.dynamicSmemBytes = hist_bytes;
  e = cudaLaunchKernelEx(&cfg, bm_count_kernel, a, w, static_cast<int>(plan_ctas));
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(static_cast<unsigned>(a.batch * a.groups));
  cfg.blockDim = dim3(kPlanThreads);
  cfg.dynamicSmemBytes = 0;
  e = cudaLaunchKernelEx(&cfg, bm_scan_kernel, a, w);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(static_cast<unsigned>(plan_ctas));
  cfg.blockDim = dim3(kBmThreads);
  cfg.dynamicSmemBytes = hist_bytes;
  e = cudaLaunchKernelEx(&cfg, bm_scatter_kernel, a, w);
  if (e != cudaSuccess) return e;
  // 2. the block-major attention, one CTA per SM, striding over the (sequence, group, block) units
  e = ensure_dynamic_smem(reinterpret_cast<const void*>(bm_attn_kernel), kTcSmem);
  if (e != cudaSuccess) return e;
  const int64_t grid = units < num_sms ? units : num_sms;
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = kTcSmem;
  e = cudaLaunchKernelEx(&cfg, bm_attn_kernel, a, w);
  if (e != cudaSuccess) return e;
  // 3. merge, a warp per (token, head)
  const int64_t rows = static_cast<int64_t>(a.batch) * a.q_len * a.groups * a.heads_per_group;
  cfg.gridDim = dim3(static_cast<unsigned>((rows + kBmThreads / 32 - 1) / (kBmThreads / 32)));
  cfg.blockDim = dim3(kBmThreads);
  cfg.dynamicSmemBytes = 0;
  e = cudaLaunchKernelEx(&cfg, bm_merge_kernel, a, w);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace msa
