// Device building blocks of the streaming index-key scan (indexer.cu): the flattened
// (sequence, page) unit list, the exact NVFP4 x FP8 score tile on mma.sync and one CTA's share
// of the scan.
//
// Scores are the plain dot products of one index query per (query token, KV group) with every
// cached index key ("vLLM liefert Day-0-Unterstützung für MiniMax-M3.1-Flash",
// §MSA-Grundlagen), with exact products: a packed E2M1 byte becomes one f16x2
// (cvt.rn.f16x2.e2m1x2), the block scale multiplies it in f16 (E2M1 x E4M3 products are
// exact in f16), the FP8 query widens exactly to f16, and only the f32 accumulation rounds.
#pragma once

#include <cuda_fp16.h>

#include "msa_device.cuh"
#include "msa_kernels.h"

namespace msa {

constexpr int kHalfData = kPageData / 2;    // 4096: E2M1 bytes of 64 keys
constexpr int kHalfScale = kPageScale / 2;  // 512: their scales
constexpr int kHalfBytes = kHalfData + kHalfScale;

__device__ __forceinline__ int find_seq(const int32_t* prefix, int batch, int64_t u) {
  // largest b with prefix[b] <= u (prefix is non-decreasing, prefix[batch] > u)
  int lo = 0, hi = batch;  // answer in [lo, hi)
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (prefix[mid] <= u) lo = mid; else hi = mid;
  }
  return lo;
}

// Walks the pages of one warp's unit range in order: unit u of sequence b is its page
// u - prefix[b].  Monotone, so the sequence index only ever moves forward.
struct PageCursor {
  int64_t u;      // first unit of the current page (within the warp's range)
  int b;          // its sequence
  int64_t b_end;  // prefix[b + 1]
  __device__ void init(const int32_t* prefix, int batch, int64_t u0, int64_t u1) {
    u = u0;
    b = (u0 < u1) ? find_seq(prefix, batch, u0) : 0;
    b_end = prefix[b + 1];
  }
  __device__ void settle(const int32_t* prefix) {
    while (u >= b_end) {
      ++b;
      b_end = prefix[b + 1];
    }
  }
};

// Pages of a sequence of length L that a scan of logical blocks [block_lo, block_hi) reads.
__device__ __forceinline__ int range_pages(int L, int block_lo, int block_hi) {
  const int nb = (L + kBlock - 1) / kBlock;
  const int hi = nb < block_hi ? nb : block_hi;
  return hi > block_lo ? hi - block_lo : 0;
}

// Exclusive prefix over sequences of their work units (their pages among logical blocks
// [block_lo, block_hi)); sequences with an invalid length get none (and flag
// MSA_DEVERR_BAD_SEQLEN once).  Block-wide scan, ends with __syncthreads.  prefix has batch + 1
// entries; warp_tot one entry per warp of the block.
__device__ __forceinline__ void build_prefix(const int32_t* seq_lens, int batch, int q_len, int max_blocks,
                                             int block_lo, int block_hi, uint32_t* err, int32_t* prefix,
                                             int32_t* warp_tot, int nwarps) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = q_len;
  const int64_t cap = static_cast<int64_t>(max_blocks) * kBlock;
  const int per = (batch + blockDim.x - 1) / blockDim.x;
  const int lo = min(batch, tid * per), hi = min(batch, lo + per);
  int local = 0;
  for (int b = lo; b < hi; ++b) {
    const int L = seq_lens[b];
    const bool ok = (L >= T) && (L <= cap);
    if (L != 0 && !ok && blockIdx.x == 0) flag_error(err, MSA_DEVERR_BAD_SEQLEN);
    local += ok ? range_pages(L, block_lo, block_hi) : 0;
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += warp_tot[w];
  int run = base + incl - local;
  for (int b = lo; b < hi; ++b) {
    prefix[b] = run;
    const int L = seq_lens[b];
    const bool ok = (L >= T) && (L <= cap);
    run += ok ? range_pages(L, block_lo, block_hi) : 0;
  }
  if (tid == blockDim.x - 1) {
    int tot = 0;
    for (int w = 0; w < nwarps; ++w) tot += warp_tot[w];
    prefix[batch] = tot;
  }
  __syncthreads();
}

// single-accumulator tile for one n-tile; scales converted once per row pair
__device__ __forceinline__ void score_tile1(const uint8_t* st, const uint8_t* ss, int r0, int t4,
                                            const uint32_t (&bq)[1][8][2], float (&acc)[4]) {
  const int r1 = r0 + 8;
  const uint4 d0 = lds128(st + r0 * kRowBytes + 16 * t4);
  const uint4 d1 = lds128(st + r1 * kRowBytes + 16 * t4);
  const uint32_t f0 = e4m3x2_to_f16x2(lds16(ss + r0 * kRowScales + 2 * t4));
  const uint32_t f1 = e4m3x2_to_f16x2(lds16(ss + r1 * kRowScales + 2 * t4));
  const uint32_t sc0[2] = {__byte_perm(f0, 0, 0x1010), __byte_perm(f0, 0, 0x3232)};
  const uint32_t sc1[2] = {__byte_perm(f1, 0, 0x1010), __byte_perm(f1, 0, 0x3232)};
  const uint32_t w0[4] = {d0.x, d0.y, d0.z, d0.w};
  const uint32_t w1[4] = {d1.x, d1.y, d1.z, d1.w};
  acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t x0, x1, x2, x3, y0, y1, y2, y3;
    e2m1x8_to_f16x2(w0[w], x0, x1, x2, x3);
    e2m1x8_to_f16x2(w1[w], y0, y1, y2, y3);
    const uint32_t sa = sc0[w >> 1], sb = sc1[w >> 1];
    x0 = hmul2(x0, sa); x1 = hmul2(x1, sa); x2 = hmul2(x2, sa); x3 = hmul2(x3, sa);
    y0 = hmul2(y0, sb); y1 = hmul2(y1, sb); y2 = hmul2(y2, sb); y3 = hmul2(y3, sb);
    mma_f16_16816(acc, x0, y0, x1, y1, bq[0][2 * w][0], bq[0][2 * w][1]);
    mma_f16_16816(acc, x2, y2, x3, y3, bq[0][2 * w + 1][0], bq[0][2 * w + 1][1]);
  }
}

// ------------------------------------------------------------------------------------------
// The streaming index scan, one CTA's share (CTA cta of ncta, kHWarps warps): see indexer.cu.
constexpr int kHWarps = 16;
constexpr int kHStages = 3;

// Dynamic shared memory of one CTA of the scan: its warps' page rings, their mbarriers and the
// sequence prefix (batch + 1 entries).
__host__ __device__ constexpr size_t index_scan_smem_bytes(int batch) {
  return static_cast<size_t>(kHWarps) * kHStages * kHalfBytes + kHWarps * kHStages * sizeof(uint64_t) +
         static_cast<size_t>(batch + 1) * sizeof(int32_t);
}

template <bool LSE>
__device__ __forceinline__ void index_scan_cta(const IndexerArgs& a, uint8_t* smem, int32_t* warp_tot, int cta,
                                               int ncta) {
  uint8_t* stages = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kHWarps * kHStages * kHalfBytes);
  int32_t* prefix = reinterpret_cast<int32_t*>(bars + kHWarps * kHStages);
  const uint64_t l2_once = l2_evict_first_policy();  // every page is read once per call
  constexpr bool lse = LSE;                             // block pooling: log-sum-exp or max
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int T = a.q_len, G = a.groups;
  const int rows = T * G;  // <= 8

  build_prefix(a.seq_lens, a.batch, a.q_len, a.max_blocks, a.block_lo, a.block_hi, a.err, prefix, warp_tot, kHWarps);
  if (lane == 0)
    for (int s = 0; s < kHStages; ++s) mbar_init(&bars[warp * kHStages + s], 1);
  fence_mbar_init();
  __syncthreads();

  const int64_t total = prefix[a.batch];
  const int64_t nwarps = static_cast<int64_t>(ncta) * kHWarps;
  const int64_t gw = static_cast<int64_t>(cta) * kHWarps + warp;
  const int64_t u0 = total * gw / nwarps, u1 = total * (gw + 1) / nwarps;
  uint8_t* my_stages = stages + warp * kHStages * kHalfBytes;
  uint64_t* my_bars = bars + warp * kHStages;

  // ---- issue side: half pages in order; the next page's block-table entry is loaded a page early
  PageCursor ic;
  ic.init(prefix, a.batch, u0, u1);
  int next_page = -1, cur_page = -1, ihalf = 0;
  auto lookup_next = [&]() {
    if (ic.u < u1) {
      ic.settle(prefix);
      next_page =
          __ldg(a.block_table + static_cast<int64_t>(ic.b) * a.max_blocks + (a.block_lo + ic.u - prefix[ic.b]));
    }
  };
  uint32_t valid_bits = 0;
  auto issue_next = [&](int stage) {
    if (ihalf == 0) {
      cur_page = next_page;
      ++ic.u;
      lookup_next();
    }
    const int page = cur_page;
    const bool ok = page >= 0 && page < a.num_pages;
    valid_bits = ok ? (valid_bits | (1u << stage)) : (valid_bits & ~(1u << stage));
    if (lane == 0) {
      uint64_t* bar = &my_bars[stage];
      if (ok) {
        uint8_t* dst = my_stages + stage * kHalfBytes;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, kHalfBytes);
        bulk_g2s_hint(dst, a.idx_data + static_cast<int64_t>(page) * kPageData + ihalf * kHalfData, kHalfData, bar,
                      l2_once);
        bulk_g2s_hint(dst + kHalfData, a.idx_scale + static_cast<int64_t>(page) * kPageScale + ihalf * kHalfScale,
                      kHalfScale, bar, l2_once);
      } else {
        if (ihalf == 0) flag_error(a.err, MSA_DEVERR_BAD_PAGE);
        mbar_arrive(bar);
      }
    }
    ihalf ^= 1;
  };
  const int nhalves = static_cast<int>(2 * (u1 - u0));  // per-warp counters fit 32 bits
  int issued = 0;
  if (u0 < u1 && !a.test_withhold) {  // (the test hook withholds every copy: the first wait runs out)
    lookup_next();
    for (; issued < kHStages && issued < nhalves; ++issued) issue_next(issued % kHStages);
  }

  // ---- consumer
  uint32_t bq[1][8][2];
  int cur_b = -1, L = 0, posc[2] = {-1, -1};
  PageCursor cc;
  cc.init(prefix, a.batch, u0, u1);
  int consumed = 0;
  bool timed_out = false;
  for (int64_t u = u0; u < u1 && !timed_out; ++u) {
    cc.u = u;
    cc.settle(prefix);
    const int b = cc.b;
    const int n = a.block_lo + static_cast<int>(u - prefix[b]);
    if (b != cur_b) {
      cur_b = b;
      L = a.seq_lens[b];
      const int r = g;  // n-tile row of this lane's B fragment
      if (r < rows) {
        const int tq = r / G, gq = r % G;
        const uint4* src = reinterpret_cast<const uint4*>(
            a.index_q + ((static_cast<int64_t>(b) * T + tq) * G + gq) * kDim + 32 * t4);
        const uint4 q0 = __ldg(src), q1 = __ldg(src + 1);
        const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          bq[0][s][0] = e4m3x2_to_f16x2(w[s]);
          bq[0][s][1] = e4m3x2_to_f16x2(w[s] >> 16);
        }
      } else {
#pragma unroll
        for (int s = 0; s < 8; ++s) bq[0][s][0] = bq[0][s][1] = 0u;
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int col = 2 * t4 + e;
        posc[e] = col < rows ? (L - T + col / G) : -1;
      }
    }
    const int pos_min = L - T;
    const bool need_mask = (n + 1) * kBlock - 1 > pos_min;
    PoolState pl[2] = {{-INFINITY, 0.f}, {-INFINITY, 0.f}};
    bool page_ok = true;
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      const int stage = consumed % kHStages;
      if (!mbar_wait_warp(&my_bars[stage], static_cast<uint32_t>((consumed / kHStages) & 1), a.spin_limit)) {
        timed_out = true;
        break;
      }
      page_ok = page_ok && ((valid_bits >> stage) & 1u);
      const uint8_t* st = my_stages + stage * kHalfBytes;
      if (page_ok) {
        float acc[4][4];
#pragma unroll
        for (int k = 0; k < 4; ++k) score_tile1(st, st + kHalfData, k * 16 + g, t4, bq, acc[k]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float v[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) v[e] = acc[k][e];
          if (need_mask) {
            const int j0 = n * kBlock + h * 64 + k * 16 + g, j1 = j0 + 8;
            if (j0 > posc[0]) v[0] = -INFINITY;
            if (j0 > posc[1]) v[1] = -INFINITY;
            if (j1 > posc[0]) v[2] = -INFINITY;
            if (j1 > posc[1]) v[3] = -INFINITY;
          }
          pool_add(pl[0], v[0], v[2], lse);
          pool_add(pl[1], v[1], v[3], lse);
        }
      }
      __syncwarp();
      ++consumed;
      if (issued < nhalves) {
        issue_next(issued % kHStages);
        ++issued;
      }
    }
    if (timed_out) break;
    float mx[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      if (!page_ok) pl[e] = {-INFINITY, 0.f};
      pool_merge_xor(pl[e], 4, lse);
      pool_merge_xor(pl[e], 8, lse);
      pool_merge_xor(pl[e], 16, lse);
      mx[e] = pool_result(pl[e], lse);
    }
    if (g == 0) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int col = 2 * t4 + e;
        if (col < rows) {
          const int tq = col / G, gq = col % G;
          a.block_scores[((static_cast<int64_t>(b) * T + tq) * G + gq) * a.max_blocks + n] = mx[e];
        }
      }
    }
  }

  if (timed_out) {
    if (lane == 0) flag_error(a.err, MSA_DEVERR_TIMEOUT);
    for (int k = consumed; k < issued; ++k)
      mbar_wait(&my_bars[k % kHStages], static_cast<uint32_t>((k / kHStages) & 1), a.spin_limit);
  }

  // ---- -inf for the blocks not scored: past each sequence's end, outside [block_lo, block_hi)
  // (and whole rows of skipped sequences)
  const int64_t nrows = static_cast<int64_t>(a.batch) * rows;
  for (int64_t row = gw; row < nrows; row += nwarps) {
    const int b = static_cast<int>(row / rows);
    const int n1 = a.block_lo + (prefix[b + 1] - prefix[b]);  // scored: [block_lo, n1)
    float* dst = a.block_scores + row * a.max_blocks;
    for (int n = lane; n < a.max_blocks; n += 32)
      if (n < a.block_lo || n >= n1) dst[n] = -INFINITY;
  }
}

}  // namespace msa
