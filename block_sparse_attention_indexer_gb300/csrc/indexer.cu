// Stage 1 of MSA decode for at most 8 query rows per sequence (T x G <= 8): indexer
// score + block pooling.
//
// Every cached key j is scored against one index query per (query token, KV group) through
// the single shared index-key head, and the scores of a 128-token block are reduced (max, or
// log-sum-exp) over the keys visible to the query ("vLLM liefert Day-0-Unterstützung für
// MiniMax-M3.1-Flash", §MSA-Grundlagen; masks from "MiniMax M3 x vLLM：百万 token 多模态推理的
// Day-0 部署", §MSA 机制细节).  Longer query rows go to the tcgen05 kernels (spec_indexer.cu
// for 9..63 rows, prefill.cu from 64 rows).
//
// Design (GB300): the path is HBM-bound (72 bytes of NVFP4 index key per token, read
// once per step), so the kernel is a persistent streaming scan:
//   * one CTA per SM, 16 independent warps; the flattened list of (sequence, page) units is
//     split into equal contiguous ranges, one per warp (balanced to one page whatever the
//     ragged lengths);
//   * each warp streams its pages as half pages (64 keys: 4 KB of E2M1 + 512 B of scales)
//     through a private 3-stage ring of shared-memory buffers filled by bulk async copies
//     (cp.async.bulk + mbarrier), so ~216 KB per SM is always in flight;
//   * scores run on the tensor cores (mma.sync m16n8k16, f16 in, f32 accumulate) with keys
//     as M (16 per tile) and the <= 8 query rows (token, group) as N: one packed E2M1 byte
//     becomes one f16x2 A register (cvt.rn.f16x2.e2m1x2), the block scale multiplies it in
//     f16 (E2M1 x E4M3 products are exact in f16), and the FP8 index query widens exactly to
//     f16, so every product is exact and only the f32 accumulation rounds -- the exact-score
//     idea of the Rubin section of the M3.1 post, instead of re-rounding keys to FP8;
//   * the contraction order over the 128 dims is permuted so that each lane reads 16
//     contiguous bytes per key row (the dot product is order-free; the queries use the same
//     permutation);
//   * the block pool is a register reduction over the key tiles of a half page, a 3-step
//     shuffle reduction, and a combine of the two halves; per-token scores never leave
//     registers.
#include <cuda_fp16.h>

#include "indexer_tile.cuh"
#include "msa_device.cuh"
#include "msa_kernels.h"

namespace msa {

// ------------------------------------------------------------------------------------------
constexpr int kHWarps = 16;
constexpr int kHStages = 3;

template <bool LSE>
__global__ void __launch_bounds__(kHWarps * 32, 1) indexer_half_kernel(const IndexerArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stages = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kHWarps * kHStages * kHalfBytes);
  int32_t* prefix = reinterpret_cast<int32_t*>(bars + kHWarps * kHStages);
  __shared__ int32_t warp_tot[kHWarps];

  grid_dependency_wait();
  grid_dependents_launch();
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
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kHWarps;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kHWarps + warp;
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

template <bool LSE>
static cudaError_t launch_half_t(const IndexerArgs& a, int num_sms, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(kHWarps) * kHStages * kHalfBytes + kHWarps * kHStages * sizeof(uint64_t) +
                      (a.batch + 1) * sizeof(int32_t);
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(indexer_half_kernel<LSE>), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kHWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, indexer_half_kernel<LSE>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

static cudaError_t launch_half(const IndexerArgs& a, int num_sms, cudaStream_t s) {
  return a.lse ? launch_half_t<true>(a, num_sms, s) : launch_half_t<false>(a, num_sms, s);
}

cudaError_t launch_indexer(const IndexerArgs& a, int num_sms, cudaStream_t s) {
  if (a.q_len * a.groups > 8) return cudaErrorInvalidValue;  // longer rows go to the tcgen05 indexers
  return launch_half(a, num_sms, s);
}

}  // namespace msa
