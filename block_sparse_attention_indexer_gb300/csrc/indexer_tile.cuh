// Device building blocks of the index-key scan shared by the streaming indexer
// (indexer.cu) and the fused decode step (decode_fused.cu): the flattened (sequence, page)
// unit list and the exact NVFP4 x FP8 score tile on mma.sync.
//
// Scores are the plain dot products of one index query per (query token, KV group) with every
// cached index key ("vLLM liefert Day-0-Unterstützung für MiniMax-M3.1-Flash",
// §MSA-Grundlagen), with exact products: a packed E2M1 byte becomes one f16x2
// (cvt.rn.f16x2.e2m1x2), the block scale multiplies it in f16 (E2M1 x E4M3 products are
// exact in f16), the FP8 query widens exactly to f16, and only the f32 accumulation rounds.
#pragma once

#include <cuda_fp16.h>

#include "msa_device.cuh"

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

}  // namespace msa
