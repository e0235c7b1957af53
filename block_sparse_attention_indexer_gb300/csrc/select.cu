// Stage 2 of MSA decode: top-k block selection with the most recent block forced.
//
// Attention runs "nur über die Top-16-Blöcke, wobei der jüngste Block immer beibehalten
// wird" ("vLLM liefert Day-0-Unterstützung für MiniMax-M3.1-Flash", §MSA-Grundlagen): the
// recent block r = pos / 128 is always kept and counted inside the 16 (local_blocks = 1,
// init_blocks = 0, the local block is not counted twice: "MiniMax M3 x vLLM：百万 token 多模态
// 推理的 Day-0 部署", §MSA 机制细节); the other 15 are the best blocks before r.  Ranking:
// higher score first, equal scores to the lower block index, NaN below -inf.  Output
// ascending, -1 padded.
//
// One warp per (sequence, query token, KV group) row.  Every candidate n < r gets the
// 64-bit key  order(score) << 32 | (0xffffffff - n)  (all keys distinct, larger = better).
//   1. each lane takes the max key of its strided share; the 15th largest lane maximum
//      is a lower bound of the 15th largest key overall (15 lanes each hold a key >= it);
//   2. keys >= that bound (at least 15, typically a few dozen) are compacted to shared
//      memory;
//   3. 15 rounds of warp arg-max over the survivors pick the winners; a lane-parallel rank
//      sort writes them ascending with r.
// If step 2 overflows its buffer (adversarial score layouts) step 3 runs over the whole
// row instead, with the same result.
#include "msa_device.cuh"
#include "msa_kernels.h"

namespace msa {

constexpr int kSelWarps = 4;
constexpr int kSelCap = 512;

__device__ __forceinline__ uint64_t cand_key(float s, int n) {
  return (static_cast<uint64_t>(score_order(s)) << 32) | static_cast<uint64_t>(0xffffffffu - static_cast<uint32_t>(n));
}

__device__ __forceinline__ uint64_t shfl_u64(uint64_t v, int src) {
  uint32_t lo = __shfl_sync(0xffffffffu, static_cast<uint32_t>(v), src);
  uint32_t hi = __shfl_sync(0xffffffffu, static_cast<uint32_t>(v >> 32), src);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int m) {
  uint32_t lo = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(v), m);
  uint32_t hi = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(v >> 32), m);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) {
    uint64_t o = shfl_xor_u64(v, m);
    v = o > v ? o : v;
  }
  return v;
}

__global__ void __launch_bounds__(kSelWarps * 32) select_kernel(const SelectArgs a) {
  __shared__ uint64_t buf[kSelWarps][kSelCap];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nrows = static_cast<int64_t>(a.batch) * a.q_len * a.groups;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kSelWarps + warp;
  if (row >= nrows) return;
  const int b = static_cast<int>(row / (static_cast<int64_t>(a.q_len) * a.groups));
  const int t = static_cast<int>((row / a.groups) % a.q_len);
  int32_t* out = a.selection + row * kTopK;
  const int L = a.seq_lens[b];
  if (L < a.q_len || L <= 0 || L > static_cast<int64_t>(a.max_blocks) * kBlock) {
    if (lane < kTopK) out[lane] = -1;
    return;
  }
  const int pos = L - a.q_len + t;
  const int r = pos / kBlock;
  const float* s = a.block_scores + row * a.max_blocks;
  if (r < kTopK) {  // every block 0..r is selected
    if (lane < kTopK) out[lane] = lane <= r ? lane : -1;
    return;
  }

  // 1. lane maxima and their 15th largest (bitonic sort across the warp, descending)
  uint64_t lmax = 0;
  for (int n = lane; n < r; n += 32) {
    const uint64_t k = cand_key(s[n], n);
    lmax = k > lmax ? k : lmax;
  }
  uint64_t v = lmax;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint64_t o = shfl_xor_u64(v, stride);
      const bool desc = ((lane & size) == 0);        // direction of this bitonic run
      const bool lower = ((lane & stride) == 0);
      const bool keep_max = (lower == desc);
      v = keep_max ? (o > v ? o : v) : (o < v ? o : v);
    }
  }
  const uint64_t bound = shfl_u64(v, kTopK - 2);    // 15th largest lane maximum

  // 2. compact keys >= bound
  uint64_t* cb = buf[warp];
  int count = 0;
  for (int n0 = 0; n0 < r; n0 += 32) {
    const int n = n0 + lane;
    uint64_t k = 0;
    bool take = false;
    if (n < r) {
      k = cand_key(s[n], n);
      take = k >= bound;
    }
    const uint32_t m = __ballot_sync(0xffffffffu, take);
    const int idx = count + __popc(m & ((1u << lane) - 1u));
    if (take && idx < kSelCap) cb[idx] = k;
    count += __popc(m);
  }
  __syncwarp();
  const bool overflow = count > kSelCap;

  // 3. 15 rounds of arg-max below the previous winner
  uint64_t prev = ~0ull;
  int mine = -1;  // lane i (< 15) keeps the i-th winner's block index
  for (int round = 0; round < kTopK - 1; ++round) {
    uint64_t best = 0;
    if (!overflow) {
      for (int i = lane; i < count; i += 32) {
        const uint64_t k = cb[i];
        if (k < prev && k > best) best = k;
      }
    } else {
      for (int n = lane; n < r; n += 32) {
        const uint64_t k = cand_key(s[n], n);
        if (k < prev && k > best) best = k;
      }
    }
    best = warp_max_u64(best);
    prev = best;
    if (lane == round) mine = static_cast<int>(0xffffffffu - static_cast<uint32_t>(best));
  }
  if (lane == kTopK - 1) mine = r;
  // rank sort of the 16 ids (all distinct)
  int rank = 0;
#pragma unroll
  for (int i = 0; i < kTopK; ++i) {
    const int other = __shfl_sync(0xffffffffu, mine, i);
    rank += (other < mine) ? 1 : 0;
  }
  if (lane < kTopK) out[rank] = mine;
}

cudaError_t launch_select(const SelectArgs& a, cudaStream_t s) {
  const int64_t nrows = static_cast<int64_t>(a.batch) * a.q_len * a.groups;
  if (nrows == 0) return cudaSuccess;
  const int64_t blocks = (nrows + kSelWarps - 1) / kSelWarps;
  select_kernel<<<static_cast<unsigned>(blocks), kSelWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace msa
