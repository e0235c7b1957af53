// Top-k block selection of one row by one warp, with the most recent block forced; used by
// the selection kernel and, on the fused decode path, by the attention kernel's producers.
//
// Attention runs only over the top-16 blocks, the most recent block always among them
// ("vLLM liefert Day-0-Unterstützung für MiniMax-M3.1-Flash", §MSA-Grundlagen): the recent
// block r = pos / 128 is kept and counted inside the 16 (local_blocks = 1, init_blocks = 0,
// the local block not counted twice: "MiniMax M3 x vLLM：百万 token 多模态推理的 Day-0 部署",
// §MSA 机制细节); the other 15 are the best blocks before r.  Ranking: higher score first,
// equal scores to the lower block index, NaN below -inf.  Output ascending, -1 padded.
//
// Every candidate n < r gets the 64-bit key  order(score) << 32 | (0xffffffff - n)  (all
// keys distinct, larger = better).
//   1. each lane takes the largest score order (32-bit, without the index) of its strided
//      share (held in registers for rows of up to 1,024 candidates); the 15th largest lane
//      maximum is a lower bound of the 15th best candidate (15 lanes each hold one at least
//      that large);
//   2. the candidates at or above that bound (at least 15, about 20 for the workloads'
//      score distributions) are compacted to shared memory as their exact 64-bit keys:
//      per-lane counts, a warp prefix sum, and every lane writes its own;
//   3. if at most 32 survive (the usual case) each survivor's rank comes from 32 pairwise
//      comparisons across the warp, and each of the 15 winners takes its place in
//      ascending block order (the recent block r, larger than every candidate, goes last);
//      otherwise 15 rounds of warp arg-max pick the winners, over the compacted survivors
//      or, if they overflowed the buffer (adversarial score layouts), over the whole row,
//      and a bitonic sort orders the 16 ids.
#pragma once

#include "msa_device.cuh"

namespace msa {

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

// Bitonic sort of one 64-bit key per lane across the warp, descending (lane 0 largest).
__device__ __forceinline__ uint64_t warp_sort_desc_u64(uint64_t v, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint64_t o = shfl_xor_u64(v, stride);
      const bool desc = ((lane & size) == 0);   // direction of this bitonic run
      const bool lower = ((lane & stride) == 0);
      v = (lower == desc) ? (o > v ? o : v) : (o < v ? o : v);
    }
  }
  return v;
}

// The same for one int per lane, ascending.
__device__ __forceinline__ int warp_sort_asc_i32(int v, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const int o = __shfl_xor_sync(0xffffffffu, v, stride);
      const bool asc = ((lane & size) == 0);
      const bool lower = ((lane & stride) == 0);
      v = (lower == asc) ? min(o, v) : max(o, v);
    }
  }
  return v;
}

// Bitonic sort of one 32-bit key per lane, descending (lane 0 largest).
__device__ __forceinline__ uint32_t warp_sort_desc_u32(uint32_t v, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint32_t o = __shfl_xor_sync(0xffffffffu, v, stride);
      const bool desc = ((lane & size) == 0);
      const bool lower = ((lane & stride) == 0);
      v = (lower == desc) ? max(o, v) : min(o, v);
    }
  }
  return v;
}

// Selection of one row with recent block r: returns, in lane i < 16, the i-th selected block
// id in ascending order (-1 past min(16, r + 1)).  s: the row's block scores (global);
// sord: optional shared staging of row_cap score orders for rows longer than 1,024
// candidates (else they are re-read from L2); cb: a shared buffer of cap >= 32 survivor keys.
// All 32 lanes call it together.
__device__ __forceinline__ int select_row_warp(const float* s, int r, int lane, uint32_t* sord, int row_cap,
                                               uint64_t* cb, int cap) {
  if (r < kTopK) return (lane < kTopK && lane <= r) ? lane : -1;  // every block 0..r
  const bool in_regs = r <= 32 * 32;      // candidate orders held in registers
  const bool staged = !in_regs && sord != nullptr && r <= row_cap;

  // 1. score orders of the candidates, with the lane maxima; the 15th largest lane maximum
  //    bounds the winners from below (15 lanes each hold a candidate at least that large)
  uint32_t o[32];
  uint32_t lmax = 0;
  if (in_regs) {
    float v[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const int n = 32 * k + lane;
      v[k] = n < r ? __ldcg(s + n) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      o[k] = (32 * k + lane < r) ? score_order(v[k]) : 0u;
      lmax = max(lmax, o[k]);
    }
  } else {
    for (int n0 = 0; n0 < r; n0 += 32 * 32) {  // 32 loads in flight per lane
      float v[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int n = n0 + 32 * k + lane;
        v[k] = n < r ? __ldcg(s + n) : 0.f;
      }
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int n = n0 + 32 * k + lane;
        if (n < r) {
          const uint32_t ord = score_order(v[k]);
          if (staged) sord[n] = ord;
          lmax = max(lmax, ord);
        }
      }
    }
  }
  const uint32_t bound = __shfl_sync(0xffffffffu, warp_sort_desc_u32(lmax, lane), kTopK - 2);
  __syncwarp();
  auto order_of = [&](int n) -> uint32_t { return staged ? sord[n] : score_order(__ldcg(s + n)); };
  auto key_of = [](uint32_t ord, int n) -> uint64_t {
    return (static_cast<uint64_t>(ord) << 32) | static_cast<uint64_t>(0xffffffffu - static_cast<uint32_t>(n));
  };

  // 2. compact the candidates whose order is >= bound (at least 15) as exact 64-bit keys:
  //    per-lane counts, a warp prefix sum, then every lane writes its own at its offset
  int cnt = 0;
  if (in_regs) {
#pragma unroll
    for (int k = 0; k < 32; ++k) cnt += (32 * k + lane < r && o[k] >= bound) ? 1 : 0;
  } else {
    for (int n = lane; n < r; n += 32) cnt += order_of(n) >= bound ? 1 : 0;
  }
  int incl = cnt;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += t;
  }
  const int count = __shfl_sync(0xffffffffu, incl, 31);
  if (count <= cap) {
    int idx = incl - cnt;
    if (in_regs) {
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int n = 32 * k + lane;
        if (n < r && o[k] >= bound) cb[idx++] = key_of(o[k], n);
      }
    } else {
      for (int n = lane; n < r; n += 32) {
        const uint32_t ord = order_of(n);
        if (ord >= bound) cb[idx++] = key_of(ord, n);
      }
    }
  }
  __syncwarp();

  // 3. the 15 winners, written in ascending block order, then the recent block
  if (count <= 32) {
    // rank of each survivor by key (keys are distinct; empty lanes hold 0, below every key),
    // then each winner's position among the winners by block index: r is larger than all
    const uint64_t k = lane < count ? cb[lane] : 0ull;
    int rank = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) rank += shfl_u64(k, j) > k ? 1 : 0;
    const bool win = lane < count && rank < kTopK - 1;
    const int id = static_cast<int>(0xffffffffu - static_cast<uint32_t>(k));
    const uint32_t wm = __ballot_sync(0xffffffffu, win);
    int at = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int idj = __shfl_sync(0xffffffffu, id, j);
      at += (((wm >> j) & 1u) && idj < id) ? 1 : 0;
    }
    __syncwarp();  // every survivor key is read: the buffer now takes the ids
    int* ids = reinterpret_cast<int*>(cb);
    if (win) ids[at] = id;
    if (lane == 0) ids[kTopK - 1] = r;
    __syncwarp();
    const int out = lane < kTopK ? ids[lane] : -1;
    __syncwarp();
    return out;
  }
  int mine = -1;  // lane i (< 15) holds the block of the i-th winner
  {
    const bool overflow = count > cap;
    uint64_t prev = ~0ull;
    for (int round = 0; round < kTopK - 1; ++round) {
      uint64_t best = 0;
      if (!overflow) {
        for (int i = lane; i < count; i += 32) {
          const uint64_t k = cb[i];
          if (k < prev && k > best) best = k;
        }
      } else if (in_regs) {  // the survivors overflowed the buffer: scan the whole row
#pragma unroll
        for (int kk = 0; kk < 32; ++kk) {
          const int n = 32 * kk + lane;
          const uint64_t k = n < r ? key_of(o[kk], n) : 0ull;
          if (k < prev && k > best) best = k;
        }
      } else {
        for (int n = lane; n < r; n += 32) {
          const uint64_t k = key_of(order_of(n), n);
          if (k < prev && k > best) best = k;
        }
      }
      best = warp_max_u64(best);
      prev = best;
      if (lane == round) mine = static_cast<int>(0xffffffffu - static_cast<uint32_t>(best));
    }
  }
  if (lane == kTopK - 1) mine = r;
  // 4. ascending order of the 16 ids (the other lanes carry INT_MAX)
  const int sorted_id = warp_sort_asc_i32(lane < kTopK ? mine : 0x7fffffff, lane);
  return lane < kTopK ? sorted_id : -1;
}


}  // namespace msa
