// Top-k block selection of one row by one warp, with forced blocks; used by the selection
// kernel.
//
// Attention runs only over the top-16 blocks, the most recent block always among them
// ("vLLM liefert Day-0-Unterstützung für MiniMax-M3.1-Flash", §MSA-Grundlagen): the recent
// block r = pos / 128 is kept and counted inside the 16 (local_blocks = 1, init_blocks = 0,
// the local block not counted twice: "MiniMax M3 x vLLM：百万 token 多模态推理的 Day-0 部署",
// §MSA 机制细节, which also names init_blocks leading and local_blocks trailing blocks as
// configuration); the other places go to the best blocks.  Ranking: higher score first,
// equal scores to the lower block index, NaN below -inf.  Output ascending, -1 padded.
//
// Every candidate n gets the 64-bit key  order(score) << 32 | (0xffffffff - n)  (all keys
// distinct, larger = better).  For W winners:
//   1. each lane takes the largest score order (32-bit, without the index) of its strided
//      share (held in registers for up to 1,024 candidates); the W-th largest lane maximum
//      is a lower bound of the W-th best candidate (W lanes each hold one at least that
//      large);
//   2. the candidates at or above that bound (at least W, about 20 for W = 15 and the
//      workloads' score distributions) are compacted to shared memory as their exact
//      64-bit keys: per-lane counts, a warp prefix sum, and every lane writes its own;
//   3. if at most 32 survive (the usual case) each survivor's rank is the number of survivor
//      keys above its own, and each winner takes its place in ascending block order, the
//      number of winners with a smaller block id; otherwise W rounds of warp arg-max pick the
//      winners, over the compacted survivors or, if they overflowed the buffer (adversarial
//      score layouts), over all candidates, and a bitonic sort orders them.
// The counts in 1 and 3 read the values they compare against back from shared memory as
// broadcast vector loads, which issue back to back; a chain of warp shuffles (a sorting
// network, or one shuffle per compared key) waits on each shuffle's latency in turn and cost
// this step several times as much.
#pragma once

#include "msa_device.cuh"
#include "msa_kernels.h"

namespace msa {

constexpr int kSelWarps = 4;   // warps per CTA of the warp-per-row selection kernels
constexpr int kSelCap = 512;   // survivor keys per warp there (a CTA per row keeps kSelCap / 8)

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

// A winner record: block id << 32 | score order (kNoWinner: none; sorts after every record).
constexpr uint64_t kNoWinner = ~0ull;

// The W best of the candidate blocks lo .. hi-1 of one row (0 <= W <= 16, W <= hi - lo):
// returns, in lane i < W, the record of the i-th winner in ascending block order (kOrdered)
// or in rank order, best first (kNoWinner in the other lanes).  s: the row's block scores
// (global); sord: optional shared staging of row_cap score orders for more than 1,024
// candidates (else they are re-read from L2); cb: a 16-byte aligned shared buffer of
// cap >= 32 survivor keys.  All 32 lanes call it together.
// KPL: candidates per lane held in registers (rows of up to 32 * KPL candidates); fewer
// registers for short rows let more warps share an SM.
template <int KPL = 32, bool kOrdered = true>
__device__ __forceinline__ uint64_t top_winners_warp(const float* s, int lo, int hi, int W, int lane, uint32_t* sord,
                                                     int row_cap, uint64_t* cb, int cap) {
  if (W <= 0) return kNoWinner;
  const int nc = hi - lo;                 // candidates
  const bool in_regs = nc <= 32 * KPL;    // candidate orders held in registers
  const bool staged = !in_regs && sord != nullptr && nc <= row_cap;

  // 1. score orders of the candidates, with the lane maxima; the W-th largest lane maximum
  //    bounds the winners from below (W lanes each hold a candidate at least that large)
  uint32_t o[KPL];
  uint32_t lmax = 0;
  if (in_regs) {
    float v[KPL];
#pragma unroll
    for (int k = 0; k < KPL; ++k) {
      const int c = 32 * k + lane;
      v[k] = c < nc ? __ldcg(s + lo + c) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < KPL; ++k) {
      o[k] = (32 * k + lane < nc) ? score_order(v[k]) : 0u;
      lmax = max(lmax, o[k]);
    }
  } else {
    for (int c0 = 0; c0 < nc; c0 += 32 * 32) {  // 32 loads in flight per lane
      float v[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int c = c0 + 32 * k + lane;
        v[k] = c < nc ? __ldcg(s + lo + c) : 0.f;
      }
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int c = c0 + 32 * k + lane;
        if (c < nc) {
          const uint32_t ord = score_order(v[k]);
          if (staged) sord[c] = ord;
          lmax = max(lmax, ord);
        }
      }
    }
  }
  // the W-th largest lane maximum: held by a lane with fewer than W maxima above its own and
  // at least W at or above it (the maxima read back from shared memory four at a time)
  uint32_t* lm = reinterpret_cast<uint32_t*>(cb);
  lm[lane] = lmax;
  __syncwarp();
  int gt = 0, ge = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint4 x = reinterpret_cast<const uint4*>(lm)[j];
    gt += (x.x > lmax ? 1 : 0) + (x.y > lmax ? 1 : 0) + (x.z > lmax ? 1 : 0) + (x.w > lmax ? 1 : 0);
    ge += (x.x >= lmax ? 1 : 0) + (x.y >= lmax ? 1 : 0) + (x.z >= lmax ? 1 : 0) + (x.w >= lmax ? 1 : 0);
  }
  const unsigned at_w = __ballot_sync(0xffffffffu, gt < W && ge >= W);
  const uint32_t bound = __shfl_sync(0xffffffffu, lmax, __ffs(at_w) - 1);
  __syncwarp();  // every lane has read the maxima: the buffer takes the survivors
  auto order_of = [&](int c) -> uint32_t { return staged ? sord[c] : score_order(__ldcg(s + lo + c)); };
  auto key_of = [](uint32_t ord, int n) -> uint64_t {
    return (static_cast<uint64_t>(ord) << 32) | static_cast<uint64_t>(0xffffffffu - static_cast<uint32_t>(n));
  };

  // 2. compact the candidates whose order is >= bound (at least W) as exact 64-bit keys:
  //    per-lane counts, a warp prefix sum, then every lane writes its own at its offset
  int cnt = 0;
  if (in_regs) {
#pragma unroll
    for (int k = 0; k < KPL; ++k) cnt += (32 * k + lane < nc && o[k] >= bound) ? 1 : 0;
  } else {
    for (int c = lane; c < nc; c += 32) cnt += order_of(c) >= bound ? 1 : 0;
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
      for (int k = 0; k < KPL; ++k) {
        const int c = 32 * k + lane;
        if (c < nc && o[k] >= bound) cb[idx++] = key_of(o[k], lo + c);
      }
    } else {
      for (int c = lane; c < nc; c += 32) {
        const uint32_t ord = order_of(c);
        if (ord >= bound) cb[idx++] = key_of(ord, lo + c);
      }
    }
  }
  if (count <= 32 && lane >= count) cb[lane] = 0ull;  // below every key
  __syncwarp();

  // 3. the W winners in ascending block order
  if (count <= 32) {
    // rank of each survivor = survivor keys above its own (keys are distinct; the padding
    // zeros are below every key), read two at a time
    const uint64_t k = cb[lane];
    int rank = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const ulonglong2 x = reinterpret_cast<const ulonglong2*>(cb)[j];
      rank += (x.x > k ? 1 : 0) + (x.y > k ? 1 : 0);
    }
    __syncwarp();  // every survivor key is read: the buffer now takes the records, by rank
    if (lane < count && rank < W)
      cb[rank] = (static_cast<uint64_t>(0xffffffffu - static_cast<uint32_t>(k)) << 32) | (k >> 32);
    __syncwarp();
    const uint64_t rec = lane < W ? cb[lane] : kNoWinner;
    if (!kOrdered) {
      __syncwarp();
      return rec;
    }
    // place of each winner in ascending block order = winners with a smaller block id
    int at = 0;
#pragma unroll
    for (int j = 0; j < kTopK; ++j) at += (j < W && cb[j] < rec) ? 1 : 0;
    __syncwarp();
    if (lane < W) cb[at] = rec;
    __syncwarp();
    const uint64_t out = lane < W ? cb[lane] : kNoWinner;
    __syncwarp();
    return out;
  }
  uint64_t mine = kNoWinner;  // lane i (< W) holds the record of the i-th winner by rank
  {
    const bool overflow = count > cap;
    uint64_t prev = ~0ull;
    for (int round = 0; round < W; ++round) {
      uint64_t best = 0;
      if (!overflow) {
        for (int i = lane; i < count; i += 32) {
          const uint64_t k = cb[i];
          if (k < prev && k > best) best = k;
        }
      } else if (in_regs) {  // the survivors overflowed the buffer: scan the whole row
#pragma unroll
        for (int kk = 0; kk < KPL; ++kk) {
          const int c = 32 * kk + lane;
          const uint64_t k = c < nc ? key_of(o[kk], lo + c) : 0ull;
          if (k < prev && k > best) best = k;
        }
      } else {
        for (int c = lane; c < nc; c += 32) {
          const uint64_t k = key_of(order_of(c), lo + c);
          if (k < prev && k > best) best = k;
        }
      }
      best = warp_max_u64(best);
      prev = best;
      if (lane == round)
        mine = (static_cast<uint64_t>(0xffffffffu - static_cast<uint32_t>(best)) << 32) | (best >> 32);
    }
  }
  if (!kOrdered) return mine;
  // 4. ascending block order of the W records (the other lanes carry kNoWinner, sorted last)
  const uint64_t sorted = ~warp_sort_desc_u64(~mine, lane);
  return lane < W ? sorted : kNoWinner;
}

// The same, as block ids (-1 in the lanes past W).
template <int KPL = 32>
__device__ __forceinline__ int top_blocks_warp(const float* s, int lo, int hi, int W, int lane, uint32_t* sord,
                                               int row_cap, uint64_t* cb, int cap) {
  const uint64_t w = top_winners_warp<KPL>(s, lo, hi, W, lane, sord, row_cap, cb, cap);
  return w == kNoWinner ? -1 : static_cast<int>(w >> 32);
}

// The selection of one row whose recent block is r: min(top_k, r + 1) blocks in ascending
// order -- the first init_blocks, the best top_k - init_blocks - local_blocks of the blocks
// between them and the local window, and the last local_blocks up to r (init_blocks +
// local_blocks <= top_k <= 16; with r + 1 <= top_k every block 0 .. r).  Lane i < 16 gets
// the i-th id (-1 past the end).  The recipe (top_k 16, init 0, local 1) is r plus the 15
// best blocks before it.
template <int KPL = 32>
__device__ __forceinline__ int select_row_warp(const float* s, int r, int top_k, int init_blocks, int local_blocks,
                                               int lane, uint32_t* sord, int row_cap, uint64_t* cb, int cap) {
  if (r + 1 <= top_k) return (lane < kTopK && lane <= r) ? lane : -1;
  // here r >= top_k, so the init blocks, the candidates and the local window are disjoint
  // and in that order: [0, I) [I, r - Lc + 1) [r - Lc + 1, r]
  const int W = top_k - init_blocks - local_blocks;
  const int win = top_blocks_warp<KPL>(s, init_blocks, r - local_blocks + 1, W, lane, sord, row_cap, cb, cap);
  const int from_win = __shfl_sync(0xffffffffu, win, (lane - init_blocks) & 31);
  if (lane < init_blocks) return lane;
  if (lane < init_blocks + W) return from_win;
  if (lane < top_k) return r - local_blocks + 1 + (lane - init_blocks - W);
  return -1;
}

// The selection of one row by NW warps (all of them call it, with the same row and the row's
// sequence length L, read by the caller): each warp takes the best of a contiguous share of the
// candidates, then every thread counts, for one of the shares' winners, the larger of the exact
// keys they left in shared memory over one half of them (a single warp ranking them all waited
// on its own chain of shared loads), and the first warp orders the row's winners.  sync() is a barrier over the NW warps; buf / part / win_ids are their shared
// scratch (buf[NW][kSelCap / 8], part[NW][16], win_ids[16]).  If a.sel_pages is set the page of
// every selected block is written beside it, from tab (the sequence's block-table row in shared
// memory) or, if tab is null, from a.block_table.
template <int NW, int KPL, typename Sync>
__device__ __forceinline__ void select_split_row(const SelectArgs& a, int64_t row, int L, int warp, int lane,
                                                 uint64_t (*buf)[kSelCap / 8], uint64_t (*part)[kTopK],
                                                 int32_t* win_ids, const int32_t* tab, Sync sync) {
  constexpr int kNK = NW * kTopK;  // the shares' winner keys, ranked by 2 x NW x 32 threads
  static_assert(2 * kNK == NW * 32, "two threads per key");
  const int b = static_cast<int>(row / (static_cast<int64_t>(a.q_len) * a.groups));
  const int t = static_cast<int>((row / a.groups) % a.q_len);
  int32_t* out = a.selection + row * kTopK;
  auto page_of = [&](int id) -> int32_t {
    if (id < 0) return -1;
    return tab != nullptr ? tab[id] : a.block_table[static_cast<int64_t>(b) * a.max_blocks + id];
  };
  if (L < a.q_len || L <= 0 || L > static_cast<int64_t>(a.max_blocks) * kBlock) {
    if (warp == 0 && lane < kTopK) {
      out[lane] = -1;
      if (a.sel_pages != nullptr) a.sel_pages[row * kTopK + lane] = -1;
    }
    return;
  }
  const int r = (L - a.q_len + t) / kBlock;
  if (r + 1 <= a.top_k) {  // every block 0 .. r
    if (warp == 0 && lane < kTopK) {
      const int v = lane <= r ? lane : -1;
      out[lane] = v;
      if (a.sel_pages != nullptr) a.sel_pages[row * kTopK + lane] = page_of(v);
    }
    return;
  }
  const float* sc = a.block_scores + row * a.max_blocks;
  const int lo = a.init_blocks, hi = r - a.local_blocks + 1, W = a.top_k - a.init_blocks - a.local_blocks;
  const int span = (hi - lo + NW - 1) / NW;
  const int wlo = min(hi, lo + warp * span), whi = min(hi, wlo + span);
  const int ww = min(W, whi - wlo);
  const uint64_t rec = top_winners_warp<KPL, false>(sc, wlo, whi, ww, lane, nullptr, 0, buf[warp], kSelCap / 8);
  // the share's winner as its exact rank key order(score) << 32 | ~id (0: none, below every key)
  if (lane < kTopK)
    part[warp][lane] = rec == kNoWinner ? 0ull
                                        : (rec << 32) | static_cast<uint64_t>(0xffffffffu - static_cast<uint32_t>(rec >> 32));
  sync();
  // rank of each of the NK shares' winners = keys larger than it (all keys distinct), counted
  // by two threads per key over one half of the keys each, the keys read back two at a time;
  // the per-warp survivor buffers are free now and take the upper halves' counts
  const int tid = warp * 32 + lane;
  const int h = tid / kNK, i = tid - h * kNK;
  const uint64_t key = (&part[0][0])[i];
  int cnt = 0;
  const ulonglong2* half = reinterpret_cast<const ulonglong2*>(&part[0][0]) + h * (kNK / 4);
#pragma unroll
  for (int j = 0; j < kNK / 4; ++j) {
    const ulonglong2 x = half[j];
    cnt += (x.x > key ? 1 : 0) + (x.y > key ? 1 : 0);
  }
  int32_t* cnt_hi = reinterpret_cast<int32_t*>(&buf[0][0]);
  if (h == 1) cnt_hi[i] = cnt;
  sync();
  if (h == 0) {
    const int rank = cnt + cnt_hi[i];
    if (key != 0ull && rank < W) win_ids[rank] = static_cast<int>(0xffffffffu - static_cast<uint32_t>(key));
  }
  sync();
  if (warp != 0) return;
  // ascending order: each winner's place = winners with a smaller block id
  const int my_id = lane < W ? win_ids[lane] : 0x7fffffff;
  int at = 0;
#pragma unroll
  for (int j = 0; j < kTopK; ++j) at += (j < W && win_ids[j] < my_id) ? 1 : 0;
  __syncwarp();
  if (lane < W) win_ids[at] = my_id;
  __syncwarp();
  const int from_win = win_ids[(lane - a.init_blocks) & (kTopK - 1)];
  int v = -1;
  if (lane < a.init_blocks)
    v = lane;
  else if (lane < a.init_blocks + W)
    v = from_win;
  else if (lane < a.top_k)
    v = r - a.local_blocks + 1 + (lane - a.init_blocks - W);
  if (lane < kTopK) {
    out[lane] = v;
    if (a.sel_pages != nullptr) a.sel_pages[row * kTopK + lane] = page_of(v);
  }
}

}  // namespace msa
