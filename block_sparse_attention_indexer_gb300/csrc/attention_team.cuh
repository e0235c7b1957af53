// The persistent team form of the query-major sparse attention and the merge of rows it splits,
// as device functions of one CTA; attention.cu wraps them in its kernels and describes the
// design.
#pragma once

#include "attention_tile.cuh"
#include "msa_device.cuh"
#include "msa_kernels.h"
#include "select_row.cuh"

namespace msa {

constexpr int kTeams = 3;                                 // teams per CTA
constexpr int kTW = 4;                                    // warps per team (one 32-key quarter each)
constexpr int kAW = kTeams * kTW;                         // consuming warps per CTA
constexpr int kAttnThreads = (kAW + kTeams) * 32;         // + one producer warp per team
constexpr int kTSl = 3;                                   // page slots per team
// per team: slots, merge area, item metadata, barriers
struct TeamBars {
  uint64_t full[kTSl];   // a page (or a marker item) is in the slot: 1 arrive (+ copy bytes)
  uint64_t empty[kTSl];  // every warp of the team is done with the slot: kTW arrives
  uint64_t merged;       // every warp wrote its segment state: kTW arrives
  uint64_t freed;        // every warp finished reading the merge area: kTW arrives
};
struct ItemMeta {
  int row;      // row of the item, -1 = end of the team's items
  int blk;      // logical block (page items)
  int page;     // page id, -1 = no page (a row with nothing to attend to)
  int pos;      // query position of the row (page items)
};

// Shared memory: page slots | mbarriers | per-warp merge areas | item metadata.  Every region
// starts on a 16-byte boundary (the slots take bulk copies, the barriers need 8 bytes).
constexpr size_t kSlotsBytes = static_cast<size_t>(kTeams) * kTSl * kSlotBytes;
constexpr size_t kBarsBytes = (static_cast<size_t>(kTeams) * sizeof(TeamBars) + 15) / 16 * 16;
constexpr size_t kRedBytes = static_cast<size_t>(kAW) * kRedFloats * sizeof(float);
static_assert(kSlotsBytes % 16 == 0 && kRedBytes % 16 == 0, "attention shared-memory regions must stay 16-byte aligned");

// the producers' ranking scratch when they select rows themselves: 32 keys each, after the
// item metadata (16-byte aligned: the ranking reads it back as 16-byte vectors)
constexpr size_t kMetaBytes = static_cast<size_t>(kTeams) * kTSl * sizeof(ItemMeta);
constexpr size_t kSelScratchOff = kSlotsBytes + kBarsBytes + kRedBytes + kMetaBytes;
static_assert(kSelScratchOff % 16 == 0, "the selection scratch must be 16-byte aligned");

__host__ __device__ constexpr size_t attn_smem_bytes() {
  return kSelScratchOff + static_cast<size_t>(kTeams) * 32 * sizeof(uint64_t);
}

// Team c of NC owns the entries [range_lo(c), range_lo(c + 1)) of the E = rows * 16 entries.
__host__ __device__ __forceinline__ int range_lo(int E, int c, int NC) {
  return static_cast<int>(static_cast<int64_t>(E) * c / NC);
}
__host__ __device__ __forceinline__ int owner_of(int E, int x, int NC) {
  return static_cast<int>((static_cast<int64_t>(x + 1) * NC - 1) / E);
}

// Row bookkeeping in 32-bit arithmetic: rows = batch * q_len * groups < 2^20 (the host
// bounds batch * q_len by 65535 and groups by 8), entries and head rows < 2^23.  The query
// heads of row (b, t, g) are the head rows row * heads_per_group + h.
struct RowInfo {
  int b, t, g, r, L;
  bool ok;
};

__device__ __forceinline__ RowInfo row_info(const AttnArgs& a, int row) {
  RowInfo ri;
  const unsigned T = static_cast<unsigned>(a.q_len), G = static_cast<unsigned>(a.groups);
  const unsigned bt = static_cast<unsigned>(row) / G;
  ri.g = static_cast<int>(static_cast<unsigned>(row) - bt * G);
  ri.b = static_cast<int>(bt / T);
  ri.t = static_cast<int>(bt - static_cast<unsigned>(ri.b) * T);
  ri.L = a.seq_lens[ri.b];
  ri.ok = ri.L > 0 && ri.L >= a.q_len && ri.L <= static_cast<int64_t>(a.max_blocks) * kBlock;
  ri.r = ri.ok ? (ri.L - a.q_len + ri.t) / kBlock : -1;
  return ri;
}

// A producer's own selection of row R (the decode step of a small batch): the row's blocks
// chosen from its block scores with the selection kernels' total order (select_row_warp:
// higher score first, lower block on ties, the forced blocks), so the selection is the one
// msa_select_blocks makes; written out when `own` (the team holds the row's first entry),
// then resolved to pages like a read selection.  cb: 32 keys of shared scratch.
__device__ __forceinline__ void select_resolve(const AttnArgs& a, int R, int lane, uint64_t* cb, bool own, int& blk,
                                               int& page, int& pos) {
  const unsigned TG = static_cast<unsigned>(a.q_len * a.groups);
  const int b = static_cast<int>(static_cast<unsigned>(R) / TG);
  const int t = static_cast<int>((static_cast<unsigned>(R) - static_cast<unsigned>(b) * TG) /
                                 static_cast<unsigned>(a.groups));
  RowRaw raw;
  raw.L = a.seq_lens[b];
  raw.page = -1;
  const bool ok = raw.L > 0 && raw.L >= a.q_len && raw.L <= static_cast<int64_t>(a.max_blocks) * kBlock;
  raw.blk = ok ? select_row_warp<8>(a.block_scores + static_cast<int64_t>(R) * a.max_blocks,
                                    (raw.L - a.q_len + t) / kBlock, a.top_k, a.init_blocks, a.local_blocks, lane,
                                    nullptr, 0, cb, 32)
               : -1;
  if (own && lane < kTopK) a.sel_out[static_cast<int64_t>(R) * kTopK + lane] = raw.blk;
  row_resolve(a, R, raw, lane, blk, page, pos);
}

// Sends one item into the team's next slot once its four warps have released it: a page
// (its K and V pages of KV head `row % groups`, by bulk copy), a marker (page -1: a row
// segment with nothing to attend to) or the end (row -1).  False if the wait gave up.
__device__ __forceinline__ bool send_item(const AttnArgs& a, int& produced, uint8_t* slots, ItemMeta* meta,
                                          TeamBars* tb, int lane, int row, int blk, int page, int pos) {
  const int slot = produced % kTSl;
  if (produced >= kTSl && !mbar_wait_warp(&tb->empty[slot], ((produced / kTSl) - 1) & 1, a.spin_limit)) return false;
  if (lane == 0) {
    uint64_t* bar = &tb->full[slot];
    meta[slot].row = row;
    meta[slot].blk = blk;
    meta[slot].page = page;
    meta[slot].pos = pos;
    if (page >= 0) {
      uint8_t* dst = slots + slot * kSlotBytes;
      const int64_t pg = static_cast<int64_t>(page) * a.groups + row % a.groups;
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, kSlotBytes);
      if (a.test_withhold) {
        // (test hook: no copy is issued, the slot never fills)
      } else if (a.q_len == 1) {  // one token per sequence: every page is read once per call
        const uint64_t pol = l2_evict_first_policy();
        bulk_g2s_hint(dst, a.k_data + pg * kPageData, kPageData, bar, pol);
        bulk_g2s_hint(dst + kPageData, a.k_scale + pg * kPageScale, kPageScale, bar, pol);
        bulk_g2s_hint(dst + kPageData + kPageScale, a.v_data + pg * kPageData, kPageData, bar, pol);
        bulk_g2s_hint(dst + 2 * kPageData + kPageScale, a.v_scale + pg * kPageScale, kPageScale, bar, pol);
      } else {  // the tokens of a sequence share most pages: keep them in L2
        bulk_g2s(dst, a.k_data + pg * kPageData, kPageData, bar);
        bulk_g2s(dst + kPageData, a.k_scale + pg * kPageScale, kPageScale, bar);
        bulk_g2s(dst + kPageData + kPageScale, a.v_data + pg * kPageData, kPageData, bar);
        bulk_g2s(dst + 2 * kPageData + kPageScale, a.v_scale + pg * kPageScale, kPageScale, bar);
      }
    } else {
      mbar_arrive(bar);
    }
  }
  ++produced;
  return true;
}

// One CTA of the persistent team attention (CTA cta of ncta; kAttnThreads threads, the dynamic
// shared memory of attn_smem_bytes() at smem).
// kOwnSelect: the producers select their rows themselves (a.block_scores set); a separate
// instance, so that the common path compiles without the selection code.
template <bool kOwnSelect>
__device__ __forceinline__ void attention_cta(const AttnArgs& a, uint8_t* smem, int cta, int ncta) {
  TeamBars* tbars = reinterpret_cast<TeamBars*>(smem + kSlotsBytes);
  float* red = reinterpret_cast<float*>(smem + kSlotsBytes + kBarsBytes);
  ItemMeta* meta = reinterpret_cast<ItemMeta*>(smem + kSlotsBytes + kBarsBytes + kRedBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, t4 = lane & 3;
  const int Hg = a.heads_per_group;
  const int NT = ncta * kTeams;
  const int rows = a.batch * a.q_len * a.groups;
  const int E = rows * kTopK;
  if (tid < kTeams) {
    TeamBars* tb = tbars + tid;
    for (int i = 0; i < kTSl; ++i) {
      mbar_init(&tb->full[i], 1);
      mbar_init(&tb->empty[i], kTW);
    }
    mbar_init(&tb->merged, kTW);
    mbar_init(&tb->freed, kTW);
  }
  fence_mbar_init();
  __syncthreads();

  // Launched as a programmatic dependent of the previous kernel on the stream (the
  // selection): the prologue above, and on the msa_decode path the consumers' first
  // queries below, run before that kernel has finished; everything that reads what it
  // writes comes after this wait.
  if (warp >= kAW) {
    grid_dependency_wait();
    grid_dependents_launch();  // the merge kernel may be scheduled as SMs free up
    // ---- producer of team `tm`: row by row over its entries, an item per entry with a
    // page (a marker for a row segment with none), then the end item
    const int tm = warp - kAW;
    const int tt = cta * kTeams + tm;
    TeamBars* tb = tbars + tm;
    uint8_t* slots = smem + static_cast<size_t>(tm) * kTSl * kSlotBytes;
    ItemMeta* my_meta = meta + tm * kTSl;
    const int x0 = range_lo(E, tt, NT), x1 = range_lo(E, tt + 1, NT);
    int produced = 0;
    bool ok = true;
    const int R_last = (x1 - 1) / kTopK;
    uint64_t* sel_cb = reinterpret_cast<uint64_t*>(smem + kSelScratchOff) + tm * 32;
    RowRaw raw = {};
    if (x0 < x1 && !kOwnSelect) raw = row_fetch(a, x0 / kTopK, lane);
    for (int R = x0 / kTopK; x0 < x1 && R <= R_last && ok; ++R) {
      int blk, page, pos;
      if (kOwnSelect) {
        select_resolve(a, R, lane, sel_cb, R * kTopK >= x0, blk, page, pos);
      } else {
        RowRaw next = {};
        if (R < R_last) next = row_fetch(a, R + 1, lane);  // in flight while row R is sent
        row_resolve(a, R, raw, lane, blk, page, pos);
        raw = next;
      }
      const int j0 = max(x0 - R * kTopK, 0), j1 = min(x1 - R * kTopK, kTopK);
      bool any = false;
      for (int j = j0; j < j1 && ok; ++j) {
        const int pj = __shfl_sync(0xffffffffu, page, j), bj = __shfl_sync(0xffffffffu, blk, j);
        if (pj < 0) continue;
        any = true;
        ok = send_item(a, produced, slots, my_meta, tb, lane, R, bj, pj, pos);
      }
      if (ok && !any) ok = send_item(a, produced, slots, my_meta, tb, lane, R, -1, -1, -1);
    }
    if (ok) ok = send_item(a, produced, slots, my_meta, tb, lane, -1, -1, -1, -1);
    if (!ok) {
      if (lane == 0) flag_error(a.err, MSA_DEVERR_TIMEOUT);
      // wait (bounded) for the copies still in flight before leaving
      for (int k = max(0, produced - kTSl); k < produced; ++k)
        mbar_wait(&tb->full[k % kTSl], (k / kTSl) & 1, a.spin_limit);
    }
    return;
  }

  // ---- consumers: team `team`, warp wt of it (one 32-key quarter of every page)
  const int team = warp / kTW, wt = warp % kTW;
  const int tt = cta * kTeams + team;
  const int x0 = range_lo(E, tt, NT), x1 = range_lo(E, tt + 1, NT);
  const int R0 = x0 / kTopK;
  uint8_t* my_slots = smem + static_cast<size_t>(team) * kTSl * kSlotBytes;
  ItemMeta* my_meta = meta + team * kTSl;
  TeamBars* tb = tbars + team;
  float* team_red = red + team * kTW * kRedFloats;

  int consumed = 0, nseg = 0;
  int cur_row = -2;
  uint32_t bq[8][2] = {};
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float o[8][4] = {};
  bool failed = false;

  auto finalize = [&](int R) -> bool {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float v = l_run[e];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      l_run[e] = v;
    }
    if (nseg > 0 && !mbar_wait_warp(&tb->freed, (nseg - 1) & 1, a.spin_limit)) return false;
    float* my_red = team_red + wt * kRedFloats;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int d0 = 16 * gq + 2 * mt;
      *reinterpret_cast<float2*>(my_red + (2 * t4) * kDim + d0) = make_float2(o[mt][0], o[mt][2]);
      *reinterpret_cast<float2*>(my_red + (2 * t4 + 1) * kDim + d0) = make_float2(o[mt][1], o[mt][3]);
    }
    if (gq == 0) {
      my_red[kHeadsMax * kDim + 2 * t4] = m_run[0];
      my_red[kHeadsMax * kDim + 2 * t4 + 1] = m_run[1];
      my_red[kHeadsMax * kDim + kHeadsMax + 2 * t4] = l_run[0];
      my_red[kHeadsMax * kDim + kHeadsMax + 2 * t4 + 1] = l_run[1];
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&tb->merged);
    if (!mbar_wait_warp(&tb->merged, nseg & 1, a.spin_limit)) return false;
    const bool whole = R * kTopK >= x0 && (R + 1) * kTopK <= x1;
    float* slot_part = whole ? nullptr : a.partial + static_cast<int64_t>(2 * tt + (R == R0 ? 0 : 1)) * kSlotFloats;
    // lane (w, h) = (lane >> 3, lane & 7): weight e^{m_w - M} of warp w's state for head h,
    // with M the heads' maximum over the team's warps, and the weighted sum of the l's
    const float* stats = team_red + kHeadsMax * kDim;
    const int lw = lane >> 3, lh = lane & 7;
    const float mw = stats[lw * kRedFloats + lh];
    float Mh = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, 8));
    Mh = fmaxf(Mh, __shfl_xor_sync(0xffffffffu, Mh, 16));
    const float fw = (mw == -INFINITY) ? 0.f : exp2f(mw - Mh);
    float den = fw * stats[lw * kRedFloats + kHeadsMax + lh];
    den += __shfl_xor_sync(0xffffffffu, den, 8);
    den += __shfl_xor_sync(0xffffffffu, den, 16);
    const int d = wt * 32 + lane;  // each warp merges 32 of the 128 dims
    for (int h = 0; h < Hg; ++h) {
      float num = 0.f;
#pragma unroll
      for (int w = 0; w < kTW; ++w) num += __shfl_sync(0xffffffffu, fw, w * 8 + h) * team_red[w * kRedFloats + h * kDim + d];
      const float M = __shfl_sync(0xffffffffu, Mh, h), dh = __shfl_sync(0xffffffffu, den, h);
      if (whole) {
        write_out(a.out, a.lse, R * Hg + h, d, num, dh, M);
      } else {
        slot_part[h * (kDim + 2) + d] = num;
        if (d == 0) {
          slot_part[h * (kDim + 2) + kDim] = M;
          slot_part[h * (kDim + 2) + kDim + 1] = dh;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&tb->freed);
    ++nseg;
    return true;
  };

  // the first row's queries load while the first pages are on their way; later rows'
  // are prefetched one row ahead (the rows of a range are consecutive)
  // (early only when the kernel before this one is the selection of the same decode step:
  // the queries were then written before that step's first kernel, which waited for them)
  uint4 qn0 = make_uint4(0u, 0u, 0u, 0u), qn1 = qn0;
  int q_row = -1;
  if (!a.q_early) grid_dependency_wait();
  if (x0 < x1) {
    load_q_raw(a.q, a.heads_per_group, R0, gq, t4, qn0, qn1);
    q_row = R0;
  }
  if (a.q_early) grid_dependency_wait();
  grid_dependents_launch();
  while (true) {
    const int slot = consumed % kTSl;
    if (!mbar_wait_warp(&tb->full[slot], (consumed / kTSl) & 1, a.spin_limit)) {
      failed = true;
      break;
    }
    const int row = my_meta[slot].row;
    const int blk = my_meta[slot].blk;
    const int page = my_meta[slot].page;
    const int pos = my_meta[slot].pos;
    if (row != cur_row) {
      if (cur_row >= 0 && !finalize(cur_row)) {
        failed = true;
        break;
      }
      if (row >= 0) {
        if (q_row != row) load_q_raw(a.q, a.heads_per_group, row, gq, t4, qn0, qn1);
        q_fragments(qn0, qn1, bq);
        if ((row + 1) * kTopK < x1) {
          load_q_raw(a.q, a.heads_per_group, row + 1, gq, t4, qn0, qn1);
          q_row = row + 1;
        }
        m_run[0] = m_run[1] = -INFINITY;
        l_run[0] = l_run[1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      }
      cur_row = row;
    }
    if (page >= 0)
      attend_quarter(my_slots + slot * kSlotBytes, wt, blk, pos / kBlock, pos, a.scale_log2, gq, t4, bq, m_run, l_run,
                     o);
    __syncwarp();
    if (lane == 0) mbar_arrive(&tb->empty[slot]);
    ++consumed;
    if (row < 0) break;
  }
  if (failed && lane == 0) flag_error(a.err, MSA_DEVERR_TIMEOUT);
}

// Rows cut by team-range boundaries: combine the partial states the teams left.  One CTA per
// boundary (the first boundary inside a row owns the row), or, with fewer rows than
// boundaries, one per row (merge_kernel); its first warp lists the row's partial slots in
// shared memory (arithmetic only, so it runs before the wait on the attention kernel), then
// one thread per (head, pair of dims) loads the slots' states eight at a time (a row has at
// most 16 slots, one per selection entry) and combines them; two CTAs fit an SM, so the CTAs
// with no row to merge clear out in one wave.  With no more rows to merge than SMs, all 16 go
// in one round (more registers, one CTA an SM: still a single wave).
constexpr int kMergeThreads = kHeadsMax * kDim / 2;

// The merge of the row cut by range boundary k (between team ranges k-1 and k) of NT, if k is
// that row's first cut; kMergeThreads threads, scratch in shared memory (s_slot[16], s_n, s_row).
// Ends with every thread past the CTA barrier, so that a CTA can take several boundaries in turn.
template <int kBatch>
__device__ __forceinline__ void merge_boundary(const AttnArgs& a, int NT, int k, int* s_slot, int* s_n, int* s_row) {
  const int tid = threadIdx.x, lane = tid & 31;
  __syncthreads();  // the scratch of a previous boundary is no longer read
  if (tid < 32) {
    const int E = a.batch * a.q_len * a.groups * kTopK;
    const int xb = range_lo(E, k, NT);
    int R = -1, ca = 0, cb = -1;
    // inside a row, and no earlier boundary inside the same row
    if (xb % kTopK != 0 && xb < E && range_lo(E, k - 1, NT) <= (xb / kTopK) * kTopK) {
      R = xb / kTopK;
      ca = owner_of(E, R * kTopK, NT);
      cb = owner_of(E, R * kTopK + kTopK - 1, NT);
    }
    int n = 0;
    for (int c0 = ca; c0 <= cb; c0 += 32) {  // the non-empty ranges among ca..cb, in order
      const int c = c0 + lane;
      int slot = -1;
      if (c <= cb) {
        const int lo = range_lo(E, c, NT), hi = range_lo(E, c + 1, NT);
        if (lo < hi) slot = 2 * c + ((lo / kTopK) == R ? 0 : 1);
      }
      const unsigned m = __ballot_sync(0xffffffffu, slot >= 0);
      const int idx = n + __popc(m & ((1u << lane) - 1u));
      if (slot >= 0 && idx < kTopK) s_slot[idx] = slot;
      n += __popc(m);
    }
    if (lane == 0) {
      *s_n = min(n, kTopK);
      *s_row = R;
    }
  }
  __syncthreads();
  const int R = *s_row, n = *s_n;
  const int h = tid / (kDim / 2), d = 2 * (tid % (kDim / 2));
  if (R < 0 || h >= a.heads_per_group) return;
  grid_dependency_wait();  // the attention kernel's partial states
  // the slots' states are loaded kBatch (8 or 16) at a time before any of them is used (one
  // round of loads in flight per batch, not one per slot), then folded into the running sums
  float M = -INFINITY, num0 = 0.f, num1 = 0.f, den = 0.f;
  for (int i0 = 0; i0 < n; i0 += kBatch) {
    float ms[kBatch], ls[kBatch];
    float2 os[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      ms[i] = -INFINITY;
      ls[i] = 0.f;
      os[i] = make_float2(0.f, 0.f);
      if (i0 + i < n) {
        const float* part = a.partial + static_cast<int64_t>(s_slot[i0 + i]) * kSlotFloats + h * (kDim + 2);
        ms[i] = __ldcg(part + kDim);
        ls[i] = __ldcg(part + kDim + 1);
        os[i] = __ldcg(reinterpret_cast<const float2*>(part + d));
      }
    }
    float Mb = M;
#pragma unroll
    for (int i = 0; i < kBatch; ++i) Mb = fmaxf(Mb, ms[i]);
    if (Mb == -INFINITY) continue;
    const float fo = (M == -INFINITY) ? 0.f : exp2f(M - Mb);  // rescale the sums so far
    num0 *= fo;
    num1 *= fo;
    den *= fo;
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      if (ms[i] == -INFINITY) continue;
      const float f = exp2f(ms[i] - Mb);
      num0 += f * os[i].x;
      num1 += f * os[i].y;
      den += f * ls[i];
    }
    M = Mb;
  }
  const int head_row = R * a.heads_per_group + h;
  write_out(a.out, a.lse, head_row, d, num0, den, M);
  write_out(a.out, a.lse, head_row, d + 1, num1, den, M);
}

}  // namespace msa
