// Device building blocks of the exact sparse GQA attention over NVFP4 K/V pages, used by the
// query-major team kernel (attention_team.cuh, attention.cu).
//
// Every query head of a KV group attends exactly to the selected blocks of that group
// ("vLLM liefert Day-0-Unterstützung für MiniMax-M3.1-Flash", §MSA-Grundlagen, Fig. 1), with
// an online softmax in the exp2 domain; partial states (o, m, l) of split work combine as
// o = sum e^{m_s-M} o_s / sum e^{m_s-M} l_s ("MiniMax M3 x vLLM：百万 token 多模态推理的
// Day-0 部署", §MiniMax 稀疏注意力后端).  One warp handles a 32-key quarter of a 128-key page:
// S^T = K Q^T on mma.sync m16n8k16 (keys as M, the <= 8 heads of the group as N), then
// O^T += V^T P^T with P packed to f16 and transposed in registers (movmatrix) and V^T built
// from two keys' bytes by a nibble transpose.  K and V are dequantised exactly (cvt
// e2m1x2 -> f16x2 times the f16 block scale).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "msa_device.cuh"
#include "msa_kernels.h"

namespace msa {

constexpr int kSlotBytes = 2 * (kPageData + kPageScale);  // one page slot: K data | K scales | V data | V scales
constexpr int kHeadsMax = 8;
constexpr int kRedFloats = kHeadsMax * kDim + 2 * kHeadsMax;   // one warp's o[8][128], m[8], l[8]
constexpr int kSlotFloats = kHeadsMax * (kDim + 2);             // one partial slot: [8][o 128, m, l]
constexpr float kLn2 = 0.69314718055994530942f;

// 2^x by the hardware approximation (ex2.approx, relative error about 2^-22), subnormal
// results flushed to zero: softmax weights below 2^-126 of the row maximum count as 0.
__device__ __forceinline__ float exp2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The raw FP8 queries of head row gq of a group's row (lane: 32 bytes of dims 32 t4 ..).
__device__ __forceinline__ void load_q_raw(const uint8_t* q, int heads_per_group, int row, int gq, int t4, uint4& q0,
                                           uint4& q1) {
  if (gq < heads_per_group) {
    const uint4* src = reinterpret_cast<const uint4*>(
        q + (static_cast<int64_t>(row) * heads_per_group + gq) * kDim + 32 * t4);
    q0 = __ldg(src);
    q1 = __ldg(src + 1);
  } else {
    q0 = q1 = make_uint4(0u, 0u, 0u, 0u);
  }
}

__device__ __forceinline__ void q_fragments(const uint4& q0, const uint4& q1, uint32_t (&bq)[8][2]) {
  const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    bq[s][0] = e4m3x2_to_f16x2(w[s]);
    bq[s][1] = e4m3x2_to_f16x2(w[s] >> 16);
  }
}

// 32 keys of one KV head into the warp's online-softmax state.  K rows (64 packed bytes each),
// K scales (8 per row), V rows and V scales are read at row rbase + i of kd / ks / vd / vs,
// i = 0..31; key i is token key0 + i of the sequence.  recent: the keys' block is the query's
// own block (only then can a key lie past the query position pos).
__device__ __forceinline__ void attend_rows32(const uint8_t* kd, const uint8_t* ks, const uint8_t* vd,
                                              const uint8_t* vs, int rbase, int key0, bool recent, int pos,
                                              float scale_log2, int gq, int t4, const uint32_t (&bq)[8][2],
                                              float (&m_run)[2], float (&l_run)[2], float (&o)[8][4]) {
  // ---- S^T = K Q^T for 32 keys (two 16-key tiles), raw (unscaled) logits
  float x[2][4];
#pragma unroll
  for (int mq = 0; mq < 2; ++mq) {
    // tile row i holds key pi(i) = i ^ ((i >> 1) & 1) of the 16 (rows 0-7 and 8-15 alike): the
    // two rows an 8-lane phase of the K loads reads then differ in parity (different bank
    // halves of their 64-byte rows: no conflict), and each PV load reads two rows of each
    // parity (its 2-way minimum)
    const int i0 = mq * 16 + (gq ^ ((gq >> 1) & 1));
    const int r0 = rbase + i0, r1 = r0 + 8;
    const uint4 d0 = lds128(kd + r0 * kRowBytes + 16 * t4);
    const uint4 d1 = lds128(kd + r1 * kRowBytes + 16 * t4);
    // the lane's two block scales of each row, as f16 pairs (s, s)
    const uint32_t f0 = e4m3x2_to_f16x2(lds16(ks + r0 * kRowScales + 2 * t4));
    const uint32_t f1 = e4m3x2_to_f16x2(lds16(ks + r1 * kRowScales + 2 * t4));
    const uint32_t sc0[2] = {__byte_perm(f0, 0, 0x1010), __byte_perm(f0, 0, 0x3232)};
    const uint32_t sc1[2] = {__byte_perm(f1, 0, 0x1010), __byte_perm(f1, 0, 0x3232)};
    const uint32_t w0[4] = {d0.x, d0.y, d0.z, d0.w};
    const uint32_t w1[4] = {d1.x, d1.y, d1.z, d1.w};
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t x0, x1, x2, x3, y0, y1, y2, y3;
      e2m1x8_to_f16x2(w0[w], x0, x1, x2, x3);
      e2m1x8_to_f16x2(w1[w], y0, y1, y2, y3);
      const uint32_t sa = sc0[w >> 1], sb = sc1[w >> 1];
      x0 = hmul2(x0, sa); x1 = hmul2(x1, sa); x2 = hmul2(x2, sa); x3 = hmul2(x3, sa);
      y0 = hmul2(y0, sb); y1 = hmul2(y1, sb); y2 = hmul2(y2, sb); y3 = hmul2(y3, sb);
      mma_f16_16816(acc, x0, y0, x1, y1, bq[2 * w][0], bq[2 * w][1]);
      mma_f16_16816(acc, x2, y2, x3, y3, bq[2 * w + 1][0], bq[2 * w + 1][1]);
    }
    const int j0 = key0 + i0, j1 = j0 + 8;
#pragma unroll
    for (int e = 0; e < 4; ++e) x[mq][e] = acc[e];
    if (recent) {
      if (j0 > pos) x[mq][0] = x[mq][1] = -INFINITY;
      if (j1 > pos) x[mq][2] = x[mq][3] = -INFINITY;
    }
  }

  // ---- online softmax per head column (2*t4 + e), in the exp2 domain: logit * scale_log2
  // (the scale is positive, so the maximum of the raw logits scales to the running maximum)
  float p[2][4], alpha[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    float mx = fmaxf(fmaxf(x[0][e], x[0][e + 2]), fmaxf(x[1][e], x[1][e + 2]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const float m_new = fmaxf(m_run[e], mx * scale_log2);
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    alpha[e] = exp2_ftz(m_run[e] - m_use);
    m_run[e] = m_new;
    float sum = 0.f;
#pragma unroll
    for (int mq = 0; mq < 2; ++mq) {
      p[mq][e] = exp2_ftz(fmaf(x[mq][e], scale_log2, -m_use));
      p[mq][e + 2] = exp2_ftz(fmaf(x[mq][e + 2], scale_log2, -m_use));
      sum += p[mq][e] + p[mq][e + 2];
    }
    l_run[e] = l_run[e] * alpha[e] + sum;
  }
  // rescale the output only when some head's running maximum moved (warp-uniform test)
  if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      o[mt][0] *= alpha[0];
      o[mt][2] *= alpha[0];
      o[mt][1] *= alpha[1];
      o[mt][3] *= alpha[1];
    }
  }

  // ---- O^T += V^T P^T, one 16-key k-step per QK tile
#pragma unroll
  for (int mq = 0; mq < 2; ++mq) {
    const uint32_t b0 = movmatrix_trans(pack_f16x2(p[mq][0], p[mq][1]));
    const uint32_t b1 = movmatrix_trans(pack_f16x2(p[mq][2], p[mq][3]));
    // k-indices 2t4, 2t4+1, 2t4+8, 2t4+9 are keys pi(.) = ka, kb, ka + 8, kb + 8 of the tile
    const int ka = rbase + mq * 16 + ((2 * t4) ^ (t4 & 1)), kb = rbase + mq * 16 + ((2 * t4 + 1) ^ (t4 & 1));
    const uint2 va = lds64(vd + ka * kRowBytes + 8 * gq);
    const uint2 vb = lds64(vd + kb * kRowBytes + 8 * gq);
    const uint2 vc = lds64(vd + (ka + 8) * kRowBytes + 8 * gq);
    const uint2 ve = lds64(vd + (kb + 8) * kRowBytes + 8 * gq);
    const uint32_t sab = e4m3x2_to_f16x2(lds8(vs + ka * kRowScales + gq) | (lds8(vs + kb * kRowScales + gq) << 8));
    const uint32_t scd = e4m3x2_to_f16x2(lds8(vs + (ka + 8) * kRowScales + gq) |
                                         (lds8(vs + (kb + 8) * kRowScales + gq) << 8));
#pragma unroll
    for (int hw = 0; hw < 2; ++hw) {
      const uint32_t wa = hw ? va.y : va.x, wb = hw ? vb.y : vb.x;
      const uint32_t wc = hw ? vc.y : vc.x, we = hw ? ve.y : ve.x;
      // byte i of lo*: low nibbles of (key a, key b); of hi*: their high nibbles
      const uint32_t lo_ab = (wa & 0x0F0F0F0Fu) | ((wb & 0x0F0F0F0Fu) << 4);
      const uint32_t hi_ab = ((wa >> 4) & 0x0F0F0F0Fu) | (wb & 0xF0F0F0F0u);
      const uint32_t lo_ce = (wc & 0x0F0F0F0Fu) | ((we & 0x0F0F0F0Fu) << 4);
      const uint32_t hi_ce = ((wc >> 4) & 0x0F0F0F0Fu) | (we & 0xF0F0F0F0u);
      uint32_t la[4], ha[4], lc[4], hc[4];
      e2m1x8_to_f16x2(lo_ab, la[0], la[1], la[2], la[3]);
      e2m1x8_to_f16x2(hi_ab, ha[0], ha[1], ha[2], ha[3]);
      e2m1x8_to_f16x2(lo_ce, lc[0], lc[1], lc[2], lc[3]);
      e2m1x8_to_f16x2(hi_ce, hc[0], hc[1], hc[2], hc[3]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int mt = hw * 4 + i;  // output dims 16*gq + 2*mt (+1)
        mma_f16_16816(o[mt], hmul2(la[i], sab), hmul2(ha[i], sab), hmul2(lc[i], scd), hmul2(hc[i], scd), b0, b1);
      }
    }
  }
}

// One 32-key quarter (qk) of one page (128 keys of one KV head: K data | K scales | V data |
// V scales at kd) into the warp's state; n is the page's logical block, r the query's.
__device__ __forceinline__ void attend_quarter(const uint8_t* kd, int qk, int n, int r, int pos, float scale_log2,
                                               int gq, int t4, const uint32_t (&bq)[8][2], float (&m_run)[2],
                                               float (&l_run)[2], float (&o)[8][4]) {
  attend_rows32(kd, kd + kPageData, kd + kPageData + kPageScale, kd + 2 * kPageData + kPageScale, qk * 32,
                n * kBlock + qk * 32, n == r, pos, scale_log2, gq, t4, bq, m_run, l_run, o);
}

// A row's selection in two steps, so that a row's loads can be in flight while the row before
// it is being streamed: row_fetch issues the loads that depend only on the row
// (its selection, lane j < 16: block id of entry j and, on the decode step, its page; the
// sequence length), row_resolve then checks them and, unless the page came with the block
// id, looks it up in the block table (-1: empty, past the recent block, or a bad block-table
// entry).
struct RowRaw {
  int blk, page, L;
};

__device__ __forceinline__ RowRaw row_fetch(const AttnArgs& a, int R, int lane) {
  RowRaw raw;
  const int64_t e = static_cast<int64_t>(R) * kTopK + lane;
  raw.blk = lane < kTopK ? a.selection[e] : -1;
  raw.page = (lane < kTopK && a.sel_pages != nullptr) ? a.sel_pages[e] : -1;
  raw.L = a.seq_lens[static_cast<unsigned>(R) / static_cast<unsigned>(a.q_len * a.groups)];
  return raw;
}

__device__ __forceinline__ void row_resolve(const AttnArgs& a, int R, const RowRaw& raw, int lane, int& blk,
                                            int& page, int& pos) {
  const unsigned TG = static_cast<unsigned>(a.q_len * a.groups);
  const int b = static_cast<int>(static_cast<unsigned>(R) / TG);
  const int t = static_cast<int>((static_cast<unsigned>(R) - static_cast<unsigned>(b) * TG) /
                                 static_cast<unsigned>(a.groups));
  const int L = raw.L;
  const bool ok = L > 0 && L >= a.q_len && L <= static_cast<int64_t>(a.max_blocks) * kBlock;
  pos = L - a.q_len + t;
  const int r = ok ? pos / kBlock : -1;
  blk = ok ? raw.blk : -1;
  // the table lookup only needs an in-range block id; its validity comes from ok and r (the
  // decode step's selection kernel has looked the pages up already: the same table entries)
  int p = -1;
  if (blk >= 0 && blk < a.max_blocks)
    p = a.sel_pages != nullptr ? raw.page : a.block_table[static_cast<int64_t>(b) * a.max_blocks + blk];
  page = -1;
  if (blk >= 0 && blk <= r) {
    if (p >= 0 && p < a.num_pages)
      page = p;
    else
      flag_error(a.err, MSA_DEVERR_BAD_PAGE);
  }
}

// Output of one (head row, dim) from its merged state: num / den rounded to bf16 (0 for a row
// with nothing to attend to), and at dim 0 the natural-log lse (-inf for such a row).
__device__ __forceinline__ void write_out(uint16_t* out, float* lse, int head_row, int d, float num, float den,
                                          float M) {
  const float v = den > 0.f ? num / den : 0.f;
  out[static_cast<int64_t>(head_row) * kDim + d] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  if (d == 0 && lse != nullptr) lse[head_row] = den > 0.f ? (M + log2f(den)) * kLn2 : -INFINITY;
}

}  // namespace msa
