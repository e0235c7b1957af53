// Stage 3 of MSA decode: exact sparse GQA attention over the selected blocks, split-K
// over the blocks with an online-softmax merge.
//
// Every query head of a KV group attends exactly, and only, to the selected blocks of that
// group ("vLLM liefert Day-0-Unterstützung für MiniMax-M3.1-Flash", §MSA-Grundlagen, Fig. 1);
// the result equals dense attention restricted to the selected set, computed with an
// online softmax ("MiniMax M3 x vLLM：百万 token 多模态推理的 Day-0 部署", §Prefill 执行
// step 4); decode consumes the selected pages and merges the partial outputs of split
// work (same page, §MiniMax 稀疏注意力后端 and §Decode 执行).
//
// Design (GB300):
//   * grid (split, group, sequence x query token); each CTA stages its <= 4 selected
//     pages of K and V (18 KB each: E2M1 bytes + E4M3 scales of one KV head) with bulk
//     async copies, 4 warps each take one 32-key quarter of every page;
//   * QK runs transposed, S^T = K Q^T on mma.sync m16n8k16 with keys as M and the (up to
//     8) heads of the group as N, so the heads fill the N=8 tile with no padding; K is
//     dequantised straight into A registers (cvt e2m1x2 -> f16x2, times the f16 block scale:
//     exact), the FP8 queries widen exactly to f16;
//   * the probabilities are packed to f16 and transposed in registers (movmatrix) into the
//     B operand of O^T = V^T P^T, whose A operand is V^T built from two keys' bytes with a
//     nibble transpose (LOP3), again exact -- no shared-memory round trip for either
//     operand;
//   * softmax in the exp2 domain with the scale folded into one multiply; a split's
//     partial state (o, m, l) is merged across warps in shared memory and across splits
//     by merge_kernel (o = sum e^{m_s-M} o_s / sum e^{m_s-M} l_s).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "msa_device.cuh"
#include "msa_kernels.h"

namespace msa {

constexpr int kAttnWarps = 4;
constexpr int kAttnSlots = 4;
constexpr int kSlotBytes = 2 * (kPageData + kPageScale);  // K data | K scales | V data | V scales
constexpr int kPartialStride = kDim + 2;                  // o[128], m (log2 units), l
constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ void store_out(const AttnArgs& a, int64_t head_row, int d, float num, float den,
                                          float M) {
  const float v = den > 0.f ? num / den : 0.f;
  a.out[head_row * kDim + d] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  if (d == 0 && a.lse != nullptr) a.lse[head_row] = den > 0.f ? (M + log2f(den)) * kLn2 : -INFINITY;
}

__global__ void __launch_bounds__(kAttnWarps * 32) attention_kernel(const AttnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kAttnSlots * kSlotBytes);
  __shared__ int s_blk[kTopK], s_page[kTopK], s_nblk;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, t4 = lane & 3;
  const int split = blockIdx.x, grp = blockIdx.y;
  const int T = a.q_len, G = a.groups, Hg = a.heads_per_group, H = G * Hg;
  const int b = blockIdx.z / T, t = blockIdx.z % T;
  const int64_t head_row0 = (static_cast<int64_t>(b) * T + t) * H + grp * Hg;
  const int L = a.seq_lens[b];
  const bool seq_ok = L > 0 && L >= T && L <= static_cast<int64_t>(a.max_blocks) * kBlock;
  const int pos = L - T + t;
  const int r = seq_ok ? pos / kBlock : -1;
  const int bps = kTopK / a.splits;

  if (tid == 0) {
    int cnt = 0;
    if (seq_ok) {
      const int32_t* sel = a.selection + ((static_cast<int64_t>(b) * T + t) * G + grp) * kTopK + split * bps;
      for (int i = 0; i < bps; ++i) {
        const int n = sel[i];
        if (n < 0 || n > r) continue;
        const int page = a.block_table[static_cast<int64_t>(b) * a.max_blocks + n];
        if (page < 0 || page >= a.num_pages) {
          flag_error(a.err, MSA_DEVERR_BAD_PAGE);
          continue;
        }
        s_blk[cnt] = n;
        s_page[cnt] = page;
        ++cnt;
      }
    }
    s_nblk = cnt;
    for (int i = 0; i < kAttnSlots; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int nblk = s_nblk;

  // B fragments of QK (k = dim, n = head): head gq, dims 32*t4 + 4s .. +3 for k-step s
  uint32_t bq[8][2];
  if (gq < Hg && seq_ok) {
    const uint4* src = reinterpret_cast<const uint4*>(a.q + (head_row0 + gq) * kDim + 32 * t4);
    const uint4 q0 = __ldg(src), q1 = __ldg(src + 1);
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      bq[s][0] = e4m3x2_to_f16x2(w[s]);
      bq[s][1] = e4m3x2_to_f16x2(w[s] >> 16);
    }
  } else {
#pragma unroll
    for (int s = 0; s < 8; ++s) bq[s][0] = bq[s][1] = 0u;
  }

  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

  for (int base = 0, round = 0; base < nblk; base += kAttnSlots, ++round) {
    const int nr = min(kAttnSlots, nblk - base);
    if (tid == 0) {
      for (int i = 0; i < nr; ++i) {
        uint8_t* slot = smem + i * kSlotBytes;
        const int64_t pg = static_cast<int64_t>(s_page[base + i]) * G + grp;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&bars[i], kSlotBytes);
        bulk_g2s(slot, a.k_data + pg * kPageData, kPageData, &bars[i]);
        bulk_g2s(slot + kPageData, a.k_scale + pg * kPageScale, kPageScale, &bars[i]);
        bulk_g2s(slot + kPageData + kPageScale, a.v_data + pg * kPageData, kPageData, &bars[i]);
        bulk_g2s(slot + 2 * kPageData + kPageScale, a.v_scale + pg * kPageScale, kPageScale, &bars[i]);
      }
    }
    for (int i = 0; i < nr; ++i) {
      if (!mbar_wait_warp(&bars[i], round & 1)) {
        if (lane == 0) flag_error(a.err, MSA_DEVERR_TIMEOUT);
        continue;
      }
      const uint8_t* kd = smem + i * kSlotBytes;
      const uint8_t* ks = kd + kPageData;
      const uint8_t* vd = ks + kPageScale;
      const uint8_t* vs = vd + kPageData;
      const int n = s_blk[base + i];
      const bool recent = (n == r);

      // ---- S^T = K Q^T for this warp's 32 keys (two 16-key tiles)
      float x[2][4];
#pragma unroll
      for (int mq = 0; mq < 2; ++mq) {
        const int r0 = warp * 32 + mq * 16 + gq, r1 = r0 + 8;
        const uint4 d0 = lds128(kd + r0 * kRowBytes + 16 * t4);
        const uint4 d1 = lds128(kd + r1 * kRowBytes + 16 * t4);
        const uint32_t s0 = lds16(ks + r0 * kRowScales + 2 * t4);
        const uint32_t s1 = lds16(ks + r1 * kRowScales + 2 * t4);
        const uint32_t sc0[2] = {e4m3_bcast_f16x2(s0, 0), e4m3_bcast_f16x2(s0, 1)};
        const uint32_t sc1[2] = {e4m3_bcast_f16x2(s1, 0), e4m3_bcast_f16x2(s1, 1)};
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
        const int j0 = n * kBlock + r0, j1 = j0 + 8;
#pragma unroll
        for (int e = 0; e < 4; ++e) x[mq][e] = acc[e] * a.scale_log2;
        if (recent) {
          if (j0 > pos) x[mq][0] = x[mq][1] = -INFINITY;
          if (j1 > pos) x[mq][2] = x[mq][3] = -INFINITY;
        }
      }

      // ---- online softmax per head column (2*t4 + e)
      float p[2][4];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float mx = fmaxf(fmaxf(x[0][e], x[0][e + 2]), fmaxf(x[1][e], x[1][e + 2]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float m_new = fmaxf(m_run[e], mx);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = exp2f(m_run[e] - m_use);
        m_run[e] = m_new;
        float sum = 0.f;
#pragma unroll
        for (int mq = 0; mq < 2; ++mq) {
          p[mq][e] = exp2f(x[mq][e] - m_use);
          p[mq][e + 2] = exp2f(x[mq][e + 2] - m_use);
          sum += p[mq][e] + p[mq][e + 2];
        }
        l_run[e] = l_run[e] * alpha + sum;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          o[mt][e] *= alpha;
          o[mt][e + 2] *= alpha;
        }
      }

      // ---- O^T += V^T P^T, one 16-key k-step per QK tile
#pragma unroll
      for (int mq = 0; mq < 2; ++mq) {
        const uint32_t b0 = movmatrix_trans(pack_f16x2(p[mq][0], p[mq][1]));
        const uint32_t b1 = movmatrix_trans(pack_f16x2(p[mq][2], p[mq][3]));
        const int ka = warp * 32 + mq * 16 + 2 * t4;  // keys ka, ka+1, ka+8, ka+9
        const uint2 va = lds64(vd + ka * kRowBytes + 8 * gq);
        const uint2 vb = lds64(vd + (ka + 1) * kRowBytes + 8 * gq);
        const uint2 vc = lds64(vd + (ka + 8) * kRowBytes + 8 * gq);
        const uint2 ve = lds64(vd + (ka + 9) * kRowBytes + 8 * gq);
        const uint32_t sab = e4m3x2_to_f16x2(lds8(vs + ka * kRowScales + gq) |
                                             (lds8(vs + (ka + 1) * kRowScales + gq) << 8));
        const uint32_t scd = e4m3x2_to_f16x2(lds8(vs + (ka + 8) * kRowScales + gq) |
                                             (lds8(vs + (ka + 9) * kRowScales + gq) << 8));
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
            mma_f16_16816(o[mt], hmul2(la[i], sab), hmul2(ha[i], sab), hmul2(lc[i], scd), hmul2(hc[i], scd), b0,
                          b1);
          }
        }
      }
    }
    __syncthreads();  // every warp is done with the slots before they are refilled / reused
  }

  // ---- merge the 4 warps' states in shared memory (aliases the page slots)
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    float v = l_run[e];
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    v += __shfl_xor_sync(0xffffffffu, v, 16);
    l_run[e] = v;
  }
  float* red_o = reinterpret_cast<float*>(smem);            // [warp][head 8][dim 128]
  float* red_m = red_o + kAttnWarps * 8 * kDim;             // [warp][8]
  float* red_l = red_m + kAttnWarps * 8;                    // [warp][8]
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int d0 = 16 * gq + 2 * mt;
    float* base = red_o + warp * 8 * kDim;
    base[(2 * t4) * kDim + d0] = o[mt][0];
    base[(2 * t4 + 1) * kDim + d0] = o[mt][1];
    base[(2 * t4) * kDim + d0 + 1] = o[mt][2];
    base[(2 * t4 + 1) * kDim + d0 + 1] = o[mt][3];
  }
  if (gq == 0) {
    red_m[warp * 8 + 2 * t4] = m_run[0];
    red_m[warp * 8 + 2 * t4 + 1] = m_run[1];
    red_l[warp * 8 + 2 * t4] = l_run[0];
    red_l[warp * 8 + 2 * t4 + 1] = l_run[1];
  }
  __syncthreads();
  const int d = tid;  // 128 threads = 128 dims
  for (int h = 0; h < Hg; ++h) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, red_m[w * 8 + h]);
    float num = 0.f, den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w) {
        const float mw = red_m[w * 8 + h];
        const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
        num += f * red_o[(w * 8 + h) * kDim + d];
        den += f * red_l[w * 8 + h];
      }
    }
    const int64_t hr = head_row0 + h;
    if (a.splits == 1) {
      store_out(a, hr, d, num, den, M);
    } else {
      float* part = a.partial + (hr * a.splits + split) * kPartialStride;
      part[d] = num;
      if (d == 0) {
        part[kDim] = M;
        part[kDim + 1] = den;
      }
    }
  }
}

// Combine the splits of one head row: 128 threads, one per dim.
__global__ void __launch_bounds__(kDim) merge_kernel(const AttnArgs a) {
  const int64_t hr = blockIdx.x;
  const int d = threadIdx.x;
  const float* part = a.partial + hr * a.splits * kPartialStride;
  float M = -INFINITY;
  for (int s = 0; s < a.splits; ++s) M = fmaxf(M, part[s * kPartialStride + kDim]);
  float num = 0.f, den = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < a.splits; ++s) {
      const float ms = part[s * kPartialStride + kDim];
      const float f = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
      num += f * part[s * kPartialStride + d];
      den += f * part[s * kPartialStride + kDim + 1];
    }
  }
  store_out(a, hr, d, num, den, M);
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t s) {
  const int64_t bt = static_cast<int64_t>(a.batch) * a.q_len;
  if (bt == 0) return cudaSuccess;
  const size_t smem = static_cast<size_t>(kAttnSlots) * kSlotBytes + kAttnSlots * sizeof(uint64_t);
  cudaError_t e = cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(a.splits, a.groups, static_cast<unsigned>(bt));
  attention_kernel<<<grid, kAttnWarps * 32, smem, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.splits == 1) return e;
  merge_kernel<<<static_cast<unsigned>(bt * a.groups * a.heads_per_group), kDim, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace msa
