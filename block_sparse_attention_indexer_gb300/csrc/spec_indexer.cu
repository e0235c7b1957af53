// Stage 1 for a few query tokens per sequence (speculative decode: 8 < T x G < 64 rows): the
// indexer on the tcgen05 tensor cores, keys as M.
//
// The scores are S[row][n] = max over the visible keys j of block n of q_row . k_j (row =
// (token, group); "MiniMax M3 x vLLM：百万 token 多模态推理的 Day-0 部署", §Decode Kernel 中的投机解码
// flattens the draft tokens of a request, each with its own causal position, and §Prefill 执行
// step 2 gives the block pooling).  With T x G = 32 rows the product per 128-key page is
// [128 keys x 128] . [128 x 32 rows]: too narrow for the query rows as M, so the keys are M and
// the rows are N (= rows rounded up to 16):
//   * a CTA owns one sequence and a range of key blocks (sized at launch so that the grid is
//     one round of two CTAs per SM); warp 8 streams the raw NVFP4 pages (6 stages): the E2M1
//     rows with a 2-D tensor copy that lands them 64-byte swizzled, the scales with a bulk
//     copy; warps 4-7 dequantise each page exactly, one key row per thread, in registers (cvt
//     e2m1x2 -> f16x2 times the f16 scale, the row's eight scales converted once; the swizzle
//     makes the eight lanes of a shared-memory phase read eight different bank groups) and
//     store the row with tcgen05.st straight into tensor memory as the MMA's A operand (2
//     stages: no shared-memory round trip for the keys); warps 0-3 convert the sequence's query
//     rows once (FP8 -> f16, the B operand in shared memory), and one thread of warp 9 issues
//     tcgen05.mma (A from TMEM: M 128 keys x N rows x K 16, eight per page) into one of two
//     TMEM accumulators;
//   * the epilogue warps (TMEM lane quarter = warp) load their 32 keys' scores 16 rows at a
//     time; the causal mask is applied only on pages holding a key some row must not see.
//     Max pooling reduces each row over the warp's keys with one warp-wide f32 max
//     (redux.sync), stages the 16 maxima so that lane j holds row j, and combines the four
//     warps with integer atomics on an order-preserving encoding, so the warps never wait on
//     each other.  Log-sum-exp pooling reduces with a butterfly that transposes as it goes
//     (31 shuffles leave lane c with row c over the warp's keys), sums e^{s - max} the same
//     way and combines through shared memory;
//   * 10 warps, ~94 KB of shared memory and 256 TMEM columns: two CTAs share an SM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "msa_device.cuh"
#include "msa_kernels.h"
#include "umma.cuh"

namespace msa {

constexpr int kSpKbMax = 64;       // key blocks per CTA at most (the launch sizes the ranges)
constexpr int kSpRawSt = 6;        // raw page stages (shared memory)
constexpr int kSpSt = 2;           // f16 key stages (TMEM, 64 columns each)
constexpr int kSpDeqWarps = 4;     // dequantisers (warps 4-7)
constexpr int kSpCopyWarp = 8, kSpMmaWarp = 9;
constexpr int kSpWarps = 10;
constexpr int kSpMaxN = 64;        // query rows (token x group) per sequence, rounded up to 16
constexpr int kSpRaw = kPageData + kPageScale;
constexpr uint32_t kSpACols = kDim / 2;                 // a key row of 128 f16 in TMEM: 64 columns
constexpr uint32_t kSpDCol = kSpSt * kSpACols;          // accumulators after the key stages
constexpr uint32_t kSpTmemCols = 256;                   // 2 x 64 (keys) + 2 x 64 (accumulators)

struct SpShared {
  uint64_t raw_full[kSpRawSt], raw_empty[kSpRawSt], k_full[kSpSt], k_empty[kSpSt], acc_full[2], acc_empty[2];
  uint64_t q_ready;
  uint32_t tmem_base;
  int32_t pages[kSpKbMax];
  float red[2][4][kSpMaxN];   // per accumulator stage: each epilogue warp's per-row maxima
  float red2[2][4][kSpMaxN];  // the same for the log-sum-exp sums
  float sbuf[kSpMaxN][kSpKbMax + 1];
  alignas(16) float wmax[4][16];  // max pooling: each epilogue warp's 16 column maxima of a chunk
};

// query tile | raw pages | shared
// (the 64-byte swizzle of the raw pages is a function of the shared address: stages on 1 KB)
static_assert((2 * kSpMaxN * 128) % 1024 == 0 && kSpRaw % 1024 == 0, "raw page stages must stay 1 KB aligned");
constexpr size_t kSpSmem = 1024 + 2 * kSpMaxN * 128 + kSpRawSt * static_cast<size_t>(kSpRaw) + sizeof(SpShared);

// 64 consecutive 32-bit columns of the warp's TMEM lane quarter, one row per thread
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&v)[64]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,"
      "%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31]), "r"(v[32]), "r"(v[33]), "r"(v[34]), "r"(v[35]), "r"(v[36]),
      "r"(v[37]), "r"(v[38]), "r"(v[39]), "r"(v[40]), "r"(v[41]), "r"(v[42]), "r"(v[43]), "r"(v[44]), "r"(v[45]),
      "r"(v[46]), "r"(v[47]), "r"(v[48]), "r"(v[49]), "r"(v[50]), "r"(v[51]), "r"(v[52]), "r"(v[53]), "r"(v[54]),
      "r"(v[55]), "r"(v[56]), "r"(v[57]), "r"(v[58]), "r"(v[59]), "r"(v[60]), "r"(v[61]), "r"(v[62]), "r"(v[63])
      : "memory");
}

// tcgen05.mma with the A operand in tensor memory (a_tmem), B from shared memory
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

// One 2-D tiled tensor copy global -> shared completing on `bar` (x, the byte offset within
// a key row, is 0 here: 16-byte aligned).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Butterfly max / sum over the warp's 32 lanes of 32 values each: afterwards lane c holds the
// reduction of value c over all lanes (at each step the lanes with bit s set keep the upper
// half of the values still in play, so the surviving index is the lane's own).
template <bool SUM>
__device__ __forceinline__ float transpose_reduce32(float (&v)[32], int lane) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool upper = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      const float keep = upper ? v[i + s] : v[i];
      const float send = upper ? v[i] : v[i + s];
      const float recv = __shfl_xor_sync(0xffffffffu, send, s);
      v[i] = SUM ? keep + recv : fmaxf(keep, recv);
    }
  }
  return v[0];
}

// Maximum of v over the warp's 32 lanes, in every lane (redux.sync on f32, sm_100 family)
__device__ __forceinline__ float warp_max_f32(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// Order-preserving map of a float onto a signed int (negative values have their magnitude
// bits flipped), so that an integer max in shared memory combines float maxima.
__device__ __forceinline__ int ord_enc(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : (i ^ 0x7fffffff);
}
__device__ __forceinline__ float ord_dec(int e) { return __int_as_float(e >= 0 ? e : (e ^ 0x7fffffff)); }

template <bool LSE>
__global__ void __launch_bounds__(kSpWarps * 32, 2) spec_indexer_kernel(const IndexerArgs a, const __grid_constant__ CUtensorMap keys_map,
                                                                   int ncols, int kb) {
  extern __shared__ uint8_t smem_raw[];
  grid_dependency_wait();
  grid_dependents_launch();
  const uint32_t base_u32 = smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024 - (base_u32 & 1023)) & 1023);
  uint8_t* q_tile = base;                               // [2 halves][ncols rows][128 B], SW128
  uint8_t* raw = q_tile + 2 * kSpMaxN * 128;            // [stage] 9 KB
  SpShared* sh = reinterpret_cast<SpShared*>(raw + kSpRawSt * kSpRaw);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.q_len, G = a.groups, rows = T * G;
  const int b = blockIdx.y;
  const int L = a.seq_lens[b];
  const bool ok = L > 0 && L >= T && L <= static_cast<int64_t>(a.max_blocks) * kBlock;
  if (!ok && L != 0 && blockIdx.x == 0 && tid == 0) flag_error(a.err, MSA_DEVERR_BAD_SEQLEN);
  const int n0 = blockIdx.x * kb;
  const int nblk = ok ? max(0, min(n0 + kb, (L + kBlock - 1) / kBlock) - n0) : 0;
  const uint32_t qhalf = static_cast<uint32_t>(ncols) * 128;  // bytes of one half of the query tile

  if (tid == 0) {
    for (int i = 0; i < kSpRawSt; ++i) {
      mbar_init(&sh->raw_full[i], 1);
      mbar_init(&sh->raw_empty[i], kSpDeqWarps);
    }
    for (int i = 0; i < kSpSt; ++i) {
      mbar_init(&sh->k_full[i], kSpDeqWarps);
      mbar_init(&sh->k_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh->acc_full[i], 1);
      mbar_init(&sh->acc_empty[i], 4);
    }
    mbar_init(&sh->q_ready, 4);
    fence_mbar_init();
  }
  if (tid < kSpKbMax) {
    int page = -1;
    if (tid < nblk) {
      page = a.block_table[static_cast<int64_t>(b) * a.max_blocks + n0 + tid];
      if (page < 0 || page >= a.num_pages) {
        flag_error(a.err, MSA_DEVERR_BAD_PAGE);
        page = -1;
      }
    }
    sh->pages[tid] = page;
  }
  if (!LSE) {  // per (row, block) maxima, combined over the epilogue warps with integer atomics
    int* sbi = reinterpret_cast<int*>(&sh->sbuf[0][0]);
    for (int i = tid; i < kSpMaxN * (kSpKbMax + 1); i += kSpWarps * 32) sbi[i] = ord_enc(-INFINITY);
  }
  if (warp == kSpMmaWarp && nblk > 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sh->tmem_base)),
                 "r"(kSpTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  bool failed = false;

  if (nblk > 0) {
    if (warp == kSpCopyWarp) {
      // ---- raw page producer
      if (lane == 0) {
        for (int k = 0; k < nblk && !failed; ++k) {
          const int s = k % kSpRawSt;
          if (k >= kSpRawSt && !mbar_wait(&sh->raw_empty[s], ((k / kSpRawSt) - 1) & 1)) {
            failed = true;
            break;
          }
          const int page = sh->pages[k];
          if (page >= 0) {
            uint8_t* dst = raw + s * kSpRaw;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&sh->raw_full[s], kSpRaw);
            tma_load_2d(dst, &keys_map, 0, page * kBlock, &sh->raw_full[s]);  // 64-byte swizzled rows
            bulk_g2s(dst + kPageData, a.idx_scale + static_cast<int64_t>(page) * kPageScale, kPageScale,
                     &sh->raw_full[s]);
          } else {
            mbar_arrive(&sh->raw_full[s]);
          }
        }
        if (failed)
          for (int k = max(0, nblk - kSpRawSt); k < nblk; ++k) mbar_wait(&sh->raw_full[k % kSpRawSt], (k / kSpRawSt) & 1);
      }
    } else if (warp >= 4 && warp < 4 + kSpDeqWarps) {
      // ---- dequantisers: thread = key row 32 (warp - 4) + lane; its 128 dims in registers,
      // then into its TMEM lane (lane quarter warp % 4) of the key stage
      const int key = (warp - 4) * 32 + lane;
      const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
      for (int k = 0; k < nblk; ++k) {
        const int rs = k % kSpRawSt, s = k % kSpSt;
        if (!mbar_wait_warp(&sh->raw_full[rs], (k / kSpRawSt) & 1) ||
            (k >= kSpSt && !mbar_wait_warp(&sh->k_empty[s], ((k / kSpSt) - 1) & 1))) {
          failed = true;
          break;
        }
        tc_fence_after();
        const uint8_t* src = raw + rs * kSpRaw;
        const uint2 scw = lds64(src + kPageData + key * kRowScales);  // the row's 8 scales
        uint32_t sc[8];  // each as an f16 pair (s, s), converted once per row
#pragma unroll
        for (int i = 0; i < 8; ++i) sc[i] = e4m3_bcast_f16x2(i < 4 ? scw.x : scw.y, i & 3);
        // register r = dims 2r, 2r+1 (f16 pair): the row laid along its TMEM lane's columns
        uint32_t hv[64];
#pragma unroll
        for (int c = 0; c < 4; ++c) {  // 16 bytes = 32 dims at a time
          // the copy swizzled the row's 16-byte chunks: chunk c sits at c ^ ((key >> 1) & 3), so
          // the eight lanes of a shared-memory phase read eight different bank groups
          const uint4 d = lds128(src + key * kRowBytes + 16 * (c ^ ((key >> 1) & 3)));
          const uint32_t wd[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {  // 8 dims 32c + 8i .. +7: scale 2c + i / 2
            const uint32_t f = sc[2 * c + (i >> 1)];
            uint32_t x0, x1, x2, x3;
            e2m1x8_to_f16x2(wd[i], x0, x1, x2, x3);
            hv[16 * c + 4 * i] = hmul2(x0, f);
            hv[16 * c + 4 * i + 1] = hmul2(x1, f);
            hv[16 * c + 4 * i + 2] = hmul2(x2, f);
            hv[16 * c + 4 * i + 3] = hmul2(x3, f);
          }
        }
        tmem_st64(trow + s * kSpACols, hv);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sh->k_full[s]);
          mbar_arrive(&sh->raw_empty[rs]);
        }
      }
    } else if (warp == kSpMmaWarp) {
      // ---- MMA issuer: D[keys][rows] = K . Q^T, eight K-steps of 16 dims per page
      if (lane == 0) {
        const uint32_t idesc = umma_idesc_f16(kBlock, ncols);
        const uint32_t qb = smem_u32(q_tile);
        failed = !mbar_wait(&sh->q_ready, 0);
        for (int k = 0; k < nblk && !failed; ++k) {
          const int s = k % kSpSt, acc = k & 1;
          if (!mbar_wait(&sh->k_full[s], (k / kSpSt) & 1) ||
              (k >= 2 && !mbar_wait(&sh->acc_empty[acc], ((k / 2) - 1) & 1))) {
            failed = true;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // 16 dims = 8 TMEM columns of A per step
            const uint32_t qo = (kk >= 4 ? qhalf : 0) + (kk & 3) * 32;
            umma_f16_ta(tmem + kSpDCol + acc * kSpMaxN, tmem + s * kSpACols + kk * 8, umma_desc(qb + qo), idesc,
                        kk > 0 ? 1u : 0u);
          }
          umma_commit(&sh->k_empty[s]);
          umma_commit(&sh->acc_full[acc]);
        }
      }
      __syncwarp();
    } else {
      // ---- warps 0-3: the query rows (FP8 -> f16, exact; rows past T x G are zero)
      for (int it = tid; it < ncols * 8; it += 128) {
        const int r = it >> 3, c = it & 7;  // dims 16c .. 16c+15
        uint32_t hq[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (r < rows) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.index_q + (static_cast<int64_t>(b) * rows + r) * kDim +
                                                               16 * c));
          const uint32_t wq[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            hq[2 * i] = e4m3x2_to_f16x2(wq[i]);
            hq[2 * i + 1] = e4m3x2_to_f16x2(wq[i] >> 16);
          }
        }
        uint8_t* tdst = q_tile + (c < 4 ? 0 : qhalf);
        const int ch = 2 * (c & 3);
        *reinterpret_cast<uint4*>(tdst + sw128(r, ch)) = make_uint4(hq[0], hq[1], hq[2], hq[3]);
        *reinterpret_cast<uint4*>(tdst + sw128(r, ch + 1)) = make_uint4(hq[4], hq[5], hq[6], hq[7]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->q_ready);

      // ---- epilogue: warp w holds keys 32w .. 32w+31 of each page (TMEM lane quarter w)
      const uint32_t tq = tmem + (static_cast<uint32_t>(warp * 32) << 16);
      const int pos0 = L - T;  // position of token 0; row c belongs to token c / G
      if (!LSE) {
        // max pooling: 16 rows at a time, each warp's maxima go straight into the shared
        // (row, block) table with an integer atomic max, so the warps never wait on each other
        int* sbi = reinterpret_cast<int*>(&sh->sbuf[0][0]);
        for (int k = 0; k < nblk && !failed; ++k) {
          const int acc = k & 1;
          if (!mbar_wait_warp(&sh->acc_full[acc], (k / 2) & 1)) {
            failed = true;
            break;
          }
          tc_fence_after();
          const int key = (n0 + k) * kBlock + warp * 32 + lane;
          // row c (token c / G) sees the key iff key <= pos0 + c / G, i.e. iff c >= cmin; only
          // the pages at the end of the sequence hold keys some row must not see
          const int cmin = key <= pos0 ? 0 : (key - pos0) * G;
          const bool masked = __any_sync(0xffffffffu, cmin > 0);
          for (int c0 = 0; c0 < ncols; c0 += 16) {
            uint32_t raw16[16];
            tmem_ld16(tq + kSpDCol + acc * kSpMaxN + c0, raw16);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            if (c0 + 16 >= ncols) {  // the accumulator is read: the next product may overwrite it
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sh->acc_empty[acc]);
            }
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(raw16[j]);
            if (masked) {
#pragma unroll
              for (int j = 0; j < 16; ++j) v[j] = (c0 + j >= cmin) ? v[j] : -INFINITY;
            }
            // the 16 columns' maxima over this warp's keys (warp-wide reductions), staged so that
            // lane j holds column c0 + j
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = warp_max_f32(v[j]);
            float* wm = sh->wmax[warp];
            if (lane == 0) {
#pragma unroll
              for (int j = 0; j < 16; j += 4) *reinterpret_cast<float4*>(wm + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            }
            __syncwarp();
            const float m = wm[lane & 15];
            __syncwarp();  // every lane has read before the next chunk restages
            const int c = c0 + lane;
            if (lane < 16 && c < rows) atomicMax(&sbi[c * (kSpKbMax + 1) + k], ord_enc(m));
          }
        }
      } else {
        // log-sum-exp pooling (every iteration reaches the named barrier below, also after a
        // timed-out wait: a warp that left the loop would stall the others there)
        for (int k = 0; k < nblk; ++k) {
          const int acc = k & 1;
          if (!failed && !mbar_wait_warp(&sh->acc_full[acc], (k / 2) & 1)) failed = true;
          tc_fence_after();
          const int key = (n0 + k) * kBlock + warp * 32 + lane;
          // row c (token c / G) sees the key iff key <= pos0 + c / G, i.e. iff c >= cmin: one
          // threshold per thread instead of a division per value
          const int cmin = key <= pos0 ? 0 : (key - pos0) * G;
          for (int c0 = 0; c0 < ncols && !failed; c0 += 32) {  // 32 rows at a time
            uint32_t raw32[32];
            tmem_ld32(tq + kSpDCol + acc * kSpMaxN + c0, raw32);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            if (c0 + 32 >= ncols) {  // the accumulator is read: the next product may overwrite it
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sh->acc_empty[acc]);
            }
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int c = c0 + j;
              v[j] = (c < rows && c >= cmin) ? __uint_as_float(raw32[j]) : -INFINITY;
            }
            float m32[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) m32[j] = v[j];
            const float mlane = transpose_reduce32<false>(m32, lane);  // row c0 + lane, this warp's keys
            sh->red[acc][warp][c0 + lane] = mlane;
            // e^{s - m_w} with the row's maximum over this warp's keys; the rows' final maximum
            // M is applied below: sum_j e^{s_j - m_w} e^{m_w - M} = sum_j e^{s_j - M}
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float mw = __shfl_sync(0xffffffffu, mlane, j);
              v[j] = (mw == -INFINITY) ? 0.f : expf(v[j] - mw);
            }
            sh->red2[acc][warp][c0 + lane] = transpose_reduce32<true>(v, lane);
          }
          if (failed) {  // defined values for the reduction below
            sh->red[acc][warp][lane] = -INFINITY;
            sh->red[acc][warp][32 + lane] = -INFINITY;
          }
          if (failed && lane == 0) mbar_arrive(&sh->acc_empty[acc]);  // (not read: keep the count)
          asm volatile("bar.sync 1, 128;" ::: "memory");  // the four warps' partial reductions
          if (warp == 0) {
            for (int c = lane; c < rows; c += 32) {
              float m = -INFINITY;
#pragma unroll
              for (int w = 0; w < 4; ++w) m = fmaxf(m, sh->red[acc][w][c]);
              if (m != -INFINITY) {
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                  const float mw = sh->red[acc][w][c];
                  if (mw != -INFINITY) sum += sh->red2[acc][w][c] * expf(mw - m);
                }
                m += logf(sum);
              }
              sh->sbuf[c][k] = sh->pages[k] >= 0 ? m : -INFINITY;
            }
          }
        }
      }
    }
  }

  // ---- scores out: one row per warp iteration, a block per lane (coalesced)
  __syncthreads();
  if (warp < 4) {
    for (int c = warp; c < rows; c += 4)
      for (int j = lane; j < kb; j += 32) {
        const int n = n0 + j;
        if (n < a.max_blocks) {
          float sc = -INFINITY;
          if (j < nblk) {
            if (LSE) sc = sh->sbuf[c][j];
            else if (sh->pages[j] >= 0) sc = ord_dec(reinterpret_cast<const int*>(&sh->sbuf[0][0])[c * (kSpKbMax + 1) + j]);
          }
          a.block_scores[(static_cast<int64_t>(b) * rows + c) * a.max_blocks + n] = sc;
        }
      }
  }
  if (failed && lane == 0) flag_error(a.err, MSA_DEVERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kSpMmaWarp && nblk > 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kSpTmemCols));
}

// Tensor map of the index-key pool viewed as rows of 64 bytes ([num_pages * 128][64]), boxes of
// one page (128 rows), 64-byte swizzle.  The encoder comes from the driver at first use.
static cudaError_t encode_keys_map(const IndexerArgs& a, CUtensorMap* map) {
  static const PFN_cuTensorMapEncodeTiled_v12000 encode = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }();
  if (encode == nullptr) return cudaErrorNotSupported;
  // row coordinates are signed 32-bit
  if (a.num_pages < 1 || a.num_pages > (static_cast<int64_t>(INT32_MAX) + 1) / kBlock) return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kRowBytes), static_cast<cuuint64_t>(a.num_pages) * kBlock};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kRowBytes)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kRowBytes), static_cast<cuuint32_t>(kBlock)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.idx_data), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <bool LSE>
static cudaError_t launch_spec_t(const IndexerArgs& a, int num_sms, cudaStream_t s) {
  const int rows = a.q_len * a.groups;
  const int ncols = (rows + 15) / 16 * 16;
  CUtensorMap keys_map;
  cudaError_t e = encode_keys_map(a, &keys_map);
  if (e != cudaSuccess) return e;
  e = ensure_dynamic_smem(reinterpret_cast<const void*>(spec_indexer_kernel<LSE>), kSpSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  // key blocks per CTA: the fewest (at most 64) that still fit the grid into one round of
  // two CTAs per SM, so that no partly filled last wave is left
  const int64_t slots = 2LL * num_sms;
  const int64_t per_seq = std::max<int64_t>(1, slots / std::max(1, a.batch));
  int kb = static_cast<int>((a.max_blocks + per_seq - 1) / per_seq);
  kb = std::min(kSpKbMax, std::max(8, kb));
  cfg.gridDim = dim3((a.max_blocks + kb - 1) / kb, static_cast<unsigned>(a.batch));
  cfg.blockDim = dim3(kSpWarps * 32);
  cfg.dynamicSmemBytes = kSpSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, spec_indexer_kernel<LSE>, a, keys_map, ncols, kb);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_spec_indexer(const IndexerArgs& a, int num_sms, cudaStream_t s) {
  return a.lse ? launch_spec_t<true>(a, num_sms, s) : launch_spec_t<false>(a, num_sms, s);
}

}  // namespace msa
