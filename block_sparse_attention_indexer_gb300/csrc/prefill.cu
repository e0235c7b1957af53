// Stage 1 for long query chunks (chunked prefill): the indexer as a dense tensor-core GEMM.
//
// In prefill the index path scores every candidate KV block for every query token and KV
// group, reduced per 128-token block with max ("MiniMax M3 x vLLM：百万 token 多模态推理的
// Day-0 部署", §Prefill 执行 step 2): S[row][n] = max over visible keys j of block n of
// q_row . k_j with row = (token, group).  With thousands of query rows this is a dense
// [rows x 128] x [128 x keys] product followed by a max-pool over each 128-key block of
// its columns, causal (key j visible to token t iff j <= pos(t)).
//
// Design (GB300, tcgen05 + TMEM):
//   * a CTA owns two tiles of 128 query rows (256 rows) and a range of 32 key blocks; the
//     query tiles are converted once (FP8 E4M3 -> f16, exact) into K-major, 128-byte-swizzled
//     shared tiles, the A operands of every MMA of the CTA;
//   * warp roles: warp 16 streams the raw NVFP4 pages (9 KB) with bulk async copies into a
//     3-stage ring; warps 8-15 dequantise each page exactly into f16 (cvt e2m1x2 -> f16x2
//     times the f16 block scale) in the same swizzled K-major layout (B operand, 2 stages) --
//     two warps per scheduler, two independent items each per page; one thread of warp 17
//     issues tcgen05.mma (M = 128 rows, N = 128 keys, K = 16, eight per block and tile) into
//     one of two accumulator stages of 2 x 128 TMEM columns, so that every dequantised key
//     page feeds both tiles (half the conversion work per MMA of a one-tile CTA); warps 0-7
//     convert the query tiles while the first pages arrive, then read the accumulators back
//     with tcgen05.ld (warp w: tile w / 4, TMEM lane quarter w % 4), apply the causal mask
//     and max-pool the 128 columns into the block's score;
#include <cuda_fp16.h>

#include "msa_device.cuh"
#include "msa_kernels.h"
#include "umma.cuh"

namespace msa {

constexpr int kPfKb = 32;                 // key blocks per CTA
constexpr int kPfRawSt = 3;               // raw NVFP4 page stages
constexpr int kPfKSt = 2;                 // f16 key tile stages
constexpr int kPfRows = 128;              // query rows per tile (MMA M)
constexpr int kPfTiles = 2;               // query tiles per CTA
constexpr int kPfM = kPfTiles * kPfRows;  // query rows per CTA
constexpr int kPfEpiWarps = 4 * kPfTiles; // query conversion, then the epilogue
constexpr int kPfDeqWarps = 8;
constexpr int kPfCopyWarp = kPfEpiWarps + kPfDeqWarps, kPfMmaWarp = kPfCopyWarp + 1;
constexpr int kPfWarps = kPfMmaWarp + 1;
constexpr int kHalfTile = kPfRows * 128;  // one [128 x 64] f16 K-major SW128 tile: 16 KB
constexpr int kRawBytes = kPageData + kPageScale;
constexpr uint32_t kPfTmemCols = 2 * kPfTiles * kBlock;  // two accumulator stages x tiles: 512

struct PfShared {
  uint64_t raw_full[kPfRawSt], raw_empty[kPfRawSt];
  uint64_t k_full[kPfKSt], k_empty[kPfKSt];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t q_ready;
  uint32_t tmem_base;
  int32_t pages[kPfKb];
};

constexpr int kSbufLd = kPfKb + 1;        // score buffer row stride (odd: conflict-free column writes)
constexpr size_t kPfSmem = 1024 /* alignment slack */ + kPfTiles * 2 * kHalfTile /* Q */ +
                           kPfKSt * 2 * kHalfTile /* K */ + kPfRawSt * kRawBytes +
                           kPfM * kSbufLd * sizeof(float) + sizeof(PfShared);

template <bool LSE>
__global__ void __launch_bounds__(kPfWarps * 32, 1) prefill_indexer_kernel(const IndexerArgs a, int tiles_per_seq) {
  extern __shared__ uint8_t smem_raw[];
  grid_dependency_wait();
  grid_dependents_launch();

  // carve shared memory (tiles 1024-byte aligned for the swizzle)
  const uint32_t base_u32 = smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024 - (base_u32 & 1023)) & 1023);
  uint8_t* q_tiles = base;                                  // [tile] A0 | A1
  uint8_t* k_tiles = q_tiles + kPfTiles * 2 * kHalfTile;    // [stage] B0 | B1
  uint8_t* raw = k_tiles + kPfKSt * 2 * kHalfTile;          // [stage] 9 KB
  float* sbuf = reinterpret_cast<float*>(raw + kPfRawSt * kRawBytes);  // [256][kSbufLd]
  PfShared* sh = reinterpret_cast<PfShared*>(sbuf + kPfM * kSbufLd);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.q_len, G = a.groups;
  const int b = blockIdx.y / tiles_per_seq, tile = blockIdx.y % tiles_per_seq;
  const int rows_seq = T * G;
  const int row0 = tile * kPfM;
  const int nrows = min(kPfM, rows_seq - row0);
  const int L = a.seq_lens[b];
  const bool ok = L > 0 && L >= T && L <= static_cast<int64_t>(a.max_blocks) * kBlock;
  if (!ok && L != 0 && blockIdx.x == 0 && tile == 0 && tid == 0) flag_error(a.err, MSA_DEVERR_BAD_SEQLEN);
  const int n0 = blockIdx.x * kPfKb;
  // blocks some row of this CTA can see: n <= r(last token of its rows), n < ceil(L / 128)
  int nblk = 0;
  if (ok && nrows > 0) {
    const int pos_last = L - T + (row0 + nrows - 1) / G;
    const int nb_eff = min((L + kBlock - 1) / kBlock, pos_last / kBlock + 1);
    nblk = max(0, min(n0 + kPfKb, nb_eff) - n0);
  }
  // tiles of this CTA with rows (the MMAs of an empty second tile are skipped)
  const int ntiles = nrows > kPfRows ? 2 : 1;

  if (tid == 0) {
    for (int i = 0; i < kPfRawSt; ++i) {
      mbar_init(&sh->raw_full[i], 1);
      mbar_init(&sh->raw_empty[i], kPfDeqWarps);
    }
    for (int i = 0; i < kPfKSt; ++i) {
      mbar_init(&sh->k_full[i], kPfDeqWarps);
      mbar_init(&sh->k_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh->acc_full[i], 1);
      mbar_init(&sh->acc_empty[i], kPfEpiWarps);
    }
    mbar_init(&sh->q_ready, kPfEpiWarps);
    fence_mbar_init();
  }
  if (tid < kPfKb) {
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
  if (warp == kPfMmaWarp && nblk > 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sh->tmem_base)),
                 "r"(kPfTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  bool failed = false;

  if (nblk > 0) {
    if (warp == kPfCopyWarp) {
      // ---- raw page producer
      if (lane == 0) {
        for (int k = 0; k < nblk && !failed; ++k) {
          const int s = k % kPfRawSt;
          if (k >= kPfRawSt && !mbar_wait(&sh->raw_empty[s], ((k / kPfRawSt) - 1) & 1)) {
            failed = true;
            break;
          }
          const int page = sh->pages[k];
          if (page >= 0) {
            uint8_t* dst = raw + s * kRawBytes;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&sh->raw_full[s], kRawBytes);
            bulk_g2s(dst, a.idx_data + static_cast<int64_t>(page) * kPageData, kPageData, &sh->raw_full[s]);
            bulk_g2s(dst + kPageData, a.idx_scale + static_cast<int64_t>(page) * kPageScale, kPageScale,
                     &sh->raw_full[s]);
          } else {
            mbar_arrive(&sh->raw_full[s]);
          }
        }
        // after a timeout, wait (bounded) for the copies still in flight before leaving
        if (failed)
          for (int k = max(0, nblk - kPfRawSt); k < nblk; ++k) mbar_wait(&sh->raw_full[k % kPfRawSt], (k / kPfRawSt) & 1);
      }
    } else if (warp >= kPfEpiWarps && warp < kPfEpiWarps + kPfDeqWarps) {
      // ---- dequantisers: every key page, two items per thread per page
      const int dt = tid - kPfEpiWarps * 32;
      for (int k = 0; k < nblk; ++k) {
        const int s = k % kPfRawSt, ks = k % kPfKSt;
        if (!mbar_wait_warp(&sh->raw_full[s], (k / kPfRawSt) & 1) ||
            (k >= kPfKSt && !mbar_wait_warp(&sh->k_empty[ks], ((k / kPfKSt) - 1) & 1))) {
          failed = true;
          break;
        }
        const uint8_t* src = raw + s * kRawBytes;
        uint8_t* kdst = k_tiles + ks * 2 * kHalfTile;
        // items (row, 32-dim chunk c) in octets (8 lanes = one shared-memory phase of 16-byte
        // accesses): two octets share a group of 4 rows, lane i of octet o takes chunk
        // c = i >> 1 of row 4 (o >> 1) + (i & 1) + 2 (((i >> 1) & 1) ^ (o & 1)).  An octet's
        // loads then hit 8 distinct 16-byte bank groups (row parity x chunk), and with the chunk
        // order of the upper half of the dims rotated by 2 so do its swizzled stores
        constexpr int kItems = kBlock * 4 / (kPfDeqWarps * 32);
        int rr[kItems], cc[kItems];
        uint4 d[kItems];
        uint32_t sc[kItems];
#pragma unroll
        for (int u = 0; u < kItems; ++u) {
          const int item = dt + u * kPfDeqWarps * 32;
          const int i8 = item & 7, oct = item >> 3;
          rr[u] = 4 * (oct >> 1) + (i8 & 1) + 2 * (((i8 >> 1) & 1) ^ (oct & 1));
          cc[u] = i8 >> 1;  // dims 32c .. 32c+31
          d[u] = lds128(src + rr[u] * kRowBytes + 16 * cc[u]);
          sc[u] = lds16(src + kPageData + rr[u] * kRowScales + 2 * cc[u]);
        }
#pragma unroll
        for (int u = 0; u < kItems; ++u) {
          const int r = rr[u], c = cc[u];
          const uint32_t s0 = e4m3_bcast_f16x2(sc[u], 0), s1 = e4m3_bcast_f16x2(sc[u], 1);
          const uint32_t w[4] = {d[u].x, d[u].y, d[u].z, d[u].w};
          uint32_t h[16];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            e2m1x8_to_f16x2(w[i], h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
            const uint32_t sca = i < 2 ? s0 : s1;
#pragma unroll
            for (int j = 0; j < 4; ++j) h[4 * i + j] = hmul2(h[4 * i + j], sca);
          }
          uint8_t* tdst = kdst + (c < 2 ? 0 : kHalfTile);
          const int ch = 4 * (c & 1);
          const bool rot = c >= 2;  // store q writes chunk q ^ 2 in the upper half
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int qq = q ^ 2;
            const uint4 v = rot ? make_uint4(h[4 * qq], h[4 * qq + 1], h[4 * qq + 2], h[4 * qq + 3])
                                : make_uint4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
            *reinterpret_cast<uint4*>(tdst + sw128(r, ch + (rot ? qq : q))) = v;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sh->k_full[ks]);
          mbar_arrive(&sh->raw_empty[s]);
        }
      }
    } else if (warp == kPfMmaWarp) {
      // ---- MMA issuer: per block, the key tile against each query tile
      if (lane == 0) {
        const uint32_t idesc = umma_idesc_f16(kPfRows, kBlock);
        failed = !mbar_wait(&sh->q_ready, 0);
        for (int k = 0; k < nblk && !failed; ++k) {
          const int ks = k % kPfKSt, acc = k & 1;
          if (!mbar_wait(&sh->k_full[ks], (k / kPfKSt) & 1) ||
              (k >= 2 && !mbar_wait(&sh->acc_empty[acc], ((k / 2) - 1) & 1))) {
            failed = true;
            break;
          }
          tc_fence_after();
          const uint32_t kb = smem_u32(k_tiles + ks * 2 * kHalfTile);
          for (int t = 0; t < ntiles; ++t) {
            const uint32_t qa = smem_u32(q_tiles + t * 2 * kHalfTile);
            const uint32_t d_tmem = tmem + static_cast<uint32_t>((acc * kPfTiles + t) * kBlock);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t off = (kk >= 4 ? kHalfTile : 0) + (kk & 3) * 32;
              umma_f16(d_tmem, umma_desc(qa + off), umma_desc(kb + off), idesc, kk > 0 ? 1u : 0u);
            }
          }
          umma_commit(&sh->k_empty[ks]);
          umma_commit(&sh->acc_full[acc]);
        }
      }
      __syncwarp();
    } else {
      // ---- warps 0-7: the query tiles (FP8 E4M3 -> f16, exact), all loads issued first
      {
        constexpr int kQItems = kPfM * 8 / (kPfEpiWarps * 32);
        uint4 qv[kQItems];
#pragma unroll
        for (int u = 0; u < kQItems; ++u) {
          const int item = tid + kPfEpiWarps * 32 * u, r = item >> 3, c = item & 7;  // dims 16c .. 16c+15
          qv[u] = r < nrows ? __ldg(reinterpret_cast<const uint4*>(
                                  a.index_q + (static_cast<int64_t>(b) * rows_seq + row0 + r) * kDim + 16 * c))
                            : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kQItems; ++u) {
          const int item = tid + kPfEpiWarps * 32 * u, r = item >> 3, c = item & 7;
          const uint32_t w[4] = {qv[u].x, qv[u].y, qv[u].z, qv[u].w};
          uint32_t h[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            h[2 * i] = e4m3x2_to_f16x2(w[i]);
            h[2 * i + 1] = e4m3x2_to_f16x2(w[i] >> 16);
          }
          uint8_t* tdst = q_tiles + (r / kPfRows) * 2 * kHalfTile + (c < 4 ? 0 : kHalfTile);
          const int rt = r % kPfRows, ch = 2 * (c & 3);
          *reinterpret_cast<uint4*>(tdst + sw128(rt, ch)) = make_uint4(h[0], h[1], h[2], h[3]);
          *reinterpret_cast<uint4*>(tdst + sw128(rt, ch + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->q_ready);
      }

      // ---- epilogue (warp w: tile w / 4, TMEM lane quarter w % 4): causal pooling per block
      const int et = warp / 4, quarter = warp % 4;
      const int r = et * kPfRows + quarter * 32 + lane;
      const bool row_ok = r < nrows;
      const int pos = row_ok ? L - T + (row0 + r) / G : -1;
      constexpr bool lse = LSE;  // block pooling: log-sum-exp or max
      const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(et * kBlock);
      const bool active = et < ntiles;  // warp-uniform: a second tile without rows has no accumulator
      for (int k = 0; k < nblk; ++k) {
        const int acc = k & 1;
        if (!mbar_wait_warp(&sh->acc_full[acc], (k / 2) & 1)) {
          failed = true;
          break;
        }
        tc_fence_after();
        float mx = -INFINITY;
        if (active) {
          const uint32_t tacc = trow + static_cast<uint32_t>(acc * kPfTiles * kBlock);
          const int lim = pos - (n0 + k) * kBlock;  // columns 0 .. lim are visible to this row
          // max: each 64-column load also returns the maximum of what it loads (tcgen05.ld.red);
          // only the half holding the causal limit is masked by hand (four independent chains)
#pragma unroll
          for (int c0 = 0; c0 < kBlock; c0 += 64) {
            uint32_t v[64];
            float hmax;
            tmem_ld64_max(tacc + c0, v, hmax);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            if (c0 + 63 <= lim) {
              mx = fmaxf(mx, hmax);
            } else {
              float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
              for (int j = 0; j < 64; ++j) m4[j & 3] = fmaxf(m4[j & 3], c0 + j <= lim ? __uint_as_float(v[j]) : -INFINITY);
              mx = fmaxf(mx, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])));
            }
          }
          if (lse) {
            // log-sum-exp pooling: a second pass over the accumulator, sum e^{s - max} (the
            // warp-collective loads run in every lane; a row with nothing visible stays -inf)
            const float m_use = mx == -INFINITY ? 0.f : mx;
            float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c0 = 0; c0 < kBlock; c0 += 64) {
              uint32_t v[2][32];
              tmem_ld32(tacc + c0, v[0]);
              tmem_ld32(tacc + c0 + 32, v[1]);
              asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
              for (int j = 0; j < 64; ++j)
                if (c0 + j <= lim) s4[j & 3] += expf(__uint_as_float(v[j >> 5][j & 31]) - m_use);
            }
            if (mx != -INFINITY) mx += logf((s4[0] + s4[1]) + (s4[2] + s4[3]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->acc_empty[acc]);
        sbuf[r * kSbufLd + k] = (row_ok && sh->pages[k] >= 0) ? mx : -INFINITY;
      }
    }
  }

  // ---- scores out: the epilogue warps write their 32 rows, a block per lane (coalesced)
  if (warp < kPfEpiWarps) {
    __syncwarp();
    const int64_t grow0 = static_cast<int64_t>(b) * rows_seq + row0;
    for (int i = 0; i < 32; ++i) {
      const int r = warp * 32 + i;
      const int n = n0 + lane;
      if (r < nrows && n < a.max_blocks)
        a.block_scores[(grow0 + r) * a.max_blocks + n] = lane < nblk ? sbuf[r * kSbufLd + lane] : -INFINITY;
    }
  }
  if (failed && lane == 0) flag_error(a.err, MSA_DEVERR_TIMEOUT);

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kPfMmaWarp && nblk > 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kPfTmemCols));
}

template <bool LSE>
static cudaError_t launch_prefill_t(const IndexerArgs& a, cudaStream_t s) {
  const int rows_seq = a.q_len * a.groups;
  const int tiles_per_seq = (rows_seq + kPfM - 1) / kPfM;
  const int ranges = (a.max_blocks + kPfKb - 1) / kPfKb;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(prefill_indexer_kernel<LSE>), kPfSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ranges, static_cast<unsigned>(a.batch * tiles_per_seq));
  cfg.blockDim = dim3(kPfWarps * 32);
  cfg.dynamicSmemBytes = kPfSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, prefill_indexer_kernel<LSE>, a, tiles_per_seq);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_prefill_indexer(const IndexerArgs& a, cudaStream_t s) {
  return a.lse ? launch_prefill_t<true>(a, s) : launch_prefill_t<false>(a, s);
}

}  // namespace msa
