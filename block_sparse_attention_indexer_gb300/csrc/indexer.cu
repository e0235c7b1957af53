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

template <bool LSE>
__global__ void __launch_bounds__(kHWarps * 32, 1) indexer_half_kernel(const IndexerArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int32_t warp_tot[kHWarps];
  grid_dependency_wait();
  grid_dependents_launch();
  index_scan_cta<LSE>(a, smem, warp_tot, blockIdx.x, gridDim.x);
}

template <bool LSE>
static cudaError_t launch_half_t(const IndexerArgs& a, int num_sms, cudaStream_t s) {
  const size_t smem = index_scan_smem_bytes(a.batch);
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
