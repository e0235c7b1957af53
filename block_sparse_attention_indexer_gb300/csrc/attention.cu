// Stage 3 of MSA decode: exact sparse GQA attention over the selected blocks.
//
// Every query head of a KV group attends exactly, and only, to the selected blocks of that
// group ("vLLM liefert Day-0-Unterstützung für MiniMax-M3.1-Flash", §MSA-Grundlagen, Fig. 1);
// the result equals dense attention restricted to the selected set, computed with an
// online softmax ("MiniMax M3 x vLLM：百万 token 多模态推理的 Day-0 部署", §Prefill 执行
// step 4); decode consumes the selected pages and merges the partial outputs of split
// work (same page, §MiniMax 稀疏注意力后端 and §Decode 执行).
//
// Design (GB300):
//   * persistent: one CTA per SM, three independent teams of four warps.  The (row = (sequence,
//     token, group), selection entry) pairs, 16 per row, are split into equal contiguous
//     ranges, one per team, so every team streams the same number of 18 KB pages (K and V of
//     one KV head, E2M1 bytes + E4M3 scales) whatever the selections;
//   * in each team one warp produces: it resolves entries (selection -> block table -> page)
//     32 at a time, one per lane, and streams the pages through a 3-slot shared-memory ring
//     with bulk async copies (cp.async.bulk), full / empty mbarriers and the item's metadata
//     in shared memory; a row with no page to attend to still gets one marker item;
//   * every warp of the team consumes every page, each on its own 32-key quarter: QK runs
//     transposed, S^T = K Q^T on mma.sync m16n8k16 (keys as M, the <= 8 heads of the group
//     as N, so the heads fill the N=8 tile), an online softmax in the exp2 domain, then
//     O^T += V^T P^T: P is packed to f16 and transposed in registers (movmatrix) into the B
//     operand, V^T is built from two keys' bytes by a nibble transpose.  K and V are
//     dequantised exactly (cvt e2m1x2 -> f16x2 times the f16 block scale);
//   * at a row change the four warps merge their states through shared memory (mbarrier
//     handshakes, every wait bounded); a row wholly inside the team's range is written out
//     at once, a row cut by a range boundary leaves a partial state (o, m, l) in one of two
//     slots of the team, combined by merge_kernel: o = sum e^{m_s-M} o_s / sum e^{m_s-M} l_s.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "attention_team.cuh"
#include "attention_tile.cuh"
#include "msa_device.cuh"
#include "msa_kernels.h"

namespace msa {

template <bool kOwnSelect>
__global__ void __launch_bounds__(kAttnThreads, 1) attention_kernel(const AttnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  attention_cta<kOwnSelect>(a, smem, blockIdx.x, gridDim.x);
}

// by_row 0: CTA i takes range boundary i + 1 (NT - 1 CTAs); by_row 1: CTA i takes row i (for
// fewer rows than boundaries), through the first boundary inside it, if any: every CTA then
// has a row to merge or leaves at once, and the grid does not outnumber the rows.
template <int kBatch>
__global__ void __launch_bounds__(kMergeThreads, kBatch == 8 ? 2 : 1) merge_kernel(const AttnArgs a, int NT, int by_row) {
  __shared__ int s_slot[kTopK];
  __shared__ int s_n, s_row;
  int k = blockIdx.x + 1;
  if (by_row) {
    const int E = a.batch * a.q_len * a.groups * kTopK, R = blockIdx.x;
    const int ca = owner_of(E, R * kTopK, NT);
    if (owner_of(E, R * kTopK + kTopK - 1, NT) == ca) return;  // the row is one team's
    k = ca + 1;
  }
  merge_boundary<kBatch>(a, NT, k, s_slot, &s_n, &s_row);
}

size_t attn_partial_bytes() {
  return static_cast<size_t>(2) * kAttnMaxCtas * kTeams * kSlotFloats * sizeof(float);
}

cudaError_t launch_attention(const AttnArgs& a, int num_sms, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(a.batch) * a.q_len * a.groups;
  if (rows == 0) return cudaSuccess;
  const int NC = num_sms < kAttnMaxCtas ? num_sms : kAttnMaxCtas;
  const size_t smem = attn_smem_bytes();
  const bool own = a.block_scores != nullptr;
  const void* kern = own ? reinterpret_cast<const void*>(attention_kernel<true>)
                         : reinterpret_cast<const void*>(attention_kernel<false>);
  cudaError_t e = ensure_dynamic_smem(kern, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(NC);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = own ? cudaLaunchKernelEx(&cfg, attention_kernel<true>, a) : cudaLaunchKernelEx(&cfg, attention_kernel<false>, a);
  if (e != cudaSuccess) return e;
  const int NT = NC * kTeams;
  const int by_row = rows < NT - 1 ? 1 : 0;
  cudaLaunchConfig_t mcfg = {};
  mcfg.gridDim = dim3(by_row ? static_cast<unsigned>(rows) : static_cast<unsigned>(NT - 1));
  mcfg.blockDim = dim3(kMergeThreads);
  mcfg.stream = s;
  mcfg.attrs = attr;
  mcfg.numAttrs = 1;
  // a row's 16 slots in one round of loads when one CTA an SM still holds every row at once
  e = by_row && rows <= NC ? cudaLaunchKernelEx(&mcfg, merge_kernel<16>, a, NT, by_row)
                           : cudaLaunchKernelEx(&mcfg, merge_kernel<8>, a, NT, by_row);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace msa
