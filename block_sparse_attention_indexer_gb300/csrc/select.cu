// Stage 2 of MSA decode: top-k block selection with the most recent block forced, one warp
// per (sequence, query token, KV group) row.  The per-row routine and its rules are in
// select_row.cuh.
#include "msa_kernels.h"
#include "select_row.cuh"

namespace msa {

constexpr int kSelWarps = 4;
constexpr int kSelCap = 512;

__global__ void __launch_bounds__(kSelWarps * 32) select_kernel(const SelectArgs a) {
  extern __shared__ __align__(16) uint32_t sord_all[];  // [kSelWarps][row_cap] staged score orders
  __shared__ uint64_t buf[kSelWarps][kSelCap];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // launched as a programmatic dependent of the previous kernel on the stream: wait for it
  // (and its memory) before touching global memory
  grid_dependency_wait();
  grid_dependents_launch();
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
  const int r = (L - a.q_len + t) / kBlock;
  const int id = select_row_warp(a.block_scores + row * a.max_blocks, r, a.top_k, a.init_blocks, a.local_blocks, lane,
                                 sord_all + static_cast<int64_t>(warp) * a.row_cap, a.row_cap, buf[warp], kSelCap);
  if (lane < kTopK) out[lane] = id;
}

cudaError_t launch_select(const SelectArgs& a0, cudaStream_t s) {
  SelectArgs a = a0;
  const int64_t nrows = static_cast<int64_t>(a.batch) * a.q_len * a.groups;
  if (nrows == 0) return cudaSuccess;
  // stage rows of up to 4096 candidates in shared memory (64 KB for 4 warps); longer rows
  // are read from L2 on each pass
  a.row_cap = a.max_blocks < 4096 ? a.max_blocks : 4096;
  const size_t smem = static_cast<size_t>(kSelWarps) * a.row_cap * sizeof(uint32_t);
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(select_kernel), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((nrows + kSelWarps - 1) / kSelWarps));
  cfg.blockDim = dim3(kSelWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, select_kernel, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace msa
