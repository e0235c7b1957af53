// Stage 2 of MSA decode: top-k block selection with the most recent block forced, one warp
// per (sequence, query token, KV group) row.  The per-row routine and its rules are in
// select_row.cuh.
#include "msa_kernels.h"
#include "select_row.cuh"

namespace msa {

constexpr int kSelWarps = 4;
constexpr int kSelCap = 512;

template <int KPL>
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
  const int id = select_row_warp<KPL>(a.block_scores + row * a.max_blocks, r, a.top_k, a.init_blocks, a.local_blocks, lane,
                                 sord_all + static_cast<int64_t>(warp) * a.row_cap, a.row_cap, buf[warp], kSelCap);
  if (lane < kTopK) out[lane] = id;
}

// Rows longer than 1,024 candidates (long contexts): one CTA per row.  Each of its eight
// warps takes the best of a contiguous eighth of the candidates (the row's winners are
// among the union of the eighths' winners), and the first warp picks the winners among
// those at most 8 x 16 by rounds of warp arg-max over their exact keys.
constexpr int kLongWarps = 8;

__global__ void __launch_bounds__(kLongWarps * 32) select_long_kernel(const SelectArgs a) {
  __shared__ uint64_t buf[kLongWarps][kSelCap / 8];
  __shared__ int32_t part[kLongWarps][kTopK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dependency_wait();
  grid_dependents_launch();
  const int64_t row = blockIdx.x;
  const int b = static_cast<int>(row / (static_cast<int64_t>(a.q_len) * a.groups));
  const int t = static_cast<int>((row / a.groups) % a.q_len);
  int32_t* out = a.selection + row * kTopK;
  const int L = a.seq_lens[b];
  if (L < a.q_len || L <= 0 || L > static_cast<int64_t>(a.max_blocks) * kBlock) {
    if (warp == 0 && lane < kTopK) out[lane] = -1;
    return;
  }
  const int r = (L - a.q_len + t) / kBlock;
  if (r + 1 <= a.top_k) {  // every block 0 .. r
    if (warp == 0 && lane < kTopK) out[lane] = lane <= r ? lane : -1;
    return;
  }
  const float* sc = a.block_scores + row * a.max_blocks;
  const int lo = a.init_blocks, hi = r - a.local_blocks + 1, W = a.top_k - a.init_blocks - a.local_blocks;
  const int span = (hi - lo + kLongWarps - 1) / kLongWarps;
  const int wlo = min(hi, lo + warp * span), whi = min(hi, wlo + span);
  const int ww = min(W, whi - wlo);
  const int id = top_blocks_warp(sc, wlo, whi, ww, lane, nullptr, 0, buf[warp], kSelCap / 8);
  if (lane < kTopK) part[warp][lane] = id;
  __syncthreads();
  if (warp != 0) return;
  // winners among the warps' winners: W rounds of warp arg-max over exact keys
  uint64_t key[kLongWarps * kTopK / 32];
#pragma unroll
  for (int i = 0; i < kLongWarps * kTopK / 32; ++i) {
    const int n = (&part[0][0])[32 * i + lane];
    key[i] = n >= 0 ? (static_cast<uint64_t>(score_order(__ldcg(sc + n))) << 32) |
                          static_cast<uint64_t>(0xffffffffu - static_cast<uint32_t>(n))
                    : 0ull;
  }
  int mine = 0x7fffffff;
  uint64_t prev = ~0ull;
  for (int round = 0; round < W; ++round) {
    uint64_t best = 0;
#pragma unroll
    for (int i = 0; i < kLongWarps * kTopK / 32; ++i)
      if (key[i] < prev && key[i] > best) best = key[i];
    best = warp_max_u64(best);
    prev = best;
    if (lane == round) mine = static_cast<int>(0xffffffffu - static_cast<uint32_t>(best));
  }
  const int sorted_id = warp_sort_asc_i32(mine, lane);
  const int from_win = __shfl_sync(0xffffffffu, sorted_id, (lane - a.init_blocks) & 31);
  int v = -1;
  if (lane < a.init_blocks)
    v = lane;
  else if (lane < a.init_blocks + W)
    v = from_win;
  else if (lane < a.top_k)
    v = r - a.local_blocks + 1 + (lane - a.init_blocks - W);
  if (lane < kTopK) out[lane] = v;
}

cudaError_t launch_select(const SelectArgs& a0, cudaStream_t s) {
  SelectArgs a = a0;
  const int64_t nrows = static_cast<int64_t>(a.batch) * a.q_len * a.groups;
  if (nrows == 0) return cudaSuccess;
  if (a.max_blocks > 32 * 32) {  // long rows: a CTA per row
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(nrows));
    cfg.blockDim = dim3(kLongWarps * 32);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, select_long_kernel, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  // stage rows of up to 4096 candidates in shared memory (64 KB for 4 warps); longer rows
  // are read from L2 on each pass
  a.row_cap = a.max_blocks < 4096 ? a.max_blocks : 4096;
  const size_t smem = static_cast<size_t>(kSelWarps) * a.row_cap * sizeof(uint32_t);
  // rows of up to 768 candidates (e.g. chunked prefill on a 96K context) keep 24 candidates
  // per lane in registers instead of 32: fewer registers, more rows in flight per SM
  const bool short_rows = a.max_blocks <= 32 * 24;
  const void* kern = short_rows ? reinterpret_cast<const void*>(select_kernel<24>)
                                : reinterpret_cast<const void*>(select_kernel<32>);
  cudaError_t e = ensure_dynamic_smem(kern, smem);
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
  e = short_rows ? cudaLaunchKernelEx(&cfg, select_kernel<24>, a) : cudaLaunchKernelEx(&cfg, select_kernel<32>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace msa
