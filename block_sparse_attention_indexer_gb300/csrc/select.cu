// Stage 2 of MSA decode: top-k block selection with the most recent block forced, one warp
// per (sequence, query token, KV group) row.  The per-row routine and its rules are in
// select_row.cuh.
#include "msa_kernels.h"
#include "select_row.cuh"

namespace msa {

constexpr int64_t kSplitMaxRows = 2048;  // rows up to which a CTA per row beats a warp per row

template <int KPL>
__global__ void __launch_bounds__(kSelWarps * 32) select_kernel(const SelectArgs a) {
  extern __shared__ __align__(16) uint32_t sord_all[];  // [kSelWarps][row_cap] staged score orders
  __shared__ __align__(16) uint64_t buf[kSelWarps][kSelCap];
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

// One CTA per row, for rows longer than 1,024 candidates (long contexts: 8 warps) and for
// batches with few rows (decode: 4 warps, so that the row's loads and ranking are split
// four ways instead of waiting on one warp).  Each warp takes the best of a contiguous
// share of the candidates (the row's winners are among the union of the shares' winners,
// at most NW x 16 keys, left in shared memory); the first warp ranks those exact keys -- each
// lane holds NW / 2 of them and counts the larger keys, read back from shared memory as
// broadcast 16-byte loads -- each of the W winners writes its block id at its rank, and each
// then takes its ascending place, the number of winners with a smaller id.
//
// On the decode step (a.sel_pages set) the CTA also stages its sequence's block-table row in
// shared memory and writes the page of every selected block, so that the attention kernel
// reads each entry's page with its block id instead of looking it up after reading the
// selection; with a.inputs_early the sequence length and the table row are read before the
// wait on the indexer, while its last CTAs are still running.
template <int NW, int KPL>
__global__ void __launch_bounds__(NW * 32) select_split_kernel(const SelectArgs a) {
  __shared__ __align__(16) uint64_t buf[NW][kSelCap / 8];
  __shared__ __align__(16) uint64_t part[NW][kTopK];
  __shared__ __align__(16) int32_t win_ids[kTopK];
  extern __shared__ int32_t tab[];  // [max_blocks] when pages are written
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = blockIdx.x;
  const int b = static_cast<int>(row / (static_cast<int64_t>(a.q_len) * a.groups));
  const bool stage_tab = a.sel_pages != nullptr;
  const int32_t* tab_src = a.block_table + static_cast<int64_t>(b) * a.max_blocks;
  int L = 0;
  if (a.inputs_early) {
    L = a.seq_lens[b];
    if (stage_tab)
      for (int i = threadIdx.x; i < a.max_blocks; i += NW * 32) tab[i] = __ldg(tab_src + i);
  }
  grid_dependency_wait();
  grid_dependents_launch();
  if (!a.inputs_early) {
    L = a.seq_lens[b];
    if (stage_tab)
      for (int i = threadIdx.x; i < a.max_blocks; i += NW * 32) tab[i] = __ldg(tab_src + i);
  }
  if (stage_tab) __syncthreads();
  select_split_row<NW, KPL>(a, row, L, warp, lane, buf, part, win_ids, stage_tab ? tab : nullptr,
                            [] { __syncthreads(); });
}

// ------------------------------------------------------------------------------------------
// Decode context parallelism ("vLLM liefert Day-0-Unterstützung für MiniMax-M3.1-Flash",
// §NVFP4-Indexer-DCP): each shard scores the blocks it holds and keeps, per (sequence, token,
// group), its best top_k - 1 blocks before the recent one; the owner merges the shards' lists
// and adds the recent block.  The merge is exact: under one strict order (score descending,
// index ascending, NaN below -inf) the best W of a union of disjoint sets are among the union
// of each set's best W.

// Shard-local candidates of every row: the best W = top_k - 1 of the blocks [lo, min(hi, r)),
// in rank order (best first), with their scores; -1 / -inf past the end of the list.
template <int KPL>
__global__ void __launch_bounds__(kSelWarps * 32) dcp_local_kernel(const SelectArgs a, int lo, int hi,
                                                                   float* cand_scores, int32_t* cand_blocks) {
  __shared__ __align__(16) uint64_t buf[kSelWarps][kSelCap / 8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dependency_wait();
  grid_dependents_launch();
  const int64_t nrows = static_cast<int64_t>(a.batch) * a.q_len * a.groups;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kSelWarps + warp;
  if (row >= nrows) return;
  const int b = static_cast<int>(row / (static_cast<int64_t>(a.q_len) * a.groups));
  const int t = static_cast<int>((row / a.groups) % a.q_len);
  const int L = a.seq_lens[b];
  const float* sc = a.block_scores + row * a.max_blocks;
  int id = -1, W = 0;
  if (L >= a.q_len && L > 0 && L <= static_cast<int64_t>(a.max_blocks) * kBlock) {
    const int r = (L - a.q_len + t) / kBlock;
    const int c1 = min(hi, r), nc = c1 - lo;
    W = max(0, min(a.top_k - 1, nc));
    if (W == nc)  // every candidate of the shard is kept
      id = lane < W ? lo + lane : -1;
    else if (W > 0)
      id = top_blocks_warp<KPL>(sc, lo, c1, W, lane, nullptr, 0, buf[warp], kSelCap / 8);
  }
  // rank order: exact keys order(score) << 32 | ~id, sorted descending across the warp
  const uint64_t key = (lane < W && id >= 0)
                           ? (static_cast<uint64_t>(score_order(__ldcg(sc + id))) << 32) |
                                 static_cast<uint64_t>(0xffffffffu - static_cast<uint32_t>(id))
                           : 0ull;
  const uint64_t k = warp_sort_desc_u64(key, lane);
  if (lane < kTopK - 1) {
    const int n = k != 0ull ? static_cast<int>(0xffffffffu - static_cast<uint32_t>(k)) : -1;
    cand_blocks[row * (kTopK - 1) + lane] = n;
    cand_scores[row * (kTopK - 1) + lane] = n >= 0 ? __ldcg(sc + n) : -INFINITY;
  }
}

// The owner's merge: the best W = top_k - 1 of the S shards' candidates (at most 8 x 15, each
// lane holding up to four exact keys, ranked by comparing every pair across the warp) plus the
// recent block, ascending; rows whose recent block is r <= top_k - 1 select every block 0 .. r.
__global__ void __launch_bounds__(kSelWarps * 32) dcp_merge_kernel(const SelectArgs a, int S, const float* cand_scores,
                                                                   const int32_t* cand_blocks) {
  constexpr int kKeys = (kDcpShardsMax * (kTopK - 1) + 31) / 32;  // 4
  __shared__ int32_t win[kSelWarps][kTopK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
  if (r + 1 <= a.top_k) {
    if (lane < kTopK) out[lane] = lane <= r ? lane : -1;
    return;
  }
  const int W = a.top_k - 1;
  const int nk = S * (kTopK - 1);
  const int64_t per_shard = nrows * (kTopK - 1);
  uint64_t key[kKeys];
#pragma unroll
  for (int i = 0; i < kKeys; ++i) {
    const int c = 32 * i + lane;  // candidate c: shard c / 15, entry c % 15
    key[i] = 0ull;
    if (c < nk) {
      const int64_t at = (c / (kTopK - 1)) * per_shard + row * (kTopK - 1) + c % (kTopK - 1);
      const int n = cand_blocks[at];
      if (n >= 0)
        key[i] = (static_cast<uint64_t>(score_order(cand_scores[at])) << 32) |
                 static_cast<uint64_t>(0xffffffffu - static_cast<uint32_t>(n));
    }
  }
  int rank[kKeys];
#pragma unroll
  for (int i = 0; i < kKeys; ++i) rank[i] = 0;
#pragma unroll
  for (int i2 = 0; i2 < kKeys; ++i2)
#pragma unroll 4
    for (int j = 0; j < 32; ++j) {
      const uint64_t other = shfl_u64(key[i2], j);
#pragma unroll
      for (int i = 0; i < kKeys; ++i) rank[i] += other > key[i] ? 1 : 0;
    }
#pragma unroll
  for (int i = 0; i < kKeys; ++i)
    if (key[i] != 0ull && rank[i] < W) win[warp][rank[i]] = static_cast<int>(0xffffffffu - static_cast<uint32_t>(key[i]));
  __syncwarp();
  // the W winners ascending (all below r), then r
  const int sorted = warp_sort_asc_i32(lane < W ? win[warp][lane] : 0x7fffffff, lane);
  if (lane < kTopK) out[lane] = lane < W ? sorted : (lane == W ? r : -1);
}

cudaError_t launch_dcp_local(const SelectArgs& a, int lo, int hi, float* cand_scores, int32_t* cand_blocks,
                             cudaStream_t s) {
  const int64_t nrows = static_cast<int64_t>(a.batch) * a.q_len * a.groups;
  if (nrows == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((nrows + kSelWarps - 1) / kSelWarps));
  cfg.blockDim = dim3(kSelWarps * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // shards of up to 1,024 candidates keep them in registers; longer ones read from L2
  cudaError_t e = cudaLaunchKernelEx(&cfg, dcp_local_kernel<32>, a, lo, hi, cand_scores, cand_blocks);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_dcp_merge(const SelectArgs& a, int S, const float* cand_scores, const int32_t* cand_blocks,
                             cudaStream_t s) {
  const int64_t nrows = static_cast<int64_t>(a.batch) * a.q_len * a.groups;
  if (nrows == 0) return cudaSuccess;
  if (S < 1 || S > kDcpShardsMax) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((nrows + kSelWarps - 1) / kSelWarps));
  cfg.blockDim = dim3(kSelWarps * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, dcp_merge_kernel, a, S, cand_scores, cand_blocks);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

namespace {
// long rows, or few rows (decode): a CTA per row; many rows (chunked prefill): a warp per row
bool cta_per_row(const SelectArgs& a) {
  const int64_t nrows = static_cast<int64_t>(a.batch) * a.q_len * a.groups;
  return a.max_blocks > 32 * 32 || nrows <= kSplitMaxRows;
}
}  // namespace

bool select_writes_pages(const SelectArgs& a) {
  return a.sel_pages != nullptr && a.block_table != nullptr && cta_per_row(a) && a.max_blocks <= kSelTableCap;
}

cudaError_t launch_select(const SelectArgs& a0, cudaStream_t s) {
  SelectArgs a = a0;
  const int64_t nrows = static_cast<int64_t>(a.batch) * a.q_len * a.groups;
  if (nrows == 0) return cudaSuccess;
  if (!select_writes_pages(a)) a.sel_pages = nullptr;
  const bool long_rows = a.max_blocks > 32 * 32;
  if (cta_per_row(a)) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(nrows));
    cfg.blockDim = dim3((long_rows ? 8 : 4) * 32);
    // the staged table row: at most kSelTableCap entries (16 KB), under the default limit
    cfg.dynamicSmemBytes = a.sel_pages != nullptr ? static_cast<size_t>(a.max_blocks) * sizeof(int32_t) : 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // shares of at most 4096 / 8 = 512 (8 warps x 16 per lane) or 1024 / 4 = 256 (4 x 8)
    // candidates stay in registers; longer rows read their shares from L2
    cudaError_t e = long_rows ? cudaLaunchKernelEx(&cfg, select_split_kernel<8, 16>, a)
                              : cudaLaunchKernelEx(&cfg, select_split_kernel<4, 8>, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  // stage rows of up to 4096 candidates in shared memory (64 KB for 4 warps); longer rows
  // are read from L2 on each pass
  a.row_cap = a.max_blocks < 4096 ? a.max_blocks : 4096;
  const size_t smem = static_cast<size_t>(kSelWarps) * a.row_cap * sizeof(uint32_t);
  // shorter rows keep fewer candidates per lane in registers (24 up to 768 candidates, e.g.
  // chunked prefill on a 96K context; 18 up to 576, a 72K context): fewer registers and
  // instructions per row, more rows in flight per SM
  const int kpl = a.max_blocks <= 32 * 18 ? 18 : (a.max_blocks <= 32 * 24 ? 24 : 32);
  const void* kern = kpl == 18 ? reinterpret_cast<const void*>(select_kernel<18>)
                               : (kpl == 24 ? reinterpret_cast<const void*>(select_kernel<24>)
                                            : reinterpret_cast<const void*>(select_kernel<32>));
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
  e = kpl == 18   ? cudaLaunchKernelEx(&cfg, select_kernel<18>, a)
      : kpl == 24 ? cudaLaunchKernelEx(&cfg, select_kernel<24>, a)
                  : cudaLaunchKernelEx(&cfg, select_kernel<32>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace msa
