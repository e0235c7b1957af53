// msa_sparse_attn_decode_noalloc: the sparse-attention stage for callers that cannot hand the
// library a workspace.
//
// Some callers cannot call cudaMalloc at all, or not at the moment they decode.  Examples: a
// plugin running inside a host application that owns every byte of device memory through its
// own pool, and code that must not allocate between decode steps.  For them this entry point
// keeps its scratch (the split-K partial states and the device error word) in a fixed
// library-owned device array instead of a caller workspace.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes (8 MiB).  Every GPU
// that loads the library holds it until the process exits.  In host code the array's name is
// only a host-side stand-in, so the device address is looked up with cudaGetSymbolAddress,
// once per device, with that device current, on the first call made on that device.  Its
// first 4 bytes are the device error word of the last call, which
// msa_noalloc_read_device_error copies out.
#include <mutex>

#include "../../include/msa.h"
#include "api_internal.h"
#include "msa_kernels.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

void* g_noalloc_ptr[kNoAllocMaxDevices] = {};
std::mutex g_noalloc_mu;

// Device address of the scratch array on the current device (set-up on first use).
msa_status_t noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return MSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MSA_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return MSA_OK;
}

}  // namespace

extern "C" msa_status_t msa_sparse_attn_decode_noalloc(const msa_config_t* cfg, const msa_cache_t* cache,
                                                       const msa_batch_t* batch, const uint8_t* q,
                                                       const int32_t* selection, uint16_t* out, float* lse,
                                                       void* stream) {
  // 0 means an invalid configuration or batch: the regular entry point names the error
  // (it validates them before it looks at the workspace)
  if (msa_workspace_bytes(MSA_OP_SPARSE_ATTN, cfg, batch) == 0)
    return msa_sparse_attn_decode(cfg, cache, batch, q, selection, out, lse, nullptr, 0, stream);
  // this entry point always runs the query-major team kernel, whose scratch does not grow
  // with the batch
  if (msa::team_attn_workspace_bytes() > kNoAllocScratchBytes) return MSA_ERR_WORKSPACE;
  void* scratch = nullptr;
  msa_status_t st = noalloc_scratch(&scratch);
  if (st != MSA_OK) return st;
  // the error word (the array's first 4 bytes) is zeroed on the stream after validation, just
  // before the launch, so that it reports this call alone; the partial states are written
  // before they are read
  return msa::sparse_attn_entry(cfg, cache, batch, q, selection, out, lse, scratch, kNoAllocScratchBytes, stream,
                                false, true);
}

extern "C" msa_status_t msa_noalloc_read_device_error(uint32_t* flags, void* stream) {
  if (flags == nullptr) return MSA_ERR_INVALID_ARG;
  void* scratch = nullptr;
  msa_status_t st = noalloc_scratch(&scratch);
  if (st != MSA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(flags, scratch, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return MSA_ERR_CUDA;
  return MSA_OK;
}
