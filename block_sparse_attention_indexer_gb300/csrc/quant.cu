// NVFP4 quantise-and-insert of cache rows, and FP8 E4M3 encoding of queries.
//
// NVFP4: E2M1 values with one E4M3 scale per 16 elements ("vLLM liefert
// Day-0-Unterstützung für MiniMax-M3.1-Flash", §Was ist neu in der MiniMax-M3.1-Architektur;
// the write into the cache is the epilogue of §QKV GEMM + Norm + RoPE + KV-Insert-Fusion).
// Rounding: scale = E4M3_rn_satfinite(amax / 6), element = E2M1_rn_satfinite(x / scale),
// both divisions correctly rounded float32, a zero scale gives zero codes.
#include "msa_device.cuh"
#include "msa_kernels.h"

namespace msa {

// Four E2M1 codes pairs from eight floats: byte i = code(v[2i]) | code(v[2i+1]) << 4.
__device__ __forceinline__ uint32_t f32x8_to_e2m1x8(const float* v) {
  uint32_t w;
  asm("{\n"
      " .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n"
      "}"
      : "=r"(w)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return w;
}

// E4M3 code of one float (round to nearest even, saturating).
__device__ __forceinline__ uint32_t f32_to_e4m3(float x) {
  unsigned short h;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(0.0f), "f"(x));
  return h & 0xFFu;
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
  uint32_t h2 = e4m3x2_to_f16x2(code);
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

// x / d correctly rounded, given y = RN(1/d) for a finite d > 0: q = RN(x y) is within an ulp
// of x / d, r = x - d q is exact (one fma), and RN(q + r y) is the correctly rounded quotient
// (Markstein's correction).  Checked on the host against exact division for every float32
// significand of x and every divisor significand 1..15 (the E4M3 scales and 6): no
// difference.  The sign is copied from x so that -0 / d stays -0.
__device__ __forceinline__ float div_rn_by_recip(float x, float d, float y) {
  const float q = __fmul_rn(x, y);
  const float r = __fmaf_rn(-d, q, x);
  return copysignf(__fmaf_rn(r, y, q), x);
}

// The 16 inputs and the slot of group gt (= row * groups-per-row + grp) of token tok.  The
// inputs are read once: streaming loads (evict first), issued together with the slot's.
__device__ __forceinline__ void insert_load(const QuantArgs& a, int64_t tok, int64_t first, float4 (&v)[4],
                                            int64_t& slot) {
  const float4* src = reinterpret_cast<const float4*>(a.x) + 4 * first;
  slot = __ldg(a.slots + tok);
#pragma unroll
  for (int j = 0; j < 4; ++j) v[j] = __ldcs(src + j);
}

// Encodes one group and writes its 8 code bytes and its scale into the token's slot (nothing
// for a slot outside the pool).
__device__ __forceinline__ void insert_store(const QuantArgs& a, int gt, int gpr, const float4 (&in)[4], int64_t slot,
                                             int64_t cap, bool slots32) {
  if (slot < 0 || slot >= cap) return;
  const float v[16] = {in[0].x, in[0].y, in[0].z, in[0].w, in[1].x, in[1].y, in[1].z, in[1].w,
                       in[2].x, in[2].y, in[2].z, in[2].w, in[3].x, in[3].y, in[3].z, in[3].w};
  const int row = static_cast<int>(static_cast<uint32_t>(gt) / static_cast<uint32_t>(gpr));
  const int grp = gt - row * gpr;
  int64_t page;
  int off;
  if (slots32) {
    const uint32_t s32 = static_cast<uint32_t>(slot), bs = static_cast<uint32_t>(a.block_size);
    const uint32_t p32 = s32 / bs;
    page = p32;
    off = static_cast<int>(s32 - p32 * bs);
  } else {
    page = slot / a.block_size;
    off = static_cast<int>(slot - page * a.block_size);
  }
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
  // the divisions are correctly rounded either way; an infinite element (amax = inf) takes
  // the plain division, whose result the reciprocal form would turn into NaN
  const bool finite = isfinite(amax);
  constexpr float kInv6 = 1.0f / 6.0f;  // RN(1/6)
  const uint32_t scode = f32_to_e4m3(finite ? div_rn_by_recip(amax, 6.0f, kInv6) : __fdiv_rn(amax, 6.0f));
  const float scale = e4m3_to_f32(scode);
  uint2 packed = make_uint2(0u, 0u);
  if (scale > 0.0f) {
    float r[16];
    if (finite) {
      const float inv = __frcp_rn(scale);
#pragma unroll
      for (int j = 0; j < 16; ++j) r[j] = div_rn_by_recip(v[j], scale, inv);
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) r[j] = __fdiv_rn(v[j], scale);
    }
    packed.x = f32x8_to_e2m1x8(r);
    packed.y = f32x8_to_e2m1x8(r + 8);
  }
  const int64_t row_index = (page * a.rows_per_token + row) * a.block_size + off;
  *reinterpret_cast<uint2*>(a.data + row_index * (a.dim / 2) + grp * 8) = packed;
  a.scale[row_index * gpr + grp] = static_cast<uint8_t>(scode);
}

// One thread per 16-element group.  The groups of all tokens are numbered token-major (group
// gt of token tok is tok * groups-per-token + gt), so group g's inputs are the 64 bytes at
// x + 64 g: consecutive threads read consecutive bytes.  A grid of kInsertCtasPerSm CTAs an SM
// strides over the groups, and each thread loads its next group before it encodes the current
// one, so that its loads stay in flight while it computes; (token, gt) advance by the stride's
// quotient and remainder instead of a division per group.
constexpr int kInsertThreads = 256;
constexpr int kInsertCtasPerSm = 4;

__global__ void __launch_bounds__(kInsertThreads, kInsertCtasPerSm) nvfp4_insert_kernel(QuantArgs a) {
  const int gpr = a.dim / 16;              // groups per row
  const int gpt = a.rows_per_token * gpr;  // groups per token
  const int64_t total = a.n_tokens * gpt;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (g >= total) return;
  const int64_t cap = a.num_pages * a.block_size;
  const bool slots32 = cap <= 0x7fffffff;
  const int64_t dq = stride / gpt;
  const int dr = static_cast<int>(stride - dq * gpt);
  int64_t tok = g / gpt;
  int gt = static_cast<int>(g - tok * gpt);
  float4 cur[4];
  int64_t slot;
  insert_load(a, tok, g, cur, slot);
  for (;;) {
    const int64_t gn = g + stride;
    int64_t tokn = tok + dq;
    int gtn = gt + dr;
    if (gtn >= gpt) {
      gtn -= gpt;
      ++tokn;
    }
    const bool more = gn < total;
    float4 nxt[4];
    int64_t slotn = -1;
    if (more) insert_load(a, tokn, gn, nxt, slotn);
    insert_store(a, gt, gpr, cur, slot, cap, slots32);
    if (!more) break;
    g = gn;
    tok = tokn;
    gt = gtn;
    slot = slotn;
#pragma unroll
    for (int j = 0; j < 4; ++j) cur[j] = nxt[j];
  }
}

__global__ void fp8_quantize_kernel(const float* __restrict__ x, int64_t n, uint8_t* __restrict__ out) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    out[i] = static_cast<uint8_t>(f32_to_e4m3(x[i]));
}

cudaError_t launch_nvfp4_insert(const QuantArgs& a, int num_sms, cudaStream_t s) {
  if (a.n_tokens == 0) return cudaSuccess;
  const int64_t total = a.n_tokens * a.rows_per_token * (a.dim / 16);
  const int64_t needed = (total + kInsertThreads - 1) / kInsertThreads;
  const int64_t resident = static_cast<int64_t>(num_sms) * kInsertCtasPerSm;
  const int64_t blocks = needed < resident ? needed : resident;
  nvfp4_insert_kernel<<<static_cast<unsigned>(blocks), kInsertThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_fp8_quantize(const float* x, int64_t n, uint8_t* out, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (n + threads - 1) / threads;
  fp8_quantize_kernel<<<static_cast<unsigned>(blocks < 65535 * 16 ? blocks : 65535 * 16), threads, 0, s>>>(x, n,
                                                                                                            out);
  return cudaGetLastError();
}

}  // namespace msa
