// Device-side building blocks of the MSA kernels (sm_103a): NVFP4/FP8 conversions,
// warp-level tensor-core MMA, mbarrier + bulk-copy staging with bounded waits.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/msa.h"
#include "msa_kernels.h"

namespace msa {

constexpr int kBlock = 128;                    // tokens per block / cache page
constexpr int kDim = 128;                      // head_dim == index_dim
constexpr int kRowBytes = kDim / 2;            // packed E2M1 bytes per row
constexpr int kRowScales = kDim / 16;          // E4M3 scales per row
constexpr int kPageData = kBlock * kRowBytes;  // 8192
constexpr int kPageScale = kBlock * kRowScales;// 1024
constexpr int kTopK = 16;
constexpr uint32_t kSpinLimit = kDefaultSpinLimit;  // default bound on every mbarrier wait loop

__device__ __forceinline__ void flag_error(uint32_t* err, uint32_t bit) {
  if (err != nullptr) atomicOr(err, bit);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ conversions
// Four packed E2M1 pairs (the four bytes of w) -> four f16x2 (exact).  In each output the
// low half is the byte's low nibble.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                uint32_t& r3) {
  asm("{\n"
      " .reg .b8 b0, b1, b2, b3;\n"
      " mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n"
      " cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n"
      " cvt.rn.f16x2.e2m1x2 %3, b3;\n"
      "}"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(w));
}

// Low two bytes of w (two E4M3 codes) -> f16x2, low byte -> low half (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w) {
  uint32_t r;
  asm("{\n"
      " .reg .b16 lo, hi;\n"
      " mov.b32 {lo, hi}, %1;\n"
      " cvt.rn.f16x2.e4m3x2 %0, lo;\n"
      "}"
      : "=r"(r)
      : "r"(w));
  return r;
}

// E4M3 code in byte `sel` of w, broadcast to both halves of an f16x2.
__device__ __forceinline__ uint32_t e4m3_bcast_f16x2(uint32_t w, int sel) {
  return e4m3x2_to_f16x2(__byte_perm(w, 0, sel * 0x1111));
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// ------------------------------------------------------------------ tensor cores
// D += A(16x16, row) * B(16x8, col), f16 inputs, f32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 b16 matrix held in the standard fragment layout across the warp.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(x));
  return d;
}

// ------------------------------------------------------------------ programmatic dependent launch
// Kernels launched with programmatic stream serialization may start while the previous
// kernel on the stream is still finishing; this waits until it has completed and its
// memory is visible (a no-op when there is no such kernel).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the next kernel on the stream (launched with programmatic stream serialization) be
// scheduled once every CTA of this grid has called it or exited; that kernel still reads
// nothing of this one's before its grid_dependency_wait, which waits for this grid's
// completion.  Called after this kernel's own grid_dependency_wait, so that everything
// before this kernel on the stream has completed by the time the next one starts.
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ mbarrier + bulk copy
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n"
      "}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on one phase: at most `limit` polls; false if it gave up (the caller flags
// MSA_DEVERR_TIMEOUT).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit = kSpinLimit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// The same, called by a whole warp; the verdict is made warp-uniform so that the warp's
// later shuffles never diverge.  (Every lane waits: a variant where lane 0 alone polls and
// broadcasts was measured slower, its divergent loop costing more than the shared polls.)
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, uint32_t limit = kSpinLimit) {
  const bool ok = mbar_wait(bar, parity, limit);
  return __all_sync(0xffffffffu, ok) != 0;
}

// Global -> shared bulk copy completing on `bar` (both addresses 16-byte aligned, bytes a
// multiple of 16).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// L2 cache policy for data read once per call: its lines are the first to be evicted.
// Streaming the index-key pages with it measured 13 % faster on GB300 than the default
// policy (the default lets 330 MB of single-use lines push each other and the rest out).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// bulk_g2s with an L2 cache policy (from createpolicy).
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

__device__ __forceinline__ uint2 lds64(const void* p) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(smem_u32(p)));
  return v;
}

__device__ __forceinline__ uint32_t lds16(const void* p) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(smem_u32(p)));
  return v;
}

__device__ __forceinline__ uint32_t lds8(const void* p) {
  unsigned short v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(smem_u32(p)));
  return v;
}

// Block pooling of key scores into one score per block ("MiniMax M3 x vLLM：百万 token 多模态推理的
// Day-0 部署", §Prefill 执行 step 2: a block-level rule such as max or log-sum-exp).  The running
// state of one column: the maximum m and, for log-sum-exp, s = sum over the values seen of
// e^{x - m}; -inf values (keys not visible) count as absent.  lse is warp-uniform.
struct PoolState {
  float m, s;
};

__device__ __forceinline__ void pool_add(PoolState& p, float a, float b, bool lse) {
  const float mn = fmaxf(p.m, fmaxf(a, b));
  if (lse && mn != -INFINITY) p.s = p.s * expf(p.m - mn) + expf(a - mn) + expf(b - mn);
  p.m = mn;
}

// Combines the states of lanes lane and lane ^ mask (all 32 lanes call it).
__device__ __forceinline__ void pool_merge_xor(PoolState& p, int mask, bool lse) {
  const float mo = __shfl_xor_sync(0xffffffffu, p.m, mask);
  const float mn = fmaxf(p.m, mo);
  if (lse) {
    const float so = __shfl_xor_sync(0xffffffffu, p.s, mask);
    if (mn != -INFINITY) p.s = p.s * expf(p.m - mn) + so * expf(mo - mn);
  }
  p.m = mn;
}

// The block score: m, or m + ln s (natural log); -inf for a block with no visible key.
__device__ __forceinline__ float pool_result(const PoolState& p, bool lse) {
  return (lse && p.m != -INFINITY) ? p.m + logf(p.s) : p.m;
}

// Order of float scores as unsigned integers: larger float -> larger key, -0 == +0,
// NaN below -inf.
__device__ __forceinline__ uint32_t score_order(float f) {
  if (f != f) return 0u;
  if (f == 0.0f) f = 0.0f;
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace msa
