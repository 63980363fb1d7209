// Device helpers shared by the kernels: activation math, bf16 packing, status reporting,
// and the bounded wait on an mbarrier.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

namespace tpk {

// ------------------------------------------------------------------ activation
// GeLU in its exact (erf) form and its derivative, with the normal tail computed once:
//   Phi(-|h|) = erfc(z) / 2,  z = |h| / sqrt 2,  erfc(z) ~ t Q(t) exp(-z^2),  t = 1 / (1 + p z),
// the form of Abramowitz & Stegun, Handbook of Mathematical Functions, 7.1.26, with p = 1/2 and
// Q of degree 8 fitted for RELATIVE error (fit_normal_tail.py, beside this file: t Q(t) is
// within 2.1e-7 of the scaled function exp(z^2) erfc(z) for every z >= 0, so Phi(h) keeps its
// relative accuracy far into the negative tail, where GeLU(h) = h Phi(h) is tiny; 7.1.26's
// own degree-4 coefficients are fitted for absolute error and drift to 38 % relative error as
// z grows). exp(-z^2) = exp(-h^2 / 2) is also the normal density's exponential, so GeLU' costs
// one exponential and one reciprocal.
constexpr float kTailP = 0.35355339059327373f;  // p / sqrt 2: t = 1 / (1 + kTailP |h|)
constexpr float kTailQ0 = 2.820921728e-01f, kTailQ1 = 2.822133577e-01f,
                kTailQ2 = 2.448138215e-01f, kTailQ3 = 1.935501536e-01f,
                kTailQ4 = 9.956123732e-04f, kTailQ5 = 2.288727022e-01f,
                kTailQ6 = -4.361299399e-01f, kTailQ7 = 2.560270581e-01f,
                kTailQ8 = -5.243482750e-02f;

struct NormalTail {
  float cdf;  // Phi(h)
  float e;    // exp(-h^2 / 2)
};

__device__ __forceinline__ NormalTail normal_tail(float h) {
  // fast division (2 ulp): the divisor 1 + p |h| / sqrt 2 lies in [1, 2^126)
  const float t = __fdividef(1.0f, fmaf(kTailP, fabsf(h), 1.0f));
  float q = fmaf(t, kTailQ8, kTailQ7);
  q = fmaf(t, q, kTailQ6);
  q = fmaf(t, q, kTailQ5);
  q = fmaf(t, q, kTailQ4);
  q = fmaf(t, q, kTailQ3);
  q = fmaf(t, q, kTailQ2);
  q = fmaf(t, q, kTailQ1);
  q = fmaf(t, q, kTailQ0);
  const float e = __expf((-0.5f * h) * h);
  const float lower = 0.5f * (t * q) * e;  // Phi(-|h|)
  return {h >= 0.0f ? 1.0f - lower : lower, e};
}

// GeLU(h) = h * Phi(h).
__device__ __forceinline__ float gelu_erf(float h) { return h * normal_tail(h).cdf; }

// d/dh GeLU(h) = Phi(h) + h * phi(h), phi(h) = exp(-h^2 / 2) / sqrt(2 pi).
__device__ __forceinline__ float gelu_erf_grad(float h) {
  const NormalTail n = normal_tail(h);
  return fmaf(h * 0.3989422804014327f, n.e, n.cdf);
}

// The same two functions for two values at once with Blackwell's paired fp32 instructions
// (__ffma2_rn, __fmul2_rn, __fadd2_rn: each half rounded exactly as the scalar operation), for
// the epilogues that are bound by instruction issue. Every operation and its order are those
// of normal_tail, gelu_erf and gelu_erf_grad, so the results are bit-identical to them; the
// exponential and the fast reciprocal stay per value.
__device__ __forceinline__ float2 splat2(float a) { return make_float2(a, a); }

__device__ __forceinline__ void normal_tail2(float2 h, float2& cdf, float2& e) {
  const float2 d = __ffma2_rn(splat2(kTailP), make_float2(fabsf(h.x), fabsf(h.y)), splat2(1.0f));
  const float2 t = make_float2(__fdividef(1.0f, d.x), __fdividef(1.0f, d.y));
  float2 q = __ffma2_rn(t, splat2(kTailQ8), splat2(kTailQ7));
  q = __ffma2_rn(t, q, splat2(kTailQ6));
  q = __ffma2_rn(t, q, splat2(kTailQ5));
  q = __ffma2_rn(t, q, splat2(kTailQ4));
  q = __ffma2_rn(t, q, splat2(kTailQ3));
  q = __ffma2_rn(t, q, splat2(kTailQ2));
  q = __ffma2_rn(t, q, splat2(kTailQ1));
  q = __ffma2_rn(t, q, splat2(kTailQ0));
  const float2 nh2 = __fmul2_rn(__fmul2_rn(splat2(-0.5f), h), h);
  e = make_float2(__expf(nh2.x), __expf(nh2.y));
  const float2 lower = __fmul2_rn(__fmul2_rn(splat2(0.5f), __fmul2_rn(t, q)), e);
  const float2 upper = __fadd2_rn(splat2(1.0f), make_float2(-lower.x, -lower.y));
  cdf = make_float2(h.x >= 0.0f ? upper.x : lower.x, h.y >= 0.0f ? upper.y : lower.y);
}

__device__ __forceinline__ float2 gelu_erf2(float2 h) {
  float2 cdf, e;
  normal_tail2(h, cdf, e);
  return __fmul2_rn(h, cdf);
}

__device__ __forceinline__ float2 gelu_erf_grad2(float2 h) {
  float2 cdf, e;
  normal_tail2(h, cdf, e);
  return __ffma2_rn(__fmul2_rn(h, splat2(0.3989422804014327f)), e, cdf);
}

// ------------------------------------------------------------------ L2 prefetch
// Ask L2 for `bytes` bytes of global memory from ptr (16-byte aligned, a multiple of 16 bytes).
__device__ __forceinline__ void prefetch_l2(const void* ptr, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(__cvta_generic_to_global(ptr)),
               "r"(bytes)
               : "memory");
}

// ------------------------------------------------------------------ bf16 packing
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
  return __bfloat1622float2(v);
}

__device__ __forceinline__ float bf16_to_f32(uint16_t u) {
  return __uint_as_float(static_cast<uint32_t>(u) << 16);
}

// ------------------------------------------------------------------ status + timeouts
// Record the first error code in the workspace status word (later codes are dropped).
__device__ __forceinline__ void report_status(int* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity of the mbarrier at shared address `bar` has
// completed. Gives up after `limit_ns` nanoseconds of global time and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++spins & 255u) == 0u && global_ns() - t0 > limit_ns) return false;
  }
}

// The same wait for a role of a warp-specialised kernel that must also notice another role's
// failure: 1 when the phase has completed, 0 when the CTA's abort flag went up first, -1 after
// `limit_ns`. The flag is read only while the wait actually polls, so a wait that succeeds at
// once costs one try_wait.
__device__ __forceinline__ int mbar_wait_or_abort(uint32_t bar, uint32_t parity,
                                                  const volatile int* abort_flag,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return 1;
  const uint64_t t0 = global_ns();
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return 1;
    if (*abort_flag) return 0;
    if ((++spins & 255u) == 0u && global_ns() - t0 > limit_ns) return -1;
  }
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Default limit of every wait inside a GEMM: far above any tile's time (a tile of the
// largest workload runs well under a millisecond) and short enough to end a stuck launch.
constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s

}  // namespace tpk
