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
// Q fitted for RELATIVE error (fit_normal_tail.py, beside this file), so that Phi(h) keeps its
// relative accuracy far into the negative tail, where GeLU(h) = h Phi(h) is tiny (7.1.26's own
// degree-4 coefficients are fitted for absolute error and drift to 38 % relative error as z
// grows). exp(-z^2) = exp(-h^2 / 2) is also the normal density's exponential, so GeLU' costs
// one exponential and one reciprocal. Two fits:
//  - degree 8 (t Q(t) within 2.1e-7 of exp(z^2) erfc(z) for every z >= 0) for the fp32 paths
//    (FFMA GEMM epilogues, the activation-gradient kernel), whose tolerance is 1e-5;
//  - degree 5 (within 5.1e-5) for the bf16 tensor-core epilogues, whose outputs are rounded
//    to bf16 (2^-9 relative) and whose instruction count sets the pace of short-K GEMMs.
// The coefficients below are Q's halved (exact in fp32), so that t Q(t) exp(-z^2) / 2 needs no
// separate multiplication.
constexpr float kTailP = 0.35355339059327373f;  // p / sqrt 2: t = 1 / (1 + kTailP |h|)
namespace tail8 {
constexpr float q0 = 0.5f * 2.820921728e-01f, q1 = 0.5f * 2.822133577e-01f,
                q2 = 0.5f * 2.448138215e-01f, q3 = 0.5f * 1.935501536e-01f,
                q4 = 0.5f * 9.956123732e-04f, q5 = 0.5f * 2.288727022e-01f,
                q6 = 0.5f * -4.361299399e-01f, q7 = 0.5f * 2.560270581e-01f,
                q8 = 0.5f * -5.243482750e-02f;
}  // namespace tail8
namespace tail5 {
constexpr float q0 = 0.5f * 2.820021294e-01f, q1 = 0.5f * 2.845312988e-01f,
                q2 = 0.5f * 2.286358539e-01f, q3 = 0.5f * 2.235169020e-01f,
                q4 = 0.5f * 6.513961987e-02f, q5 = 0.5f * -8.387641932e-02f;
}  // namespace tail5
constexpr float kInvSqrt2Pi = 0.3989422804014327f;

// Phi(-|h|) = lower and exp(-h^2 / 2) = e, degree-8 fit. GeLU and GeLU' then follow without a
// branch: GeLU(h) = max(h, 0) - |h| lower, GeLU'(h) = [h >= 0] + e (h / sqrt(2 pi) -+ t Q / 2)
// (the sign of t Q / 2 = lower / e opposite to h's), each with one final fused multiply-add.
// Both the step and the sign are taken from h's sign bit, so h = -0 gives GeLU'(0) = 1/2 too.
struct NormalTail {
  float tq;  // t Q(t) / 2 = Phi(-|h|) / exp(-h^2 / 2)
  float e;   // exp(-h^2 / 2)
};

__device__ __forceinline__ NormalTail normal_tail(float h) {
  using namespace tail8;
  // fast division (2 ulp): the divisor 1 + p |h| / sqrt 2 lies in [1, 2^126)
  const float t = __fdividef(1.0f, fmaf(kTailP, fabsf(h), 1.0f));
  float q = fmaf(t, q8, q7);
  q = fmaf(t, q, q6);
  q = fmaf(t, q, q5);
  q = fmaf(t, q, q4);
  q = fmaf(t, q, q3);
  q = fmaf(t, q, q2);
  q = fmaf(t, q, q1);
  q = fmaf(t, q, q0);
  return {t * q, __expf((-0.5f * h) * h)};
}

// GeLU(h) = h Phi(h) = max(h, 0) - |h| Phi(-|h|).
__device__ __forceinline__ float gelu_erf(float h) {
  const NormalTail n = normal_tail(h);
  return fmaf(-fabsf(h), n.tq * n.e, fmaxf(h, 0.0f));
}

// d/dh GeLU(h) = Phi(h) + h phi(h), phi(h) = exp(-h^2 / 2) / sqrt(2 pi).
__device__ __forceinline__ float gelu_erf_grad(float h) {
  const NormalTail n = normal_tail(h);
  return fmaf(n.e, fmaf(kInvSqrt2Pi, h, copysignf(n.tq, -h)), signbit(h) ? 0.0f : 1.0f);
}

// The bf16 epilogues' versions, two values at once with Blackwell's paired fp32 instructions
// (__ffma2_rn, __fmul2_rn: each half rounded as the scalar operation), degree-5 fit; the same
// formulas as above. The exponential and the fast reciprocal stay per value.
__device__ __forceinline__ float2 splat2(float a) { return make_float2(a, a); }

__device__ __forceinline__ void normal_tail2(float2 h, float2& tq, float2& e) {
  using namespace tail5;
  const float2 d = __ffma2_rn(splat2(kTailP), make_float2(fabsf(h.x), fabsf(h.y)), splat2(1.0f));
  const float2 t = make_float2(__fdividef(1.0f, d.x), __fdividef(1.0f, d.y));
  float2 q = __ffma2_rn(t, splat2(q5), splat2(q4));
  q = __ffma2_rn(t, q, splat2(q3));
  q = __ffma2_rn(t, q, splat2(q2));
  q = __ffma2_rn(t, q, splat2(q1));
  q = __ffma2_rn(t, q, splat2(q0));
  tq = __fmul2_rn(t, q);
  const float2 nh2 = __fmul2_rn(__fmul2_rn(splat2(-0.5f), h), h);
  e = make_float2(__expf(nh2.x), __expf(nh2.y));
}

__device__ __forceinline__ float2 gelu_erf2(float2 h) {
  float2 tq, e;
  normal_tail2(h, tq, e);
  return __ffma2_rn(make_float2(-fabsf(h.x), -fabsf(h.y)), __fmul2_rn(tq, e),
                    make_float2(fmaxf(h.x, 0.0f), fmaxf(h.y, 0.0f)));
}

__device__ __forceinline__ float2 gelu_erf_grad2(float2 h) {
  float2 tq, e;
  normal_tail2(h, tq, e);
  const float2 s = __ffma2_rn(splat2(kInvSqrt2Pi), h,
                              make_float2(copysignf(tq.x, -h.x), copysignf(tq.y, -h.y)));
  return __ffma2_rn(e, s, make_float2(signbit(h.x) ? 0.0f : 1.0f, signbit(h.y) ? 0.0f : 1.0f));
}

// ------------------------------------------------------------------ programmatic dependent launch
// A kernel launched with programmatic stream serialisation may start while the kernel before it
// on the stream is still running: it does its set-up (barriers, TMEM, shared memory), then
// waits here until that kernel has completed and its memory operations are visible, before its
// first global load or store. Without that launch attribute the wait returns at once.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Lets the next kernel on the stream be scheduled (it still waits in grid_dependency_wait for
// this one to complete); called by every CTA once it is running, after its own wait.
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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

// Non-blocking test of the same phase: returns at once (try_wait may suspend the thread until
// the phase completes or a system-dependent time limit passes, which is what a wait wants but
// not a look-ahead placed between two instruction issues).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
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
