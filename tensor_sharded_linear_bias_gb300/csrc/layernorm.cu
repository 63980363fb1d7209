// LayerNorm with the hidden dimension split into tp_degree column shards ("Tensor Parallelism:
// principle and practice", section 4.2: each device computes the mean and variance of its own
// part and the statistics are synchronised by an All-Reduce). All shards live on this GPU as
// separate buffers; the All-Reduce of the statistics is a combination, in shard order, inside
// the block that owns the token row.
//
// Forward, one block per token row, its warps taking the shards in turn (warp w: shards w,
// w + 8, ...):
//   1. per shard i: every lane sums x - k_i and (x - k_i)^2 over its elements (k_i = the
//      shard's first element of the row: a shift that keeps the sums well conditioned), the
//      warp adds the lanes in a fixed butterfly, giving the shard's count, mean and M2;
//   2. the shards' (count, mean, M2) are combined in shard order 0..n-1 with the pairwise
//      update of Chan, Golub and LeVeque ("Updating formulae and a pairwise algorithm for
//      computing sample variances", 1979): the row's mean and biased variance;
//   3. y = (x - mean) * rstd * gamma + beta for every shard (the row's bytes are re-read from
//      L1/L2), and mean, rstd are stored for the backward.
// Backward dX, one block per row likewise: the row statistics sum(dY*gamma) and
// sum(dY*gamma*xhat) are summed per shard, then over the shards in order, and
// dX = rstd * (g - (s1 + xhat s2) / H).
// Backward dgamma, dbeta: column sums over the tokens, split over the warps of a block and the
// blocks of a cluster, combined in warp and block order (distributed shared memory for the
// blocks): deterministic, no atomics.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "device_common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace tpk {
namespace {

constexpr int kLnWarps = 8;  // warps per block (one token row per block, warps over its shards)
constexpr int kUnrollFwd = 4;  // 16-byte loads in flight per lane: forward (one operand)
constexpr int kUnrollBwd = 4;  // ... and backward (two operands)

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// VEC consecutive elements of one row: one 16-byte access when VEC * sizeof(T) == 16 (the
// alignment makes the compiler emit a single vector load or store).
template <typename T, int VEC>
struct alignas(sizeof(T) * VEC) Vec {
  T v[VEC];
};
template <typename T, int VEC>
__device__ __forceinline__ void load_vec(const T* p, float* out) {
  const Vec<T, VEC> r = *reinterpret_cast<const Vec<T, VEC>*>(p);
#pragma unroll
  for (int j = 0; j < VEC; ++j) out[j] = to_f(r.v[j]);
}
template <typename T, int VEC>
__device__ __forceinline__ void store_vec(T* p, const float* in) {
  Vec<T, VEC> r;
#pragma unroll
  for (int j = 0; j < VEC; ++j) r.v[j] = from_f<T>(in[j]);
  *reinterpret_cast<Vec<T, VEC>*>(p) = r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

struct LnParams {
  const void* X[kMaxShards];
  const void* gamma[kMaxShards];
  const void* beta[kMaxShards];
  void* Y[kMaxShards];   // forward output / backward dX
  const void* dY[kMaxShards];
  float* dgamma[kMaxShards];
  float* dbeta[kMaxShards];
  float* mean;
  float* rstd;
  long long T, Hs;
  int n;
  float eps;
};

template <typename T, int VEC>
__global__ void __launch_bounds__(kLnWarps * 32) ln_forward_kernel(const __grid_constant__ LnParams p) {
  __shared__ float stat[kMaxShards][2];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, W = blockDim.x >> 5;
  const long long t = blockIdx.x;
  const long long row = t * p.Hs;
  // 1: every warp takes shards warp, warp + W, ...: the shard's shifted sums -> (mean_i, M2_i)
  for (int i = warp; i < p.n; i += W) {
    const T* x = static_cast<const T*>(p.X[i]) + row;
    const float k = to_f(x[0]);
    float s1 = 0.f, s2 = 0.f;
    constexpr int kUnroll = kUnrollFwd;
    for (long long c0 = static_cast<long long>(lane) * VEC; c0 < p.Hs; c0 += 32LL * VEC * kUnroll) {
      float v[kUnroll][VEC];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {  // kUnroll loads in flight
        const long long c = c0 + 32LL * VEC * u;
        if (c < p.Hs) load_vec<T, VEC>(x + c, v[u]);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (c0 + 32LL * VEC * u >= p.Hs) break;
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
          const float d = v[u][j] - k;
          s1 += d;
          s2 = fmaf(d, d, s2);
        }
      }
    }
    s1 = warp_sum(s1);
    s2 = warp_sum(s2);
    const float ci = static_cast<float>(p.Hs);
    if (lane == 0) {
      stat[i][0] = k + s1 / ci;
      stat[i][1] = fmaxf(s2 - s1 * (s1 / ci), 0.f);
    }
  }
  __syncthreads();
  // 2: the shards' statistics combined in shard order (every thread, same result)
  float cnt = 0.f, mean = 0.f, m2 = 0.f;
  const float ci = static_cast<float>(p.Hs);
  for (int i = 0; i < p.n; ++i) {
    const float c2 = cnt + ci;
    const float d = stat[i][0] - mean;
    mean += d * (ci / c2);
    m2 += stat[i][1] + d * d * (cnt * ci / c2);
    cnt = c2;
  }
  const float rstd = rsqrtf(m2 / cnt + p.eps);
  if (threadIdx.x == 0) {
    if (p.mean != nullptr) p.mean[t] = mean;
    if (p.rstd != nullptr) p.rstd[t] = rstd;
  }
  // 3: normalise, scale, shift (each warp its shards again: the bytes are in L1/L2)
  for (int i = warp; i < p.n; i += W) {
    const T* x = static_cast<const T*>(p.X[i]) + row;
    T* y = static_cast<T*>(p.Y[i]) + row;
    const T* g = static_cast<const T*>(p.gamma[i]);
    const T* b = static_cast<const T*>(p.beta[i]);
    for (long long c = static_cast<long long>(lane) * VEC; c < p.Hs; c += 32LL * VEC) {
      float v[VEC], gv[VEC], bv[VEC];
      load_vec<T, VEC>(x + c, v);
      if (g != nullptr) load_vec<T, VEC>(g + c, gv);
      if (b != nullptr) load_vec<T, VEC>(b + c, bv);
#pragma unroll
      for (int j = 0; j < VEC; ++j) {
        const float h = (v[j] - mean) * rstd;
        v[j] = fmaf(h, g != nullptr ? gv[j] : 1.f, b != nullptr ? bv[j] : 0.f);
      }
      store_vec<T, VEC>(y + c, v);
    }
  }
}

template <typename T, int VEC>
__global__ void __launch_bounds__(kLnWarps * 32, 3) ln_backward_dx_kernel(const __grid_constant__ LnParams p) {
  __shared__ float stat[kMaxShards][2];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, W = blockDim.x >> 5;
  const long long t = blockIdx.x;
  const long long row = t * p.Hs;
  const float mean = p.mean[t], rstd = p.rstd[t];
  // the two row statistics: per shard (warps over shards), then summed over the shards in order
  for (int i = warp; i < p.n; i += W) {
    const T* x = static_cast<const T*>(p.X[i]) + row;
    const T* dy = static_cast<const T*>(p.dY[i]) + row;
    const T* g = static_cast<const T*>(p.gamma[i]);
    float a1 = 0.f, a2 = 0.f;
    constexpr int kUnroll = kUnrollBwd;
    for (long long c0 = static_cast<long long>(lane) * VEC; c0 < p.Hs; c0 += 32LL * VEC * kUnroll) {
      float v[kUnroll][VEC], d[kUnroll][VEC];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const long long c = c0 + 32LL * VEC * u;
        if (c < p.Hs) {
          load_vec<T, VEC>(x + c, v[u]);
          load_vec<T, VEC>(dy + c, d[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const long long c = c0 + 32LL * VEC * u;
        if (c >= p.Hs) break;
        float gv[VEC];
        if (g != nullptr) load_vec<T, VEC>(g + c, gv);
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
          const float gg = d[u][j] * (g != nullptr ? gv[j] : 1.f);
          a1 += gg;
          a2 = fmaf(gg, (v[u][j] - mean) * rstd, a2);
        }
      }
    }
    a1 = warp_sum(a1);
    a2 = warp_sum(a2);
    if (lane == 0) {
      stat[i][0] = a1;
      stat[i][1] = a2;
    }
  }
  __syncthreads();
  float s1 = 0.f, s2 = 0.f;
  for (int i = 0; i < p.n; ++i) {
    s1 += stat[i][0];
    s2 += stat[i][1];
  }
  const float inv_h = 1.f / static_cast<float>(p.Hs * p.n);
  const float m1 = s1 * inv_h, m2 = s2 * inv_h;
  for (int i = warp; i < p.n; i += W) {
    const T* x = static_cast<const T*>(p.X[i]) + row;
    const T* dy = static_cast<const T*>(p.dY[i]) + row;
    const T* g = static_cast<const T*>(p.gamma[i]);
    T* dx = static_cast<T*>(p.Y[i]) + row;
    for (long long c = static_cast<long long>(lane) * VEC; c < p.Hs; c += 32LL * VEC) {
      float v[VEC], d[VEC], gv[VEC];
      load_vec<T, VEC>(x + c, v);
      load_vec<T, VEC>(dy + c, d);
      if (g != nullptr) load_vec<T, VEC>(g + c, gv);
#pragma unroll
      for (int j = 0; j < VEC; ++j) {
        const float gg = d[j] * (g != nullptr ? gv[j] : 1.f);
        const float h = (v[j] - mean) * rstd;
        v[j] = rstd * (gg - m1 - h * m2);
      }
      store_vec<T, VEC>(dx + c, v);
    }
  }
}

// Register-resident variants for rows whose shards fit in NV 16-byte vectors per lane (one
// warp per shard, n <= kLnWarps): every lane issues all loads of its part of the row at once
// (one DRAM round trip per block instead of one per kUnroll vectors plus a second pass that
// re-reads the row), keeps the raw vectors in registers for the second pass, and reads only
// gamma / beta again (the same few KB for every row: L1 hits). The arithmetic is that of the
// kernels above, in the same order (lane l's vectors l, l + 32, ... ascending): the results
// are bit-identical.
template <typename T, int NV>
__device__ __forceinline__ void load_row_part(const T* src, long long Hs, int lane, uint4* raw) {
  constexpr int VEC = 16 / sizeof(T);
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const long long c = static_cast<long long>(v * 32 + lane) * VEC;
    raw[v] = c < Hs ? *reinterpret_cast<const uint4*>(src + c) : make_uint4(0u, 0u, 0u, 0u);
  }
}

// The VEC values of a raw 16-byte vector as fp32, with register operations only (a bf16 is
// the upper half of the fp32 with the same bits).
template <typename T>
__device__ __forceinline__ void unpack16(const uint4& r, float* out);
template <>
__device__ __forceinline__ void unpack16<float>(const uint4& r, float* out) {
  out[0] = __uint_as_float(r.x);
  out[1] = __uint_as_float(r.y);
  out[2] = __uint_as_float(r.z);
  out[3] = __uint_as_float(r.w);
}
template <>
__device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4& r, float* out) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    out[2 * q] = __uint_as_float(w[q] << 16);
    out[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
  }
}

template <typename T, int NV>
__global__ void __launch_bounds__(kLnWarps * 32) ln_forward_reg_kernel(const __grid_constant__ LnParams p) {
  constexpr int VEC = 16 / sizeof(T);
  __shared__ float stat[kLnWarps][2];
  const int lane = threadIdx.x & 31, i = threadIdx.x >> 5;  // warp i: shard i
  const long long t = blockIdx.x;
  const long long row = t * p.Hs;
  const T* x = static_cast<const T*>(p.X[i]) + row;
  uint4 raw[NV];
  load_row_part<T, NV>(x, p.Hs, lane, raw);
  float first[VEC];
  unpack16<T>(raw[0], first);
  const float k = __shfl_sync(0xffffffffu, first[0], 0);  // the shard's first element
  float s1 = 0.f, s2 = 0.f;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    if (static_cast<long long>(v * 32 + lane) * VEC >= p.Hs) break;
    float f[VEC];
    unpack16<T>(raw[v], f);
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
      const float d = f[j] - k;
      s1 += d;
      s2 = fmaf(d, d, s2);
    }
  }
  s1 = warp_sum(s1);
  s2 = warp_sum(s2);
  const float ci = static_cast<float>(p.Hs);
  if (lane == 0) {
    stat[i][0] = k + s1 / ci;
    stat[i][1] = fmaxf(s2 - s1 * (s1 / ci), 0.f);
  }
  __syncthreads();
  float cnt = 0.f, mean = 0.f, m2 = 0.f;
  for (int s = 0; s < p.n; ++s) {
    const float c2 = cnt + ci;
    const float d = stat[s][0] - mean;
    mean += d * (ci / c2);
    m2 += stat[s][1] + d * d * (cnt * ci / c2);
    cnt = c2;
  }
  const float rstd = rsqrtf(m2 / cnt + p.eps);
  if (threadIdx.x == 0) {
    if (p.mean != nullptr) p.mean[t] = mean;
    if (p.rstd != nullptr) p.rstd[t] = rstd;
  }
  T* y = static_cast<T*>(p.Y[i]) + row;
  const T* g = static_cast<const T*>(p.gamma[i]);
  const T* b = static_cast<const T*>(p.beta[i]);
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const long long c = static_cast<long long>(v * 32 + lane) * VEC;
    if (c >= p.Hs) break;
    float f[VEC], gv[VEC], bv[VEC];
    unpack16<T>(raw[v], f);
    if (g != nullptr) load_vec<T, VEC>(g + c, gv);
    if (b != nullptr) load_vec<T, VEC>(b + c, bv);
    // the two-pass kernel's (x - mean) * rstd and fma, two columns per paired instruction
    // (each half rounded as the scalar operation: the same results)
#pragma unroll
    for (int j = 0; j < VEC; j += 2) {
      const float2 h = __fmul2_rn(__fadd2_rn(make_float2(f[j], f[j + 1]), splat2(-mean)),
                                  splat2(rstd));
      const float2 y = __ffma2_rn(h, g != nullptr ? make_float2(gv[j], gv[j + 1]) : splat2(1.f),
                                  b != nullptr ? make_float2(bv[j], bv[j + 1]) : splat2(0.f));
      f[j] = y.x;
      f[j + 1] = y.y;
    }
    store_vec<T, VEC>(y + c, f);
  }
}

template <typename T, int NV>
__global__ void __launch_bounds__(kLnWarps * 32, 3) ln_backward_dx_reg_kernel(const __grid_constant__ LnParams p) {
  constexpr int VEC = 16 / sizeof(T);
  __shared__ float stat[kLnWarps][2];
  const int lane = threadIdx.x & 31, i = threadIdx.x >> 5;
  const long long t = blockIdx.x;
  const long long row = t * p.Hs;
  uint4 xr[NV], dr[NV];
  load_row_part<T, NV>(static_cast<const T*>(p.X[i]) + row, p.Hs, lane, xr);
  load_row_part<T, NV>(static_cast<const T*>(p.dY[i]) + row, p.Hs, lane, dr);
  const float mean = p.mean[t], rstd = p.rstd[t];
  const T* g = static_cast<const T*>(p.gamma[i]);
  float a1 = 0.f, a2 = 0.f;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const long long c = static_cast<long long>(v * 32 + lane) * VEC;
    if (c >= p.Hs) break;
    float f[VEC], d[VEC], gv[VEC];
    unpack16<T>(xr[v], f);
    unpack16<T>(dr[v], d);
    if (g != nullptr) load_vec<T, VEC>(g + c, gv);
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
      const float gg = d[j] * (g != nullptr ? gv[j] : 1.f);
      a1 += gg;
      a2 = fmaf(gg, (f[j] - mean) * rstd, a2);
    }
  }
  a1 = warp_sum(a1);
  a2 = warp_sum(a2);
  if (lane == 0) {
    stat[i][0] = a1;
    stat[i][1] = a2;
  }
  __syncthreads();
  float s1 = 0.f, s2 = 0.f;
  for (int s = 0; s < p.n; ++s) {
    s1 += stat[s][0];
    s2 += stat[s][1];
  }
  const float inv_h = 1.f / static_cast<float>(p.Hs * p.n);
  const float m1 = s1 * inv_h, m2 = s2 * inv_h;
  T* dx = static_cast<T*>(p.Y[i]) + row;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const long long c = static_cast<long long>(v * 32 + lane) * VEC;
    if (c >= p.Hs) break;
    float f[VEC], d[VEC], gv[VEC];
    unpack16<T>(xr[v], f);
    unpack16<T>(dr[v], d);
    if (g != nullptr) load_vec<T, VEC>(g + c, gv);
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
      const float gg = d[j] * (g != nullptr ? gv[j] : 1.f);
      const float h = (f[j] - mean) * rstd;
      f[j] = rstd * (gg - m1 - h * m2);
    }
    store_vec<T, VEC>(dx + c, f);
  }
}

// dgamma_i[c] = sum_t dY_i[t,c] * xhat[t,c], dbeta_i[c] = sum_t dY_i[t,c]. blockIdx.x: a strip
// of 32 * VEC columns of one shard (strips of shard i are consecutive); lane l of every warp
// owns columns [strip + VEC l, strip + VEC l + VEC) (one 16-byte access per row where the rows
// allow it). blockIdx.y = q: tokens [q T / R, (q+1) T / R) of a cluster of R blocks, of which
// warp w takes every kPgWarps-th from the w-th, U rows' loads in flight, added in token order.
// The warps' sums are added in warp order, then the R blocks' in block order through
// distributed shared memory: deterministic, no atomics.
constexpr int kPgWarps = 16;

template <typename T, int VEC>
__global__ void __launch_bounds__(kPgWarps * 32) ln_param_grads_kernel(const __grid_constant__ LnParams p) {
  constexpr int U = 4;
  constexpr int COLS = 32 * VEC;
  __shared__ float part[kPgWarps][2][COLS];
  __shared__ float blk[2][COLS];
  const long long strips = (p.Hs + COLS - 1) / COLS;
  const int i = static_cast<int>(blockIdx.x / strips);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long c = (blockIdx.x % strips) * COLS + static_cast<long long>(lane) * VEC;
  const int R = static_cast<int>(gridDim.y), q = static_cast<int>(blockIdx.y);
  const long long t0 = p.T * q / R, t1 = p.T * (q + 1) / R;
  float sg[VEC], sb[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) sg[e] = sb[e] = 0.f;
  if (c < p.Hs) {
    const T* x = static_cast<const T*>(p.X[i]) + c;
    const T* dy = static_cast<const T*>(p.dY[i]) + c;
    long long t = t0 + warp;
    for (; t + (U - 1) * kPgWarps < t1; t += U * kPgWarps) {
      float xv[U][VEC], dv[U][VEC], mv[U], rv[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const long long tt = t + u * kPgWarps;
        load_vec<T, VEC>(x + tt * p.Hs, xv[u]);
        load_vec<T, VEC>(dy + tt * p.Hs, dv[u]);
        mv[u] = p.mean[tt];
        rv[u] = p.rstd[tt];
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          sg[e] = fmaf(dv[u][e], (xv[u][e] - mv[u]) * rv[u], sg[e]);
          sb[e] += dv[u][e];
        }
    }
    for (; t < t1; t += kPgWarps) {
      float xv[VEC], dv[VEC];
      load_vec<T, VEC>(x + t * p.Hs, xv);
      load_vec<T, VEC>(dy + t * p.Hs, dv);
      const float m = p.mean[t], r = p.rstd[t];
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        sg[e] = fmaf(dv[e], (xv[e] - m) * r, sg[e]);
        sb[e] += dv[e];
      }
    }
  }
#pragma unroll
  for (int e = 0; e < VEC; ++e) {
    part[warp][0][lane * VEC + e] = sg[e];
    part[warp][1][lane * VEC + e] = sb[e];
  }
  __syncthreads();
  // the block's sums: warps in order (thread k < 2 * COLS sums one of the 2 * COLS values)
  for (int k = threadIdx.x; k < 2 * COLS; k += kPgWarps * 32) {
    float v = 0.f;
    for (int w = 0; w < kPgWarps; ++w) v += part[w][k / COLS][k % COLS];
    blk[k / COLS][k % COLS] = v;
  }
  auto store = [&](int k, float v) {
    const long long col = (blockIdx.x % strips) * COLS + (k % COLS);
    if (col >= p.Hs) return;
    float* out = k < COLS ? p.dgamma[i] : p.dbeta[i];
    if (out != nullptr) out[col] = v;
  };
  if (R == 1) {
    __syncthreads();
    for (int k = threadIdx.x; k < 2 * COLS; k += kPgWarps * 32) store(k, blk[k / COLS][k % COLS]);
    return;
  }
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  if (q == 0) {
    for (int k = threadIdx.x; k < 2 * COLS; k += kPgWarps * 32) {
      float v = 0.f;
      for (int r = 0; r < R; ++r) v += cluster.map_shared_rank(&blk[0][0], r)[k];
      store(k, v);
    }
  }
  cluster.sync();
}

bool aligned16(const void* ptr) { return reinterpret_cast<uintptr_t>(ptr) % 16 == 0; }

// Vector width usable for every row of every shard (16-byte accesses need 16-byte-aligned
// shard bases and rows whose byte length is a multiple of 16).
template <typename T>
int vec_width(const LnParams& p, bool backward) {
  constexpr int V = 16 / sizeof(T);
  if (p.Hs % V != 0) return 1;
  for (int i = 0; i < p.n; ++i) {
    if (!aligned16(p.X[i]) || !aligned16(p.Y[i])) return 1;
    if (p.gamma[i] != nullptr && !aligned16(p.gamma[i])) return 1;
    if (!backward && p.beta[i] != nullptr && !aligned16(p.beta[i])) return 1;
    if (backward && !aligned16(p.dY[i])) return 1;
  }
  return V;
}

// Register-resident kernels where they apply; TP_TUNE_LN_REG = 0 keeps the two-pass kernels.
bool ln_reg_enabled() {
  if (const int v = tuning(TP_TUNE_LN_REG); v != TP_TUNE_AUTO) return v != 0;
  return true;
}

template <typename T, int NV>
void launch_rows_reg(const LnParams& p, bool backward, dim3 grid, int threads, cudaStream_t st) {
  if (!backward)
    ln_forward_reg_kernel<T, NV><<<grid, threads, 0, st>>>(p);
  else
    ln_backward_dx_reg_kernel<T, NV><<<grid, threads, 0, st>>>(p);
}

template <typename T>
cudaError_t launch_rows(const LnParams& p, bool backward, cudaStream_t st) {
  constexpr int V = 16 / sizeof(T);
  if (p.T > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(p.T));                 // one block per token row
  const int threads = 32 * std::min(p.n, kLnWarps);          // one warp per shard (or more)
  const bool vec = vec_width<T>(p, backward) == V;
  const long long nv = (p.Hs + 32LL * V - 1) / (32LL * V);    // 16-byte vectors per lane
  if (vec && p.n <= kLnWarps && nv <= 8 && ln_reg_enabled()) {
    if (nv <= 2)
      launch_rows_reg<T, 2>(p, backward, grid, threads, st);
    else if (nv <= 4)
      launch_rows_reg<T, 4>(p, backward, grid, threads, st);
    else if (nv <= 6)
      launch_rows_reg<T, 6>(p, backward, grid, threads, st);
    else
      launch_rows_reg<T, 8>(p, backward, grid, threads, st);
    return cudaGetLastError();
  }
  if (!backward) {
    if (vec)
      ln_forward_kernel<T, V><<<grid, threads, 0, st>>>(p);
    else
      ln_forward_kernel<T, 1><<<grid, threads, 0, st>>>(p);
  } else {
    if (vec)
      ln_backward_dx_kernel<T, V><<<grid, threads, 0, st>>>(p);
    else
      ln_backward_dx_kernel<T, 1><<<grid, threads, 0, st>>>(p);
  }
  return cudaGetLastError();
}

template <typename T, int VEC>
cudaLaunchConfig_t param_grads_config(long long strips, int R, cudaStream_t st,
                                      cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(strips), static_cast<unsigned>(R), 1);
  cfg.blockDim = dim3(kPgWarps * 32, 1, 1);
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = static_cast<unsigned>(R);
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// How many clusters of R blocks of the column-sum kernel the device holds at once (cached per
// device; the driver's answer, which accounts for clusters having to fit within one GPC).
template <typename T, int VEC>
int param_grads_max_clusters(int R) {
  static int cache[64][9] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev][R] == 0) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = param_grads_config<T, VEC>(1, R, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, ln_param_grads_kernel<T, VEC>, &cfg) != cudaSuccess)
      n = 0;
    cache[dev][R] = n > 0 ? n : -1;
  }
  return cache[dev][R];
}

template <typename T, int VEC>
cudaError_t launch_param_grads_v(const LnParams& p, cudaStream_t st) {
  const long long strips = ((p.Hs + 32LL * VEC - 1) / (32LL * VEC)) * p.n;
  if (strips > 0x7fffffffLL) return cudaErrorInvalidValue;
  // blocks per strip (a cluster): the most, up to 8 and at least 256 tokens each, for which
  // all strips' clusters are resident at once (a second, partial wave would double the time)
  int R = 1;
  for (int r = static_cast<int>(std::min(8LL, std::max(1LL, p.T / 256))); r > 1; --r) {
    if (param_grads_max_clusters<T, VEC>(r) >= strips) {
      R = r;
      break;
    }
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = param_grads_config<T, VEC>(strips, R, st, attr);
  return cudaLaunchKernelEx(&cfg, ln_param_grads_kernel<T, VEC>, p);
}

template <typename T>
cudaError_t launch_param_grads(const LnParams& p, cudaStream_t st) {
  constexpr int V = 16 / sizeof(T);
  bool vec = p.Hs % V == 0;
  for (int i = 0; i < p.n && vec; ++i) vec = aligned16(p.X[i]) && aligned16(p.dY[i]);
  return vec ? launch_param_grads_v<T, V>(p, st) : launch_param_grads_v<T, 1>(p, st);
}

LnParams make(const LnArgs& a) {
  LnParams p{};
  for (int i = 0; i < a.n; ++i) {
    p.X[i] = a.X[i];
    p.gamma[i] = a.gamma ? a.gamma[i] : nullptr;
    p.beta[i] = a.beta ? a.beta[i] : nullptr;
    p.Y[i] = a.Y ? a.Y[i] : nullptr;
    p.dY[i] = a.dY ? a.dY[i] : nullptr;
    p.dgamma[i] = a.dgamma ? a.dgamma[i] : nullptr;
    p.dbeta[i] = a.dbeta ? a.dbeta[i] : nullptr;
  }
  p.mean = a.mean;
  p.rstd = a.rstd;
  p.T = a.T;
  p.Hs = a.Hs;
  p.n = a.n;
  p.eps = a.eps;
  return p;
}

}  // namespace

cudaError_t launch_ln_forward(const LnArgs& a, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  const LnParams p = make(a);
  return a.bf16 ? launch_rows<__nv_bfloat16>(p, false, st) : launch_rows<float>(p, false, st);
}

cudaError_t launch_ln_backward_dx(const LnArgs& a, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  const LnParams p = make(a);
  return a.bf16 ? launch_rows<__nv_bfloat16>(p, true, st) : launch_rows<float>(p, true, st);
}

cudaError_t launch_ln_param_grads(const LnArgs& a, cudaStream_t st) {
  const LnParams p = make(a);
  if (a.T == 0) {
    for (int i = 0; i < a.n; ++i) {
      if (p.dgamma[i] != nullptr) {
        cudaError_t e = cudaMemsetAsync(p.dgamma[i], 0, size_t(a.Hs) * 4, st);
        if (e != cudaSuccess) return e;
      }
      if (p.dbeta[i] != nullptr) {
        cudaError_t e = cudaMemsetAsync(p.dbeta[i], 0, size_t(a.Hs) * 4, st);
        if (e != cudaSuccess) return e;
      }
    }
    return cudaSuccess;
  }
  return a.bf16 ? launch_param_grads<__nv_bfloat16>(p, st) : launch_param_grads<float>(p, st);
}

}  // namespace tpk
