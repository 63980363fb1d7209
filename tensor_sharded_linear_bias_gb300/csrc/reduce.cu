// Bandwidth-bound kernels of the path:
//  * shard_reduce: Z = sum_i P_i + bias over fp32 shard partials (the pages' All-Reduce SUM,
//    done on the device in fixed shard order), 128-bit coalesced loads and stores;
//  * colsum: bias gradients, sums over tokens of dZ / dH_i, deterministic (fixed order);
//  * dact: dH = dY * GeLU'(H) for the stand-alone column backward;
//  * the one-block self-test of the bounded wait.
#include <cuda_runtime.h>

#include <cooperative_groups.h>

#include <algorithm>

#include "device_common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace tpk {

int device_sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

namespace {

// ------------------------------------------------------------------ shard reduce
constexpr int kReduceThreads = 256;

__device__ __forceinline__ float4 ld_stream(const float4* p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void add4(float4& a, const float4& b) {
  a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
}

__device__ __forceinline__ float4 bias4(const void* bias, int bf16, long long col) {
  if (bias == nullptr) return make_float4(0.f, 0.f, 0.f, 0.f);
  if (bf16) {
    const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(bias) + col);
    const float2 lo = unpack_bf16x2(u.x), hi = unpack_bf16x2(u.y);
    return make_float4(lo.x, lo.y, hi.x, hi.y);
  }
  return *reinterpret_cast<const float4*>(static_cast<const float*>(bias) + col);
}

// P holds n partials of count4 float4 each, back to back. Shards are added in order
// 0..n-1; loads are issued four shards at a time to keep enough bytes in flight.
__global__ void __launch_bounds__(kReduceThreads) shard_reduce_v4(const float4* __restrict__ P,
                                                                  int n, long long count4,
                                                                  long long n4,
                                                                  const void* bias, int bias_bf16,
                                                                  float4* __restrict__ Z) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
       idx < count4; idx += stride) {
    float4 s = ld_stream(P + idx);
    int i = 1;
    for (; i + 3 < n; i += 4) {
      const float4 a = ld_stream(P + (i + 0) * count4 + idx);
      const float4 b = ld_stream(P + (i + 1) * count4 + idx);
      const float4 c = ld_stream(P + (i + 2) * count4 + idx);
      const float4 d = ld_stream(P + (i + 3) * count4 + idx);
      add4(s, a); add4(s, b); add4(s, c); add4(s, d);
    }
    for (; i < n; ++i) add4(s, ld_stream(P + i * count4 + idx));
    add4(s, bias4(bias, bias_bf16, (idx % n4) * 4));
    Z[idx] = s;
  }
}

__global__ void shard_reduce_scalar(const float* __restrict__ P, int n, long long count,
                                    long long N, const void* bias, int bias_bf16,
                                    float* __restrict__ Z) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
       idx < count; idx += stride) {
    float s = P[idx];
    for (int i = 1; i < n; ++i) s += P[i * count + idx];
    if (bias != nullptr) {
      const long long c = idx % N;
      s += bias_bf16 ? bf16_to_f32(static_cast<const uint16_t*>(bias)[c])
                     : static_cast<const float*>(bias)[c];
    }
    Z[idx] = s;
  }
}

// Eight bf16 partial values per thread and shard (one 16-byte load each), summed in fp32 in
// shard order, plus the bias; two 16-byte fp32 stores.
__global__ void __launch_bounds__(kReduceThreads) shard_reduce_bf16_v8(
    const uint4* __restrict__ P, int n, long long count8, long long n8, const void* bias,
    float4* __restrict__ Z) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
       idx < count8; idx += stride) {
    float s[8] = {};
    for (int i = 0; i < n; ++i) {
      uint4 u;
      asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
                   : "l"(P + i * count8 + idx));
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = unpack_bf16x2(w[j]);
        s[2 * j] += f.x;
        s[2 * j + 1] += f.y;
      }
    }
    if (bias != nullptr) {
      const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(bias) + (idx % n8) * 8);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = unpack_bf16x2(w[j]);
        s[2 * j] += f.x;
        s[2 * j + 1] += f.y;
      }
    }
    Z[2 * idx] = make_float4(s[0], s[1], s[2], s[3]);
    Z[2 * idx + 1] = make_float4(s[4], s[5], s[6], s[7]);
  }
}

// ------------------------------------------------------------------ token-shard copies
struct ShardCopyParams {
  void* shards[kMaxShards];
  void* full;
  long long bytes;   // per shard
  int n;
  int gather;
};

// Grid-stride copy over n blocks, 16 bytes per thread and step when every block allows it.
__global__ void shard_copy_kernel(const __grid_constant__ ShardCopyParams p) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const bool vec = (p.bytes % 16 == 0) && (reinterpret_cast<uintptr_t>(p.full) % 16 == 0);
  for (int j = 0; j < p.n; ++j) {
    char* sh = static_cast<char*>(p.shards[j]);
    char* fu = static_cast<char*>(p.full) + static_cast<long long>(j) * p.bytes;
    char* dst = p.gather ? fu : sh;
    const char* src = p.gather ? sh : fu;
    if (vec && reinterpret_cast<uintptr_t>(sh) % 16 == 0) {
      const long long n16 = p.bytes / 16;
      for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
           i += stride)
        reinterpret_cast<uint4*>(dst)[i] = reinterpret_cast<const uint4*>(src)[i];
    } else {
      for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
           i < p.bytes; i += stride)
        dst[i] = src[i];
    }
  }
}

// ------------------------------------------------------------------ column sums
// One cluster of R blocks per (segment, strip of 256 columns); block q of the cluster sums
// rows [q*rows/R, (q+1)*rows/R) with 16 warps. Lane l of warp w owns columns
// [strip + 8l, strip + 8l + 8) and every 16th row of the block's range from w; it keeps eight
// of its rows' 16-byte loads in flight and adds them in row order. The 16 warps' sums are
// added in warp order, then block 0 adds the R blocks' sums in block order, reading them from
// the other blocks' shared memory (distributed shared memory of the cluster). R > 1 only when
// the strips alone would leave SMs idle (few columns); R <= 16. Every addition happens in a
// fixed order for a given shape, so the result is the same on every run.
constexpr int kColsumWarps = 16;
constexpr int kColsumUnroll = 8;
constexpr int kMaxColsumSegs = kMaxShards + 1;

struct ColsumParams {
  ColsumSeg seg[kMaxColsumSegs];
  int strip_start[kMaxColsumSegs + 1];  // prefix sums of strips per segment
  int nseg;
  long long rows;
  int bf16;
};

__device__ __forceinline__ void load8(const void* base, int bf16, long long off, float* v,
                                      int valid) {
  if (bf16 && valid == 8) {
    const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + off);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = unpack_bf16x2(w[j]);
      v[2 * j] = f.x;
      v[2 * j + 1] = f.y;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      v[j] = (j < valid) ? (bf16 ? bf16_to_f32(static_cast<const uint16_t*>(base)[off + j])
                                 : static_cast<const float*>(base)[off + j])
                         : 0.f;
  }
}

__global__ void __launch_bounds__(kColsumWarps * 32) colsum_kernel(const __grid_constant__ ColsumParams p) {
  __shared__ float part[kColsumWarps][256];
  __shared__ float block_sum[256];
  grid_dependency_wait();
  grid_dependents_launch();
  int s = 0;
  while (s + 1 < p.nseg && static_cast<int>(blockIdx.x) >= p.strip_start[s + 1]) ++s;
  const ColsumSeg seg = p.seg[s];
  const long long c0 = static_cast<long long>(blockIdx.x - p.strip_start[s]) * 256;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const long long col = c0 + 8 * lane;
  const int valid = static_cast<int>(max(0LL, min(8LL, seg.cols - col)));
  const int R = static_cast<int>(gridDim.y);  // blocks per cluster (cluster dims 1 x R x 1)
  const int q = static_cast<int>(blockIdx.y);
  const long long r_end = p.rows * (q + 1) / R;
  float acc[8] = {};
  if (valid > 0) {
    const long long step = kColsumWarps;
    long long r = p.rows * q / R + warp;
    if (p.bf16 && valid == 8) {
      // Raw 16-byte loads first (8 rows in flight), then unpack and add in row order.
      const uint16_t* in = static_cast<const uint16_t*>(seg.in);
      for (; r + (kColsumUnroll - 1) * step < r_end; r += kColsumUnroll * step) {
        uint4 raw[kColsumUnroll];
#pragma unroll
        for (int u = 0; u < kColsumUnroll; ++u)
          raw[u] = *reinterpret_cast<const uint4*>(in + (r + u * step) * seg.ld + col);
#pragma unroll
        for (int u = 0; u < kColsumUnroll; ++u) {
          const uint32_t w[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 f = unpack_bf16x2(w[j]);
            acc[2 * j] += f.x;
            acc[2 * j + 1] += f.y;
          }
        }
      }
    }
    for (; r < r_end; r += step) {
      float v[8];
      load8(seg.in, p.bf16, r * seg.ld + col, v, valid);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] += v[j];
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) part[warp][8 * lane + j] = acc[j];
  __syncthreads();
  const long long c = c0 + threadIdx.x;
  if (threadIdx.x < 256) {
    float t = 0.f;
#pragma unroll 8
    for (int w = 0; w < kColsumWarps; ++w) t += part[w][threadIdx.x];
    if (R == 1) {
      if (c < seg.cols) seg.out[c] = t;
    } else {
      block_sum[threadIdx.x] = t;
    }
  }
  if (R == 1) return;
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();  // every block's sums are in its shared memory
  if (q == 0 && threadIdx.x < 256 && c < seg.cols) {
    float t = 0.f;
    for (int b = 0; b < R; ++b) t += cluster.map_shared_rank(block_sum, b)[threadIdx.x];
    seg.out[c] = t;
  }
  cluster.sync();  // no block leaves while block 0 may still read its shared memory
}

// ------------------------------------------------------------------ dH = dY * act'(H)
struct DactParams {
  const void* dY[kMaxShards];
  const void* H[kMaxShards];
  void* dH[kMaxShards];
  long long ld_dy, T, w;
  int act, bf16;
};

__global__ void dact_kernel(const __grid_constant__ DactParams p) {
  const int g = blockIdx.y;
  const long long total = p.T * p.w;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const long long t = i / p.w, c = i % p.w;
    float dy, h;
    if (p.bf16) {
      dy = bf16_to_f32(static_cast<const uint16_t*>(p.dY[g])[t * p.ld_dy + c]);
      h = bf16_to_f32(static_cast<const uint16_t*>(p.H[g])[i]);
    } else {
      dy = static_cast<const float*>(p.dY[g])[t * p.ld_dy + c];
      h = static_cast<const float*>(p.H[g])[i];
    }
    const float v = (p.act == TP_ACT_GELU_ERF) ? dy * gelu_erf_grad(h) : dy;
    if (p.bf16) {
      static_cast<__nv_bfloat16*>(p.dH[g])[i] = __float2bfloat16_rn(v);
    } else {
      static_cast<float*>(p.dH[g])[i] = v;
    }
  }
}

// ------------------------------------------------------------------ wait self-test
// One warp: allocates a TMEM block, waits on an mbarrier that nothing arrives on, gives up
// after limit_ns, reports the timeout, frees TMEM and returns.
__global__ void wait_selftest_kernel(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_slot;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_mbarrier_init();
  }
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 32;" ::"r"(
                   smem_addr(&tmem_slot))
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncwarp();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_slot;
  const bool ok = mbar_wait_bounded(smem_addr(&bar), 0, limit_ns);
  if (!ok && threadIdx.x == 0) report_status(status, kDevTimeoutBase | 0x70);
  __syncwarp();
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 32;" ::"r"(tmem) : "memory");
}

}  // namespace

cudaError_t launch_shard_reduce(const float* P, int n, int64_t T, int64_t N, const void* bias,
                                int bias_bf16, float* Z, cudaStream_t st) {
  const long long count = static_cast<long long>(T) * N;
  if (count == 0) return cudaSuccess;
  const int sms = device_sm_count();
  const bool vec = (N % 4 == 0) && (reinterpret_cast<uintptr_t>(P) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(Z) % 16 == 0) &&
                   (bias == nullptr || reinterpret_cast<uintptr_t>(bias) % (bias_bf16 ? 8 : 16) == 0);
  if (vec) {
    const long long count4 = count / 4;
    const long long blocks = std::min<long long>((count4 + kReduceThreads - 1) / kReduceThreads,
                                                 static_cast<long long>(sms) * 8);
    shard_reduce_v4<<<static_cast<unsigned>(blocks), kReduceThreads, 0, st>>>(
        reinterpret_cast<const float4*>(P), n, count4, N / 4, bias, bias_bf16,
        reinterpret_cast<float4*>(Z));
  } else {
    const long long blocks = std::min<long long>((count + kReduceThreads - 1) / kReduceThreads,
                                                 static_cast<long long>(sms) * 8);
    shard_reduce_scalar<<<static_cast<unsigned>(blocks), kReduceThreads, 0, st>>>(
        P, n, count, N, bias, bias_bf16, Z);
  }
  return cudaGetLastError();
}

cudaError_t launch_shard_reduce_bf16(const uint16_t* P, int n, int64_t T, int64_t N,
                                     const void* bias, float* Z, cudaStream_t st) {
  const long long count = static_cast<long long>(T) * N;
  if (count == 0) return cudaSuccess;
  if (N % 8 != 0 || reinterpret_cast<uintptr_t>(P) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(Z) % 16 != 0 ||
      (bias != nullptr && reinterpret_cast<uintptr_t>(bias) % 16 != 0))
    return cudaErrorInvalidValue;
  const long long count8 = count / 8;
  const long long blocks = std::min<long long>((count8 + kReduceThreads - 1) / kReduceThreads,
                                               static_cast<long long>(device_sm_count()) * 8);
  shard_reduce_bf16_v8<<<static_cast<unsigned>(blocks), kReduceThreads, 0, st>>>(
      reinterpret_cast<const uint4*>(P), n, count8, N / 8, bias, reinterpret_cast<float4*>(Z));
  return cudaGetLastError();
}

cudaError_t launch_shard_copy(void* const* shards, void* full, int n, size_t bytes, int gather,
                              cudaStream_t st) {
  if (n < 1 || n > kMaxShards) return cudaErrorInvalidValue;
  if (bytes == 0) return cudaSuccess;
  ShardCopyParams p{};
  for (int j = 0; j < n; ++j) p.shards[j] = shards[j];
  p.full = full;
  p.bytes = static_cast<long long>(bytes);
  p.n = n;
  p.gather = gather;
  const long long blocks = std::min<long long>((static_cast<long long>(bytes) / 16 + 255) / 256 + 1,
                                               static_cast<long long>(device_sm_count()) * 8);
  shard_copy_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_colsum(const ColsumSeg* segs, int nseg, int64_t rows, int in_bf16,
                          cudaStream_t st) {
  if (nseg <= 0) return cudaSuccess;
  if (nseg > kMaxColsumSegs) return cudaErrorInvalidValue;
  ColsumParams p{};
  p.nseg = nseg;
  p.rows = rows;
  p.bf16 = in_bf16;
  int strips = 0;
  for (int s = 0; s < nseg; ++s) {
    p.seg[s] = segs[s];
    p.strip_start[s] = strips;
    strips += static_cast<int>((segs[s].cols + 255) / 256);
  }
  p.strip_start[nseg] = strips;
  if (strips == 0) return cudaSuccess;
  // Blocks per strip: enough for about four blocks per SM, at least 256 rows each, at most a
  // cluster of 16 (above 8: the non-portable size; measured on GB300, 4096 tokens and 20
  // strips: 12.4 us with clusters of 16 against 14.6 with 8, and 18.3 with 7 fitted to one wave).
  const long long want = (4LL * device_sm_count() + strips - 1) / strips;
  const int R = static_cast<int>(std::max(1LL, std::min({want, static_cast<long long>(rows) / 256, 16LL})));
  if (R > 8) {
    static bool allowed[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !allowed[dev]) {
      e = cudaFuncSetAttribute(colsum_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) allowed[dev] = true;
    }
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(strips), static_cast<unsigned>(R), 1);
  cfg.blockDim = dim3(kColsumWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = static_cast<unsigned>(R);
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = tuning(TP_TUNE_PDL) != 0 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, colsum_kernel, p);
}

cudaError_t launch_dact(const void* const* dY, int64_t ld_dy, const void* const* H,
                        void* const* dH, int n, int64_t T, int64_t w, int act, int bf16,
                        cudaStream_t st) {
  if (n < 1 || n > kMaxShards) return cudaErrorInvalidValue;
  if (T * w == 0) return cudaSuccess;
  DactParams p{};
  for (int g = 0; g < n; ++g) {
    p.dY[g] = dY[g];
    p.H[g] = H[g];
    p.dH[g] = dH[g];
  }
  p.ld_dy = ld_dy;
  p.T = T;
  p.w = w;
  p.act = act;
  p.bf16 = bf16;
  const long long total = static_cast<long long>(T) * w;
  const unsigned bx = static_cast<unsigned>(
      std::min<long long>((total + 255) / 256, std::max(1, device_sm_count() * 4 / n)));
  dact_kernel<<<dim3(bx, n), 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(status, static_cast<unsigned long long>(limit_ns));
  return cudaGetLastError();
}

}  // namespace tpk
