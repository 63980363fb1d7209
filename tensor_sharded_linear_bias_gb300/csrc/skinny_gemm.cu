// fp32 GEMM for products of at most 32 rows (the pages' batch-32 example and other few-token
// calls), FFMA only: A K-major [M, K] (M <= 32), B MN-major [K, N], per-shard outputs or the shard
// sum, epilogue bias (+ GeLU).
//
// With 32 rows the weights (B) are the whole cost: every element of B is used exactly 32 times,
// once per row. So each lane keeps all 32 rows x C consecutive columns of the output in
// registers and streams its columns of B straight from global memory into registers (C
// floats per K step, one coalesced 8- or 16-byte load: a warp reads 32 C consecutive floats of a
// row of B), several K steps ahead; A's K slice is staged once in shared memory, transposed
// ([k][32 rows]), and read as broadcasts (every lane of a warp reads the same 32 values). Per K
// step a lane does 32 C FFMAs for one global load and eight 16-byte shared loads.
//
// A CTA (8 warps) owns 32 C output columns and one K slice; its warps split the slice into 8
// contiguous parts and add their 32 x 32 C partial tiles in warp order through shared memory.
// The S CTAs of a thread-block cluster take S contiguous K slices (over all summed shards) of the
// same columns; after a cluster barrier CTA q adds the S partial tiles of rows q M/S .. (q+1) M/S
// - 1 in CTA order (distributed shared memory), applies the epilogue and stores. Every sum is in
// a fixed order for a shape: results repeat bit for bit.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "device_common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace tpk {
namespace {

constexpr int kSkinnyRows = 32;
constexpr int kSkinnyWarps = 8;
constexpr int kSkinnyThreads = 32 * kSkinnyWarps;
constexpr int kSkinnyMaxSplit = 16;   // CTAs per cluster (above 8: non-portable size)
constexpr int kSkinnyMaxSlice = 512;  // K steps per CTA: A's slice in shared memory <= 64 KiB
constexpr int kPrefetch = 4;          // K steps of B in registers ahead of the one in use

struct SkinnyParams {
  const float* A[kMaxShards];
  const float* B[kMaxShards];
  float* D[kMaxShards];
  float* D2[kMaxShards];
  const float* bias[kMaxShards];
  long long lda, ldb, ldd, ldd2;
  int M, N, K;
  int groups, ksum, epi, act;
  int slices;  // CTAs per cluster = K slices
};

template <int C>
struct SkinnySmem {
  static constexpr int kPartialFloats = kSkinnyWarps * kSkinnyRows * 32 * C;
  static constexpr int kSliceFloats = kSkinnyMaxSlice * kSkinnyRows;
  // A's slice ([k][32 rows]) first; after the K loop the same space holds the warps' partial
  // tiles, then (warp 0's part) the CTA's summed tile that the cluster reads
  static constexpr int kFloats = kPartialFloats > kSliceFloats ? kPartialFloats : kSliceFloats;
  static constexpr int kBytes = kFloats * 4;
};

template <int C>
struct BVec;
template <>
struct BVec<2> {
  __device__ static void load(const float* p, float* b) {
    const float2 v = *reinterpret_cast<const float2*>(p);
    b[0] = v.x;
    b[1] = v.y;
  }
};
template <>
struct BVec<4> {
  __device__ static void load(const float* p, float* b) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    b[0] = v.x;
    b[1] = v.y;
    b[2] = v.z;
    b[3] = v.w;
  }
};

__device__ __forceinline__ void skinny_epilogue(const SkinnyParams& p, int og, int m, int n,
                                                float v) {
  if (p.bias[og] != nullptr) v += p.bias[og][n];
  if (p.epi == EPI_BIAS_ACT) {
    if (p.D[og] != nullptr) p.D[og][static_cast<long long>(m) * p.ldd + n] = v;
    p.D2[og][static_cast<long long>(m) * p.ldd2 + n] = (p.act == TP_ACT_GELU_ERF) ? gelu_erf(v) : v;
  } else {
    p.D[og][static_cast<long long>(m) * p.ldd + n] = v;
  }
}

template <int C>
__global__ void __launch_bounds__(kSkinnyThreads, 1)
    skinny_gemm_kernel(const __grid_constant__ SkinnyParams p) {
  constexpr int TN = 32 * C;  // columns per CTA
  extern __shared__ __align__(16) float skinny_smem[];
  float* As = skinny_smem;  // [kk][32]
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int S = p.slices;
  const int q = static_cast<int>(blockIdx.x);  // K slice = rank in the cluster
  const int og = static_cast<int>(blockIdx.z);
  const int n0 = static_cast<int>(blockIdx.y) * TN;
  const int kgroups = p.ksum ? p.groups : 1;
  const long long Ktot = static_cast<long long>(p.K) * kgroups;
  const int k_lo = static_cast<int>(Ktot * q / S), k_hi = static_cast<int>(Ktot * (q + 1) / S);
  const int klen = k_hi - k_lo;

  grid_dependency_wait();

  // A's slice, transposed into [kk][row]; rows >= M are zeros. k' = k_lo + kk is column k' % K of
  // shard k' / K (summed shards) or column k' of this output's shard.
  for (int e = threadIdx.x; e < klen * kSkinnyRows; e += kSkinnyThreads) {
    const int m = e / klen, kk = e % klen;  // consecutive threads: consecutive k of one row
    const int kp = k_lo + kk;
    const int g = p.ksum ? kp / p.K : og;
    const int k = p.ksum ? kp % p.K : kp;
    As[kk * kSkinnyRows + m] = m < p.M ? p.A[g][static_cast<long long>(m) * p.lda + k] : 0.0f;
  }

  // this warp's part of the slice and its columns
  const int w_lo = klen * warp / kSkinnyWarps, w_hi = klen * (warp + 1) / kSkinnyWarps;
  const int n = n0 + C * lane;
  const bool col_in = n < p.N;  // N % C == 0: a lane's C columns are all in or all out
  float acc[kSkinnyRows][C];
#pragma unroll
  for (int m = 0; m < kSkinnyRows; ++m)
#pragma unroll
    for (int c = 0; c < C; ++c) acc[m][c] = 0.0f;

  // B's rows are loaded in slice order: the next one to load is row ld_k of shard ld_g
  int ld_g = og, ld_k = k_lo + w_lo;
  if (p.ksum) {
    ld_g = ld_k / p.K;
    ld_k -= ld_g * p.K;
  }
  auto load_next = [&](float* dst) {
    if (col_in) BVec<C>::load(p.B[ld_g] + static_cast<long long>(ld_k) * p.ldb + n, dst);
    if (++ld_k == p.K && p.ksum) {
      ld_k = 0;
      ++ld_g;
    }
  };
  float bq[kPrefetch][C];
#pragma unroll
  for (int i = 0; i < kPrefetch; ++i) {
#pragma unroll
    for (int c = 0; c < C; ++c) bq[i][c] = 0.0f;
    if (w_lo + i < w_hi) load_next(bq[i]);
  }
  __syncthreads();  // A's slice is in shared memory

  for (int kb = w_lo; kb < w_hi; kb += kPrefetch) {
#pragma unroll
    for (int i = 0; i < kPrefetch; ++i) {
      const int kk = kb + i;
      if (kk < w_hi) {
        float b[C];
#pragma unroll
        for (int c = 0; c < C; ++c) b[c] = bq[i][c];
        // refill this register slot with step kk + kPrefetch
        if (kk + kPrefetch < w_hi) load_next(bq[i]);
        const float4* a4 = reinterpret_cast<const float4*>(As + kk * kSkinnyRows);
#pragma unroll
        for (int r = 0; r < kSkinnyRows / 4; ++r) {
          const float4 a = a4[r];
#pragma unroll
          for (int c = 0; c < C; ++c) {
            acc[4 * r + 0][c] = fmaf(a.x, b[c], acc[4 * r + 0][c]);
            acc[4 * r + 1][c] = fmaf(a.y, b[c], acc[4 * r + 1][c]);
            acc[4 * r + 2][c] = fmaf(a.z, b[c], acc[4 * r + 2][c]);
            acc[4 * r + 3][c] = fmaf(a.w, b[c], acc[4 * r + 3][c]);
          }
        }
      }
    }
  }
  grid_dependents_launch();

  // the warps' partial tiles, then their sum in warp order: part[w][m][col]
  __syncthreads();  // every warp is done reading A's slice
  float* part = skinny_smem;
#pragma unroll
  for (int m = 0; m < kSkinnyRows; ++m)
#pragma unroll
    for (int c = 0; c < C; ++c)
      part[(warp * kSkinnyRows + m) * TN + C * lane + c] = acc[m][c];
  __syncthreads();
  for (int e = threadIdx.x; e < kSkinnyRows * TN; e += kSkinnyThreads) {
    float t = part[e];
#pragma unroll
    for (int w = 1; w < kSkinnyWarps; ++w) t += part[w * kSkinnyRows * TN + e];
    part[e] = t;  // warp 0's part now holds the CTA's tile
  }
  __syncthreads();

  if (S == 1) {
    for (int e = threadIdx.x; e < p.M * TN; e += kSkinnyThreads) {
      const int m = e / TN, col = n0 + e % TN;
      if (col < p.N) skinny_epilogue(p, og, m, col, part[e]);
    }
    return;
  }
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();  // every CTA's tile is summed
  const int r0 = p.M * q / S, r1 = p.M * (q + 1) / S;
  for (int e = threadIdx.x; e < (r1 - r0) * TN; e += kSkinnyThreads) {
    const int m = r0 + e / TN, cc = e % TN, col = n0 + cc;
    float v = 0.0f;
    for (int s = 0; s < S; ++s) v += cluster.map_shared_rank(part, s)[m * TN + cc];
    if (col < p.N) skinny_epilogue(p, og, m, col, v);
  }
  cluster.sync();  // no CTA leaves while another may still read its shared memory
}

template <int C>
int skinny_max_active_clusters(int S) {
  static int cache[64][kSkinnyMaxSplit + 1][2] = {};
  int dev = 0;
  if (S < 2 || S > kSkinnyMaxSplit || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return 0;
  int& slot = cache[dev][S][C == 4 ? 1 : 0];
  if (slot == 0) {
    int n = 0;
    auto kern = skinny_gemm_kernel<C>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SkinnySmem<C>::kBytes) == cudaSuccess &&
        (S <= 8 ||
         cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
             cudaSuccess)) {
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = dim3(static_cast<unsigned>(S), 1, 1);
      cfg.blockDim = dim3(kSkinnyThreads, 1, 1);
      cfg.dynamicSmemBytes = SkinnySmem<C>::kBytes;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = static_cast<unsigned>(S);
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
    slot = n > 0 ? n : -1;
  }
  return slot;
}

template <int C>
cudaError_t launch_skinny_c(const SkinnyParams& p0, int outs, int col_blocks, cudaStream_t st) {
  SkinnyParams p = p0;
  const long long Ktot = static_cast<long long>(p.K) * (p.ksum ? p.groups : 1);
  // about one CTA per SM: S K slices per column block, each at least 8 steps per warp and at
  // most kSkinnyMaxSlice steps, every cluster resident at once
  const long long blocks = static_cast<long long>(outs) * col_blocks;
  long long S = std::max(1LL, (device_sm_count() + blocks / 2) / blocks);
  S = std::min<long long>(S, kSkinnyMaxSplit);
  S = std::min<long long>(S, std::max(1LL, Ktot / (8 * kSkinnyWarps)));
  S = std::max<long long>(S, (Ktot + kSkinnyMaxSlice - 1) / kSkinnyMaxSlice);
  if (S > kSkinnyMaxSplit) return cudaErrorNotSupported;
  // every cluster resident at once (a second, partial wave would take as long as the first)
  while (S > 1) {
    const int c = skinny_max_active_clusters<C>(static_cast<int>(S));
    if (c <= 0 || c >= blocks) break;
    if ((Ktot + S - 2) / (S - 1) > kSkinnyMaxSlice) break;  // the slice must fit in shared memory
    --S;
  }
  p.slices = static_cast<int>(S);
  auto kern = skinny_gemm_kernel<C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SkinnySmem<C>::kBytes);
  if (e != cudaSuccess) return e;
  if (S > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(S), static_cast<unsigned>(col_blocks),
                     static_cast<unsigned>(outs));
  cfg.blockDim = dim3(kSkinnyThreads, 1, 1);
  cfg.dynamicSmemBytes = SkinnySmem<C>::kBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(S);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = tuning(TP_TUNE_PDL) != 0 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

bool aligned_to(const void* ptr, int bytes) {
  return reinterpret_cast<uintptr_t>(ptr) % static_cast<uintptr_t>(bytes) == 0;
}

}  // namespace

bool skinny_gemm_applies(const GemmSpec& s) {
  if (tuning(TP_TUNE_SKINNY) == 0) return false;
  if (s.M < 1 || s.M > kSkinnyRows || s.a_mn || !s.b_mn) return false;
  if (s.epi != EPI_STORE_F32 && s.epi != EPI_BIAS_ACT) return false;
  if (s.N % 2 != 0 || s.ldb % 2 != 0) return false;
  const long long ktot = s.K * (s.ksum ? s.groups : 1);
  if (ktot > static_cast<long long>(kSkinnyMaxSplit) * kSkinnyMaxSlice) return false;
  for (int g = 0; g < s.groups; ++g)
    if (!aligned_to(s.B[g], 8)) return false;
  return true;
}

cudaError_t launch_skinny_gemm(const GemmSpec& s, cudaStream_t st) {
  if (s.M <= 0 || s.N <= 0 || s.K <= 0) return cudaSuccess;
  SkinnyParams p{};
  for (int g = 0; g < s.groups; ++g) {
    p.A[g] = static_cast<const float*>(s.A[g]);
    p.B[g] = static_cast<const float*>(s.B[g]);
    p.D[g] = static_cast<float*>(s.D[g]);
    p.D2[g] = static_cast<float*>(s.D2[g]);
    p.bias[g] = static_cast<const float*>(s.bias[g]);
  }
  p.lda = s.lda;
  p.ldb = s.ldb;
  p.ldd = s.ldd;
  p.ldd2 = s.ldd2;
  p.M = static_cast<int>(s.M);
  p.N = static_cast<int>(s.N);
  p.K = static_cast<int>(s.K);
  p.groups = s.groups;
  p.ksum = s.ksum ? 1 : 0;  // as the general FFMA kernel: one summed output, or one per shard
  p.epi = s.epi;
  p.act = s.act;
  const int outs = p.ksum ? 1 : s.groups;
  bool vec4 = s.N % 4 == 0 && s.ldb % 4 == 0;
  for (int g = 0; g < s.groups && vec4; ++g) vec4 = aligned_to(s.B[g], 16);
  // 4 columns per lane unless that leaves too few CTAs to spread over the SMs
  const int blocks4 = static_cast<int>((s.N + 127) / 128) * outs;
  if (vec4 && blocks4 * kSkinnyMaxSplit >= device_sm_count())
    return launch_skinny_c<4>(p, outs, static_cast<int>((s.N + 127) / 128), st);
  return launch_skinny_c<2>(p, outs, static_cast<int>((s.N + 63) / 64), st);
}

}  // namespace tpk
