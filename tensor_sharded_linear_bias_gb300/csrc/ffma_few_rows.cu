// fp32 GEMM for products of at most 32 rows (few tokens: the pages' batch-32 example), FFMA
// only, forward layouts: A K-major [M, K] (M <= 32), B N-contiguous [K, N]; per-shard outputs or
// the shard sum, epilogue bias (+ GeLU).
//
// With so few rows the weights are the whole cost and every weight element is used M <= 32
// times, so the kernel is built around moving B once, in bulk, with as many bytes in flight as
// the SM can hold. A CTA owns 32 rows x 64 output columns and one contiguous slice of K (over
// all summed shards); its loader thread requests the slice in 64-deep chunks, up to eight
// chunks ahead (the 192 KiB ring: a slice of at most 8 chunks is requested at once): per chunk
// one TMA box of B (64 x 64) and one of A (32 x 64; rows past M read as zeros), both
// completing on one mbarrier. (One bulk copy per 256-byte row instead ran at
// ~3 us per chunk on GB300: the copy engine's cost is per operation, not per byte.) Eight
// compute warps split every chunk's 64 K steps into eight runs of 8; lane l keeps the 32 x 2
// outputs of columns 2l, 2l+1 in registers, and per 4 K steps does 4 8-byte shared loads of B,
// 32 16-byte broadcast loads of A and 128 paired FMAs (256 FMAs).
//
// Sums, all in a fixed order for a shape (results repeat bit for bit): per output, each warp
// over its K steps in order; the warps' partial tiles in warp order through shared memory; the
// S CTAs of a thread-block cluster (the K slices, S <= 8) in CTA order: each CTA pushes its
// sums into receive slots of the CTA that finishes them (distributed shared memory), CTA q
// finishing the q-th S-part of the tile's outputs (epilogue and store).
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "device_common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace tpk {
namespace {

constexpr int kFrRows = 32;                        // rows a CTA holds (M <= 32)
constexpr int kFrCols = 64;                        // output columns per CTA
constexpr int kFrChunk = 64;                       // K steps per pipeline stage
constexpr int kFrStages = 8;                       // chunks in flight: all of a slice of <= 8
constexpr int kFrWarps = 8;                        // compute warps; warp kFrWarps loads
constexpr int kFrThreads = 32 * (kFrWarps + 1);
constexpr int kFrMaxSlices = 8;                    // CTAs per cluster (portable size)
constexpr uint32_t kFrBBytes = kFrChunk * kFrCols * 4;     // B block of a chunk: 16 KiB
constexpr uint32_t kFrABytes = kFrRows * kFrChunk * 4;     // A block of a chunk: 8 KiB
constexpr uint32_t kFrStageBytes = kFrBBytes + kFrABytes;  // 24 KiB
constexpr int kFrTileFloats = kFrRows * kFrCols;           // 2048
// The ring is reused after the K loop for the warps' partial tiles.
static_assert(kFrWarps * kFrTileFloats * 4 <= kFrStages * kFrStageBytes, "partials fit");
// after the ring: the receive slots of the cluster sum (S slots of ceil(512 / S) groups of 4
// floats: at most kFrTileFloats + 28), then the barriers and a flag
constexpr int kFrRecvFloats = kFrTileFloats + 32;
constexpr int kFrSmem = kFrStages * kFrStageBytes + kFrRecvFloats * 4 + 2 * kFrStages * 8 + 16;

struct FewRowsParams {
  CUtensorMap tmA[kMaxShards];  // A_g [M][K]: boxes of 32 rows x 64 K
  CUtensorMap tmB[kMaxShards];  // B_g [K][N]: boxes of 64 K x 64 columns
  float* D[kMaxShards];
  float* D2[kMaxShards];
  const float* bias[kMaxShards];
  long long ldd, ldd2;
  int M, N, K;
  int groups, ksum, epi, act;
  int slices;  // CTAs per cluster = K slices of every output tile (1: no cluster)
  int* status;
  int b_early;  // B may be requested before the grid dependency wait (GemmSpec::b_early)
};

// One 2-D TMA box (x = inner coordinate, a multiple of 64 elements here) into this CTA's
// shared memory, completing on the mbarrier at bar.
__device__ __forceinline__ void tma_box(uint32_t dst, const CUtensorMap* map, int x, int y,
                                        uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// bias: the output column's bias value, loaded by the caller ahead of the sums (0 without one)
__device__ __forceinline__ void few_rows_epilogue(const FewRowsParams& p, int og, int m, int n,
                                                  float v, float bias) {
  if (p.bias[og] != nullptr) v += bias;
  if (p.epi == EPI_BIAS_ACT) {
    if (p.D[og] != nullptr) p.D[og][static_cast<long long>(m) * p.ldd + n] = v;
    p.D2[og][static_cast<long long>(m) * p.ldd2 + n] = (p.act == TP_ACT_GELU_ERF) ? gelu_erf(v) : v;
  } else {
    p.D[og][static_cast<long long>(m) * p.ldd + n] = v;
  }
}

__global__ void __launch_bounds__(kFrThreads, 1)
    few_rows_gemm_kernel(const __grid_constant__ FewRowsParams p) {
  extern __shared__ __align__(128) unsigned char fr_smem[];
  float* ring = reinterpret_cast<float*>(fr_smem);
  float* recv = reinterpret_cast<float*>(fr_smem + kFrStages * kFrStageBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(recv + kFrRecvFloats);
  volatile int* failed_flag = reinterpret_cast<volatile int*>(bars + 2 * kFrStages);
  const uint32_t ring_base = smem_addr(ring);
  const uint32_t bar_base = smem_addr(bars);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (kFrStages + s); };

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int S = p.slices;
  const int q = static_cast<int>(blockIdx.x);  // K slice = rank in the cluster
  const int n0 = static_cast<int>(blockIdx.y) * kFrCols;
  const int og = static_cast<int>(blockIdx.z);
  const int kgroups = p.ksum ? p.groups : 1;
  const int chunks_per_group = p.K / kFrChunk;
  const long long chunks = static_cast<long long>(chunks_per_group) * kgroups;
  const int c_lo = static_cast<int>(chunks * q / S);
  const int nchunks = static_cast<int>(chunks * (q + 1) / S) - c_lo;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kFrStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kFrWarps);
    }
    *failed_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  // With a programmatic launch this CTA may start while the previous kernel still runs. Where
  // B is known not to be that kernel's output, the first chunks' B boxes are requested now
  // (their A boxes, possibly the previous kernel's output, only after the wait below).
  int b_pre = 0;
  if (p.b_early && warp == kFrWarps && lane == 0) {
    b_pre = min(nchunks, kFrStages);
    for (int i = 0; i < b_pre; ++i) {
      const int c = c_lo + i;
      const int kg = c / chunks_per_group;
      const uint32_t sb = ring_base + static_cast<uint32_t>(i) * kFrStageBytes;
      mbar_arrive_expect_tx(full_bar(i), kFrStageBytes);
      tma_box(sb, &p.tmB[p.ksum ? kg : og], n0, (c - kg * chunks_per_group) * kFrChunk, full_bar(i));
    }
  }
  // from here on the previous kernel's results are visible
  grid_dependency_wait();
  grid_dependents_launch();

  // the two columns of a row as one pair: Blackwell's paired fp32 FMA (each half rounded as
  // the scalar fmaf) does both in one instruction, leaving issue slots for the shared loads
  float2 acc[kFrRows];
#pragma unroll
  for (int r = 0; r < kFrRows; ++r) acc[r] = make_float2(0.0f, 0.0f);

  if (warp == kFrWarps) {
    // ---------------------------------------------------------------- loader warp
    int issued = 0;
    for (int i = 0; i < nchunks && lane == 0; ++i) {
      const int s = i % kFrStages;
      const uint32_t ph = static_cast<uint32_t>(i / kFrStages) & 1u;
      if (i >= kFrStages &&  // the stage's previous chunk consumed by all compute warps
          !mbar_wait_bounded(empty_bar(s), ph ^ 1u, kWaitLimitNs)) {
        report_status(p.status, kDevTimeoutBase | 0x70);
        *failed_flag = 1;
        break;
      }
      const int c = c_lo + i;
      const int kg = c / chunks_per_group;
      const int kk = (c - kg * chunks_per_group) * kFrChunk;
      const int g = p.ksum ? kg : og;
      const uint32_t sb = ring_base + static_cast<uint32_t>(s) * kFrStageBytes;
      // full boxes land (zeros outside the arrays), so every chunk brings the same bytes
      if (i >= b_pre) {
        mbar_arrive_expect_tx(full_bar(s), kFrStageBytes);
        tma_box(sb, &p.tmB[g], n0, kk, full_bar(s));
      }
      tma_box(sb + kFrBBytes, &p.tmA[g], kk, 0, full_bar(s));
      ++issued;
    }
    __syncwarp();
    if (issued > 0 && *failed_flag) {
      // a compute warp gave up: copies it never waited for may still be landing
      const uint64_t t0 = global_ns();
      while (global_ns() - t0 < 2000000ull) {
      }
    }
  } else {
    // ---------------------------------------------------------------- compute warps
    for (int i = 0; i < nchunks; ++i) {
      const int s = i % kFrStages;
      const uint32_t ph = static_cast<uint32_t>(i / kFrStages) & 1u;
      if (!mbar_wait_bounded(full_bar(s), ph, kWaitLimitNs)) {
        if (lane == 0) {
          report_status(p.status, kDevTimeoutBase | 0x71);
          *failed_flag = 1;
        }
        break;
      }
      const float* Bs = ring + s * (kFrStageBytes / 4) + warp * 8 * kFrCols + 2 * lane;
      const float* As = ring + s * (kFrStageBytes / 4) + kFrBBytes / 4 + warp * 8;
#pragma unroll
      for (int kb = 0; kb < 2; ++kb) {
        float2 b[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          b[j] = *reinterpret_cast<const float2*>(Bs + (4 * kb + j) * kFrCols);
#pragma unroll
        for (int r = 0; r < kFrRows; ++r) {
          const float4 a = *reinterpret_cast<const float4*>(As + r * kFrChunk + 4 * kb);
          acc[r] = __ffma2_rn(make_float2(a.x, a.x), b[0], acc[r]);
          acc[r] = __ffma2_rn(make_float2(a.y, a.y), b[1], acc[r]);
          acc[r] = __ffma2_rn(make_float2(a.z, a.z), b[2], acc[r]);
          acc[r] = __ffma2_rn(make_float2(a.w, a.w), b[3], acc[r]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(s));
    }
  }

  // ------------------------------------------------------------------ sums and epilogue
  // Outputs go in groups of 4 consecutive columns of one row (512 groups per tile); CTA r of
  // the cluster finishes groups [r 512 / S, (r + 1) 512 / S). Each CTA adds its warps' partial
  // tiles in warp order and pushes every group's sum into the receive slot (its own rank) of
  // the CTA that finishes the group (remote shared-memory stores: no round trip waits on them);
  // after one cluster barrier each CTA adds its slots in CTA order and runs the epilogue.
  __syncthreads();  // every chunk consumed (or abandoned): the ring is free
  float* part = ring;  // [warp][row][col]
  if (warp < kFrWarps) {
#pragma unroll
    for (int r = 0; r < kFrRows; ++r)
      *reinterpret_cast<float2*>(part + (warp * kFrRows + r) * kFrCols + 2 * lane) =
          acc[r];
  }
  const bool ok = *failed_flag == 0;  // read before the barrier that makes every write visible
  const float* bias = p.bias[og];
  constexpr int kGroups = kFrTileFloats / 4;                       // 512
  constexpr int kPer = (kGroups + kFrThreads - 1) / kFrThreads;    // groups per thread
  const int g_lo = kGroups * q / S, g_hi = kGroups * (q + 1) / S;  // this CTA's groups
  const int slot = 4 * ((kGroups + S - 1) / S);                    // floats per receive slot
  // the bias of this CTA's groups, fetched while the sums are formed
  float4 bv[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int gi = g_lo + static_cast<int>(threadIdx.x) + j * kFrThreads;
    const int n = n0 + (4 * gi) % kFrCols;  // N % 4 == 0: a group's columns are all in or out
    bv[j] = (bias != nullptr && gi < g_hi && n < p.N)
                ? *reinterpret_cast<const float4*>(bias + n)
                : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  __syncthreads();
  auto warp_sum = [&](int gi) {
    float4 v = *reinterpret_cast<const float4*>(part + 4 * gi);
#pragma unroll
    for (int w = 1; w < kFrWarps; ++w) {
      const float4 x = *reinterpret_cast<const float4*>(part + w * kFrTileFloats + 4 * gi);
      v.x += x.x;
      v.y += x.y;
      v.z += x.z;
      v.w += x.w;
    }
    return v;
  };
  auto finish = [&](int gi, float4 v, float4 b) {
    const int o = 4 * gi, m = o / kFrCols, n = n0 + o % kFrCols;
    if (!ok || m >= p.M || n >= p.N) return;
    few_rows_epilogue(p, og, m, n, v.x, b.x);
    few_rows_epilogue(p, og, m, n + 1, v.y, b.y);
    few_rows_epilogue(p, og, m, n + 2, v.z, b.z);
    few_rows_epilogue(p, og, m, n + 3, v.w, b.w);
  };
  if (S == 1) {
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int gi = static_cast<int>(threadIdx.x) + j * kFrThreads;
      if (gi < kGroups) finish(gi, warp_sum(gi), bv[j]);
    }
    return;
  }
  cg::cluster_group cluster = cg::this_cluster();
  for (int gi = threadIdx.x; gi < kGroups; gi += kFrThreads) {
    // the finishing CTA: the r with r 512 / S <= gi < (r + 1) 512 / S
    int r = min(S - 1, gi * S / kGroups);
    while (r > 0 && gi < kGroups * r / S) --r;
    while (r + 1 < S && gi >= kGroups * (r + 1) / S) ++r;
    const int pos = 4 * (gi - kGroups * r / S);
    float* dst = cluster.map_shared_rank(recv, r) + q * slot + pos;
    *reinterpret_cast<float4*>(dst) = warp_sum(gi);
  }
  cluster.sync();  // every push has landed; after this no CTA touches another's memory
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int gi = g_lo + static_cast<int>(threadIdx.x) + j * kFrThreads;
    if (gi >= g_hi) continue;
    const int pos = 4 * (gi - g_lo);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int r = 0; r < S; ++r) {
      const float4 x = *reinterpret_cast<const float4*>(recv + r * slot + pos);
      v.x += x.x;
      v.y += x.y;
      v.z += x.z;
      v.w += x.w;
    }
    finish(gi, v, bv[j]);
  }
}

// How many clusters of S CTAs the device holds at once (the driver's answer, which accounts
// for a cluster having to fit within one GPC); cached per device.
int max_active_few_rows_clusters(int S) {
  static int cache[64][kFrMaxSlices + 1] = {};
  int dev = 0;
  if (S < 1 || S > kFrMaxSlices || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return 0;
  if (cache[dev][S] == 0) {
    int n = 0;
    if (cudaFuncSetAttribute(few_rows_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kFrSmem) == cudaSuccess) {
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = dim3(static_cast<unsigned>(S), 1, 1);
      cfg.blockDim = dim3(kFrThreads, 1, 1);
      cfg.dynamicSmemBytes = kFrSmem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = static_cast<unsigned>(S);
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, few_rows_gemm_kernel, &cfg) != cudaSuccess) n = 0;
    }
    cache[dev][S] = n > 0 ? n : -1;
  }
  return cache[dev][S];
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

}  // namespace

bool few_rows_eligible(const GemmSpec& s) {
  if (tuning(TP_TUNE_FEW_ROWS) == 0) return false;
  if (s.M < 1 || s.M > kFrRows || s.N < 1 || s.K < kFrChunk) return false;
  if (s.a_mn || !s.b_mn) return false;
  if (s.epi != EPI_STORE_F32 && s.epi != EPI_BIAS_ACT) return false;
  if (s.K % kFrChunk != 0 || s.N % 4 != 0 || s.lda % 4 != 0 || s.ldb % 4 != 0) return false;
  if (s.groups < 1 || s.groups > kMaxShards) return false;
  // outputs: one per group, or one sum of all groups (no partial grouping)
  if (s.kpo > 1 && !(s.ksum && s.kpo == s.groups)) return false;
  if ((s.N + kFrCols - 1) / kFrCols > 65535) return false;
  for (int g = 0; g < s.groups; ++g)
    if (!aligned16(s.A[g]) || !aligned16(s.B[g]) || !aligned16(s.bias[g])) return false;
  return true;
}

cudaError_t launch_few_rows_gemm(const GemmSpec& s, cudaStream_t st) {
  const int outs = s.ksum ? 1 : s.groups;
  const int col_tiles = static_cast<int>((s.N + kFrCols - 1) / kFrCols);
  const long long tiles = static_cast<long long>(col_tiles) * outs;
  const long long chunks = (s.K / kFrChunk) * (s.ksum ? s.groups : 1);
  // K slices: fill the SMs with one CTA each, at most 8 per cluster, at least one chunk per
  // slice, and every tile's cluster resident at once
  long long S = std::max<long long>(1, device_sm_count() / std::max<long long>(1, tiles));
  S = std::min<long long>({S, kFrMaxSlices, chunks});
  while (S > 1) {
    const int c = max_active_few_rows_clusters(static_cast<int>(S));
    if (c <= 0 || c >= tiles) break;  // c <= 0: no answer, keep the plan
    --S;
  }

  alignas(128) static thread_local FewRowsParams p;
  std::memset(static_cast<void*>(&p), 0, sizeof(p));
  static_assert(sizeof(FewRowsParams) <= 32764, "kernel parameter block too large");
  for (int g = 0; g < s.groups; ++g) {
    if (!encode_f32_rows(&p.tmA[g], s.A[g], s.K, s.M, s.lda, kFrChunk, kFrRows) ||
        !encode_f32_rows(&p.tmB[g], s.B[g], s.N, s.K, s.ldb, kFrCols, kFrChunk))
      return cudaErrorInvalidValue;
    p.D[g] = static_cast<float*>(s.D[g]);
    p.D2[g] = static_cast<float*>(s.D2[g]);
    p.bias[g] = static_cast<const float*>(s.bias[g]);
  }
  p.ldd = s.ldd;
  p.ldd2 = s.ldd2;
  p.M = static_cast<int>(s.M);
  p.N = static_cast<int>(s.N);
  p.K = static_cast<int>(s.K);
  p.groups = s.groups;
  p.ksum = s.ksum;
  p.epi = s.epi;
  p.act = s.act;
  p.slices = static_cast<int>(S);
  p.status = s.status;
  p.b_early = s.b_early;

  cudaError_t e = opt_in_dynamic_smem(reinterpret_cast<const void*>(few_rows_gemm_kernel), kFrSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(S), static_cast<unsigned>(col_tiles),
                     static_cast<unsigned>(outs));
  cfg.blockDim = dim3(kFrThreads, 1, 1);
  cfg.dynamicSmemBytes = kFrSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (S > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = static_cast<unsigned>(S);
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (tuning(TP_TUNE_PDL) != 0) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, few_rows_gemm_kernel, p);
}

}  // namespace tpk
