// fp32 GEMM on the CUDA cores (FFMA): the fp32 path, where tensor-core TF32 would not keep
// fp32 accuracy. Same grouping (per-shard outputs or a shard-summed output) and epilogues as
// the tensor-core GEMM, with fp32 everywhere.
//
// Tiles of TM x 64 outputs (TM = 64, or 32 when the product has at most 32 rows), K steps of
// 32, a ring of STAGES shared-memory buffers filled by cp.async, so that several K steps' loads
// are in flight while one is multiplied. 256 threads: thread (ty, tx) owns rows RM*ty ..
// RM*ty+RM-1 (RM = TM/16) and columns 4tx .. 4tx+3; each K element costs one vector shared load
// of A, one of B and 4*RM FFMAs.
//
// Split K: when the output tiles alone cannot fill the GPU (few tokens, as in the pages'
// batch-32 example), the K steps of every tile (over all summed shards) are cut into S <= 16
// contiguous ranges computed by the S CTAs of one thread-block cluster. Each CTA parks its
// partial tile in its shared memory; after a cluster barrier, CTA q adds rows q*TM/S ..
// (q+1)*TM/S-1 of all S partial tiles in CTA order (distributed shared memory), applies the
// epilogue and stores them. The order is fixed for a shape, so results repeat bit for bit;
// no partial tile goes through global memory.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "device_common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace tpk {
namespace {

constexpr int TN = 64, TK = 32, STAGES = 4;
constexpr long long kMinSplitSteps = 4;  // K steps (of TK) a split slice keeps at least
constexpr int kMaxSplit = 16;            // CTAs of a cluster (above 8: non-portable size)

struct SimtParams {
  const float* A[kMaxShards];
  const float* B[kMaxShards];
  float* D[kMaxShards];
  float* D2[kMaxShards];
  const float* bias[kMaxShards];
  const float* aux[kMaxShards];
  long long sam, sak, sbk, sbn;
  long long ldd, ldd2, ldaux;
  long long M, N, K;
  int groups, ksum, epi, act;
  int slices;  // CTAs (one cluster) per output tile; 1: no split
};

// The epilogue of output element (m, n) of output og, given its accumulated value v.
__device__ __forceinline__ void epilogue(const SimtParams& p, int og, long long m, long long n,
                                         float v) {
  if (p.epi == EPI_STORE_F32) {
    if (p.bias[og] != nullptr) v += p.bias[og][n];
    p.D[og][m * p.ldd + n] = v;
  } else if (p.epi == EPI_BIAS_ACT) {
    if (p.bias[og] != nullptr) v += p.bias[og][n];
    if (p.D[og] != nullptr) p.D[og][m * p.ldd + n] = v;
    p.D2[og][m * p.ldd2 + n] = (p.act == TP_ACT_GELU_ERF) ? gelu_erf(v) : v;
  } else {  // EPI_DACT
    if (p.act == TP_ACT_GELU_ERF) v *= gelu_erf_grad(p.aux[og][m * p.ldaux + n]);
    p.D[og][m * p.ldd + n] = v;
  }
}

// 4-byte asynchronous copy global -> shared; with pred false nothing is read (src-size 0) and
// the 4 bytes are zero-filled (src must still be a valid address: the operand's base).
__device__ __forceinline__ void cp_async4(uint32_t d, const float* src, bool pred) {
  const int bytes = pred ? 4 : 0;
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(d),
               "l"(__cvta_generic_to_global(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int RM>
struct RowVec;
template <>
struct RowVec<2> {
  __device__ static void load(const float* p, float* a) {
    const float2 v = *reinterpret_cast<const float2*>(p);
    a[0] = v.x;
    a[1] = v.y;
  }
};
template <>
struct RowVec<4> {
  __device__ static void load(const float* p, float* a) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    a[0] = v.x;
    a[1] = v.y;
    a[2] = v.z;
    a[3] = v.w;
  }
};

template <int TM>
struct SimtSmem {
  float A[STAGES][TK][TM + 4];  // [k][m]: rows of 16-byte multiples for the vector reads
  float B[STAGES][TK][TN + 4];  // [k][n]
};

template <int TM>
__global__ void __launch_bounds__(256) simt_gemm_kernel(const __grid_constant__ SimtParams p) {
  constexpr int RM = TM / 16;
  constexpr int LOADS_A = TM * TK / 256;  // elements of A each thread copies per K step
  constexpr int LOADS_B = TK * TN / 256;  // elements of B
  extern __shared__ __align__(16) unsigned char simt_smem_raw[];
  SimtSmem<TM>& sm = *reinterpret_cast<SimtSmem<TM>*>(simt_smem_raw);
  const int S = p.slices;
  const int g = static_cast<int>(blockIdx.z) / S;      // output (or group)
  const int slice = static_cast<int>(blockIdx.z) % S;  // = rank in the cluster when S > 1
  const long long m0 = static_cast<long long>(blockIdx.y) * TM;
  const long long n0 = static_cast<long long>(blockIdx.x) * TN;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[RM][4] = {};

  const int kgroups = p.ksum ? p.groups : 1;
  const long long ksteps = (p.K + TK - 1) / TK;
  const long long all_steps = ksteps * kgroups;
  const long long s_begin = all_steps * slice / S;
  const long long s_end = all_steps * (slice + 1) / S;

  // Element e of a step's tile -> coordinates; consecutive threads follow whichever of the two
  // coordinates is contiguous in global memory (coalesced). A thread's elements keep their
  // coordinates from step to step, so their offsets are computed once: per step only the K
  // origin (and, summing shards, the operand) moves.
  long long a_off[LOADS_A], b_off[LOADS_B];
  int a_kk[LOADS_A], b_kk[LOADS_B];  // K coordinate inside the step; -1: row/column outside
  uint32_t a_dst[LOADS_A], b_dst[LOADS_B];  // shared addresses in stage 0
#pragma unroll
  for (int j = 0; j < LOADS_A; ++j) {
    const int e = threadIdx.x + 256 * j;
    int mm, kk;
    if (p.sak == 1) { kk = e % TK; mm = e / TK; } else { mm = e % TM; kk = e / TM; }
    const long long m = m0 + mm;
    a_off[j] = m * p.sam + kk * p.sak;
    a_kk[j] = m < p.M ? kk : -1;
    a_dst[j] = smem_addr(&sm.A[0][kk][mm]);
  }
#pragma unroll
  for (int j = 0; j < LOADS_B; ++j) {
    const int e = threadIdx.x + 256 * j;
    int nn, kk;
    if (p.sbk == 1) { kk = e % TK; nn = e / TK; } else { nn = e % TN; kk = e / TN; }
    const long long n = n0 + nn;
    b_off[j] = kk * p.sbk + n * p.sbn;
    b_kk[j] = n < p.N ? kk : -1;
    b_dst[j] = smem_addr(&sm.B[0][kk][nn]);
  }
  constexpr uint32_t A_STAGE = sizeof(float) * TK * (TM + 4);
  constexpr uint32_t B_STAGE = sizeof(float) * TK * (TN + 4);
  auto issue = [&](long long step, int buf) {
    const int kg = static_cast<int>(step / ksteps);
    const long long k0 = (step % ksteps) * TK;
    const int kmax = static_cast<int>(min(static_cast<long long>(TK), p.K - k0));
    const float* A = p.A[p.ksum ? kg : g] + k0 * p.sak;
    const float* B = p.B[p.ksum ? kg : g] + k0 * p.sbk;
#pragma unroll
    for (int j = 0; j < LOADS_A; ++j) {
      const bool in = a_kk[j] >= 0 && a_kk[j] < kmax;
      cp_async4(a_dst[j] + buf * A_STAGE, in ? A + a_off[j] : A, in);
    }
#pragma unroll
    for (int j = 0; j < LOADS_B; ++j) {
      const bool in = b_kk[j] >= 0 && b_kk[j] < kmax;
      cp_async4(b_dst[j] + buf * B_STAGE, in ? B + b_off[j] : B, in);
    }
  };

  // prologue: the first STAGES-1 steps in flight (one commit group per step, empty past the end)
#pragma unroll
  for (int i = 0; i < STAGES - 1; ++i) {
    if (s_begin + i < s_end) issue(s_begin + i, i);
    cp_async_commit();
  }
  for (long long step = s_begin; step < s_end; ++step) {
    const int buf = static_cast<int>((step - s_begin) % STAGES);
    cp_async_wait<STAGES - 2>();  // this step's group has landed (this thread's copies)
    __syncthreads();              // ... everyone's; and the buffer refilled below is free
    const long long nxt = step + STAGES - 1;
    if (nxt < s_end) issue(nxt, static_cast<int>((nxt - s_begin) % STAGES));
    cp_async_commit();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[RM], b[4];
      RowVec<RM>::load(&sm.A[buf][kk][RM * ty], a);
      RowVec<4>::load(&sm.B[buf][kk][4 * tx], b);
#pragma unroll
      for (int r = 0; r < RM; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
    }
  }
  cp_async_wait<0>();

  const int og = p.ksum ? 0 : g;
  if (S == 1) {
#pragma unroll
    for (int r = 0; r < RM; ++r) {
      const long long m = m0 + RM * ty + r;
      if (m >= p.M) continue;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const long long n = n0 + 4 * tx + c;
        if (n < p.N) epilogue(p, og, m, n, acc[r][c]);
      }
    }
    return;
  }

  // split K: park the partial tile in shared memory (the ring's A buffers, TM x TN floats),
  // then sum this CTA's share of rows over the cluster's CTAs in CTA order
  __syncthreads();  // every thread is done reading the ring
  float* part = &sm.A[0][0][0];
  static_assert(sizeof(sm.A) >= sizeof(float) * TM * TN, "partial tile fits the A ring");
#pragma unroll
  for (int r = 0; r < RM; ++r)
    *reinterpret_cast<float4*>(part + (RM * ty + r) * TN + 4 * tx) =
        make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  const int r0 = TM * slice / S, r1 = TM * (slice + 1) / S;
  for (int e = threadIdx.x; e < (r1 - r0) * TN; e += 256) {
    const int rr = r0 + e / TN, cc = e % TN;
    const long long m = m0 + rr, n = n0 + cc;
    float v = 0.0f;
    for (int q = 0; q < S; ++q) v += cluster.map_shared_rank(part, q)[rr * TN + cc];
    if (m < p.M && n < p.N) epilogue(p, og, m, n, v);
  }
  cluster.sync();  // no CTA leaves while another may still read its shared memory
}

int tile_rows(int64_t M) { return M <= 32 ? 32 : 64; }

SimtParams make_params(const GemmSpec& s) {
  SimtParams p{};
  for (int g = 0; g < s.groups; ++g) {
    p.A[g] = static_cast<const float*>(s.A[g]);
    p.B[g] = static_cast<const float*>(s.B[g]);
    p.D[g] = static_cast<float*>(s.D[g]);
    p.D2[g] = static_cast<float*>(s.D2[g]);
    p.bias[g] = static_cast<const float*>(s.bias[g]);
    p.aux[g] = static_cast<const float*>(s.aux[g]);
  }
  p.sam = s.a_mn ? 1 : s.lda;
  p.sak = s.a_mn ? s.lda : 1;
  p.sbk = s.b_mn ? s.ldb : 1;
  p.sbn = s.b_mn ? 1 : s.ldb;
  p.ldd = s.ldd;
  p.ldd2 = s.ldd2;
  p.ldaux = s.ldaux;
  p.M = s.M;
  p.N = s.N;
  p.K = s.K;
  p.groups = s.groups;
  p.ksum = s.ksum;
  p.epi = s.epi;
  p.act = s.act;
  p.slices = 1;
  return p;
}

template <int TM>
cudaError_t launch(const SimtParams& p, dim3 grid, cudaStream_t st) {
  constexpr int smem = static_cast<int>(sizeof(SimtSmem<TM>));  // > 48 KiB: opt in
  cudaError_t e = opt_in_dynamic_smem(reinterpret_cast<const void*>(simt_gemm_kernel<TM>), smem);
  if (e != cudaSuccess) return e;
  if (p.slices > 8) {
    e = cudaFuncSetAttribute(simt_gemm_kernel<TM>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  if (p.slices == 1) {
    simt_gemm_kernel<TM><<<grid, 256, smem, st>>>(p);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = static_cast<unsigned>(p.slices);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, simt_gemm_kernel<TM>, p);
}

// How many clusters of S CTAs of simt_gemm_kernel<TM> the device holds at once (the driver's
// answer, which accounts for a cluster having to fit within one GPC); cached per device.
template <int TM>
int max_active_clusters(int S) {
  static int cache[64][kMaxSplit + 1] = {};
  int dev = 0;
  if (S < 2 || S > kMaxSplit || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return 0;
  if (cache[dev][S] == 0) {
    constexpr int smem = static_cast<int>(sizeof(SimtSmem<TM>));
    int n = 0;
    if (cudaFuncSetAttribute(simt_gemm_kernel<TM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) == cudaSuccess &&
        (S <= 8 || cudaFuncSetAttribute(simt_gemm_kernel<TM>,
                                        cudaFuncAttributeNonPortableClusterSizeAllowed,
                                        1) == cudaSuccess)) {
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = dim3(1, 1, static_cast<unsigned>(S));
      cfg.blockDim = dim3(256, 1, 1);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 1;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = static_cast<unsigned>(S);
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, simt_gemm_kernel<TM>, &cfg) != cudaSuccess) n = 0;
    }
    cache[dev][S] = n > 0 ? n : -1;
  }
  return cache[dev][S];
}

}  // namespace

int plan_simt_split(const GemmSpec& s) {
  if (s.M <= 0 || s.N <= 0 || s.K <= 0) return 1;
  if (tuning(TP_TUNE_SIMT_SPLIT) == 0) return 1;
  const long long outs = s.ksum ? 1 : s.groups;
  const long long TM = tile_rows(s.M);
  const long long tiles = ((s.N + TN - 1) / TN) * ((s.M + TM - 1) / TM) * outs;
  const long long target = 2LL * device_sm_count();  // CTAs: two per SM
  if (tiles >= target) return 1;
  const long long steps = ((s.K + TK - 1) / TK) * (s.ksum ? s.groups : 1);
  long long S = (target + tiles - 1) / tiles;
  S = std::min(S, steps / kMinSplitSteps);  // enough K steps per slice
  S = std::min<long long>(S, kMaxSplit);
  // every tile's cluster resident at once: a second, partial wave of clusters would take as
  // long as the first
  while (S > 1) {
    const int c = TM == 32 ? max_active_clusters<32>(static_cast<int>(S))
                           : max_active_clusters<64>(static_cast<int>(S));
    if (c <= 0 || c >= tiles) break;  // c <= 0: no answer, keep the plan
    --S;
  }
  return S > 1 ? static_cast<int>(S) : 1;
}

cudaError_t launch_simt_gemm(const GemmSpec& s, cudaStream_t st) {
  if (s.M <= 0 || s.N <= 0 || s.K <= 0) return cudaSuccess;
  if (s.groups < 1 || s.groups > kMaxShards) return cudaErrorInvalidValue;
  if (s.kslices < 1 || s.kslices > kMaxSplit) return cudaErrorInvalidValue;
  SimtParams p = make_params(s);
  p.slices = s.kslices;
  const unsigned zg = s.ksum ? 1u : static_cast<unsigned>(s.groups);
  const int TM = tile_rows(s.M);
  const dim3 grid(static_cast<unsigned>((s.N + TN - 1) / TN),
                  static_cast<unsigned>((s.M + TM - 1) / TM), zg * static_cast<unsigned>(p.slices));
  if (grid.y > 65535u || grid.z > 65535u) return cudaErrorInvalidValue;
  return TM == 32 ? launch<32>(p, grid, st) : launch<64>(p, grid, st);
}

}  // namespace tpk
