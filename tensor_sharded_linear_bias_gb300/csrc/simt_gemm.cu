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
// Products of at most 32 rows whose B is N-contiguous take skinny_gemm_kernel instead (below).
//
// Split K: when the output tiles alone cannot fill the GPU (few tokens), the K steps of every tile (over all summed shards) are cut into S <= 8
// contiguous ranges computed by the S CTAs of one thread-block cluster. Each CTA parks its
// partial tile in its shared memory; after a cluster barrier, CTA q adds rows q*TM/S ..
// (q+1)*TM/S-1 of all S partial tiles in CTA order (distributed shared memory), applies the
// epilogue and stores them. The order is fixed for a shape, so results repeat bit for bit;
// no partial tile goes through global memory.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>

#include "device_common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace tpk {
namespace {

constexpr int TN = 64, TK = 32, STAGES = 4;
constexpr long long kMinSplitSteps = 4;  // K steps (of TK) a split slice keeps at least
constexpr int kMaxSplit = 8;             // CTAs of a portable cluster

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

// ------------------------------------------------------------------ at most 32 rows
// Products of at most 32 rows with A row-major (K contiguous) and B N-contiguous -- the forward
// at few tokens, as in the pages' batch-32 example. The weights are streamed once: a block of
// 8 warps owns 64 output columns (2 per lane) for all <= 32 rows; its K range (a slice of the
// summed K when the cluster splits K) is staged transposed in shared memory once, each warp
// takes an eighth of it, and per K element a lane issues 8 vector shared loads (the 32 A values,
// broadcast), 2 B loads and 64 FFMAs. The warps' partial tiles are added in warp order, then the
// cluster's blocks in block order through distributed shared memory, then the epilogue.
constexpr int kSkCols = 64;          // output columns per block
constexpr int kSkRows = 32;          // rows held (M <= 32, zero-padded)
constexpr int kSkStride = 36;        // floats per staged K row (16-byte multiple)
constexpr int kSkMaxK = 640;         // staged K elements per block
constexpr int kSkPart = 8 * kSkRows * kSkCols;  // floats of the warps' partial tiles

__global__ void __launch_bounds__(256) skinny_gemm_kernel(const __grid_constant__ SimtParams p) {
  extern __shared__ __align__(16) float sk[];
  const int S = p.slices;
  const int g = static_cast<int>(blockIdx.z) / S;
  const int slice = static_cast<int>(blockIdx.z) % S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long n0 = static_cast<long long>(blockIdx.x) * kSkCols;
  const int kgroups = p.ksum ? p.groups : 1;
  const long long Kall = p.K * kgroups;
  const long long kb = Kall * slice / S, ke = Kall * (slice + 1) / S;
  const int L = static_cast<int>(ke - kb);
  float* As = sk;                               // [L][kSkStride], rows m >= M are 0
  float* red = sk + max(L * kSkStride, kSkPart);
  // stage A^T for this block's K range (consecutive threads: consecutive k of one row)
  for (int e = threadIdx.x; e < kSkRows * L; e += 256) {
    const int m = e / L, kl = e % L;
    const long long k = kb + kl;
    const int kg = static_cast<int>(k / p.K);
    const long long kk = k - kg * p.K;
    float v = 0.f;
    if (m < p.M) v = p.A[p.ksum ? kg : g][m * p.sam + kk];
    As[kl * kSkStride + m] = v;
  }
  __syncthreads();
  // this warp's share of the K range
  const int w0 = L * warp / 8, w1 = L * (warp + 1) / 8;
  const long long n = n0 + 2 * lane;
  float acc[kSkRows][2];
#pragma unroll
  for (int m = 0; m < kSkRows; ++m) acc[m][0] = acc[m][1] = 0.f;
  long long k = kb + w0;
  int kg = static_cast<int>(k / p.K);
  long long kk = k - kg * p.K;
  for (int kl = w0; kl < w1; ++kl) {
    const float* B = p.B[p.ksum ? kg : g] + kk * p.sbk;
    const float b0 = n < p.N ? B[n] : 0.f;
    const float b1 = n + 1 < p.N ? B[n + 1] : 0.f;
    const float4* a4 = reinterpret_cast<const float4*>(As + kl * kSkStride);
#pragma unroll
    for (int q = 0; q < kSkRows / 4; ++q) {
      const float4 a = a4[q];
      acc[4 * q][0] = fmaf(a.x, b0, acc[4 * q][0]);
      acc[4 * q][1] = fmaf(a.x, b1, acc[4 * q][1]);
      acc[4 * q + 1][0] = fmaf(a.y, b0, acc[4 * q + 1][0]);
      acc[4 * q + 1][1] = fmaf(a.y, b1, acc[4 * q + 1][1]);
      acc[4 * q + 2][0] = fmaf(a.z, b0, acc[4 * q + 2][0]);
      acc[4 * q + 2][1] = fmaf(a.z, b1, acc[4 * q + 2][1]);
      acc[4 * q + 3][0] = fmaf(a.w, b0, acc[4 * q + 3][0]);
      acc[4 * q + 3][1] = fmaf(a.w, b1, acc[4 * q + 3][1]);
    }
    if (++kk == p.K) {
      kk = 0;
      ++kg;
    }
  }
  __syncthreads();  // every warp is done reading As: its space takes the partial tiles
  float* part = sk;  // [warp][m][col]
#pragma unroll
  for (int m = 0; m < kSkRows; ++m) {
    part[(warp * kSkRows + m) * kSkCols + 2 * lane] = acc[m][0];
    part[(warp * kSkRows + m) * kSkCols + 2 * lane + 1] = acc[m][1];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < kSkRows * kSkCols; e += 256) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) v += part[w * kSkRows * kSkCols + e];
    red[e] = v;
  }
  const int og = p.ksum ? 0 : g;
  if (S == 1) {
    __syncthreads();
    for (int e = threadIdx.x; e < kSkRows * kSkCols; e += 256) {
      const int m = e / kSkCols;
      const long long c = n0 + e % kSkCols;
      if (m < p.M && c < p.N) epilogue(p, og, m, c, red[e]);
    }
    return;
  }
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  const int e0 = kSkRows * kSkCols * slice / S, e1 = kSkRows * kSkCols * (slice + 1) / S;
  for (int e = e0 + static_cast<int>(threadIdx.x); e < e1; e += 256) {
    float v = 0.f;
    for (int q = 0; q < S; ++q) v += cluster.map_shared_rank(red, q)[e];
    const int m = e / kSkCols;
    const long long c = n0 + e % kSkCols;
    if (m < p.M && c < p.N) epilogue(p, og, m, c, v);
  }
  cluster.sync();
}

// Blocks of the K split for the skinny kernel (0: not applicable).
int plan_skinny(const GemmSpec& s) {
  if (const char* env = std::getenv("TPMLP_SIMT_SKINNY"))
    if (std::atoi(env) == 0) return 0;
  if (s.M > kSkRows || s.a_mn || !s.b_mn) return 0;
  const long long outs = s.ksum ? 1 : s.groups;
  const long long blocks = ((s.N + kSkCols - 1) / kSkCols) * outs;
  const long long Kall = s.K * (s.ksum ? s.groups : 1);
  const long long target = 2LL * device_sm_count();
  long long S = std::max((target + blocks - 1) / blocks, (Kall + kSkMaxK - 1) / kSkMaxK);
  S = std::min<long long>(S, std::max(1LL, Kall / 64));  // at least 64 K elements per block
  S = std::min<long long>(S, kMaxSplit);                  // a portable cluster
  if ((Kall + S - 1) / S > kSkMaxK) return 0;             // the block's K range must fit
  return static_cast<int>(std::max(1LL, S));
}

cudaError_t launch_skinny(const SimtParams& p, long long col_blocks, cudaStream_t st) {
  const long long Kall = p.K * (p.ksum ? p.groups : 1);
  const int L = static_cast<int>((Kall + p.slices - 1) / p.slices);
  const int smem = static_cast<int>(sizeof(float)) *
                   (std::max(L * kSkStride, kSkPart) + kSkRows * kSkCols);
  cudaError_t e = cudaFuncSetAttribute(skinny_gemm_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned zg = p.ksum ? 1u : static_cast<unsigned>(p.groups);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(col_blocks), 1, zg * static_cast<unsigned>(p.slices));
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = static_cast<unsigned>(p.slices);
  cfg.attrs = attr;
  cfg.numAttrs = p.slices > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, skinny_gemm_kernel, p);
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
  cudaError_t e =
      cudaFuncSetAttribute(simt_gemm_kernel<TM>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
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

}  // namespace

int plan_simt_split(const GemmSpec& s) {
  if (s.M <= 0 || s.N <= 0 || s.K <= 0) return 1;
  if (const char* env = std::getenv("TPMLP_SIMT_SPLIT"))
    if (std::atoi(env) == 0) return 1;
  const long long outs = s.ksum ? 1 : s.groups;
  const long long TM = tile_rows(s.M);
  const long long tiles = ((s.N + TN - 1) / TN) * ((s.M + TM - 1) / TM) * outs;
  const long long target = 2LL * device_sm_count();  // CTAs: two per SM
  if (tiles >= target) return 1;
  const long long steps = ((s.K + TK - 1) / TK) * (s.ksum ? s.groups : 1);
  long long S = (target + tiles - 1) / tiles;
  S = std::min(S, steps / kMinSplitSteps);  // enough K steps per slice
  S = std::min<long long>(S, kMaxSplit);
  return S > 1 ? static_cast<int>(S) : 1;
}

cudaError_t launch_simt_gemm(const GemmSpec& s, cudaStream_t st) {
  if (s.M <= 0 || s.N <= 0 || s.K <= 0) return cudaSuccess;
  if (s.groups < 1 || s.groups > kMaxShards) return cudaErrorInvalidValue;
  if (s.kslices < 1 || s.kslices > kMaxSplit) return cudaErrorInvalidValue;
  const int skinny = plan_skinny(s);
  if (skinny > 0) {
    SimtParams p = make_params(s);
    p.slices = skinny;
    return launch_skinny(p, (s.N + kSkCols - 1) / kSkCols, st);
  }
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
