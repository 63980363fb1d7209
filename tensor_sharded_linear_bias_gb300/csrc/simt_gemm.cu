// fp32 GEMM on the CUDA cores (FFMA): the fp32 path, where tensor-core TF32 would not keep
// fp32 accuracy. Same grouping (per-shard outputs or a shard-summed output) and epilogues as
// the tensor-core GEMM, with fp32 everywhere.
//
// Split K: when the output tiles alone cannot fill the GPU (few tokens, as in the pages'
// batch-32 example), the K steps of every tile (over all summed shards) are cut into
// `slices` contiguous ranges, one CTA each. Each CTA writes its raw partial tile to scratch;
// simt_split_sum_kernel then adds the slices in slice order (a fixed order: the result does
// not depend on scheduling) and applies the epilogue.
#include <cuda_runtime.h>

#include <algorithm>

#include "device_common.cuh"
#include "internal.h"

namespace tpk {
namespace {

// Tiles of TM x 64 outputs (TM = 64, or 32 when the product has at most 32 rows), K steps of 32.
// 256 threads: thread (ty, tx) owns rows RM*ty .. RM*ty+RM-1 (RM = TM/16) and columns
// 4tx .. 4tx+3, so each K element costs one vector shared load of A, one of B and 4*RM FFMAs.
constexpr int TN = 64, TK = 32;
constexpr long long kMinSplitSteps = 4;    // K steps (of TK) a split slice keeps at least
constexpr long long kMaxSplitSlices = 64;

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
  float* P;    // split K: partial tiles [slices][outs][M][N]
  int slices;  // 1: no split
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

// Two shared-memory buffers and a register prefetch: while the block multiplies the K step in
// one buffer, the loads of the next step are in flight, so the K loop is not a chain of
// load-latency-bound steps.
template <int TM>
__global__ void __launch_bounds__(256) simt_gemm_kernel(const __grid_constant__ SimtParams p) {
  constexpr int RM = TM / 16;
  constexpr int LOADS_A = TM * TK / 256;  // elements of A each thread stages per K step
  constexpr int LOADS_B = TK * TN / 256;  // elements of B
  __shared__ __align__(16) float As[2][TK][TM + 4];
  __shared__ __align__(16) float Bs[2][TK][TN + 4];
  const int zg = p.ksum ? 1 : p.groups;  // outputs
  const int g = static_cast<int>(blockIdx.z % zg);
  const int slice = static_cast<int>(blockIdx.z / zg);
  const long long m0 = static_cast<long long>(blockIdx.y) * TM;
  const long long n0 = static_cast<long long>(blockIdx.x) * TN;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[RM][4] = {};

  const int kgroups = p.ksum ? p.groups : 1;
  const long long ksteps = (p.K + TK - 1) / TK;
  const long long all_steps = ksteps * kgroups;
  // this CTA's contiguous range of K steps (all of them without a split)
  const long long s_begin = all_steps * slice / p.slices;
  const long long s_end = all_steps * (slice + 1) / p.slices;
  float ra[LOADS_A], rb[LOADS_B];

  // element e of a step's A tile -> (mm, kk); coalesced along whichever of m, k is contiguous
  auto a_coord = [&](int e, int& mm, int& kk) {
    if (p.sak == 1) { kk = e % TK; mm = e / TK; } else { mm = e % TM; kk = e / TM; }
  };
  auto b_coord = [&](int e, int& nn, int& kk) {
    if (p.sbk == 1) { kk = e % TK; nn = e / TK; } else { nn = e % TN; kk = e / TN; }
  };
  auto load = [&](long long step) {
    const int kg = static_cast<int>(step / ksteps);
    const long long k0 = (step % ksteps) * TK;
    const float* A = p.A[p.ksum ? kg : g];
    const float* B = p.B[p.ksum ? kg : g];
#pragma unroll
    for (int j = 0; j < LOADS_A; ++j) {
      int mm, kk;
      a_coord(threadIdx.x + 256 * j, mm, kk);
      const long long m = m0 + mm, k = k0 + kk;
      ra[j] = (m < p.M && k < p.K) ? A[m * p.sam + k * p.sak] : 0.0f;
    }
#pragma unroll
    for (int j = 0; j < LOADS_B; ++j) {
      int nn, kb;
      b_coord(threadIdx.x + 256 * j, nn, kb);
      const long long n = n0 + nn, k2 = k0 + kb;
      rb[j] = (n < p.N && k2 < p.K) ? B[k2 * p.sbk + n * p.sbn] : 0.0f;
    }
  };
  auto stash = [&](int buf) {
#pragma unroll
    for (int j = 0; j < LOADS_A; ++j) {
      int mm, kk;
      a_coord(threadIdx.x + 256 * j, mm, kk);
      As[buf][kk][mm] = ra[j];
    }
#pragma unroll
    for (int j = 0; j < LOADS_B; ++j) {
      int nn, kb;
      b_coord(threadIdx.x + 256 * j, nn, kb);
      Bs[buf][kb][nn] = rb[j];
    }
  };

  if (s_begin < s_end) {
    load(s_begin);
    stash(0);
  }
  __syncthreads();
  for (long long step = s_begin; step < s_end; ++step) {
    const int buf = static_cast<int>((step - s_begin) & 1);
    if (step + 1 < s_end) load(step + 1);
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[RM], b[4];
      RowVec<RM>::load(&As[buf][kk][RM * ty], a);
      RowVec<4>::load(&Bs[buf][kk][4 * tx], b);
#pragma unroll
      for (int r = 0; r < RM; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
    }
    if (step + 1 < s_end) stash(buf ^ 1);
    __syncthreads();
  }

  const int og = p.ksum ? 0 : g;
  float* part = p.slices > 1 ? p.P + (static_cast<long long>(slice) * zg + og) * p.M * p.N : nullptr;
#pragma unroll
  for (int r = 0; r < RM; ++r) {
    const long long m = m0 + RM * ty + r;
    if (m >= p.M) continue;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const long long n = n0 + 4 * tx + c;
      if (n >= p.N) continue;
      if (part != nullptr)
        part[m * p.N + n] = acc[r][c];
      else
        epilogue(p, og, m, n, acc[r][c]);
    }
  }
}

// Sum of the K-slice partials in slice order, then the epilogue; one thread per element of
// [outs][M][N] (consecutive threads along n: coalesced).
__global__ void __launch_bounds__(256) simt_split_sum_kernel(const __grid_constant__ SimtParams p) {
  const int zg = p.ksum ? 1 : p.groups;
  const long long mn = p.M * p.N;
  const long long total = zg * mn;
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < total; i += 256LL * gridDim.x) {
    const int og = static_cast<int>(i / mn);
    const long long r = i - og * mn;
    // eight slices' loads in flight at a time, added in slice order
    const float* src = p.P + static_cast<long long>(og) * mn + r;
    const long long slice_stride = zg * mn;
    float v = 0.0f;
    int s = 0;
    for (; s + 8 <= p.slices; s += 8) {
      float t[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) t[u] = src[(s + u) * slice_stride];
#pragma unroll
      for (int u = 0; u < 8; ++u) v += t[u];
    }
    for (; s < p.slices; ++s) v += src[s * slice_stride];
    epilogue(p, og, r / p.N, r % p.N, v);
  }
}

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
  p.slices = s.kslices > 1 ? s.kslices : 1;
  p.P = p.slices > 1 ? s.split : nullptr;
  return p;
}

}  // namespace

namespace {
int tile_rows(int64_t M) { return M <= 32 ? 32 : 64; }
}  // namespace

int plan_simt_split(const GemmSpec& s, size_t scratch_bytes) {
  if (s.M <= 0 || s.N <= 0 || s.K <= 0) return 1;
  const long long outs = s.ksum ? 1 : s.groups;
  const long long TM = tile_rows(s.M);
  const long long tiles = ((s.N + TN - 1) / TN) * ((s.M + TM - 1) / TM) * outs;
  const long long target = 2LL * device_sm_count();  // CTAs: two per SM
  if (tiles >= target) return 1;
  const long long steps = ((s.K + TK - 1) / TK) * (s.ksum ? s.groups : 1);
  long long S = (target + tiles - 1) / tiles;
  S = std::min(S, steps / kMinSplitSteps);                        // enough K steps per slice
  S = std::min<long long>(S, kMaxSplitSlices);
  const long long per_slice = outs * s.M * s.N * 4;
  if (per_slice > 0) S = std::min<long long>(S, static_cast<long long>(scratch_bytes) / per_slice);
  return S > 1 ? static_cast<int>(S) : 1;
}

cudaError_t launch_simt_gemm(const GemmSpec& s, cudaStream_t st) {
  if (s.M <= 0 || s.N <= 0 || s.K <= 0) return cudaSuccess;
  if (s.groups < 1 || s.groups > kMaxShards) return cudaErrorInvalidValue;
  if (s.kslices > 1 && s.split == nullptr) return cudaErrorInvalidValue;
  const SimtParams p = make_params(s);
  const unsigned zg = s.ksum ? 1u : static_cast<unsigned>(s.groups);
  const int TM = tile_rows(s.M);
  const dim3 grid(static_cast<unsigned>((s.N + TN - 1) / TN),
                  static_cast<unsigned>((s.M + TM - 1) / TM), zg * static_cast<unsigned>(p.slices));
  if (grid.y > 65535u || grid.z > 65535u) return cudaErrorInvalidValue;
  if (TM == 32)
    simt_gemm_kernel<32><<<grid, 256, 0, st>>>(p);
  else
    simt_gemm_kernel<64><<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_simt_split_sum(const GemmSpec& s, cudaStream_t st) {
  if (s.M <= 0 || s.N <= 0 || s.kslices <= 1) return cudaSuccess;
  if (s.split == nullptr) return cudaErrorInvalidValue;
  const SimtParams p = make_params(s);
  const long long total = (s.ksum ? 1LL : s.groups) * s.M * s.N;
  const long long blocks = std::min<long long>((total + 255) / 256, 8LL * device_sm_count());
  simt_split_sum_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace tpk
