// fp32 GEMM on the CUDA cores (FFMA): the fp32 path, where tensor-core TF32 would not keep
// fp32 accuracy. Same grouping (per-shard outputs or a shard-summed output) and epilogues as
// the tensor-core GEMM, with fp32 everywhere.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"

namespace tpk {
namespace {

constexpr int TM = 64, TN = 64, TK = 16;

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
};

__global__ void __launch_bounds__(256) simt_gemm_kernel(const __grid_constant__ SimtParams p) {
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  const int g = blockIdx.z;
  const long long m0 = static_cast<long long>(blockIdx.y) * TM;
  const long long n0 = static_cast<long long>(blockIdx.x) * TN;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};

  const int kgroups = p.ksum ? p.groups : 1;
  for (int kg = 0; kg < kgroups; ++kg) {
    const float* A = p.A[p.ksum ? kg : g];
    const float* B = p.B[p.ksum ? kg : g];
    for (long long k0 = 0; k0 < p.K; k0 += TK) {
      for (int i = threadIdx.x; i < TM * TK; i += 256) {
        int mm, kk;
        if (p.sak == 1) { kk = i % TK; mm = i / TK; } else { mm = i % TM; kk = i / TM; }
        const long long m = m0 + mm, k = k0 + kk;
        As[kk][mm] = (m < p.M && k < p.K) ? A[m * p.sam + k * p.sak] : 0.0f;
      }
      for (int i = threadIdx.x; i < TN * TK; i += 256) {
        int nn, kk;
        if (p.sbk == 1) { kk = i % TK; nn = i / TK; } else { nn = i % TN; kk = i / TN; }
        const long long n = n0 + nn, k = k0 + kk;
        Bs[kk][nn] = (n < p.N && k < p.K) ? B[k * p.sbk + n * p.sbn] : 0.0f;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < TK; ++kk) {
        float a[4], b[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) a[r] = As[kk][ty + 16 * r];
#pragma unroll
        for (int c = 0; c < 4; ++c) b[c] = Bs[kk][tx + 16 * c];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
      }
      __syncthreads();
    }
  }

  const int og = p.ksum ? 0 : g;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const long long m = m0 + ty + 16 * r;
    if (m >= p.M) continue;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const long long n = n0 + tx + 16 * c;
      if (n >= p.N) continue;
      float v = acc[r][c];
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
  }
}

}  // namespace

cudaError_t launch_simt_gemm(const GemmSpec& s, cudaStream_t st) {
  if (s.M <= 0 || s.N <= 0 || s.K <= 0) return cudaSuccess;
  if (s.groups < 1 || s.groups > kMaxShards) return cudaErrorInvalidValue;
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
  const dim3 grid(static_cast<unsigned>((s.N + TN - 1) / TN),
                  static_cast<unsigned>((s.M + TM - 1) / TM), s.ksum ? 1u : s.groups);
  if (grid.y > 65535u) return cudaErrorInvalidValue;
  simt_gemm_kernel<<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace tpk
