// Host-side interface between the C ABI layer (tp_api.cu) and the kernel launchers.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "tp_mlp.h"
#include "tp_mlp_tuning.h"

namespace tpk {

constexpr int kMaxShards = 64;

// Workspace layout: a 256-byte status block, then scratch (256-byte aligned).
constexpr size_t kStatusBytes = 256;
// bf16 calls reserve kTailBytes right after the status block: the fp32 pieces of the tensor-core GEMM's split
// tail tiles (at most kTailUnits pieces of 256 x 256 fp32), then one counter per (tile, 32-row
// block) of the split tiles.
constexpr int kTailUnits = 80;
constexpr size_t kTailPieceBytes = size_t(256) * 256 * 4;
constexpr size_t kTailCounterBytes = 4096;
constexpr size_t kTailBytes = TP_BF16_TAIL_SCRATCH_BYTES;
static_assert(kTailBytes == kTailUnits * kTailPieceBytes + kTailCounterBytes, "tail region");

// Device status codes written by kernels (first error wins).
constexpr int kDevTimeoutBase = 0x100;  // | (role << 4) | wait site

enum EpiKind : int {
  EPI_STORE_F32 = 0,      // D (fp32) = acc (+ bias[n] once, when bias != nullptr)
  EPI_BIAS_ACT = 1,       // H = acc + bias[n] -> D (optional), Y = act(H) -> D2  (bf16 / fp32)
  EPI_DACT = 2,           // D = acc * act'(aux[m,n])                               (bf16 / fp32)
  EPI_STORE_BF16 = 3,     // D (bf16) = acc (+ bias[n])                   (tensor-core GEMM only)
  EPI_PARTIAL_REDUCE = 4, // D[og] (fp32 partial og); the last writer of each block sums the
                          // partials into Z (+ zbias)                   (tensor-core GEMM only)
};

// One launch of a (grouped) GEMM: D_g[M,N] = A_g[M,K] * B_g[K,N] for every group g, or,
// with ksum, one D[M,N] = sum_g A_g B_g (K spans the groups in group order).
//  A element (m,k) at A[g] + (a_mn ? k*lda + m : m*lda + k)
//  B element (k,n) at B[g] + (b_mn ? k*ldb + n : n*ldb + k)
//  D element (m,n) at D[g] + m*ldd + n
struct GemmSpec {
  int64_t M = 0, N = 0, K = 0;
  int groups = 1;
  int ksum = 0;   // 1: one output, sum over all groups (shorthand for kpo = groups)
  int kpo = 0;    // groups summed per output (tensor-core GEMM only; 0: from ksum)
  int a_mn = 0, b_mn = 0;
  const void* A[kMaxShards] = {};
  const void* B[kMaxShards] = {};
  void* D[kMaxShards] = {};
  void* D2[kMaxShards] = {};
  const void* bias[kMaxShards] = {};
  const void* aux[kMaxShards] = {};
  int64_t lda = 0, ldb = 0, ldd = 0, ldd2 = 0, ldaux = 0;
  int epi = EPI_STORE_F32;
  int act = TP_ACT_NONE;
  int raster = 0;   // tensor-core GEMM tile order: 0 = m fastest, 1 = n fastest
  int* counters = nullptr;   // EPI_PARTIAL_REDUCE: one int per (32-row, 256-column) block, zero
  float* Z = nullptr;
  int64_t ldz = 0;
  const void* zbias = nullptr;
  int* status = nullptr;
  int kslices = 1;  // FFMA GEMM: K steps split over a cluster of this many CTAs per tile (1: none)
  // B is not written by the launch before this one on the stream (the caller knows: the row GEMM
  // of tp_mlp_forward follows the column GEMM, which writes only H_i and Y_i), so the few-row
  // fp32 GEMM may request B before waiting for that launch to finish
  int b_early = 0;
  // tensor-core GEMM on SM pairs: scratch for split tail tiles (nullptr: never split)
  float* tail_ws = nullptr;
  int* tail_counters = nullptr;
};

// bf16 inputs, tcgen05 tensor cores (sm_103a). Returns cudaSuccess or the launch error.
cudaError_t launch_tc_gemm(const GemmSpec& s, cudaStream_t st);
// Two independent bf16 GEMMs in one SM-pair launch, s0 with both operands MN-major, s1 with
// both K-major, at most 16 groups each, no EPI_PARTIAL_REDUCE. tc_dual_eligible says whether
// the two fit and (TP_TUNE_DUAL at AUTO) whether one launch is expected to beat two.
bool tc_dual_eligible(const GemmSpec& s0, const GemmSpec& s1);
cudaError_t launch_tc_gemm_dual(const GemmSpec& s0, const GemmSpec& s1, cudaStream_t st);
// fp32 inputs, FFMA (no TF32); kslices > 1 splits every tile's K steps over a cluster.
cudaError_t launch_simt_gemm(const GemmSpec& s, cudaStream_t st);
// The dynamic shared memory opt-in (cudaFuncSetAttribute) of kernel `kern` for at least
// `bytes` on the current device, made once per kernel and device: a driver call on every
// launch costs a few-microsecond launch measurable host time.
cudaError_t opt_in_dynamic_smem(const void* kern, int bytes);

// Tensor map of a 2-D fp32 row-major array [outer][inner] (row pitch ld elements), no swizzle,
// box box_outer x box_inner; false if the driver rejects it (alignment, sizes).
bool encode_f32_rows(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint64_t ld,
                     uint32_t box_inner, uint32_t box_outer);
// fp32 FFMA GEMM for at most 32 rows with bulk-copied operands (forward layouts: A K-major, B
// N-contiguous; K % 64 == 0, N % 4 == 0, 16-byte aligned rows; epilogue bias (+ act) only).
// few_rows_eligible says whether s fits it (and TP_TUNE_FEW_ROWS is not 0).
bool few_rows_eligible(const GemmSpec& s);
cudaError_t launch_few_rows_gemm(const GemmSpec& s, cudaStream_t st);
// K slices (cluster size, <= 8) for an FFMA GEMM whose tiles alone would leave SMs idle
// (1: no split). TP_TUNE_SIMT_SPLIT = 0 turns the split off.
int plan_simt_split(const GemmSpec& s);

// Z[T,N] = sum_{i<n} P[i][T,N] + bias (bias may be null; bias dtype: bf16 if bias_bf16).
cudaError_t launch_shard_reduce(const float* P, int n, int64_t T, int64_t N,
                                const void* bias, int bias_bf16, float* Z, cudaStream_t st);

// The same over bf16 partials (summed in fp32); N % 8 == 0.
cudaError_t launch_shard_reduce_bf16(const uint16_t* P, int n, int64_t T, int64_t N,
                                     const void* bias, float* Z, cudaStream_t st);

// n equal, contiguous blocks of `bytes` each: gather (full[j*bytes..] <- shard[j]) or scatter
// (shard[j] <- full[j*bytes..]), one launch for all blocks.
cudaError_t launch_shard_copy(void* const* shards, void* full, int n, size_t bytes, int gather,
                              cudaStream_t st);

// Column sums: out_s[c] = sum_{r<rows} in_s[r*ld_s + c] for every segment s.
struct ColsumSeg {
  const void* in;
  float* out;
  int64_t cols;
  int64_t ld;
};
cudaError_t launch_colsum(const ColsumSeg* segs, int nseg, int64_t rows, int in_bf16,
                          cudaStream_t st);

// dH = dY * act'(H) elementwise over n shards of [T, w] (ld for dY may differ: gathered).
cudaError_t launch_dact(const void* const* dY, int64_t ld_dy, const void* const* H,
                        void* const* dH, int n, int64_t T, int64_t w, int act, int bf16,
                        cudaStream_t st);

// LayerNorm over a hidden dimension split into n column shards of Hs columns (dtype bf16 or
// fp32 for X, Y, dY, gamma, beta; mean, rstd, dgamma, dbeta fp32). Arrays of n pointers;
// gamma, beta, dgamma, dbeta may be NULL arrays.
struct LnArgs {
  const void* const* X = nullptr;
  const void* const* gamma = nullptr;
  const void* const* beta = nullptr;
  void* const* Y = nullptr;  // forward: Y; backward: dX
  const void* const* dY = nullptr;
  float* const* dgamma = nullptr;
  float* const* dbeta = nullptr;
  float* mean = nullptr;
  float* rstd = nullptr;
  int64_t T = 0, Hs = 0;
  int n = 0;
  float eps = 0.f;
  int bf16 = 0;
};
cudaError_t launch_ln_forward(const LnArgs& a, cudaStream_t st);
cudaError_t launch_ln_backward_dx(const LnArgs& a, cudaStream_t st);
cudaError_t launch_ln_param_grads(const LnArgs& a, cudaStream_t st);

// One-block self-test of the bounded wait (see tp_selftest_wait_timeout).
cudaError_t launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t st);

// Number of partial outputs to split a shard-summed GEMM into (a divisor of n; 1 = fully
// fused): balances the tile waves against the extra reduction traffic.
int plan_shard_split(int64_t M, int64_t N, int64_t K_per_group, int n);

// Override of a measured kernel choice (tp_mlp_tuning.h): TP_TUNE_AUTO when none is set.
int tuning(int knob);

// Device facts (cached per device).
int device_sm_count();

// Sets the thread-local message that tp_last_error() returns.
void set_last_error(const char* msg);

}  // namespace tpk
