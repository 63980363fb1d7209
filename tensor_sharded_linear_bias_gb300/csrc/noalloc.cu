// Row-parallel linear forward (partials form) for callers that cannot allocate device memory:
// its scratch -- the status word and the per-shard fp32 partial products -- lives in one
// file-scope static device array that the library carries, instead of a caller-allocated
// workspace. It reuses the library's GEMM and shard-reduction launchers unchanged.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "internal.h"
#include "tp_mlp.h"

namespace {

// 32 MiB: 256 bytes of status block + up to (32 MiB - 256 B) / 4 fp32 partial elements
// (n * T * N of them). Every GPU that loads the library holds this array until exit.
constexpr size_t kScratchBytes = size_t(32) << 20;
constexpr size_t kStatusBytes = tpk::kStatusBytes;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

tp_status fail(tp_status st, const char* msg) {
  tpk::set_last_error(msg);
  return st;
}

// Device address of the array on the current device. In host code the array's name is only
// a host-side stand-in, so the address is looked up once per device (with that device
// current) and cached.
cudaError_t scratch_on_current_device(void** out) {
  static void* addr[kMaxDevices] = {};
  static std::mutex mu;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

// After the shard reduction: if a GEMM wait ran out (a code in the static status word, which
// no caller can read), Z is overwritten with NaN so that the failure cannot pass for a
// result. One block; it reads the word and returns at once when it is zero.
__global__ void poison_on_timeout(const int* status, float* Z, long long count) {
  if (*reinterpret_cast<const volatile int*>(status) == 0) return;
  const float nan = __int_as_float(0x7fc00000);
  for (long long i = threadIdx.x; i < count; i += blockDim.x) Z[i] = nan;
}

bool aligned(const void* p, int dtype) {
  return reinterpret_cast<uintptr_t>(p) % (dtype == TP_BF16 ? 16 : 4) == 0;
}

}  // namespace

extern "C" tp_status tp_linear_row_forward_noalloc(const tp_linear_desc* desc,
                                                   const void* const* X, const void* const* W,
                                                   const void* bias, void* Z, void* stream) {
  char msg[256];
  if (desc == nullptr) return fail(TP_ERR_NULL, "desc is NULL");
  const int dt = desc->dtype;
  const int n = desc->tp_degree;
  const int64_t T = desc->tokens, K = desc->in_features, N = desc->out_features;
  if (dt != TP_F32 && dt != TP_BF16) return fail(TP_ERR_DTYPE, "unknown dtype");
  if (desc->act != TP_ACT_NONE) return fail(TP_ERR_DTYPE, "a row-parallel linear has no activation");
  if (desc->gather != 0) return fail(TP_ERR_DTYPE, "gather applies to column-parallel linears only");
  if (n < 1 || n > tpk::kMaxShards) return fail(TP_ERR_SHAPE, "tp_degree outside 1..64");
  const int64_t kMaxDim = int64_t(1) << 30;
  if (T < 0 || T > kMaxDim || K < 1 || K > kMaxDim || N < 1 || N > kMaxDim)
    return fail(TP_ERR_SHAPE, "tokens, in_features or out_features out of range");
  if (K % n != 0) return fail(TP_ERR_INDIVISIBLE, "in_features is not divisible by tp_degree");
  const int64_t Ks = K / n;
  if (dt == TP_BF16 && (Ks % 8 != 0 || N % 8 != 0))
    return fail(TP_ERR_ALIGN, "bf16 needs in_features / tp_degree and out_features to be multiples of 8");
  // n * T * N fp32 partials must fit behind the status block; checked factor by factor so
  // that no product can wrap around before the comparison
  const uint64_t max_elems = (kScratchBytes - kStatusBytes) / 4;
  const uint64_t per_token = uint64_t(n) * uint64_t(N);  // <= 2^36: no wrap
  if (per_token > max_elems || (T > 0 && uint64_t(T) > max_elems / per_token)) {
    std::snprintf(msg, sizeof(msg),
                  "needs %llu x %lld x %lld fp32 partials (tp_degree x tokens x out_features) "
                  "plus 256 bytes of scratch; the static scratch of this entry point holds %zu "
                  "bytes",
                  static_cast<unsigned long long>(n), static_cast<long long>(T),
                  static_cast<long long>(N), kScratchBytes);
    return fail(TP_ERR_WORKSPACE, msg);
  }
  if (T > 0) {
    if (X == nullptr || Z == nullptr) return fail(TP_ERR_NULL, "X (array) or Z is NULL");
    if (!aligned(Z, dt)) return fail(TP_ERR_ALIGN, "Z is not aligned");
    for (int i = 0; i < n; ++i)
      if (X[i] == nullptr || !aligned(X[i], dt)) return fail(TP_ERR_ALIGN, "X[i] is NULL or not aligned");
  }
  if (W == nullptr) return fail(TP_ERR_NULL, "W (array) is NULL");
  for (int i = 0; i < n; ++i)
    if (W[i] == nullptr || !aligned(W[i], dt)) return fail(TP_ERR_ALIGN, "W[i] is NULL or not aligned");
  if (bias != nullptr && !aligned(bias, dt)) return fail(TP_ERR_ALIGN, "bias is not aligned");

  int dev = -1, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return fail(TP_ERR_ARCH, "no CUDA device is available");
  }
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return fail(TP_ERR_ARCH, "this library is built for sm_103a");
  if (T == 0) {
    tpk::set_last_error("");
    return TP_OK;
  }

  void* scratch = nullptr;
  cudaError_t e = scratch_on_current_device(&scratch);
  if (e != cudaSuccess) {
    std::snprintf(msg, sizeof(msg), "cudaGetSymbolAddress of the static scratch: %s",
                  cudaGetErrorString(e));
    return fail(TP_ERR_CUDA, msg);
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = static_cast<int*>(scratch);
  float* P = reinterpret_cast<float*>(static_cast<unsigned char*>(scratch) + kStatusBytes);

  // The status word must start at zero; the partials are fully overwritten by the GEMM.
  e = cudaMemsetAsync(status, 0, kStatusBytes, st);
  if (e == cudaSuccess) {
    tpk::GemmSpec s;
    s.M = T;
    s.N = N;
    s.K = Ks;
    s.groups = n;
    s.ksum = 0;
    s.a_mn = 0;
    s.b_mn = 1;
    s.lda = Ks;
    s.ldb = N;
    s.ldd = N;
    s.epi = tpk::EPI_STORE_F32;
    s.status = status;
    for (int i = 0; i < n; ++i) {
      s.A[i] = X[i];
      s.B[i] = W[i];
      s.D[i] = P + size_t(i) * size_t(T) * size_t(N);
    }
    e = dt == TP_BF16 ? tpk::launch_tc_gemm(s, st) : tpk::launch_simt_gemm(s, st);
  }
  if (e == cudaSuccess)
    e = tpk::launch_shard_reduce(P, n, T, N, bias, dt == TP_BF16, static_cast<float*>(Z), st);
  if (e == cudaSuccess) {
    poison_on_timeout<<<1, 256, 0, st>>>(status, static_cast<float*>(Z), T * N);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    std::snprintf(msg, sizeof(msg), "launch: %s", cudaGetErrorString(e));
    return fail(TP_ERR_CUDA, msg);
  }
  tpk::set_last_error("");
  return TP_OK;
}
