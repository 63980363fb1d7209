// The C ABI (include/tp_mlp.h): argument validation, workspace sizing, and the launch plan
// of each entry point. Every step of the computation runs in this library's kernels; the
// host code only checks arguments and enqueues launches on the caller's stream.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"
#include "tp_mlp.h"

using namespace tpk;

namespace {

thread_local std::string g_last_error;

}  // namespace

void tpk::set_last_error(const char* msg) { g_last_error = msg; }

namespace {

tp_status fail(tp_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

tp_status ok() {
  g_last_error.clear();
  return TP_OK;
}

constexpr int64_t kMaxDim = int64_t(1) << 30;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t elem_size(int dtype) { return dtype == TP_BF16 ? 2 : 4; }

tp_status check_common(int64_t tokens, int tp, int dtype, int act, int reduce) {
  if (dtype != TP_F32 && dtype != TP_BF16) return fail(TP_ERR_DTYPE, "unknown dtype %d", dtype);
  if (act != TP_ACT_NONE && act != TP_ACT_GELU_ERF)
    return fail(TP_ERR_DTYPE, "unknown activation %d", act);
  if (reduce < TP_REDUCE_FUSED || reduce > TP_REDUCE_OVERLAP)
    return fail(TP_ERR_DTYPE, "unknown reduce mode %d", reduce);
  if ((reduce == TP_REDUCE_PARTIALS_BF16 || reduce == TP_REDUCE_OVERLAP) && dtype != TP_BF16)
    return fail(TP_ERR_DTYPE, "reduce mode %d needs bf16 inputs", reduce);
  if (tp < 1 || tp > kMaxShards)
    return fail(TP_ERR_SHAPE, "tp_degree %d outside 1..%d", tp, kMaxShards);
  if (tokens < 0 || tokens > kMaxDim) return fail(TP_ERR_SHAPE, "tokens %lld out of range",
                                                  static_cast<long long>(tokens));
  return TP_OK;
}

tp_status check_dim(const char* name, int64_t v) {
  if (v < 1 || v > kMaxDim)
    return fail(TP_ERR_SHAPE, "%s = %lld out of range 1..2^30", name, static_cast<long long>(v));
  return TP_OK;
}

// bf16: 16-byte pointers and widths that are multiples of 8 (TMA rows of 16-byte multiples).
tp_status check_width(int dtype, const char* name, int64_t v) {
  if (dtype == TP_BF16 && v % 8 != 0)
    return fail(TP_ERR_ALIGN, "bf16 needs %s (%lld) to be a multiple of 8", name,
                static_cast<long long>(v));
  return TP_OK;
}

tp_status check_ptr(int dtype, const char* name, const void* p, bool required) {
  if (p == nullptr) {
    if (required) return fail(TP_ERR_NULL, "%s is NULL", name);
    return TP_OK;
  }
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  const uintptr_t need = dtype == TP_BF16 ? 16 : 4;
  if (a % need != 0)
    return fail(TP_ERR_ALIGN, "%s is not %u-byte aligned", name, static_cast<unsigned>(need));
  return TP_OK;
}

// A host array of n device pointers. `required`: the array must be given. `elems`: when the
// array is given, every element must be non-NULL (token-sized buffers of a call with zero
// tokens may be NULL: they are never touched).
tp_status check_ptr_array(int dtype, const char* name, const void* const* arr, int n,
                          bool required, bool elems = true) {
  if (arr == nullptr) {
    if (required) return fail(TP_ERR_NULL, "%s (array) is NULL", name);
    return TP_OK;
  }
  char buf[64];
  for (int i = 0; i < n; ++i) {
    std::snprintf(buf, sizeof(buf), "%s[%d]", name, i);
    tp_status s = check_ptr(dtype, buf, arr[i], elems);
    if (s != TP_OK) return s;
  }
  return TP_OK;
}


tp_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (ws == nullptr) return fail(TP_ERR_WORKSPACE, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(ws) % 256 != 0)
    return fail(TP_ERR_ALIGN, "workspace must be 256-byte aligned");
  if (ws_bytes < need)
    return fail(TP_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed",
                ws_bytes, need);
  return TP_OK;
}

tp_status check_arch() {
  static int arch_state[64] = {};  // 0 unknown, 1 ok, 2 bad
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return fail(TP_ERR_ARCH, "no CUDA device is available");
  }
  if (dev >= 64) return fail(TP_ERR_ARCH, "device index %d out of range", dev);
  if (arch_state[dev] == 0) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    arch_state[dev] = (major == 10 && minor == 3) ? 1 : 2;
    if (arch_state[dev] == 2)
      return fail(TP_ERR_ARCH, "device %d is sm_%d%d; this library is built for sm_103a", dev,
                  major, minor);
  }
  if (arch_state[dev] == 2) return fail(TP_ERR_ARCH, "device %d is not sm_103", dev);
  return TP_OK;
}

tp_status cuda_fail(cudaError_t e, const char* what) {
  return fail(TP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int* status_word(void* ws) { return static_cast<int*>(ws); }

// First byte of a call's scratch: after the status block and, for bf16, the split tail tiles.
size_t scratch_base(int dtype) { return kStatusBytes + (dtype == TP_BF16 ? kTailBytes : 0); }

// A GEMM's view of the workspace: the status word and, for bf16, the tail-split region.
void bind_ws(GemmSpec& s, void* ws, int dtype) {
  char* region = static_cast<char*>(ws) + kStatusBytes;
  s.status = status_word(ws);
  s.tail_ws = dtype == TP_BF16 ? reinterpret_cast<float*>(region) : nullptr;
  s.tail_counters =
      dtype == TP_BF16 ? reinterpret_cast<int*>(region + kTailUnits * kTailPieceBytes) : nullptr;
}

template <typename T>
T* ws_at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// ---------------------------------------------------------------- launch tracing
struct TraceSlot {
  cudaEvent_t start = nullptr, stop = nullptr;
  int kernel = 0, tag = 0, groups = 0;
  double flops = 0, bytes = 0;
  bool recorded = false;
};

struct Trace {
  std::mutex mu;
  bool on = false;
  std::vector<TraceSlot> slots;
  size_t used = 0;
};

Trace& trace() {
  static Trace t;
  return t;
}

// Runs `launch` on stream st; while tracing is on, brackets it with two events and notes
// the launch's algorithmic work.
template <class F>
cudaError_t traced(int kernel, int tag, int groups, double flops, double bytes, cudaStream_t st,
                   F&& launch) {
  Trace& t = trace();
  TraceSlot* slot = nullptr;
  {
    std::lock_guard<std::mutex> lk(t.mu);
    if (t.on && t.used < t.slots.size()) slot = &t.slots[t.used++];
  }
  if (slot != nullptr) cudaEventRecord(slot->start, st);
  const cudaError_t e = launch();
  if (slot != nullptr) {
    cudaEventRecord(slot->stop, st);
    slot->kernel = kernel;
    slot->tag = tag;
    slot->groups = groups;
    slot->flops = flops;
    slot->bytes = bytes;
    slot->recorded = true;
  }
  return e;
}

// Algorithmic work of a GEMM launch: 2*M*N*K per shard; every distinct operand buffer read
// once, every output written once.
void gemm_work(const GemmSpec& s, int dtype, double* flops, double* bytes) {
  const double e = dtype == TP_BF16 ? 2.0 : 4.0;
  const double M = double(s.M), N = double(s.N), K = double(s.K);
  *flops = 2.0 * M * N * K * s.groups;
  int distinctA = 0, distinctB = 0;
  for (int g = 0; g < s.groups; ++g) {
    bool seenA = false, seenB = false;
    for (int h = 0; h < g; ++h) {
      seenA = seenA || s.A[h] == s.A[g];
      seenB = seenB || s.B[h] == s.B[g];
    }
    distinctA += !seenA;
    distinctB += !seenB;
  }
  const int outs = s.groups / (s.kpo > 0 ? s.kpo : (s.ksum ? s.groups : 1));
  double out_e = 4.0;
  if (s.epi != EPI_STORE_F32) out_e = e * ((s.epi == EPI_BIAS_ACT && s.D[0] != nullptr) ? 2 : 1);
  double aux = (s.epi == EPI_DACT && s.act != TP_ACT_NONE) ? e * M * N * outs : 0.0;
  *bytes = e * (M * K * distinctA + K * N * distinctB) + out_e * M * N * outs + aux;
}

cudaError_t run_gemm(const GemmSpec& s, int dtype, cudaStream_t st, int tag) {
  double flops = 0, bytes = 0;
  gemm_work(s, dtype, &flops, &bytes);
  if (dtype == TP_BF16)
    return traced(TP_K_GEMM_TC, tag, s.groups, flops, bytes, st, [&] { return launch_tc_gemm(s, st); });
  if (few_rows_eligible(s))
    return traced(TP_K_GEMM_FFMA, tag, s.groups, flops, bytes, st,
                  [&] { return launch_few_rows_gemm(s, st); });
  GemmSpec t = s;
  t.kslices = plan_simt_split(s);
  return traced(TP_K_GEMM_FFMA, tag, s.groups, flops, bytes, st,
                [&] { return launch_simt_gemm(t, st); });
}

// Two independent bf16 GEMMs in one launch (tc_dual_eligible), traced as one launch.
cudaError_t run_gemm_dual(const GemmSpec& s0, const GemmSpec& s1, int dtype, cudaStream_t st,
                          int tag) {
  double f0 = 0, b0 = 0, f1 = 0, b1 = 0;
  gemm_work(s0, dtype, &f0, &b0);
  gemm_work(s1, dtype, &f1, &b1);
  return traced(TP_K_GEMM_TC, tag, s0.groups + s1.groups, f0 + f1, b0 + b1, st,
                [&] { return launch_tc_gemm_dual(s0, s1, st); });
}

// Zero `rows` x `cols` fp32 outputs (a GEMM over zero tokens).
cudaError_t zero_f32(void* p, int64_t count, cudaStream_t st) {
  if (p == nullptr || count == 0) return cudaSuccess;
  return cudaMemsetAsync(p, 0, static_cast<size_t>(count) * 4, st);
}

#define TP_TRY(expr)                    \
  do {                                  \
    tp_status _s = (expr);              \
    if (_s != TP_OK) return _s;         \
  } while (0)

#define TP_CUDA(expr, what)                          \
  do {                                               \
    cudaError_t _e = (expr);                         \
    if (_e != cudaSuccess) return cuda_fail(_e, what); \
  } while (0)

// Bytes of one element of a shard partial.
size_t partial_bytes(int reduce) { return reduce == TP_REDUCE_PARTIALS_BF16 ? 2 : 4; }

// Counters of the overlapped reduction: one int per (32-row, 256-column) block of [M, N].
size_t counter_bytes(int reduce, int64_t M, int64_t N) {
  if (reduce != TP_REDUCE_OVERLAP) return 0;
  return align256(size_t((M + 31) / 32) * size_t((N + 255) / 256) * 4);
}

// Scratch of one shard-summed product: n partials, then the counters.
size_t partials_region(int reduce, int n, int64_t M, int64_t N) {
  if (reduce == TP_REDUCE_FUSED) return 0;
  return align256(size_t(n) * size_t(M) * size_t(N) * partial_bytes(reduce)) +
         counter_bytes(reduce, M, N);
}

// ---------------------------------------------------------------- MLP sizes
struct MlpSizes {
  int64_t T, H, F, Fs;
  int n;
  size_t partials_fwd, dH, partials_bwd, total;
};

tp_status mlp_validate(const tp_mlp_desc* d, MlpSizes* z) {
  if (d == nullptr) return fail(TP_ERR_NULL, "desc is NULL");
  TP_TRY(check_common(d->tokens, d->tp_degree, d->dtype, d->act, d->reduce));
  TP_TRY(check_dim("hidden", d->hidden));
  TP_TRY(check_dim("ffn", d->ffn));
  if (d->ffn % d->tp_degree != 0)
    return fail(TP_ERR_INDIVISIBLE, "ffn %lld is not divisible by tp_degree %d",
                static_cast<long long>(d->ffn), d->tp_degree);
  z->T = d->tokens;
  z->H = d->hidden;
  z->F = d->ffn;
  z->n = d->tp_degree;
  z->Fs = d->ffn / d->tp_degree;
  TP_TRY(check_width(d->dtype, "hidden", z->H));
  TP_TRY(check_width(d->dtype, "ffn / tp_degree", z->Fs));
  const size_t e = elem_size(d->dtype);
  z->partials_fwd =
      partials_region(d->reduce, z->n, z->T, z->H);
  z->dH = align256(size_t(z->T) * z->F * e);
  z->partials_bwd = z->partials_fwd;
  z->total = scratch_base(d->dtype) + std::max(z->partials_fwd, z->dH + z->partials_bwd);
  return TP_OK;
}

// ---------------------------------------------------------------- linear sizes
struct LinSizes {
  int64_t T, K, N, Ks, Ns;
  int n;
  size_t partials_fwd, dH, partials_bwd, total;
};

tp_status lin_validate(const tp_linear_desc* d, int kind, LinSizes* z) {
  if (d == nullptr) return fail(TP_ERR_NULL, "desc is NULL");
  if (kind != TP_COLUMN && kind != TP_ROW) return fail(TP_ERR_DTYPE, "unknown linear kind %d", kind);
  TP_TRY(check_common(d->tokens, d->tp_degree, d->dtype, d->act, d->reduce));
  TP_TRY(check_dim("in_features", d->in_features));
  TP_TRY(check_dim("out_features", d->out_features));
  if (d->gather != 0 && d->gather != 1) return fail(TP_ERR_DTYPE, "gather must be 0 or 1");
  z->T = d->tokens;
  z->K = d->in_features;
  z->N = d->out_features;
  z->n = d->tp_degree;
  const size_t e = elem_size(d->dtype);
  if (kind == TP_COLUMN) {
    if (z->N % z->n != 0)
      return fail(TP_ERR_INDIVISIBLE, "out_features %lld is not divisible by tp_degree %d",
                  static_cast<long long>(z->N), z->n);
    z->Ns = z->N / z->n;
    z->Ks = z->K;
    TP_TRY(check_width(d->dtype, "in_features", z->K));
    TP_TRY(check_width(d->dtype, "out_features / tp_degree", z->Ns));
    z->partials_fwd = 0;
    z->dH = d->act != TP_ACT_NONE ? align256(size_t(z->T) * z->N * e) : 0;
    z->partials_bwd =
        partials_region(d->reduce, z->n, z->T, z->K);
  } else {
    if (d->act != TP_ACT_NONE) return fail(TP_ERR_DTYPE, "a row-parallel linear has no activation");
    if (d->gather != 0) return fail(TP_ERR_DTYPE, "gather applies to column-parallel linears only");
    if (z->K % z->n != 0)
      return fail(TP_ERR_INDIVISIBLE, "in_features %lld is not divisible by tp_degree %d",
                  static_cast<long long>(z->K), z->n);
    z->Ks = z->K / z->n;
    z->Ns = z->N;
    TP_TRY(check_width(d->dtype, "in_features / tp_degree", z->Ks));
    TP_TRY(check_width(d->dtype, "out_features", z->N));
    z->partials_fwd =
        partials_region(d->reduce, z->n, z->T, z->N);
    z->dH = 0;
    z->partials_bwd = 0;
  }
  z->total = scratch_base(d->dtype) + std::max(z->partials_fwd, z->dH + z->partials_bwd);
  return TP_OK;
}

// Number of partial outputs of a shard-summed product: 1 (fused), n (partials), or the
// planner's choice (bf16 AUTO).
int shard_split(int reduce, int dtype, int64_t M, int64_t N, int64_t K, int n) {
  if (reduce == TP_REDUCE_FUSED) return 1;
  if (reduce == TP_REDUCE_PARTIALS || reduce == TP_REDUCE_PARTIALS_BF16) return n;
  return dtype == TP_BF16 ? plan_shard_split(M, N, K, n) : 1;  // AUTO, OVERLAP
}

// The overlapped form of a split shard sum: S partials in the workspace, counters after the
// n-partial region, Z written by the GEMM's own epilogue warps.
tp_status overlapped_sum(GemmSpec& s, int dtype, int S, int n, int64_t M, int64_t N,
                         const void* bias, float* Z, void* ws, size_t partials_off,
                         cudaStream_t st, int tag, const char* what) {
  float* P = ws_at<float>(ws, partials_off);
  int* counters = ws_at<int>(ws, partials_off + align256(size_t(n) * M * N * 4));
  TP_CUDA(cudaMemsetAsync(counters, 0, counter_bytes(TP_REDUCE_OVERLAP, M, N), st),
          "clearing the partial-sum counters");
  s.kpo = n / S;
  s.epi = EPI_PARTIAL_REDUCE;
  for (int i = 0; i < S; ++i) s.D[i] = P + size_t(i) * M * N;
  s.counters = counters;
  s.Z = Z;
  s.ldz = N;
  s.zbias = bias;
  TP_CUDA(run_gemm(s, dtype, st, tag), what);
  return TP_OK;
}

cudaError_t reduce_traced(const float* P, int n, int64_t T, int64_t N, const void* bias,
                          int bias_bf16, float* Z, cudaStream_t st) {
  const double bytes = (4.0 * n + 4.0) * double(T) * N + (bias ? (bias_bf16 ? 2.0 : 4.0) * N : 0.0);
  return traced(TP_K_SHARD_REDUCE, TP_TAG_REDUCE, n, double(n - 1) * T * N + (bias ? T * N : 0),
                bytes, st, [&] { return launch_shard_reduce(P, n, T, N, bias, bias_bf16, Z, st); });
}

cudaError_t reduce_bf16_traced(const uint16_t* P, int n, int64_t T, int64_t N, const void* bias,
                               float* Z, cudaStream_t st) {
  const double bytes = (2.0 * n + 4.0) * double(T) * N + (bias ? 2.0 * N : 0.0);
  return traced(TP_K_SHARD_REDUCE, TP_TAG_REDUCE, n, double(n - 1) * T * N + (bias ? T * N : 0),
                bytes, st, [&] { return launch_shard_reduce_bf16(P, n, T, N, bias, Z, st); });
}

// Row-parallel product Z = sum_i X_i W_i + bias, fused or through partials.
// X_i [T, Ks] (ld ldx), W_i [Ks, N] row-major (MN-major B), Z fp32 [T, N].
tp_status row_product(int dtype, int reduce, int n, int64_t T, int64_t Ks, int64_t N,
                      const void* const* X, int64_t ldx, const void* const* W, const void* bias,
                      float* Z, void* ws, size_t partials_off, cudaStream_t st, const char* what,
                      bool w_early = false) {
  GemmSpec s;
  s.b_early = w_early ? 1 : 0;
  s.M = T;
  s.N = N;
  s.K = Ks;
  s.groups = n;
  s.a_mn = 0;
  s.b_mn = 1;
  s.lda = ldx;
  s.ldb = N;
  s.ldd = N;
  s.epi = EPI_STORE_F32;
  bind_ws(s, ws, dtype);
  for (int i = 0; i < n; ++i) {
    s.A[i] = X[i];
    s.B[i] = W[i];
  }
  const int S = shard_split(reduce, dtype, T, N, Ks, n);
  if (S == 1) {
    s.ksum = 1;
    s.D[0] = Z;
    s.bias[0] = bias;
    TP_CUDA(run_gemm(s, dtype, st, TP_TAG_ROW_FWD), what);
  } else if (reduce == TP_REDUCE_OVERLAP) {
    TP_TRY(overlapped_sum(s, dtype, S, n, T, N, bias, Z, ws, partials_off, st, TP_TAG_ROW_FWD,
                          what));
  } else {
    s.kpo = n / S;
    if (reduce == TP_REDUCE_PARTIALS_BF16) {
      uint16_t* P = ws_at<uint16_t>(ws, partials_off);
      s.epi = EPI_STORE_BF16;
      for (int i = 0; i < S; ++i) s.D[i] = P + size_t(i) * T * N;
      TP_CUDA(run_gemm(s, dtype, st, TP_TAG_ROW_FWD), what);
      TP_CUDA(reduce_bf16_traced(P, S, T, N, bias, Z, st), "shard reduce");
    } else {
      float* P = ws_at<float>(ws, partials_off);
      for (int i = 0; i < S; ++i) s.D[i] = P + size_t(i) * T * N;
      TP_CUDA(run_gemm(s, dtype, st, TP_TAG_ROW_FWD), what);
      TP_CUDA(reduce_traced(P, S, T, N, bias, dtype == TP_BF16, Z, st), "shard reduce");
    }
  }
  return TP_OK;
}

// dX = sum_i dH_i W_i^T, dH_i [T, w] (ld ldh), W_i [Kd, w] row-major (K-major B).
// dX = sum_i dH_i W_i^T before its outputs are set: dH_i [T, w] (ld ldh), W_i [Kd, w], both
// K-major operands.
GemmSpec dgrad_spec(int dtype, int n, int64_t T, int64_t w, int64_t Kd, const void* const* dH,
                    int64_t ldh, const void* const* W, void* ws) {
  GemmSpec s;
  s.M = T;
  s.N = Kd;
  s.K = w;
  s.groups = n;
  s.a_mn = 0;
  s.b_mn = 0;
  s.lda = ldh;
  s.ldb = w;
  s.ldd = Kd;
  s.epi = EPI_STORE_F32;
  bind_ws(s, ws, dtype);
  for (int i = 0; i < n; ++i) {
    s.A[i] = dH[i];
    s.B[i] = W[i];
  }
  return s;
}

tp_status input_grad_sum(int dtype, int reduce, int n, int64_t T, int64_t w, int64_t Kd,
                         const void* const* dH, int64_t ldh, const void* const* W, float* dX,
                         void* ws, size_t partials_off, cudaStream_t st) {
  GemmSpec s = dgrad_spec(dtype, n, T, w, Kd, dH, ldh, W, ws);
  const int S = shard_split(reduce, dtype, T, Kd, w, n);
  if (S == 1) {
    s.ksum = 1;
    s.D[0] = dX;
    TP_CUDA(run_gemm(s, dtype, st, TP_TAG_COLUMN_DGRAD), "input-gradient GEMM");
  } else if (reduce == TP_REDUCE_OVERLAP) {
    TP_TRY(overlapped_sum(s, dtype, S, n, T, Kd, nullptr, dX, ws, partials_off, st,
                          TP_TAG_COLUMN_DGRAD, "input-gradient GEMM"));
  } else {
    s.kpo = n / S;
    if (reduce == TP_REDUCE_PARTIALS_BF16) {
      uint16_t* P = ws_at<uint16_t>(ws, partials_off);
      s.epi = EPI_STORE_BF16;
      for (int i = 0; i < S; ++i) s.D[i] = P + size_t(i) * T * Kd;
      TP_CUDA(run_gemm(s, dtype, st, TP_TAG_COLUMN_DGRAD), "input-gradient GEMM");
      TP_CUDA(reduce_bf16_traced(P, S, T, Kd, nullptr, dX, st), "shard reduce");
    } else {
      float* P = ws_at<float>(ws, partials_off);
      for (int i = 0; i < S; ++i) s.D[i] = P + size_t(i) * T * Kd;
      TP_CUDA(run_gemm(s, dtype, st, TP_TAG_COLUMN_DGRAD), "input-gradient GEMM");
      TP_CUDA(reduce_traced(P, S, T, Kd, nullptr, 0, dX, st), "shard reduce");
    }
  }
  return TP_OK;
}

// dW_i = Xa_i^T Gb_i for every shard: Xa_i [T, M] (ld lda), Gb_i [T, N] (ld ldb): both
// MN-major operands of a GEMM over the T tokens. dW_i fp32 [M, N].
GemmSpec wgrad_spec(int dtype, int n, int64_t T, int64_t M, int64_t N, const void* const* Xa,
                    int64_t lda, const void* const* Gb, int64_t ldb, void* const* dW, void* ws) {
  GemmSpec s;
  s.M = M;
  s.N = N;
  s.K = T;
  s.groups = n;
  s.a_mn = 1;
  s.b_mn = 1;
  s.lda = lda;
  s.ldb = ldb;
  s.ldd = N;
  s.epi = EPI_STORE_F32;
  bind_ws(s, ws, dtype);
  for (int i = 0; i < n; ++i) {
    s.A[i] = Xa[i];
    s.B[i] = Gb[i];
    s.D[i] = dW[i];
  }
  return s;
}

tp_status weight_grads(int dtype, int n, int64_t T, int64_t M, int64_t N,
                       const void* const* Xa, int64_t lda, const void* const* Gb, int64_t ldb,
                       void* const* dW, void* ws, cudaStream_t st, int tag) {
  if (T == 0) {
    for (int i = 0; i < n; ++i) TP_CUDA(zero_f32(dW[i], M * N, st), "zeroing weight gradient");
    return TP_OK;
  }
  const GemmSpec s = wgrad_spec(dtype, n, T, M, N, Xa, lda, Gb, ldb, dW, ws);
  TP_CUDA(run_gemm(s, dtype, st, tag), "weight-gradient GEMM");
  return TP_OK;
}

tp_status colsums(int dtype, int64_t T, const ColsumSeg* segs, int nseg, cudaStream_t st) {
  if (nseg == 0) return TP_OK;
  if (T == 0) {
    for (int s = 0; s < nseg; ++s) TP_CUDA(zero_f32(segs[s].out, segs[s].cols, st), "zeroing bias gradient");
    return TP_OK;
  }
  double bytes = 0;
  for (int s = 0; s < nseg; ++s) bytes += double(segs[s].cols) * (double(T) * (dtype == TP_BF16 ? 2 : 4) + 4);
  TP_CUDA(traced(TP_K_COLSUM, TP_TAG_BIAS_GRAD, nseg, 0.0, bytes, st,
                 [&] { return launch_colsum(segs, nseg, T, dtype == TP_BF16, st); }),
          "bias-gradient column sums");
  return TP_OK;
}

}  // namespace

extern "C" {

int32_t tp_version(void) { return 100; }

const char* tp_last_error(void) { return g_last_error.c_str(); }

tp_status tp_mlp_workspace_size(const tp_mlp_desc* desc, size_t* bytes) {
  if (bytes == nullptr) return fail(TP_ERR_NULL, "bytes is NULL");
  MlpSizes z{};
  TP_TRY(mlp_validate(desc, &z));
  *bytes = z.total;
  return ok();
}

tp_status tp_linear_workspace_size(const tp_linear_desc* desc, int32_t kind, size_t* bytes) {
  if (bytes == nullptr) return fail(TP_ERR_NULL, "bytes is NULL");
  LinSizes z{};
  TP_TRY(lin_validate(desc, kind, &z));
  *bytes = z.total;
  return ok();
}

tp_status tp_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  TP_TRY(check_ws(ws, ws_bytes, kStatusBytes));
  TP_TRY(check_arch());
  TP_CUDA(cudaMemsetAsync(ws, 0, kStatusBytes, static_cast<cudaStream_t>(stream)),
          "clearing the status word");
  return ok();
}

tp_status tp_check_status(void* ws, size_t ws_bytes, void* stream) {
  TP_TRY(check_ws(ws, ws_bytes, kStatusBytes));
  TP_TRY(check_arch());
  int code = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  TP_CUDA(cudaMemcpyAsync(&code, ws, sizeof(int), cudaMemcpyDeviceToHost, st), "reading status");
  TP_CUDA(cudaStreamSynchronize(st), "stream synchronise");
  if (code != 0)
    return fail(TP_ERR_DEVICE_TIMEOUT, "a device-side wait ran out (status code 0x%x)", code);
  return ok();
}

tp_status tp_trace_start(int32_t capacity) {
  if (capacity < 1 || capacity > 1000000)
    return fail(TP_ERR_SHAPE, "trace capacity %d outside 1..1000000", capacity);
  TP_TRY(check_arch());
  Trace& t = trace();
  std::lock_guard<std::mutex> lk(t.mu);
  if (t.on) return fail(TP_ERR_DTYPE, "tracing is already on");
  t.slots.assign(size_t(capacity), TraceSlot{});
  for (auto& sl : t.slots) {
    if (cudaEventCreate(&sl.start) != cudaSuccess || cudaEventCreate(&sl.stop) != cudaSuccess)
      return cuda_fail(cudaGetLastError(), "creating trace events");
  }
  t.used = 0;
  t.on = true;
  return ok();
}

tp_status tp_trace_stop(tp_trace_record* out, int32_t capacity, int32_t* count) {
  if (count == nullptr) return fail(TP_ERR_NULL, "count is NULL");
  if (out == nullptr && capacity > 0) return fail(TP_ERR_NULL, "out is NULL");
  Trace& t = trace();
  std::lock_guard<std::mutex> lk(t.mu);
  if (!t.on) return fail(TP_ERR_DTYPE, "tracing is not on");
  t.on = false;
  tp_status st = TP_OK;
  int32_t k = 0;
  for (size_t i = 0; i < t.used; ++i) {
    TraceSlot& sl = t.slots[i];
    if (!sl.recorded) continue;
    float ms = 0.f;
    if (cudaEventSynchronize(sl.stop) != cudaSuccess ||
        cudaEventElapsedTime(&ms, sl.start, sl.stop) != cudaSuccess) {
      st = cuda_fail(cudaGetLastError(), "reading trace events");
      break;
    }
    if (k < capacity) {
      out[k].kernel = sl.kernel;
      out[k].tag = sl.tag;
      out[k].flops = sl.flops;
      out[k].bytes = sl.bytes;
      out[k].ms = ms;
      out[k].groups = sl.groups;
    }
    ++k;
  }
  for (auto& sl : t.slots) {
    if (sl.start) cudaEventDestroy(sl.start);
    if (sl.stop) cudaEventDestroy(sl.stop);
  }
  t.slots.clear();
  t.used = 0;
  *count = std::min(k, capacity);
  if (st != TP_OK) return st;
  return ok();
}

tp_status tp_selftest_wait_timeout(void* ws, size_t ws_bytes, uint32_t limit_us, void* stream) {
  TP_TRY(check_ws(ws, ws_bytes, kStatusBytes));
  if (limit_us < 1 || limit_us > 1000000)
    return fail(TP_ERR_SHAPE, "limit_us %u outside 1..1000000", limit_us);
  TP_TRY(check_arch());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  TP_CUDA(traced(TP_K_SELFTEST, TP_TAG_OTHER, 1, 0.0, 0.0, st,
                 [&] { return launch_wait_selftest(status_word(ws), uint64_t(limit_us) * 1000, st); }),
          "wait self-test launch");
  return ok();
}

// ------------------------------------------------------------------ MLP
tp_status tp_mlp_forward(const tp_mlp_desc* desc, const void* X, const void* const* A,
                         const void* const* a, const void* const* B, const void* b, void* Z,
                         void* const* Hsave, void* const* Ysave, void* ws, size_t ws_bytes,
                         void* stream) {
  MlpSizes z{};
  TP_TRY(mlp_validate(desc, &z));
  const int dt = desc->dtype;
  const int n = z.n;
  TP_TRY(check_ptr(dt, "X", X, z.T > 0));
  TP_TRY(check_ptr_array(dt, "A", A, n, true));
  TP_TRY(check_ptr_array(dt, "a", a, n, false));
  TP_TRY(check_ptr_array(dt, "B", B, n, true));
  TP_TRY(check_ptr(dt, "b", b, false));
  TP_TRY(check_ptr(dt, "Z", Z, z.T > 0));
  TP_TRY(check_ptr_array(dt, "Ysave", reinterpret_cast<const void* const*>(Ysave), n, z.T > 0, z.T > 0));
  TP_TRY(check_ptr_array(dt, "Hsave", reinterpret_cast<const void* const*>(Hsave), n,
                         z.T > 0 && desc->act != TP_ACT_NONE, z.T > 0));
  TP_TRY(check_ws(ws, ws_bytes, z.total));
  TP_TRY(check_arch());
  if (z.T == 0) return ok();
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  // Column-parallel linear with the bias + activation epilogue: H_i, Y_i = act(H_i).
  GemmSpec c;
  c.M = z.T;
  c.N = z.Fs;
  c.K = z.H;
  c.groups = n;
  c.a_mn = 0;
  c.b_mn = 1;
  c.lda = z.H;
  c.ldb = z.Fs;
  c.ldd = z.Fs;
  c.ldd2 = z.Fs;
  c.epi = EPI_BIAS_ACT;
  c.act = desc->act;
  bind_ws(c, ws, dt);
  for (int i = 0; i < n; ++i) {
    c.A[i] = X;
    c.B[i] = A[i];
    c.bias[i] = a ? a[i] : nullptr;
    c.D[i] = Hsave ? Hsave[i] : nullptr;
    c.D2[i] = Ysave[i];
  }
  TP_CUDA(run_gemm(c, dt, st, TP_TAG_COLUMN_FWD), "column GEMM");

  // Row-parallel linear: Z = sum_i Y_i B_i + b.
  TP_TRY(row_product(dt, desc->reduce, n, z.T, z.Fs, z.H,
                     reinterpret_cast<const void* const*>(Ysave), z.Fs, B, b,
                     static_cast<float*>(Z), ws, scratch_base(dt), st, "row GEMM",
                     /*w_early=*/true));
  return ok();
}

tp_status tp_mlp_backward(const tp_mlp_desc* desc, const void* X, const void* const* A,
                          const void* const* B, const void* const* Hsave,
                          const void* const* Ysave, const void* dZ, void* dX, void* const* dA,
                          void* const* da, void* const* dB, void* db, void* ws, size_t ws_bytes,
                          void* stream) {
  MlpSizes z{};
  TP_TRY(mlp_validate(desc, &z));
  const int dt = desc->dtype;
  const int n = z.n;
  TP_TRY(check_ptr(dt, "X", X, z.T > 0));
  TP_TRY(check_ptr_array(dt, "A", A, n, true));
  TP_TRY(check_ptr_array(dt, "B", B, n, true));
  TP_TRY(check_ptr_array(dt, "Hsave", Hsave, n, z.T > 0 && desc->act != TP_ACT_NONE, z.T > 0));
  TP_TRY(check_ptr_array(dt, "Ysave", Ysave, n, z.T > 0, z.T > 0));
  TP_TRY(check_ptr(dt, "dZ", dZ, z.T > 0));
  TP_TRY(check_ptr(dt, "dX", dX, z.T > 0));
  TP_TRY(check_ptr_array(dt, "dA", reinterpret_cast<const void* const*>(dA), n, true));
  TP_TRY(check_ptr_array(dt, "da", reinterpret_cast<const void* const*>(da), n, false));
  TP_TRY(check_ptr_array(dt, "dB", reinterpret_cast<const void* const*>(dB), n, true));
  TP_TRY(check_ptr(dt, "db", db, false));
  TP_TRY(check_ws(ws, ws_bytes, z.total));
  TP_TRY(check_arch());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t e = elem_size(dt);

  // dH_i = (dZ B_i^T) * act'(H_i), kept in the workspace in the input dtype.
  const size_t dh_off = scratch_base(dt);
  const void* dHp[kMaxShards] = {};
  const void* dZs[kMaxShards] = {};
  const void* Xs[kMaxShards] = {};
  for (int i = 0; i < n; ++i) {
    dZs[i] = dZ;
    Xs[i] = X;
  }
  bool dB_done = false;
  if (z.T > 0) {
    GemmSpec s;
    s.M = z.T;
    s.N = z.Fs;
    s.K = z.H;
    s.groups = n;
    s.a_mn = 0;
    s.b_mn = 0;
    s.lda = z.H;
    s.ldb = z.H;
    s.ldd = z.Fs;
    s.ldaux = z.Fs;
    s.epi = EPI_DACT;
    s.act = desc->act;
    bind_ws(s, ws, dt);
    for (int i = 0; i < n; ++i) {
      s.A[i] = dZ;
      s.B[i] = B[i];
      s.D[i] = ws_at<char>(ws, dh_off + size_t(i) * z.T * z.Fs * e);
      s.aux[i] = Hsave ? Hsave[i] : nullptr;
      dHp[i] = s.D[i];
    }
    // dB_i = Y_i^T dZ needs only the forward's values: where the two fit one launch, its tiles
    // and dH_i's share the pairs
    const GemmSpec sb = wgrad_spec(dt, n, z.T, z.Fs, z.H, Ysave, z.Fs, dZs, z.H, dB, ws);
    if (dt == TP_BF16 && tc_dual_eligible(sb, s)) {
      TP_CUDA(run_gemm_dual(sb, s, dt, st, TP_TAG_ROW_GRADS), "dB and dY GEMMs");
      dB_done = true;
    } else {
      TP_CUDA(run_gemm(s, dt, st, TP_TAG_ROW_DGRAD), "dY GEMM");
    }
  } else {
    for (int i = 0; i < n; ++i) dHp[i] = ws_at<char>(ws, dh_off);
  }

  // dB_i = Y_i^T dZ.
  if (!dB_done)
    TP_TRY(weight_grads(dt, n, z.T, z.Fs, z.H, Ysave, z.Fs, dZs, z.H, dB, ws, st, TP_TAG_ROW_WGRAD));
  // dA_i = X^T dH_i and dX = sum_i dH_i A_i^T: both need only dH_i; one launch where they fit
  // it and the shard sum stays inside the dX GEMM's accumulator.
  bool column_done = false;
  if (z.T > 0 && dt == TP_BF16 && shard_split(desc->reduce, dt, z.T, z.H, z.Fs, n) == 1) {
    const GemmSpec sa = wgrad_spec(dt, n, z.T, z.H, z.Fs, Xs, z.H, dHp, z.Fs, dA, ws);
    GemmSpec sx = dgrad_spec(dt, n, z.T, z.Fs, z.H, dHp, z.Fs, A, ws);
    sx.ksum = 1;
    sx.D[0] = dX;
    if (tc_dual_eligible(sa, sx)) {
      TP_CUDA(run_gemm_dual(sa, sx, dt, st, TP_TAG_COLUMN_GRADS), "dA and dX GEMMs");
      column_done = true;
    }
  }
  if (!column_done) {
    TP_TRY(weight_grads(dt, n, z.T, z.H, z.Fs, Xs, z.H, dHp, z.Fs, dA, ws, st, TP_TAG_COLUMN_WGRAD));
    if (z.T > 0)
      TP_TRY(input_grad_sum(dt, desc->reduce, n, z.T, z.Fs, z.H, dHp, z.Fs, A,
                            static_cast<float*>(dX), ws, dh_off + z.dH, st));
  }
  // db = sum_t dZ, da_i = sum_t dH_i.
  ColsumSeg segs[kMaxShards + 1];
  int nseg = 0;
  if (db != nullptr) segs[nseg++] = ColsumSeg{dZ, static_cast<float*>(db), z.H, z.H};
  if (da != nullptr)
    for (int i = 0; i < n; ++i) segs[nseg++] = ColsumSeg{dHp[i], static_cast<float*>(da[i]), z.Fs, z.Fs};
  TP_TRY(colsums(dt, z.T, segs, nseg, st));
  return ok();
}

}  // extern "C"

// ------------------------------------------------------------------ sequence-parallel MLP
namespace {

struct SpLayout {
  size_t base, xg, zf, dzg, dxf, total;
};

tp_status sp_layout(const tp_mlp_desc* d, SpLayout* L, MlpSizes* z) {
  TP_TRY(mlp_validate(d, z));
  if (z->T % z->n != 0)
    return fail(TP_ERR_INDIVISIBLE, "tokens %lld are not divisible by tp_degree %d",
                static_cast<long long>(z->T), z->n);
  const size_t e = elem_size(d->dtype);
  const size_t th = size_t(z->T) * size_t(z->H);
  L->base = align256(z->total);
  L->xg = L->base;
  L->zf = L->xg + align256(th * e);
  L->dzg = L->zf + align256(th * 4);
  L->dxf = L->dzg + align256(th * e);
  L->total = L->dxf + align256(th * 4);
  return TP_OK;
}

cudaError_t copy_traced(void* const* shards, void* full, int n, size_t bytes, int gather,
                        cudaStream_t st) {
  return traced(TP_K_SHARD_COPY, gather ? TP_TAG_SP_GATHER : TP_TAG_SP_SCATTER, n, 0.0,
                2.0 * double(bytes) * n, st,
                [&] { return launch_shard_copy(shards, full, n, bytes, gather, st); });
}

}  // namespace

extern "C" {

tp_status tp_mlp_sp_workspace_size(const tp_mlp_desc* desc, size_t* bytes) {
  if (bytes == nullptr) return fail(TP_ERR_NULL, "bytes is NULL");
  SpLayout L{};
  MlpSizes z{};
  TP_TRY(sp_layout(desc, &L, &z));
  *bytes = L.total;
  return ok();
}

tp_status tp_mlp_forward_sp(const tp_mlp_desc* desc, const void* const* X_shards,
                            const void* const* A, const void* const* a, const void* const* B,
                            const void* b, void* const* Z_shards, void* const* Hsave,
                            void* const* Ysave, void* ws, size_t ws_bytes, void* stream) {
  SpLayout L{};
  MlpSizes z{};
  TP_TRY(sp_layout(desc, &L, &z));
  const int dt = desc->dtype;
  TP_TRY(check_ptr_array(dt, "X_shards", X_shards, z.n, z.T > 0, z.T > 0));
  TP_TRY(check_ptr_array(dt, "Z_shards", reinterpret_cast<const void* const*>(Z_shards), z.n,
                         z.T > 0, z.T > 0));
  TP_TRY(check_ws(ws, ws_bytes, L.total));
  TP_TRY(check_arch());
  if (z.T == 0) return ok();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t e = elem_size(dt);
  const size_t rows = size_t(z.T / z.n);
  void* xg = ws_at<char>(ws, L.xg);
  void* zf = ws_at<char>(ws, L.zf);
  TP_CUDA(copy_traced(const_cast<void* const*>(X_shards), xg, z.n, rows * z.H * e, 1, st),
          "all-gather of the token shards");
  TP_TRY(tp_mlp_forward(desc, xg, A, a, B, b, zf, Hsave, Ysave, ws, L.base, stream));
  TP_CUDA(copy_traced(Z_shards, zf, z.n, rows * z.H * 4, 0, st), "scatter of Z");
  return ok();
}

tp_status tp_mlp_backward_sp(const tp_mlp_desc* desc, const void* const* X_shards,
                             const void* const* A, const void* const* B,
                             const void* const* Hsave, const void* const* Ysave,
                             const void* const* dZ_shards, void* const* dX_shards,
                             void* const* dA, void* const* da, void* const* dB, void* db,
                             void* ws, size_t ws_bytes, void* stream) {
  SpLayout L{};
  MlpSizes z{};
  TP_TRY(sp_layout(desc, &L, &z));
  const int dt = desc->dtype;
  TP_TRY(check_ptr_array(dt, "X_shards", X_shards, z.n, z.T > 0, z.T > 0));
  TP_TRY(check_ptr_array(dt, "dZ_shards", dZ_shards, z.n, z.T > 0, z.T > 0));
  TP_TRY(check_ptr_array(dt, "dX_shards", reinterpret_cast<const void* const*>(dX_shards), z.n,
                         z.T > 0, z.T > 0));
  TP_TRY(check_ws(ws, ws_bytes, L.total));
  TP_TRY(check_arch());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t e = elem_size(dt);
  const size_t rows = size_t(z.T / z.n);
  void* xg = ws_at<char>(ws, L.xg);
  void* dzg = ws_at<char>(ws, L.dzg);
  void* dxf = ws_at<char>(ws, L.dxf);
  if (z.T > 0) {
    TP_CUDA(copy_traced(const_cast<void* const*>(X_shards), xg, z.n, rows * z.H * e, 1, st),
            "all-gather of the token shards");
    TP_CUDA(copy_traced(const_cast<void* const*>(dZ_shards), dzg, z.n, rows * z.H * e, 1, st),
            "all-gather of dZ");
  }
  TP_TRY(tp_mlp_backward(desc, xg, A, B, Hsave, Ysave, dzg, dxf, dA, da, dB, db, ws, L.base,
                         stream));
  if (z.T > 0)
    TP_CUDA(copy_traced(dX_shards, dxf, z.n, rows * z.H * 4, 0, st), "scatter of dX");
  return ok();
}

// ------------------------------------------------------------------ column-parallel linear
tp_status tp_linear_column_forward(const tp_linear_desc* desc, const void* X,
                                   const void* const* W, const void* const* bias,
                                   void* const* Y, void* const* Hsave, void* ws,
                                   size_t ws_bytes, void* stream) {
  LinSizes z{};
  TP_TRY(lin_validate(desc, TP_COLUMN, &z));
  const int dt = desc->dtype;
  const int n = z.n;
  const int ny = desc->gather ? 1 : n;
  TP_TRY(check_ptr(dt, "X", X, z.T > 0));
  TP_TRY(check_ptr_array(dt, "W", W, n, true));
  TP_TRY(check_ptr_array(dt, "bias", bias, n, false));
  TP_TRY(check_ptr_array(dt, "Y", reinterpret_cast<const void* const*>(Y), ny, z.T > 0, z.T > 0));
  TP_TRY(check_ptr_array(dt, "Hsave", reinterpret_cast<const void* const*>(Hsave), n,
                         z.T > 0 && desc->act != TP_ACT_NONE, z.T > 0));
  TP_TRY(check_ws(ws, ws_bytes, z.total));
  TP_TRY(check_arch());
  if (z.T == 0) return ok();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t e = elem_size(dt);
  GemmSpec c;
  c.M = z.T;
  c.N = z.Ns;
  c.K = z.K;
  c.groups = n;
  c.a_mn = 0;
  c.b_mn = 1;
  c.lda = z.K;
  c.ldb = z.Ns;
  c.ldd = z.Ns;
  c.ldd2 = desc->gather ? z.N : z.Ns;
  c.epi = EPI_BIAS_ACT;
  c.act = desc->act;
  bind_ws(c, ws, dt);
  for (int i = 0; i < n; ++i) {
    c.A[i] = X;
    c.B[i] = W[i];
    c.bias[i] = bias ? bias[i] : nullptr;
    c.D[i] = Hsave ? Hsave[i] : nullptr;
    c.D2[i] = desc->gather ? static_cast<char*>(Y[0]) + size_t(i) * z.Ns * e : Y[i];
  }
  TP_CUDA(run_gemm(c, dt, st, TP_TAG_COLUMN_FWD), "column GEMM");
  return ok();
}

tp_status tp_linear_column_backward(const tp_linear_desc* desc, const void* X,
                                    const void* const* W, const void* const* Hsave,
                                    const void* const* dY, void* dX, void* const* dW,
                                    void* const* dbias, void* ws, size_t ws_bytes, void* stream) {
  LinSizes z{};
  TP_TRY(lin_validate(desc, TP_COLUMN, &z));
  const int dt = desc->dtype;
  const int n = z.n;
  const int ny = desc->gather ? 1 : n;
  TP_TRY(check_ptr(dt, "X", X, z.T > 0));
  TP_TRY(check_ptr_array(dt, "W", W, n, true));
  TP_TRY(check_ptr_array(dt, "Hsave", Hsave, n, z.T > 0 && desc->act != TP_ACT_NONE, z.T > 0));
  TP_TRY(check_ptr_array(dt, "dY", dY, ny, z.T > 0, z.T > 0));
  TP_TRY(check_ptr(dt, "dX", dX, z.T > 0));
  TP_TRY(check_ptr_array(dt, "dW", reinterpret_cast<const void* const*>(dW), n, true));
  TP_TRY(check_ptr_array(dt, "dbias", reinterpret_cast<const void* const*>(dbias), n, false));
  TP_TRY(check_ws(ws, ws_bytes, z.total));
  TP_TRY(check_arch());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t e = elem_size(dt);

  // The shard views of dY (gathered: column blocks of one [T, N] buffer).
  const void* dYv[kMaxShards] = {};
  for (int i = 0; i < n && dY != nullptr; ++i)
    dYv[i] = desc->gather ? static_cast<const char*>(dY[0]) + size_t(i) * z.Ns * e : dY[i];
  const int64_t ld_dy = desc->gather ? z.N : z.Ns;

  const void* dHp[kMaxShards] = {};
  int64_t ldh = ld_dy;
  const size_t dh_off = scratch_base(dt);
  if (desc->act != TP_ACT_NONE) {
    void* dHw[kMaxShards] = {};
    for (int i = 0; i < n; ++i) {
      dHw[i] = ws_at<char>(ws, dh_off + size_t(i) * z.T * z.Ns * e);
      dHp[i] = dHw[i];
    }
    if (z.T > 0)
      TP_CUDA(traced(TP_K_DACT, TP_TAG_ACT_GRAD, n, 0.0, 3.0 * double(z.T) * z.N * e, st,
                     [&] {
                       return launch_dact(dYv, ld_dy, Hsave, dHw, n, z.T, z.Ns, desc->act,
                                          dt == TP_BF16, st);
                     }),
              "activation gradient");
    ldh = z.Ns;
  } else {
    for (int i = 0; i < n; ++i) dHp[i] = dYv[i];
  }
  const void* Xs[kMaxShards] = {};
  for (int i = 0; i < n; ++i) Xs[i] = X;
  // dW_i = X^T dH_i and dX = sum_i dH_i W_i^T: one launch where they fit it and the shard sum
  // stays inside the dX GEMM's accumulator (tc_dual_eligible)
  bool shared = false;
  if (z.T > 0 && dt == TP_BF16 && shard_split(desc->reduce, dt, z.T, z.K, z.Ns, n) == 1) {
    const GemmSpec sw = wgrad_spec(dt, n, z.T, z.K, z.Ns, Xs, z.K, dHp, ldh, dW, ws);
    GemmSpec sx = dgrad_spec(dt, n, z.T, z.Ns, z.K, dHp, ldh, W, ws);
    sx.ksum = 1;
    sx.D[0] = dX;
    if (tc_dual_eligible(sw, sx)) {
      TP_CUDA(run_gemm_dual(sw, sx, dt, st, TP_TAG_COLUMN_GRADS), "dW and dX GEMMs");
      shared = true;
    }
  }
  if (!shared) {
    TP_TRY(weight_grads(dt, n, z.T, z.K, z.Ns, Xs, z.K, dHp, ldh, dW, ws, st, TP_TAG_COLUMN_WGRAD));
    if (z.T > 0)
      TP_TRY(input_grad_sum(dt, desc->reduce, n, z.T, z.Ns, z.K, dHp, ldh, W,
                            static_cast<float*>(dX), ws, dh_off + z.dH, st));
  }
  if (dbias != nullptr) {
    ColsumSeg segs[kMaxShards];
    for (int i = 0; i < n; ++i) segs[i] = ColsumSeg{dHp[i], static_cast<float*>(dbias[i]), z.Ns, ldh};
    TP_TRY(colsums(dt, z.T, segs, n, st));
  }
  return ok();
}

// ------------------------------------------------------------------ row-parallel linear
tp_status tp_linear_row_forward(const tp_linear_desc* desc, const void* const* X,
                                const void* const* W, const void* bias, void* Z, void* ws,
                                size_t ws_bytes, void* stream) {
  LinSizes z{};
  TP_TRY(lin_validate(desc, TP_ROW, &z));
  const int dt = desc->dtype;
  const int n = z.n;
  TP_TRY(check_ptr_array(dt, "X", X, n, z.T > 0, z.T > 0));
  TP_TRY(check_ptr_array(dt, "W", W, n, true));
  TP_TRY(check_ptr(dt, "bias", bias, false));
  TP_TRY(check_ptr(dt, "Z", Z, z.T > 0));
  TP_TRY(check_ws(ws, ws_bytes, z.total));
  TP_TRY(check_arch());
  if (z.T == 0) return ok();
  TP_TRY(row_product(dt, desc->reduce, n, z.T, z.Ks, z.N, X, z.Ks, W, bias,
                     static_cast<float*>(Z), ws, scratch_base(dt), static_cast<cudaStream_t>(stream),
                     "row GEMM"));
  return ok();
}

tp_status tp_linear_row_backward(const tp_linear_desc* desc, const void* const* X,
                                 const void* const* W, const void* dZ, void* const* dX,
                                 void* const* dW, void* dbias, void* ws, size_t ws_bytes,
                                 void* stream) {
  LinSizes z{};
  TP_TRY(lin_validate(desc, TP_ROW, &z));
  const int dt = desc->dtype;
  const int n = z.n;
  TP_TRY(check_ptr_array(dt, "X", X, n, z.T > 0, z.T > 0));
  TP_TRY(check_ptr_array(dt, "W", W, n, true));
  TP_TRY(check_ptr(dt, "dZ", dZ, z.T > 0));
  TP_TRY(check_ptr_array(dt, "dX", reinterpret_cast<const void* const*>(dX), n, z.T > 0, z.T > 0));
  TP_TRY(check_ptr_array(dt, "dW", reinterpret_cast<const void* const*>(dW), n, true));
  TP_TRY(check_ptr(dt, "dbias", dbias, false));
  TP_TRY(check_ws(ws, ws_bytes, z.total));
  TP_TRY(check_arch());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (z.T > 0) {
    // dX_i = dZ W_i^T: W_i [Ks, N] read as the K-major [N-rows = Ks][K = N] operand.
    GemmSpec s;
    s.M = z.T;
    s.N = z.Ks;
    s.K = z.N;
    s.groups = n;
    s.a_mn = 0;
    s.b_mn = 0;
    s.lda = z.N;
    s.ldb = z.N;
    s.ldd = z.Ks;
    s.epi = EPI_STORE_F32;
    bind_ws(s, ws, dt);
    for (int i = 0; i < n; ++i) {
      s.A[i] = dZ;
      s.B[i] = W[i];
      s.D[i] = dX[i];
    }
    // dW_i = X_i^T dZ needs only the inputs: one launch with dX_i where they fit it
    const void* dZs[kMaxShards] = {};
    for (int i = 0; i < n; ++i) dZs[i] = dZ;
    const GemmSpec sw = wgrad_spec(dt, n, z.T, z.Ks, z.N, X, z.Ks, dZs, z.N, dW, ws);
    if (dt == TP_BF16 && tc_dual_eligible(sw, s)) {
      TP_CUDA(run_gemm_dual(sw, s, dt, st, TP_TAG_ROW_GRADS), "dW and dX GEMMs");
      if (dbias != nullptr) {
        ColsumSeg seg{dZ, static_cast<float*>(dbias), z.N, z.N};
        TP_TRY(colsums(dt, z.T, &seg, 1, st));
      }
      return ok();
    }
    TP_CUDA(run_gemm(s, dt, st, TP_TAG_ROW_DGRAD), "row input-gradient GEMM");
  }
  const void* dZs[kMaxShards] = {};
  for (int i = 0; i < n; ++i) dZs[i] = dZ;
  TP_TRY(weight_grads(dt, n, z.T, z.Ks, z.N, X, z.Ks, dZs, z.N, dW, ws, st, TP_TAG_ROW_WGRAD));
  if (dbias != nullptr) {
    ColsumSeg seg{dZ, static_cast<float*>(dbias), z.N, z.N};
    TP_TRY(colsums(dt, z.T, &seg, 1, st));
  }
  return ok();
}

// ------------------------------------------------------------------ hidden-split LayerNorm
}  // extern "C"

namespace {

tp_status ln_validate(const tp_layernorm_desc* d, int64_t* Hs) {
  if (d == nullptr) return fail(TP_ERR_NULL, "desc is NULL");
  TP_TRY(check_common(d->tokens, d->tp_degree, d->dtype, TP_ACT_NONE, TP_REDUCE_FUSED));
  TP_TRY(check_dim("hidden", d->hidden));
  if (d->hidden % d->tp_degree != 0)
    return fail(TP_ERR_INDIVISIBLE, "hidden %lld is not divisible by tp_degree %d",
                static_cast<long long>(d->hidden), d->tp_degree);
  if (!(d->eps > 0.0f) || !std::isfinite(d->eps)) return fail(TP_ERR_SHAPE, "eps must be > 0");
  *Hs = d->hidden / d->tp_degree;
  TP_TRY(check_width(d->dtype, "hidden / tp_degree", *Hs));
  return TP_OK;
}

tp_status check_f32_ptr(const char* name, const void* p, bool required) {
  return check_ptr(TP_F32, name, p, required);
}

}  // namespace

extern "C" {

tp_status tp_layernorm_forward(const tp_layernorm_desc* desc, const void* const* X,
                               const void* const* gamma, const void* const* beta, void* const* Y,
                               float* mean, float* rstd, void* stream) {
  int64_t Hs = 0;
  TP_TRY(ln_validate(desc, &Hs));
  const int dt = desc->dtype, n = desc->tp_degree;
  const int64_t T = desc->tokens;
  TP_TRY(check_ptr_array(dt, "X", X, n, T > 0, T > 0));
  TP_TRY(check_ptr_array(dt, "gamma", gamma, n, false));
  TP_TRY(check_ptr_array(dt, "beta", beta, n, false));
  TP_TRY(check_ptr_array(dt, "Y", reinterpret_cast<const void* const*>(Y), n, T > 0, T > 0));
  TP_TRY(check_f32_ptr("mean", mean, false));
  TP_TRY(check_f32_ptr("rstd", rstd, false));
  TP_TRY(check_arch());
  if (T == 0) return ok();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  LnArgs a;
  a.X = X;
  a.gamma = gamma;
  a.beta = beta;
  a.Y = Y;
  a.mean = mean;
  a.rstd = rstd;
  a.T = T;
  a.Hs = Hs;
  a.n = n;
  a.eps = desc->eps;
  a.bf16 = dt == TP_BF16;
  const double e = elem_size(dt), H = double(Hs) * n;
  const double bytes = double(T) * H * 2.0 * e + ((gamma ? 1 : 0) + (beta ? 1 : 0)) * H * e +
                       (mean ? 4.0 * T : 0.0) + (rstd ? 4.0 * T : 0.0);
  TP_CUDA(traced(TP_K_LAYERNORM, TP_TAG_LN_FWD, n, 0.0, bytes, st,
                 [&] { return launch_ln_forward(a, st); }),
          "LayerNorm forward");
  return ok();
}

tp_status tp_layernorm_backward(const tp_layernorm_desc* desc, const void* const* X,
                                const void* const* gamma, const float* mean, const float* rstd,
                                const void* const* dY, void* const* dX, float* const* dgamma,
                                float* const* dbeta, void* stream) {
  int64_t Hs = 0;
  TP_TRY(ln_validate(desc, &Hs));
  const int dt = desc->dtype, n = desc->tp_degree;
  const int64_t T = desc->tokens;
  TP_TRY(check_ptr_array(dt, "X", X, n, T > 0, T > 0));
  TP_TRY(check_ptr_array(dt, "gamma", gamma, n, false));
  TP_TRY(check_ptr_array(dt, "dY", dY, n, T > 0, T > 0));
  TP_TRY(check_ptr_array(dt, "dX", reinterpret_cast<const void* const*>(dX), n, T > 0, T > 0));
  TP_TRY(check_ptr_array(TP_F32, "dgamma", reinterpret_cast<const void* const*>(dgamma), n, false));
  TP_TRY(check_ptr_array(TP_F32, "dbeta", reinterpret_cast<const void* const*>(dbeta), n, false));
  TP_TRY(check_f32_ptr("mean", mean, T > 0));
  TP_TRY(check_f32_ptr("rstd", rstd, T > 0));
  TP_TRY(check_arch());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  LnArgs a;
  a.X = X;
  a.gamma = gamma;
  a.Y = dX;
  a.dY = dY;
  a.dgamma = dgamma;
  a.dbeta = dbeta;
  a.mean = const_cast<float*>(mean);
  a.rstd = const_cast<float*>(rstd);
  a.T = T;
  a.Hs = Hs;
  a.n = n;
  a.eps = desc->eps;
  a.bf16 = dt == TP_BF16;
  const double e = elem_size(dt), H = double(Hs) * n;
  if (T > 0)
    TP_CUDA(traced(TP_K_LAYERNORM, TP_TAG_LN_DGRAD, n, 0.0,
                   double(T) * H * 3.0 * e + (gamma ? H * e : 0.0) + 8.0 * T, st,
                   [&] { return launch_ln_backward_dx(a, st); }),
            "LayerNorm input gradient");
  if (dgamma != nullptr || dbeta != nullptr)
    TP_CUDA(traced(TP_K_LN_PARAM_GRAD, TP_TAG_LN_PARAM_GRAD, n, 0.0,
                   double(T) * H * 2.0 * e + 8.0 * T + 8.0 * H, st,
                   [&] { return launch_ln_param_grads(a, st); }),
            "LayerNorm parameter gradients");
  return ok();
}

}  // extern "C"
