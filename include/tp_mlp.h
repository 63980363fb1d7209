/*
 * tp_mlp.h -- C ABI of the GB300 (sm_103a) tensor-parallel MLP library (libtpmlp.so).
 *
 * The operations are those of Megatron-style tensor parallelism as the pages describe it:
 *
 *  - "What tensor parallelism is: core principles of large-model training", section
 *    "Core working mechanism": X is replicated, the first weight A is split by columns
 *    (Y_i = X A_i), the next linear's weight is split by rows so that Y_i is its shard
 *    input, and the partial products are summed by an All-Reduce.
 *  - "Tensor Parallelism: principle and practice", section 3.1 (Megatron-LM): column
 *    parallel forward X W_i with weight gradient X^T dL/dY_i; row parallel forward X_i W
 *    summed by All-Reduce, input gradient (dL/dY) W^T; section 2.1: XW = sum_i X_i W_i.
 *  - "Tensor parallelism in practice: from theory to complete PyTorch code", section
 *    "PyTorch implementation example": per-shard weight [in, out/world_size] and bias
 *    [out/world_size], forward X W_i + b_i, shard outputs gathered and concatenated along
 *    the last dimension; out_features must divide by world_size.
 *  - "PaddlePaddle tensor parallelism: from principle to industrial deployment": the
 *    input gradient of a column-split layer is summed over the devices.
 *
 * All tp_degree shards live on ONE GPU as separate device buffers. The All-Reduce of the
 * pages is an on-device reduction: either accumulated over the shards inside one tensor-core
 * accumulator (TP_REDUCE_FUSED), or written as per-shard fp32 partials and summed by a
 * reduction kernel (TP_REDUCE_PARTIALS). No collective and no second GPU are involved.
 *
 * Conventions (every entry point):
 *  - Matrices are row-major and dense (leading dimension = number of columns).
 *  - Device pointers are owned by the caller; the library never allocates or frees device
 *    memory. Pointer arrays ("const void* const* W") are HOST arrays of tp_degree DEVICE
 *    pointers, read during the call only.
 *  - "stream" is a cudaStream_t (NULL = the legacy default stream). Every call only
 *    enqueues work on it and returns; nothing is synchronised except in tp_check_status.
 *  - Arguments are validated on the host before any launch; on an error nothing is
 *    enqueued and tp_last_error() returns a message (thread-local).
 *  - TP_BF16: inputs (activations, weights, biases, upstream gradients) are bf16; the
 *    tensor cores multiply bf16 and accumulate in fp32. Saved activations (Hsave, Ysave)
 *    and column outputs are bf16. Summed outputs (Z, dX) and all parameter gradients
 *    (dW, dbias) are fp32. Pointers must be 16-byte aligned and hidden / in / out / shard
 *    widths multiples of 8.
 *    TP_F32: everything is fp32 and computed with fp32 FMA (no TF32); pointers 4-byte
 *    aligned, no other size rule.
 *  - The workspace (see the *_workspace_size calls) holds a device status word followed by
 *    scratch; call tp_workspace_init once after allocating it. A device-side wait that
 *    runs out writes an error code into the status word; tp_check_status reports it.
 *    TP_BF16 calls reserve TP_BF16_TAIL_SCRATCH_BYTES of the workspace right after the
 *    status block: when a GEMM's tiles leave its last wave of SM pairs partly idle, each tile
 *    of that wave is computed as K pieces on otherwise idle pairs, and the pieces are added
 *    in piece order (deterministic) before the epilogue.
 *  - Requires an sm_103 device (GB300); on any other device calls return TP_ERR_ARCH.
 */
#ifndef TP_MLP_H
#define TP_MLP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum tp_dtype { TP_F32 = 0, TP_BF16 = 1 } tp_dtype;

/* Activation of the column-parallel linear. The pages name none; GeLU is the exact erf
 * form h * (1 + erf(h / sqrt 2)) / 2. */
typedef enum tp_act { TP_ACT_NONE = 0, TP_ACT_GELU_ERF = 1 } tp_act;

/* How the shard sum (the pages' All-Reduce) is done on the device.
 *  FUSED:    one accumulator sums every shard's K range (no scratch).
 *  PARTIALS: one fp32 partial per shard, then a reduction kernel.
 *  AUTO:     the shards are summed in S groups (S a divisor of tp_degree chosen from the
 *            shape and the SM count to balance tile waves against reduction traffic; S = 1 is
 *            FUSED), then a reduction of the S partials. bf16 only; fp32 uses FUSED.
 *            Workspace is sized as for PARTIALS.
 *  PARTIALS_BF16: one bf16 partial per shard (half the bytes of PARTIALS), summed in fp32 by
 *            the reduction kernel -- the reduced-precision "communication" of "Tensor
 *            Parallelism: principle and practice", section 5.2. bf16 only.
 *  OVERLAP:  as AUTO, but with S > 1 the partials are summed inside the GEMM launch, while
 *            other tiles still compute: the epilogue warp that writes the last partial of a
 *            (32-row, 256-column) block adds the S partials in order, plus the bias, into the
 *            output (the single-GPU counterpart of overlapping the All-Reduce with compute,
 *            "Tensor Parallelism: principle and practice", section 5.2). bf16 only; the
 *            workspace adds one counter per block. */
typedef enum tp_reduce {
  TP_REDUCE_FUSED = 0,
  TP_REDUCE_PARTIALS = 1,
  TP_REDUCE_AUTO = 2,
  TP_REDUCE_PARTIALS_BF16 = 3,
  TP_REDUCE_OVERLAP = 4
} tp_reduce;

typedef enum tp_status {
  TP_OK = 0,
  TP_ERR_NULL = 1,            /* a required pointer is NULL */
  TP_ERR_SHAPE = 2,           /* a size is < 1, too large, or tp_degree is outside 1..64 */
  TP_ERR_INDIVISIBLE = 3,     /* the split dimension does not divide by tp_degree */
  TP_ERR_ALIGN = 4,           /* pointer or size alignment rule broken (see above) */
  TP_ERR_DTYPE = 5,           /* unknown dtype, activation, reduce mode or flag */
  TP_ERR_WORKSPACE = 6,       /* workspace missing or smaller than *_workspace_size */
  TP_ERR_ARCH = 7,            /* no CUDA device, or the device is not sm_103 */
  TP_ERR_CUDA = 8,            /* a CUDA runtime / driver call or a launch failed */
  TP_ERR_DEVICE_TIMEOUT = 9   /* a kernel's bounded wait ran out (from tp_check_status) */
} tp_status;

/* The MLP: X [T,H]; A [H,F] split by columns into A_i [H,F/n] with bias a_i [F/n];
 * B [F,H] split by rows into B_i [F/n,H]; bias b [H] added once after the shard sum.
 *   H_i = X A_i + a_i;  Y_i = act(H_i);  Z = sum_i Y_i B_i + b. */
typedef struct tp_mlp_desc {
  int64_t tokens;     /* T */
  int64_t hidden;     /* H */
  int64_t ffn;        /* F; must divide by tp_degree */
  int32_t tp_degree;  /* n, 1..64 */
  int32_t dtype;      /* tp_dtype */
  int32_t act;        /* tp_act */
  int32_t reduce;     /* tp_reduce */
} tp_mlp_desc;

/* One parallel linear: X [T,K] times W [K,N].
 *  column: W split by columns into W_i [K,N/n], bias_i [N/n]; Y_i = act(X W_i + bias_i).
 *  row:    W split by rows into W_i [K/n,N]; input shards X_i [T,K/n];
 *          Z = sum_i X_i W_i + bias (bias [N], once). */
typedef struct tp_linear_desc {
  int64_t tokens;        /* T */
  int64_t in_features;   /* K */
  int64_t out_features;  /* N */
  int32_t tp_degree;     /* n, 1..64; column: N % n == 0; row: K % n == 0 */
  int32_t dtype;         /* tp_dtype */
  int32_t act;           /* tp_act (column only; row must be TP_ACT_NONE) */
  int32_t reduce;        /* tp_reduce (row forward; column backward's dX sum) */
  int32_t gather;        /* column only: 1 = the shard outputs (and dY in the backward)
                            are the column blocks of ONE [T,N] buffer, passed as Y[0]
                            (the gather + concatenation of the pages' example) */
} tp_linear_desc;

typedef enum tp_linear_kind { TP_COLUMN = 0, TP_ROW = 1 } tp_linear_kind;

/* Workspace bytes that every TP_BF16 call reserves after the 256-byte status block: up to 80
 * fp32 accumulator pieces of 256 x 256 for the GEMM's split last wave, and their counters. */
#define TP_BF16_TAIL_SCRATCH_BYTES ((size_t)80 * 256 * 256 * 4 + 4096)

/* Version of this ABI (major * 100 + minor). */
int32_t tp_version(void);

/* Message of the last error on this thread ("" if none). Never NULL. */
const char* tp_last_error(void);

/* Bytes of workspace that tp_mlp_forward and tp_mlp_backward need for *desc (the larger of
 * the two): a 256-byte status block, TP_BF16_TAIL_SCRATCH_BYTES for TP_BF16, plus n fp32
 * partials [T,H] in TP_REDUCE_PARTIALS mode, or the backward's per-shard gradients
 * dH_i [T,F/n] at the pre-activation. */
tp_status tp_mlp_workspace_size(const tp_mlp_desc* desc, size_t* bytes);

/* Bytes of workspace that the forward and backward of one column or row linear need. */
tp_status tp_linear_workspace_size(const tp_linear_desc* desc, int32_t kind, size_t* bytes);

/* Zero the workspace's status word (enqueued on stream). Call once after allocation. */
tp_status tp_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Synchronise stream and return TP_ERR_DEVICE_TIMEOUT if a kernel that used this
 * workspace reported a wait that ran out (the code stays in the status word until
 * tp_workspace_init clears it), TP_ERR_CUDA if the stream reports an error, else TP_OK. */
tp_status tp_check_status(void* ws, size_t ws_bytes, void* stream);

/* MLP forward. X [T,H]; A[i] [H,F/n]; a[i] [F/n] (a may be NULL: no column bias);
 * B[i] [F/n,H]; b [H] (may be NULL). Writes Z [T,H] (fp32 for TP_BF16, else fp32),
 * Hsave[i] = H_i and Ysave[i] = Y_i, each [T,F/n] in the input dtype (both required:
 * they are the backward's inputs; with TP_ACT_NONE, Hsave may be NULL). */
tp_status tp_mlp_forward(const tp_mlp_desc* desc, const void* X, const void* const* A,
                         const void* const* a, const void* const* B, const void* b,
                         void* Z, void* const* Hsave, void* const* Ysave,
                         void* ws, size_t ws_bytes, void* stream);

/* MLP backward for upstream gradient dZ [T,H] (input dtype). Writes
 *   dB_i = Y_i^T dZ [F/n,H]; db = sum_t dZ [H]; dH_i = (dZ B_i^T) * act'(H_i);
 *   dA_i = X^T dH_i [H,F/n]; da_i = sum_t dH_i [F/n]; dX = sum_i dH_i A_i^T [T,H].
 * All outputs fp32. da and db may be NULL (not computed). dH_i lives in the workspace. */
tp_status tp_mlp_backward(const tp_mlp_desc* desc, const void* X, const void* const* A,
                          const void* const* B, const void* const* Hsave,
                          const void* const* Ysave, const void* dZ, void* dX,
                          void* const* dA, void* const* da, void* const* dB, void* db,
                          void* ws, size_t ws_bytes, void* stream);

/* Sequence-parallel MLP ("What tensor parallelism is", section on sequence parallelism; the
 * ReduceScatter of "PaddlePaddle tensor parallelism"). The tokens are split across the shards:
 * X_shards[j] and Z_shards[j] (backward: dZ_shards[j], dX_shards[j]) hold rows
 * j*T/n .. (j+1)*T/n - 1, each [T/n, H]; T must divide by tp_degree (else
 * TP_ERR_INDIVISIBLE). The token shards are all-gathered on the device, the MLP runs as in
 * tp_mlp_forward / tp_mlp_backward, and the shard sum Z (dX) is scattered back by token rows
 * (a reduce-scatter: each token shard receives the full sum for its rows). Hsave, Ysave, the
 * weight and bias gradients are as in the non-sequence-parallel calls. The workspace
 * (tp_mlp_sp_workspace_size) adds gathered copies of X and dZ and the full Z / dX. */
tp_status tp_mlp_sp_workspace_size(const tp_mlp_desc* desc, size_t* bytes);
tp_status tp_mlp_forward_sp(const tp_mlp_desc* desc, const void* const* X_shards,
                            const void* const* A, const void* const* a, const void* const* B,
                            const void* b, void* const* Z_shards, void* const* Hsave,
                            void* const* Ysave, void* ws, size_t ws_bytes, void* stream);
tp_status tp_mlp_backward_sp(const tp_mlp_desc* desc, const void* const* X_shards,
                             const void* const* A, const void* const* B,
                             const void* const* Hsave, const void* const* Ysave,
                             const void* const* dZ_shards, void* const* dX_shards,
                             void* const* dA, void* const* da, void* const* dB, void* db,
                             void* ws, size_t ws_bytes, void* stream);

/* Column-parallel linear forward: Y_i = act(X W_i + bias_i). X [T,K]; W[i] [K,N/n];
 * bias[i] [N/n] or bias NULL; Y[i] [T,N/n] in the input dtype (gather=1: Y[0] is [T,N]).
 * Hsave[i] [T,N/n] receives X W_i + bias_i when act != NONE (required then), else may be
 * NULL. */
tp_status tp_linear_column_forward(const tp_linear_desc* desc, const void* X,
                                   const void* const* W, const void* const* bias,
                                   void* const* Y, void* const* Hsave,
                                   void* ws, size_t ws_bytes, void* stream);

/* Column-parallel linear backward for dY[i] [T,N/n] (gather=1: dY[0] is [T,N]), input
 * dtype. dH_i = dY_i * act'(Hsave_i) (= dY_i with TP_ACT_NONE); dW[i] = X^T dH_i
 * [K,N/n]; dbias[i] = sum_t dH_i [N/n] (dbias may be NULL); dX = sum_i dH_i W_i^T [T,K].
 * Outputs fp32. */
tp_status tp_linear_column_backward(const tp_linear_desc* desc, const void* X,
                                    const void* const* W, const void* const* Hsave,
                                    const void* const* dY, void* dX, void* const* dW,
                                    void* const* dbias, void* ws, size_t ws_bytes,
                                    void* stream);

/* Row-parallel linear forward: Z = sum_i X_i W_i + bias. X[i] [T,K/n]; W[i] [K/n,N];
 * bias [N] or NULL; Z [T,N] fp32. */
tp_status tp_linear_row_forward(const tp_linear_desc* desc, const void* const* X,
                                const void* const* W, const void* bias, void* Z,
                                void* ws, size_t ws_bytes, void* stream);

/* Row-parallel linear backward for dZ [T,N] (input dtype): dX[i] = dZ W_i^T [T,K/n];
 * dW[i] = X_i^T dZ [K/n,N]; dbias = sum_t dZ [N] (may be NULL). Outputs fp32. */
tp_status tp_linear_row_backward(const tp_linear_desc* desc, const void* const* X,
                                 const void* const* W, const void* dZ, void* const* dX,
                                 void* const* dW, void* dbias, void* ws, size_t ws_bytes,
                                 void* stream);

/* ---------------------------------------------------------------------------------------
 * LayerNorm with the hidden dimension split over the shards ("Tensor Parallelism: principle
 * and practice", section 4.2: each device computes the mean and variance of its own part and
 * the statistics are synchronised by an All-Reduce). Shard i holds columns i*H/n ..
 * (i+1)*H/n - 1 of every token row as its own buffer X[i] [T, H/n] (row-major), with its
 * slices gamma[i], beta[i] [H/n]. The row statistics are the mean and the biased variance of
 * the whole row (H columns), eps added inside the square root:
 *   Y[i] = (X[i] - mean) / sqrt(var + eps) * gamma[i] + beta[i].
 * On this GPU the All-Reduce is the combination of the shards' (count, mean, M2) in shard
 * order inside the kernel (deterministic). dtype TP_BF16 or TP_F32 applies to X, Y, dY, dX,
 * gamma and beta; mean, rstd, dgamma, dbeta are fp32. bf16 needs H/n % 8 == 0 and 16-byte
 * aligned pointers; fp32 takes any width (16-byte accesses where rows and pointers allow).
 * No workspace; calls enqueue on `stream`; TP_ERR_* as for the other entry points. */
typedef struct tp_layernorm_desc {
  int64_t tokens;     /* T (>= 0) */
  int64_t hidden;     /* H, divisible by tp_degree */
  int32_t tp_degree;  /* n, 1..64 */
  int32_t dtype;      /* tp_dtype */
  float eps;          /* > 0 */
} tp_layernorm_desc;

/* Forward. gamma / beta: arrays of n pointers, or NULL for 1 / 0. mean, rstd: fp32 [T] or NULL
 * (not stored); the backward needs them. */
tp_status tp_layernorm_forward(const tp_layernorm_desc* desc, const void* const* X,
                               const void* const* gamma, const void* const* beta, void* const* Y,
                               float* mean, float* rstd, void* stream);

/* Backward for dY[i] [T, H/n]: dX[i] [T, H/n] (dtype) = rstd * (g - mean_row(g) - xhat *
 * mean_row(g * xhat)) with g = dY * gamma and xhat = (X - mean) * rstd over the whole row;
 * dgamma[i] = sum_t dY[i] * xhat, dbeta[i] = sum_t dY[i] (fp32 [H/n], arrays may be NULL: not
 * computed). mean, rstd: the forward's. */
tp_status tp_layernorm_backward(const tp_layernorm_desc* desc, const void* const* X,
                                const void* const* gamma, const float* mean, const float* rstd,
                                const void* const* dY, void* const* dX, float* const* dgamma,
                                float* const* dbeta, void* stream);

/* Launch tracing (profiling aid). While tracing is on, every kernel launch this library makes
 * (in any thread) is bracketed by two CUDA events recorded on the launch's stream, and the
 * launch's algorithmic work is noted: flops = 2*M*N*K per GEMM over all its shards; bytes =
 * each operand buffer read once plus each output written once. tp_trace_start(capacity) turns
 * tracing on for up to `capacity` launches (1..1000000; launches beyond it are not traced);
 * tp_trace_stop synchronises the recorded events, writes up to `capacity` records to `out`
 * (a host array), their number to *count, and turns tracing off. Events are created at start
 * and destroyed at stop: call both outside any stream capture. */
typedef enum tp_kernel_kind {
  TP_K_GEMM_TC = 1,        /* tcgen05 bf16 GEMM (any epilogue) */
  TP_K_GEMM_FFMA = 2,      /* fp32 FFMA GEMM */
  TP_K_SHARD_REDUCE = 3,   /* sum of fp32 shard partials (+ bias) */
  TP_K_COLSUM = 4,         /* bias gradients: column sums over tokens */
  TP_K_DACT = 5,           /* dH = dY * act'(H) */
  TP_K_SELFTEST = 6,
  TP_K_SHARD_COPY = 7,     /* token-shard gather / scatter (sequence parallel) */
  TP_K_LAYERNORM = 8,      /* hidden-split LayerNorm: row statistics + normalise (fwd, bwd dX) */
  TP_K_LN_PARAM_GRAD = 9   /* hidden-split LayerNorm: dgamma, dbeta column sums */
} tp_kernel_kind;

typedef enum tp_trace_tag {
  TP_TAG_COLUMN_FWD = 1,   /* H_i, Y_i = act(X A_i + a_i) */
  TP_TAG_ROW_FWD = 2,      /* Z = sum_i Y_i B_i + b (fused) or the partials */
  TP_TAG_ROW_DGRAD = 3,    /* dY_i = dZ B_i^T (MLP: times act'(H_i) -> dH_i) */
  TP_TAG_ROW_WGRAD = 4,    /* dB_i = Y_i^T dZ */
  TP_TAG_COLUMN_WGRAD = 5, /* dA_i = X^T dH_i */
  TP_TAG_COLUMN_DGRAD = 6, /* dX = sum_i dH_i A_i^T */
  TP_TAG_REDUCE = 7,       /* shard reduction of partials */
  TP_TAG_BIAS_GRAD = 8,    /* db, da_i */
  TP_TAG_ACT_GRAD = 9,     /* stand-alone dH = dY * act'(H) */
  TP_TAG_OTHER = 10,
  TP_TAG_SP_GATHER = 11,   /* all-gather of token shards */
  TP_TAG_SP_SCATTER = 12,  /* scatter of the summed rows to token shards */
  TP_TAG_LN_FWD = 13,      /* LayerNorm forward */
  TP_TAG_LN_DGRAD = 14,    /* LayerNorm input gradient */
  TP_TAG_LN_PARAM_GRAD = 15, /* LayerNorm dgamma, dbeta */
  TP_TAG_ROW_GRADS = 16,   /* dY_i (times act'(H_i)) and dB_i in one launch */
  TP_TAG_COLUMN_GRADS = 17 /* dA_i and dX in one launch */
} tp_trace_tag;

typedef struct tp_trace_record {
  int32_t kernel;   /* tp_kernel_kind */
  int32_t tag;      /* tp_trace_tag */
  double flops;     /* algorithmic flops of the launch */
  double bytes;     /* algorithmic bytes of the launch */
  float ms;         /* device time between the two events */
  int32_t groups;   /* shards handled by the launch */
} tp_trace_record;

tp_status tp_trace_start(int32_t capacity);
tp_status tp_trace_stop(tp_trace_record* out, int32_t capacity, int32_t* count);

/* Row-parallel linear forward for callers that cannot allocate device memory. The pages have
 * no counterpart to this entry point.
 *
 * Some callers have no way to call cudaMalloc: a plug-in running inside a host application
 * that owns every device allocation and forbids side allocations, or a process whose device
 * memory budget is fixed when it starts. This entry point takes no workspace: it computes the
 * same Z = sum_i X_i W_i + bias as tp_linear_row_forward in TP_REDUCE_PARTIALS form (desc->
 * reduce is ignored), with its status word and the per-shard fp32 partials in one static
 * device array of 32 MiB inside the library (every GPU that loads the library holds it until
 * the process exits). It allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 * call.
 *  - Limit: 256 + tp_degree * tokens * out_features * 4 bytes must fit in 32 MiB; larger calls
 *    return TP_ERR_WORKSPACE before anything is enqueued.
 *  - The first call on each device looks up the array's device address (once per device,
 *    with that device current); make that first call before any stream capture.
 *  - Every call on a device shares the one array and leaves its partials there; each call
 *    clears the status word itself. Calls whose work overlaps on the GPU (on different
 *    streams, or from different threads) race on the array: order them on one stream.
 *  - A device-side wait that runs out writes its code into the array's status word. With no
 *    workspace there is no tp_check_status to read it, so the call's last launch checks the
 *    word and, when it is set, fills Z with NaN: a timed-out call leaves Z all NaN, never a
 *    plausible-looking sum. The next call clears the word.
 * Arguments, layouts, dtypes and the other errors are those of tp_linear_row_forward. */
tp_status tp_linear_row_forward_noalloc(const tp_linear_desc* desc, const void* const* X,
                                        const void* const* W, const void* bias, void* Z,
                                        void* stream);

/* Self-test of the device-side timeout path: launches one block that waits on a barrier
 * nothing completes, with a limit of limit_us microseconds (1..1000000). The wait runs
 * out, the kernel writes TP_ERR_DEVICE_TIMEOUT's code into the workspace status word and
 * returns; a following tp_check_status returns TP_ERR_DEVICE_TIMEOUT. */
tp_status tp_selftest_wait_timeout(void* ws, size_t ws_bytes, uint32_t limit_us,
                                   void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TP_MLP_H */
