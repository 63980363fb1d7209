/*
 * tp_mlp_tuning.h -- test and measurement hook of libtpmlp.so (not for production callers).
 *
 * The library picks, per launch, among kernel variants by measurement on GB300: SM-pair or
 * one-SM tensor-core GEMM, 4 or 8 epilogue warps, tile order, one 3-D or several 2-D TMA
 * boxes, one or two producer threads, the issue loops' barrier probes, the K split of a
 * last partial wave, the shard-sum grouping, the fp32 GEMM kernel for few rows and its K split
 * over a cluster, and the LayerNorm kernels. Every variant computes the same operation (none of them is a different
 * reading of the pages); those marked "bit-identical" give the same bits as the default, the
 * others differ from it only in the fp32 summation order. The tests pin each variant against
 * the default and the oracle through this hook, and A/B timings use it.
 *
 * Overrides are process-wide, held in the library (no environment variable is read), and
 * take effect at the next launch; a value of TP_TUNE_AUTO gives the choice back to the
 * library. They are meant to be set between calls from one thread: a launch that runs while
 * another thread changes a knob sees either value.
 */
#ifndef TP_MLP_TUNING_H
#define TP_MLP_TUNING_H

#include <stdint.h>

#include "tp_mlp.h"

#ifdef __cplusplus
extern "C" {
#endif

#define TP_TUNE_AUTO (-1)

typedef enum tp_tune_knob {
  TP_TUNE_GEMM_PAIR = 0,    /* 0: one-SM tcgen05 GEMM, 1: SM pairs (default: pairs when M > 128) */
  TP_TUNE_EPI_WARPS = 1,    /* 4, 8 or 12 epilogue warps in the SM-pair GEMM (bit-identical;
                               12: whole tiles only, one K block per ring stage) */
  TP_TUNE_RASTER = 2,       /* tile order inside an output: 0 m fastest, 1 n fastest (bit-identical) */
  TP_TUNE_TMA_3D = 3,       /* 0/1: MN-major operands as 2-D boxes / one 3-D box (bit-identical) */
  TP_TUNE_SPLIT_LOADS = 4,  /* 0/1: A and B loads from one / two producer threads (bit-identical) */
  TP_TUNE_MMA_PROBE = 5,    /* 0/1: MMA issuer's early look at the next stage (bit-identical) */
  TP_TUNE_LOAD_PROBE = 6,   /* 0/1: producers' early look at the next stage (bit-identical) */
  TP_TUNE_TAIL_SPLIT = 7,   /* 0/1: K split of the last partial wave's tiles */
  TP_TUNE_TAIL_WAVES = 8,   /* wave limit (>= 1) below which shallow tiles are tail-split */
  TP_TUNE_SHARD_SPLIT = 9,  /* S partial outputs of a shard sum under TP_REDUCE_AUTO/OVERLAP
                               (a divisor of tp_degree; others fall back to the library's) */
  TP_TUNE_SIMT_SPLIT = 10,  /* 0: no K split over a cluster in the fp32 FFMA GEMM */
  TP_TUNE_LN_REG = 11,      /* 0/1: two-pass / register-resident LayerNorm kernels (bit-identical) */
  TP_TUNE_PDL = 12,         /* 0/1: SM-pair GEMMs and column sums launched without / with
                               programmatic stream serialisation (default on: each launch's
                               set-up overlaps the previous kernel's end; bit-identical) */
  TP_TUNE_STAGE_BLOCKS = 13, /* 1 or 2: 64-deep K blocks per operand-ring stage of the SM-pair
                               GEMM (6 stages of 64 or 3 of 128; bit-identical) */
  TP_TUNE_TAIL_PIECES = 14, /* upper bound (>= 1) on the K pieces of a split tail tile */
  TP_TUNE_FEW_ROWS = 15,    /* 0: fp32 products of <= 32 rows on the general FFMA kernel instead
                               of the bulk-copy one (forward layouts) */
  TP_TUNE_DUAL = 16,        /* 0/1: the backward's independent bf16 GEMMs (MLP: dY_i with dB_i, dA_i
                               with dX; linear layers: dW_i with dX) in separate launches / in one
                               SM-pair launch wherever they fit it (default: where one of them has
                               at most one wave of tiles; bit-identical) */
  TP_TUNE_COUNT = 17
} tp_tune_knob;

/* Sets knob to value (TP_TUNE_AUTO: the library's choice). TP_ERR_DTYPE for an unknown
 * knob; TP_ERR_SHAPE for a value below TP_TUNE_AUTO. Never touches the GPU. */
tp_status tp_tuning_set(int32_t knob, int32_t value);

/* The current override of knob (TP_TUNE_AUTO when none), or TP_TUNE_AUTO - 1 for an
 * unknown knob. */
int32_t tp_tuning_get(int32_t knob);

#ifdef __cplusplus
}
#endif

#endif /* TP_MLP_TUNING_H */
