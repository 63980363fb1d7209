// Persistent, warp-specialised bf16 GEMM on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// One CTA per SM loops over output tiles of 128 x 256. Roles:
//   warp 0 (one lane)  : TMA producer -- streams 64-wide K slices of A and B into a
//                        4-stage ring of 128B-swizzled shared-memory tiles.
//   warp 1 (one lane)  : MMA issuer  -- tcgen05.mma (M=128, N=256, K=16, bf16 x bf16 -> fp32)
//                        into one of two TMEM accumulators (2 x 256 columns), so the
//                        epilogue of tile i overlaps the main loop of tile i+1.
//   warps 2..5         : epilogue    -- tcgen05.ld of the accumulator (one row per thread),
//                        the fused epilogue (bias, GeLU, GeLU'), coalesced fp32 / bf16 stores
//                        through a per-warp shared-memory staging buffer.
//
// Grouping: the tp_degree shards are groups of one launch. Output og accumulates the K ranges
// of groups og*kpo .. og*kpo + kpo - 1 into one TMEM accumulator, in group order: kpo = 1
// gives every group its own output; kpo = groups is the on-device form of the pages'
// All-Reduce (one output, the shard sum inside the accumulator); in between, the shard sum
// is split into groups/kpo partial outputs that a reduction kernel adds.
//
// Operand layouts: A is K-major ([M,K] row-major) or MN-major ([K,M] row-major); likewise
// B ([N,K] or [K,N]). The MN-major forms let the backward use X^T, Y_i^T, B_i^T and A_i^T
// straight from the forward's row-major buffers without a transpose.
//
// Every mbarrier wait is bounded (kWaitLimitNs); a wait that runs out records an error code
// in the status word, raises a CTA-wide abort flag, drains the copies and MMAs in flight,
// frees TMEM and returns.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "device_common.cuh"
#include "internal.h"

namespace tpk {
namespace tc {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;                       // one 128-byte swizzle row of bf16
constexpr int STAGES = 4;
constexpr int ACC_BUFS = 2;
constexpr int TMEM_COLS = ACC_BUFS * BN;     // 512 (all of TMEM)
constexpr int A_BYTES = BM * BK * 2;         // 16 KiB
constexpr int B_BYTES = BN * BK * 2;         // 32 KiB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int MN_BOX_BYTES = 64 * BK * 2;    // one [64 K rows][64 MN] box: 8 KiB
constexpr int NUM_THREADS = 192;
constexpr int NUM_BARS = 2 * STAGES + 2 * ACC_BUFS + 1;
constexpr int EPI_WARPS = 4;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_WARPS * 32 * 128 + 1024 + 256;

// The parameters of one grouped GEMM, for up to NM groups (tensor maps, outputs, bias and aux
// pointers per group). A launch of one GEMM takes NM = kMaxShards; a launch of two
// (TcDual) takes two blocks of kDualMaxShards, so that both fit in the kernel parameter space.
template <int NM>
struct __align__(128) TcParamsT {
  CUtensorMap tmA[NM];
  CUtensorMap tmB[NM];
  void* D[NM];
  void* D2[NM];
  const void* bias[NM];
  const void* aux[NM];
  long long ldd, ldd2, ldaux;
  int M, N;
  int kblocks;      // K blocks of 64 per group
  int groups;
  int kpo;          // groups summed into each output (1: one output per group)
  int tiles_m, tiles_n, num_tiles;
  int tiles_n_out;  // 256-column blocks of one output (for the partial-sum counters)
  int epi, act;
  int raster;       // tile order inside an output: 0 = m fastest, 1 = n fastest
  int a3d, b3d;     // MN-major operand mapped as [MN/64][K][64]: one TMA load per tile
  // EPI_PARTIAL_REDUCE: D[og] are the nsplit fp32 partials; the warp completing a
  // (32-row, 256-column) block's count sums them (+ zbias, bf16) into Z.
  int* counters;
  float* Z;
  long long ldz;
  const void* zbias;
  int nsplit;
  // Tail split (SM-pair kernel): units [0, full_tiles) are whole tiles; every tile t >=
  // full_tiles is computed as ksplit units ("pieces") of consecutive K blocks. A piece stores
  // its fp32 accumulator in tail_ws; the warp completing a (tile, 32-row block) count in
  // tail_counters adds the pieces in piece order and runs the tile's epilogue.
  int full_tiles, ksplit, num_units;
  float* tail_ws;
  int* tail_counters;
  int split_loads;  // SM-pair kernel: A and B loads issued by two threads (two warps)
  int mma_probe;    // SM-pair kernel: probe the next block's full barrier during the MMAs
  int load_probe;   // ... and the next block's empty barrier between the loads
  int* status;
};
using TcParams = TcParamsT<kMaxShards>;

// Two independent GEMMs in one SM-pair launch: work units [0, units0) are q[0]'s, the rest
// q[1]'s (unit u of the launch is unit u - units0 of q[1]); one queue deals them all to the pairs.
constexpr int kDualMaxShards = 16;
struct __align__(128) TcDual {
  TcParamsT<kDualMaxShards> q[2];
  int units0;
  int num_units;
};

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// One load of `chunks` consecutive 64-wide MN chunks of an MN-major operand, through its 3-D
// view [MN/64][K][64]: lands in shared memory exactly like `chunks` 2-D boxes of [64 K][64 MN].
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Shared-memory matrix descriptor of a 128B-swizzled operand tile (tcgen05 format:
// start >> 4 at bit 0, leading byte offset >> 4 at bit 16, stride byte offset >> 4 at bit
// 32, descriptor version 1 at bit 46, swizzle mode "128B" = 2 at bit 61).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, operand majors,
// N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 lanes x 32 consecutive fp32 columns: thread t of the warp gets row (quadrant + t).
// The wait is in the same asm statement, so no use of r[] can be scheduled before it.
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
      "[%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ------------------------------------------------------------------ tile decode
// Tile t -> output index og, m block, n block. With m fastest, the tiles running at the same
// time share B blocks and sweep all of A; with n fastest, they share A blocks and sweep B.
template <class P>
__device__ __forceinline__ void decode_tile(const P& p, int t, int& g, int& mb, int& nb) {
  const int per = p.tiles_m * p.tiles_n;
  g = t / per;
  const int r = t - g * per;
  if (p.raster == 0) {
    mb = r % p.tiles_m;
    nb = r / p.tiles_m;
  } else {
    nb = r % p.tiles_n;
    mb = r / p.tiles_n;
  }
}

// Work unit u -> tile t and its K blocks [kb0, kb1); piece = -1 for a whole tile.
template <class P>
__device__ __forceinline__ void decode_unit(const P& p, int u, int total_kb, int& t,
                                            int& kb0, int& kb1, int& piece) {
  if (u < p.full_tiles) {
    t = u;
    kb0 = 0;
    kb1 = total_kb;
    piece = -1;
    return;
  }
  const int v = u - p.full_tiles;
  t = p.full_tiles + v / p.ksplit;
  piece = v % p.ksplit;
  kb0 = static_cast<int>(static_cast<long long>(total_kb) * piece / p.ksplit);
  kb1 = static_cast<int>(static_cast<long long>(total_kb) * (piece + 1) / p.ksplit);
}

// ------------------------------------------------------------------ epilogue (32 rows x 32 cols per warp)
// Each lane of an epilogue warp holds 32 consecutive accumulator columns of one row
// (row = row0 + lane). Global memory is touched through the warp's 4 KiB staging buffer so
// that every store (and the GeLU' input load) moves whole row segments: 4 rows x 128 B per
// instruction for fp32, 8 rows x 64 B for bf16. 16-byte chunks are XOR-swizzled by row in the
// staging buffer, which keeps both the row-wise and the column-wise accesses free of bank
// conflicts.
constexpr int STAGE_WARP_BYTES = 32 * 128;

__device__ __forceinline__ void warp_store_f32(uint8_t* stage, const float* v, float* D,
                                               long long ldd, int row0, int col0, int M,
                                               int valid) {
  const int lane = threadIdx.x & 31;
  float4* s4 = reinterpret_cast<float4*>(stage);
#pragma unroll
  for (int q = 0; q < 8; ++q)
    s4[lane * 8 + (q ^ (lane & 7))] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  __syncwarp();
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int r = 4 * it + (lane >> 3);
    const int c = lane & 7;
    const float4 x = s4[r * 8 + (c ^ (r & 7))];
    if (row0 + r < M && 4 * c < valid)
      *reinterpret_cast<float4*>(D + static_cast<long long>(row0 + r) * ldd + col0 + 4 * c) = x;
  }
  __syncwarp();
}

__device__ __forceinline__ void warp_store_bf16(uint8_t* stage, const float* v, uint16_t* D,
                                                long long ldd, int row0, int col0, int M,
                                                int valid) {
  const int lane = threadIdx.x & 31;
  uint4* s = reinterpret_cast<uint4*>(stage);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    u.x = pack_bf16x2(v[q * 8 + 0], v[q * 8 + 1]);
    u.y = pack_bf16x2(v[q * 8 + 2], v[q * 8 + 3]);
    u.z = pack_bf16x2(v[q * 8 + 4], v[q * 8 + 5]);
    u.w = pack_bf16x2(v[q * 8 + 6], v[q * 8 + 7]);
    s[lane * 4 + (q ^ ((lane >> 1) & 3))] = u;
  }
  __syncwarp();
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int r = 8 * it + (lane >> 2);
    const int c = lane & 3;
    const uint4 x = s[r * 4 + (c ^ ((r >> 1) & 3))];
    if (row0 + r < M && 8 * c < valid)
      *reinterpret_cast<uint4*>(D + static_cast<long long>(row0 + r) * ldd + col0 + 8 * c) = x;
  }
  __syncwarp();
}

// The transpose of warp_store_bf16, in two halves so that the loads can be issued ahead of
// their use. warp_fetch_bf16: coalesced 16-byte loads of the 32 x 32 bf16 block at
// src[row0.., col0..] into four registers per lane (0 outside the matrix).
__device__ __forceinline__ void warp_fetch_bf16(const uint16_t* src, long long ld, int row0,
                                                int col0, int M, int valid, uint4* raw) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int r = 8 * it + (lane >> 2);
    const int c = lane & 3;
    raw[it] = make_uint4(0u, 0u, 0u, 0u);
    if (row0 + r < M && 8 * c < valid)
      raw[it] = *reinterpret_cast<const uint4*>(src + static_cast<long long>(row0 + r) * ld + col0 + 8 * c);
  }
}

// warp_unpack_bf16: through the warp's staging buffer, lane l gets the 32 values of row
// row0 + l of a fetched block, as fp32.
__device__ __forceinline__ void warp_unpack_bf16(uint8_t* stage, const uint4* raw, float* out) {
  const int lane = threadIdx.x & 31;
  uint4* s = reinterpret_cast<uint4*>(stage);
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int r = 8 * it + (lane >> 2);
    const int c = lane & 3;
    s[r * 4 + (c ^ ((r >> 1) & 3))] = raw[it];
  }
  __syncwarp();
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 u = s[lane * 4 + (q ^ ((lane >> 1) & 3))];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = unpack_bf16x2(w[j]);
      out[q * 8 + 2 * j] = f.x;
      out[q * 8 + 2 * j + 1] = f.y;
    }
  }
  __syncwarp();
}

// EPI_DACT with an activation reads the saved pre-activation at every output element.
template <class P>
__device__ __forceinline__ bool dact_reads_aux(const P& p) {
  return p.epi == EPI_DACT && p.act == TP_ACT_GELU_ERF;
}

// Lane l asks L2 for row row0 + l of the pre-activation block [row0.., col0.., up to ncols
// columns] of group g: one bulk prefetch per row (16-byte aligned start, a multiple of 16
// bytes long: bf16 rows and N are multiples of 8, col0 of 256).
template <class P>
__device__ __forceinline__ void prefetch_aux_rows(const P& p, int g, int row0, int col0,
                                                  int ncols) {
  const int lane = threadIdx.x & 31;
  const int row = row0 + lane;
  const int cols = min(ncols, p.N - col0);
  if (row < p.M && cols > 0)
    prefetch_l2(static_cast<const uint16_t*>(p.aux[g]) + static_cast<long long>(row) * p.ldaux + col0,
                static_cast<uint32_t>(cols) * 2u);
}

// Per-column bias (bf16), the same 32 values for every lane: broadcast loads. Columns at or
// beyond `valid` (a multiple of 8) read as 0.
__device__ __forceinline__ void add_bias_bf16x32(const uint16_t* bias, int valid, float* v) {
  const uint4* s = reinterpret_cast<const uint4*>(bias);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (q * 8 < valid) {
      const uint4 u = s[q];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __fadd2_rn(make_float2(v[q * 8 + 2 * j], v[q * 8 + 2 * j + 1]),
                                    unpack_bf16x2(w[j]));
        v[q * 8 + 2 * j] = f.x;
        v[q * 8 + 2 * j + 1] = f.y;
      }
    }
  }
}

__device__ __forceinline__ float4 ld_cg_f4(const float* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// The shard sum overlapped with the GEMM (EPI_PARTIAL_REDUCE), warp-wide, after the warp has
// stored its 32 rows of partial og (all 256 columns of the block, or its share of them when
// warps_per_block warps split the columns): the warp makes its stores visible and counts
// itself in for the block; the warp that completes the count (one per block, whichever
// partial it computed) reads the nsplit partials of the block in partial order, adds the bias
// and writes Z, then resets the counter for the next launch. No warp waits for another.
template <class P>
__device__ __forceinline__ void partial_reduce_rows(const P& p, int row0, int nb,
                                                   int warps_per_block = 1) {
  const int lane = threadIdx.x & 31;
  if (row0 >= p.M) return;  // no rows of this block exist (edge tile): nothing was stored
  __threadfence();
  __syncwarp();
  const int block = (row0 >> 5) * p.tiles_n_out + nb;
  int last = 0;
  if (lane == 0) last = atomicAdd(p.counters + block, 1) == p.nsplit * warps_per_block - 1;
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __threadfence();
  const int col = nb * 256 + lane * 8;  // N % 8 == 0: a lane's 8 columns are all in or all out
  if (col < p.N) {
    float b[8] = {};
    if (p.zbias != nullptr) {
      const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.zbias) + col);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = unpack_bf16x2(w[j]);
        b[2 * j] = f.x;
        b[2 * j + 1] = f.y;
      }
    }
    for (int r = 0; r < 32 && row0 + r < p.M; ++r) {
      const long long row = row0 + r;
      float acc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = 0.f;
      for (int sp = 0; sp < p.nsplit; ++sp) {
        const float* src = static_cast<const float*>(p.D[sp]) + row * p.ldd + col;
        const float4 x0 = ld_cg_f4(src), x1 = ld_cg_f4(src + 4);
        acc[0] += x0.x; acc[1] += x0.y; acc[2] += x0.z; acc[3] += x0.w;
        acc[4] += x1.x; acc[5] += x1.y; acc[6] += x1.z; acc[7] += x1.w;
      }
      float* dst = p.Z + row * p.ldz + col;
      reinterpret_cast<float4*>(dst)[0] = make_float4(acc[0] + b[0], acc[1] + b[1], acc[2] + b[2], acc[3] + b[3]);
      reinterpret_cast<float4*>(dst)[1] = make_float4(acc[4] + b[4], acc[5] + b[5], acc[6] + b[6], acc[7] + b[7]);
    }
  }
  __syncwarp();
  if (lane == 0) atomicExch(p.counters + block, 0);
}

// Warp-wide: all 32 lanes call this for the same (row0, col0).
template <class P>
__device__ __forceinline__ void epilogue_chunk(const P& p, int g, int row0, int col0,
                                               float* v, uint8_t* stage) {
  const int valid = min(32, p.N - col0);  // a multiple of 8 (N % 8 == 0)
  const int og = g;
  if (p.epi == EPI_STORE_F32 || p.epi == EPI_PARTIAL_REDUCE) {
    if (p.bias[og] != nullptr) add_bias_bf16x32(static_cast<const uint16_t*>(p.bias[og]) + col0, valid, v);
    warp_store_f32(stage, v, static_cast<float*>(p.D[og]), p.ldd, row0, col0, p.M, valid);
  } else if (p.epi == EPI_STORE_BF16) {
    if (p.bias[og] != nullptr) add_bias_bf16x32(static_cast<const uint16_t*>(p.bias[og]) + col0, valid, v);
    warp_store_bf16(stage, v, static_cast<uint16_t*>(p.D[og]), p.ldd, row0, col0, p.M, valid);
  } else if (p.epi == EPI_BIAS_ACT) {
    if (p.bias[og] != nullptr) add_bias_bf16x32(static_cast<const uint16_t*>(p.bias[og]) + col0, valid, v);
    if (p.D[og] != nullptr)
      warp_store_bf16(stage, v, static_cast<uint16_t*>(p.D[og]), p.ldd, row0, col0, p.M, valid);
    if (p.act == TP_ACT_GELU_ERF) {
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float2 y = gelu_erf2(make_float2(v[i], v[i + 1]));
        v[i] = y.x;
        v[i + 1] = y.y;
      }
    }
    warp_store_bf16(stage, v, static_cast<uint16_t*>(p.D2[og]), p.ldd2, row0, col0, p.M, valid);
  } else {  // EPI_DACT (aux = the saved pre-activation, read only with an activation)
    if (p.act == TP_ACT_GELU_ERF) {
      float h[32];
      uint4 raw[4];
      warp_fetch_bf16(static_cast<const uint16_t*>(p.aux[og]), p.ldaux, row0, col0, p.M, valid, raw);
      warp_unpack_bf16(stage, raw, h);
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float2 y = __fmul2_rn(make_float2(v[i], v[i + 1]),
                                    gelu_erf_grad2(make_float2(h[i], h[i + 1])));
        v[i] = y.x;
        v[i + 1] = y.y;
      }
    }
    warp_store_bf16(stage, v, static_cast<uint16_t*>(p.D[og]), p.ldd, row0, col0, p.M, valid);
  }
}

// One warp's 32 rows x NCOLS columns (from colbase) of a finished accumulator at TMEM address
// trow, 32 columns at a time. With EPI_DACT + activation, the pre-activation loads of the
// next 32 columns are issued before the current ones are used, so each chunk's DRAM/L2 round
// trip overlaps the previous chunk's work instead of stalling the warp.
template <int NCOLS, class P>
__device__ __forceinline__ void epilogue_rows(const P& p, int g, int row0, int colbase,
                                              uint32_t trow, uint8_t* stage) {
  if (!dact_reads_aux(p)) {
    for (int c0 = 0; c0 < NCOLS; c0 += 32) {
      const int col0 = colbase + c0;
      if (col0 >= p.N) break;  // uniform across the warp
      float v[32];
      tmem_ld_32cols(trow + c0, v);
      epilogue_chunk(p, g, row0, col0, v, stage);
    }
    return;
  }
  const uint16_t* aux = static_cast<const uint16_t*>(p.aux[g]);
  uint4 nxt[4];
  warp_fetch_bf16(aux, p.ldaux, row0, colbase, p.M, min(32, p.N - colbase), nxt);
  for (int c0 = 0; c0 < NCOLS; c0 += 32) {
    const int col0 = colbase + c0;
    if (col0 >= p.N) break;
    const uint4 cur[4] = {nxt[0], nxt[1], nxt[2], nxt[3]};
    if (c0 + 32 < NCOLS && col0 + 32 < p.N)
      warp_fetch_bf16(aux, p.ldaux, row0, col0 + 32, p.M, min(32, p.N - col0 - 32), nxt);
    float v[32], h[32];
    tmem_ld_32cols(trow + c0, v);
    warp_unpack_bf16(stage, cur, h);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const float2 y = __fmul2_rn(make_float2(v[i], v[i + 1]),
                                  gelu_erf_grad2(make_float2(h[i], h[i + 1])));
      v[i] = y.x;
      v[i + 1] = y.y;
    }
    warp_store_bf16(stage, v, static_cast<uint16_t*>(p.D[g]), p.ldd, row0, col0, p.M,
                    min(32, p.N - col0));
  }
}

// The same for a column count known only at run time (the SM-pair kernel with 12 epilogue
// warps, whose warps take 96 or 64 columns). A separate copy, so that the loops of the
// fixed-width form above compile as they always have.
template <class P>
__device__ __forceinline__ void epilogue_rows_n(const P& p, int g, int row0, int colbase,
                                                int ncols, uint32_t trow, uint8_t* stage) {
  if (!dact_reads_aux(p)) {
#pragma unroll 1
    for (int c0 = 0; c0 < ncols; c0 += 32) {
      const int col0 = colbase + c0;
      if (col0 >= p.N) break;  // uniform across the warp
      float v[32];
      tmem_ld_32cols(trow + c0, v);
      epilogue_chunk(p, g, row0, col0, v, stage);
    }
    return;
  }
  const uint16_t* aux = static_cast<const uint16_t*>(p.aux[g]);
  uint4 nxt[4];
  warp_fetch_bf16(aux, p.ldaux, row0, colbase, p.M, min(32, p.N - colbase), nxt);
#pragma unroll 1
  for (int c0 = 0; c0 < ncols; c0 += 32) {
    const int col0 = colbase + c0;
    if (col0 >= p.N) break;
    const uint4 cur[4] = {nxt[0], nxt[1], nxt[2], nxt[3]};
    if (c0 + 32 < ncols && col0 + 32 < p.N)
      warp_fetch_bf16(aux, p.ldaux, row0, col0 + 32, p.M, min(32, p.N - col0 - 32), nxt);
    float v[32], h[32];
    tmem_ld_32cols(trow + c0, v);
    warp_unpack_bf16(stage, cur, h);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const float2 y = __fmul2_rn(make_float2(v[i], v[i + 1]),
                                  gelu_erf_grad2(make_float2(h[i], h[i + 1])));
      v[i] = y.x;
      v[i + 1] = y.y;
    }
    warp_store_bf16(stage, v, static_cast<uint16_t*>(p.D[g]), p.ldd, row0, col0, p.M,
                    min(32, p.N - col0));
  }
}

// ------------------------------------------------------------------ the kernel
template <bool A_MN, bool B_MN>
__global__ void __launch_bounds__(NUM_THREADS, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* epi_stage = smem + STAGES * STAGE_BYTES;  // EPI_WARPS x 4 KiB
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi_stage + EPI_WARPS * STAGE_WARP_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const uint32_t smem_base = smem_addr(smem);
  const uint32_t bar_base = smem_addr(bars);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + ACC_BUFS + a); };
  const uint32_t drain_bar = bar_base + 8u * (2 * STAGES + 2 * ACC_BUFS);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < ACC_BUFS; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int total_kb = p.kblocks * p.kpo;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      // The loop is kept short (no division, the abort flag read only while a wait polls):
      // this one thread issues every load of the CTA.
      uint32_t stage = 0, phase = 0;
      long long issued = 0;
      bool failed = false;
      const int kend = p.kblocks * BK;
      for (int t = blockIdx.x; t < p.num_tiles && !failed; t += gridDim.x) {
        int g, mb, nb;
        decode_tile(p, t, g, mb, nb);
        int kg = g * p.kpo, kk = 0;
        for (int kb = 0; kb < total_kb; ++kb) {
          const int w = mbar_wait_or_abort(empty_bar(stage), phase ^ 1u, abort_flag, kWaitLimitNs);
          if (w <= 0) {
            if (w < 0) {
              report_status(p.status, kDevTimeoutBase | 0x10);
              *abort_flag = 1;
            }
            failed = true;
            break;
          }
          const uint32_t fb = full_bar(stage);
          const uint32_t sa = smem_base + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          if (!A_MN) {
            tma_load_2d(sa, &p.tmA[kg], kk, mb * BM, fb);
          } else if (p.a3d) {
            tma_load_3d(sa, &p.tmA[kg], 0, kk, mb * BM / 64, fb);
          } else {
#pragma unroll
            for (int j = 0; j < BM / 64; ++j)
              tma_load_2d(sa + j * MN_BOX_BYTES, &p.tmA[kg], mb * BM + 64 * j, kk, fb);
          }
          if (!B_MN) {
            tma_load_2d(sb, &p.tmB[kg], kk, nb * BN, fb);
          } else if (p.b3d) {
            tma_load_3d(sb, &p.tmB[kg], 0, kk, nb * BN / 64, fb);
          } else {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_2d(sb + j * MN_BOX_BYTES, &p.tmB[kg], nb * BN + 64 * j, kk, fb);
          }
          ++issued;
          kk += BK;
          if (kk == kend) { kk = 0; ++kg; }
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // another role may have given up after this thread's last wait
      if (!failed && *abort_flag) failed = true;
      if (failed) {
        // Drain: wait (bounded) until every copy this thread issued has landed.
        for (int s = 0; s < STAGES; ++s) {
          if (issued > s) {
            const long long last = s + ((issued - 1 - s) / STAGES) * STAGES;
            mbar_wait_bounded(full_bar(s), static_cast<uint32_t>((last / STAGES) & 1), 100000000ull);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = idesc_bf16(BM, BN, A_MN, B_MN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool failed = false;
      for (int t = blockIdx.x; t < p.num_tiles && !failed; t += gridDim.x) {
        const int we = mbar_wait_or_abort(tempty_bar(acc), acc_phase ^ 1u, abort_flag, kWaitLimitNs);
        if (we <= 0) {
          if (we < 0) {
            report_status(p.status, kDevTimeoutBase | 0x20);
            *abort_flag = 1;
          }
          failed = true;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < total_kb; ++kb) {
          const int w = mbar_wait_or_abort(full_bar(stage), phase, abort_flag, kWaitLimitNs);
          if (w <= 0) {
            if (w < 0) {
              report_status(p.status, kDevTimeoutBase | 0x21);
              *abort_flag = 1;
            }
            failed = true;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_base + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = A_MN ? sdesc_sw128(sa + k * 2048, MN_BOX_BYTES, 1024)
                                     : sdesc_sw128(sa + k * 32, 16, 1024);
            const uint64_t bd = B_MN ? sdesc_sw128(sb + k * 2048, MN_BOX_BYTES, 1024)
                                     : sdesc_sw128(sb + k * 32, 16, 1024);
            umma_bf16(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit(empty_bar(stage));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (failed) break;
        umma_commit(tfull_bar(acc));
        if (++acc == ACC_BUFS) { acc = 0; acc_phase ^= 1u; }
      }
      if (!failed && *abort_flag) failed = true;   // MMAs of a tile no epilogue will read
      if (failed) {
        // Drain: all MMAs issued so far complete before TMEM is freed.
        umma_commit(drain_bar);
        mbar_wait_bounded(drain_bar, 0, 100000000ull);
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue warps 2..5
    const int quad = warp & 3;  // TMEM lanes this warp may read: 32*quad .. 32*quad+31
    uint32_t acc = 0, acc_phase = 0;
    // With the GeLU' epilogue, each tile's pre-activation rows are requested into L2 one tile
    // ahead (the first tile's here), while the tile before it is being finished.
    const bool aux_ahead = dact_reads_aux(p);
    if (aux_ahead && static_cast<int>(blockIdx.x) < p.num_tiles) {
      int g1, mb1, nb1;
      decode_tile(p, blockIdx.x, g1, mb1, nb1);
      prefetch_aux_rows(p, g1, mb1 * BM + quad * 32, nb1 * BN, BN);
    }
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      int g, mb, nb;
      decode_tile(p, t, g, mb, nb);
      if (aux_ahead && t + static_cast<int>(gridDim.x) < p.num_tiles) {
        int g1, mb1, nb1;
        decode_tile(p, t + gridDim.x, g1, mb1, nb1);
        prefetch_aux_rows(p, g1, mb1 * BM + quad * 32, nb1 * BN, BN);
      }
      if (!mbar_wait_bounded(tfull_bar(acc), acc_phase, kWaitLimitNs)) {
        if (lane == 0) report_status(p.status, kDevTimeoutBase | 0x30);
        *abort_flag = 1;
        break;
      }
      if (*abort_flag) break;
      tc_fence_after();
      const int row0 = mb * BM + quad * 32;  // this warp's 32 rows
      const uint32_t trow = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN;
      uint8_t* stage = epi_stage + (warp - 2) * STAGE_WARP_BYTES;
      epilogue_rows<BN>(p, g, row0, nb * BN, trow, stage);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
      if (p.epi == EPI_PARTIAL_REDUCE) partial_reduce_rows(p, row0, nb);
      if (++acc == ACC_BUFS) { acc = 0; acc_phase ^= 1u; }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

}  // namespace tc
}  // namespace tpk
