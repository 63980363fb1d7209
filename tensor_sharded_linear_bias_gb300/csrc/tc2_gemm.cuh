// The same grouped bf16 GEMM on pairs of SMs: tcgen05.mma.cta_group::2.
//
// A cluster of two CTAs (one per SM) computes a 256 x 256 output tile. Each CTA stages its own
// 128 rows of A and its own 128-column half of B (32 KiB per 64-deep K block, a ring of 6
// blocks, 5 with 12 epilogue warps); one MMA issued by the even CTA reads both CTAs' shared
// memory and writes each CTA's 128 accumulator rows (all 256 columns) into that CTA's TMEM. Per
// k block an SM takes in 32 KiB instead of the 48 KiB of the one-SM 128 x 256 tile, for the
// same tensor work per SM. The clusters are persistent and walk a queue of work units (tiles,
// or K pieces of split tail tiles) of one grouped GEMM, or of two independent GEMMs.
//
// Synchronisation (mbarriers; the even CTA is the "leader"):
//   full[s]   leader only: the leader's A producer posts expect_tx for both halves (64 KiB);
//             both CTAs' TMA loads complete their bytes on it (.cta_group::2 loads).
//   empty[s]  in both CTAs: the leader's MMA commit arrives on both (multicast).
//   tfull[a]  in both CTAs: the leader's commit after a tile's last MMA (multicast).
//   tempty[a] leader only: the EPI_W epilogue warps of both CTAs arrive (count 2 EPI_W).
// The issue loops are single threads (one MMA issuer, one or two producers per CTA): each
// keeps its per-block work short and looks at the next block's barrier while the current
// block's last MMA (or load) issues, so that a wait that would succeed at once costs nothing.
// TMEM (all 512 columns, two 256-column accumulators) is allocated and freed by warp 1 of
// both CTAs together (cta_group::2). Cluster barriers after set-up and before the end keep
// either CTA from touching the other's shared memory before it is ready or after it is gone.
//
// Every mbarrier wait is bounded as in the one-SM kernel; a wait that runs out records a
// code in the status word, raises the CTA's abort flag and lets the CTA wind down.
#pragma once

#include "tc_gemm.cuh"

namespace tpk {
namespace tc2 {

using tc::BK;
using tc::TcParams;

constexpr int BM = 256;                      // rows per CTA pair (128 per CTA)
constexpr int BN = 256;                      // columns per tile (128 of B staged per CTA)
constexpr int HALF = 128;
constexpr int ACC_BUFS = 2;
constexpr int TMEM_COLS = ACC_BUFS * BN;     // 512
constexpr int A_BYTES = HALF * BK * 2;       // 16 KiB
constexpr int B_BYTES = HALF * BK * 2;       // 16 KiB
constexpr int BLOCK_BYTES = A_BYTES + B_BYTES;  // one 64-deep K block of A and B per CTA: 32 KiB
constexpr int RING_BLOCKS = 6;                  // K blocks the operand ring holds (192 KiB)
// The ring is cut into stages of SUB K blocks (SUB = 1: 6 stages of 64; SUB = 2: 3 stages of
// 128). Each stage has one full and one empty barrier, so the MMA issuer's fixed work per stage
// (the barrier wait or look-ahead, the commit that releases the stage) is paid once per SUB K
// blocks; the price is a coarser release (a stage is refilled only when all its blocks are
// consumed). Inside a stage, block j sits at j * BLOCK_BYTES with the layout of a one-block
// stage, so TMA boxes and MMA descriptors are the same for both.
template <int SUB, int BLOCKS = RING_BLOCKS>
struct Ring {
  static_assert(SUB == 1 || SUB == 2, "1 or 2 K blocks per stage");
  static_assert(BLOCKS % SUB == 0, "whole stages");
  static constexpr int STAGES = BLOCKS / SUB;
  static constexpr int STAGE_BYTES = SUB * BLOCK_BYTES;
};
constexpr int MN_BOX_BYTES = 64 * BK * 2;    // 8 KiB
// Warp 0: TMA producer (A); warp 1: MMA issuer; warps 2..: EPI_W epilogue warps; the last
// warp: TMA producer (B), so that no single thread's issue loop paces the ring. A warp may only
// read the 32 TMEM lanes of quadrant warp % 4, so with 4 epilogue warps each takes all 256
// columns of its 32 rows, with 8 two warps share a quadrant and take 128 columns each (for
// epilogue-heavy tiles, GeLU or GeLU', whose K loops are too short to hide 4 warps' work), and
// with 12 three warps take 96, 96 and 64 columns (their 12 staging buffers leave room for a
// ring of 5 K blocks; whole tiles only, no split tail pieces).
template <int EPI_W>
struct EpiShape {
  static_assert(EPI_W == 4 || EPI_W == 8 || EPI_W == 12, "4, 8 or 12 epilogue warps");
  static constexpr int WARPS = EPI_W;
  static constexpr int PER_QUAD = EPI_W / 4;  // warps sharing a TMEM quadrant
  // columns of the warp that is j-th in its quadrant (the largest: COLS)
  static constexpr int COLS = EPI_W == 12 ? 96 : BN * 4 / EPI_W;
  __device__ static int cofs(int j) { return j * COLS; }
  __device__ static int ncols(int j) { return j == PER_QUAD - 1 ? BN - j * COLS : COLS; }
  static constexpr int B_WARP = 2 + EPI_W;         // the B producer, after the epilogue warps
  static constexpr int THREADS = 96 + 32 * EPI_W;
  static constexpr int RING = EPI_W == 12 ? 5 : RING_BLOCKS;  // K blocks of the operand ring
  static constexpr int SMEM = RING * BLOCK_BYTES + EPI_W * tc::STAGE_WARP_BYTES + 1024 + 256;
};
constexpr int NUM_BARS = 2 * RING_BLOCKS + 2 * ACC_BUFS + 1;  // sized for the most stages

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// Shared::cluster address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// TMA load into this CTA's shared memory whose completion is counted on an mbarrier that may
// live in the peer CTA (`bar` is a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                 uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                 int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// Arrives on the mbarrier at shared offset `bar` in every CTA of `mask` once all MMAs issued
// so far by this thread have completed.
__device__ __forceinline__ void umma_commit_pair_multicast(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

// ------------------------------------------------------------------ tail split
// A piece's accumulator in the tail workspace: [piece][256 rows][256 columns] fp32 per tile.
constexpr int PIECE_FLOATS = BM * BN;
// one counter per (tile, CTA, column part, lane quadrant): the rows and columns of one warp
constexpr int TAIL_COUNTERS_PER_TILE = 2 * 2 * 4;

// One warp stores its 32 accumulator rows (tile-local rows lrow0..lrow0+31) x COLS columns
// (from tile column cofs; trow addresses that column) of a piece, through its staging buffer.
template <int COLS>
__device__ __forceinline__ void store_piece_rows(float* piece_ws, int lrow0, int cofs,
                                                 uint32_t trow, uint8_t* stage) {
  for (int c0 = 0; c0 < COLS; c0 += 32) {
    float v[32];
    tc::tmem_ld_32cols(trow + c0, v);
    tc::warp_store_f32(stage, v, piece_ws, BN, lrow0, cofs + c0, BM, 32);
  }
}

// Warp-wide, after the warp's piece rows are stored: make them visible and count the warp in
// for its (tile, 32-row block). True for the warp that completes the count (it then sees every
// piece's rows).
__device__ __forceinline__ bool tail_last_arrival(int* counter, int pieces) {
  const int lane = threadIdx.x & 31;
  __threadfence();
  __syncwarp();
  int last = 0;
  if (lane == 0) last = atomicAdd(counter, 1) == pieces - 1;
  last = __shfl_sync(0xffffffffu, last, 0);
  if (last) __threadfence();
  return last != 0;
}

// The completing warp adds its 32 rows of every piece in piece order, 32 columns at a time, and
// runs the tile's epilogue on the sums as for an unsplit tile. Reads are coalesced (each
// instruction covers 4 rows x 128 bytes) and two pieces' loads are in flight at once; the
// 32 x 32 sum is turned into one row per lane through the warp's staging buffer.
template <int COLS, class P>
__device__ __forceinline__ void tail_fixup_rows(const P& p, int g, int row0, int colbase,
                                                const float* tile_ws, int lrow0, int cofs,
                                                uint8_t* stage) {
  const int lane = threadIdx.x & 31;
  const int rr = lane >> 3, cc = lane & 7;  // row (of 4) and float4 column (of 8) per step
  float4* s4 = reinterpret_cast<float4*>(stage);
  for (int c0 = cofs; c0 < cofs + COLS; c0 += 32) {
    const int col0 = colbase + c0;
    if (col0 >= p.N) break;  // uniform across the warp
    float4 acc[8];
#pragma unroll
    for (int it = 0; it < 8; ++it) acc[it] = make_float4(0.f, 0.f, 0.f, 0.f);
    const float* src = tile_ws + static_cast<long long>(lrow0 + rr) * BN + c0 + 4 * cc;
    int pc = 0;
    for (; pc + 2 <= p.ksplit; pc += 2) {
      float4 x0[8], x1[8];
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        x0[it] = tc::ld_cg_f4(src + static_cast<long long>(pc) * PIECE_FLOATS + 4 * it * BN);
        x1[it] = tc::ld_cg_f4(src + static_cast<long long>(pc + 1) * PIECE_FLOATS + 4 * it * BN);
      }
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        acc[it].x += x0[it].x; acc[it].y += x0[it].y; acc[it].z += x0[it].z; acc[it].w += x0[it].w;
        acc[it].x += x1[it].x; acc[it].y += x1[it].y; acc[it].z += x1[it].z; acc[it].w += x1[it].w;
      }
    }
    for (; pc < p.ksplit; ++pc) {
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const float4 x = tc::ld_cg_f4(src + static_cast<long long>(pc) * PIECE_FLOATS + 4 * it * BN);
        acc[it].x += x.x; acc[it].y += x.y; acc[it].z += x.z; acc[it].w += x.w;
      }
    }
    // element (row 4*it + rr, columns 4*cc..) -> the swizzled slot warp_store_f32 uses
#pragma unroll
    for (int it = 0; it < 8; ++it) {
      const int r = 4 * it + rr;
      s4[r * 8 + (cc ^ (r & 7))] = acc[it];
    }
    __syncwarp();
    float v[32];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 x = s4[lane * 8 + (q ^ (lane & 7))];
      v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
    }
    __syncwarp();
    tc::epilogue_chunk(p, g, row0, col0, v, stage);
  }
}

// The operand layouts of one GEMM of a launch, as a type.
template <bool A_MN_, bool B_MN_>
struct Layout {
  static constexpr bool A_MN = A_MN_;
  static constexpr bool B_MN = B_MN_;
};

// The GEMMs of one launch. visit(u, f) calls f(params, unit of that GEMM, layout) for work unit
// u of the launch: one grouped GEMM (OneGemm), or two independent ones (TwoGemms) whose units
// follow each other in one queue, so that the second GEMM's tiles fill the pairs the first
// leaves idle and its epilogues overlap the other's main loops. Both GEMMs of a launch use the
// same producer split (split_loads).
template <bool A_MN, bool B_MN>
struct OneGemm {
  const TcParams& p;
  __device__ __forceinline__ int units() const { return p.num_units; }
  __device__ __forceinline__ int split_loads() const { return p.split_loads; }
  template <class F>
  __device__ __forceinline__ void visit(int u, F&& f) const {
    f(p, u, Layout<A_MN, B_MN>{});
  }
};

template <bool A0, bool B0, bool A1, bool B1>
struct TwoGemms {
  const tc::TcDual& d;
  __device__ __forceinline__ int units() const { return d.num_units; }
  __device__ __forceinline__ int split_loads() const { return d.q[0].split_loads; }
  template <class F>
  __device__ __forceinline__ void visit(int u, F&& f) const {
    if (u < d.units0)
      f(d.q[0], u, Layout<A0, B0>{});
    else
      f(d.q[1], u - d.units0, Layout<A1, B1>{});
  }
};

template <int EPI_W, int SUB, class Set>
__device__ __forceinline__ void pair_gemm(const Set& set) {
  using E = EpiShape<EPI_W>;
  constexpr int RB = E::RING;
  constexpr int STAGES = Ring<SUB, RB>::STAGES;
  constexpr int STAGE_BYTES = Ring<SUB, RB>::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* epi_stage = smem + RB * BLOCK_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi_stage + E::WARPS * tc::STAGE_WARP_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const uint32_t smem_base = smem_addr(smem);
  const uint32_t bar_base = smem_addr(bars);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (RB + s); };
  auto tfull_bar = [&](int a) { return bar_base + 8u * (2 * RB + a); };
  auto tempty_bar = [&](int a) { return bar_base + 8u * (2 * RB + ACC_BUFS + a); };
  const uint32_t drain_bar = bar_base + 8u * (2 * RB + 2 * ACC_BUFS);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();      // 0: leader (issues the MMAs), 1: peer
  const int cluster = static_cast<int>(cluster_id_x());
  const int nclusters = static_cast<int>(num_clusters_x());
  const int num_units = set.units();

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < ACC_BUFS; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 2 * E::WARPS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc::tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Set-up done without touching global memory; with a programmatic launch this is where the
  // previous kernel's results become visible.
  grid_dependency_wait();
  grid_dependents_launch();

  if (warp == 0 || warp == E::B_WARP) {
    // ------------------------------------------------------------ TMA producers (both CTAs)
    // Lane 0 of warp 0 loads A (and posts the leader's expect_tx), lane 0 of the last warp
    // loads B; with split_loads == 0 warp 0 loads both. Each loop is kept short: per K
    // block one try_wait, one or two TMA issues and no division (the shard map and K offset
    // advance incrementally); the abort flag is read only while a wait actually polls.
    const bool b_warp = warp == E::B_WARP;
    const bool do_a = !b_warp;
    const bool do_b = b_warp == (set.split_loads() != 0);
    if (lane == 0 && (do_a || do_b)) {
      uint32_t stage = 0, phase = 0;
      bool failed = false;
      long long issued = 0;
      const uint32_t full_leader = map_to_rank(full_bar(0), 0);   // the leader's full[0]
      for (int u = cluster; u < num_units && !failed; u += nclusters) {
        set.visit(u, [&](const auto& p, int lu, auto lay) {
          constexpr bool A_MN = decltype(lay)::A_MN;
          constexpr bool B_MN = decltype(lay)::B_MN;
          const int total_kb = p.kblocks * p.kpo;
          const int kend = p.kblocks * BK;
          int t, kb0, kb1, piece;
          tc::decode_unit(p, lu, total_kb, t, kb0, kb1, piece);
          int g, mb, nb;
          tc::decode_tile(p, t, g, mb, nb);
          const int arow = mb * BM + static_cast<int>(rank) * HALF;   // this CTA's A rows
          const int bcol = nb * BN + static_cast<int>(rank) * HALF;   // this CTA's B half
          int kg = g * p.kpo + kb0 / p.kblocks;                       // shard of block kb0
          int kk = (kb0 % p.kblocks) * BK;                            // its K offset
          bool free_next = false;  // the next stage seen free by an earlier probe
          for (int kb = kb0; kb < kb1; kb += SUB) {
            const int nsub = min(SUB, kb1 - kb);  // K blocks in this stage (fewer at a range's end)
            if (!free_next) {
              const int w = mbar_wait_or_abort(empty_bar(stage), phase ^ 1u, abort_flag, kWaitLimitNs);
              if (w <= 0) {
                if (w < 0) {
                  report_status(p.status, kDevTimeoutBase | 0x40);
                  *abort_flag = 1;
                }
                failed = true;
                break;
              }
            }
            uint32_t nstage = stage + 1, nphase = phase;
            if (nstage == STAGES) { nstage = 0; nphase ^= 1u; }
            const uint32_t fb = full_leader + 8u * stage;
            const uint32_t s0 = smem_base + stage * STAGE_BYTES;
            // probe the next stage between the last block's loads, as the MMA issuer does
            const bool probe = p.load_probe != 0 && kb + nsub < kb1;
            if (!do_a && probe) free_next = mbar_test_wait(empty_bar(nstage), nphase ^ 1u);
            if (do_a && rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2 * nsub * BLOCK_BYTES);
#pragma unroll
            for (int j = 0; j < SUB; ++j) {
              if (j < nsub) {
                const uint32_t sa = s0 + j * BLOCK_BYTES;
                const uint32_t sb = sa + A_BYTES;
                if (do_a) {
                  if (!A_MN) {
                    tma_load_2d_pair(sa, &p.tmA[kg], kk, arow, fb);
                  } else if (p.a3d) {
                    tma_load_3d_pair(sa, &p.tmA[kg], 0, kk, arow / 64, fb);
                  } else {
#pragma unroll
                    for (int c = 0; c < HALF / 64; ++c)
                      tma_load_2d_pair(sa + c * MN_BOX_BYTES, &p.tmA[kg], arow + 64 * c, kk, fb);
                  }
                }
                if (do_a && probe && j == nsub - 1)
                  free_next = mbar_test_wait(empty_bar(nstage), nphase ^ 1u);
                if (do_b) {
                  if (!B_MN) {
                    tma_load_2d_pair(sb, &p.tmB[kg], kk, bcol, fb);
                  } else if (p.b3d) {
                    tma_load_3d_pair(sb, &p.tmB[kg], 0, kk, bcol / 64, fb);
                  } else {
#pragma unroll
                    for (int c = 0; c < HALF / 64; ++c)
                      tma_load_2d_pair(sb + c * MN_BOX_BYTES, &p.tmB[kg], bcol + 64 * c, kk, fb);
                  }
                }
                kk += BK;
                if (kk == kend) { kk = 0; ++kg; }
              }
            }
            ++issued;
            stage = nstage;
            phase = nphase;
          }
        });
      }
      // another role may have given up after this thread's last wait: its copies in flight
      // are then never consumed
      if (!failed && *abort_flag) failed = true;
      if (failed && issued > 0) {
        // The copies signal the leader's barriers; give any still in flight time to land
        // before this CTA can leave.
        const uint64_t t0 = global_ns();
        while (global_ns() - t0 < 2000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------------------------------------ MMA issuer (leader)
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool failed = false;
      for (int u = cluster; u < num_units && !failed; u += nclusters) {
        set.visit(u, [&](const auto& p, int lu, auto lay) {
          constexpr bool A_MN = decltype(lay)::A_MN;
          constexpr bool B_MN = decltype(lay)::B_MN;
          constexpr uint32_t idesc = tc::idesc_bf16(BM, BN, A_MN, B_MN);
          int t, kb0, kb1, piece;
          tc::decode_unit(p, lu, p.kblocks * p.kpo, t, kb0, kb1, piece);
          const int we = mbar_wait_or_abort(tempty_bar(acc), acc_phase ^ 1u, abort_flag, kWaitLimitNs);
          if (we <= 0) {
            if (we < 0) {
              report_status(p.status, kDevTimeoutBase | 0x50);
              *abort_flag = 1;
            }
            failed = true;
            return;
          }
          tc::tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * BN;
          // `ready`: the next block's full barrier was seen complete by a probe issued before the
          // current block's last MMA (its latency then hides behind the MMA issue instead of
          // adding to the gap between blocks)
          bool ready = false;
          for (int kb = kb0; kb < kb1; kb += SUB) {
            const int nsub = min(SUB, kb1 - kb);
            if (!ready) {
              const int w = mbar_wait_or_abort(full_bar(stage), phase, abort_flag, kWaitLimitNs);
              if (w <= 0) {
                if (w < 0) {
                  report_status(p.status, kDevTimeoutBase | 0x51);
                  *abort_flag = 1;
                }
                failed = true;
                break;
              }
            }
            tc::tc_fence_after();
            uint32_t nstage = stage + 1, nphase = phase;
            if (nstage == STAGES) { nstage = 0; nphase ^= 1u; }
            const uint32_t s0 = smem_base + stage * STAGE_BYTES;
#pragma unroll
            for (int j = 0; j < SUB; ++j) {
              if (j < nsub) {
                const uint32_t sa = s0 + j * BLOCK_BYTES;
                const uint32_t sb = sa + A_BYTES;
#pragma unroll
                for (int k = 0; k < BK / 16; ++k) {
                  if (j == nsub - 1 && k == BK / 16 - 1)
                    ready = p.mma_probe != 0 && kb + nsub < kb1 &&
                            mbar_test_wait(full_bar(nstage), nphase);
                  const uint64_t ad = A_MN ? tc::sdesc_sw128(sa + k * 2048, MN_BOX_BYTES, 1024)
                                           : tc::sdesc_sw128(sa + k * 32, 16, 1024);
                  const uint64_t bd = B_MN ? tc::sdesc_sw128(sb + k * 2048, MN_BOX_BYTES, 1024)
                                           : tc::sdesc_sw128(sb + k * 32, 16, 1024);
                  umma_bf16_pair(d_tmem, ad, bd, idesc, (kb > kb0 || j > 0 || k > 0) ? 1u : 0u);
                }
              }
            }
            umma_commit_pair_multicast(empty_bar(stage), 0x3);
            stage = nstage;
            phase = nphase;
          }
          if (failed) return;
          umma_commit_pair_multicast(tfull_bar(acc), 0x3);
          if (++acc == ACC_BUFS) { acc = 0; acc_phase ^= 1u; }
        });
      }
      if (!failed && *abort_flag) failed = true;   // MMAs of a tile no epilogue will read
      if (failed) {
        umma_commit_pair_multicast(drain_bar, 0x1);
        mbar_wait_bounded(drain_bar, 0, 100000000ull);
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue warps 2..
    const int quad = warp & 3;
    const int jq = (warp - 2) >> 2;      // this warp's place among those sharing its quadrant
    const int cofs = E::cofs(jq);        // its columns of the tile: cofs .. cofs + ncols - 1
    const int ncols = E::ncols(jq);
    uint32_t acc = 0, acc_phase = 0;
    const int my_rows = static_cast<int>(rank) * HALF + quad * 32;
    // With the GeLU' epilogue, each tile's pre-activation rows are requested into L2 one unit
    // ahead (the first unit's here), while the unit before it is being finished.
    auto prefetch_unit = [&](int u) {
      set.visit(u, [&](const auto& p, int lu, auto) {
        if (!tc::dact_reads_aux(p)) return;
        int t1, a0, a1, pc1, g1, mb1, nb1;
        tc::decode_unit(p, lu, p.kblocks * p.kpo, t1, a0, a1, pc1);
        tc::decode_tile(p, t1, g1, mb1, nb1);
        tc::prefetch_aux_rows(p, g1, mb1 * BM + my_rows, nb1 * BN + cofs, ncols);
      });
    };
    if (cluster < num_units) prefetch_unit(cluster);
    bool stop = false;
    for (int u = cluster; u < num_units && !stop; u += nclusters) {
      if (u + nclusters < num_units) prefetch_unit(u + nclusters);
      set.visit(u, [&](const auto& p, int lu, auto) {
        int t, kb0, kb1, piece;
        tc::decode_unit(p, lu, p.kblocks * p.kpo, t, kb0, kb1, piece);
        int g, mb, nb;
        tc::decode_tile(p, t, g, mb, nb);
        if (!mbar_wait_bounded(tfull_bar(acc), acc_phase, kWaitLimitNs)) {
          if (lane == 0) report_status(p.status, kDevTimeoutBase | 0x60);
          *abort_flag = 1;
          stop = true;
          return;
        }
        if (*abort_flag) {
          stop = true;
          return;
        }
        tc::tc_fence_after();
        const int row0 = mb * BM + static_cast<int>(rank) * HALF + quad * 32;
        const uint32_t trow =
            tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN + static_cast<uint32_t>(cofs);
        uint8_t* stg = epi_stage + (warp - 2) * tc::STAGE_WARP_BYTES;
        if (piece < 0) {
          if constexpr (EPI_W == 12)
            tc::epilogue_rows_n(p, g, row0, nb * BN + cofs, ncols, trow, stg);
          else
            tc::epilogue_rows<E::COLS>(p, g, row0, nb * BN + cofs, trow, stg);
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(map_to_rank(tempty_bar(acc), 0));
          if (p.epi == EPI_PARTIAL_REDUCE) tc::partial_reduce_rows(p, row0, nb, E::PER_QUAD);
        } else if constexpr (EPI_W == 12) {
          // never launched with split tail tiles (their per-warp counters are laid out for 4 or
          // 8 warps): free the accumulator and report the misuse instead of summing pieces
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive_cluster(map_to_rank(tempty_bar(acc), 0));
            report_status(p.status, kDevTimeoutBase | 0x6f);
          }
        } else {
          // one piece of a split tile: park the accumulator rows, free TMEM, and finish the
          // tile's rows if this warp completes their count
          const int split_tile = t - p.full_tiles;
          float* tile_ws = p.tail_ws + static_cast<long long>(split_tile) * p.ksplit * PIECE_FLOATS;
          store_piece_rows<E::COLS>(tile_ws + static_cast<long long>(piece) * PIECE_FLOATS, my_rows,
                                    cofs, trow, stg);
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(map_to_rank(tempty_bar(acc), 0));
          int* counter = p.tail_counters + split_tile * TAIL_COUNTERS_PER_TILE +
                         static_cast<int>(rank) * 8 + (cofs / E::COLS) * 4 + quad;
          if (tail_last_arrival(counter, p.ksplit)) {
            tail_fixup_rows<E::COLS>(p, g, row0, nb * BN, tile_ws, my_rows, cofs, stg);
            if (p.epi == EPI_PARTIAL_REDUCE) tc::partial_reduce_rows(p, row0, nb, E::PER_QUAD);
            __syncwarp();
            if (lane == 0) atomicExch(counter, 0);
          }
        }
        if (++acc == ACC_BUFS) { acc = 0; acc_phase ^= 1u; }
      });
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    tc::tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

template <bool A_MN, bool B_MN, int EPI_W, int SUB>
__global__ void __launch_bounds__(EpiShape<EPI_W>::THREADS, 1)
    tc2_gemm_kernel(const __grid_constant__ TcParams p) {
  pair_gemm<EPI_W, SUB>(OneGemm<A_MN, B_MN>{p});
}

// Two GEMMs in one launch with the given operand layouts (A0/B0 of the first, A1/B1 of the
// second; true = MN-major). One K block per ring stage.
template <bool A0, bool B0, bool A1, bool B1, int EPI_W>
__global__ void __launch_bounds__(EpiShape<EPI_W>::THREADS, 1)
    tc2_dual_kernel(const __grid_constant__ tc::TcDual d) {
  pair_gemm<EPI_W, 1>(TwoGemms<A0, B0, A1, B1>{d});
}

// Launch `kern` on clusters of two CTAs; max_clusters != nullptr asks for the occupancy limit
// only.
template <int EPI_W, class Kern, class Params>
cudaError_t launch_pair_kernel(Kern kern, const Params& p, int clusters, cudaStream_t st,
                               int* max_clusters) {
  using E = EpiShape<EPI_W>;
  cudaError_t e = opt_in_dynamic_smem(reinterpret_cast<const void*>(kern), E::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(E::THREADS, 1, 1);
  cfg.dynamicSmemBytes = E::SMEM;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_clusters != nullptr) {
    cfg.gridDim = dim3(2, 1, 1);
    return cudaOccupancyMaxActiveClusters(max_clusters, kern, &cfg);
  }
  // overlap this launch's set-up with the previous kernel's end (measured on GB300: the
  // 4096 x 1024 x 4096 step 1.4 % faster, the GPT-3-shaped step unchanged); TP_TUNE_PDL = 0
  // turns it off
  if (tuning(TP_TUNE_PDL) != 0) cfg.numAttrs = 2;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <bool A_MN, bool B_MN, int EPI_W, int SUB>
cudaError_t launch_pair(const TcParams& p, int clusters, cudaStream_t st, int* max_clusters) {
  return launch_pair_kernel<EPI_W>(tc2_gemm_kernel<A_MN, B_MN, EPI_W, SUB>, p, clusters, st,
                                   max_clusters);
}

template <bool A0, bool B0, bool A1, bool B1, int EPI_W>
cudaError_t launch_dual(const tc::TcDual& d, int clusters, cudaStream_t st, int* max_clusters) {
  return launch_pair_kernel<EPI_W>(tc2_dual_kernel<A0, B0, A1, B1, EPI_W>, d, clusters, st,
                                   max_clusters);
}

// The five instantiations of one operand layout: 4 or 8 epilogue warps with 1 or 2 K blocks
// per ring stage, 12 with one.
template <bool A_MN, bool B_MN>
cudaError_t launch_pair_variant(const TcParams& p, int clusters, cudaStream_t st,
                                int* max_clusters, int epi_warps, int sub) {
  if (epi_warps == 12) return launch_pair<A_MN, B_MN, 12, 1>(p, clusters, st, max_clusters);
  if (epi_warps == 8)
    return sub == 2 ? launch_pair<A_MN, B_MN, 8, 2>(p, clusters, st, max_clusters)
                    : launch_pair<A_MN, B_MN, 8, 1>(p, clusters, st, max_clusters);
  return sub == 2 ? launch_pair<A_MN, B_MN, 4, 2>(p, clusters, st, max_clusters)
                  : launch_pair<A_MN, B_MN, 4, 1>(p, clusters, st, max_clusters);
}

}  // namespace tc2
}  // namespace tpk
