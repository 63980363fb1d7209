// The grouped bf16 GEMM on two SM pairs that share their B tiles: clusters of four CTAs.
//
// A cluster of four CTAs (ranks 0..3) computes a 512 x 256 output tile as two 256 x 256 pair
// tiles stacked in M: pair p = rank / 2 (ranks 2p, 2p + 1; the even one issues the pair's
// tcgen05.mma.cta_group::2) owns rows 256p .. 256p + 255. Both pairs need the same B tile, and
// CTA r of a pair holds B columns 128r .. 128r + 127 (its half) as in the pair kernel. The two
// CTAs holding the same half ("twins": ranks q and q ^ 2) each load one 64-column quarter of
// it with a TMA multicast to both, so every SM takes in 16 KiB of A and 8 KiB of B per K block
// instead of 16 + 16 KiB: a quarter fewer bytes from L2 for the same tensor work.
//
// Synchronisation (all mbarrier waits bounded, as in the other kernels):
//   full[s]      pair leader: its producer posts expect_tx for its own A, its peer's A (both
//                land through .cta_group::2 loads on the leader's barrier) and its own B
//                (two multicast quarters): 48 KiB; count 2 = that post + the peer's relay.
//                pair peer: its producer posts expect_tx for its own B (16 KiB); count 1.
//                The peer's warp 1 waits on it and relays an arrival to the leader's full[s],
//                so the leader's MMAs start only when all four halves of the pair are in.
//   consumed[s]  in both CTAs of a pair: the pair leader's MMA commit (multicast in the pair).
//   empty[s]     count 2: this CTA's producer arrives once its own pair has consumed the stage,
//                and its twin's producer arrives remotely once the twin's pair has. A producer
//                refills stage s (with a multicast into its twin too) only when empty[s] shows
//                both pairs done with the previous fill.
//   tfull/tempty per pair, as in the pair kernel (commit multicast within the pair; the
//                pair's 8 epilogue warps arrive on the leader's tempty).
// No instruction here multicasts across pairs except the plain (non-cta_group) TMA loads of B;
// MMA commits stay inside their pair.
#pragma once

#include "tc2_gemm.cuh"

namespace tpk {
namespace tc4 {

using tc::BK;
using tc::TcParams;
using tc2::BN;
using tc2::HALF;
using tc2::STAGES;
using tc2::ACC_BUFS;
using tc2::TMEM_COLS;
using tc2::A_BYTES;
using tc2::B_BYTES;
using tc2::STAGE_BYTES;
using tc2::MN_BOX_BYTES;
using tc2::cluster_ctarank;
using tc2::cluster_id_x;
using tc2::num_clusters_x;
using tc2::map_to_rank;
using tc2::cluster_sync_all;
using tc2::mbar_arrive_cluster;
using tc2::tma_load_2d_pair;
using tc2::tma_load_3d_pair;
using tc2::umma_bf16_pair;
using tc2::umma_commit_pair_multicast;

constexpr int BM = 512;       // rows per cluster tile (256 per pair)
constexpr int PAIR_ROWS = 256;
constexpr int QUARTER = 64;   // B columns one CTA loads per K block
constexpr int QUARTER_BYTES = QUARTER * BK * 2;  // 8 KiB
constexpr int EPI_WARPS = 4;
constexpr int NUM_THREADS = 64 + 32 * EPI_WARPS;
constexpr int NUM_BARS = 3 * STAGES + 2 * ACC_BUFS + 1;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_WARPS * tc::STAGE_WARP_BYTES + 1024 + 512;

__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const CUtensorMap* map, int x, int y,
                                               uint32_t bar, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "h"(mask)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_mc(uint32_t dst, const CUtensorMap* map, int x, int y,
                                               int z, uint32_t bar, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "h"(mask)
      : "memory");
}

// Cluster tile t -> output group g, 512-row block mb, 256-column block nb (m fastest inside an
// output, or n fastest when raster = 1).
__device__ __forceinline__ void decode_quad(const TcParams& p, int t, int& g, int& mb, int& nb) {
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

template <bool A_MN, bool B_MN>
__global__ void __launch_bounds__(NUM_THREADS, 1) tc4_gemm_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* epi_stage = smem + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi_stage + EPI_WARPS * tc::STAGE_WARP_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const uint32_t smem_base = smem_addr(smem);
  const uint32_t bar_base = smem_addr(bars);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto consumed_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
  auto empty_bar = [&](int s) { return bar_base + 8u * (2 * STAGES + s); };
  auto tfull_bar = [&](int a) { return bar_base + 8u * (3 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar_base + 8u * (3 * STAGES + ACC_BUFS + a); };
  const uint32_t drain_bar = bar_base + 8u * (3 * STAGES + 2 * ACC_BUFS);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();  // 0..3
  const uint32_t pair = rank >> 1;          // which 256-row half of the cluster tile
  const uint32_t prank = rank & 1u;         // 0: pair leader (issues the MMAs), 1: peer
  const uint32_t leader = rank & ~1u;
  const uint32_t twin = rank ^ 2u;          // holds the same B half in the other pair
  const uint16_t pair_mask = static_cast<uint16_t>(3u << (2 * pair));
  const uint16_t twin_mask = static_cast<uint16_t>((1u << rank) | (1u << twin));
  const int cluster = static_cast<int>(cluster_id_x());
  const int nclusters = static_cast<int>(num_clusters_x());

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), prank == 0 ? 2 : 1);
      mbar_init(consumed_bar(s), 1);
      mbar_init(empty_bar(s), 2);
    }
    for (int a = 0; a < ACC_BUFS; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 2 * EPI_WARPS);
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

  const int total_kb = p.kblocks * p.kpo;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer (all CTAs)
      uint32_t stage = 0, phase = 0;
      bool failed = false;
      long long issued = 0;
      long long fill = 0;  // K blocks issued so far (fill index of the ring)
      for (int t = cluster; t < p.num_tiles && !failed; t += nclusters) {
        int g, mb, nb;
        decode_quad(p, t, g, mb, nb);
        const int arow = mb * BM + static_cast<int>(pair) * PAIR_ROWS + static_cast<int>(prank) * HALF;
        const int bq = nb * BN + static_cast<int>(prank) * HALF + static_cast<int>(pair) * QUARTER;
        for (int kb = 0; kb < total_kb; ++kb, ++fill) {
          if (*abort_flag) { failed = true; break; }
          if (fill >= STAGES) {
            // the previous fill of this stage: own pair done -> tell self and twin, then wait
            // until the twin's pair is done too
            if (!mbar_wait_bounded(consumed_bar(stage), phase ^ 1u, kWaitLimitNs)) {
              report_status(p.status, kDevTimeoutBase | 0x41);
              *abort_flag = 1;
              failed = true;
              break;
            }
            mbar_arrive(empty_bar(stage));
            mbar_arrive_cluster(map_to_rank(empty_bar(stage), twin));
            if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, kWaitLimitNs)) {
              report_status(p.status, kDevTimeoutBase | 0x42);
              *abort_flag = 1;
              failed = true;
              break;
            }
          }
          const int kg = g * p.kpo + kb / p.kblocks;
          const int kk = (kb % p.kblocks) * BK;
          const uint32_t fb = map_to_rank(full_bar(stage), leader);
          const uint32_t sa = smem_base + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
          // bytes this CTA's full[s] receives: leader 2 x A + own B; peer own B
          mbar_arrive_expect_tx(full_bar(stage), prank == 0 ? 2 * A_BYTES + B_BYTES : B_BYTES);
          if (!A_MN) {
            tma_load_2d_pair(sa, &p.tmA[kg], kk, arow, fb);
          } else if (p.a3d) {
            tma_load_3d_pair(sa, &p.tmA[kg], 0, kk, arow / 64, fb);
          } else {
#pragma unroll
            for (int j = 0; j < HALF / 64; ++j)
              tma_load_2d_pair(sa + j * MN_BOX_BYTES, &p.tmA[kg], arow + 64 * j, kk, fb);
          }
          // this CTA's quarter of the B half, into the same place in itself and its twin
          const uint32_t dq = sb + pair * QUARTER_BYTES;
          if (!B_MN)
            tma_load_2d_mc(dq, &p.tmB[kg], kk, bq, full_bar(stage), twin_mask);
          else if (p.b3d)
            tma_load_3d_mc(dq, &p.tmB[kg], 0, kk, bq / 64, full_bar(stage), twin_mask);
          else
            tma_load_2d_mc(dq, &p.tmB[kg], bq, kk, full_bar(stage), twin_mask);
          ++issued;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (failed && issued > 0) {
        const uint64_t t0 = global_ns();
        while (global_ns() - t0 < 2000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && prank == 0) {
      // ------------------------------------------------------------ MMA issuer (pair leaders)
      constexpr uint32_t idesc = tc::idesc_bf16(PAIR_ROWS, BN, A_MN, B_MN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool failed = false;
      for (int t = cluster; t < p.num_tiles && !failed; t += nclusters) {
        if (!mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u, kWaitLimitNs)) {
          report_status(p.status, kDevTimeoutBase | 0x52);
          *abort_flag = 1;
          failed = true;
          break;
        }
        tc::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < total_kb; ++kb) {
          if (*abort_flag) { failed = true; break; }
          if (!mbar_wait_bounded(full_bar(stage), phase, kWaitLimitNs)) {
            report_status(p.status, kDevTimeoutBase | 0x53);
            *abort_flag = 1;
            failed = true;
            break;
          }
          tc::tc_fence_after();
          const uint32_t sa = smem_base + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = A_MN ? tc::sdesc_sw128(sa + k * 2048, MN_BOX_BYTES, 1024)
                                     : tc::sdesc_sw128(sa + k * 32, 16, 1024);
            const uint64_t bd = B_MN ? tc::sdesc_sw128(sb + k * 2048, MN_BOX_BYTES, 1024)
                                     : tc::sdesc_sw128(sb + k * 32, 16, 1024);
            umma_bf16_pair(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit_pair_multicast(consumed_bar(stage), pair_mask);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (failed) break;
        umma_commit_pair_multicast(tfull_bar(acc), pair_mask);
        if (++acc == ACC_BUFS) { acc = 0; acc_phase ^= 1u; }
      }
      if (failed) {
        umma_commit_pair_multicast(drain_bar, static_cast<uint16_t>(1u << rank));
        mbar_wait_bounded(drain_bar, 0, 100000000ull);
      }
    } else if (lane == 0) {
      // ------------------------------------------------------------ relay (pair peers)
      // The peer's B lands on its own full[s]; pass each completed fill on to the leader.
      uint32_t stage = 0, phase = 0;
      bool failed = false;
      for (int t = cluster; t < p.num_tiles && !failed; t += nclusters) {
        for (int kb = 0; kb < total_kb; ++kb) {
          if (*abort_flag) { failed = true; break; }
          if (!mbar_wait_bounded(full_bar(stage), phase, kWaitLimitNs)) {
            report_status(p.status, kDevTimeoutBase | 0x54);
            *abort_flag = 1;
            failed = true;
            break;
          }
          mbar_arrive_cluster(map_to_rank(full_bar(stage), leader));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue warps 2..5
    const int quad = warp & 3;
    uint32_t acc = 0, acc_phase = 0;
    const int my_rows = static_cast<int>(pair) * PAIR_ROWS + static_cast<int>(prank) * HALF + quad * 32;
    const bool aux_ahead = tc::dact_reads_aux(p);
    if (aux_ahead && cluster < p.num_tiles) {
      int g1, mb1, nb1;
      decode_quad(p, cluster, g1, mb1, nb1);
      tc::prefetch_aux_rows(p, g1, mb1 * BM + my_rows, nb1 * BN, BN);
    }
    for (int t = cluster; t < p.num_tiles; t += nclusters) {
      int g, mb, nb;
      decode_quad(p, t, g, mb, nb);
      if (aux_ahead && t + nclusters < p.num_tiles) {
        int g1, mb1, nb1;
        decode_quad(p, t + nclusters, g1, mb1, nb1);
        tc::prefetch_aux_rows(p, g1, mb1 * BM + my_rows, nb1 * BN, BN);
      }
      if (!mbar_wait_bounded(tfull_bar(acc), acc_phase, kWaitLimitNs)) {
        if (lane == 0) report_status(p.status, kDevTimeoutBase | 0x61);
        *abort_flag = 1;
        break;
      }
      if (*abort_flag) break;
      tc::tc_fence_after();
      const int row0 = mb * BM + my_rows;
      const uint32_t trow = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN;
      uint8_t* stg = epi_stage + (warp - 2) * tc::STAGE_WARP_BYTES;
      tc::epilogue_rows<BN>(p, g, row0, nb * BN, trow, stg);
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_to_rank(tempty_bar(acc), leader));
      if (++acc == ACC_BUFS) { acc = 0; acc_phase ^= 1u; }
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

// Launch on clusters of four CTAs; max_clusters != nullptr asks for the occupancy limit only.
template <bool A_MN, bool B_MN>
cudaError_t launch_quad(const TcParams& p, int clusters, cudaStream_t st, int* max_clusters) {
  auto kern = tc4_gemm_kernel<A_MN, B_MN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 4;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_clusters != nullptr) {
    cfg.gridDim = dim3(4, 1, 1);
    return cudaOccupancyMaxActiveClusters(max_clusters, kern, &cfg);
  }
  cfg.gridDim = dim3(4 * clusters, 1, 1);
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace tc4
}  // namespace tpk
