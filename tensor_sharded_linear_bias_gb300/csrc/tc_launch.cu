// Host side of the tcgen05 GEMM: TMA descriptor encoding, tile counts, grid sizing.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "tc2_gemm.cuh"

namespace tpk {
namespace tc {
cudaError_t run_kmn(const TcParams& p, int grid, cudaStream_t st);
cudaError_t run_kk(const TcParams& p, int grid, cudaStream_t st);
cudaError_t run_mnmn(const TcParams& p, int grid, cudaStream_t st);
cudaError_t run_pair_kmn(const TcParams& p, int clusters, cudaStream_t st, int* max_clusters,
                         int epi_warps, int sub);
cudaError_t run_pair_kk(const TcParams& p, int clusters, cudaStream_t st, int* max_clusters,
                        int epi_warps, int sub);
cudaError_t run_pair_mnmn(const TcParams& p, int clusters, cudaStream_t st, int* max_clusters,
                          int epi_warps, int sub);
cudaError_t run_pair_dual(const TcDual& d, int clusters, cudaStream_t st, int* max_clusters,
                          int epi_warps);
}  // namespace tc

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// Tensor maps are encoded on the host for every launch; a launch of a few microseconds (few
// tokens) would otherwise wait for its encodes (~1 us each). So each thread keeps the maps it
// made, keyed by everything that goes into them (a map holds only the address, shape, strides,
// box and modes, so a hit is exactly the map a new encode would give), in a small
// direct-mapped table.
struct MapKey {
  const void* ptr;
  cuuint64_t dims[3];
  cuuint64_t strides[2];
  cuuint32_t box[3];
  uint32_t rank;
  int dtype, swizzle;
  bool operator==(const MapKey& o) const { return std::memcmp(this, &o, sizeof(MapKey)) == 0; }
};

bool encode_cached(CUtensorMap* m, CUtensorMapDataType dtype, uint32_t rank, const void* ptr,
                   const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                   CUtensorMapSwizzle swizzle) {
  MapKey k;
  std::memset(&k, 0, sizeof(k));  // padding too: keys compare byte for byte
  k.ptr = ptr;
  for (uint32_t i = 0; i < rank; ++i) {
    k.dims[i] = dims[i];
    k.box[i] = box[i];
    if (i + 1 < rank) k.strides[i] = strides[i];
  }
  k.rank = rank;
  k.dtype = static_cast<int>(dtype);
  k.swizzle = static_cast<int>(swizzle);
  uint64_t h = 1469598103934665603ull;  // FNV-1a over the key's bytes
  const unsigned char* b = reinterpret_cast<const unsigned char*>(&k);
  for (size_t i = 0; i < sizeof(k); ++i) h = (h ^ b[i]) * 1099511628211ull;
  struct Entry {
    bool valid = false;
    MapKey key;
    CUtensorMap map;
  };
  static thread_local Entry table[256];
  Entry& e = table[h & 255u];
  if (e.valid && e.key == k) {
    *m = e.map;
    return true;
  }
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  if (fn(m, dtype, rank, const_cast<void*>(ptr), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  e.valid = true;
  e.key = k;
  e.map = *m;
  return true;
}

// 2-D bf16 row-major tensor [outer][inner] with row pitch ld (elements), 128B swizzle.
bool encode_bf16(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint64_t ld,
                 uint32_t box_inner, uint32_t box_outer) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {ld * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  return encode_cached(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_128B);
}

// The SM-pair kernel computes 256-row tiles; below that the one-SM kernel's 128-row tiles
// waste less. TP_TUNE_GEMM_PAIR forces the choice (tests and A/B timing).
bool use_pair_kernel(int64_t M) {
  if (const int v = tuning(TP_TUNE_GEMM_PAIR); v != TP_TUNE_AUTO) return v != 0;
  return M > tc::BM;
}

cudaError_t run_pair(int layout, const tc::TcParams& p, int clusters, cudaStream_t st,
                     int* max_clusters, int epi_warps, int sub = 1) {
  if (layout == 0) return tc::run_pair_kmn(p, clusters, st, max_clusters, epi_warps, sub);
  if (layout == 1) return tc::run_pair_kk(p, clusters, st, max_clusters, epi_warps, sub);
  return tc::run_pair_mnmn(p, clusters, st, max_clusters, epi_warps, sub);
}

// K blocks per ring stage of the pair kernel (tc2::Ring). The single MMA-issuing thread needs
// ~360 cycles to issue the four MMAs of a 64-deep block (~85 each, measured with cycle counters in
// an instrumented copy) plus ~150 for the block's barrier look-ahead, wait and commit: about as
// long as the 512 cycles the tensor pipe takes for the block, so the pipe idled ~15 %. Two blocks
// per stage pay the barrier work once per 128; the coarser release (a stage is refilled only when
// both blocks are consumed) costs more on short tiles. Measured on GB300, same box, alternating
// (stage of 2 vs 1): GPT-3-shaped step 8.92-8.94 vs 9.18-9.33 ms (its forward and input-gradient
// GEMMs 4-7 % faster, its weight gradients of 32 blocks 2 % slower); sweep T 16384 28.6 vs 30.0
// ms (weight gradients of 256 blocks faster too); 4096 x 1024 x 4096 step slightly slower (tiles
// of 16 blocks). So: 2 for tiles of at least 64 blocks (128 with both operands MN-major), else 1.
// TP_TUNE_STAGE_BLOCKS overrides.
int pair_sub_blocks(int layout, int total_kb) {
  if (const int v = tuning(TP_TUNE_STAGE_BLOCKS); v != TP_TUNE_AUTO) return v == 2 ? 2 : 1;
  return total_kb >= (layout == 2 ? 128 : 64) ? 2 : 1;
}

// Largest number of co-resident 2-CTA clusters of the pair kernel (cached per device, operand
// layout and epilogue warp count); falls back to half the SM count.
int pair_clusters(int layout, int epi_warps = 4) {
  static int cached[64][3][3] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return device_sm_count() / 2;
  const int v = epi_warps == 12 ? 2 : epi_warps == 8 ? 1 : 0;
  if (cached[dev][layout][v] == 0) {
    int n = 0;
    cudaError_t e = run_pair(layout, tc::TcParams{}, 0, nullptr, &n, epi_warps);
    if (e != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = device_sm_count() / 2;
    }
    cached[dev][layout][v] = n;
  }
  return cached[dev][layout][v];
}

// Epilogue warps of the pair kernel: 8 where 4 warps' epilogue of a tile would outlast the next
// tile's main loop: GeLU or GeLU' tiles with at most 64 K blocks of 64, any tile with at most
// 16; else 4, which is faster for deep tiles (measured on GB300, same box: the GPT-3-shaped
// step 1494 vs 1484 TFLOP/s with 4; the 4096 x 1024 x 4096 step 753 vs 710 with 8 on its
// GeLU / GeLU' GEMMs; weight gradients over 512 tokens 0.253 vs 0.265 ms with 8). The launch
// may raise 8 to 12 for GeLU / GeLU' tiles (see launch_tc_gemm). TP_TUNE_EPI_WARPS forces the
// count (4, 8 or 12).
int pair_epi_warps(int epi, int act, int total_kb) {
  if (const int v = tuning(TP_TUNE_EPI_WARPS); v != TP_TUNE_AUTO) return v == 12 ? 12 : v == 8 ? 8 : 4;
  const bool heavy = (epi == EPI_BIAS_ACT || epi == EPI_DACT) && act == TP_ACT_GELU_ERF;
  return (heavy && total_kb <= 64) || total_kb <= 16 ? 8 : 4;
}

// Tile order of a launch (inside each output; m fastest or n fastest). Two estimates:
//  1. Working set in flight: the tiles running at the same time (one per SM, or per SM pair)
//     touch, in m-fastest order, all tiles_m row blocks of A plus C / tiles_m column blocks of
//     B (C = tiles in flight); in n-fastest order, the converse. Each block is 256 x K bf16
//     (128 x K for one-SM A blocks). m fastest unless its working set exceeds half of L2 and n
//     fastest needs a quarter less. (Measured on GB300: m fastest is 5 % faster for the
//     GPT-3-shaped MLP's forward and input-gradient GEMMs, n fastest 1.5 % faster at 8192
//     tokens.)
//  2. DRAM reads per output: the blocks of the slow axis are read once; the set of fast-axis
//     blocks is read once if it fits in a share of L2 (kRasterL2Budget, leaving room for the
//     streamed operand and the outputs), else once per wave that cycles through it. Where one
//     order reads less than half of the other, that order wins over estimate 1. (The GPT-3
//     column weight gradient: m fastest cycles 48 MB of X per column of dH_i and its 2.4 GB of
//     fp32 output evicted X in between -- ncu read 2.16 GB for 0.25 GB of operands; n fastest
//     keeps the shard's 24 MB of dH_i resident.)
// TP_TUNE_RASTER forces the order.
constexpr double kRasterL2Budget = 40.0e6;

double raster_reads(double n_fast, double fast_block, double n_slow, double slow_block,
                    double inflight) {
  const double fast_set = n_fast * fast_block;
  const double cycles = fast_set <= kRasterL2Budget
                            ? 1.0
                            : std::max(1.0, n_slow * std::min(1.0, n_fast / inflight));
  return n_slow * slow_block + fast_set * cycles;
}

int choose_raster(int tiles_m, int tiles_n, int64_t k_total, int sms, bool pair) {
  if (const int v = tuning(TP_TUNE_RASTER); v != TP_TUNE_AUTO) return v != 0;
  const double inflight = pair ? sms / 2.0 : double(sms);
  const double a_block = (pair ? 256.0 : 128.0) * double(k_total) * 2.0;
  const double b_block = 256.0 * double(k_total) * 2.0;
  const double reads_m = raster_reads(tiles_m, a_block, tiles_n, b_block, inflight);
  const double reads_n = raster_reads(tiles_n, b_block, tiles_m, a_block, inflight);
  if (reads_n < 0.5 * reads_m) return 1;
  if (reads_m < 0.5 * reads_n) return 0;
  const double fm = std::min<double>(tiles_m, inflight) * a_block +
                    std::ceil(inflight / std::max(1, tiles_m)) * b_block;
  const double fn = std::min<double>(tiles_n, inflight) * b_block +
                    std::ceil(inflight / std::max(1, tiles_n)) * a_block;
  const double half_l2 = 64.0e6;
  return (fm > half_l2 && fn < 0.75 * fm) ? 1 : 0;
}

// 3-D view of an MN-major bf16 operand [K][MN] (row pitch ld): dims {64, K, MN/64}, strides
// {ld * 2, 128} bytes, box {64, 64, chunks}. One load then brings `chunks` 64-wide MN chunks
// of 64 K rows, laid out in shared memory like `chunks` 2-D boxes. Only for MN % 64 == 0 (a
// partial last chunk would read past the rows). Returns false if the driver refuses it.
bool encode_bf16_mn3d(CUtensorMap* m, const void* ptr, uint64_t mn, uint64_t k, uint64_t ld,
                      uint32_t chunks) {
  if (mn % 64 != 0) return false;
  const cuuint64_t dims[3] = {64, k, mn / 64};
  const cuuint64_t strides[2] = {ld * 2, 128};
  const cuuint32_t box[3] = {64, 64, chunks};
  return encode_cached(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_128B);
}

// One-load MN-major tiles (3-D maps); TP_TUNE_TMA_3D = 0 keeps the 2-D boxes.
bool mn3d_enabled() {
  if (const int v = tuning(TP_TUNE_TMA_3D); v != TP_TUNE_AUTO) return v != 0;
  return true;
}

// A and B loads of the SM-pair kernel from two producer threads: where both operands are
// MN-major (weight gradients), whose two 3-D boxes per K block make the longest issue loop
// (measured 1-2 % faster there, 0.5-1 % slower for the other layouts); TP_TUNE_SPLIT_LOADS
// overrides.
bool split_loads_enabled(int layout) {
  if (const int v = tuning(TP_TUNE_SPLIT_LOADS); v != TP_TUNE_AUTO) return v != 0;
  return layout == 2;
}

// The MMA issuer's early look at the next block's barrier; TP_TUNE_MMA_PROBE overrides.
bool mma_probe_enabled() {
  if (const int v = tuning(TP_TUNE_MMA_PROBE); v != TP_TUNE_AUTO) return v != 0;
  return true;
}

// The producers' early look at the next block's stage: for A K-major with B MN-major (the
// forward GEMMs: 4-5 % faster), not for the other layouts (both K-major: 0.5-2 % slower, both
// MN-major: no change); TP_TUNE_LOAD_PROBE overrides.
bool load_probe_enabled(int layout) {
  if (const int v = tuning(TP_TUNE_LOAD_PROBE); v != TP_TUNE_AUTO) return v != 0;
  return layout == 0;
}

// Split tail; TP_TUNE_TAIL_SPLIT = 0 turns it off.
bool tail_split_enabled() {
  if (const int v = tuning(TP_TUNE_TAIL_SPLIT); v != TP_TUNE_AUTO) return v != 0;
  return true;
}

constexpr int kMinPieceKb = 16;  // K blocks of 64 a piece keeps at least
// Shallow tiles are split only when there are at most this many waves (in a deeper queue of
// short tiles the partly idle last wave matters less than the pieces' round trip: the GPT-3
// weight gradients, 121 waves of 32 K blocks, were 1 % slower split); tiles of at least
// kDeepTileKb K blocks are split at any number of waves (the GPT-3 column forward and dY GEMMs,
// 20 waves of 192 K blocks: 0.6-1.3 % faster; T 8192: 1-3 %).
constexpr int kMaxSplitWaves = 8;
constexpr int kDeepTileKb = 64;

// Work units of an SM-pair launch over `clusters` pairs. Tiles are dealt to the pairs round
// robin, so the last wave holds L = num_tiles mod clusters tiles (all of them when there are
// fewer tiles than pairs) and leaves the other pairs idle for a whole tile. Each of those L
// tiles is cut into S = clusters / L pieces of consecutive K blocks (capped by kMinPieceKb and
// the kTailUnits pieces the workspace holds), which run side by side on the idle pairs: the
// last wave takes about 1/S of a tile's time, plus the pieces' fp32 round trip through L2.
// Pieces per split tile. The last wave takes about (tile time) / P for the pieces, plus the sum of
// the P parked accumulators by the warp that completes a tile's count: it reads them from L2 two
// at a time, 8 chunks of 32 columns each, ~3 us per piece (per-CTA timestamps on GB300: 19 pieces
// of a 768-block tile ended 52-66 us after the other CTAs, 4 pieces of a 192-block tile ~30 us).
// The sum tile/P + 3 P is smallest near P = sqrt(tile / 3 us), a 64-deep block taking ~0.28 us:
// ~8 pieces for 768 blocks, ~4 for 192. TP_TUNE_TAIL_PIECES overrides the cap.
int tail_pieces_cap(int total_kb) {
  if (const int v = tuning(TP_TUNE_TAIL_PIECES); v != TP_TUNE_AUTO) return std::max(1, v);
  const double tile_us = total_kb * 0.28;
  return std::max(2, static_cast<int>(std::lround(std::sqrt(tile_us / 3.0))));
}

void plan_tail(tc::TcParams& p, int clusters, int total_kb, bool have_ws) {
  p.full_tiles = p.num_tiles;
  p.ksplit = 1;
  p.num_units = p.num_tiles;
  if (!have_ws || !tail_split_enabled() || clusters < 2) return;
  int max_waves = total_kb >= kDeepTileKb ? 1 << 20 : kMaxSplitWaves;
  if (const int v = tuning(TP_TUNE_TAIL_WAVES); v != TP_TUNE_AUTO) max_waves = v;
  if (p.num_tiles > static_cast<long long>(max_waves) * clusters) return;
  const int L = p.num_tiles % clusters;
  if (L == 0) return;
  int S = clusters / L;
  S = std::min(S, total_kb / kMinPieceKb);
  S = std::min(S, kTailUnits / L);
  S = std::min(S, tail_pieces_cap(total_kb));
  if (S < 2) return;
  p.full_tiles = p.num_tiles - L;
  p.ksplit = S;
  p.num_units = p.full_tiles + L * S;
}

}  // namespace

cudaError_t opt_in_dynamic_smem(const void* kern, int bytes) {
  struct Entry {
    const void* kern;
    int dev, bytes;
  };
  static std::mutex mu;
  static Entry done[256];
  static int n_done = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_done; ++i)
      if (done[i].kern == kern && done[i].dev == dev && done[i].bytes >= bytes) return cudaSuccess;
  }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (n_done < 256) done[n_done++] = {kern, dev, bytes};
  return cudaSuccess;
}

// 2-D fp32 row-major tensor [outer][inner] with row pitch ld (elements), no swizzle: a box
// lands in shared memory as box_outer rows of box_inner consecutive floats; elements outside
// the tensor read as zeros.
bool encode_f32_rows(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint64_t ld,
                     uint32_t box_inner, uint32_t box_outer) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {ld * 4};
  const cuuint32_t box[2] = {box_inner, box_outer};
  return encode_cached(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_NONE);
}


int plan_shard_split(int64_t M, int64_t N, int64_t K_per_group, int n) {
  using namespace tc;
  if (const int v = tuning(TP_TUNE_SHARD_SPLIT); v != TP_TUNE_AUTO) {
    if (v >= 1 && v <= n && n % v == 0) return v;
  }
  // Model on SM pairs (the kernel for every M > 128): 256 x 256 tiles dealt to C = SMs / 2
  // pairs; a 64-deep K block of a pair tile costs ~512 tensor cycles (~0.27 us). A last wave
  // that leaves pairs idle costs a whole tile, unless the tail split applies (at most 8 waves
  // or tiles of >= 64 K blocks; >= 32 K blocks per tile), which cuts its L tiles into P pieces
  // (~1/P of a tile, plus a
  // little for the piece sums). A reduction of S fp32 partials moves (4 S + 4) M N bytes at
  // ~6.5 TB/s. (Measured on GB300, GPT-3-shaped step: fused 1525-1528 TFLOP/s with the tail
  // split vs 1499-1506 for S = 4 and 1499 fused without it.)
  const double C = std::max(1, device_sm_count() / 2);
  const double tiles1 = double((M + 255) / 256) * double((N + BN - 1) / BN);
  const double kb = double((K_per_group + BK - 1) / BK);
  const double t_kb_us = 512.0 / 1.9e3;
  const double hbm_bytes_per_us = 6.5e6;
  int best = 1;
  double best_cost = 1e300;
  for (int S = 1; S <= n; ++S) {
    if (n % S != 0) continue;
    const double per_tile_kb = kb * (n / S);
    const double tiles = S * tiles1;
    double waves = std::ceil(tiles / C);
    const double L = tiles - C * std::floor(tiles / C);
    if (L > 0 && (tiles <= kMaxSplitWaves * C || per_tile_kb >= kDeepTileKb) &&
        tail_split_enabled()) {
      const double P = std::min({std::floor(C / L), std::floor(per_tile_kb / kMinPieceKb),
                                 std::floor(kTailUnits / L),
                                 double(tail_pieces_cap(static_cast<int>(per_tile_kb)))});
      if (P >= 2) waves = std::floor(tiles / C) + 1.0 / P + 0.05;
    }
    double cost = waves * per_tile_kb * t_kb_us;
    if (S > 1) cost += (4.0 * S + 4.0) * double(M) * double(N) / hbm_bytes_per_us;
    if (cost < best_cost * 0.995) {
      best_cost = cost;
      best = S;
    }
  }
  return best;
}

namespace {

// The kernel parameters of GEMM s (tensor maps, outputs, tile counts, tile order), for the
// SM-pair kernel (pair) or the one-SM kernel; *layout = 0 (A K-major, B MN-major), 1 (both
// K-major) or 2 (both MN-major). p holds at least s.groups groups (checked by the caller).
template <class P>
cudaError_t fill_tc_params(P& p, const GemmSpec& s, bool pair, int* layout) {
  using namespace tc;
  std::memset(static_cast<void*>(&p), 0, sizeof(p));
  // K-major boxes: 128 rows of A; 256 rows of B (one SM) or 128 (each SM of a pair).
  const uint32_t b_rows = pair ? static_cast<uint32_t>(tc2::HALF) : static_cast<uint32_t>(BN);
  // MN chunks per CTA tile: A 128 rows (one SM or each SM of a pair); B 256 or 128 columns.
  const uint32_t a_chunks = 2;
  const uint32_t b_chunks = pair ? 2 : 4;
  p.a3d = s.a_mn && mn3d_enabled() && s.M % 64 == 0;
  p.b3d = s.b_mn && mn3d_enabled() && s.N % 64 == 0;
  for (int g = 0; g < s.groups && p.a3d; ++g)
    p.a3d = encode_bf16_mn3d(&p.tmA[g], s.A[g], s.M, s.K, s.lda, a_chunks);
  for (int g = 0; g < s.groups && p.b3d; ++g)
    p.b3d = encode_bf16_mn3d(&p.tmB[g], s.B[g], s.N, s.K, s.ldb, b_chunks);
  for (int g = 0; g < s.groups; ++g) {
    const bool okA = p.a3d ? true
                     : s.a_mn ? encode_bf16(&p.tmA[g], s.A[g], s.M, s.K, s.lda, 64, 64)
                              : encode_bf16(&p.tmA[g], s.A[g], s.K, s.M, s.lda, 64, BM);
    const bool okB = p.b3d ? true
                     : s.b_mn ? encode_bf16(&p.tmB[g], s.B[g], s.N, s.K, s.ldb, 64, 64)
                              : encode_bf16(&p.tmB[g], s.B[g], s.K, s.N, s.ldb, 64, b_rows);
    if (!okA || !okB) return cudaErrorInvalidValue;
    p.D[g] = s.D[g];
    p.D2[g] = s.D2[g];
    p.bias[g] = s.bias[g];
    p.aux[g] = s.aux[g];
  }
  p.ldd = s.ldd;
  p.ldd2 = s.ldd2;
  p.ldaux = s.ldaux;
  p.M = static_cast<int>(s.M);
  p.N = static_cast<int>(s.N);
  p.kblocks = static_cast<int>((s.K + BK - 1) / BK);
  p.groups = s.groups;
  const int kpo = s.kpo > 0 ? s.kpo : (s.ksum ? s.groups : 1);
  if (s.groups % kpo != 0) return cudaErrorInvalidValue;
  p.kpo = kpo;
  const int tile_rows = pair ? tc2::BM : BM;
  p.tiles_m = static_cast<int>((s.M + tile_rows - 1) / tile_rows);
  p.tiles_n = static_cast<int>((s.N + BN - 1) / BN);
  p.num_tiles = (s.groups / kpo) * p.tiles_m * p.tiles_n;
  p.tiles_n_out = p.tiles_n;
  p.counters = s.counters;
  p.Z = s.Z;
  p.ldz = s.ldz;
  p.zbias = s.zbias;
  p.nsplit = s.groups / kpo;
  p.epi = s.epi;
  p.act = s.act;
  p.raster = choose_raster(p.tiles_m, p.tiles_n, s.K * p.kpo,
                           pair ? 2 * pair_clusters(0) : device_sm_count(), pair);
  p.status = s.status;
  *layout = (!s.a_mn && s.b_mn) ? 0 : (!s.a_mn && !s.b_mn) ? 1 : (s.a_mn && s.b_mn) ? 2 : -1;
  if (*layout < 0) return cudaErrorNotSupported;
  p.full_tiles = p.num_tiles;
  p.ksplit = 1;
  p.num_units = p.num_tiles;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_tc_gemm(const GemmSpec& s, cudaStream_t st) {
  using namespace tc;
  if (s.M <= 0 || s.N <= 0 || s.K <= 0) return cudaSuccess;
  if (s.groups < 1 || s.groups > kMaxShards) return cudaErrorInvalidValue;
  static_assert(sizeof(TcParams) <= 32764, "kernel parameter block too large");

  const bool pair = use_pair_kernel(s.M);
  alignas(128) static thread_local TcParams p;
  int layout = -1;
  if (const cudaError_t e = fill_tc_params(p, s, pair, &layout); e != cudaSuccess) return e;
  if (pair) {
    int epi_warps = pair_epi_warps(p.epi, p.act, p.kblocks * p.kpo);
    int max_clusters = pair_clusters(layout, epi_warps);
    // 12 epilogue warps take whole tiles only (no split tail pieces)
    plan_tail(p, max_clusters, p.kblocks * p.kpo,
              epi_warps != 12 && s.tail_ws != nullptr && s.tail_counters != nullptr);
    // 8 epilogue warps also where the epilogue work is exposed at the end of the launch: split
    // tail tiles, whose pieces the completing warps sum (with 8 warps each sums half as many
    // columns), and launches of at most one tile per pair (no next tile hides the epilogue).
    // Measured on GB300, same box: the GPT-3-shaped forward and input-gradient GEMMs 1-2 %
    // faster, the 4096 x 1024 x 4096 step 0.2317 vs 0.2346 ms.
    if (epi_warps == 4 && tuning(TP_TUNE_EPI_WARPS) == TP_TUNE_AUTO &&
        (p.ksplit > 1 || p.num_units <= max_clusters)) {
      epi_warps = 8;
      max_clusters = pair_clusters(layout, epi_warps);
      if (p.ksplit > 1 && max_clusters != pair_clusters(layout, 4))
        plan_tail(p, max_clusters, p.kblocks * p.kpo, true);
    }
    // 12 epilogue warps for the GeLU / GeLU' tiles that 8 serve (short K) when the launch has
    // no split tail tiles, and for launches of at most one tile per pair (whose one epilogue is
    // all exposed). Measured on GB300, same box, 4096 x 1024 x 4096 step: the GeLU / GeLU' GEMMs
    // 3-4 % faster (column forward 46.7 vs 48.2 us, dY 50.1 vs 52.1), the step 1 % faster; its
    // row GEMM (64 tiles of 64 K blocks) 33.8 vs 35.0 us. Forced on every GEMM of many tiles,
    // the weight gradients and the input gradient were slower.
    const bool one_tile_each = p.num_units <= pair_clusters(layout, 12);
    if (epi_warps == 8 && p.ksplit == 1 && tuning(TP_TUNE_EPI_WARPS) == TP_TUNE_AUTO &&
        (((p.epi == EPI_BIAS_ACT || p.epi == EPI_DACT) && p.act == TP_ACT_GELU_ERF &&
          p.kblocks * p.kpo <= 64) ||
         one_tile_each)) {
      epi_warps = 12;
      max_clusters = std::min(max_clusters, pair_clusters(layout, epi_warps));
    }
    if (p.ksplit > 1) {
      p.tail_ws = s.tail_ws;
      p.tail_counters = s.tail_counters;
      const size_t counters =
          size_t(p.num_tiles - p.full_tiles) * tc2::TAIL_COUNTERS_PER_TILE * sizeof(int);
      if (counters > kTailCounterBytes) return cudaErrorInvalidValue;
      cudaError_t e = cudaMemsetAsync(s.tail_counters, 0, counters, st);
      if (e != cudaSuccess) return e;
    }
    p.split_loads = split_loads_enabled(layout) ? 1 : 0;
    p.mma_probe = mma_probe_enabled() ? 1 : 0;
    p.load_probe = load_probe_enabled(layout) ? 1 : 0;
    const int clusters = std::min(p.num_units, max_clusters);
    return run_pair(layout, p, clusters, st, nullptr, epi_warps,
                    epi_warps == 12 ? 1 : pair_sub_blocks(layout, p.kblocks * p.kpo));
  }
  const int grid = std::min(p.num_tiles, device_sm_count());
  if (!s.a_mn && s.b_mn) return run_kmn(p, grid, st);
  if (!s.a_mn && !s.b_mn) return run_kk(p, grid, st);
  if (s.a_mn && s.b_mn) return run_mnmn(p, grid, st);
  return cudaErrorNotSupported;
}


// ---------------------------------------------------------------- two GEMMs in one launch
namespace {

// Largest number of co-resident 2-CTA clusters of the two-GEMM kernel (cached per device and
// epilogue warp count); falls back to half the SM count.
int dual_clusters(int epi_warps) {
  static int cached[64][2] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return device_sm_count() / 2;
  const int v = epi_warps == 12 ? 1 : 0;
  if (cached[dev][v] == 0) {
    alignas(128) static tc::TcDual probe;  // only the kernel's resources matter here
    int n = 0;
    cudaError_t e = tc::run_pair_dual(probe, 0, nullptr, &n, epi_warps);
    if (e != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = device_sm_count() / 2;
    }
    cached[dev][v] = n;
  }
  return cached[dev][v];
}

int64_t pair_tiles(const GemmSpec& s) {
  const int kpo = s.kpo > 0 ? s.kpo : (s.ksum ? s.groups : 1);
  return int64_t(s.groups / std::max(1, kpo)) * ((s.M + tc2::BM - 1) / tc2::BM) *
         ((s.N + tc2::BN - 1) / tc2::BN);
}

// A shared launch pays off where a GEMM alone leaves pairs idle: one of the two has at most
// one wave of tiles (its launch ramp, its partly idle wave and its last, exposed epilogue are
// then a large part of its time), and together they make few waves (with many waves there is
// nothing to fill, and the one-GEMM launch keeps its split tail tiles).
constexpr int kDualMaxWaves = 8;

}  // namespace

bool tc_dual_eligible(const GemmSpec& s0, const GemmSpec& s1) {
  const int v = tuning(TP_TUNE_DUAL);
  if (v == 0) return false;
  const auto fits = [](const GemmSpec& s) {
    const int kpo = s.kpo > 0 ? s.kpo : (s.ksum ? s.groups : 1);
    return s.M > 0 && s.N > 0 && s.K > 0 && s.groups >= 1 && s.groups <= tc::kDualMaxShards &&
           s.groups % kpo == 0 && use_pair_kernel(s.M) && s.epi != EPI_PARTIAL_REDUCE;
  };
  if (!(s0.a_mn && s0.b_mn && !s1.a_mn && !s1.b_mn && fits(s0) && fits(s1))) return false;
  if (v != TP_TUNE_AUTO) return true;
  const int64_t C = std::max(1, device_sm_count() / 2);
  const int64_t t0 = pair_tiles(s0), t1 = pair_tiles(s1);
  return std::min(t0, t1) <= C && t0 + t1 <= kDualMaxWaves * C;
}

cudaError_t launch_tc_gemm_dual(const GemmSpec& s0, const GemmSpec& s1, cudaStream_t st) {
  using namespace tc;
  static_assert(sizeof(TcDual) <= 32764, "kernel parameter block too large");
  alignas(128) static thread_local TcDual d;
  int l0 = -1, l1 = -1;
  if (const cudaError_t e = fill_tc_params(d.q[0], s0, true, &l0); e != cudaSuccess) return e;
  if (const cudaError_t e = fill_tc_params(d.q[1], s1, true, &l1); e != cudaSuccess) return e;
  if (l0 != 2 || l1 != 1) return cudaErrorNotSupported;
  // 12 epilogue warps: GeLU' tiles of few K blocks are paced by their epilogues, and the last
  // tiles' epilogues are exposed (measured on GB300, 4096 x 1024 x 4096 step: 0.2065 vs
  // 0.2131 ms with 8). Both GEMMs load A and B from two producer threads.
  const int epi_warps = tuning(TP_TUNE_EPI_WARPS) == 8 ? 8 : 12;
  for (int i = 0; i < 2; ++i) {
    d.q[i].split_loads = 1;
    d.q[i].mma_probe = mma_probe_enabled() ? 1 : 0;
    d.q[i].load_probe = load_probe_enabled(i == 0 ? l0 : l1) ? 1 : 0;
  }
  d.units0 = d.q[0].num_units;
  d.num_units = d.q[0].num_units + d.q[1].num_units;
  if (d.num_units == 0) return cudaSuccess;
  const int clusters = std::min(d.num_units, dual_clusters(epi_warps));
  return run_pair_dual(d, clusters, st, nullptr, epi_warps);
}

}  // namespace tpk
