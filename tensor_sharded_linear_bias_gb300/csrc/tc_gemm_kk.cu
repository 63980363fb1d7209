// Instantiations of the tcgen05 GEMM (one-SM and SM-pair kernels) for A K-major, B K-major.
#include "tc2_gemm.cuh"

namespace tpk {
namespace tc {

cudaError_t run_kk(const TcParams& p, int grid, cudaStream_t st) {
  auto kern = tc_gemm_kernel<false, false>;
  cudaError_t e = opt_in_dynamic_smem(reinterpret_cast<const void*>(kern), SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<grid, NUM_THREADS, SMEM_BYTES, st>>>(p);
  return cudaGetLastError();
}

// SM-pair kernel: clusters of two CTAs, 4 or 8 epilogue warps. max_clusters != nullptr asks
// for the occupancy limit only.
cudaError_t run_pair_kk(const TcParams& p, int clusters, cudaStream_t st, int* max_clusters,
                         int epi_warps, int sub) {
  return tc2::launch_pair_variant<false, false>(p, clusters, st, max_clusters, epi_warps, sub);
}

}  // namespace tc
}  // namespace tpk
