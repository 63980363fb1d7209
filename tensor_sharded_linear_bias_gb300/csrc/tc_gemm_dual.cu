// Instantiations of the SM-pair kernel that runs two GEMMs in one launch: the first with both
// operands MN-major (weight gradients), the second with both K-major (input gradients).
#include "tc2_gemm.cuh"

namespace tpk {
namespace tc {

// 8 or 12 epilogue warps; max_clusters != nullptr asks for the occupancy limit only.
cudaError_t run_pair_dual(const TcDual& d, int clusters, cudaStream_t st, int* max_clusters,
                          int epi_warps) {
  if (epi_warps == 12)
    return tc2::launch_dual<true, true, false, false, 12>(d, clusters, st, max_clusters);
  return tc2::launch_dual<true, true, false, false, 8>(d, clusters, st, max_clusters);
}

}  // namespace tc
}  // namespace tpk
