// Instantiations of the tcgen05 GEMM (one-SM and SM-pair kernels) for A K-major, B K-major.
#include "tc2_gemm.cuh"

namespace tpk {
namespace tc {

cudaError_t run_kk(const TcParams& p, int grid, cudaStream_t st) {
  auto kern = tc_gemm_kernel<false, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<grid, NUM_THREADS, SMEM_BYTES, st>>>(p);
  return cudaGetLastError();
}

// SM-pair kernel: clusters of two CTAs. max_clusters == 0 asks for the occupancy limit only.
cudaError_t run_pair_kk(const TcParams& p, int clusters, cudaStream_t st, int* max_clusters) {
  auto kern = tc2::tc2_gemm_kernel<false, false>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, tc2::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(tc2::NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = tc2::SMEM_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_clusters != nullptr) {
    cfg.gridDim = dim3(2, 1, 1);
    return cudaOccupancyMaxActiveClusters(max_clusters, kern, &cfg);
  }
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace tc
}  // namespace tpk
