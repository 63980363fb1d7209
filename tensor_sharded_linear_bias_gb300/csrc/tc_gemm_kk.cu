// Instantiation of the tcgen05 GEMM for A K-major, B K-major.
#include "tc_gemm.cuh"

namespace tpk {
namespace tc {

cudaError_t run_kk(const TcParams& p, int grid, cudaStream_t st) {
  auto kern = tc_gemm_kernel<false, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<grid, NUM_THREADS, SMEM_BYTES, st>>>(p);
  return cudaGetLastError();
}

}  // namespace tc
}  // namespace tpk
