// GEMM kernel instantiations for launches of up to 1 block product(s).
#include "kernel_instances.cuh"

namespace axonn {
template cudaError_t kernels_init<1>(bool*);
template cudaError_t kernels_launch<1>(int, const GemmParams<1>&, int, bool, cudaStream_t);
template cudaError_t kernels_take_status<1>(unsigned long long*, cudaStream_t);

cudaError_t pair_clusters_resident(int sms, int* clusters) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * sms, 1, 1);
  cfg.blockDim = dim3(cta_threads<1>(), 1, 1);
  cfg.dynamicSmemBytes = PairSmemLayout<256, kPairStages, 1>::kBytes;
  return cudaOccupancyMaxActiveClusters(
      clusters, reinterpret_cast<const void*>(&fc_gemm_tcgen05_pair_kernel<256, kPairStages, 1, 1>),
      &cfg);
}
}  // namespace axonn
