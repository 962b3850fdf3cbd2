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

// The reduction-split kernel: 128 x 128 tiles, 3 stages of 32 KB beside the
// 66 KB staging tile and the 58 KB inbox (226 KB in all).  Pieces are short
// (num_k / S stages), so a deeper ring buys little.
constexpr int kSplitStages = 3;
using SplitLayout = SmemLayout<128, 64, kSplitStages, 1, true>;
#define AXONN_SPLIT_KERNEL fc_gemm_tcgen05_kernel<128, 64, kSplitStages, 1, 1, true>
static_assert(SplitLayout::kBytes <= 227 * 1024, "split kernel shared memory");

cudaError_t split_kernel_init() {
  return cudaFuncSetAttribute(AXONN_SPLIT_KERNEL, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              SplitLayout::kBytes);
}

cudaError_t split_clusters_resident(int sms, int pieces, int* clusters) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(sms / pieces * pieces), 1, 1);
  cfg.blockDim = dim3(cta_threads<1>(), 1, 1);
  cfg.dynamicSmemBytes = SplitLayout::kBytes;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  cfg.numAttrs = static_cast<unsigned>(launch_attrs(attr, false, pieces));
  return cudaOccupancyMaxActiveClusters(clusters, reinterpret_cast<const void*>(&AXONN_SPLIT_KERNEL),
                                        &cfg);
}

cudaError_t split_kernel_launch(const GemmParams<1>& P, int pieces, int clusters, bool pdl,
                                cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * pieces), 1, 1);
  cfg.blockDim = dim3(cta_threads<1>(), 1, 1);
  cfg.dynamicSmemBytes = SplitLayout::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  cfg.numAttrs = static_cast<unsigned>(launch_attrs(attr, pdl, pieces));
  return cudaLaunchKernelEx(&cfg, AXONN_SPLIT_KERNEL, P);
}
#undef AXONN_SPLIT_KERNEL
}  // namespace axonn
