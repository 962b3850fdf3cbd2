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

// The reduction-split kernels.  128 x 128 tiles: 3 stages of 32 KB beside
// the 66 KB staging tile and the 58 KB inbox (226 KB in all).  128 x 64
// tiles: 6 stages of 24 KB beside a 34 KB staging tile and a 30 KB inbox
// (209 KB).  Pieces are short (num_k / S stages), so a deeper ring buys
// little.
constexpr int kSplitStages = 3;
constexpr int kSplit64Stages = 6;
using SplitLayout = SmemLayout<128, 64, kSplitStages, 1, true>;
using Split64Layout = SmemLayout<64, 64, kSplit64Stages, 1, true>;
#define AXONN_SPLIT_KERNEL fc_gemm_tcgen05_kernel<128, 64, kSplitStages, 1, 1, true>
#define AXONN_SPLIT64_KERNEL fc_gemm_tcgen05_kernel<64, 64, kSplit64Stages, 1, 1, true>
static_assert(SplitLayout::kBytes <= 227 * 1024, "split kernel shared memory");
static_assert(Split64Layout::kBytes <= 227 * 1024, "split kernel shared memory");

cudaError_t split_kernel_init() {
  cudaError_t e = cudaFuncSetAttribute(AXONN_SPLIT_KERNEL, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SplitLayout::kBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(AXONN_SPLIT64_KERNEL, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Split64Layout::kBytes);
  return e;
}

namespace {
cudaLaunchConfig_t split_config_for(int pieces, int ctas, int bn, cudaLaunchAttribute (&attr)[2],
                                    bool pdl, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
  cfg.blockDim = dim3(cta_threads<1>(), 1, 1);
  cfg.dynamicSmemBytes = bn == 64 ? Split64Layout::kBytes : SplitLayout::kBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = static_cast<unsigned>(launch_attrs(attr, pdl, pieces));
  return cfg;
}
}  // namespace

cudaError_t split_clusters_resident(int sms, int pieces, int bn, int* clusters) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = split_config_for(pieces, sms / pieces * pieces, bn, attr, false, nullptr);
  return bn == 64
             ? cudaOccupancyMaxActiveClusters(clusters, reinterpret_cast<const void*>(&AXONN_SPLIT64_KERNEL), &cfg)
             : cudaOccupancyMaxActiveClusters(clusters, reinterpret_cast<const void*>(&AXONN_SPLIT_KERNEL), &cfg);
}

cudaError_t split_kernel_launch(const GemmParams<1>& P, int pieces, int clusters, int bn, bool pdl,
                                cudaStream_t stream) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = split_config_for(pieces, clusters * pieces, bn, attr, pdl, stream);
  return bn == 64 ? cudaLaunchKernelEx(&cfg, AXONN_SPLIT64_KERNEL, P)
                  : cudaLaunchKernelEx(&cfg, AXONN_SPLIT_KERNEL, P);
}
#undef AXONN_SPLIT64_KERNEL
#undef AXONN_SPLIT_KERNEL
}  // namespace axonn
