// Host interface of the GEMM kernel instantiations.  Each size of the
// problem table (MAXP = 1, 8, 64 block products per launch) is compiled in a
// translation unit of its own (kernels_p1.cu, kernels_p8.cu, kernels_p64.cu)
// so that the library builds in parallel; the host code calls these
// functions and never names a kernel template itself.
#pragma once
#include <cuda_runtime.h>

#include "gemm_kernel.cuh"

namespace axonn {

// Kernel configurations by index (the host's configuration table uses the
// same order): 0 1cta_128x128, 1 1cta_128x256, 2 pair_256x256,
// 3 1cta_256x256, 4 1cta_128x192, 5 1cta_256x192, 6 pair_512x256,
// 7 1cta_128x64.
constexpr int kKernelConfigs = 8;

// Sets the dynamic shared memory limit of every instantiation for this
// MAXP on the current device, and checks that each 12-warp kernel was built
// with the register count its setmaxnreg split assumes (*split_ok = false
// if not).
template <int MAXP>
cudaError_t kernels_init(bool* split_ok);

// Launches configuration `config` over `units` persistent CTAs, or CTA pairs
// for the pair configurations; with `pdl` as a programmatic dependent launch
// (its set-up overlaps the previous kernel in the stream).
template <int MAXP>
cudaError_t kernels_launch(int config, const GemmParams<MAXP>& P, int units, bool pdl,
                           cudaStream_t stream);

// Reads, and clears if set, the device error word of this MAXP's kernels
// (each translation unit that instantiates kernels holds its own copy of
// g_status_word), in order on `stream`; *word = 0 when no wait expired.
template <int MAXP>
cudaError_t kernels_take_status(unsigned long long* word, cudaStream_t stream);

// Clusters of 2 of the pair kernels that can be resident at once.
cudaError_t pair_clusters_resident(int sms, int* clusters);

// The reduction-split kernels (one problem; see fc_gemm_tcgen05_kernel's
// kSplit), with 128 x 128 tiles (bn = 128) or 128 x 64 tiles (bn = 64):
// their shared-memory limits, how many of their clusters of `pieces` CTAs
// (2, 4 or 8) can be resident at once, and a launch of `clusters` such
// clusters.
cudaError_t split_kernel_init();
cudaError_t split_clusters_resident(int sms, int pieces, int bn, int* clusters);
cudaError_t split_kernel_launch(const GemmParams<1>& P, int pieces, int clusters, int bn, bool pdl,
                                cudaStream_t stream);

}  // namespace axonn
