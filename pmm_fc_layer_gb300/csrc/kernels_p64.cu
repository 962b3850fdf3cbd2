// GEMM kernel instantiations for launches of up to 64 block product(s).
#include "kernel_instances.cuh"

namespace axonn {
template cudaError_t kernels_init<64>(bool*);
template cudaError_t kernels_launch<64>(int, const GemmParams<64>&, int, bool, cudaStream_t);
template cudaError_t kernels_take_status<64>(unsigned long long*, cudaStream_t);
}  // namespace axonn
