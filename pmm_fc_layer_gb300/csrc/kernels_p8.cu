// GEMM kernel instantiations for launches of up to 8 block product(s).
#include "kernel_instances.cuh"

namespace axonn {
template cudaError_t kernels_init<8>(bool*);
template cudaError_t kernels_launch<8>(int, const GemmParams<8>&, int, bool, cudaStream_t);
template cudaError_t kernels_take_status<8>(unsigned long long*, cudaStream_t);
}  // namespace axonn
