// Definitions behind kernel_launch.h, instantiated once per MAXP by the
// kernels_p*.cu translation units.
#pragma once
#include "gemm_pair_kernel.cuh"
#include "kernel_launch.h"

namespace axonn {

constexpr int kPairStages = 6;   // 256 x 256 pair tiles, 32 KB stages
constexpr int kPair2Stages = 4;  // 512 x 256 pair tiles, 48 KB stages

// Launch attributes: programmatic stream serialization (pdl) and, when
// cluster > 0, the cluster size along x.
inline int launch_attrs(cudaLaunchAttribute (&attr)[2], bool pdl, int cluster) {
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  return n;
}

// Launches `kernel` with cudaLaunchKernelEx; with `pdl` the launch may begin
// while the previous kernel in the stream finishes (programmatic stream
// serialization; the kernel waits for it with griddepcontrol.wait).
template <typename K, int MAXP>
cudaError_t launch_ex(K kernel, const GemmParams<MAXP>& P, int ctas, int threads, int smem,
                      bool pdl, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  cfg.numAttrs = static_cast<unsigned>(launch_attrs(attr, pdl, 0));
  return cudaLaunchKernelEx(&cfg, kernel, P);
}

template <int BN, int BK, int STAGES, int MAXP, int MH>
struct Single {
  static cudaError_t init() {
    return cudaFuncSetAttribute(fc_gemm_tcgen05_kernel<BN, BK, STAGES, MAXP, MH>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                SmemLayout<BN, BK, STAGES, MH>::kBytes);
  }
  static cudaError_t launch(const GemmParams<MAXP>& P, int ctas, bool pdl, cudaStream_t s) {
    return launch_ex(fc_gemm_tcgen05_kernel<BN, BK, STAGES, MAXP, MH>, P, ctas, cta_threads<MH>(),
                     SmemLayout<BN, BK, STAGES, MH>::kBytes, pdl, s);
  }
};

template <int BN, int STAGES, int MAXP, int MH>
struct Pair {
  static cudaError_t init() {
    return cudaFuncSetAttribute(fc_gemm_tcgen05_pair_kernel<BN, STAGES, MAXP, MH>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                PairSmemLayout<BN, STAGES, MH>::kBytes);
  }
  // The 12-warp (register split) variant must have exactly the launch
  // allocation its split adds up to: fewer registers per thread would make
  // the epilogue's setmaxnreg increase wait forever.
  static cudaError_t check_regs(bool* ok) {
    if (MH != 2) return cudaSuccess;
    cudaFuncAttributes a = {};
    const cudaError_t e = cudaFuncGetAttributes(
        &a, reinterpret_cast<const void*>(fc_gemm_tcgen05_pair_kernel<BN, STAGES, MAXP, MH>));
    if (e == cudaSuccess && a.numRegs != kRegsAtLaunch) *ok = false;
    return e;
  }
  static cudaError_t launch(const GemmParams<MAXP>& P, int pairs, bool pdl, cudaStream_t s) {
    return launch_ex(fc_gemm_tcgen05_pair_kernel<BN, STAGES, MAXP, MH>, P, 2 * pairs,
                     cta_threads<MH, MH == 2>(), PairSmemLayout<BN, STAGES, MH>::kBytes, pdl, s);
  }
};

template <int MAXP>
using C0 = Single<128, 64, 6, MAXP, 1>;
template <int MAXP>
using C1 = Single<256, 64, 4, MAXP, 1>;
template <int MAXP>
using C2 = Pair<256, kPairStages, MAXP, 1>;
template <int MAXP>
using C3 = Single<256, 64, 3, MAXP, 2>;
template <int MAXP>
using C4 = Single<192, 64, 5, MAXP, 1>;
template <int MAXP>
using C5 = Single<192, 64, 4, MAXP, 2>;
template <int MAXP>
using C6 = Pair<256, kPair2Stages, MAXP, 2>;
template <int MAXP>
using C7 = Single<64, 64, 8, MAXP, 1>;  // 128 x 64 tiles, 24 KB stages

template <int MAXP>
cudaError_t kernels_init(bool* split_ok) {
  const cudaError_t es[] = {C0<MAXP>::init(), C1<MAXP>::init(), C2<MAXP>::init(),
                            C3<MAXP>::init(), C4<MAXP>::init(), C5<MAXP>::init(),
                            C6<MAXP>::init(), C7<MAXP>::init(), C6<MAXP>::check_regs(split_ok)};
  for (cudaError_t e : es)
    if (e != cudaSuccess) return e;
  return cudaSuccess;
}

template <int MAXP>
cudaError_t kernels_launch(int config, const GemmParams<MAXP>& P, int units, bool pdl,
                           cudaStream_t s) {
  switch (config) {
    case 0: return C0<MAXP>::launch(P, units, pdl, s);
    case 1: return C1<MAXP>::launch(P, units, pdl, s);
    case 2: return C2<MAXP>::launch(P, units, pdl, s);
    case 3: return C3<MAXP>::launch(P, units, pdl, s);
    case 4: return C4<MAXP>::launch(P, units, pdl, s);
    case 5: return C5<MAXP>::launch(P, units, pdl, s);
    case 6: return C6<MAXP>::launch(P, units, pdl, s);
    case 7: return C7<MAXP>::launch(P, units, pdl, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int MAXP>
cudaError_t kernels_take_status(unsigned long long* word, cudaStream_t stream) {
  *word = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(word, g_status_word, sizeof(*word), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess || *word == 0) return e;
  const unsigned long long zero = 0;
  e = cudaMemcpyToSymbolAsync(g_status_word, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return e;
}

}  // namespace axonn
