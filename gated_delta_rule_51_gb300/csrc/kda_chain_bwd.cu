// kda_chain_bwd.cu -- the backward's chain kernels: kda_chain_kernel with kChainBwd, for the
// gate with a lower bound and each setting of the beta and L2-norm switches.  One launch runs
// both kinds of run side by side: forward runs that store every chunk's entering state and Vn,
// and reverse runs that carry dS from each sequence's end to its start (kModeReverse).  When a
// sequence is split in two, a second launch (kChainAux) runs the correction runs that carry the
// true state across the split (kModeCorrect forward, kModeReverseCorrect reverse).
#include "kda_chain.cuh"

namespace kda {

cudaError_t launch_chain_bwd(const ChainParams& p, int grid, cudaStream_t s, bool corrections) {
  using Kernel = void (*)(ChainParams);
  // indexed by the caller-side flags kBetaPreactivated | kNoQkL2Norm (the gate is the safe one),
  // then the correction runs of split sequences (kChainAux)
  constexpr int kC = kChainBwd | kChainAux;
  static constexpr Kernel kernels[8] = {kda_chain_kernel<kChainBwd + 0>, kda_chain_kernel<kChainBwd + 2>,
                                        kda_chain_kernel<kChainBwd + 4>, kda_chain_kernel<kChainBwd + 6>,
                                        kda_chain_kernel<kC + 0>, kda_chain_kernel<kC + 2>,
                                        kda_chain_kernel<kC + 4>, kda_chain_kernel<kC + 6>};
  constexpr size_t smem = chain_smem_bytes_t<false>();
  constexpr int kMaxDevices = 64;
  static std::atomic<bool> opted_in[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices || !opted_in[dev].load(std::memory_order_acquire)) {
    for (Kernel k : kernels) {
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    if (dev >= 0 && dev < kMaxDevices) opted_in[dev].store(true, std::memory_order_release);
  }
  if (grid <= 0) return cudaSuccess;
  if ((p.flags & (kGatePreactivated | kGateSoftplus)) != 0 || p.kdim != 128 || p.vrows != 128 || p.precise)
    return cudaErrorInvalidValue;
  const Kernel k = kernels[((p.flags & (kBetaPreactivated | kNoQkL2Norm)) >> 1) + (corrections ? 4 : 0)];
  if (!corrections) {
    k<<<grid, kThreads, smem, s>>>(p);
    return cudaGetLastError();
  }
  // the corrections start beside the runs (programmatic dependent launch): they load their
  // first chunks' inputs and prepare their operands, and wait for the runs before they read a
  // slot or a stored copy
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, p);
}

}  // namespace kda
