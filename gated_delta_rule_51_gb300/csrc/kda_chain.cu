// kda_chain.cu -- the usual variants of the chunked forward kernel (kda_chain.cuh) for forward
// runs, and the launch entry that picks them or the precise-state ones (kda_chain_precise.cu).
// The segment scan's correction and transition runs have kernels of their own (kda_chain_aux.cu).
#include "kda_chain.cuh"

namespace kda {

cudaError_t launch_chain(const ChainParams& p, int grid, cudaStream_t s, bool overlap_prev) {
  if (p.precise) return launch_chain_precise(p, grid, s, overlap_prev);
  return launch_chain_table<0>(p, grid, s, overlap_prev);
}

}  // namespace kda
