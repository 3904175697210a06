// kda_chain.cu -- the usual variants of the chunked forward kernel (kda_chain.cuh) and the
// launch entry that picks them or the precise-state ones (kda_chain_precise.cu).
#include "kda_chain.cuh"

namespace kda {

cudaError_t launch_chain(const ChainParams& p, int grid, cudaStream_t s) {
  if (p.precise) return launch_chain_precise(p, grid, s);
  return launch_chain_table<0>(p, grid, s);
}

}  // namespace kda
