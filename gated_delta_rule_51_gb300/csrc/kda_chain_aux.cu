// kda_chain_aux.cu -- the segment scan's correction and transition runs (kda_chain.cuh with
// kChainAux): the recurrence with v taken as zero, stopped once the state it carries is
// exactly zero in fp32.  A translation unit of its own, so that the forward runs' kernels
// carry none of this code and the families compile in parallel.
#include "kda_chain.cuh"

namespace kda {

cudaError_t launch_chain_aux(const ChainParams& p, int grid, cudaStream_t s, bool overlap_prev) {
  if (p.precise) return launch_chain_table<kChainAux | kChainPrecise>(p, grid, s, overlap_prev);
  return launch_chain_table<kChainAux>(p, grid, s, overlap_prev);
}

}  // namespace kda
