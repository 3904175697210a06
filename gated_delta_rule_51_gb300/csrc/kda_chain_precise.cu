// kda_chain_precise.cu -- the precise-state variants of the chunked forward kernel
// (kda_chain.cuh with kChainPrecise): the carried state, W and the tile W is made from are
// read as bf16 hi + lo, for gates that hardly decay.  A translation unit of its own, so the
// two families compile in parallel.
#include "kda_chain.cuh"

namespace kda {

cudaError_t launch_chain_precise(const ChainParams& p, int grid, cudaStream_t s, bool overlap_prev) {
  return launch_chain_table<kChainPrecise>(p, grid, s, overlap_prev);
}

}  // namespace kda
