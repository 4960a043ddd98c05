// The E4M3-weight variants of the projection kernel (gemm_kernel.cuh),
// instantiated apart from the bf16 ones so the two compile in parallel.
#include "gemm_kernel.cuh"

namespace dflash {

cudaError_t launch_tc_w8(dflash_ctx* c, const GemmLaunch& g, int bn, const CUtensorMap& tw, const CUtensorMap& tx,
                         const CUtensorMap& txlo, cudaStream_t s) {
  return g.X_lo != nullptr ? launch_tc_bn<true, true>(c, g, bn, tw, tx, txlo, s)
                           : launch_tc_bn<false, true>(c, g, bn, tw, tx, txlo, s);
}

}  // namespace dflash
