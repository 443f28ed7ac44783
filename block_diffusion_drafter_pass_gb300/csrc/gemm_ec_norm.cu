// gemm_ec_norm.cu - GEMM kernel instantiations for one epilogue class
// (compiled separately so the library builds in parallel).
#include "gemm_kernel.cuh"

namespace dfl {
namespace gk {

cudaError_t launch_ec_norm(const AMaps& amaps, const ARegions& rg, const CUtensorMap& xmap, const GemmArgs& a,
                           const GemmEpi& e, int BN, cudaStream_t stream) {
  return launch_class_bn<kEcNorm>(amaps, rg, xmap, a, e, BN, stream);
}

}  // namespace gk
}  // namespace dfl
