// Tensor-core fused weight-gradient + nadam step: every (weight dtype,
// moment dtype, tile width, pipeline depth) instantiation for this rule.
#include "wgrad_tc_dispatch.cuh"

namespace forge {

cudaError_t launch_wgrad_tc_nadam(const WgradTcParams& p, const TcLaunch& l) {
  return launch_opt<OPT_NADAM>(p, l);
}

}  // namespace forge
