// Tensor-core fused weight-gradient + radam step: every (weight dtype,
// moment dtype, tile width, pipeline depth) instantiation for this rule.
#include "wgrad_tc_dispatch.cuh"

namespace forge {

cudaError_t launch_wgrad_tc_radam(const WgradTcParams& p, const TcLaunch& l) {
  return launch_opt<OPT_RADAM>(p, l);
}

}  // namespace forge
