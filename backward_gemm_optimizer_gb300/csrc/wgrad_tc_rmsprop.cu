// Tensor-core fused weight-gradient + rmsprop step: every (weight dtype,
// moment dtype, tile width, pipeline depth) instantiation for this rule.
#include "wgrad_tc_dispatch.cuh"

namespace forge {

cudaError_t launch_wgrad_tc_rmsprop(const WgradTcParams& p, const TcLaunch& l) {
  return launch_opt<OPT_RMSPROP>(p, l);
}

}  // namespace forge
