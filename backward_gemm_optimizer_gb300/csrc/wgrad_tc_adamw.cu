// Tensor-core fused weight-gradient + adamw step: every (weight dtype,
// moment dtype, tile width, pipeline depth) instantiation for this rule.
#include "wgrad_tc_dispatch.cuh"

namespace forge {

cudaError_t launch_wgrad_tc_adamw(const WgradTcParams& p, const TcLaunch& l) {
  return launch_opt<OPT_ADAMW>(p, l);
}

}  // namespace forge
