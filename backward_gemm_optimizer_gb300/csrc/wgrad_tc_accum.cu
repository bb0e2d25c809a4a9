// Gradient accumulation over micro-batches (FORGE, Appendix L, the exact
// mode): the weight-gradient GEMM of each micro-batch adds its tiles into an
// fp32 accumulator G_acc in HBM (or, on the first micro-batch, writes them
// there), through the same tile kernel as the fused step with the
// accumulator in place of the weights -- optionally with the micro-batch's
// input gradient dX = dY W formed in the same pass, as in the fused
// backward step. The step itself fires once, at the last micro-batch,
// through the accumulated-gradient variant of the rule kernels.
#include "wgrad_tc_dispatch.cuh"

namespace forge {

namespace {

template <int OPT>
cudaError_t launch_accum(const WgradTcParams& p, const TcLaunch& l) {
  if (l.ga || l.narrow) return cudaErrorInvalidValue;
  if (l.dx) {
    // With the input gradient of the same micro-batch (wk: the dtype of the
    // weights read for dX); three 128-token operand stages, since the
    // accumulator alone leaves the state ring little to do.
    if (l.bn != 64 || !l.deep) return cudaErrorInvalidValue;
    return l.wk == W_F32 ? launch_dx<OPT, W_F32, M_F32, false, true>(p, l.grid, l.stream)
                         : launch_dx<OPT, W_BF16, M_F32, false, true>(p, l.grid, l.stream);
  }
  if (l.wk != W_F32) return cudaErrorInvalidValue;
  if (l.bn == 64) {
    if (l.deep) return cudaErrorInvalidValue;
    return launch_one<OPT, W_F32, M_F32, 64, 0>(p, l.grid, l.stream);
  }
  return l.deep ? launch_one<OPT, W_F32, M_F32, 128, 1>(p, l.grid, l.stream)
                : launch_one<OPT, W_F32, M_F32, 128, 0>(p, l.grid, l.stream);
}

}  // namespace

cudaError_t launch_wgrad_tc_accum(const WgradTcParams& p, const TcLaunch& l) {
  return l.opt == OPT_ACCSET ? launch_accum<OPT_ACCSET>(p, l) : launch_accum<OPT_ACCUM>(p, l);
}

}  // namespace forge
