// wgrad_tc_dispatch.cuh -- compile-time choice of pipeline depths and the
// runtime dispatch over (weight dtype, moment dtype, tile width, depth) for
// one optimizer. Included once per optimizer translation unit.
#pragma once

#include "wgrad_tc.cuh"

namespace forge {

// Shared memory available to the dynamic ring after the kernel's static
// shared memory (barriers + the 8 KB absmax exchange) is accounted for.
constexpr int kDynSmemBudget = 227 * 1024 - 9 * 1024;

template <int OPT, int WK, int MK, int BN, int STAGES, bool DX = false, bool GA = false, bool NARROW = false,
          bool WIDE = false, bool PAIR = false>
constexpr int slots_that_fit() {
  using C = TcCfg<OPT, WK, MK, BN, STAGES, 2, DX, GA, NARROW, WIDE, PAIR>;
  const int avail = kDynSmemBudget - 1024 - STAGES * C::STAGE_BYTES - C::WB_BYTES;
  const int n = avail / C::SLOT_BYTES;
  return n > 8 ? 8 : n;
}

// Operand stages: 2 for short token axes (the step is bound by the state
// stream); for long ones as many as leave room for the state ring (4, else
// 3, else 2). CTA pairs, whose stages are a third smaller, take up to PS
// (5, or 4 where the state stream is heavy) beside at least two slots.
template <int OPT, int WK, int MK, int BN, int DEEP, bool WIDE = false, bool NARROW = false, bool PAIR = false,
          int PS = 5>
constexpr int pick_stages() {
  if (!DEEP) return 2;
  constexpr int need = (MK == M_Q8) ? 4 : 2;
  if constexpr (PAIR)
    if (PS >= 5 && slots_that_fit<OPT, WK, MK, BN, 5, false, false, NARROW, WIDE, PAIR>() >= need) return 5;
  if (slots_that_fit<OPT, WK, MK, BN, 4, false, false, NARROW, WIDE, PAIR>() >= need) return 4;
  if (slots_that_fit<OPT, WK, MK, BN, 3, false, false, NARROW, WIDE, PAIR>() >= need) return 3;
  return 2;
}

template <int OPT, int WK, int MK, int BN, int DEEP, bool WIDE = false, bool NARROW = false, bool PAIR = false,
          int PS = 5>
cudaError_t launch_one(const WgradTcParams& p, int grid, cudaStream_t stream) {
  constexpr int S = pick_stages<OPT, WK, MK, BN, DEEP, WIDE, NARROW, PAIR, PS>();
  constexpr int N = slots_that_fit<OPT, WK, MK, BN, S, false, false, NARROW, WIDE, PAIR>();
  static_assert(N >= ((MK == M_Q8) ? 4 : 2), "state ring does not fit");
  return launch_tc_variant<OPT, WK, MK, BN, S, N, false, false, NARROW, WIDE, PAIR>(p, grid, stream);
}

// Step with an accumulated gradient (the last micro-batch): two operand
// stages, the state ring also carries the fp32 G_acc chunks.
template <int OPT, int WK, int MK, int BN>
cudaError_t launch_ga(const WgradTcParams& p, int grid, cudaStream_t stream) {
  constexpr int N = slots_that_fit<OPT, WK, MK, BN, 2, false, true>();
  static_assert(N >= 2, "state ring does not fit");
  return launch_tc_variant<OPT, WK, MK, BN, 2, N, false, true>(p, grid, stream);
}

// Fused input gradient: 64-column tiles, two 128-token operand stages, or
// three (DEEP: long token axes, where the mainloop sets the pace) when the
// state ring still keeps two slots.
template <int OPT, int WK, int MK, bool NARROW = false, bool DEEP = false>
cudaError_t launch_dx(const WgradTcParams& p, int grid, cudaStream_t stream) {
  constexpr int S = (DEEP && slots_that_fit<OPT, WK, MK, 64, 3, true, false, NARROW>() >= 2) ? 3 : 2;
  constexpr int N = slots_that_fit<OPT, WK, MK, 64, S, true, false, NARROW>();
  static_assert(N >= 2, "state ring does not fit");
  return launch_tc_variant<OPT, WK, MK, 64, S, N, true, false, NARROW>(p, grid, stream);
}

template <int OPT, int WK, int MK>
cudaError_t launch_mk(const WgradTcParams& p, const TcLaunch& l) {
  if (l.pair && (l.ga || l.dx || l.wide || l.bn != 256 || MK == M_Q8)) return cudaErrorInvalidValue;
  if (l.ga) {
    if constexpr (MK == M_Q8) return cudaErrorInvalidValue;
    else {
      if (l.dx || l.deep) return cudaErrorInvalidValue;
      return l.bn == 64 ? launch_ga<OPT, WK, MK, 64>(p, l.grid, l.stream)
                        : launch_ga<OPT, WK, MK, 128>(p, l.grid, l.stream);
    }
  }
  if (l.dx) {
    if constexpr (MK == M_Q8) return cudaErrorInvalidValue;
    else {
      if (l.bn != 64) return cudaErrorInvalidValue;
      if constexpr (WK == W_F32 && MK == M_F32 && opt_nstate(OPT) >= 1)
        if (l.narrow)
          return l.deep ? launch_dx<OPT, WK, MK, true, true>(p, l.grid, l.stream)
                        : launch_dx<OPT, WK, MK, true, false>(p, l.grid, l.stream);
      if (l.narrow) return cudaErrorInvalidValue;
      return l.deep ? launch_dx<OPT, WK, MK, false, true>(p, l.grid, l.stream)
                    : launch_dx<OPT, WK, MK, false, false>(p, l.grid, l.stream);
    }
  }
  if constexpr (MK == M_Q8) {
    if (l.bn != 128) return cudaErrorInvalidValue;
    return l.deep ? launch_one<OPT, WK, MK, 128, 1>(p, l.grid, l.stream)
                  : launch_one<OPT, WK, MK, 128, 0>(p, l.grid, l.stream);
  } else {
    if (l.bn == 64) {
      if (l.deep || l.wide) return cudaErrorInvalidValue;
      return launch_one<OPT, WK, MK, 64, 0>(p, l.grid, l.stream);
    }
    if constexpr (WK == W_BF16 && MK == M_BF16 && opt_nstate(OPT) >= 1) {
      // 64-column state chunks (128-column tiles only).
      if (l.wide) {
        if (l.bn != 128) return cudaErrorInvalidValue;
        return l.deep ? launch_one<OPT, WK, MK, 128, 1, true>(p, l.grid, l.stream)
                      : launch_one<OPT, WK, MK, 128, 0, true>(p, l.grid, l.stream);
      }
    }
    if (l.wide) return cudaErrorInvalidValue;
    if (l.bn == 256) {
      // 128 x 256 tiles for long token axes: a quarter less operand traffic
      // per gradient element than 128 x 128, half the MMA instructions.
      if (!l.deep) return cudaErrorInvalidValue;
      // l.pair: 0, or the CTA pair's operand stages (5; 4 for fp32 W with
      // two fp32 moments below 4096 tokens).
      if constexpr (WK == W_F32 && MK == M_F32 && opt_nstate(OPT) >= 1) {
        if (l.narrow) {
          if (l.pair == 0) return launch_one<OPT, WK, MK, 256, 1, false, true>(p, l.grid, l.stream);
          if constexpr (opt_nstate(OPT) == 2)
            if (l.pair == 4) return launch_one<OPT, WK, MK, 256, 1, false, true, true, 4>(p, l.grid, l.stream);
          if (l.pair != 5) return cudaErrorInvalidValue;
          return launch_one<OPT, WK, MK, 256, 1, false, true, true, 5>(p, l.grid, l.stream);
        }
      }
      if (l.narrow || (l.pair != 0 && l.pair != 5)) return cudaErrorInvalidValue;
      return l.pair ? launch_one<OPT, WK, MK, 256, 1, false, false, true, 5>(p, l.grid, l.stream)
                    : launch_one<OPT, WK, MK, 256, 1>(p, l.grid, l.stream);
    }
    if constexpr (WK == W_F32 && MK == M_F32 && opt_nstate(OPT) >= 1)
      if (l.narrow && l.deep) return launch_one<OPT, WK, MK, 128, 1, false, true>(p, l.grid, l.stream);
    if (l.narrow || l.pair) return cudaErrorInvalidValue;
    return l.deep ? launch_one<OPT, WK, MK, 128, 1>(p, l.grid, l.stream)
                  : launch_one<OPT, WK, MK, 128, 0>(p, l.grid, l.stream);
  }
}

template <int OPT>
cudaError_t launch_opt(const WgradTcParams& p, const TcLaunch& l) {
  constexpr bool kQ8 = (OPT == OPT_ADAMW || OPT == OPT_SGDM || OPT == OPT_LION);
  if constexpr (opt_nstate(OPT) == 0) {
    // No state tensor: the moment storage does not matter.
    return l.wk == W_F32 ? launch_mk<OPT, W_F32, M_F32>(p, l) : launch_mk<OPT, W_BF16, M_F32>(p, l);
  } else {
    if (l.wk == W_F32) {
      if (l.mk == M_F32) return launch_mk<OPT, W_F32, M_F32>(p, l);
      if (l.mk == M_BF16) return launch_mk<OPT, W_F32, M_BF16>(p, l);
      if constexpr (kQ8)
        if (l.mk == M_Q8) return launch_mk<OPT, W_F32, M_Q8>(p, l);
    } else {
      if (l.mk == M_F32) return launch_mk<OPT, W_BF16, M_F32>(p, l);
      if (l.mk == M_BF16) return launch_mk<OPT, W_BF16, M_BF16>(p, l);
      if constexpr (kQ8)
        if (l.mk == M_Q8) return launch_mk<OPT, W_BF16, M_Q8>(p, l);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace forge
