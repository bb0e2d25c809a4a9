// wgrad_simt.cu -- fused weight-gradient + optimizer step for fp32 X / dY
// on the CUDA cores (FORGE, Algorithm 1, for inputs the bf16 tensor-core
// path cannot take without rounding them).
//
// A CTA of 128 threads owns a 16 x 128 tile of G: thread t owns column
// q0 + t and accumulates its 16 rows over the token axis with fp32 fused
// multiply-adds in ascending token order (Eq. 5 with T_K = 1). The
// epilogue then steps those 16 elements in registers, exactly as the
// tensor-core kernel does, and writes W and the moments back. The 8-bit
// variant reduces each row's block absmax across the 128 threads (the
// tile row is one 128-element block).
#include <cstdint>

#include "forge_math.cuh"
#include "forge_params.h"

namespace forge {

namespace {

constexpr int SR = 16;   // rows per tile
constexpr int SC = 128;  // columns per tile (one 8-bit block)
constexpr int TT = 32;   // tokens staged per step

template <int KIND>
__device__ __forceinline__ float ld_val(const void* base, int64_t off) {
  if constexpr (KIND == 0) return static_cast<const float*>(base)[off];
  else return bf16_bits_to_f32(static_cast<const uint16_t*>(base)[off]);
}

__device__ __forceinline__ uint32_t draw16(uint64_t idx, uint32_t step, uint32_t site, uint32_t lo, uint32_t hi) {
  const U4 r = sr_block(idx >> 3, step, site, lo, hi);
  return sr_lane(r, static_cast<int>(idx & 7));
}

template <int OPT, int WK, int MK>
__global__ void __launch_bounds__(128) wgrad_step_simt_kernel(const WgradSimtParams p) {
  __shared__ float dys[TT][SR];
  __shared__ float red[2][4][SR];
  constexpr int NST = opt_nstate(OPT);
  constexpr bool TWO = (NST == 2);
  const int t = threadIdx.x;
  const int q = blockIdx.x * SC + t;
  const int p0 = blockIdx.y * SR;
  const bool qok = q < p.d_in;

  // ---- Phase 1: G[p0 .. p0+15][q] over all tokens.
  float g[SR];
#pragma unroll
  for (int i = 0; i < SR; ++i) g[i] = 0.0f;
  for (int k0 = 0; k0 < p.bt; k0 += TT) {
    __syncthreads();
    for (int e = t; e < TT * SR; e += 128) {
      const int kk = e / SR, ii = e % SR;
      const int tok = k0 + kk, row = p0 + ii;
      dys[kk][ii] = (tok < p.bt && row < p.d_out) ? p.dY[static_cast<int64_t>(tok) * p.ld_dy + row] : 0.0f;
    }
    __syncthreads();
    const int kn = min(TT, p.bt - k0);
    for (int kk = 0; kk < kn; ++kk) {
      const float x = qok ? p.X[static_cast<int64_t>(k0 + kk) * p.ld_x + q] : 0.0f;
#pragma unroll
      for (int i = 0; i < SR; ++i) g[i] = __fmaf_rn(dys[kk][i], x, g[i]);
    }
  }

  // ---- Phase 2 + 3.
  const StepScalars s = p.sc;
  float w1[SR], m1[SR], v1[SR];
  float sm_old[SR], sv_old[SR];
  const int jb = blockIdx.x;  // 8-bit block column
#pragma unroll
  for (int i = 0; i < SR; ++i) {
    const int row = p0 + i;
    w1[i] = m1[i] = v1[i] = 0.0f;
    sm_old[i] = sv_old[i] = 0.0f;
    if (row >= p.d_out) continue;
    if constexpr (MK == M_Q8) {
      sm_old[i] = p.m_scale[static_cast<int64_t>(jb) * p.d_out + row];
      if constexpr (TWO) sv_old[i] = p.v_scale[static_cast<int64_t>(jb) * p.d_out + row];
    }
    if (!qok) continue;
    float w = ld_val<WK == W_F32 ? 0 : 1>(p.W, static_cast<int64_t>(row) * p.ld_w + q);
    float m = 0.0f, v = 0.0f;
    if constexpr (MK == M_Q8) {
      m = dequant_m(small_int_to_f32(static_cast<const int8_t*>(p.m)[static_cast<int64_t>(row) * p.ld_m + q]),
                    sm_old[i]);
      if constexpr (TWO)
        v = dequant_v(small_int_to_f32(static_cast<const uint8_t*>(p.v)[static_cast<int64_t>(row) * p.ld_v + q]),
                      sv_old[i]);
    } else {
      if constexpr (NST >= 1) m = ld_val<MK == M_F32 ? 0 : 1>(p.m, static_cast<int64_t>(row) * p.ld_m + q);
      if constexpr (TWO) v = ld_val<MK == M_F32 ? 0 : 1>(p.v, static_cast<int64_t>(row) * p.ld_v + q);
    }
    step_elem<OPT>(g[i], w, m, v, s);
    w1[i] = w; m1[i] = m; v1[i] = v;
  }

  float sm_new[SR], sv_new[SR];
  if constexpr (MK == M_Q8) {
    // Block absmax of the new moments over the tile row (128 threads).
    const int warp = t >> 5, lane = t & 31;
#pragma unroll
    for (int i = 0; i < SR; ++i) {
      float am = fabsf(m1[i]);
      float au = TWO ? v1[i] : 0.0f;     // max v'; sqrt(max v') = max sqrt(v')
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, o));
        au = fmaxf(au, __shfl_xor_sync(0xFFFFFFFFu, au, o));
      }
      if (lane == 0) { red[0][warp][i] = am; red[1][warp][i] = au; }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < SR; ++i) {
      const float am = fmaxf(fmaxf(red[0][0][i], red[0][1][i]), fmaxf(red[0][2][i], red[0][3][i]));
      const float au = fmaxf(fmaxf(red[1][0][i], red[1][1][i]), fmaxf(red[1][2][i], red[1][3][i]));
      sm_new[i] = __fdiv_rn(am, 127.0f);
      sv_new[i] = __fdiv_rn(__fsqrt_rn(au), 255.0f);
    }
    __syncthreads();  // every thread has read the old scales and the reduction
    if (t == 0) {
      for (int i = 0; i < SR; ++i) {
        const int row = p0 + i;
        if (row >= p.d_out) continue;
        p.m_scale[static_cast<int64_t>(jb) * p.d_out + row] = sm_new[i];
        if constexpr (TWO) p.v_scale[static_cast<int64_t>(jb) * p.d_out + row] = sv_new[i];
      }
    }
  }

  if (!qok) return;
#pragma unroll
  for (int i = 0; i < SR; ++i) {
    const int row = p0 + i;
    if (row >= p.d_out) continue;
    const uint64_t idx = static_cast<uint64_t>(row) * static_cast<uint64_t>(p.d_in) + q;
    if constexpr (WK == W_F32) {
      static_cast<float*>(p.W)[static_cast<int64_t>(row) * p.ld_w + q] = w1[i];
    } else {
      const uint32_t b = p.sr_w ? f32_to_bf16_sr(w1[i], draw16(idx, p.step, 0u, p.seed_lo, p.seed_hi))
                                : f32_to_bf16_rne(w1[i]);
      static_cast<uint16_t*>(p.W)[static_cast<int64_t>(row) * p.ld_w + q] = static_cast<uint16_t>(b);
    }
    if constexpr (NST == 0) {
    } else if constexpr (MK == M_F32) {
      static_cast<float*>(p.m)[static_cast<int64_t>(row) * p.ld_m + q] = m1[i];
      if constexpr (TWO) static_cast<float*>(p.v)[static_cast<int64_t>(row) * p.ld_v + q] = v1[i];
    } else if constexpr (MK == M_BF16) {
      const uint32_t bm = p.sr_m ? f32_to_bf16_sr(m1[i], draw16(idx, p.step, 1u, p.seed_lo, p.seed_hi))
                                 : f32_to_bf16_rne(m1[i]);
      static_cast<uint16_t*>(p.m)[static_cast<int64_t>(row) * p.ld_m + q] = static_cast<uint16_t>(bm);
      if constexpr (TWO) {
        const uint32_t bv = p.sr_m ? f32_to_bf16_sr(v1[i], draw16(idx, p.step, 2u, p.seed_lo, p.seed_hi))
                                   : f32_to_bf16_rne(v1[i]);
        static_cast<uint16_t*>(p.v)[static_cast<int64_t>(row) * p.ld_v + q] = static_cast<uint16_t>(bv);
      }
    } else {
      static_cast<int8_t*>(p.m)[static_cast<int64_t>(row) * p.ld_m + q] =
          static_cast<int8_t>(quant_m(m1[i], sm_new[i], block_inv(sm_new[i])));
      if constexpr (TWO)
        static_cast<uint8_t*>(p.v)[static_cast<int64_t>(row) * p.ld_v + q] =
            static_cast<uint8_t>(quant_v(v1[i], __fsqrt_rn(v1[i]), sv_new[i], block_inv(sv_new[i])));
    }
  }
}

template <int OPT, int WK, int MK>
cudaError_t launch3(const WgradSimtParams& p, cudaStream_t stream) {
  const dim3 grid((p.d_in + SC - 1) / SC, (p.d_out + SR - 1) / SR);
  wgrad_step_simt_kernel<OPT, WK, MK><<<grid, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

template <int OPT, int WK>
cudaError_t launch2(const WgradSimtParams& p, int mk, cudaStream_t stream) {
  if (mk == M_F32) return launch3<OPT, WK, M_F32>(p, stream);
  if (mk == M_BF16) return launch3<OPT, WK, M_BF16>(p, stream);
  if constexpr (OPT == OPT_ADAMW || OPT == OPT_SGDM || OPT == OPT_LION)
    if (mk == M_Q8) return launch3<OPT, WK, M_Q8>(p, stream);
  return cudaErrorInvalidValue;
}

template <int OPT>
cudaError_t launch1(const WgradSimtParams& p, int wk, int mk, cudaStream_t stream) {
  return wk == W_F32 ? launch2<OPT, W_F32>(p, mk, stream) : launch2<OPT, W_BF16>(p, mk, stream);
}

}  // namespace

cudaError_t launch_wgrad_simt(const WgradSimtParams& p, int opt, int wk, int mk, cudaStream_t stream) {
  if (opt == OPT_ADAMW) return launch1<OPT_ADAMW>(p, wk, mk, stream);
  if (opt == OPT_SGDM) return launch1<OPT_SGDM>(p, wk, mk, stream);
  if (opt == OPT_LION) return launch1<OPT_LION>(p, wk, mk, stream);
  if (opt == OPT_SGD) return launch1<OPT_SGD>(p, wk, mk, stream);
  if (opt == OPT_RMSPROP) return launch1<OPT_RMSPROP>(p, wk, mk, stream);
  if (opt == OPT_ADAGRAD) return launch1<OPT_ADAGRAD>(p, wk, mk, stream);
  if (opt == OPT_NADAM) return launch1<OPT_NADAM>(p, wk, mk, stream);
  if (opt == OPT_RADAM) return launch1<OPT_RADAM>(p, wk, mk, stream);
  return cudaErrorInvalidValue;
}

}  // namespace forge
