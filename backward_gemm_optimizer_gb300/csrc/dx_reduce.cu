// dx_reduce.cu -- the second half of the fused backward pass: the input
// gradient dX = dY W_old (FORGE, Appendix A, Remark 1) arrives from the
// fused kernel as fp32 partial sums, one slab per (CTA, tile column) that
// CTA visited; this kernel adds a column's slabs in increasing CTA order --
// a fixed order, so dX is bit-reproducible -- and stores dX.
//
// The fused kernel's CTA c owns the contiguous tile range
// [c T / G, (c + 1) T / G) of the column-major tile order (T tiles, G CTAs,
// tiles_m tiles per column), so the CTAs that touched column q are
// owner(q tiles_m) .. owner(q tiles_m + tiles_m - 1), with
// owner(L) = floor(((L + 1) G - 1) / T), and the slot of column q in CTA c's
// slab list is q - floor(first tile of c / tiles_m).
#include <cstdint>

#include "forge_math.cuh"
#include "forge_params.h"

namespace forge {

namespace {

constexpr int kBN = 64;  // columns per tile of the fused kernel

// One block per (tile column q, 64 tokens): 64 x 64 outputs, four float4
// per thread; consecutive threads read consecutive 16-byte pieces of a
// token's 256-byte slab row.
constexpr int kTokens = 64;

__global__ void __launch_bounds__(256) dx_reduce_kernel(const DxReduceParams p) {
  // Launched as a programmatic dependent of the fused kernel: the blocks may
  // start while it finishes; its slab writes are visible after this wait.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int q = blockIdx.x;
  const int t0 = blockIdx.y * kTokens;
  const int64_t T = p.num_tiles, G = p.grid;
  const int64_t l0 = static_cast<int64_t>(q) * p.tiles_m;
  const int64_t l1 = l0 + p.tiles_m - 1;
  const int64_t c0 = ((l0 + 1) * G - 1) / T, c1 = ((l1 + 1) * G - 1) / T;
  const int col = (threadIdx.x & 15) * 4;
  const int i = q * kBN + col;
  float4 acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  // Two slabs' loads in flight per thread, added in increasing CTA order.
  for (int64_t c = c0; c <= c1; c += 2) {
    float4 v[2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int64_t cc = c + u;
      const float* slab =
          cc <= c1 ? p.ws + (cc * p.runs + (q - (cc * T / G) / p.tiles_m)) * p.slab + col : nullptr;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int t = t0 + (threadIdx.x >> 4) + 16 * k;
        v[u][k] = (slab != nullptr && t < p.bt)
                      ? __ldcg(reinterpret_cast<const float4*>(slab + static_cast<int64_t>(t) * kBN))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (c + u > c1) break;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[k].x = __fadd_rn(acc[k].x, v[u][k].x);
        acc[k].y = __fadd_rn(acc[k].y, v[u][k].y);
        acc[k].z = __fadd_rn(acc[k].z, v[u][k].z);
        acc[k].w = __fadd_rn(acc[k].w, v[u][k].w);
      }
    }
  }
  if (i >= p.d_in) return;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int t = t0 + (threadIdx.x >> 4) + 16 * k;
    if (t >= p.bt) continue;
    if (p.dx_bf16) {
      uint2* out = reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.dX) + static_cast<int64_t>(t) * p.ld_dx + i);
      *out = make_uint2(pack_bf16x2_rn(acc[k].x, acc[k].y), pack_bf16x2_rn(acc[k].z, acc[k].w));
    } else {
      *reinterpret_cast<float4*>(static_cast<float*>(p.dX) + static_cast<int64_t>(t) * p.ld_dx + i) = acc[k];
    }
  }
}

}  // namespace

cudaError_t launch_dx_reduce(const DxReduceParams& p, int, cudaStream_t stream) {
  if (p.bt == 0 || p.d_in == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((p.d_in + kBN - 1) / kBN), static_cast<unsigned>((p.bt + kTokens - 1) / kTokens));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, dx_reduce_kernel, p);
}

}  // namespace forge
