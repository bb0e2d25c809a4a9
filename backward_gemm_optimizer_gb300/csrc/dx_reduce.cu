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
//
// When the fused kernel stored the slabs evict-last (small slab sets), they
// are read here from L2 and, with `discard`, each line is then dropped from
// L2 (the slabs are dead scratch), so that it is never written back to DRAM.
#include <cstdint>

#include "forge_math.cuh"
#include "forge_params.h"
#include "forge_ptx.cuh"

namespace forge {

namespace {

constexpr int kBN = 64;      // columns per tile of the fused kernel
constexpr int kTokens = 32;  // token rows per block
constexpr int kSlabsInFlight = 4;

// One block per (tile column q, 32 tokens): 16 threads per token row (4
// columns each, consecutive 16-byte pieces of a 256-byte slab row), each
// thread two rows; the loads of up to four slabs are in flight before they
// are added in increasing CTA order (up-projection BT 512, fused backward
// pass: 296.6 -> 283 us against one block per 64 tokens with two slabs in
// flight).
__global__ void __launch_bounds__(256) dx_reduce_kernel(const DxReduceParams p) {
  // Launched as a programmatic dependent of the fused kernel: the blocks may
  // start while it finishes; its slab writes are visible after this wait.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // The next kernel may be scheduled once every block is running.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int q = blockIdx.x;
  const int64_t T = p.num_tiles, G = p.grid;
  const int64_t l0 = static_cast<int64_t>(q) * p.tiles_m;
  const int64_t l1 = l0 + p.tiles_m - 1;
  const int c0 = static_cast<int>(((l0 + 1) * G - 1) / T), c1 = static_cast<int>(((l1 + 1) * G - 1) / T);
  const int col = (threadIdx.x & 15) * 4;
  const int i = q * kBN + col;
  const int row0 = static_cast<int>(blockIdx.y) * kTokens + static_cast<int>(threadIdx.x >> 4);
  float4 acc[2];
  acc[0] = acc[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c = c0; c <= c1; c += kSlabsInFlight) {
    float4 v[kSlabsInFlight][2];
#pragma unroll
    for (int u = 0; u < kSlabsInFlight; ++u) {
      const int cc = c + u;
      const float* slab =
          p.ws + (static_cast<int64_t>(cc) * p.runs + (q - (static_cast<int64_t>(cc) * T / G) / p.tiles_m)) * p.slab +
          col;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int t = row0 + 16 * k;
        v[u][k] = (cc <= c1 && t < p.bt)
                      ? __ldcg(reinterpret_cast<const float4*>(slab + static_cast<int64_t>(t) * kBN))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < kSlabsInFlight; ++u) {
      if (c + u > c1) break;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        acc[k].x = __fadd_rn(acc[k].x, v[u][k].x);
        acc[k].y = __fadd_rn(acc[k].y, v[u][k].y);
        acc[k].z = __fadd_rn(acc[k].z, v[u][k].z);
        acc[k].w = __fadd_rn(acc[k].w, v[u][k].w);
      }
    }
  }
  if (i < p.d_in) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int t = row0 + 16 * k;
      if (t >= p.bt) continue;
      if (p.dx_bf16) {
        uint2* out = reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.dX) + static_cast<int64_t>(t) * p.ld_dx + i);
        *out = make_uint2(pack_bf16x2_rn(acc[k].x, acc[k].y), pack_bf16x2_rn(acc[k].z, acc[k].w));
      } else {
        *reinterpret_cast<float4*>(static_cast<float*>(p.dX) + static_cast<int64_t>(t) * p.ld_dx + i) = acc[k];
      }
    }
  }
  if (p.discard) {
    // Every slab row of this block -- token rows past BT included, which the
    // fused kernel wrote too -- has been read by this block only.
    __syncthreads();
    if ((threadIdx.x & 7) == 0) {
      for (int c = c0; c <= c1; ++c) {
        const float* slab =
            p.ws + (static_cast<int64_t>(c) * p.runs + (q - (static_cast<int64_t>(c) * T / G) / p.tiles_m)) * p.slab +
            col;
#pragma unroll
        for (int k = 0; k < 2; ++k) l2_discard_line(slab + static_cast<int64_t>(row0 + 16 * k) * kBN);
      }
    }
  }
}

}  // namespace

cudaError_t launch_dx_reduce(const DxReduceParams& p, int, cudaStream_t stream) {
  if (p.bt == 0 || p.d_in == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  // With discard, the blocks cover every slab row the fused kernel wrote
  // (ceil(BT / 128) * 128); otherwise the rows of dX.
  const int64_t rows = p.discard ? p.slab / kBN : p.bt;
  cfg.gridDim = dim3(static_cast<unsigned>((p.d_in + kBN - 1) / kBN), static_cast<unsigned>((rows + kTokens - 1) / kTokens));
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
