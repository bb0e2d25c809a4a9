// dgrad_tc.cu -- input gradient dX = dY W_old on tcgen05 tensor cores
// (FORGE, Remark 1 in Appendix A: the input gradient must read the weights
// before the fused step overwrites them, so it is enqueued first).
//
// Tiles of 128 tokens x 128 input features; the contraction runs over
// D_out in 64-wide stages. A = dY is K-major (D_out contiguous), B = W is
// MN-major (D_in contiguous). bf16 weights are fed by TMA directly; fp32
// master weights are staged by TMA and four converter warps round them to
// bf16 (round-to-nearest-even) into the swizzled operand layout before the
// MMA consumes them.
//
// Warp roles (384 threads): 0 TMA producer, 1 MMA issuer + TMEM owner,
// 4-7 epilogue (TMEM lane quadrant = warp % 4, thread = token row),
// 8-11 converters (fp32 weights only). All waits are bounded.
#include <cstdint>

#include "forge_math.cuh"
#include "forge_params.h"
#include "forge_ptx.cuh"

namespace forge {

namespace {

constexpr int BM = 128, BN = 128, BK = 64;
constexpr int A_BYTES = BM * BK * 2;       // 16 KB
constexpr int B_BYTES = BK * BN * 2;       // 16 KB
constexpr int STG_BYTES = BK * BN * 4;     // 32 KB: fp32 W tile as four 32-column swizzled boxes
constexpr int TMEM_COLS = 256;
constexpr uint32_t IDESC = make_idesc_bf16(BM, BN, 0, 1);

template <bool F32W>
struct DCfg {
  static constexpr int STAGES = F32W ? 3 : 4;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + (F32W ? STG_BYTES : 0);
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES;
};

__device__ __forceinline__ bool dwait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                      unsigned int* status, uint32_t code, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 7u) == 0u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        atomicCAS(status, 0u, code);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void dtile(int tile, int tiles_m, int tiles_n, int group_m, int& tm, int& tn) {
  const int per_group = group_m * tiles_n;
  const int g = tile / per_group;
  const int first_m = g * group_m;
  const int rem = tiles_m - first_m;
  const int gsize = rem < group_m ? rem : group_m;
  const int in_g = tile - g * per_group;
  tm = first_m + in_g % gsize;
  tn = in_g / gsize;
}

template <bool F32W>
__global__ void __launch_bounds__(384, 1) dgrad_tc_kernel(const __grid_constant__ DgradParams p) {
  using C = DCfg<F32W>;
  constexpr int S = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[S], conv[S], empty[S];
  __shared__ __align__(8) uint64_t tm_full[2], tm_empty[2], drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &abort_sh;
  const uint64_t lim = p.timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&conv[s], 128);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) { mbar_init(&tm_full[b], 1); mbar_init(&tm_empty[b], 4); }
    mbar_init(&drain_bar, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) { prefetch_tmap(&p.tm_dy); prefetch_tmap(&p.tm_w); }
  if (warp == 1) { tmem_alloc(&tmem_base_sh, TMEM_COLS); tmem_relinquish(); }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = tmem_base_sh;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t kseq = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        int tm, tn;
        dtile(tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
        for (int kb = 0; kb < p.num_kb; ++kb, ++kseq) {
          const int s = static_cast<int>(kseq % S);
          if (!dwait(&empty[s], ((kseq / S) & 1u) ^ 1u, abort_flag, p.status, WAIT_OP_EMPTY, lim)) {
            ok = false;
            break;
          }
          uint8_t* a = smem + s * C::STAGE_BYTES;
          uint8_t* b = a + A_BYTES;
          if constexpr (F32W) {
            uint8_t* stg = b + B_BYTES;
            mbar_arrive_expect_tx(&full[s], A_BYTES + STG_BYTES);
            tma_load_2d(a, &p.tm_dy, &full[s], kb * BK, tm * BM);
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) tma_load_2d(stg + bb * 8192, &p.tm_w, &full[s], tn * BN + bb * 32, kb * BK);
          } else {
            mbar_arrive_expect_tx(&full[s], A_BYTES + B_BYTES);
            tma_load_2d(a, &p.tm_dy, &full[s], kb * BK, tm * BM);
            tma_load_2d(b, &p.tm_w, &full[s], tn * BN, kb * BK);
            tma_load_2d(b + 8192, &p.tm_w, &full[s], tn * BN + 64, kb * BK);
          }
        }
      }
      if (!ok) {
        const uint32_t first = kseq > static_cast<uint32_t>(S) ? kseq - S : 0u;
        for (uint32_t k = first; k < kseq; ++k) {
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(&full[k % S], (k / S) & 1u))
            if (globaltimer_ns() - t0 > 200000000ull) { atomicCAS(p.status, 0u, WAIT_DRAIN); break; }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t kseq = 0;
      bool ok = true;
      int it = 0;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x, ++it) {
        const int buf = it & 1;
        if (!dwait(&tm_empty[buf], ((it >> 1) & 1) ^ 1u, abort_flag, p.status, WAIT_TMEM_EMPTY, lim)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d = tmem_base + static_cast<uint32_t>(buf * BN);
        for (int kb = 0; kb < p.num_kb; ++kb, ++kseq) {
          const int s = static_cast<int>(kseq % S);
          const uint32_t ph = (kseq / S) & 1u;
          uint64_t* ready = F32W ? &conv[s] : &full[s];
          if (!dwait(ready, ph, abort_flag, p.status, WAIT_OP_FULL, lim)) { ok = false; break; }
          tc_fence_after_sync();
          const uint32_t a0 = smem_u32(smem + s * C::STAGE_BYTES);
          const uint32_t b0 = a0 + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // A: K-major, 128-byte swizzle, 8-row groups 1024 bytes apart; a
            // K step of 16 elements advances the start by 32 bytes.
            const uint64_t ad = make_smem_desc(a0 + kk * 32, 16, 1024, 2);
            // B: MN-major, 64-column atoms 8192 bytes apart, 8-row K groups of 1024 bytes.
            const uint64_t bd = make_smem_desc(b0 + kk * 2048, 8192, 1024, 2);
            umma_f16(d, ad, bd, IDESC, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&empty[s]);
        }
        if (!ok) break;
        umma_commit(&tm_full[buf]);
      }
      if (!ok) {
        umma_commit(&drain_bar);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&drain_bar, 0))
          if (globaltimer_ns() - t0 > 200000000ull) { atomicCAS(p.status, 0u, WAIT_MMA_DRAIN); break; }
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int r = q * 32 + lane;
    int it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x, ++it) {
      int tm, tn;
      dtile(tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
      const int buf = it & 1;
      ok = dwait(&tm_full[buf], (it >> 1) & 1, abort_flag, p.status, WAIT_TMEM_FULL, lim);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      const int row = tm * BM + r;
      const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * BN);
#pragma unroll 1
      for (int c = 0; c < BN / 16; ++c) {
        uint32_t acc[16];
        if (p.num_kb > 0) {
          tmem_ld_32x32b_x16(t_lane + c * 16, acc);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[j] = 0u;
        }
        const int col0 = tn * BN + c * 16;
        if (row >= p.bt || col0 >= p.d_in) continue;
        const bool full_chunk = col0 + 16 <= p.d_in;
        if (p.dx_bf16) {
          uint16_t* out = static_cast<uint16_t*>(p.dX) + static_cast<int64_t>(row) * p.ld_dx + col0;
          if (full_chunk) {
            uint32_t b[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
              b[j] = f32_to_bf16_rne(__uint_as_float(acc[2 * j])) |
                     (f32_to_bf16_rne(__uint_as_float(acc[2 * j + 1])) << 16);
            reinterpret_cast<uint4*>(out)[0] = make_uint4(b[0], b[1], b[2], b[3]);
            reinterpret_cast<uint4*>(out)[1] = make_uint4(b[4], b[5], b[6], b[7]);
          } else {
            for (int j = 0; j < 16 && col0 + j < p.d_in; ++j)
              out[j] = static_cast<uint16_t>(f32_to_bf16_rne(__uint_as_float(acc[j])));
          }
        } else {
          float* out = static_cast<float*>(p.dX) + static_cast<int64_t>(row) * p.ld_dx + col0;
          if (full_chunk) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              reinterpret_cast<float4*>(out)[j] =
                  make_float4(__uint_as_float(acc[4 * j]), __uint_as_float(acc[4 * j + 1]),
                              __uint_as_float(acc[4 * j + 2]), __uint_as_float(acc[4 * j + 3]));
          } else {
            for (int j = 0; j < 16 && col0 + j < p.d_in; ++j) out[j] = __uint_as_float(acc[j]);
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tm_empty[buf]);
    }
  } else if (warp >= 8 && F32W) {
    // ------------------------------------------------------------ fp32 -> bf16 converters
    // The fp32 tile landed by TMA as four [64 rows][32 columns] boxes with
    // the 128-byte swizzle. Work item = (box, K row, 8-column group): read
    // two 16-byte chunks, round to bf16, write one 16-byte chunk of the
    // MN-major swizzled operand. Consecutive threads take consecutive K
    // rows, so both the reads and the writes are bank-conflict free.
    const int ct = threadIdx.x - 256;
    uint32_t kseq = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
      for (int kb = 0; kb < p.num_kb; ++kb, ++kseq) {
        const int s = static_cast<int>(kseq % S);
        const uint32_t ph = (kseq / S) & 1u;
        ok = dwait(&full[s], ph, abort_flag, p.status, WAIT_OP_FULL, lim);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) break;
        uint8_t* b = smem + s * C::STAGE_BYTES + A_BYTES;
        const uint8_t* stg = b + B_BYTES;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int i = ct + 128 * j;
          const int k = i & 63;              // K row
          const int hh = (i >> 6) & 3;       // 8-column group within the 32-column box
          const int bb = i >> 8;             // box (32 columns)
          const uint8_t* src = stg + bb * 8192 + k * 128;
          const float4 u0 = *reinterpret_cast<const float4*>(src + (((2 * hh) ^ (k & 7)) << 4));
          const float4 u1 = *reinterpret_cast<const float4*>(src + (((2 * hh + 1) ^ (k & 7)) << 4));
          uint4 o;
          o.x = f32_to_bf16_rne(u0.x) | (f32_to_bf16_rne(u0.y) << 16);
          o.y = f32_to_bf16_rne(u0.z) | (f32_to_bf16_rne(u0.w) << 16);
          o.z = f32_to_bf16_rne(u1.x) | (f32_to_bf16_rne(u1.y) << 16);
          o.w = f32_to_bf16_rne(u1.z) | (f32_to_bf16_rne(u1.w) << 16);
          const int n = bb * 32 + hh * 8;    // column within the 128-wide tile
          const int atom = n >> 6;
          const int chunk = ((n & 63) >> 3) ^ (k & 7);
          *reinterpret_cast<uint4*>(b + atom * 8192 + k * 128 + (chunk << 4)) = o;
        }
        fence_proxy_async_smem();
        mbar_arrive(&conv[s]);
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <bool F32W>
cudaError_t launch_d(const DgradParams& p, int grid, cudaStream_t stream) {
  auto kern = dgrad_tc_kernel<F32W>;
  static unsigned long long attr_mask = 0ull;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(__atomic_load_n(&attr_mask, __ATOMIC_ACQUIRE) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DCfg<F32W>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&attr_mask, bit, __ATOMIC_ACQ_REL);
  }
  kern<<<grid, 384, DCfg<F32W>::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dgrad_tc(const DgradParams& p, int grid, cudaStream_t stream) {
  return p.w_f32 ? launch_d<true>(p, grid, stream) : launch_d<false>(p, grid, stream);
}

}  // namespace forge
