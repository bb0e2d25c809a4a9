// forge_selftest.cu -- enumeration checks of the branch-free divide and
// square root of forge_math.cuh against the correctly rounded hardware
// operations (__fsqrt_rn, __frcp_rn, __fdiv_rn), behind
// forge_selftest_math in include/forge.h. Each launch walks a range of
// cases with a grid-stride loop, counts disagreements and values the fast
// path declines (outside its range), and touches no memory but two
// counters.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/forge.h"
#include "forge_math.cuh"

namespace forge {
namespace {

__device__ unsigned long long g_counts[2];   // mismatches, declined

__device__ __forceinline__ void add_counts(unsigned long long mism, unsigned long long declined) {
  if (mism) atomicAdd(&g_counts[0], mism);
  if (declined) atomicAdd(&g_counts[1], declined);
}

// Every float whose bit pattern is in [first, first + count): sqrt_fast
// against __fsqrt_rn inside [2^-100, 2^100] (the rest counted as declined).
__global__ void __launch_bounds__(256) sqrt_check_kernel(uint64_t first, uint64_t count) {
  unsigned long long mism = 0, declined = 0;
  for (uint64_t i = blockIdx.x * 256ull + threadIdx.x; i < count; i += 256ull * gridDim.x) {
    const float x = __uint_as_float(static_cast<uint32_t>(first + i));
    if (!(x >= 0x1p-100f && x <= 0x1p100f)) { ++declined; continue; }
    if (__float_as_uint(sqrt_fast(x)) != __float_as_uint(__fsqrt_rn(x))) ++mism;
  }
  add_counts(mism, declined);
}

// Every divisor whose bit pattern is in [first, first + count): the refined
// reciprocal against __frcp_rn (inside the quotient's divisor range).
__global__ void __launch_bounds__(256) rcp_check_kernel(uint64_t first, uint64_t count) {
  unsigned long long mism = 0, declined = 0;
  for (uint64_t i = blockIdx.x * 256ull + threadIdx.x; i < count; i += 256ull * gridDim.x) {
    const float d = __uint_as_float(static_cast<uint32_t>(first + i));
    if (!(d >= 0x1p-60f && d <= 0x1p60f)) { ++declined; continue; }
    if (__float_as_uint(rcp_refined(d)) != __float_as_uint(__frcp_rn(d))) ++mism;
  }
  add_counts(mism, declined);
}

// Pairs of significands: case i is n = 1 + (i >> 23) 2^-23, d = 1 + (i mod
// 2^23) 2^-23, for i in [first, first + count) (2^46 cases in all): div_fast
// against __fdiv_rn.
__global__ void __launch_bounds__(256) div_check_kernel(uint64_t first, uint64_t count) {
  unsigned long long mism = 0, declined = 0;
  for (uint64_t i = blockIdx.x * 256ull + threadIdx.x; i < count; i += 256ull * gridDim.x) {
    const uint64_t c = first + i;
    const float n = __uint_as_float(0x3F800000u | static_cast<uint32_t>((c >> 23) & 0x7FFFFFu));
    const float d = __uint_as_float(0x3F800000u | static_cast<uint32_t>(c & 0x7FFFFFu));
    if (__float_as_uint(div_fast(n, d)) != __float_as_uint(__fdiv_rn(n, d))) ++mism;
  }
  add_counts(mism, declined);
}

}  // namespace
}  // namespace forge

extern "C" forge_status forge_selftest_math(int which, uint64_t first, uint64_t count, uint64_t* mismatches,
                                            uint64_t* declined) {
  using namespace forge;
  if (mismatches == nullptr || declined == nullptr || which < 0 || which > 2) return FORGE_ERR_INVALID_ARG;
  const uint64_t limit = which == 2 ? (1ull << 46) : (1ull << 32);
  if (first > limit || count > limit - first) return FORGE_ERR_INVALID_ARG;
  *mismatches = 0;
  *declined = 0;
  if (count == 0) return FORGE_OK;
  const unsigned long long zero[2] = {0ull, 0ull};
  if (cudaMemcpyToSymbol(g_counts, zero, sizeof(zero)) != cudaSuccess) return FORGE_ERR_CUDA;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FORGE_ERR_CUDA;
  const uint64_t blocks_needed = (count + 255) / 256;
  const unsigned grid = static_cast<unsigned>(blocks_needed < 8ull * sms ? blocks_needed : 8ull * sms);
  if (which == 0) sqrt_check_kernel<<<grid, 256>>>(first, count);
  else if (which == 1) rcp_check_kernel<<<grid, 256>>>(first, count);
  else div_check_kernel<<<grid, 256>>>(first, count);
  if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) return FORGE_ERR_CUDA;
  unsigned long long out[2];
  if (cudaMemcpyFromSymbol(out, g_counts, sizeof(out)) != cudaSuccess) return FORGE_ERR_CUDA;
  *mismatches = out[0];
  *declined = out[1];
  return FORGE_OK;
}
