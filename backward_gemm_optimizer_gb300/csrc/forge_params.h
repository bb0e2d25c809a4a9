// forge_params.h -- kernel parameter blocks and launcher declarations
// shared between the C-ABI translation unit and the kernel translation
// units. Host and device code both include it.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "forge_math.cuh"

namespace forge {

// Device status word codes (first failure wins). The low byte names the
// wait that gave up.
enum : uint32_t {
  STATUS_OK = 0,
  WAIT_OP_EMPTY = 0xF001,     // operand producer: free operand stage
  WAIT_OP_FULL = 0xF002,      // MMA issuer: operand stage landed
  WAIT_TMEM_EMPTY = 0xF003,   // MMA issuer: accumulator buffer drained
  WAIT_ST_EMPTY = 0xF004,     // state producer: free state slot
  WAIT_ST_WRITTEN = 0xF005,   // state storer: epilogue finished a slot
  WAIT_TMEM_FULL = 0xF006,    // epilogue: accumulator ready
  WAIT_ST_FULL = 0xF007,      // epilogue: state slot landed
  WAIT_RED = 0xF008,          // epilogue: 8-bit block absmax exchange
  WAIT_TEST_HOOK = 0xF009,    // epilogue: the forced-timeout test barrier
  WAIT_MMA_DRAIN = 0xF00A,    // MMA issuer: in-flight MMAs after an abort
  WAIT_DRAIN = 0xF00B,        // a producer's in-flight loads after an abort
  WAIT_WB_FULL = 0xF00C,      // MMA issuer: bf16 W_old tile converted (fused dX)
  WAIT_WB_EMPTY = 0xF00D,     // converters: previous W_old tile consumed
  WAIT_DX_FULL = 0xF00E,      // converters: dX partial complete
  WAIT_DX_EMPTY = 0xF00F,     // MMA issuer: dX partial written out
};

constexpr uint32_t FLAG_TILE_N_MASK = 7u;
constexpr uint32_t FLAG_TEST_FORCE_TIMEOUT = 0x100u;

// Tensor-core fused step (bf16 X / dY).
struct alignas(128) WgradTcParams {
  CUtensorMap tm_dy;  // dY  [BT][D_out] bf16, box 64 x 64, 128-byte swizzle
  CUtensorMap tm_x;   // X   [BT][D_in]  bf16, box 64 x 64, 128-byte swizzle
  CUtensorMap tm_w;   // W   [D_out][D_in], box 32 cols x 128 rows
  CUtensorMap tm_m;   // m   (values or 8-bit codes), box 32 x 128
  CUtensorMap tm_v;   // v   (AdamW only)
  CUtensorMap tm_g;   // G_acc fp32 [D_out][D_in], box 32 x 128 (accumulated-gradient step only)
  StepScalars sc;
  float* m_scale;     // 8-bit state: [D_in/128][D_out]
  float* v_scale;
  unsigned int* status;
  int d_out, d_in, bt;
  int tiles_m, tiles_n, num_tiles, num_kb;
  int group_m;
  uint32_t step, seed_lo, seed_hi;
  int sr_w, sr_m;
  uint32_t flags;
  uint64_t timeout_ns;
  // Operand residency: with op_hint the X / dY loads carry an L2 evict-last
  // policy (every tile of a column / row re-reads them, while the state
  // streams through L2 once); at the end each CTA returns its share of the
  // operands' whole 128-byte lines, [op_lo[i], op_hi[i]), to normal priority.
  int op_hint;
  const uint8_t* op_lo[2];
  const uint8_t* op_hi[2];
  // Fused input gradient (DX kernels only).
  void* w_ptr;        // W_old, read by the converters
  int64_t ld_w;
  float* dx_ws;       // workspace: [grid][dx_runs] slabs of dx_slab floats
  int dx_runs;        // column runs per CTA (slab slots)
  int64_t dx_slab;    // floats per slab: num_kb * 128 * 64
  int dx_l2;          // 1: slabs are stored evict-last (the reduction reads them from L2 and drops them)
};

// Deterministic reduction of the dX partial slabs into dX.
struct DxReduceParams {
  const float* ws;
  void* dX;
  int64_t ld_dx;
  int dx_bf16;
  int bt, d_in;
  int tiles_m, num_tiles, grid, runs;
  int64_t slab;
  int discard;        // 1: drop each slab line from L2 once read (the slabs are dead scratch)
};

// fp32 fused step (fp32 X / dY), plain CUDA cores.
struct WgradSimtParams {
  const float* X;
  const float* dY;
  void* W;
  void* m;
  void* v;
  float* m_scale;
  float* v_scale;
  int64_t ld_x, ld_dy, ld_w, ld_m, ld_v;
  int d_out, d_in, bt;
  StepScalars sc;
  uint32_t step, seed_lo, seed_hi;
  int sr_w, sr_m;
};

// Input gradient dX = dY W (tensor cores).
struct alignas(128) DgradParams {
  CUtensorMap tm_dy;  // dY [BT][D_out] bf16, box 64 (K) x 128 (M rows), 128-byte swizzle
  CUtensorMap tm_w;   // W [D_out][D_in]: bf16, box 64 (N) x bk (K); or fp32, box 32 (N) x stg_rows (K); 128-byte swizzle
  const float* w_f32; // W fp32 (staged and rounded to bf16 by the kernel) or null
  int64_t ld_w32;
  void* dX;           // [BT][D_in]
  int64_t ld_dx;
  int dx_bf16;
  unsigned int* status;
  int bt, d_out, d_in;
  int tiles_m, tiles_n, num_tiles, num_kb;
  int group_m;
  int bn;             // tile width (input features): 128, or 256 for bf16 W
  int bk;             // rows of D_out per stage (128, or 64 with bn 256 or mb > 1); must match the kernel's
  int mb;             // 128-token blocks per tile: 1, or 2 / 4 (all tokens of BT <= 256 / 512; tiles_m = 1)
  int stg_rows;       // fp32 W: rows per staging slot (64, or 32 with mb > 1); must match the kernel's
  int k_rotate;       // 1: tiles of a row start their stage walks at evenly spaced stages
  uint32_t flags;
  uint64_t timeout_ns;
  // Split contraction (splitk = S >= 2; grid = num_tiles * S): CTA c runs
  // stages [s num_kb / S, (s + 1) num_kb / S) of tile c % num_tiles,
  // s = c / num_tiles, and stores its fp32 partial sum to
  // part + c * mb * 128 * bn (mb * 128 x bn, row-major); dgrad_fixup_kernel
  // adds a tile's parts in order.
  int splitk;
  float* part;
};

// Sum of the partial tiles of a split dgrad (see DgradParams::splitk).
struct DgradFixupParams {
  const float* part;
  void* dX;
  int64_t ld_dx;
  int dx_bf16;
  int bt, d_in;
  int bn, tiles_m, tiles_n, group_m, num_tiles, parts;
  int rows;  // token rows per tile (mb * 128)
};

struct TcLaunch {
  int opt, wk, mk;
  int bn;       // tile width (64, 128 or 256)
  int deep;     // 1: deeper operand pipeline for long token axes
  int dx;       // 1: fused input gradient (64-column tiles, fp32 / bf16 state)
  int ga;       // 1: add the accumulated gradient G_acc (tm_g) to each tile
  int narrow;   // 1: 16-column state chunks (fused kernel, fp32 W and moments, short token axes)
  int wide;     // 1: 64-column state chunks (plain step, bf16 W and bf16 moments)
  int pair;     // CTA pairs on 256 x 256 tiles (plain step, bn 256; grid = 2 x pairs): 0, or their operand stages (4, 5)
  int grid;
  cudaStream_t stream;
};

// Defined in the kernel translation units.
cudaError_t launch_wgrad_tc_adamw(const WgradTcParams& p, const TcLaunch& l);
cudaError_t launch_wgrad_tc_sgdm(const WgradTcParams& p, const TcLaunch& l);
cudaError_t launch_wgrad_tc_lion(const WgradTcParams& p, const TcLaunch& l);
cudaError_t launch_wgrad_tc_sgd(const WgradTcParams& p, const TcLaunch& l);
cudaError_t launch_wgrad_tc_rmsprop(const WgradTcParams& p, const TcLaunch& l);
cudaError_t launch_wgrad_tc_adagrad(const WgradTcParams& p, const TcLaunch& l);
cudaError_t launch_wgrad_tc_nadam(const WgradTcParams& p, const TcLaunch& l);
cudaError_t launch_wgrad_tc_radam(const WgradTcParams& p, const TcLaunch& l);
cudaError_t launch_wgrad_tc_accum(const WgradTcParams& p, const TcLaunch& l);
cudaError_t launch_wgrad_simt(const WgradSimtParams& p, int opt, int wk, int mk, cudaStream_t stream);
cudaError_t launch_dgrad_tc(const DgradParams& p, int grid, cudaStream_t stream);
cudaError_t launch_dgrad_fixup(const DgradFixupParams& p, cudaStream_t stream);
cudaError_t launch_dx_reduce(const DxReduceParams& p, int sms, cudaStream_t stream);

// Whether a (opt, wk, mk, bn, deep) variant has a tensor-core kernel.
bool wgrad_tc_supported(int opt, int wk, int mk, int bn, int deep);

}  // namespace forge
