// wgrad_tc.cuh -- the fused weight-gradient + optimizer-step kernel for
// sm_103a (FORGE, Algorithm 1, re-designed for tcgen05 tensor cores).
//
// One persistent CTA per SM walks a grouped raster of 128 x BN gradient
// tiles G_ij = sum_k dY_k,i^T X_k,j (Eq. 5), BN = 64, 128 or 256. Warp
// roles (640 threads; 768 or 800 with the fused input gradient, below):
//
//   warp 0      operand producer: TMA loads of the BK-token slabs of dY and
//               X (BK = 64, or 128 with the fused input gradient) into a
//               STAGES-deep shared-memory ring;
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M = 128, N = BN,
//               K = 16) into a double-buffered fp32 TMEM accumulator; the
//               warp also owns the TMEM allocation;
//   warp 2      state producer: TMA loads of the W / m / v tiles (and of an
//               accumulated gradient G_acc, GA), in CW-column chunks
//               (CW = 32, or 16: NARROW), into an NBUF-deep slot ring;
//   warp 3      state storer: TMA stores of each finished chunk;
//   warps 4-19  epilogue: warp w reads TMEM lane quadrant w % 4 (row p of
//               the tile = TMEM lane) and column quarter (w - 4) / 4 of each
//               chunk, applies the optimizer element-wise in fp32 and writes
//               the new W / m / v back into the slot (Algorithm 1 phase 2-3).
//               Four epilogue warps per scheduler hide the latency of the
//               per-element arithmetic (divide, square root, Philox rounds).
//
// The same template serves gradient accumulation over micro-batches
// (Appendix L): with the OPT_ACCUM / OPT_ACCSET rules the "weight" is an fp32
// accumulator G_acc that the tile is added to (or written to), and with GA
// the step of any rule adds a streamed G_acc chunk to each tile first.
//
// With DX (the fused backward pass) the same kernel also forms the input
// gradient dX = dY W_old from the W tile it is about to update (Appendix A,
// Remark 1: dX must see the weights before the step):
//
//   * operand stages hold 128 tokens, so each dY stage serves both
//     products -- read MN-major as the A operand of G = dY^T X, and K-major
//     as the A operand of dX = dY W;
//   * warps 20-23 (converters) read each tile's W_old from global memory
//     ahead of its MMAs, round it to bf16 and write it as the MN-major B
//     operand of dX (Wb); the state ring reads the same W again for the
//     update, mostly from L2;
//   * the dX MMAs (M = 128 tokens, N = 64, K = 16 rows of the tile) are
//     issued by warp 1 after each stage's weight-gradient MMAs, or, where
//     the state stream is light, by a warp of their own (warp 24): with
//     64-column tiles the two products need 64 MMAs per tile, which one
//     issuing thread barely keeps up with; a stage returns to the producer
//     once every issuer's MMAs on it have completed;
//   * each CTA walks a contiguous range of tiles ordered column by column,
//     and a persistent fp32 dX partial (all tokens x the tile's 64 columns)
//     accumulates in TMEM beside the gradient accumulators while the CTA
//     stays in one column; when the column changes, the converter warps
//     (which between them reach all four TMEM lane quadrants) write the
//     partial to a workspace slab, and a separate reduction sums a
//     column's slabs in a fixed order (deterministic dX).
//
// With PAIR (long token axes) two CTAs of a cluster share 256 x 256 tiles:
// each loads its own 128 rows of dY^T and half (128 columns) of X, one
// thread of the pair's first CTA issues tcgen05.mma.cta_group::2 (M = 256,
// N = 256) that reads both CTAs' shared memory, and each CTA's epilogue
// steps its own 128 x 256 accumulator half. Both CTAs' operand bytes are
// counted on the first CTA's stage barriers; its commits arrive on the
// stage and accumulator barriers of both; both epilogues release the
// accumulator on the first CTA's barrier. Per CTA, an operand stage holds
// a third less than a 128 x 256 tile's, for the same MMA work.
//
// The accumulator never leaves TMEM / registers: no gradient tile is ever
// written to global memory (Proposition 3). Both operands are token-major
// in memory, so A = dY^T and B = X are fed to the tensor cores as MN-major
// shared-memory matrices (no transpose is materialised).
//
// Every wait is bounded: a wait that gives up records a status code, sets
// a shared abort flag seen by every other role, and the CTA drains what it
// has in flight and exits; it never traps and never waits forever.
#pragma once

#include <cstdint>

#include "forge_math.cuh"
#include "forge_params.h"
#include "forge_ptx.cuh"

namespace forge {

template <int OPT, int WK, int MK, int BN_, int STAGES_, int NBUF_, bool DX_ = false, bool GA_ = false,
          bool NARROW_ = false, bool WIDE_ = false, bool PAIR_ = false>
struct TcCfg {
  static constexpr bool DX = DX_;      // fused input gradient (see above)
  static constexpr bool GA = GA_;      // add an fp32 accumulated gradient G_acc to each tile
  static constexpr bool LOAD_W = OPT != OPT_ACCSET;  // the set-accumulator rule never reads its target
  static constexpr int BM = 128;       // tile rows (D_out), one per TMEM lane
  static constexpr int BN = BN_;       // tile columns (D_in)
  // A CTA pair (see above): 256 x BN tiles, this CTA's rows and B columns.
  static constexpr bool PAIR = PAIR_;
  static constexpr int BN_CTA = PAIR ? BN / 2 : BN;   // columns of X one CTA loads
  static constexpr int BK = DX ? 128 : 64;  // tokens per operand stage
  static constexpr int BOX = BK * 128; // bytes of one 64-column operand box (BK rows of 128 bytes)
  // State chunk width (columns): 32, or 16 (NARROW) with fp32 W and fp32
  // state in the fused-input-gradient kernel and the deep-ring step --
  // shared memory holds two 48 KB slots of 32 columns or four of 16: on
  // short token axes the deeper state ring pays for the extra chunk turns,
  // and on long ones the narrow slots leave room for a third operand stage.
  static constexpr bool NARROW = NARROW_;
  // 64 (WIDE) for the plain step with bf16 W and bf16 moments: 48 KB slots
  // instead of 24 KB ones, half the chunk turns per byte of state.
  static constexpr bool WIDE = WIDE_;
  static constexpr int CW = NARROW ? 16 : (WIDE ? 64 : 32);
  static constexpr int QC = CW / 4;    // columns per epilogue thread per chunk (one quarter)
  static constexpr int STAGES = STAGES_;
  static constexpr int NBUF = NBUF_;
  static constexpr int NCH = BN / CW;  // chunks per tile
  static constexpr int NST = opt_nstate(OPT);      // state tensors (0, 1, 2)
  static constexpr bool TWO = (NST == 2);           // a second state tensor
  static constexpr bool Q8 = (MK == M_Q8);
  // The accumulation rules keep the fp32 accumulator G_acc where the other
  // rules keep W; with the fused input gradient, WK then names the dtype of
  // the weights the converter warps read for dX.
  static constexpr bool ACC = (OPT == OPT_ACCUM || OPT == OPT_ACCSET);
  static constexpr bool SLOT_F32 = (WK == W_F32) || ACC;  // fp32 values in the slot's first tensor
  // AdamW with bf16 or 8-bit moments in the plain step: the branch-free
  // divide and square root (forge_math.cuh, adamw_group_fast; up-projection,
  // BT 512: bf16 state 172.4 -> 161.2 us, 8-bit 221 -> 210 us with 30 % zero
  // rows, 201 us without). Not in the fused input-gradient kernel (bf16
  // state 226 -> 227 us, with spills around the out-of-line guarded path),
  // on 128 x 256 tiles (BT 2048 250 -> 272 us, BT 8192 771 -> 793 us) nor
  // with fp32 state (no faster; fused pass 269.5 -> 274.8 us).
  static constexpr bool FASTDIV = OPT == OPT_ADAMW && (MK == M_BF16 || MK == M_Q8) && !DX && BN_ != 256;
  static constexpr int WE = SLOT_F32 ? 4 : 2;
  static constexpr int ME = (MK == M_F32) ? 4 : (MK == M_BF16 ? 2 : 1);
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN_CTA * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int W_CH = BM * CW * WE;
  static constexpr int M_CH = NST >= 1 ? BM * CW * ME : 0;
  static constexpr int V_CH = TWO ? M_CH : 0;
  static constexpr int G_CH = GA ? BM * CW * 4 : 0;
  static constexpr int G_OFF = W_CH + M_CH + V_CH;   // G_acc chunk after W, m, v in a slot
  static constexpr int LOAD_BYTES = (LOAD_W ? W_CH : 0) + M_CH + V_CH + G_CH;
  static constexpr int SLOT_BYTES = ((W_CH + M_CH + V_CH + G_CH + 1023) / 1024) * 1024;
  static constexpr int WB_BYTES = DX ? BM * BN * 2 : 0;   // bf16 W_old tile (B operand of dX)
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + WB_BYTES + NBUF * SLOT_BYTES;
  static constexpr int TMEM_COLS =
      (DX || Q8) ? 512 : ((2 * BN <= 128) ? 128 : (2 * BN <= 256 ? 256 : 512));
  static constexpr int DX_COL = 2 * BN;          // first TMEM column of the dX partial
  static constexpr int KEEP_COL = 2 * BN;        // 8-bit moments: the new moments of the tile in the epilogue
  static constexpr int DX_MAX_BLOCKS = DX ? (512 - DX_COL) / BN : 0;  // 128-token blocks that fit
  static constexpr int EPI_WARPS = 16;
  static constexpr int EPI_THREADS = EPI_WARPS * 32;
  static constexpr int CONV_THREADS = DX ? 128 : 0;  // warps 20-23
  // DX: where the state stream is light (bf16 or one-tensor state, the
  // accumulation rules), warp 24 issues the dX MMAs while warp 1 issues the
  // weight-gradient ones -- one issuing thread would set the pass's pace.
  // With fp32 W and two fp32 moments the state stream does, and warp 1
  // issues both (measured: 291.5 us against 294.5 us with two issuers on the
  // Llama-3.1-8B up-projection at BT 512; the bf16-state pass goes from 238
  // to 230 us with two).
  static constexpr bool DX_ISSUER = DX && !(WK == W_F32 && MK == M_F32 && NST == 2);
  static constexpr int DXMMA_WARP = 4 + EPI_WARPS + 4;
  static constexpr int NUM_THREADS = 128 + EPI_THREADS + CONV_THREADS + (DX_ISSUER ? 32 : 0);
  static constexpr uint32_t IDESC = make_idesc_bf16(PAIR ? 2 * BM : BM, BN, 1, 1);
  // dX: A = dY (M = 128 tokens, K-major), B = Wb (N = BN, MN-major).
  static constexpr uint32_t IDESC_DX = make_idesc_bf16(128, BN, 0, 1);

};

// Byte offset of 16-byte chunk `c` of row `r` in a TMA tile whose rows are
// 32 * E bytes, written with the matching swizzle (128, 64 or 32 bytes):
// the chunk index is XOR-ed with address bits 7.. of the row start.
template <int E>
__device__ __forceinline__ uint32_t swz(int r, int c) {
  constexpr int RB = 32 * E;
  const int x = (RB == 128) ? (r & 7) : (RB == 64 ? ((r >> 1) & 3) : ((r >> 2) & 1));
  return static_cast<uint32_t>(r * RB + ((c ^ x) << 4));
}

// 8 consecutive values of row r, columns [8h, 8h + 8) of a 32-column chunk.
template <int KIND>  // 0: f32, 1: bf16
__device__ __forceinline__ void ld8(const uint8_t* base, int r, int h, float (&o)[8]) {
  if constexpr (KIND == 0) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float4 t = *reinterpret_cast<const float4*>(base + swz<4>(r, 2 * h + k));
      o[4 * k + 0] = t.x; o[4 * k + 1] = t.y; o[4 * k + 2] = t.z; o[4 * k + 3] = t.w;
    }
  } else {
    const uint4 t = *reinterpret_cast<const uint4*>(base + swz<2>(r, h));
    const uint32_t wv[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i + 0] = bf16_bits_to_f32(wv[i] & 0xFFFFu);
      o[2 * i + 1] = bf16_bits_to_f32(wv[i] >> 16);
    }
  }
}

__device__ __forceinline__ void st8_f32(uint8_t* base, int r, int h, const float (&o)[8]) {
#pragma unroll
  for (int k = 0; k < 2; ++k)
    *reinterpret_cast<float4*>(base + swz<4>(r, 2 * h + k)) =
        make_float4(o[4 * k + 0], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
}

// 4 consecutive fp32 values of row r, columns [4h, 4h + 4) of a 16-column
// chunk (64-byte rows, 64-byte swizzle: one 16-byte piece).
__device__ __forceinline__ void ld4_f32(const uint8_t* base, int r, int h, float (&o)[4]) {
  const float4 t = *reinterpret_cast<const float4*>(base + swz<2>(r, h));
  o[0] = t.x; o[1] = t.y; o[2] = t.z; o[3] = t.w;
}

__device__ __forceinline__ void st4_f32(uint8_t* base, int r, int h, const float (&o)[4]) {
  *reinterpret_cast<float4*>(base + swz<2>(r, h)) = make_float4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ void st8_bf16(uint8_t* base, int r, int h, const uint4& t) {
  *reinterpret_cast<uint4*>(base + swz<2>(r, h)) = t;
}

// 8 consecutive bf16 values of row r, 16-byte piece hq of a 64-column chunk
// (128-byte rows, 128-byte swizzle), as floats; and the matching store.
__device__ __forceinline__ void ld8_bf16_w(const uint8_t* base, int r, int hq, float (&o)[8]) {
  const uint4 t = *reinterpret_cast<const uint4*>(base + swz<4>(r, hq));
  const uint32_t wv[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i + 0] = bf16_bits_to_f32(wv[i] & 0xFFFFu);
    o[2 * i + 1] = bf16_bits_to_f32(wv[i] >> 16);
  }
}

__device__ __forceinline__ void st8_bf16_w(uint8_t* base, int r, int hq, const uint4& t) {
  *reinterpret_cast<uint4*>(base + swz<4>(r, hq)) = t;
}

// The 8 codes of row r, columns [8h, 8h + 8) of a 32-column chunk (half
// h % 2 of 16-byte chunk h / 2) as two words, byte i = column 8h + i.
__device__ __forceinline__ uint2 ld8_code_words(const uint8_t* base, int r, int h) {
  return *reinterpret_cast<const uint2*>(base + swz<1>(r, h >> 1) + (h & 1) * 8);
}

// Stores the low bytes of c[0..7] as those 8 codes.
__device__ __forceinline__ void st8_codes(uint8_t* base, int r, int h, const uint32_t (&c)[8]) {
  *reinterpret_cast<uint2*>(base + swz<1>(r, h >> 1) + (h & 1) * 8) =
      make_uint2(pack_low_bytes(c[0], c[1], c[2], c[3]), pack_low_bytes(c[4], c[5], c[6], c[7]));
}

// Eight bf16 stores of `x` packed in four words: stochastic rounding with
// the Philox block of elements idx8 * 8 .. idx8 * 8 + 7 at `site`, or
// round-to-nearest-even.
// BATCH_NAN: the NaN test is made once for the eight values, and without a
// NaN the draws are added to the bit patterns directly (plain step, bf16
// state, up-projection: AdamW BT 512 174.1 -> 171.6 us, Lion 137.2 -> 131.5;
// in the fused input-gradient kernel it measured 225 -> 230 us, which keeps
// the per-value test).
template <bool BATCH_NAN>
__device__ __forceinline__ void to_bf16x8(const float (&x)[8], bool sr, uint64_t idx8, uint32_t site,
                                          const WgradTcParams& p, uint4& o) {
  if (sr) {
    // Lanes 2i and 2i + 1 take the low and high half of Philox word i.
    const U4 rr = sr_block(idx8, p.step, site, p.seed_lo, p.seed_hi);
    bool any_nan = !BATCH_NAN;
    if constexpr (BATCH_NAN) {
#pragma unroll
      for (int j = 0; j < 8; ++j) any_nan |= x[j] != x[j];
    }
    if (__builtin_expect(!any_nan, 1)) {
      o = make_uint4(sr_bf16x2_finite(x[0], x[1], rr.x), sr_bf16x2_finite(x[2], x[3], rr.y),
                     sr_bf16x2_finite(x[4], x[5], rr.z), sr_bf16x2_finite(x[6], x[7], rr.w));
    } else {
      o = make_uint4(sr_bf16x2(x[0], x[1], rr.x & 0xFFFFu, rr.x >> 16),
                     sr_bf16x2(x[2], x[3], rr.y & 0xFFFFu, rr.y >> 16),
                     sr_bf16x2(x[4], x[5], rr.z & 0xFFFFu, rr.z >> 16),
                     sr_bf16x2(x[6], x[7], rr.w & 0xFFFFu, rr.w >> 16));
    }
  } else {
    o = make_uint4(pack_bf16x2_rn(x[0], x[1]), pack_bf16x2_rn(x[2], x[3]), pack_bf16x2_rn(x[4], x[5]),
                   pack_bf16x2_rn(x[6], x[7]));
  }
}

__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int group_m, int& tm, int& tn) {
  const int per_group = group_m * tiles_n;
  const int g = tile / per_group;
  const int first_m = g * group_m;
  const int rem = tiles_m - first_m;
  const int gsize = rem < group_m ? rem : group_m;
  const int in_g = tile - g * per_group;
  tm = first_m + in_g % gsize;
  tn = in_g / gsize;
}

// The tiles one CTA processes: a grid-stride walk of the grouped raster, or
// (fused input gradient) a contiguous range of the column-major tile order,
// so that consecutive tiles share a column and its dX partial.
struct TileWalk {
  int first, step, end;
};

template <bool DX, bool PAIR>
__device__ __forceinline__ TileWalk tile_walk(const WgradTcParams& p) {
  if constexpr (DX) {
    const int64_t T = p.num_tiles, G = gridDim.x, c = blockIdx.x;
    return TileWalk{static_cast<int>(c * T / G), 1, static_cast<int>((c + 1) * T / G)};
  } else if constexpr (PAIR) {
    // A pair (cluster) walks the raster of 256-row tiles.
    return TileWalk{static_cast<int>(blockIdx.x >> 1), static_cast<int>(gridDim.x >> 1), p.num_tiles};
  } else {
    return TileWalk{static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), p.num_tiles};
  }
}

// tm: this CTA's 128-row tile (PAIR: half `prank` of the pair's 256 rows).
template <bool DX, bool PAIR>
__device__ __forceinline__ void walk_coords(const WgradTcParams& p, int tile, int prank, int& tm, int& tn) {
  if constexpr (DX) {
    tm = tile % p.tiles_m;
    tn = tile / p.tiles_m;
  } else {
    tile_coords(tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
    if constexpr (PAIR) tm = 2 * tm + prank;
  }
}

// Write a CTA's dX partial (tokens x BN fp32, token-major) from tensor
// memory to its workspace slab: the warp with TMEM lane quadrant q writes
// tokens 32q .. 32q + 31 of every 128-token block, one token row per
// thread. Runs once per tile column of the CTA.
// With l2 the slab is stored evict-last, and the reduction that follows this
// kernel reads it from L2 and drops it, so that it need not reach DRAM.
template <int BN>
__device__ __forceinline__ void write_dx_partial(float* slab, uint32_t tmem_dx, int q, int lane, int num_kb,
                                                 bool l2) {
  const uint64_t pol = l2_policy_evict_last();
  for (int b = 0; b < num_kb; ++b) {
    const int tok = b * 128 + q * 32 + lane;
    const uint32_t ta = tmem_dx + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * BN);
    float* dst = slab + static_cast<int64_t>(tok) * BN;
#pragma unroll 1
    for (int c16 = 0; c16 < BN / 16; ++c16) {
      uint32_t d[16];
      tmem_ld_32x32b_x16(ta + c16 * 16, d);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float* o = dst + c16 * 16 + 4 * j;
        const float a = __uint_as_float(d[4 * j]), bb = __uint_as_float(d[4 * j + 1]);
        const float c = __uint_as_float(d[4 * j + 2]), e = __uint_as_float(d[4 * j + 3]);
        if (l2) st_global_v4_hint(o, a, bb, c, e, pol);
        else *reinterpret_cast<float4*>(o) = make_float4(a, bb, c, e);
      }
    }
  }
}

// Bounded wait on an mbarrier phase. Returns false if the CTA is aborting
// (another role gave up) or if this wait exceeded `limit_ns`, in which case
// it raises the abort flag and records `code` in the device status word.

// CL: acquire at cluster scope (phases completed by the other CTA of a pair).
template <bool CL = false>
__device__ __forceinline__ bool bwait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                      unsigned int* status, uint32_t code, uint64_t limit_ns) {
  auto try_wait = [&]() { return CL ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  if (try_wait()) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (try_wait()) return true;
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

// After an abort: wait (bounded) for the last fills a producer issued on a
// ring of barriers, so that no TMA write lands after the CTA has exited.
__device__ __forceinline__ void drain_ring(uint64_t* full, int ring, uint32_t issued, unsigned int* status) {
  const uint32_t first = issued > static_cast<uint32_t>(ring) ? issued - ring : 0u;
  for (uint32_t k = first; k < issued; ++k) {
    const int s = static_cast<int>(k % ring);
    const uint32_t ph = (k / ring) & 1u;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(&full[s], ph)) {
      if (globaltimer_ns() - t0 > 200000000ull) {  // 0.2 s: a load never takes this long
        atomicCAS(status, 0u, WAIT_DRAIN);
        break;
      }
    }
  }
}

// The dX MMAs of operand stage kb of a tile: dX[128 tokens of the stage][BN]
// += dY[tokens][128 rows of the tile] * Wb, into the persistent partial of
// the tile column (a fresh one on the column's first tile). A: dY K-major
// (K = D_out rows of the tile, 64 per 128-byte box row), 8-token groups
// 1024 bytes apart, a K step of 16 advancing 32 bytes. B: Wb MN-major,
// 8-row K groups of 1024 bytes, 16 rows = 2048 bytes.
template <class C>
__device__ __forceinline__ void issue_dx_stage(uint32_t a0, uint32_t wb, uint32_t tmem_base, int kb,
                                               bool run_first) {
  const uint32_t dx_tmem = tmem_base + static_cast<uint32_t>(C::DX_COL + kb * C::BN);
  const uint64_t xa0 = make_smem_desc(a0, 16, 1024, 2);
  const uint64_t xb0 = make_smem_desc(wb, 8192, 1024, 2);
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t astep = static_cast<uint64_t>((hh * C::BOX + kk * 32) >> 4);
      const uint64_t bstep = static_cast<uint64_t>(((hh * 4 + kk) * 2048) >> 4);
      umma_f16(dx_tmem, xa0 + astep, xb0 + bstep, C::IDESC_DX, (run_first && hh == 0 && kk == 0) ? 0u : 1u);
    }
  }
}

// Before a tile's first dX MMAs: the previous column's partial must have
// been written out (at a column's first tile), and this tile's bf16 W_old
// must be in place. False if a wait gave up.
__device__ __forceinline__ bool dx_tile_ready(bool run_first, uint32_t runs_done, int it, uint64_t* dx_empty,
                                              uint64_t* wb_full, volatile int* abort_flag, unsigned int* status,
                                              uint64_t lim) {
  if (run_first && runs_done > 0 && !bwait(dx_empty, (runs_done - 1) & 1u, abort_flag, status, WAIT_DX_EMPTY, lim))
    return false;
  return bwait(wb_full, it & 1, abort_flag, status, WAIT_WB_FULL, lim);
}

template <int OPT, int WK, int MK, int BN, int STAGES, int NBUF, bool DX, bool GA, bool NARROW, bool WIDE,
          bool PAIR>
__global__ void __launch_bounds__(TcCfg<OPT, WK, MK, BN, STAGES, NBUF, DX, GA, NARROW, WIDE, PAIR>::NUM_THREADS, 1)
    wgrad_step_tc_kernel(const __grid_constant__ WgradTcParams p) {
  using C = TcCfg<OPT, WK, MK, BN, STAGES, NBUF, DX, GA, NARROW, WIDE, PAIR>;
  static_assert(!WIDE || (WK == W_BF16 && MK == M_BF16 && !DX && !GA && !C::ACC),
                "64-column chunks: plain step with bf16 W and bf16 moments");
  static_assert(!NARROW || ((DX || BN >= 128) && WK == W_F32 && MK == M_F32 && C::NST >= 1 && !C::ACC && !GA),
                "16-column chunks: fused kernel or deep step tiles with fp32 W and fp32 state");
  static_assert(!GA || (!DX && !C::Q8), "accumulated-gradient step: split path, fp32 / bf16 state");
  static_assert(!C::ACC || ((WK == W_F32 || DX) && !GA), "fp32 gradient accumulator");
  static_assert(BN == 64 || BN == 128 || BN == 256, "tile width");
  static_assert(BN != 256 || (!C::Q8 && !DX && !GA), "256-column tiles: plain step, fp32 / bf16 state");
  static_assert(!DX || (BN == 64 && !C::Q8), "fused input gradient: 64-column tiles, fp32 / bf16 state");
  static_assert(!C::Q8 || BN == 128, "8-bit blocks span one 128-column tile row");
  static_assert(!C::Q8 || OPT == OPT_ADAMW || OPT == OPT_SGDM || OPT == OPT_LION, "8-bit state rules");
  static_assert(!C::Q8 || NBUF >= C::NCH, "8-bit moments hold a whole tile of slots");
  static_assert(!PAIR || (BN == 256 && !DX && !GA && !C::Q8 && !C::ACC), "CTA pairs: 256-column plain-step tiles");
  static_assert(NBUF >= 2 && STAGES >= 2, "pipelines");
  static_assert(C::SMEM_BYTES <= 227 * 1024, "shared memory");

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t op_full[STAGES], op_empty[STAGES];
  __shared__ __align__(8) uint64_t st_full[NBUF], st_empty[NBUF], st_written[NBUF];
  __shared__ __align__(8) uint64_t tm_full[2], tm_empty[2];
  __shared__ __align__(8) uint64_t red_bar[2];
  __shared__ __align__(8) uint64_t never_bar, mma_drain_bar, dx_drain_bar;
  __shared__ __align__(8) uint64_t wb_full, wb_empty, dx_full, dx_empty;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ float red_sh[C::Q8 ? 2 : 1][2][4][128];  // [tile parity][|m'| | v'][column quarter][row]

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* op_base = smem;
  uint8_t* wb_base = smem + STAGES * C::STAGE_BYTES;
  uint8_t* st_base = wb_base + C::WB_BYTES;
  const TileWalk tw = tile_walk<DX, PAIR>(p);
  // Rank in the CTA pair: 0 issues the pair's MMAs and owns the operand barriers.
  const int prank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &abort_sh;

  if (threadIdx.x == 0) {
    // With a dX issuer a stage is released by both MMA-issuing threads.
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&op_full[s], 1);
      mbar_init(&op_empty[s], C::DX_ISSUER ? 2 : 1);
    }
    for (int s = 0; s < NBUF; ++s) {
      mbar_init(&st_full[s], 1);
      mbar_init(&st_empty[s], 1);
      mbar_init(&st_written[s], C::EPI_THREADS);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tm_full[b], 1);
      mbar_init(&tm_empty[b], PAIR ? 2 * C::EPI_WARPS : C::EPI_WARPS);  // both halves' epilogues
      mbar_init(&red_bar[b], C::EPI_THREADS);
    }
    mbar_init(&never_bar, 1);
    mbar_init(&mma_drain_bar, 1);
    mbar_init(&dx_drain_bar, 1);
    mbar_init(&wb_full, C::CONV_THREADS > 0 ? C::CONV_THREADS : 1);
    mbar_init(&wb_empty, 1);
    mbar_init(&dx_full, 1);
    mbar_init(&dx_empty, 4);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    if (p.num_kb > 0) { prefetch_tmap(&p.tm_dy); prefetch_tmap(&p.tm_x); }
    prefetch_tmap(&p.tm_w);
    if constexpr (GA) prefetch_tmap(&p.tm_g);
    if constexpr (C::NST >= 1) prefetch_tmap(&p.tm_m);
    if constexpr (C::TWO) prefetch_tmap(&p.tm_v);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(&tmem_base_sh, C::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&tmem_base_sh, C::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  // The other CTA's barriers are initialised before any load or arrival
  // reaches them.
  if constexpr (PAIR) cluster_sync_all();
  tc_fence_after_sync();
  // Launched as a programmatic dependent: everything above (barriers, tensor
  // memory, tensor-map prefetch) overlaps the previous kernel's tail; global
  // memory is touched only after it has completed. The next kernel may be
  // scheduled from here on (its CTAs take SMs as this grid's CTAs leave).
  griddep_launch_dependents();
  griddep_wait();
  const uint32_t tmem_base = tmem_base_sh;
  const uint64_t lim = p.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ operand producer
    if (lane == 0) {
      uint32_t kseq = 0;
      bool ok = true;
      for (int tile = tw.first; ok && tile < tw.end; tile += tw.step) {
        int tm, tn;
        walk_coords<DX, PAIR>(p, tile, prank, tm, tn);
        for (int kb = 0; kb < p.num_kb; ++kb, ++kseq) {
          const int s = static_cast<int>(kseq % STAGES);
          const uint32_t ph = (kseq / STAGES) & 1u;
          if (!bwait(&op_empty[s], ph ^ 1u, abort_flag, p.status, WAIT_OP_EMPTY, lim)) { ok = false; break; }
          uint8_t* a = op_base + s * C::STAGE_BYTES;
          uint8_t* b = a + C::A_BYTES;
          if constexpr (PAIR) {
            // Both CTAs' bytes complete on the first CTA's stage barrier.
            if (prank == 0) mbar_arrive_expect_tx(&op_full[s], 2 * C::STAGE_BYTES);
            const uint32_t fb = cluster_map(smem_u32(&op_full[s]), 0u);
            const int xb = tn * BN + prank * C::BN_CTA;
            if (p.op_hint) {
              const uint64_t pol = l2_policy_evict_last();
              tma_load_2d_pair_hint(a, &p.tm_dy, fb, tm * C::BM, kb * C::BK, pol);
              tma_load_2d_pair_hint(a + C::BOX, &p.tm_dy, fb, tm * C::BM + 64, kb * C::BK, pol);
#pragma unroll
              for (int bb = 0; bb < C::BN_CTA / 64; ++bb)
                tma_load_2d_pair_hint(b + bb * C::BOX, &p.tm_x, fb, xb + bb * 64, kb * C::BK, pol);
            } else {
              tma_load_2d_pair(a, &p.tm_dy, fb, tm * C::BM, kb * C::BK);
              tma_load_2d_pair(a + C::BOX, &p.tm_dy, fb, tm * C::BM + 64, kb * C::BK);
#pragma unroll
              for (int bb = 0; bb < C::BN_CTA / 64; ++bb)
                tma_load_2d_pair(b + bb * C::BOX, &p.tm_x, fb, xb + bb * 64, kb * C::BK);
            }
            continue;
          }
          mbar_arrive_expect_tx(&op_full[s], C::STAGE_BYTES);
          if (p.op_hint) {
            const uint64_t pol = l2_policy_evict_last();
            tma_load_2d_hint(a, &p.tm_dy, &op_full[s], tm * C::BM, kb * C::BK, pol);
            tma_load_2d_hint(a + C::BOX, &p.tm_dy, &op_full[s], tm * C::BM + 64, kb * C::BK, pol);
#pragma unroll
            for (int bb = 0; bb < BN / 64; ++bb)
              tma_load_2d_hint(b + bb * C::BOX, &p.tm_x, &op_full[s], tn * BN + bb * 64, kb * C::BK, pol);
          } else {
            tma_load_2d(a, &p.tm_dy, &op_full[s], tm * C::BM, kb * C::BK);
            tma_load_2d(a + C::BOX, &p.tm_dy, &op_full[s], tm * C::BM + 64, kb * C::BK);
#pragma unroll
            for (int bb = 0; bb < BN / 64; ++bb)
              tma_load_2d(b + bb * C::BOX, &p.tm_x, &op_full[s], tn * BN + bb * 64, kb * C::BK);
          }
        }
      }
      // (PAIR: the second CTA's loads complete on the first CTA's barriers,
      // which that CTA drains.)
      if (!ok && prank == 0) drain_ring(op_full, STAGES, kseq, p.status);
    }
    if (p.op_hint) {
      // This CTA's share of the operands' lines back to normal priority, so
      // that evict-last lines do not pile up in L2 across calls.
      __syncwarp();
#pragma unroll 1
      for (int i = 0; i < 2; ++i) {
        // fewer than 2^20 lines (the host takes operands of at most 96 MB)
        const uint32_t lines = static_cast<uint32_t>((p.op_hi[i] - p.op_lo[i]) >> 7);
        const uint32_t l1 = lines * (blockIdx.x + 1) / gridDim.x;
        const uint8_t* base = p.op_lo[i];
#pragma unroll 1
        for (uint32_t l = lines * blockIdx.x / gridDim.x + lane; l < l1; l += 32) l2_demote_line(base + (l << 7));
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (weight gradient)
    // (PAIR: the first CTA's thread issues for both.)
    if (lane == 0 && prank == 0) {
      uint32_t kseq = 0;
      bool ok = true;
      int it = 0;
      uint32_t runs_done = 0;  // dX partials handed to the converter warps (no dX issuer)
      for (int tile = tw.first; ok && tile < tw.end; tile += tw.step, ++it) {
        const int buf = it & 1;
        const uint32_t eph = ((it >> 1) & 1) ^ 1u;
        if (!bwait<PAIR>(&tm_empty[buf], eph, abort_flag, p.status, WAIT_TMEM_EMPTY, lim)) { ok = false; break; }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
        // dX issued here too (no dX issuer warp): the column's first tile
        // starts a fresh partial.
        constexpr bool DX_HERE = DX && !C::DX_ISSUER;
        const bool run_first = DX_HERE && (tile == tw.first || tile % p.tiles_m == 0);
        const bool run_last = DX_HERE && (tile + 1 == tw.end || (tile + 1) % p.tiles_m == 0);
        for (int kb = 0; kb < p.num_kb; ++kb, ++kseq) {
          const int s = static_cast<int>(kseq % STAGES);
          const uint32_t ph = (kseq / STAGES) & 1u;
          if (!bwait(&op_full[s], ph, abort_flag, p.status, WAIT_OP_FULL, lim)) { ok = false; break; }
          tc_fence_after_sync();
          const uint32_t a0 = smem_u32(op_base + s * C::STAGE_BYTES);
          const uint32_t b0 = a0 + C::A_BYTES;
          // Descriptors are built once per stage; a K step only moves the
          // 14-bit start-address field (16-byte units; shared addresses stay
          // below 2^18 bytes, so the field never carries into its neighbour).
          const uint64_t ad0 = make_smem_desc(a0, C::BOX, 1024, 2);
          const uint64_t bd0 = make_smem_desc(b0, C::BOX, 1024, 2);
#pragma unroll
          for (int kk = 0; kk < C::BK / 16; ++kk) {
            // 16 tokens = two 8-row K groups of 1024 bytes; MN atoms one box apart.
            const uint64_t step = static_cast<uint64_t>(kk * 2048 >> 4);
            if constexpr (PAIR) umma_f16_pair(d_tmem, ad0 + step, bd0 + step, C::IDESC, (kb > 0 || kk > 0) ? 1u : 0u);
            else umma_f16(d_tmem, ad0 + step, bd0 + step, C::IDESC, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          if constexpr (DX_HERE) {
            if (kb == 0) {
              if (!dx_tile_ready(run_first, runs_done, it, &dx_empty, &wb_full, abort_flag, p.status, lim)) {
                ok = false;
                break;
              }
              tc_fence_after_sync();
            }
            issue_dx_stage<C>(a0, smem_u32(wb_base), tmem_base, kb, run_first);
          }
          if constexpr (PAIR) umma_commit_pair(&op_empty[s], 3);   // the stage in both CTAs
          else umma_commit(&op_empty[s]);
        }
        if (!ok) break;
        if constexpr (DX_HERE) {
          if (p.num_kb > 0) {
            umma_commit(&wb_empty);
            if (run_last) { umma_commit(&dx_full); ++runs_done; }
          }
        }
        if constexpr (PAIR) umma_commit_pair(&tm_full[buf], 3);   // both halves' epilogues
        else umma_commit(&tm_full[buf]);
      }
      if (!ok) {
        // Let every MMA already issued finish before TMEM is released.
        if constexpr (PAIR) umma_commit_pair(&mma_drain_bar, 1);
        else umma_commit(&mma_drain_bar);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&mma_drain_bar, 0)) {
          if (globaltimer_ns() - t0 > 200000000ull) { atomicCAS(p.status, 0u, WAIT_MMA_DRAIN); break; }
        }
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ state producer
    if (lane == 0) {
      uint32_t cseq = 0;
      bool ok = true;
      for (int tile = tw.first; ok && tile < tw.end; tile += tw.step) {
        int tm, tn;
        walk_coords<DX, PAIR>(p, tile, prank, tm, tn);
        for (int c = 0; c < C::NCH; ++c, ++cseq) {
          const int s = static_cast<int>(cseq % NBUF);
          const uint32_t ph = (cseq / NBUF) & 1u;
          if (!bwait(&st_empty[s], ph ^ 1u, abort_flag, p.status, WAIT_ST_EMPTY, lim)) { ok = false; break; }
          uint8_t* slot = st_base + s * C::SLOT_BYTES;
          const int x = tn * BN + c * C::CW, y = tm * C::BM;
          mbar_arrive_expect_tx(&st_full[s], C::LOAD_BYTES);
          if constexpr (C::LOAD_W) tma_load_2d(slot, &p.tm_w, &st_full[s], x, y);
          if constexpr (C::NST >= 1) tma_load_2d(slot + C::W_CH, &p.tm_m, &st_full[s], x, y);
          if constexpr (C::TWO) tma_load_2d(slot + C::W_CH + C::M_CH, &p.tm_v, &st_full[s], x, y);
          if constexpr (GA) tma_load_2d(slot + C::G_OFF, &p.tm_g, &st_full[s], x, y);
        }
      }
      if (!ok) drain_ring(st_full, NBUF, cseq, p.status);
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ state storer
    if (lane == 0) {
      uint32_t cseq = 0;
      bool ok = true;
      for (int tile = tw.first; ok && tile < tw.end; tile += tw.step) {
        int tm, tn;
        walk_coords<DX, PAIR>(p, tile, prank, tm, tn);
        for (int c = 0; c < C::NCH; ++c, ++cseq) {
          const int s = static_cast<int>(cseq % NBUF);
          const uint32_t ph = (cseq / NBUF) & 1u;
          if (!bwait(&st_written[s], ph, abort_flag, p.status, WAIT_ST_WRITTEN, lim)) { ok = false; break; }
          const uint8_t* slot = st_base + s * C::SLOT_BYTES;
          const int x = tn * BN + c * C::CW, y = tm * C::BM;
          tma_store_2d(&p.tm_w, slot, x, y);
          if constexpr (C::NST >= 1) tma_store_2d(&p.tm_m, slot + C::W_CH, x, y);
          if constexpr (C::TWO) tma_store_2d(&p.tm_v, slot + C::W_CH + C::M_CH, x, y);
          bulk_commit_group();
          bulk_wait_group_read0();
          mbar_arrive(&st_empty[s]);
        }
      }
      bulk_wait_group0();
    }
  } else if (warp < 4 + C::EPI_WARPS) {
    // ------------------------------------------------------------ epilogue (warps 4..19)
    const int q = warp & 3;          // TMEM lane quadrant this warp may access
    const int h = (warp - 4) >> 2;   // 8-column quarter of each 32-column chunk
    const int r = q * 32 + lane;     // tile row == TMEM lane
    const StepScalars sc = p.sc;
    uint32_t cseq = 0;
    int it = 0;
    bool ok = true;

    if (p.flags & FLAG_TEST_FORCE_TIMEOUT) {
      // Test hook: a barrier nothing signals, with a short bound.
      ok = bwait(&never_bar, 0, abort_flag, p.status, WAIT_TEST_HOOK, 1000000ull);
      ok = __all_sync(0xFFFFFFFFu, ok);
    }

    for (int tile = tw.first; ok && tile < tw.end; tile += tw.step, ++it) {
      int tm, tn;
      walk_coords<DX, PAIR>(p, tile, prank, tm, tn);
      const int buf = it & 1;
      ok = bwait(&tm_full[buf], (it >> 1) & 1, abort_flag, p.status, WAIT_TMEM_FULL, lim);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      const int row = tm * C::BM + r;
      const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * BN);

      if constexpr (!C::Q8) {
        for (int c = 0; c < C::NCH; ++c, ++cseq) {
          const int s = static_cast<int>(cseq % NBUF);
          ok = bwait(&st_full[s], (cseq / NBUF) & 1u, abort_flag, p.status, WAIT_ST_FULL, lim);
          ok = __all_sync(0xFFFFFFFFu, ok);
          if (!ok) break;
          if constexpr (WIDE) {
            // 16 columns per thread per chunk, as two groups of 8: the same
            // per-element code as 32-column chunks, one slot hand-over per 16.
            uint8_t* slot = st_base + s * C::SLOT_BYTES;
#pragma unroll 1
            for (int sub = 0; sub < 2; ++sub) {
              const int col = h * 16 + sub * 8;  // within the chunk
              const int hq = 2 * h + sub;        // 16-byte piece of the 128-byte row
              uint32_t gr[8];
              if (p.num_kb > 0) {
                tmem_ld_32x32b_x8(t_lane + c * C::CW + col, gr);
                tmem_ld_wait();
              } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) gr[j] = 0u;
              }
              float w[8], m[8], v[8], g[8];
              ld8_bf16_w(slot, r, hq, w);
              if constexpr (C::NST >= 1) ld8_bf16_w(slot + C::W_CH, r, hq, m);
              if constexpr (C::TWO) ld8_bf16_w(slot + C::W_CH + C::M_CH, r, hq, v);
#pragma unroll
              for (int j = 0; j < 8; ++j) g[j] = __uint_as_float(gr[j]);
              if constexpr (C::FASTDIV) {
                adamw_group_fast(g, w, m, v, sc);
              } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) step_elem<OPT>(g[j], w[j], m[j], v[j], sc);
              }
              const uint64_t idx8 =
                  (static_cast<uint64_t>(row) * static_cast<uint64_t>(p.d_in) + (tn * BN + c * C::CW + col)) >> 3;
              uint4 b;
              to_bf16x8<!DX>(w, p.sr_w != 0, idx8, 0u, p, b);
              st8_bf16_w(slot, r, hq, b);
              if constexpr (C::NST >= 1) {
                to_bf16x8<!DX>(m, p.sr_m != 0, idx8, 1u, p, b);
                st8_bf16_w(slot + C::W_CH, r, hq, b);
              }
              if constexpr (C::TWO) {
                to_bf16x8<!DX>(v, p.sr_m != 0, idx8, 2u, p, b);
                st8_bf16_w(slot + C::W_CH + C::M_CH, r, hq, b);
              }
            }
            fence_proxy_async_smem();
            mbar_arrive(&st_written[s]);
          } else {
          constexpr int Q = C::QC;
          uint32_t gr[Q];
          if (p.num_kb > 0) {
            if constexpr (Q == 8) tmem_ld_32x32b_x8(t_lane + c * C::CW + h * Q, gr);
            else tmem_ld_32x32b_x4(t_lane + c * C::CW + h * Q, gr);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int j = 0; j < Q; ++j) gr[j] = 0u;
          }
          uint8_t* slot = st_base + s * C::SLOT_BYTES;
          uint8_t* sw = slot;
          uint8_t* sm = slot + C::W_CH;
          uint8_t* sv = slot + C::W_CH + C::M_CH;
          float w[Q], m[Q], v[Q], g[Q];
          if constexpr (Q == 4) {  // fp32 W and moments (the 16-column chunks)
            ld4_f32(sw, r, h, w);
            ld4_f32(sm, r, h, m);
            if constexpr (C::TWO) ld4_f32(sv, r, h, v);
          } else {
            if constexpr (C::LOAD_W) ld8<C::SLOT_F32 ? 0 : 1>(sw, r, h, w);
            if constexpr (C::NST >= 1) ld8<MK == M_F32 ? 0 : 1>(sm, r, h, m);
            if constexpr (C::TWO) ld8<MK == M_F32 ? 0 : 1>(sv, r, h, v);
          }
#pragma unroll
          for (int j = 0; j < Q; ++j) g[j] = __uint_as_float(gr[j]);
          if constexpr (GA) {
            // The micro-batches accumulated so far: G = G_acc + this tile's G.
            float ga[8];
            ld8<0>(slot + C::G_OFF, r, h, ga);
#pragma unroll
            for (int j = 0; j < 8; ++j) g[j] = __fadd_rn(ga[j], g[j]);
          }
          if constexpr (C::FASTDIV) {
            adamw_group_fast(g, w, m, v, sc);
          } else {
#pragma unroll
            for (int j = 0; j < Q; ++j) step_elem<OPT>(g[j], w[j], m[j], v[j], sc);
          }
          if constexpr (Q == 4) {
            st4_f32(sw, r, h, w);
            st4_f32(sm, r, h, m);
            if constexpr (C::TWO) st4_f32(sv, r, h, v);
            fence_proxy_async_smem();
            mbar_arrive(&st_written[s]);
            continue;
          } else {
          // Element index of this thread's first column; 8-aligned (D_in % 8 == 0).
          const uint64_t idx8 =
              (static_cast<uint64_t>(row) * static_cast<uint64_t>(p.d_in) + (tn * BN + c * C::CW + h * 8)) >> 3;
          if constexpr (C::SLOT_F32) {
            st8_f32(sw, r, h, w);
          } else {
            uint4 b;
            to_bf16x8<!DX>(w, p.sr_w != 0, idx8, 0u, p, b);
            st8_bf16(sw, r, h, b);
          }
          if constexpr (C::NST == 0) {
          } else if constexpr (MK == M_F32) {
            st8_f32(sm, r, h, m);
            if constexpr (C::TWO) st8_f32(sv, r, h, v);
          } else {
            uint4 b;
            to_bf16x8<!DX>(m, p.sr_m != 0, idx8, 1u, p, b);
            st8_bf16(sm, r, h, b);
            if constexpr (C::TWO) {
              to_bf16x8<!DX>(v, p.sr_m != 0, idx8, 2u, p, b);
              st8_bf16(sv, r, h, b);
            }
          }
          fence_proxy_async_smem();
          mbar_arrive(&st_written[s]);
          }
          }
        }
        if (!ok) break;
      } else {
        // -------------------------------------------------- 8-bit block moments
        // The 128 columns of this tile row are one quantisation block, so the
        // new block absmax needs every chunk. Pass 1 forms the new moments
        // (Lion: and its update direction), keeps them in the free half of
        // tensor memory and takes their absmax; the accumulator buffer is
        // then handed back. Pass 2 reads them back, steps W and quantises.
        const int jb = tn;  // block column (BN == 128)
        const uint32_t t_keep = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(C::KEEP_COL);
        constexpr bool KEEP2 = OPT != OPT_SGDM;   // a second kept value: v' (AdamW), the direction (Lion)
        float sm_old = 0.0f, sv_old = 0.0f;
        if (row < p.d_out) {
          sm_old = p.m_scale[static_cast<int64_t>(jb) * p.d_out + row];
          if constexpr (C::TWO) sv_old = p.v_scale[static_cast<int64_t>(jb) * p.d_out + row];
        }
        float am = 0.0f, au = 0.0f;
        for (int c = 0; c < C::NCH; ++c) {
          const uint32_t k = cseq + c;
          const int s = static_cast<int>(k % NBUF);
          ok = bwait(&st_full[s], (k / NBUF) & 1u, abort_flag, p.status, WAIT_ST_FULL, lim);
          ok = __all_sync(0xFFFFFFFFu, ok);
          if (!ok) break;
          uint32_t gr[8];
          if (p.num_kb > 0) {
            tmem_ld_32x32b_x8(t_lane + c * C::CW + h * 8, gr);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) gr[j] = 0u;
          }
          const uint8_t* slot = st_base + s * C::SLOT_BYTES;
          float c0[8], c1[8], w[8];
          const uint2 tm8 = ld8_code_words(slot + C::W_CH, r, h);
          codes_s8_to_f32(tm8.x, tm8.y, c0);
          if constexpr (C::TWO) {
            const uint2 tv8 = ld8_code_words(slot + C::W_CH + C::M_CH, r, h);
            codes_u8_to_f32(tv8.x, tv8.y, c1);
          }
          if constexpr (OPT == OPT_SGDM) ld8<WK == W_F32 ? 0 : 1>(slot, r, h, w);
          uint32_t k0[8], k1[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float g = __uint_as_float(gr[j]);
            const float m0 = dequant_m(c0[j], sm_old);
            float m1;
            if constexpr (OPT == OPT_ADAMW) {
              float v1;
              adamw_moments(g, m0, dequant_v(c1[j], sv_old), sc, m1, v1);
              au = fmaxf(au, v1);     // max v'; sqrt is taken once per row below
              k1[j] = __float_as_uint(v1);
            } else if constexpr (OPT == OPT_SGDM) {
              m1 = sgdm_moment(g, w[j], m0, sc);
            } else {
              k1[j] = __float_as_uint(lion_dir(g, m0, sc));
              m1 = lion_moment(g, m0, sc);
            }
            am = fmaxf(am, fabsf(m1));
            k0[j] = __float_as_uint(m1);
          }
          tmem_st_32x32b_x8(t_keep + c * C::CW + h * 8, k0);
          if constexpr (KEEP2) tmem_st_32x32b_x8(t_keep + BN + c * C::CW + h * 8, k1);
        }
        tmem_st_wait();
        if (!ok) break;
        // The accumulator is not read again for this tile.
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tm_empty[buf]);
        // Combine the four column quarters of each row (bounded, abort-aware).
        red_sh[it & 1][0][h][r] = am;
        red_sh[it & 1][1][h][r] = au;
        mbar_arrive(&red_bar[it & 1]);
        ok = bwait(&red_bar[it & 1], (it >> 1) & 1, abort_flag, p.status, WAIT_RED, lim);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) break;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          am = fmaxf(am, red_sh[it & 1][0][k][r]);
          au = fmaxf(au, red_sh[it & 1][1][k][r]);
        }
        // sqrt is monotonic and correctly rounded: max sqrt(v') = sqrt(max v').
        const float sm_new = div_rn(am, 127.0f);
        const float sv_new = div_rn(sqrt_rn(au), 255.0f);
        const float im_new = block_inv(sm_new), iv_new = block_inv(sv_new);
        if (h == 0 && row < p.d_out) {
          p.m_scale[static_cast<int64_t>(jb) * p.d_out + row] = sm_new;
          if constexpr (C::TWO) p.v_scale[static_cast<int64_t>(jb) * p.d_out + row] = sv_new;
        }
        for (int c = 0; c < C::NCH; ++c, ++cseq) {
          const int s = static_cast<int>(cseq % NBUF);
          uint32_t k0[8], k1[8];
          tmem_ld_32x32b_x8(t_keep + c * C::CW + h * 8, k0);
          if constexpr (KEEP2) tmem_ld_32x32b_x8(t_keep + BN + c * C::CW + h * 8, k1);
          tmem_ld_wait();
          uint8_t* slot = st_base + s * C::SLOT_BYTES;
          uint8_t* sw = slot;
          uint8_t* smc = slot + C::W_CH;
          uint8_t* svc = slot + C::W_CH + C::M_CH;
          uint32_t cm[8], cv[8];
          float w[8];
          ld8<WK == W_F32 ? 0 : 1>(sw, r, h, w);
          bool near = false;  // a product within 1e-4 of a half-integer: decide those codes exactly
          // AdamW: the weight update and sqrt(v') of the 8 values with the
          // branch-free divide and square root, recomputed with the guarded
          // correctly rounded ones if an operand is outside their ranges.
          // A row whose new moments are all zero (its block maxima am, au are
          // 0) takes u = m' (0 / d, signed) and sqrt(v') = v' directly.
          float wn[8], sq[8];
          if constexpr (OPT == OPT_ADAMW) {
            if (am == 0.0f && au == 0.0f) {
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                wn[j] = __fsub_rn(__fmul_rn(sc.decay, w[j]), __fmul_rn(sc.step_size, __uint_as_float(k0[j])));
                sq[j] = __uint_as_float(k1[j]);
              }
            } else {
              bool bad = false;
#pragma unroll
              for (int j = 0; j < 8; ++j)
                adamw_apply_fast(w[j], __uint_as_float(k0[j]), __uint_as_float(k1[j]), sc, wn[j], sq[j], bad);
              if (__builtin_expect(bad, 0)) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const AdamWOut o = adamw_value_guarded(0.0f, w[j], __uint_as_float(k0[j]), __uint_as_float(k1[j]),
                                                         sc.b1, sc.omb1, sc.b2, sc.omb2, sc.decay, sc.step_size,
                                                         sc.inv_sqrt_bc2, sc.eps, 1);
                  wn[j] = o.w;
                  sq[j] = o.sq;
                }
              }
            }
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float m1 = __uint_as_float(k0[j]);
            float w1;
            if constexpr (OPT == OPT_ADAMW) {
              const float v1 = __uint_as_float(k1[j]);
              w1 = wn[j];
              cv[j] = quant_v_byte_fast(v1, sq[j], sv_new, iv_new, near);
            } else if constexpr (OPT == OPT_SGDM) {
              w1 = sgdm_apply(w[j], m1, sc);
            } else {
              w1 = lion_apply(w[j], __uint_as_float(k1[j]), sc);
            }
            w[j] = w1;
            cm[j] = quant_m_byte_fast(m1, sm_new, im_new, near);
          }
          // Rare (a product within 1e-4 of a half-integer): decide this
          // thread's 8 codes exactly. The new moments are read again from
          // tensor memory (a warp-wide load, hence the warp-uniform branch)
          // rather than kept in registers across the loop above.
          if (__any_sync(0xFFFFFFFFu, near)) {
            uint32_t r0[8], r1[8];
            tmem_ld_32x32b_x8(t_keep + c * C::CW + h * 8, r0);
            if constexpr (OPT == OPT_ADAMW) tmem_ld_32x32b_x8(t_keep + BN + c * C::CW + h * 8, r1);
            tmem_ld_wait();
            if (near) {
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                cm[j] = quant_m_byte(__uint_as_float(r0[j]), sm_new, im_new);
                if constexpr (OPT == OPT_ADAMW) {
                  const float v1 = __uint_as_float(r1[j]);
                  cv[j] = quant_v_byte(v1, sqrt_rn(v1), sv_new, iv_new);
                }
              }
            }
          }
          if constexpr (WK == W_F32) {
            st8_f32(sw, r, h, w);
          } else {
            uint4 b;
            const uint64_t idx8 =
                (static_cast<uint64_t>(row) * static_cast<uint64_t>(p.d_in) + (tn * BN + c * C::CW + h * 8)) >> 3;
            to_bf16x8<!DX>(w, p.sr_w != 0, idx8, 0u, p, b);
            st8_bf16(sw, r, h, b);
          }
          st8_codes(smc, r, h, cm);
          if constexpr (C::TWO) st8_codes(svc, r, h, cv);
          fence_proxy_async_smem();
          mbar_arrive(&st_written[s]);
        }
      }
      if constexpr (!C::Q8) {
        tc_fence_before_sync();
        __syncwarp();
        if constexpr (PAIR) {
          if (lane == 0) mbar_arrive_cluster(cluster_map(smem_u32(&tm_empty[buf]), 0u));
        } else {
          if (lane == 0) mbar_arrive(&tm_empty[buf]);
        }
      }
    }
  }
  if constexpr (DX) {
    if (warp >= 4 + C::EPI_WARPS && warp < C::DXMMA_WARP) {
      // ---------------------------------------------------------- converters (warps 20-23)
      // Per tile: load this thread's 8 items of W_old (tile row r = item / 8,
      // 8-column group g = item % 8), round to bf16, and once the MMAs of
      // the previous tile have released Wb, write them MN-major with the
      // 128-byte swizzle (row r is 128 bytes, group g lands at g ^ (r % 8)).
      // After the last tile of a column: write the dX partial out.
      const int ct = threadIdx.x - (128 + C::EPI_THREADS);
      const int q = warp & 3;  // TMEM lane quadrant of this warp
      int it = 0;
      uint32_t run_seq = 0;
      bool ok = p.num_kb > 0;
      for (int tile = tw.first; ok && tile < tw.end; tile += tw.step, ++it) {
        int tm, tn;
        walk_coords<DX, PAIR>(p, tile, prank, tm, tn);
        uint4 o[8];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          if constexpr (WK == W_F32) {
            float4 u[4][2];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int item = ct + 128 * (half * 4 + j);
              const int orow = tm * C::BM + (item >> 3), col = tn * BN + (item & 7) * 8;
              if (orow < p.d_out && col < p.d_in) {  // D_in % 8 == 0: all 8 columns or none
                const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.w_ptr) +
                                                                    static_cast<int64_t>(orow) * p.ld_w + col);
                u[j][0] = __ldcg(src);
                u[j][1] = __ldcg(src + 1);
              } else {
                u[j][0] = make_float4(0.f, 0.f, 0.f, 0.f);
                u[j][1] = u[j][0];
              }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
              o[half * 4 + j] = make_uint4(pack_bf16x2_rn(u[j][0].x, u[j][0].y), pack_bf16x2_rn(u[j][0].z, u[j][0].w),
                                           pack_bf16x2_rn(u[j][1].x, u[j][1].y), pack_bf16x2_rn(u[j][1].z, u[j][1].w));
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int item = ct + 128 * (half * 4 + j);
              const int orow = tm * C::BM + (item >> 3), col = tn * BN + (item & 7) * 8;
              o[half * 4 + j] = (orow < p.d_out && col < p.d_in)
                                    ? __ldcg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.w_ptr) +
                                                                            static_cast<int64_t>(orow) * p.ld_w + col))
                                    : make_uint4(0u, 0u, 0u, 0u);
            }
          }
        }
        ok = bwait(&wb_empty, (it & 1) ^ 1u, abort_flag, p.status, WAIT_WB_EMPTY, lim);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) break;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int item = ct + 128 * j;
          const int rr = item >> 3, g = item & 7;
          *reinterpret_cast<uint4*>(wb_base + rr * 128 + ((g ^ (rr & 7)) << 4)) = o[j];
        }
        fence_proxy_async_smem();
        mbar_arrive(&wb_full);

        if (tile + 1 == tw.end || (tile + 1) % p.tiles_m == 0) {
          ok = bwait(&dx_full, run_seq & 1u, abort_flag, p.status, WAIT_DX_FULL, lim);
          ok = __all_sync(0xFFFFFFFFu, ok);
          if (!ok) break;
          tc_fence_after_sync();
          const int run = tn - tw.first / p.tiles_m;
          float* slab = p.dx_ws + (static_cast<int64_t>(blockIdx.x) * p.dx_runs + run) * p.dx_slab;
          write_dx_partial<BN>(slab, tmem_base + static_cast<uint32_t>(C::DX_COL), q, lane, p.num_kb, p.dx_l2 != 0);
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&dx_empty);
          ++run_seq;
        }
      }
    }
  }

  if constexpr (C::DX_ISSUER) {
    if (warp == C::DXMMA_WARP && lane == 0) {
      // ---------------------------------------------------------- MMA issuer (input gradient, warp 24)
      // dX[128 tokens of stage kb][BN] += dY[tokens][128 rows of the tile] * Wb,
      // into the persistent partial of the current tile column; the stage is
      // released once both issuers' MMAs on it have completed.
      uint32_t kseq = 0;
      bool ok = true;
      int it = 0;
      uint32_t runs_done = 0;  // dX partials handed to the converter warps
      for (int tile = tw.first; ok && tile < tw.end; tile += tw.step, ++it) {
        // The first tile of a column starts a fresh partial.
        const bool run_first = tile == tw.first || tile % p.tiles_m == 0;
        const bool run_last = tile + 1 == tw.end || (tile + 1) % p.tiles_m == 0;
        for (int kb = 0; kb < p.num_kb; ++kb, ++kseq) {
          const int s = static_cast<int>(kseq % STAGES);
          const uint32_t ph = (kseq / STAGES) & 1u;
          if (!bwait(&op_full[s], ph, abort_flag, p.status, WAIT_OP_FULL, lim)) { ok = false; break; }
          if (kb == 0 && !dx_tile_ready(run_first, runs_done, it, &dx_empty, &wb_full, abort_flag, p.status, lim)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          issue_dx_stage<C>(smem_u32(op_base + s * C::STAGE_BYTES), smem_u32(wb_base), tmem_base, kb, run_first);
          umma_commit(&op_empty[s]);
        }
        if (!ok) break;
        if (p.num_kb > 0) {
          umma_commit(&wb_empty);
          if (run_last) { umma_commit(&dx_full); ++runs_done; }
        }
      }
      if (!ok) {
        // Let every dX MMA already issued finish before TMEM is released.
        umma_commit(&dx_drain_bar);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&dx_drain_bar, 0)) {
          if (globaltimer_ns() - t0 > 200000000ull) { atomicCAS(p.status, 0u, WAIT_MMA_DRAIN); break; }
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  // Neither CTA of a pair leaves (or frees tensor memory) while the other
  // may still arrive on its barriers or read its accumulator half.
  if constexpr (PAIR) cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <int OPT, int WK, int MK, int BN, int STAGES, int NBUF, bool DX, bool GA = false, bool NARROW = false,
          bool WIDE = false, bool PAIR = false>
cudaError_t launch_tc_variant(const WgradTcParams& p, int grid, cudaStream_t stream) {
  using C = TcCfg<OPT, WK, MK, BN, STAGES, NBUF, DX, GA, NARROW, WIDE, PAIR>;
  auto kern = wgrad_step_tc_kernel<OPT, WK, MK, BN, STAGES, NBUF, DX, GA, NARROW, WIDE, PAIR>;
  // The opt-in shared-memory size is a per-device function attribute: set
  // it once per device (bit d of the mask) before the first launch there.
  static unsigned long long attr_mask = 0ull;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(__atomic_load_n(&attr_mask, __ATOMIC_ACQUIRE) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&attr_mask, bit, __ATOMIC_ACQ_REL);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(C::NUM_THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see griddep_wait() in the kernel
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if constexpr (PAIR) {
    // Clusters of two; at most as many pairs as the device keeps resident
    // at once (each pair walks its own share of the tiles).
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
    static int max_pairs[64] = {};
    int mp = __atomic_load_n(&max_pairs[dev & 63], __ATOMIC_ACQUIRE);
    if (mp == 0) {
      cudaLaunchConfig_t q = cfg;
      q.gridDim = dim3(2);
      q.attrs = &attr[1];  // the cluster shape alone
      q.numAttrs = 1;
      e = cudaOccupancyMaxActiveClusters(&mp, kern, &q);
      if (e != cudaSuccess) return e;
      if (mp < 1) return cudaErrorInvalidConfiguration;
      __atomic_store_n(&max_pairs[dev & 63], mp, __ATOMIC_RELEASE);
    }
    int pairs = grid / 2;
    if (pairs > mp) pairs = mp;
    if (pairs < 1) return cudaErrorInvalidValue;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
  } else {
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
  }
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace forge
