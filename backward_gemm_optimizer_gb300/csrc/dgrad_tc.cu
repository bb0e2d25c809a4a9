// dgrad_tc.cu -- input gradient dX = dY W_old on tcgen05 tensor cores
// (FORGE, Remark 1 in Appendix A: the input gradient must read the weights
// before the fused step overwrites them, so it is enqueued first).
//
// Tiles of 128 tokens x 128 input features (128 x 256 for bf16 weights on
// long token axes), or, on short token axes (BT <= 512), of all the tokens
// (MB = 2 or 4 blocks of 128, one accumulator each in tensor memory) x 128
// features; the contraction runs over D_out in 128-row stages (64 on the
// wider and on the all-token tiles). A = dY is K-major (D_out contiguous), B = W is
// MN-major (D_in contiguous). bf16 weights are fed by TMA directly; fp32
// master weights are staged by TMA in 64-row slots and eight converter
// warps round them to bf16 (round-to-nearest-even) into the swizzled
// operand layout before the MMA consumes them.
//
// With a workspace, layers with at most half as many tiles as SMs split the
// contraction over D_out into S equal parts run by S CTAs each (one wave);
// the parts' fp32 partial sums are added in a fixed order by a fix-up
// kernel, so more SMs work on a skinny dX.
//
// What a CTA takes in from L2 sets the pace: each SM receives about
// 110 GB/s (128 x 128 tiles with fp32 weights: 11 MB per CTA in 110 us;
// bf16 weights 7.3 MB in 66 us), so a tile's operand bytes per output
// decide. An all-token tile reads each weight once instead of once per
// 128-token block (up-projection, BT 512, fp32 weights: 5.5 MB instead of
// 11 MB per CTA).
//
// Warp roles (512 threads): 0 dY producer, 1 MMA issuer + TMEM owner,
// 2 W producer, 4-7 epilogue (TMEM lane quadrant = warp % 4, thread =
// token row), 8-15 converters (fp32 weights only). All waits are bounded.
#include <cstdint>

#include "forge_math.cuh"
#include "forge_params.h"
#include "forge_ptx.cuh"

namespace forge {

namespace {

constexpr int BM = 128;
constexpr int NUM_THREADS = 512;
constexpr int CONV_THREADS = 256;          // warps 8-15

// Rings: dY tiles and bf16 W tiles (filled by TMA, or by the converters
// from the fp32 staging ring), of the same depth and released together by
// one MMA commit per stage (a commit is not free: 68 -> 66 us with one
// instead of two), and the fp32 staging tiles (released by the converters
// once read). 128-token tiles are BN = 128 input features wide, or 256 for
// bf16 weights when the wider tiles still fill the GPU (half the operand
// traffic of dY per output).
template <bool F32W, int BN_, int MB_ = 1>
struct DCfg {
  static constexpr int BN = BN_;
  static constexpr int MB = MB_;   // 128-token blocks per tile
  // Rows of D_out per stage: 128 on 128-column tiles -- each stage costs a
  // fixed hand-over time besides its bytes, so fewer, larger stages win
  // (up-projection, BT 512, bf16 weights: 105 -> 72 us); fp32 weights are
  // staged in 64-row slots, two per stage. 64 on 128 x 256 tiles, whose
  // ring would shrink to two stages (measured slower).
  // All-token tiles: 64-row stages (32-row ones, with the 64-byte swizzle
  // and twice the ring depth, measured slower: 81 -> 86 us on the
  // down-projection with fp32 weights, 46 -> 61 us at BT 256 with bf16).
  static constexpr int BK = MB > 1 ? 64 : (BN == 256 ? 64 : 128);
  // dY boxes: 64 K columns x 128 token rows (128-byte rows, 128-byte swizzle).
  static constexpr int A_BOX_K = 64;              // K columns per box
  static constexpr int A_BOX = BM * 128;          // bytes per box
  static constexpr int A_BLOCK = BM * BK * 2;    // one token block of dY, K-major: BK / 64 boxes, A_BOX apart
  static constexpr int A_BYTES = MB * A_BLOCK;   // the stage's token blocks, A_BLOCK apart
  static constexpr int B_BYTES = BK * BN * 2;    // bf16 W tile, MN-major, 64-column atoms BK * 128 bytes apart
  static constexpr int ATOM = BK * 128;          // bytes of one 64-column atom (box) of the bf16 W tile
  // fp32 staging slot: 64 rows of the stage (two per 128-row stage), 32 on
  // all-token tiles (whose dY stages leave room for four small slots), as
  // four 32-column swizzled boxes.
  static constexpr int STG_ROWS = MB > 1 ? 32 : 64;
  static constexpr int STG_BYTES = STG_ROWS * BN * 4;
  // Ring depths (stages). All-token tiles: two stages of four token blocks
  // (a ring of one (stage, block) entry per 16 KB, each released once its
  // products were done, measured slower: 81 -> 99 us on the down-projection
  // with fp32 weights), three or four of two.
  static constexpr int SA = MB == 4 ? 2 : MB == 2 ? (F32W ? 3 : 4) : (F32W ? 2 : (BN == 256 ? 4 : 3));
  static constexpr int SB = SA;
  static constexpr int SS = F32W ? (MB > 1 ? 4 : 3) : 0;
  static constexpr int A_OFF = 0;
  static constexpr int B_OFF = SA * A_BYTES;
  static constexpr int S_OFF = B_OFF + SB * B_BYTES;
  static constexpr int SMEM_BYTES = 1024 + S_OFF + SS * STG_BYTES;
  // Accumulator buffers: two (the next tile's products run while the last
  // one is drained) where they fit in the 512 columns, else one.
  static constexpr int NBUF = 2 * MB * BN <= 512 ? 2 : 1;
  static constexpr int TMEM_COLS = NBUF * MB * BN;
  // 128-token tiles: A = dY (M = 128 tokens, K-major), B = W (N = BN
  // features, MN-major). All-token tiles swap the operands: A = W (M = 128
  // features, MN-major), B = dY (N = 256 tokens, K-major) -- one product per
  // 256 tokens instead of one per 128, a third fewer operand bytes read from
  // shared memory per multiply-add; the accumulator is then dX transposed
  // (tensor-memory lane = feature, column = token).
  static constexpr bool SWAP = MB > 1;
  static constexpr int DRAIN_WARPS = SWAP ? 12 : 4;   // warps that drain the accumulator
  static constexpr int NT = 256;                  // tokens per product (swapped)
  static constexpr uint32_t IDESC = SWAP ? make_idesc_bf16(BM, NT, 1, 0) : make_idesc_bf16(BM, BN, 0, 1);
  static_assert(!F32W || BN == 128, "fp32 weight staging is sized for 128-column tiles");
  static_assert(MB == 1 || (BN == 128 && (MB == 2 || MB == 4)), "all-token tiles: 2 or 4 blocks x 128 columns");
  static_assert(!SWAP || (MB * BM) % NT == 0, "whole 256-token products");
  static_assert(BK % A_BOX_K == 0 && (!F32W || BK % STG_ROWS == 0), "stage rows");
  static_assert(SA == SB, "one empty barrier per stage serves the dY and the bf16 W ring");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
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

// After an abort: wait (bounded) for the last fills issued on a ring.
__device__ __forceinline__ void ddrain(uint64_t* full, int ring, uint32_t issued, unsigned int* status) {
  const uint32_t first = issued > static_cast<uint32_t>(ring) ? issued - ring : 0u;
  for (uint32_t k = first; k < issued; ++k) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(&full[k % ring], (k / ring) & 1u))
      if (globaltimer_ns() - t0 > 200000000ull) { atomicCAS(status, 0u, WAIT_DRAIN); break; }
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

// The (tile, stage range) segments a CTA processes, in order: whole tiles
// blockIdx.x, blockIdx.x + gridDim.x, ... or, with the contraction split in
// S = splitk parts (grid = num_tiles * S, one wave), the single segment
// (tile c % num_tiles, stages [s num_kb / S, (s + 1) num_kb / S)) with
// s = c / num_tiles: the token tiles that share a column of W read the same
// rows of it at the same time, so W comes from DRAM once. Every role walks
// the same sequence.
// (The split is a template parameter: the one-kernel walk compiles to the
// plain tile loop -- a runtime walk cost the one-kernel dgrad 4-6 %.)
struct SegWalk {
  int pos, end, stride;
};

template <bool SPLIT>
__device__ __forceinline__ SegWalk seg_walk(const DgradParams& p) {
  if constexpr (SPLIT) return SegWalk{0, 1, 0};
  else return SegWalk{static_cast<int>(blockIdx.x), p.num_tiles, static_cast<int>(gridDim.x)};
}

template <bool SPLIT>
__device__ __forceinline__ bool seg_next(const DgradParams& p, SegWalk& w, int& tile, int& kb0, int& kb1, int& rot) {
  if (w.pos >= w.end) return false;
  if constexpr (SPLIT) {
    const int part = static_cast<int>(blockIdx.x) / p.num_tiles;
    tile = static_cast<int>(blockIdx.x) % p.num_tiles;
    kb0 = static_cast<int>(static_cast<int64_t>(part) * p.num_kb / p.splitk);
    kb1 = static_cast<int>(static_cast<int64_t>(part + 1) * p.num_kb / p.splitk);
    w.pos = 1;
  } else {
    tile = w.pos;
    kb0 = 0;
    kb1 = p.num_kb;
    w.pos += w.stride;
  }
  // With k_rotate, the tiles of a row of tiles (which share the dY rows of
  // every stage) start their stage walks at evenly spaced offsets: column
  // tn at stage kb0 + tn * (kb1 - kb0) / tiles_n, wrapping round.
  rot = 0;
  if (p.k_rotate && kb1 > kb0) {
    int tm, tn;
    dtile(tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
    rot = static_cast<int>(static_cast<int64_t>(tn) * (kb1 - kb0) / p.tiles_n);
  }
  return true;
}

// Stage i of a segment's walk [kb0, kb1) started at kb0 + rot.
__device__ __forceinline__ int stage_at(int kb0, int kb1, int rot, int i) {
  const int kb = kb0 + rot + i;
  return kb >= kb1 ? kb - (kb1 - kb0) : kb;
}

template <bool F32W, int BN, bool SPLIT, int MB>
__global__ void __launch_bounds__(NUM_THREADS, 1) dgrad_tc_kernel(const __grid_constant__ DgradParams p) {
  using C = DCfg<F32W, BN, MB>;
  constexpr int NBUF = C::NBUF;
  constexpr int A_BYTES = C::A_BYTES, B_BYTES = C::B_BYTES, STG_BYTES = C::STG_BYTES, TMEM_COLS = C::TMEM_COLS;
  constexpr int BK = C::BK;
  constexpr uint32_t IDESC = C::IDESC;
  constexpr int SA = C::SA, SB = C::SB, SS = C::SS > 0 ? C::SS : 1;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t a_full[SA], a_empty[SA], b_full[SB], s_full[SS], s_empty[SS];
  __shared__ __align__(8) uint64_t tm_full[NBUF], tm_empty[NBUF], drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a_ring = smem + C::A_OFF;
  uint8_t* b_ring = smem + C::B_OFF;
  uint8_t* s_ring = smem + C::S_OFF;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &abort_sh;
  const uint64_t lim = p.timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SA; ++s) { mbar_init(&a_full[s], 1); mbar_init(&a_empty[s], 1); }
    for (int s = 0; s < SB; ++s) mbar_init(&b_full[s], F32W ? CONV_THREADS : 1);
    for (int s = 0; s < SS; ++s) { mbar_init(&s_full[s], 1); mbar_init(&s_empty[s], CONV_THREADS); }
    for (int b = 0; b < NBUF; ++b) { mbar_init(&tm_full[b], 1); mbar_init(&tm_empty[b], C::DRAIN_WARPS); }
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
  // A programmatic dependent (as the step kernel): the set-up above overlaps
  // the previous kernel's tail; memory is touched after it completes.
  griddep_launch_dependents();
  griddep_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ dY producer
    if (lane == 0) {
      uint32_t k = 0;
      bool ok = true;
      SegWalk w = seg_walk<SPLIT>(p);
      int tile, kb0, kb1, rot;
      while (ok && seg_next<SPLIT>(p, w, tile, kb0, kb1, rot)) {
        int tm, tn;
        dtile(tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
        for (int i = 0; i < kb1 - kb0; ++i, ++k) {
          const int kb = stage_at(kb0, kb1, rot, i);
          const int s = static_cast<int>(k % SA);
          if (!dwait(&a_empty[s], ((k / SA) & 1u) ^ 1u, abort_flag, p.status, WAIT_OP_EMPTY, lim)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&a_full[s], A_BYTES);
#pragma unroll
          for (int b = 0; b < MB; ++b)
#pragma unroll
            for (int h = 0; h < BK / C::A_BOX_K; ++h)
              tma_load_2d(a_ring + s * A_BYTES + b * C::A_BLOCK + h * C::A_BOX, &p.tm_dy, &a_full[s],
                          kb * BK + h * C::A_BOX_K, (tm * MB + b) * BM);
        }
      }
      if (!ok) ddrain(a_full, SA, k, p.status);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ W producer
    if (lane == 0) {
      uint32_t k = 0;
      uint32_t ks = 0;  // fp32 staging slots filled
      bool ok = true;
      SegWalk w = seg_walk<SPLIT>(p);
      int tile, kb0, kb1, rot;
      while (ok && seg_next<SPLIT>(p, w, tile, kb0, kb1, rot)) {
        int tm, tn;
        dtile(tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
        for (int i = 0; i < kb1 - kb0; ++i, ++k) {
          const int kb = stage_at(kb0, kb1, rot, i);
          if constexpr (F32W) {
            for (int half = 0; half < BK / C::STG_ROWS; ++half, ++ks) {
              const int s = static_cast<int>(ks % SS);
              if (!dwait(&s_empty[s], ((ks / SS) & 1u) ^ 1u, abort_flag, p.status, WAIT_OP_EMPTY, lim)) {
                ok = false;
                break;
              }
              uint8_t* stg = s_ring + s * STG_BYTES;
              mbar_arrive_expect_tx(&s_full[s], STG_BYTES);
#pragma unroll
              for (int bb = 0; bb < 4; ++bb)
                tma_load_2d(stg + bb * (C::STG_ROWS * 128), &p.tm_w, &s_full[s], tn * BN + bb * 32,
                            kb * BK + half * C::STG_ROWS);
            }
            if (!ok) break;
          } else {
            // Both rings have the same depth and one commit per stage
            // releases the dY and W slots together (a_empty).
            const int s = static_cast<int>(k % SB);
            if (!dwait(&a_empty[s], ((k / SB) & 1u) ^ 1u, abort_flag, p.status, WAIT_OP_EMPTY, lim)) {
              ok = false;
              break;
            }
            uint8_t* b = b_ring + s * B_BYTES;
            mbar_arrive_expect_tx(&b_full[s], B_BYTES);
#pragma unroll
            for (int bb = 0; bb < BN / 64; ++bb)
              tma_load_2d(b + bb * C::ATOM, &p.tm_w, &b_full[s], tn * BN + bb * 64, kb * BK);
          }
        }
      }
      if (!ok) {
        if constexpr (F32W) ddrain(s_full, SS, ks, p.status);
        else ddrain(b_full, SB, k, p.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t k = 0;
      bool ok = true;
      int it = 0;
      SegWalk w = seg_walk<SPLIT>(p);
      int tile, kb0, kb1, rot;
      for (; ok && seg_next<SPLIT>(p, w, tile, kb0, kb1, rot); ++it) {
        const int buf = it % NBUF;
        if (!dwait(&tm_empty[buf], ((it / NBUF) & 1) ^ 1u, abort_flag, p.status, WAIT_TMEM_EMPTY, lim)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d = tmem_base + static_cast<uint32_t>(buf * MB * BN);
        for (int i = 0; i < kb1 - kb0; ++i, ++k) {
          const int kb = stage_at(kb0, kb1, rot, i);
          const int sa = static_cast<int>(k % SA), sb = static_cast<int>(k % SB);
          if (!dwait(&a_full[sa], (k / SA) & 1u, abort_flag, p.status, WAIT_OP_FULL, lim) ||
              !dwait(&b_full[sb], (k / SB) & 1u, abort_flag, p.status, WAIT_OP_FULL, lim)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a0 = smem_u32(a_ring + sa * A_BYTES);
          const uint32_t b0 = smem_u32(b_ring + sb * B_BYTES);
          // dY: K-major, 128-byte swizzle, 8-row groups 1024 bytes apart.
          // W: MN-major, 64-column atoms C::ATOM bytes apart, 8-row K groups
          // of 1024 bytes. Both descriptors are built once per stage; a K
          // step only moves the 14-bit start-address field (16-byte units;
          // shared addresses stay below 2^18 bytes, so it never carries).
          const uint64_t ad0 = make_smem_desc(a0, 16, 1024, 2);
          const uint64_t bd0 = make_smem_desc(b0, C::ATOM, 1024, 2);
          if constexpr (C::SWAP) {
            // A = the W tile (descriptor bd0), B = 256 tokens of dY: token
            // blocks 2 nb and 2 nb + 1, contiguous (ad0 + nb * 2 A_BLOCK).
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t wstep = static_cast<uint64_t>((kk * 2048) >> 4);
              const uint64_t ystep = static_cast<uint64_t>(((kk % 4) * 32) >> 4);
#pragma unroll
              for (int nb = 0; nb < MB * BM / C::NT; ++nb)
                umma_f16(d + static_cast<uint32_t>(nb * C::NT), bd0 + wstep,
                         ad0 + static_cast<uint64_t>((nb * 2 * C::A_BLOCK) >> 4) + ystep, IDESC,
                         (i > 0 || kk > 0) ? 1u : 0u);
            }
          } else {
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // A K step of 16 elements advances 32 bytes within a box (boxes
            // A_BOX bytes apart); B's advances 16 rows = 2048 bytes.
            constexpr int KPB = C::A_BOX_K / 16;  // K steps per box
            const uint64_t astep = static_cast<uint64_t>(((kk / KPB) * C::A_BOX + (kk % KPB) * 32) >> 4);
            const uint64_t bstep = static_cast<uint64_t>((kk * 2048) >> 4);
            // Token block b: its own A tile (A_BLOCK bytes on) and
            // accumulator (BN columns on), the same B.
#pragma unroll
            for (int b = 0; b < MB; ++b)
              umma_f16(d + static_cast<uint32_t>(b * BN), ad0 + static_cast<uint64_t>((b * C::A_BLOCK) >> 4) + astep,
                       bd0 + bstep, IDESC, (i > 0 || kk > 0) ? 1u : 0u);
          }
          }
          umma_commit(&a_empty[sa]);  // releases the stage's dY slot and its bf16 W slot
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
  } else if (warp >= 4) {
    if (warp >= 8 && F32W) {
      // ------------------------------------------------------------ fp32 -> bf16 converters
      // The fp32 rows landed by TMA as four [STG_ROWS rows][32 columns] boxes
      // with the 128-byte swizzle. Work item = (box, K row, 8-column group): read
      // two 16-byte chunks, round to bf16, write one 16-byte chunk of the
      // MN-major swizzled operand. Consecutive threads take consecutive K
      // rows, so both the reads and the writes are bank-conflict free.
      const int ct = threadIdx.x - 256;
      uint32_t k = 0, ks = 0;
      bool ok = true;
      SegWalk w = seg_walk<SPLIT>(p);
      int tile, kb0, kb1, rot;
      while (ok && seg_next<SPLIT>(p, w, tile, kb0, kb1, rot)) {
        for (int i = 0; i < kb1 - kb0; ++i, ++k) {
          const int kb = stage_at(kb0, kb1, rot, i);
          const int sb = static_cast<int>(k % SB);
          uint8_t* b = b_ring + sb * B_BYTES;
          // A stage's BK rows arrive as BK / 64 staging slots of 64 rows.
          for (int half = 0; half < BK / C::STG_ROWS; ++half, ++ks) {
            const int ss = static_cast<int>(ks % SS);
            ok = dwait(&s_full[ss], (ks / SS) & 1u, abort_flag, p.status, WAIT_OP_FULL, lim) &&
                 (half > 0 || dwait(&a_empty[sb], ((k / SB) & 1u) ^ 1u, abort_flag, p.status, WAIT_OP_EMPTY, lim));
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) break;
            const uint8_t* stg = s_ring + ss * STG_BYTES;
            // Work items of the slot: 4 boxes x STG_ROWS rows x 4 groups of 8
            // columns, STG_ROWS / 16 per thread.
            constexpr int NJ = C::STG_ROWS / 16;
            uint4 o[NJ];
            int dst[NJ];
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
              const int i = ct + CONV_THREADS * j;
              const int kr = i % C::STG_ROWS;                // row within the staging slot
              const int hh = (i / C::STG_ROWS) & 3;          // 8-column group within the 32-column box
              const int bb = i / (4 * C::STG_ROWS);          // box (32 columns)
              const uint8_t* src = stg + bb * (C::STG_ROWS * 128) + kr * 128;
              const float4 u0 = *reinterpret_cast<const float4*>(src + (((2 * hh) ^ (kr & 7)) << 4));
              const float4 u1 = *reinterpret_cast<const float4*>(src + (((2 * hh + 1) ^ (kr & 7)) << 4));
              o[j].x = pack_bf16x2_rn(u0.x, u0.y);
              o[j].y = pack_bf16x2_rn(u0.z, u0.w);
              o[j].z = pack_bf16x2_rn(u1.x, u1.y);
              o[j].w = pack_bf16x2_rn(u1.z, u1.w);
              const int n = bb * 32 + hh * 8;    // column within the 128-wide tile
              const int row = half * C::STG_ROWS + kr;  // K row of the stage (row % 8 == kr % 8)
              dst[j] = (n >> 6) * C::ATOM + row * 128 + ((((n & 63) >> 3) ^ (kr & 7)) << 4);
            }
#pragma unroll
            for (int j = 0; j < NJ; ++j) *reinterpret_cast<uint4*>(b + dst[j]) = o[j];
            fence_proxy_async_smem();
            // Release the staging slot only now: the stores above consume every
            // value loaded from it, so those loads have returned before the next
            // TMA fill may overwrite the slot.
            mbar_arrive(&s_empty[ss]);
          }
          if (!ok) break;
          mbar_arrive(&b_full[sb]);
        }
      }
    }
    // All-token tiles drain their transposed accumulator with warps 4-15
    // (three groups of four, one warp per lane quadrant in each); the
    // converters join once their last stage is written.
    if (warp < 8 || C::SWAP) {
      // ------------------------------------------------------------ epilogue
      const int q = warp & 3;
      const int r = q * 32 + lane;
      int it = 0;
      bool ok = true;
      SegWalk w = seg_walk<SPLIT>(p);
      int tile, kb0, kb1, rot;
      for (; ok && seg_next<SPLIT>(p, w, tile, kb0, kb1, rot); ++it) {
        int tm, tn;
        dtile(tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
        const int buf = it % NBUF;
        ok = dwait(&tm_full[buf], (it / NBUF) & 1, abort_flag, p.status, WAIT_TMEM_FULL, lim);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) break;
        tc_fence_after_sync();
        if constexpr (C::SWAP) {
          // Transposed accumulator: this thread's lane is feature r of the
          // tile, its columns the tokens. Each load brings 16 tokens; a warp's
          // store of one token covers 32 consecutive features.
          const int col = tn * BN + r;
          const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * MB * BN);
          float* slot = SPLIT ? p.part + static_cast<int64_t>(blockIdx.x) * MB * BM * BN + r : nullptr;
          const int group = (warp - 4) >> 2;   // 0..2: token chunks group, group + 3, ...
#pragma unroll 1
          for (int c = group; c < MB * BM / 16; c += 3) {
            uint32_t acc[16];
            if (p.num_kb > 0) {
              tmem_ld_32x32b_x16(t_lane + c * 16, acc);
              tmem_ld_wait();
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j) acc[j] = 0u;
            }
            const int t0 = tm * MB * BM + c * 16;
            if constexpr (SPLIT) {
#pragma unroll
              for (int j = 0; j < 16; ++j) slot[static_cast<int64_t>(c * 16 + j) * BN] = __uint_as_float(acc[j]);
              continue;
            }
            if (col >= p.d_in) continue;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int t = t0 + j;
              if (t >= p.bt) break;
              if (p.dx_bf16)
                static_cast<uint16_t*>(p.dX)[static_cast<int64_t>(t) * p.ld_dx + col] =
                    static_cast<uint16_t>(f32_to_bf16_rne(__uint_as_float(acc[j])));
              else
                static_cast<float*>(p.dX)[static_cast<int64_t>(t) * p.ld_dx + col] = __uint_as_float(acc[j]);
            }
          }
        } else {
#pragma unroll 1
        for (int blk = 0; blk < MB; ++blk) {
          const int row = (tm * MB + blk) * BM + r;
          const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                  static_cast<uint32_t>((buf * MB + blk) * BN);
          // A split contraction: this CTA's fp32 partial sum goes to its slot
          // (row blk * 128 + r of an MB * 128 x BN slab), for the fix-up kernel
          // to add in order.
          constexpr bool partial = SPLIT;
          float* slot = partial ? p.part + ((static_cast<int64_t>(blockIdx.x) * MB + blk) * BM + r) * BN : nullptr;
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
            if (partial) {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                reinterpret_cast<float4*>(slot + c * 16)[j] =
                    make_float4(__uint_as_float(acc[4 * j]), __uint_as_float(acc[4 * j + 1]),
                                __uint_as_float(acc[4 * j + 2]), __uint_as_float(acc[4 * j + 3]));
              continue;
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
                  b[j] = pack_bf16x2_rn(__uint_as_float(acc[2 * j]), __uint_as_float(acc[2 * j + 1]));
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
        }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tm_empty[buf]);
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

// The second half of a split dgrad: for each tile, adds the partial sums of
// its S parts in increasing part order -- the order of the contraction, and
// a fixed one, so dX is bit-reproducible -- and stores dX. Part s of tile t
// is CTA t + s * num_tiles's slot of `rows` x bn values. One block per
// (tile, 16 token rows).
__global__ void __launch_bounds__(256) dgrad_fixup_kernel(const DgradFixupParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // the step may be scheduled
  const int tile = blockIdx.x;
  int tm, tn;
  dtile(tile, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
  const int nq = p.bn / 4;  // 16-byte pieces per row
  for (int idx = threadIdx.x; idx < 16 * nq; idx += blockDim.x) {
    const int rr = static_cast<int>(blockIdx.y) * 16 + idx / nq;
    const int col = (idx % nq) * 4;
    const int t = tm * p.rows + rr, i = tn * p.bn + col;
    if (t >= p.bt || i >= p.d_in) continue;  // D_in % 8 == 0: 4 columns all in or all out
    float4 v[4];
#pragma unroll
    for (int s = 0; s < 4; ++s)
      v[s] = s < p.parts ? __ldcg(reinterpret_cast<const float4*>(
                               p.part + ((static_cast<int64_t>(s) * p.num_tiles + tile) * p.rows + rr) * p.bn + col))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    auto add = [&acc](const float4& u) {
      acc.x = __fadd_rn(acc.x, u.x);
      acc.y = __fadd_rn(acc.y, u.y);
      acc.z = __fadd_rn(acc.z, u.z);
      acc.w = __fadd_rn(acc.w, u.w);
    };
#pragma unroll
    for (int s = 0; s < 4; ++s)
      if (s < p.parts) add(v[s]);
    for (int s = 4; s < p.parts; ++s)
      add(__ldcg(reinterpret_cast<const float4*>(
          p.part + ((static_cast<int64_t>(s) * p.num_tiles + tile) * p.rows + rr) * p.bn + col)));
    if (p.dx_bf16) {
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.dX) + static_cast<int64_t>(t) * p.ld_dx + i) =
          make_uint2(pack_bf16x2_rn(acc.x, acc.y), pack_bf16x2_rn(acc.z, acc.w));
    } else {
      *reinterpret_cast<float4*>(static_cast<float*>(p.dX) + static_cast<int64_t>(t) * p.ld_dx + i) = acc;
    }
  }
}

template <bool F32W, int BN, bool SPLIT, int MB = 1>
cudaError_t launch_d(const DgradParams& p, int grid, cudaStream_t stream) {
  using C = DCfg<F32W, BN, MB>;
  // The stage depth and staging rows the host encoded the tensor maps and
  // num_kb for must be the kernel's: a mismatch would overfill the
  // shared-memory rings.
  if (p.bk != C::BK || p.mb != MB || (F32W && p.stg_rows != C::STG_ROWS) || (p.w_f32 != nullptr) != F32W ||
      (p.splitk != 0) != SPLIT)
    return cudaErrorInvalidValue;
  auto kern = dgrad_tc_kernel<F32W, BN, SPLIT, MB>;
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
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

cudaError_t launch_dgrad_fixup(const DgradFixupParams& p, cudaStream_t stream) {
  if (p.bt == 0 || p.d_in == 0 || p.num_tiles == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  if (p.rows % 16 != 0) return cudaErrorInvalidValue;
  cfg.gridDim = dim3(static_cast<unsigned>(p.num_tiles), static_cast<unsigned>(p.rows / 16));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, dgrad_fixup_kernel, p);
}

// All-token tiles (MB = 2 or 4 blocks of 128 tokens, 128 columns).
template <int MB>
cudaError_t launch_mb(const DgradParams& p, int grid, cudaStream_t stream) {
  if (p.bn != 128) return cudaErrorInvalidValue;
  if (p.splitk)
    return p.w_f32 ? launch_d<true, 128, true, MB>(p, grid, stream) : launch_d<false, 128, true, MB>(p, grid, stream);
  return p.w_f32 ? launch_d<true, 128, false, MB>(p, grid, stream) : launch_d<false, 128, false, MB>(p, grid, stream);
}

cudaError_t launch_dgrad_tc(const DgradParams& p, int grid, cudaStream_t stream) {
  if (p.mb == 4) return launch_mb<4>(p, grid, stream);
  if (p.mb == 2) return launch_mb<2>(p, grid, stream);
  if (p.mb != 1) return cudaErrorInvalidValue;
  if (p.splitk) {
    if (p.w_f32) return p.bn == 128 ? launch_d<true, 128, true>(p, grid, stream) : cudaErrorInvalidValue;
    return p.bn == 256 ? launch_d<false, 256, true>(p, grid, stream) : cudaErrorInvalidValue;
  }
  if (p.w_f32) return p.bn == 128 ? launch_d<true, 128, false>(p, grid, stream) : cudaErrorInvalidValue;
  return p.bn == 256 ? launch_d<false, 256, false>(p, grid, stream) : launch_d<false, 128, false>(p, grid, stream);
}

}  // namespace forge
