/*
 * forge.h -- C ABI of the fused weight-gradient + optimizer-step library
 * for one NVIDIA GB300 GPU (sm_103a).
 *
 * What it computes (FORGE, "Fused On-Register Gradient Elimination for
 * Memory-Efficient LLM Training", arXiv 2606.22932):
 *
 *   For a linear layer Y = X W^T (section 2.1, Eq. 2) with
 *     X  : BT x D_in   (saved input),
 *     dY : BT x D_out  (upstream gradient),
 *     W  : D_out x D_in,
 *   the weight gradient G = dY^T X (Eq. 3) is formed one 128-row tile at a
 *   time, accumulated over the token axis in fp32 (Eq. 5, Algorithm 1
 *   phase 1), and each accumulator tile is consumed at once by an
 *   element-wise optimizer step (Algorithm 1 phase 2). Only the updated
 *   weight and moment tiles are written (Algorithm 1 phase 3); G is never
 *   stored and no gradient-sized buffer is ever allocated (Proposition 3).
 *   Proposition 1 (Appendix A) makes the result equal to "materialise G,
 *   then step" up to the summation order of G (Corollary 1).
 *
 * Conventions shared by every entry point
 *   - All tensors are row-major 2-D views described by forge_tensor.
 *     "ld" is the distance in elements between consecutive rows
 *     (ld >= cols). The caller allocates and owns every buffer; the
 *     library never allocates device memory on these calls.
 *   - Device tensors: base address 16-byte aligned and ld * element size
 *     a multiple of 16 bytes (the tensor-memory-accelerator rule); the
 *     column counts D_in and D_out must be multiples of 8. BT may be any
 *     value >= 0 (BT = 0 is a step with a zero gradient).
 *   - Every call is enqueued on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and returns without synchronising. Argument
 *     and launch errors are returned as a forge_status; the message is
 *     available from forge_last_error() on the calling thread. No C++
 *     exception crosses this interface.
 *   - Device-side failures (a bounded wait inside a kernel that gave up)
 *     are recorded in a per-device status word and reported by
 *     forge_sync_status(). Kernels never trap and never wait unboundedly.
 *   - There is no CPU fallback: a variant without a GPU kernel returns
 *     FORGE_ERR_UNSUPPORTED.
 */
#ifndef FORGE_H_
#define FORGE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Compatible with cudaStream_t (a pointer to the runtime's opaque stream). */
struct CUstream_st;
typedef struct CUstream_st* forge_stream_t;

typedef enum {
  FORGE_OK = 0,
  FORGE_ERR_INVALID_ARG = 1, /* null pointer, bad shape, bad step, bad hyper-parameter */
  FORGE_ERR_UNSUPPORTED = 2, /* a dtype / option combination with no kernel */
  FORGE_ERR_ALIGNMENT = 3,   /* base address or row pitch breaks the 16-byte rule */
  FORGE_ERR_CUDA = 4,        /* a CUDA runtime or driver call failed */
  FORGE_ERR_TIMEOUT = 5      /* a kernel's bounded wait gave up (forge_sync_status) */
} forge_status;

typedef enum {
  FORGE_F32 = 0,
  FORGE_BF16 = 1,
  /* 8-bit block-quantised moment (section 2.3; Appendix B), one fp32 scale
   * s per 128 consecutive elements of a row (D_in must be a multiple of
   * 128). First moment: int8 codes, m = code * s, s = absmax(m) / 127.
   * Second moment: uint8 codes of sqrt(v), v = (code * s)^2,
   * s = absmax(sqrt(v)) / 255. Code 0 is reserved for an exactly zero
   * moment. `scale` points to fp32 scales laid out [D_in/128][D_out]
   * (contiguous; block column major), so one 128-row tile reads 512
   * contiguous bytes. */
  FORGE_I8B128 = 2
} forge_dtype;

typedef struct {
  void* data;        /* device pointer to element (0, 0) */
  int32_t dtype;     /* forge_dtype */
  int64_t rows;
  int64_t cols;
  int64_t ld;        /* elements between rows (codes for FORGE_I8B128) */
  void* scale;       /* FORGE_I8B128 only: fp32 scales [cols/128][rows]; else NULL */
} forge_tensor;

/* Flags (forge_hyper.flags). */
#define FORGE_FLAG_TILE_N_AUTO 0u   /* tile width chosen by the scheduler policy */
#define FORGE_FLAG_TILE_N_128 1u    /* force 128 x 128 gradient tiles */
#define FORGE_FLAG_TILE_N_64 2u     /* force 128 x 64 gradient tiles */
#define FORGE_FLAG_TILE_N_256 3u    /* force 128 x 256 gradient tiles (fp32 / bf16 state) */
/* force 256 x 256 gradient tiles shared by a cluster of two CTAs (one
 * 128-row half each; plain step, fp32 / bf16 state) */
#define FORGE_FLAG_TILE_PAIR_256 4u
#define FORGE_FLAG_TILE_N_MASK 7u
/* Test hook for the device-side failure path: the epilogue waits on a
 * barrier that nothing signals, with a ~1 ms bound, gives up, and the
 * step returns without touching W or its moments; forge_sync_status() then
 * reports FORGE_ERR_TIMEOUT. */
#define FORGE_FLAG_TEST_FORCE_TIMEOUT 0x100u
/* forge_backward_step (in forge_hyper.flags) and forge_backward_accumulate
 * (its flags argument) only: force the fused input gradient (an error if
 * this layer or workspace cannot take it), or force the two-kernel path. */
#define FORGE_FLAG_BACKWARD_FUSED 0x200u
#define FORGE_FLAG_BACKWARD_SPLIT 0x400u
/* forge_backward_step only, split path (either flag implies it): the tiles
 * of the input gradient dX = dY W_old -- 128 tokens each, or all the tokens
 * (2 or 4 blocks of 128, for 128 < BT <= 512; FORGE_ERR_UNSUPPORTED
 * otherwise). Without either, the library costs both and takes the
 * cheaper. dX differs between them only in the fp32 summation order. */
#define FORGE_FLAG_DGRAD_TOKENS_128 0x800u
#define FORGE_FLAG_DGRAD_ALL_TOKENS 0x1000u

/* Optimizer rule of forge_backward_step. */
typedef enum {
  FORGE_RULE_ADAMW = 0,
  FORGE_RULE_SGDM = 1,
  FORGE_RULE_LION = 2,
  FORGE_RULE_SGD = 3,
  FORGE_RULE_RMSPROP = 4,
  FORGE_RULE_ADAGRAD = 5,
  FORGE_RULE_NADAM = 6,
  FORGE_RULE_RADAM = 7
} forge_rule;

typedef struct {
  double lr;            /* eta */
  double beta1;         /* AdamW / Lion beta1; SGD-momentum: momentum mu */
  double beta2;         /* AdamW beta2; Lion: decay of the stored moment */
  double eps;           /* AdamW epsilon (added outside the square root) */
  double weight_decay;  /* lambda: decoupled for AdamW and Lion, L2 for SGD-momentum */
  int32_t sr_w;         /* bf16 W only: 1 = stochastic rounding, 0 = round-to-nearest-even */
  int32_t sr_moments;   /* bf16 moments only: 1 = stochastic rounding, 0 = RNE */
  uint32_t flags;       /* FORGE_FLAG_* */
  double momentum_decay; /* NAdam psi (PyTorch's default is 4e-3); unused by the other rules */
} forge_hyper;

/*
 * forge_wgrad_step_adamw -- fused G = dY^T X and AdamW step, in place.
 *
 * Computes, per element (p, q), with t = step (Algorithm 1, phase 2):
 *   m' = b1 m + (1 - b1) g
 *   v' = b2 v + (1 - b2) g^2
 *   W' = (1 - lr wd) W - lr (m' / (1 - b1^t)) / (sqrt(v' / (1 - b2^t)) + eps)
 * where g = G[p][q]. The arithmetic is fp32: the scalars 1 - b1, 1 - b2,
 * 1 - lr wd, lr / (1 - b1^t) and 1 / sqrt(1 - b2^t) are folded in double on
 * the host and rounded to float once; each element then evaluates
 *   m' = b1*m + (1-b1)*g;  v' = b2*v + (1-b2)*(g*g);
 *   d = sqrt(v')*(1/sqrt(1-b2^t)) + eps;  W' = (1-lr wd)*W - (lr/(1-b1^t))*(m'/d)
 * with every operation correctly rounded and no fused multiply-add.
 * The new moments used by the update are the unrounded fp32 values;
 * storage rounding applies to what is written.
 *
 * X, dY: both FORGE_BF16 (tensor-core path) or both FORGE_F32 (an fp32
 *   path for small problems). X is BT x D_in, dY is BT x D_out.
 * W: FORGE_F32 (master weights) or FORGE_BF16, D_out x D_in, updated in place.
 *   bf16 W is written with stochastic rounding when h->sr_w (Appendix C,
 *   Proposition 5): the 16-bit draw of element idx = p * D_in + q is half
 *   (idx % 2) of word (idx % 8) / 2 of Philox4x32-10 with key
 *   (seed lo, seed hi) and counter (idx / 8 lo, idx / 8 hi, step, site),
 *   site 0 for W, 1 for m, 2 for v.
 * m, v: both FORGE_F32, both FORGE_BF16 or both FORGE_I8B128, D_out x D_in,
 *   updated in place (scales too).
 * step: t >= 1 (FORGE_ERR_INVALID_ARG otherwise).
 * Precondition (Remark 1): W is overwritten, so the input gradient
 *   dX = dY W must already have been enqueued (forge_dgrad) on the same
 *   stream, and W must have no other gradient consumer in this step.
 * W, m and v must not overlap X, dY or each other.
 */
forge_status forge_wgrad_step_adamw(const forge_tensor* X, const forge_tensor* dY,
                                    forge_tensor* W, forge_tensor* m, forge_tensor* v,
                                    const forge_hyper* h, int64_t step, uint64_t seed,
                                    forge_stream_t stream);

/*
 * forge_wgrad_step_sgdm -- fused G = dY^T X and SGD with momentum, in place.
 *
 * The paper lists SGD-momentum among the fully fused element-wise rules
 * (Appendix N (i), item 8: "single moment") without printing it; this
 * library implements the common rule with coupled L2 decay, no dampening
 * and no Nesterov term, mu = h->beta1:
 *   g~ = g + wd*W;  m' = mu*m + g~;  W' = W - lr*m'     (fp32, no FMA).
 * Arguments as for forge_wgrad_step_adamw without v (m: F32, BF16 or
 * I8B128 with the first-moment code rule). h->beta2 and h->eps are unused.
 */
forge_status forge_wgrad_step_sgdm(const forge_tensor* X, const forge_tensor* dY,
                                   forge_tensor* W, forge_tensor* m,
                                   const forge_hyper* h, int64_t step, uint64_t seed,
                                   forge_stream_t stream);

/*
 * forge_wgrad_step_lion -- fused G = dY^T X and Lion, in place.
 *
 * Appendix N (i), item 4 ("sign-of-momentum update with a single moment
 * buffer"), following Chen et al. 2023, sign(0) = 0:
 *   c = b1*m + (1-b1)*g;  W' = (1-lr wd)*W - lr*sign(c);  m' = b2*m + (1-b2)*g.
 * Arguments as for forge_wgrad_step_sgdm; h->eps is unused.
 */
forge_status forge_wgrad_step_lion(const forge_tensor* X, const forge_tensor* dY,
                                   forge_tensor* W, forge_tensor* m,
                                   const forge_hyper* h, int64_t step, uint64_t seed,
                                   forge_stream_t stream);

/*
 * The remaining element-wise rules the paper fuses (Appendix N (i): SGD,
 * RMSprop, AdaGrad, NAdam, RAdam) are named there without formulas; each
 * follows the PyTorch optimizer of the same name with its defaults
 * (coupled L2 weight decay g~ = g + wd*W, no momentum / centring / lr decay
 * for RMSprop and AdaGrad, initial accumulator 0). Arguments as for
 * forge_wgrad_step_adamw; the state tensors are FORGE_F32 or FORGE_BF16
 * (no 8-bit variant). fp32 op sequences (correctly rounded, no FMA):
 *
 * forge_wgrad_step_sgd:      g~ = g + wd*W;  W' = W - lr*g~.  No state.
 * forge_wgrad_step_rmsprop:  v' = a*v + (1-a)*(g~*g~);  W' = W - lr*(g~/(sqrt(v') + eps)),
 *                            a = h->beta2 (PyTorch's alpha).
 * forge_wgrad_step_adagrad:  v' = v + g~*g~;  W' = W - lr*(g~/(sqrt(v') + eps)).
 * forge_wgrad_step_nadam:    m' = b1*m + (1-b1)*g~;  v' = b2*v + (1-b2)*(g~*g~);
 *                            d = sqrt(v')*(1/sqrt(1-b2^t)) + eps;
 *                            W' = W - (c1*g~ + c2*m')/d, with mu_i = b1 (1 - 0.5*0.96^(i psi)),
 *                            P_t = prod_{i<=t} mu_i, c1 = lr (1 - mu_t)/(1 - P_t),
 *                            c2 = lr mu_{t+1}/(1 - P_t mu_{t+1}), psi = h->momentum_decay.
 * forge_wgrad_step_radam:    m', v' as NAdam; rho_inf = 2/(1-b2) - 1,
 *                            rho_t = rho_inf - 2 t b2^t/(1-b2^t); if rho_t > 5:
 *                            r_t = sqrt((rho_t-4)(rho_t-2) rho_inf/((rho_inf-4)(rho_inf-2) rho_t)),
 *                            W' = W - (lr r_t sqrt(1-b2^t)/(1-b1^t))*(m'/(sqrt(v') + eps));
 *                            else W' = W - (lr/(1-b1^t))*m'.
 * The per-step scalars (c1, c2, r_t, ...) are computed in double on the host
 * and rounded to float once.
 */
forge_status forge_wgrad_step_sgd(const forge_tensor* X, const forge_tensor* dY, forge_tensor* W,
                                  const forge_hyper* h, int64_t step, uint64_t seed, forge_stream_t stream);
forge_status forge_wgrad_step_rmsprop(const forge_tensor* X, const forge_tensor* dY, forge_tensor* W,
                                      forge_tensor* v, const forge_hyper* h, int64_t step, uint64_t seed,
                                      forge_stream_t stream);
forge_status forge_wgrad_step_adagrad(const forge_tensor* X, const forge_tensor* dY, forge_tensor* W,
                                      forge_tensor* v, const forge_hyper* h, int64_t step, uint64_t seed,
                                      forge_stream_t stream);
forge_status forge_wgrad_step_nadam(const forge_tensor* X, const forge_tensor* dY, forge_tensor* W,
                                    forge_tensor* m, forge_tensor* v, const forge_hyper* h, int64_t step,
                                    uint64_t seed, forge_stream_t stream);
forge_status forge_wgrad_step_radam(const forge_tensor* X, const forge_tensor* dY, forge_tensor* W,
                                    forge_tensor* m, forge_tensor* v, const forge_hyper* h, int64_t step,
                                    uint64_t seed, forge_stream_t stream);

/*
 * forge_dgrad -- input gradient dX = dY W_old (Remark 1, Appendix A).
 *
 * Must be enqueued before the step that overwrites W, on the same stream,
 * so that it reads the pre-update weights. dY: FORGE_BF16, BT x D_out.
 * W_old: FORGE_BF16 or FORGE_F32 (fp32 master weights are rounded to bf16
 * as they are staged for the tensor cores), D_out x D_in. dX: FORGE_BF16
 * or FORGE_F32, BT x D_in (fp32 accumulation, one rounding at the store).
 */
forge_status forge_dgrad(const forge_tensor* dY, const forge_tensor* W_old, forge_tensor* dX,
                         forge_stream_t stream);

/*
 * forge_dgrad_ws -- the same product with a device workspace (16-byte
 * aligned, caller-owned, not shared by calls in flight; contents need not
 * be initialised): given forge_workspace_bytes(D_out, D_in, BT) bytes, a
 * layer with few dX tiles splits its contraction over D_out across the SMs
 * and a second kernel adds the parts in a fixed order (dX bit-reproducible;
 * it differs from forge_dgrad's only in the fp32 summation order). Less
 * workspace (or NULL) gives forge_dgrad's plan. This is the input gradient
 * of forge_backward_step's split path.
 */
forge_status forge_dgrad_ws(const forge_tensor* dY, const forge_tensor* W_old, forge_tensor* dX, void* workspace,
                            size_t workspace_bytes, forge_stream_t stream);

/*
 * forge_backward_step -- the whole backward pass of one linear layer with
 * its optimizer step: dX = dY W_old (Remark 1, Appendix A) and the fused
 * weight-gradient step of `rule` (Algorithm 1 for AdamW; Appendix N (i)
 * for the other element-wise rules).
 *
 * s0, s1: the rule's state, as the forge_wgrad_step_<rule> call takes it
 * (AdamW / NAdam / RAdam: m, v; SGD-momentum / Lion: m; RMSprop /
 * AdaGrad: v; SGD: none -- pass NULL for unused slots). dX: FORGE_BF16 or
 * FORGE_F32, BT x D_in.
 *
 * Two paths. The fused path reads each W tile once: the tile that is about
 * to be updated also feeds a second tensor-core product, dY_tile x
 * W_old_tile, whose fp32 partial sums accumulate in tensor memory per
 * column of tiles and are added up in a fixed order by a second kernel
 * (deterministic dX). It needs bf16 X / dY, fp32 or bf16 state,
 * 1 <= BT <= 768, and `workspace` of forge_workspace_bytes(D_out, D_in, BT)
 * bytes (device memory, 16-byte aligned, owned by the caller, contents
 * need not be initialised; it must not be shared by calls in flight at the
 * same time). The split path enqueues the input gradient (forge_dgrad's
 * kernel; given that workspace and few tiles, its contraction is split
 * over several SMs and a second kernel adds the partial sums in a fixed
 * order) and then the step. 8-bit state takes the split
 * path.
 * With no FORGE_FLAG_BACKWARD_* flag the library takes the fused path when
 * it applies, the workspace is large enough, and the layer is one where it
 * measured faster: fp32 W; bf16 W with two state tensors and D_in < D_out
 * (otherwise the split path); FORGE_FLAG_BACKWARD_FUSED /
 * FORGE_FLAG_BACKWARD_SPLIT force a path. The fused path uses 128 x 64
 * gradient tiles (a FORGE_FLAG_TILE_N_128 request selects the split path).
 * dX differs between the paths only in the fp32 summation order.
 */
forge_status forge_backward_step(forge_rule rule, const forge_tensor* X, const forge_tensor* dY, forge_tensor* W,
                                 forge_tensor* s0, forge_tensor* s1, forge_tensor* dX, const forge_hyper* h,
                                 int64_t step, uint64_t seed, void* workspace, size_t workspace_bytes,
                                 forge_stream_t stream);

/*
 * forge_wgrad_accumulate -- one micro-batch of exact gradient accumulation
 * (Appendix L): G_acc = G_acc + dY^T X, or G_acc = dY^T X when `overwrite`
 * is nonzero (the first micro-batch of a window). Each 128-row tile of
 * dY^T X is formed in tensor memory exactly as the fused step forms it and
 * added to G_acc in fp32 (one rounding per micro-batch).
 *
 * G_acc: FORGE_F32, D_out x D_in, caller-owned; it is the one
 * gradient-shaped buffer of this mode and lives for the accumulation
 * window. X, dY: FORGE_BF16. The micro-batch's input gradient is a
 * separate forge_dgrad (or forge_dgrad_ws) call, or use forge_backward_accumulate for both.
 */
forge_status forge_wgrad_accumulate(const forge_tensor* X, const forge_tensor* dY, forge_tensor* G_acc, int overwrite,
                                    forge_stream_t stream);

/*
 * forge_backward_accumulate -- the whole backward pass of a layer for one
 * micro-batch of an accumulation window other than its last (Appendix L):
 * dX = dY W (the weights are not updated inside the window, so dX always
 * reads the current W) and the accumulation of forge_wgrad_accumulate,
 * G_acc = [G_acc +] dY^T X (`overwrite` nonzero: the window's first
 * micro-batch). Where the layer allows it (bf16 X / dY, 1 <= BT <= 768)
 * both run in one pass: the 128 x 64 tile kernel of the fused backward
 * step, with G_acc in place of the state and the W tile read once, rounded
 * to bf16, as the B operand of the dX product; dX is summed from fp32
 * partials in a fixed order, as in forge_backward_step. Otherwise
 * forge_dgrad and forge_wgrad_accumulate run one after the other.
 *
 * W: FORGE_F32 or FORGE_BF16, D_out x D_in, read only. G_acc: FORGE_F32.
 * dX: BT x D_in, FORGE_BF16 or FORGE_F32. workspace / workspace_bytes: as
 * for forge_backward_step (forge_workspace_bytes(D_out, D_in, BT) bytes
 * enable the fused pass). flags: 0 (the library chooses: fused when it
 * applies and the workspace suffices), FORGE_FLAG_BACKWARD_FUSED or
 * FORGE_FLAG_BACKWARD_SPLIT; any other bit is FORGE_ERR_INVALID_ARG. G_acc
 * is identical on both paths up to the fp32 summation order inside a tile
 * (bit-identical when the tile sums are exact); so is dX.
 */
forge_status forge_backward_accumulate(const forge_tensor* X, const forge_tensor* dY, const forge_tensor* W,
                                       forge_tensor* G_acc, forge_tensor* dX, int overwrite, uint32_t flags,
                                       void* workspace, size_t workspace_bytes, forge_stream_t stream);

/*
 * forge_wgrad_step_accumulated -- the last micro-batch of the window: each
 * tile's gradient is G_acc + dY^T X (G_acc is read, not written) and the
 * fused step of `rule` fires once on it, so the result is the step of the
 * whole effective batch (Appendix L). X / dY may be empty (BT = 0): the step
 * then uses G_acc alone. s0, s1 as for forge_backward_step; fp32 or bf16
 * state (no 8-bit variant); bf16 X / dY.
 */
forge_status forge_wgrad_step_accumulated(forge_rule rule, const forge_tensor* X, const forge_tensor* dY,
                                          const forge_tensor* G_acc, forge_tensor* W, forge_tensor* s0,
                                          forge_tensor* s1, const forge_hyper* h, int64_t step, uint64_t seed,
                                          forge_stream_t stream);

/*
 * forge_backward_step_no_alloc -- forge_backward_step on the fused path,
 * for callers that cannot allocate device memory: code running under a
 * framework whose allocator owns the whole device, plug-ins that get
 * tensors but no allocator, or hosts that forbid allocation once training
 * has started. The paper has no counterpart of this entry point.
 *
 * Same arguments and results as forge_backward_step with
 * FORGE_FLAG_BACKWARD_FUSED, minus the workspace: the dX partial sums go
 * to a 64 MiB array compiled into the library (held on every GPU that
 * loads this part of the library, until the process exits). It calls no
 * allocator. A layer whose forge_workspace_bytes() exceeds 64 MiB is
 * rejected with FORGE_ERR_UNSUPPORTED before any work; every
 * Llama-3.1-8B projection fits at BT <= 512 on a 152-SM GPU. Layers the
 * fused path does not take (8-bit state, BT > 768) return
 * FORGE_ERR_UNSUPPORTED as well.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * With CUDA's lazy module loading that first call is also when the driver
 * loads this part of the library on the device and reserves the 64 MiB, so
 * it can fail (FORGE_ERR_CUDA) if the device is already full: make it at
 * start-up, before a framework allocator takes the device's memory. The
 * address is kept per device for the life of the process; after a
 * cudaDeviceReset it no longer points at the array, so do not call this
 * entry point again in a process that has reset the device.
 * All calls share the one array and it keeps what the last call left
 * there; nothing in it needs to start at zero, since every partial sum is
 * written before it is read. Calls whose kernels overlap on the GPU (on
 * different streams, or from different threads) race on the array: order
 * them on one stream.
 */
forge_status forge_backward_step_no_alloc(forge_rule rule, const forge_tensor* X, const forge_tensor* dY,
                                          forge_tensor* W, forge_tensor* s0, forge_tensor* s1, forge_tensor* dX,
                                          const forge_hyper* h, int64_t step, uint64_t seed,
                                          forge_stream_t stream);

/*
 * forge_sync_status -- synchronise `stream`, then read and clear the
 * device status word of the current device. Returns FORGE_ERR_TIMEOUT if
 * a kernel's bounded wait gave up since the last call (the message names
 * the wait), FORGE_ERR_CUDA if synchronisation failed, else FORGE_OK.
 */
forge_status forge_sync_status(forge_stream_t stream);

/* Message of the last failed call on this thread ("" if none). */
const char* forge_last_error(void);

/* Library version, e.g. "0.3.0". */
const char* forge_version(void);

/*
 * forge_workspace_bytes -- device scratch for a layer of this shape on the
 * current device, the larger of:
 *   - the fused paths of forge_backward_step and forge_backward_accumulate:
 *     one fp32 slab of ceil(BT/128)*128 x 64 dX partial sums per (CTA, tile
 *     column) pair (1 <= BT <= 768);
 *   - the split path's input gradient where its plan splits the
 *     contraction over D_out: one fp32 partial sum per part (S = min(4,
 *     SMs / tiles) parts run side by side), which a second kernel adds in a
 *     fixed order (dX stays bit-reproducible). Tiles of 128 tokens split in
 *     parts of at least 2048 rows where 128 x 128 tiles would leave at least
 *     half the SMs idle (128 x 256 tiles for bf16 W); tiles of all the
 *     tokens (128 < BT <= 512) in parts of at least 256 rows. The plan with
 *     the least shared-memory traffic per SM is taken.
 * 0 when neither applies or the device cannot be queried. Passing less only
 * forgoes these paths (forced fused paths then fail). The forge_wgrad_step_*
 * calls and forge_dgrad need no scratch: their schedulers keep their state on
 * chip and the gradient never leaves the tensor-memory accumulators.
 */
size_t forge_workspace_bytes(int64_t d_out, int64_t d_in, int64_t bt);

/*
 * forge_selftest_math -- test hook: enumerates cases of the branch-free
 * correctly rounded divide and square root the AdamW epilogues use with
 * bf16 / 8-bit moments, on the current device, and counts disagreements
 * with the hardware's correctly rounded operations. which = 0: the square
 * root of every float whose bit pattern is in [first, first + count)
 * (< 2^32); 1: the refined reciprocal of every such divisor in
 * [2^-60, 2^60]; 2: the quotient n / d over pairs of significands, case i
 * being n = 1 + floor(i / 2^23) 2^-23, d = 1 + (i mod 2^23) 2^-23
 * (i < 2^46). *mismatches receives the disagreements, *declined the cases
 * the fast path leaves to the guarded functions (outside its range).
 * Synchronous (waits for the device); FORGE_ERR_INVALID_ARG for a bad
 * `which`, range or null pointer, FORGE_ERR_CUDA if a CUDA call fails; sets
 * no forge_last_error message.
 */
forge_status forge_selftest_math(int which, uint64_t first, uint64_t count, uint64_t* mismatches,
                                 uint64_t* declined);

#ifdef __cplusplus
}
#endif

#endif /* FORGE_H_ */
