// forge_api.cu -- the C ABI declared in include/forge.h: argument
// validation, tensor-map encoding, the tile-scheduler / tile-shape policy,
// host folding of the per-step scalars, launch, and the device status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/forge.h"
#include "forge_params.h"

using namespace forge;

// Device status word (per device): 0, or the code of the first bounded wait
// that gave up since it was last read.
__device__ unsigned int forge_device_status[4];

namespace {

thread_local std::string g_last_error;

forge_status fail(forge_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

forge_status ok() {
  g_last_error.clear();
  return FORGE_OK;
}

}  // namespace

namespace forge {

// Records `msg` as the calling thread's forge_last_error() and returns `st`
// (for entry points defined in other translation units).
forge_status set_error(forge_status st, const char* msg) { return fail(st, "%s", msg); }

}  // namespace forge

namespace {

// ------------------------------------------------------------------ driver entry points

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

struct DeviceInfo {
  int sms = 0;
  unsigned int* status = nullptr;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

forge_status device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FORGE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(FORGE_ERR_CUDA, "device id %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (d.status == nullptr) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
      return fail(FORGE_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", dev,
                  major, minor);
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(FORGE_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, forge_device_status);
    if (e != cudaSuccess) return fail(FORGE_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    d.status = static_cast<unsigned int*>(p);
  }
  *out = &d;
  return FORGE_OK;
}

// ------------------------------------------------------------------ validation

const char* dtype_name(int dt) {
  switch (dt) {
    case FORGE_F32: return "f32";
    case FORGE_BF16: return "bf16";
    case FORGE_I8B128: return "i8b128";
    default: return "?";
  }
}

int elem_bytes(int dt) { return dt == FORGE_F32 ? 4 : dt == FORGE_BF16 ? 2 : 1; }

forge_status check_tensor(const forge_tensor* t, const char* name, int64_t rows, int64_t cols, bool needs_tma) {
  if (t == nullptr) return fail(FORGE_ERR_INVALID_ARG, "%s: null descriptor", name);
  if (t->dtype != FORGE_F32 && t->dtype != FORGE_BF16 && t->dtype != FORGE_I8B128)
    return fail(FORGE_ERR_INVALID_ARG, "%s: unknown dtype %d", name, t->dtype);
  if (t->rows != rows || t->cols != cols)
    return fail(FORGE_ERR_INVALID_ARG, "%s: shape %lld x %lld, expected %lld x %lld", name, (long long)t->rows,
                (long long)t->cols, (long long)rows, (long long)cols);
  if (t->ld < t->cols) return fail(FORGE_ERR_INVALID_ARG, "%s: ld %lld < cols %lld", name, (long long)t->ld,
                                   (long long)t->cols);
  if (rows > 0 && cols > 0 && t->data == nullptr) return fail(FORGE_ERR_INVALID_ARG, "%s: null data", name);
  if (t->dtype == FORGE_I8B128 && t->scale == nullptr && rows > 0 && cols > 0)
    return fail(FORGE_ERR_INVALID_ARG, "%s: 8-bit block state needs its scale array", name);
  if (needs_tma) {
    if (reinterpret_cast<uintptr_t>(t->data) % 16 != 0)
      return fail(FORGE_ERR_ALIGNMENT, "%s: base address not 16-byte aligned", name);
    if ((t->ld * elem_bytes(t->dtype)) % 16 != 0)
      return fail(FORGE_ERR_ALIGNMENT, "%s: row pitch %lld bytes is not a multiple of 16", name,
                  (long long)(t->ld * elem_bytes(t->dtype)));
  }
  if (t->dtype == FORGE_I8B128 && reinterpret_cast<uintptr_t>(t->scale) % 16 != 0)
    return fail(FORGE_ERR_ALIGNMENT, "%s: scale array not 16-byte aligned", name);
  return FORGE_OK;
}

bool finite(double x) { return std::isfinite(x); }

// ------------------------------------------------------------------ tensor maps

forge_status encode_2d(CUtensorMap* map, const forge_tensor* t, CUtensorMapDataType dt, int esize, uint32_t box_x,
                       uint32_t box_y, CUtensorMapSwizzle swz, const char* name) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return fail(FORGE_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(t->cols), static_cast<cuuint64_t>(t->rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(t->ld) * esize};
  const cuuint32_t box[2] = {box_x, box_y};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dt, 2, t->data, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FORGE_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed: %d", name, (int)r);
  return FORGE_OK;
}

// Chunk maps of the W / m / v tiles: `cw` columns (32, or 16 for the fp32
// fused-input-gradient kernel) x 128 rows, swizzle = row bytes.
forge_status encode_state(CUtensorMap* map, const forge_tensor* t, const char* name, int cw = 32) {
  CUtensorMapDataType dt;
  int es;
  if (t->dtype == FORGE_F32) { dt = CU_TENSOR_MAP_DATA_TYPE_FLOAT32; es = 4; }
  else if (t->dtype == FORGE_BF16) { dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16; es = 2; }
  else { dt = CU_TENSOR_MAP_DATA_TYPE_UINT8; es = 1; }
  const int row_bytes = cw * es;
  const CUtensorMapSwizzle swz = row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                   : CU_TENSOR_MAP_SWIZZLE_32B;
  return encode_2d(map, t, dt, es, static_cast<uint32_t>(cw), 128, swz, name);
}

// ------------------------------------------------------------------ scalars

// NAdam's momentum schedule mu_i = b1 (1 - 0.5 * 0.96^(i psi)) and its running
// product prod_{i<=t} mu_i. The product is extended from the last value this
// thread computed when the step advances (O(1) per step in a training loop).
double nadam_mu(double b1, double psi, double i) { return b1 * (1.0 - 0.5 * std::pow(0.96, i * psi)); }

double nadam_mu_product(double b1, double psi, int64_t t) {
  thread_local double c_b1 = -1.0, c_psi = -1.0, c_prod = 1.0;
  thread_local int64_t c_t = 0;
  if (c_b1 != b1 || c_psi != psi || t < c_t) { c_b1 = b1; c_psi = psi; c_t = 0; c_prod = 1.0; }
  for (int64_t i = c_t + 1; i <= t; ++i) c_prod *= nadam_mu(b1, psi, static_cast<double>(i));
  c_t = t;
  return c_prod;
}

StepScalars fold(int opt, const forge_hyper* h, int64_t t) {
  StepScalars s{};
  const double td = static_cast<double>(t);
  s.b1 = static_cast<float>(h->beta1);
  s.omb1 = static_cast<float>(1.0 - h->beta1);
  s.b2 = static_cast<float>(h->beta2);
  s.omb2 = static_cast<float>(1.0 - h->beta2);
  s.decay = static_cast<float>(1.0 - h->lr * h->weight_decay);
  s.eps = static_cast<float>(h->eps);
  s.wd = static_cast<float>(h->weight_decay);
  s.step_size = static_cast<float>(h->lr);
  s.inv_sqrt_bc2 = 1.0f;
  s.c2 = 0.0f;
  s.rect = 0;
  const double bc1 = 1.0 - std::pow(h->beta1, td), bc2 = 1.0 - std::pow(h->beta2, td);
  if (opt == OPT_ADAMW) {
    s.step_size = static_cast<float>(h->lr / bc1);
    s.inv_sqrt_bc2 = static_cast<float>(1.0 / std::sqrt(bc2));
  } else if (opt == OPT_NADAM) {
    const double mu_t = nadam_mu(h->beta1, h->momentum_decay, td);
    const double mu_n = nadam_mu(h->beta1, h->momentum_decay, td + 1.0);
    const double prod = nadam_mu_product(h->beta1, h->momentum_decay, t);
    s.step_size = static_cast<float>(h->lr * (1.0 - mu_t) / (1.0 - prod));
    s.c2 = static_cast<float>(h->lr * mu_n / (1.0 - prod * mu_n));
    s.inv_sqrt_bc2 = static_cast<float>(1.0 / std::sqrt(bc2));
  } else if (opt == OPT_RADAM) {
    const double rho_inf = 2.0 / (1.0 - h->beta2) - 1.0;
    const double rho_t = rho_inf - 2.0 * td * std::pow(h->beta2, td) / bc2;
    if (rho_t > 5.0) {
      const double r = std::sqrt((rho_t - 4.0) * (rho_t - 2.0) * rho_inf / ((rho_inf - 4.0) * (rho_inf - 2.0) * rho_t));
      s.rect = 1;
      s.step_size = static_cast<float>(h->lr * r * std::sqrt(bc2) / bc1);
    } else {
      s.step_size = static_cast<float>(h->lr / bc1);
    }
  }
  return s;
}

const char* opt_name(int opt) {
  switch (opt) {
    case OPT_ADAMW: return "adamw";
    case OPT_SGDM: return "sgdm";
    case OPT_LION: return "lion";
    case OPT_SGD: return "sgd";
    case OPT_RMSPROP: return "rmsprop";
    case OPT_ADAGRAD: return "adagrad";
    case OPT_NADAM: return "nadam";
    case OPT_RADAM: return "radam";
    case OPT_ACCUM: return "accumulate";
    default: return "accumulate(first)";
  }
}

int mkind(int dt) { return dt == FORGE_F32 ? M_F32 : dt == FORGE_BF16 ? M_BF16 : M_Q8; }

constexpr uint64_t kTimeoutNs = 4000000000ull;  // 4 s: far beyond any healthy wait
// X + dY up to 96 MB: the up-projection at BT 2048 (75 MB) gains too (fp32
// state step 391 -> 380 us); at BT 8192 (302 MB) the policy lost (762 -> 772).
constexpr int64_t kOperandHintBytes = int64_t(96) << 20;
constexpr size_t kDxL2SlabBytes = size_t(16) << 20;        // dX partial slabs kept in L2 up to 16 MB

// ------------------------------------------------------------------ fused input gradient: geometry

// The fused backward kernel uses 64-column tiles, walks them column by
// column in contiguous per-CTA ranges, and keeps a dX partial for up to six
// 128-token blocks in tensor memory beside its two gradient accumulators.
constexpr int kDxBN = 64;
constexpr int64_t kDxMaxTokens = 768;

struct DxGeometry {
  int tiles_m = 0, tiles_n = 0, num_tiles = 0, grid = 0, runs = 0, num_kb = 0;
  int64_t slab = 0;    // floats per partial slab
  size_t bytes = 0;    // workspace bytes
};

DxGeometry dx_geometry(int64_t d_out, int64_t d_in, int64_t bt, int sms) {
  DxGeometry g;
  if (bt < 1 || bt > kDxMaxTokens || d_out < 1 || d_in < 1 || sms < 1) return g;
  g.tiles_m = static_cast<int>((d_out + 127) / 128);
  g.tiles_n = static_cast<int>((d_in + kDxBN - 1) / kDxBN);
  g.num_tiles = g.tiles_m * g.tiles_n;
  g.grid = g.num_tiles < sms ? g.num_tiles : sms;
  // The fewest CTAs that keep the same most tiles per CTA, where that
  // leaves a tenth of the SMs or more idle: small layers then write fewer
  // dX slabs, which stay in L2 (k/v projection 1024 x 4096: 128 CTAs of 4
  // tiles, each half a tile column, 16 MB of slabs instead of 27.6 MB).
  {
    const int per = (g.num_tiles + g.grid - 1) / g.grid;
    const int fewest = (g.num_tiles + per - 1) / per;
    if (10 * fewest <= 9 * g.grid) g.grid = fewest;
  }
  const int64_t T = g.num_tiles, G = g.grid;
  for (int64_t c = 0; c < G; ++c) {
    const int64_t lo = c * T / G, hi = (c + 1) * T / G;
    if (hi <= lo) continue;
    const int r = static_cast<int>((hi - 1) / g.tiles_m - lo / g.tiles_m + 1);
    if (r > g.runs) g.runs = r;
  }
  g.num_kb = static_cast<int>((bt + 127) / 128);
  g.slab = static_cast<int64_t>(g.num_kb) * 128 * kDxBN;
  g.bytes = static_cast<size_t>(G) * g.runs * g.slab * sizeof(float);
  return g;
}

// The split contraction of the input gradient (dgrad with a workspace): a
// layer whose 128 x 128 tiles would leave at least half the SMs idle runs
// S = SMs / tiles parts of each tile's contraction on S CTAs (one wave),
// S <= 4, each part at least 32 stages long; the fix-up kernel adds the
// parts' fp32 sums in order. bf16 weights use 128 x 256 tiles there (twice
// the work per MMA instruction, which one thread issues). Measured (Lion,
// bf16 state, split path): up-projection BT 256 176.6 -> 159 us; where the
// tiles already fill half the GPU, or the contraction is short, the split
// lost (BT 512: q/o 72 -> 83 us, k/v 34 -> 46 us, up-projection even).
// How the input gradient is tiled, and whether its contraction over D_out
// is split over several CTAs (parts >= 2; needs `bytes` of workspace for
// the fp32 partial sums, which dgrad_fixup_kernel adds in a fixed order).
struct DgradPlan {
  int mb = 1;         // 128-token blocks per tile (2 / 4: all tokens of BT <= 256 / 512)
  int bn = 128;       // tile width (input features)
  int bk = 128;       // rows of D_out per stage
  int stg_rows = 64;  // fp32 W: rows per staging slot
  int tiles_m = 0, tiles_n = 0, num_tiles = 0, num_kb = 0;
  int parts = 0;
  size_t bytes = 0;
  double cost = 0.0;  // bytes through the busiest SM's shared memory (dgrad_cost)
};

// The kernel is bound by shared-memory bandwidth (about 128 bytes per
// clock per SM): the TMA writes of dY and W, the fp32-to-bf16 converters'
// reads and writes, and the tensor cores' operand reads. Per multiply-add,
// with tiles of MB blocks of 128 tokens x BN features:
//   dY written 2/BN + W written (and converted) (wb + 6 [fp32]) / (128 MB)
//   + operands read 2/N + 2/M bytes for M x N products (128 tokens x BN
//   features; all-token tiles: 128 features x 256 tokens).
// This model gives the measured times within 0.7-1.0 (128 x 128 tiles,
// fp32 weights: 29.4 MB through shared memory per CTA, 117 us). A plan's
// cost is waves x that per CTA (token blocks padded to 128), x 1.2 for
// all-token tiles (their two-stage rings and transposed drain: on the
// down-projection with bf16 weights they take 73 us where the model puts
// them 9 % below the 68 us of 128 x 256 tiles) and x 1.4 for four blocks
// with bf16 weights (up-projection, BT 512, split path: 141 against
// 135 us with 128-token tiles), plus, for a split, 740 KB for the fix-up
// launch (3 us).
double dgrad_cost(const DgradPlan& g, int64_t d_out, int wbytes, bool f32w, int sms) {
  const int parts = g.parts >= 2 ? g.parts : 1;
  const int64_t ctas = static_cast<int64_t>(g.num_tiles) * parts;
  const double waves = static_cast<double>((ctas + sms - 1) / sms);
  const double operands = g.mb > 1 ? 2.0 / 256.0 + 2.0 / 128.0 : 2.0 / g.bn + 2.0 / 128.0;
  const double per_mac = 2.0 / g.bn + (wbytes + (f32w ? 6.0 : 0.0)) / (128.0 * g.mb) + operands;
  const double macs = 128.0 * g.mb * g.bn * (static_cast<double>(d_out) / parts);
  double c = waves * macs * per_mac;
  if (g.mb > 1) c *= (g.mb == 4 && wbytes == 2) ? 1.4 : 1.2;
  if (g.parts >= 2) c += 740e3;
  return c;
}

// force: 0 the cheapest plan, 1 128-token tiles only, 2 all-token tiles only
// (an empty plan, num_tiles == 0, where they do not apply).
DgradPlan dgrad_plan(int64_t d_out, int64_t d_in, int64_t bt, bool w_bf16, int sms, bool may_split, int force = 0) {
  DgradPlan best;
  if (bt < 1 || d_out < 1 || d_in < 1 || sms < 1) return best;
  const int wbytes = w_bf16 ? 2 : 4;
  auto finish = [&](DgradPlan g) {
    g.tiles_n = static_cast<int>((d_in + g.bn - 1) / g.bn);
    g.num_tiles = g.tiles_m * g.tiles_n;
    g.num_kb = static_cast<int>((d_out + g.bk - 1) / g.bk);
    g.cost = dgrad_cost(g, d_out, wbytes, !w_bf16, sms);
    g.bytes = g.parts >= 2 ? static_cast<size_t>(g.num_tiles) * g.parts * 128 * g.mb * g.bn * sizeof(float) : 0;
    return g;
  };
  // 1. 128-token tiles, 128 x 256 for bf16 weights when those still fill
  //    the GPU (half the dY traffic per output of 128 x 128).
  {
    DgradPlan g;
    g.tiles_m = static_cast<int>((bt + 127) / 128);
    g.bn = (w_bf16 && g.tiles_m * ((d_in + 255) / 256) >= sms) ? 256 : 128;
    g.bk = g.bn == 128 ? 128 : 64;
    best = finish(g);
    if (force == 2) best = DgradPlan{};
  }
  // 2. The same tiles with the contraction split in S = min(4, SMs / tiles)
  //    parts of >= 2048 rows, where that puts >= 1.5x as many SMs to work
  //    as whole 128 x 128 tiles would (bf16 weights on 128 x 256 tiles).
  if (may_split && force != 2) {
    DgradPlan g;
    g.tiles_m = static_cast<int>((bt + 127) / 128);
    g.bn = w_bf16 ? 256 : 128;
    g.bk = g.bn == 128 ? 128 : 64;
    g = finish(g);
    const int64_t tiles128 = static_cast<int64_t>(g.tiles_m) * ((d_in + 127) / 128);
    int parts = sms / g.num_tiles;
    if (parts > 4) parts = 4;
    while (parts >= 2 && g.num_kb * (g.bk / 64) < 32 * parts) --parts;
    if (parts >= 2 && 2 * tiles128 <= sms && 2 * g.num_tiles * parts >= 3 * tiles128) {
      g.parts = parts;
      g = finish(g);
      if (g.cost < best.cost) best = g;
    }
  }
  // 3. All-token tiles on short token axes: 2 or 4 blocks of 128 tokens x
  //    128 columns (one weight read and conversion per tile instead of one
  //    per 128 tokens) in 64-row stages, the contraction split in
  //    S = min(4, SMs / tiles) parts of >= 256 rows where a workspace allows.
  if (bt > 128 && bt <= 512 && force != 1) {
    DgradPlan g;
    g.mb = bt <= 256 ? 2 : 4;
    g.tiles_m = 1;
    g.bn = 128;
    g.bk = 64;
    g.stg_rows = 32;
    g = finish(g);
    if (may_split) {
      int parts = sms / g.num_tiles;
      if (parts > 4) parts = 4;
      while (parts >= 2 && g.num_kb * g.bk < 256 * parts) --parts;
      if (parts >= 2) g.parts = parts;
      g = finish(g);
    }
    if (force == 2 || g.cost < best.cost) best = g;
  }
  return best;
}

// Extra arguments of the fused backward pass (dX and its workspace). W_dx:
// the weights dX is formed from when they are not the step's first tensor
// (the accumulation rules, whose first tensor is G_acc); null otherwise.
struct DxArgs {
  forge_tensor* dX;
  void* ws;
  size_t ws_bytes;
  const forge_tensor* W_dx;
};

// ------------------------------------------------------------------ the fused step

forge_status wgrad_step(int opt, const forge_tensor* X, const forge_tensor* dY, forge_tensor* W, forge_tensor* m,
                        forge_tensor* v, const forge_hyper* h, int64_t step, uint64_t seed, forge_stream_t stream,
                        const DxArgs* dx = nullptr, const forge_tensor* G_acc = nullptr) {
  const char* oname = opt_name(opt);
  const int nst = opt_nstate(opt);
  if (X == nullptr || dY == nullptr || W == nullptr || h == nullptr || (nst >= 1 && m == nullptr))
    return fail(FORGE_ERR_INVALID_ARG, "%s: null argument", oname);
  if (nst == 2 && v == nullptr) return fail(FORGE_ERR_INVALID_ARG, "%s: null v", oname);
  const bool two_betas = opt == OPT_ADAMW || opt == OPT_NADAM || opt == OPT_RADAM;
  if (two_betas && (h->beta1 >= 1.0 || h->beta2 >= 1.0 || h->beta1 < 0.0 || h->beta2 < 0.0))
    return fail(FORGE_ERR_INVALID_ARG, "%s: betas must lie in [0, 1)", oname);
  if (opt == OPT_RMSPROP && (h->beta2 >= 1.0 || h->beta2 < 0.0))
    return fail(FORGE_ERR_INVALID_ARG, "rmsprop: alpha (beta2) must lie in [0, 1)");
  if (opt == OPT_NADAM && !std::isfinite(h->momentum_decay))
    return fail(FORGE_ERR_INVALID_ARG, "nadam: non-finite momentum_decay");
  if (step < 1) return fail(FORGE_ERR_INVALID_ARG, "%s: step must be >= 1 (got %lld)", oname, (long long)step);
  if (step > 0xFFFFFFFFll) return fail(FORGE_ERR_INVALID_ARG, "%s: step exceeds 2^32 - 1", oname);
  if (!finite(h->lr) || !finite(h->beta1) || !finite(h->beta2) || !finite(h->eps) || !finite(h->weight_decay))
    return fail(FORGE_ERR_INVALID_ARG, "%s: non-finite hyper-parameter", oname);
  if (h->flags & ~(FORGE_FLAG_TILE_N_MASK | FORGE_FLAG_TEST_FORCE_TIMEOUT | FORGE_FLAG_BACKWARD_FUSED |
                   FORGE_FLAG_BACKWARD_SPLIT))
    return fail(FORGE_ERR_INVALID_ARG, "%s: unknown flags 0x%x", oname, h->flags);

  const int64_t bt = X->rows, d_in = X->cols, d_out = dY->cols;
  if (bt < 0 || d_in < 0 || d_out < 0) return fail(FORGE_ERR_INVALID_ARG, "%s: negative size", oname);
  if (X->dtype != dY->dtype || (X->dtype != FORGE_BF16 && X->dtype != FORGE_F32))
    return fail(FORGE_ERR_UNSUPPORTED, "%s: X and dY must both be bf16 or both f32 (got %s, %s)", oname,
                dtype_name(X->dtype), dtype_name(dY->dtype));
  const bool tc = X->dtype == FORGE_BF16;
  const bool accum = opt == OPT_ACCUM || opt == OPT_ACCSET;
  forge_status st;
  if ((accum || G_acc != nullptr) && !tc)
    return fail(FORGE_ERR_UNSUPPORTED, "%s: gradient accumulation runs on the tensor-core path (bf16 X, dY)", oname);
  if (accum && W != nullptr && W->dtype != FORGE_F32)
    return fail(FORGE_ERR_UNSUPPORTED, "%s: the gradient accumulator must be f32", oname);
  if (G_acc != nullptr) {
    if ((st = check_tensor(G_acc, "G_acc", d_out, d_in, true)) != FORGE_OK) return st;
    if (G_acc->dtype != FORGE_F32) return fail(FORGE_ERR_UNSUPPORTED, "%s: G_acc must be f32", oname);
    if (dx != nullptr) return fail(FORGE_ERR_UNSUPPORTED, "%s: no fused input gradient with G_acc", oname);
  }
  if ((st = check_tensor(X, "X", bt, d_in, true)) != FORGE_OK) return st;
  if ((st = check_tensor(dY, "dY", bt, d_out, true)) != FORGE_OK) return st;
  if ((st = check_tensor(W, "W", d_out, d_in, true)) != FORGE_OK) return st;
  if (nst >= 1 && (st = check_tensor(m, nst == 2 ? "m" : "state", d_out, d_in, true)) != FORGE_OK) return st;
  if (nst == 2 && (st = check_tensor(v, "v", d_out, d_in, true)) != FORGE_OK) return st;
  if (W->dtype == FORGE_I8B128) return fail(FORGE_ERR_UNSUPPORTED, "%s: W must be f32 or bf16", oname);
  if (nst == 2 && v->dtype != m->dtype)
    return fail(FORGE_ERR_UNSUPPORTED, "%s: m and v must share a dtype (got %s, %s)", oname, dtype_name(m->dtype),
                dtype_name(v->dtype));
  const int mdt = nst >= 1 ? m->dtype : FORGE_F32;
  if (mdt == FORGE_I8B128 && !(opt == OPT_ADAMW || opt == OPT_SGDM || opt == OPT_LION))
    return fail(FORGE_ERR_UNSUPPORTED, "%s: 8-bit block state exists for adamw, sgdm and lion", oname);
  if (d_in % 8 != 0 || d_out % 8 != 0)
    return fail(FORGE_ERR_UNSUPPORTED, "%s: D_in (%lld) and D_out (%lld) must be multiples of 8", oname,
                (long long)d_in, (long long)d_out);
  if (mdt == FORGE_I8B128 && d_in % 128 != 0)
    return fail(FORGE_ERR_UNSUPPORTED, "%s: 8-bit block moments need D_in %% 128 == 0 (got %lld)", oname,
                (long long)d_in);
  if (h->sr_w && W->dtype != FORGE_BF16)
    return fail(FORGE_ERR_INVALID_ARG, "%s: sr_w requires bf16 W", oname);
  if (h->sr_moments && mdt != FORGE_BF16)
    return fail(FORGE_ERR_INVALID_ARG, "%s: sr_moments requires bf16 moments", oname);
  if (bt > 0x7FFFFFFF || d_in > 0x7FFFFFFF || d_out > 0x7FFFFFFF)
    return fail(FORGE_ERR_INVALID_ARG, "%s: dimension exceeds 2^31 - 1", oname);
  if (d_in == 0 || d_out == 0) return ok();

  const forge_tensor* w_dx = (dx != nullptr && dx->W_dx != nullptr) ? dx->W_dx : W;
  if (w_dx != W) {
    if ((st = check_tensor(w_dx, "W", d_out, d_in, true)) != FORGE_OK) return st;
    if (w_dx->dtype != FORGE_F32 && w_dx->dtype != FORGE_BF16)
      return fail(FORGE_ERR_UNSUPPORTED, "%s: W must be f32 or bf16", oname);
  }

  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != FORGE_OK) return st;
  const StepScalars sc = fold(opt, h, step);
  // With the fused input gradient of an accumulation rule, the kernel's
  // weight kind is that of the weights read for dX (the slot holds G_acc).
  const int wk = w_dx->dtype == FORGE_F32 ? W_F32 : W_BF16;
  const int mk = mkind(mdt);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  if (!tc) {
    if (h->flags & FORGE_FLAG_TEST_FORCE_TIMEOUT)
      return fail(FORGE_ERR_UNSUPPORTED, "%s: the timeout test hook exists on the tensor-core path only", oname);
    WgradSimtParams p{};
    p.X = static_cast<const float*>(X->data);
    p.dY = static_cast<const float*>(dY->data);
    p.W = W->data;
    p.m = nst >= 1 ? m->data : nullptr;
    p.v = nst == 2 ? v->data : nullptr;
    p.m_scale = nst >= 1 ? static_cast<float*>(m->scale) : nullptr;
    p.v_scale = nst == 2 ? static_cast<float*>(v->scale) : nullptr;
    p.ld_x = X->ld; p.ld_dy = dY->ld; p.ld_w = W->ld; p.ld_m = nst >= 1 ? m->ld : 0; p.ld_v = nst == 2 ? v->ld : 0;
    p.d_out = static_cast<int>(d_out); p.d_in = static_cast<int>(d_in); p.bt = static_cast<int>(bt);
    p.sc = sc;
    p.step = static_cast<uint32_t>(step);
    p.seed_lo = static_cast<uint32_t>(seed); p.seed_hi = static_cast<uint32_t>(seed >> 32);
    p.sr_w = h->sr_w ? 1 : 0; p.sr_m = h->sr_moments ? 1 : 0;
    cudaError_t e = launch_wgrad_simt(p, opt, wk, mk, s);
    if (e != cudaSuccess) return fail(FORGE_ERR_CUDA, "%s (fp32 path) launch: %s", oname, cudaGetErrorString(e));
    return ok();
  }

  // ---- tensor-core path: tile-shape / scheduler policy
  const int tiles_m = static_cast<int>((d_out + 127) / 128);
  // W and state bytes per parameter (read once; written once).
  const int state_bytes = (wk == W_F32 ? 4 : 2) + nst * (mk == M_F32 ? 4 : mk == M_BF16 ? 2 : 1);
  int bn = 128;
  bool pair = false;  // CTA pairs on 256 x 256 tiles
  const uint32_t force = h->flags & FORGE_FLAG_TILE_N_MASK;
  if (dx != nullptr) bn = kDxBN;  // the fused input gradient fixes the tile width
  else if (force == FORGE_FLAG_TILE_N_64) bn = 64;
  else if (force == FORGE_FLAG_TILE_N_128) bn = 128;
  else if (force == FORGE_FLAG_TILE_N_256) bn = 256;
  else if (force == FORGE_FLAG_TILE_PAIR_256) { bn = 256; pair = true; }
  else if (force != FORGE_FLAG_TILE_N_AUTO) return fail(FORGE_ERR_INVALID_ARG, "%s: bad tile flag", oname);
  else if (mk != M_Q8 && tiles_m * ((d_in + 127) / 128) < dev->sms) bn = 64;  // too few tiles for one wave
  else if (mk != M_Q8 && !accum && G_acc == nullptr && tiles_m * ((d_in + 255) / 256) >= dev->sms &&
           (bt >= 1024 || (bt >= 512 && state_bytes <= 4)))
    // Long token axes (the GEMM dominates) and, from 512 tokens, light state
    // (<= 4 bytes per parameter): wider tiles cut the operand pipeline's
    // share (up-projection, BT 512, step alone: SGD bf16 W 108 -> 75 us,
    // SGD fp32 W 129 -> 92, Lion bf16 129 -> 110, SGD-momentum bf16
    // 117 -> 104.5; Lion fp32 188 -> 202, AdamW fp32 238 -> 267, AdamW
    // bf16 173 either way; BT 256: 128 columns everywhere).
    bn = 256;
  // From 2048 tokens the 256-column tiles are shared by CTA pairs (256 x 256
  // tiles; per CTA a third fewer operand bytes per stage for the same MMA
  // work, and a deeper operand ring). Up-projection, step alone, single CTA
  // / pair: AdamW bf16 state BT 2048 250 / 225.5 us, 4096 426 / 358, 8192
  // 775 / 624; fp32 state 314 / 293 (four pair stages), 487 / 404, 827 /
  // 660; Lion bf16 BT 2048 227 / 207.5, fp32 258 / 220. Below 2048 tokens
  // the pair lost (BT 1024 AdamW bf16 180 / 188.6 at best; light state at
  // BT 512: Lion bf16 110.5 / 128.5).
  if (force == FORGE_FLAG_TILE_N_AUTO && dx == nullptr && bn == 256 && bt >= 2048) pair = true;
  if (mk == M_Q8 && bn != 128)
    return fail(FORGE_ERR_UNSUPPORTED, "%s: 8-bit block moments need 128-column tiles", oname);
  if (bn == 256 && (accum || G_acc != nullptr))
    return fail(FORGE_ERR_UNSUPPORTED, "%s: 256-column tiles exist for the plain step only", oname);
  if (pair && mk == M_Q8)
    return fail(FORGE_ERR_UNSUPPORTED, "%s: CTA-pair tiles need fp32 or bf16 state", oname);
  if (mk == M_Q8 && G_acc != nullptr)
    return fail(FORGE_ERR_UNSUPPORTED, "%s: the accumulated-gradient step has no 8-bit state variant", oname);
  // Deep operand ring for long token axes, and for the accumulation rules at
  // any length: their slots hold only the fp32 accumulator, so shared memory
  // has room for four operand stages, and their tile time is the mainloop's.
  // Measured on the up-projection (step alone): bf16 W + bf16 moments at
  // BT 512 181 -> 178 us, BT 768 211 -> 180 us; 8-bit moments at BT 512
  // 227.5 -> 220 us; fp32 state at BT 768 277 -> 268 us but at BT 512
  // 240 -> 262 us (its state ring loses slots).
  // The stateless rule (SGD) takes it from 256 tokens (BT 256: bf16 W
  // 69 -> 60 us, fp32 W 86.5 -> 84 us).
  const bool deep128 = dx == nullptr && G_acc == nullptr && bn == 128 &&
                       (bt >= 768 || accum || (bt >= 256 && nst == 0) ||
                        (bt >= 512 && ((wk == W_BF16 && mk == M_BF16) || mk == M_Q8)));
  // 256-column tiles always use the deep ring; the fused input gradient takes
  // a third operand stage past 512 tokens (its mainloop then sets the pace).
  // The fused input gradient takes a third operand stage past 512 tokens, and
  // with the accumulation rules at any length (their state is one fp32 tensor).
  // The fused pass with bf16 weights takes its third operand stage from 512
  // tokens (up-projection, bf16 state: 230 -> 226.5 us); with fp32 weights
  // the state ring would lose its slots (270 -> 336 us).
  const int deep = (deep128 || bn == 256 ||
                    (dx != nullptr && (bt > 512 || accum || (bt == 512 && wk == W_BF16)))) ? 1 : 0;
  const int tiles_n = static_cast<int>((d_in + bn - 1) / bn);
  const uint32_t box_tokens = dx != nullptr ? 128u : 64u;  // tokens per operand stage

  WgradTcParams p;
  std::memset(&p, 0, sizeof(p));
  if (bt > 0) {  // with BT = 0 the kernel issues no operand loads and needs no operand maps
    if ((st = encode_2d(&p.tm_dy, dY, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, box_tokens,
                        CU_TENSOR_MAP_SWIZZLE_128B, "dY")) != FORGE_OK)
      return st;
    if ((st = encode_2d(&p.tm_x, X, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, box_tokens, CU_TENSOR_MAP_SWIZZLE_128B,
                        "X")) != FORGE_OK)
      return st;
  }
  // State chunk width: 16 columns for the fused input gradient with fp32 W
  // and two fp32 moments (four 24 KB state slots instead of two 48 KB
  // ones): up-projection at BT 256 282 -> 259 us, at BT 512 283.7 -> 269.3 us
  // (with the evict-last operand loads; before them the extra chunk turns
  // cost more than the deeper ring gained at BT 512), and past 512 tokens
  // the narrow slots leave room for a third operand stage (398 -> 351 us at
  // BT 768). One-state rules (fp32 W + fp32 m) take them from 512 tokens:
  // Lion up-projection 225.3 -> 220.6 us, SGD-momentum unchanged, both a
  // little slower at 256.
  // On the plain step's 128 x 256 tiles the narrow slots make room for a
  // third operand stage beside three (two moments) or four (one) slots,
  // where 32-column slots left two stages and two slots (up-projection, step
  // alone: AdamW BT 2048 381 -> 314 us, BT 8192 1123 -> 824 us; Lion BT
  // 8192 779 -> 771 us); on deep 128 x 128 tiles (768 tokens) a fourth
  // operand stage (AdamW 268.8 -> 256 us, Lion 203 -> 164, SGD-momentum
  // 197 -> 163).
  const bool narrow = wk == W_F32 && mk == M_F32 && nst >= 1 &&
                      ((dx != nullptr && (nst == 2 || bt >= 512)) ||
                       (dx == nullptr && G_acc == nullptr && !accum && (bn == 256 || deep128)));
  // 64-column chunks for the plain step with bf16 W and bf16 moments on
  // 128-column tiles below 768 tokens: half as many slot hand-overs for the
  // same bytes in flight (up-projection, AdamW: BT 256 176.4 -> 168.2 us,
  // BT 512 178.0 -> 175.5 us). From 768 tokens the 48 KB slots cost the ring
  // its fourth operand stage (181 -> 184 us), and on 256-column tiles its
  // third (BT 2048: 253 -> 319 us).
  const bool wide = dx == nullptr && G_acc == nullptr && !accum && wk == W_BF16 && mk == M_BF16 && nst >= 1 &&
                    bn == 128 && bt < 768;
  const int cw = narrow ? 16 : (wide ? 64 : 32);
  if ((st = encode_state(&p.tm_w, W, "W", cw)) != FORGE_OK) return st;
  if (nst >= 1) {
    if ((st = encode_state(&p.tm_m, m, "m", cw)) != FORGE_OK) return st;
  } else {
    p.tm_m = p.tm_w;  // unused
  }
  if (nst == 2) {
    if ((st = encode_state(&p.tm_v, v, "v", cw)) != FORGE_OK) return st;
  } else {
    p.tm_v = p.tm_m;  // unused
  }
  if (G_acc != nullptr) {
    if ((st = encode_state(&p.tm_g, G_acc, "G_acc")) != FORGE_OK) return st;
  } else {
    p.tm_g = p.tm_w;  // unused
  }
  p.sc = sc;
  p.m_scale = nst >= 1 ? static_cast<float*>(m->scale) : nullptr;
  p.v_scale = nst == 2 ? static_cast<float*>(v->scale) : nullptr;
  p.status = dev->status;
  p.d_out = static_cast<int>(d_out);
  p.d_in = static_cast<int>(d_in);
  p.bt = static_cast<int>(bt);
  // CTA pairs walk 256-row tiles (each CTA steps one 128-row half).
  p.tiles_m = pair ? static_cast<int>((d_out + 255) / 256) : tiles_m;
  p.tiles_n = tiles_n;
  p.num_tiles = p.tiles_m * tiles_n;
  p.num_kb = static_cast<int>((bt + box_tokens - 1) / box_tokens);
  // Grouped raster: tile rows per group. With 128 x 256 tiles (long token
  // axes, operands far larger than L2) 16 rows keep fewer X column blocks
  // live per window of in-flight tiles (BT 8192 up-projection: 791 -> 775 us
  // with bf16 state); 8 elsewhere.
  p.group_m = pair ? 8 : (bn == 256 ? 16 : 8);   // 2048 rows either way on 256-column tiles
  p.step = static_cast<uint32_t>(step);
  p.seed_lo = static_cast<uint32_t>(seed);
  p.seed_hi = static_cast<uint32_t>(seed >> 32);
  p.sr_w = h->sr_w ? 1 : 0;
  p.sr_m = h->sr_moments ? 1 : 0;
  p.flags = h->flags;
  p.timeout_ns = kTimeoutNs;
  // Operands that fit in L2 are loaded evict-last: every tile of
  // a row (column) of tiles re-reads the same dY (X) slabs while the state
  // streams through L2 once and would otherwise push them out (up-projection
  // BT 512: fused backward 68 MB fewer DRAM reads, 290 -> 283 us; split step
  // 262 -> 239 us). Not for the fused pass with bf16 weights, where it
  // measured 235 -> 239 us.
  const int64_t op_bytes = 2 * bt * (d_in + d_out);
  if (bt > 0 && op_bytes <= kOperandHintBytes && !(dx != nullptr && wk == W_BF16)) {
    p.op_hint = 1;
    const forge_tensor* ops[2] = {X, dY};
    for (int i = 0; i < 2; ++i) {
      const uintptr_t a = reinterpret_cast<uintptr_t>(ops[i]->data);
      const uintptr_t e = a + static_cast<uintptr_t>((ops[i]->rows - 1) * ops[i]->ld + ops[i]->cols) * 2u;
      p.op_lo[i] = reinterpret_cast<const uint8_t*>((a + 127u) & ~uintptr_t(127));   // whole lines only
      p.op_hi[i] = reinterpret_cast<const uint8_t*>(e & ~uintptr_t(127));
      if (p.op_hi[i] < p.op_lo[i]) p.op_hi[i] = p.op_lo[i];
    }
  }

  TcLaunch l{};
  l.opt = opt; l.wk = wk; l.mk = mk; l.bn = bn; l.deep = deep; l.dx = dx != nullptr ? 1 : 0;
  l.ga = G_acc != nullptr ? 1 : 0;
  l.narrow = narrow ? 1 : 0;
  l.wide = wide ? 1 : 0;
  // The pair's operand stages: 5 beside two state slots, or 4 beside three
  // for fp32 W with two fp32 moments below 4096 tokens (BT 2048: 333 us with
  // five stages, 293 with four; from 4096 five win: 404 / 431 us).
  l.pair = !pair ? 0 : ((wk == W_F32 && mk == M_F32 && nst == 2 && bt < 4096) ? 4 : 5);
  l.grid = pair ? 2 * (p.num_tiles < dev->sms / 2 ? p.num_tiles : dev->sms / 2)
                : (p.num_tiles < dev->sms ? p.num_tiles : dev->sms);
  l.stream = s;
  DxGeometry g;
  if (dx != nullptr) {
    g = dx_geometry(d_out, d_in, bt, dev->sms);
    l.grid = g.grid;
    if (g.num_tiles != p.num_tiles || g.num_kb != p.num_kb)
      return fail(FORGE_ERR_INVALID_ARG, "%s: internal geometry mismatch", oname);
    if (dx->ws == nullptr || dx->ws_bytes < g.bytes)
      return fail(FORGE_ERR_INVALID_ARG, "%s: fused backward needs %zu workspace bytes (got %zu)", oname, g.bytes,
                  dx->ws_bytes);
    if (reinterpret_cast<uintptr_t>(dx->ws) % 16 != 0)
      return fail(FORGE_ERR_ALIGNMENT, "%s: workspace not 16-byte aligned", oname);
    p.w_ptr = w_dx->data;
    p.ld_w = w_dx->ld;
    p.dx_ws = static_cast<float*>(dx->ws);
    p.dx_runs = g.runs;
    p.dx_slab = g.slab;
    // Small slab sets stay in L2 until the reduction reads and drops them
    // (whole lines only: a 128-byte aligned workspace).
    p.dx_l2 = (g.bytes <= kDxL2SlabBytes && reinterpret_cast<uintptr_t>(dx->ws) % 128 == 0) ? 1 : 0;
  }
  cudaError_t e;
  switch (opt) {
    case OPT_ADAMW: e = launch_wgrad_tc_adamw(p, l); break;
    case OPT_SGDM: e = launch_wgrad_tc_sgdm(p, l); break;
    case OPT_LION: e = launch_wgrad_tc_lion(p, l); break;
    case OPT_SGD: e = launch_wgrad_tc_sgd(p, l); break;
    case OPT_RMSPROP: e = launch_wgrad_tc_rmsprop(p, l); break;
    case OPT_ADAGRAD: e = launch_wgrad_tc_adagrad(p, l); break;
    case OPT_NADAM: e = launch_wgrad_tc_nadam(p, l); break;
    case OPT_RADAM: e = launch_wgrad_tc_radam(p, l); break;
    default: e = launch_wgrad_tc_accum(p, l); break;
  }
  if (e != cudaSuccess) return fail(FORGE_ERR_CUDA, "%s launch: %s", oname, cudaGetErrorString(e));
  if (dx != nullptr) {
    DxReduceParams r{};
    r.ws = static_cast<const float*>(dx->ws);
    r.dX = dx->dX->data;
    r.ld_dx = dx->dX->ld;
    r.dx_bf16 = dx->dX->dtype == FORGE_BF16 ? 1 : 0;
    r.bt = static_cast<int>(bt);
    r.d_in = static_cast<int>(d_in);
    r.tiles_m = g.tiles_m;
    r.num_tiles = g.num_tiles;
    r.grid = g.grid;
    r.runs = g.runs;
    r.slab = g.slab;
    r.discard = p.dx_l2;
    e = launch_dx_reduce(r, dev->sms, s);
    if (e != cudaSuccess) return fail(FORGE_ERR_CUDA, "%s: dX reduction launch: %s", oname, cudaGetErrorString(e));
  }
  return ok();
}

// Whether the fused backward pass beats dgrad + step for this layer: it
// saves the split path's dgrad (its read of W, its launches) and costs
// writing and re-reading one fp32 dX partial slab per (CTA, column) pair,
// with 64-column instead of 128-column step tiles. Measured at BT 512 on the
// Llama-3.1-8B projections (forge_backward_step fused / split, us):
//   fp32 W, fp32 state: fused everywhere -- up 269 / 318 (AdamW),
//     220 / 271 (Lion); down 290 / 322; q/o 102 / 118; k/v 50 / 58.
//   bf16 W, two bf16 moments: fused where D_in < D_out -- up 227 / 246;
//     split where it is as wide or wider -- q/o 88.7 / 79.7 (with the
//     branch-free divide in the split step), down 247 / 238, k/v 44 / 38.
//   bf16 W, one or no state tensor: split -- the step is bound by its
//     per-element arithmetic (stochastic rounding of W) and the fused
//     pass's slabs and narrower tiles do not pay: down Lion 226 / 197,
//     k/v 42 / 33, up 206 / 203, q/o 82 / 84 (within 2 %).
bool dx_worthwhile(const DxGeometry&, int64_t d_out, int64_t d_in, int w_bytes, int nst) {
  if (w_bytes == 4) return true;
  if (nst < 2) return false;
  return d_in < d_out;
}

forge_status dgrad_impl(const forge_tensor* dY, const forge_tensor* W_old, forge_tensor* dX, forge_stream_t stream,
                        void* ws = nullptr, size_t ws_bytes = 0, uint32_t flags = 0);

// forge_backward_step's own flags, taken off before the step.
constexpr uint32_t kBackwardOnlyFlags =
    FORGE_FLAG_BACKWARD_FUSED | FORGE_FLAG_BACKWARD_SPLIT | FORGE_FLAG_DGRAD_TOKENS_128 | FORGE_FLAG_DGRAD_ALL_TOKENS;

forge_status backward_step(int opt, const forge_tensor* X, const forge_tensor* dY, forge_tensor* W, forge_tensor* s0,
                           forge_tensor* s1, forge_tensor* dX, const forge_hyper* h, int64_t step, uint64_t seed,
                           void* ws, size_t ws_bytes, forge_stream_t stream) {
  const char* oname = opt_name(opt);
  if (X == nullptr || dY == nullptr || W == nullptr || dX == nullptr || h == nullptr)
    return fail(FORGE_ERR_INVALID_ARG, "backward_step(%s): null argument", oname);
  const bool want_fused = (h->flags & FORGE_FLAG_BACKWARD_FUSED) != 0;
  const bool dgrad_tiles = (h->flags & (FORGE_FLAG_DGRAD_TOKENS_128 | FORGE_FLAG_DGRAD_ALL_TOKENS)) != 0;
  const bool want_split = (h->flags & FORGE_FLAG_BACKWARD_SPLIT) != 0 || dgrad_tiles;
  if (want_fused && (h->flags & FORGE_FLAG_BACKWARD_SPLIT))
    return fail(FORGE_ERR_INVALID_ARG, "backward_step(%s): both BACKWARD_FUSED and BACKWARD_SPLIT set", oname);
  if (want_fused && dgrad_tiles)
    return fail(FORGE_ERR_INVALID_ARG, "backward_step(%s): DGRAD_* tile flags apply to the split path only", oname);
  if ((h->flags & FORGE_FLAG_DGRAD_TOKENS_128) && (h->flags & FORGE_FLAG_DGRAD_ALL_TOKENS))
    return fail(FORGE_ERR_INVALID_ARG, "backward_step(%s): both DGRAD_TOKENS_128 and DGRAD_ALL_TOKENS set", oname);
  const int64_t bt = X->rows, d_in = X->cols, d_out = dY->cols;
  if (dX->dtype != FORGE_BF16 && dX->dtype != FORGE_F32)
    return fail(FORGE_ERR_UNSUPPORTED, "backward_step(%s): dX must be bf16 or f32", oname);
  forge_status st;
  if ((st = check_tensor(dX, "dX", bt, d_in, true)) != FORGE_OK) return st;
  const int nst = opt_nstate(opt);
  const bool q8 = nst >= 1 && s0 != nullptr && s0->dtype == FORGE_I8B128;
  const uint32_t tile = h->flags & FORGE_FLAG_TILE_N_MASK;
  const bool possible = X->dtype == FORGE_BF16 && !q8 && bt >= 1 && bt <= kDxMaxTokens && d_in > 0 && d_out > 0 &&
                        (tile == FORGE_FLAG_TILE_N_AUTO || tile == FORGE_FLAG_TILE_N_64);
  bool fused = false;
  if (possible && !want_split) {
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev)) != FORGE_OK) return st;
    const DxGeometry g = dx_geometry(d_out, d_in, bt, dev->sms);
    fused = want_fused || (ws != nullptr && ws_bytes >= g.bytes &&
                           dx_worthwhile(g, d_out, d_in, W->dtype == FORGE_F32 ? 4 : 2, nst));
  }
  if (want_fused && !fused)
    return fail(FORGE_ERR_UNSUPPORTED,
                "backward_step(%s): the fused input gradient needs bf16 X/dY, fp32 or bf16 state, 1 <= BT <= %lld "
                "and 64-column tiles",
                oname, (long long)kDxMaxTokens);
  if (fused) {
    const DxArgs a{dX, ws, ws_bytes, nullptr};
    return wgrad_step(opt, X, dY, W, s0, s1, h, step, seed, stream, &a);
  }
  // Split path: dX from the weights before the step, then the step.
  if (X->dtype != FORGE_BF16)
    return fail(FORGE_ERR_UNSUPPORTED, "backward_step(%s): dX needs bf16 dY (the fp32-input step has no dgrad)",
                oname);
  if ((st = dgrad_impl(dY, W, dX, stream, ws, ws_bytes, h->flags)) != FORGE_OK) return st;
  forge_hyper h2 = *h;
  h2.flags &= ~kBackwardOnlyFlags;
  return wgrad_step(opt, X, dY, W, s0, s1, &h2, step, seed, stream);
}

// One micro-batch of an accumulation window that is not its last: dX from
// the (unchanged) weights and G_acc (+)= dY^T X, fused into one pass when
// the layer allows it, else dgrad and the accumulation kernel.
forge_status backward_accumulate(const forge_tensor* X, const forge_tensor* dY, const forge_tensor* W,
                                 forge_tensor* G_acc, forge_tensor* dX, int overwrite, uint32_t flags, void* ws,
                                 size_t ws_bytes, forge_stream_t stream) {
  if (X == nullptr || dY == nullptr || W == nullptr || G_acc == nullptr || dX == nullptr)
    return fail(FORGE_ERR_INVALID_ARG, "backward_accumulate: null argument");
  if (flags & ~(FORGE_FLAG_BACKWARD_FUSED | FORGE_FLAG_BACKWARD_SPLIT))
    return fail(FORGE_ERR_INVALID_ARG, "backward_accumulate: unknown flags 0x%x", flags);
  const bool want_fused = (flags & FORGE_FLAG_BACKWARD_FUSED) != 0;
  const bool want_split = (flags & FORGE_FLAG_BACKWARD_SPLIT) != 0;
  if (want_fused && want_split)
    return fail(FORGE_ERR_INVALID_ARG, "backward_accumulate: both BACKWARD_FUSED and BACKWARD_SPLIT set");
  const int64_t bt = X->rows, d_in = X->cols, d_out = dY->cols;
  if (dX->dtype != FORGE_BF16 && dX->dtype != FORGE_F32)
    return fail(FORGE_ERR_UNSUPPORTED, "backward_accumulate: dX must be bf16 or f32");
  forge_status st;
  if ((st = check_tensor(dX, "dX", bt, d_in, true)) != FORGE_OK) return st;
  if ((st = check_tensor(W, "W", d_out, d_in, true)) != FORGE_OK) return st;
  if (W->dtype != FORGE_F32 && W->dtype != FORGE_BF16)
    return fail(FORGE_ERR_UNSUPPORTED, "backward_accumulate: W must be f32 or bf16");
  const int opt = overwrite ? OPT_ACCSET : OPT_ACCUM;
  forge_hyper h;
  std::memset(&h, 0, sizeof(h));
  bool fused = false;
  if (X->dtype == FORGE_BF16 && bt >= 1 && bt <= kDxMaxTokens && d_in > 0 && d_out > 0 && !want_split) {
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev)) != FORGE_OK) return st;
    const DxGeometry g = dx_geometry(d_out, d_in, bt, dev->sms);
    fused = want_fused || (ws != nullptr && ws_bytes >= g.bytes);
  }
  if (want_fused && !fused)
    return fail(FORGE_ERR_UNSUPPORTED,
                "backward_accumulate: the fused input gradient needs bf16 X/dY and 1 <= BT <= %lld",
                (long long)kDxMaxTokens);
  if (fused) {
    const DxArgs a{dX, ws, ws_bytes, W};
    return wgrad_step(opt, X, dY, G_acc, nullptr, nullptr, &h, 1, 0, stream, &a);
  }
  if (X->dtype != FORGE_BF16)
    return fail(FORGE_ERR_UNSUPPORTED, "backward_accumulate: gradient accumulation needs bf16 X, dY");
  if ((st = dgrad_impl(dY, W, dX, stream, ws, ws_bytes)) != FORGE_OK) return st;
  return wgrad_step(opt, X, dY, G_acc, nullptr, nullptr, &h, 1, 0, stream);
}

}  // namespace

extern "C" {

forge_status forge_wgrad_step_adamw(const forge_tensor* X, const forge_tensor* dY, forge_tensor* W, forge_tensor* m,
                                    forge_tensor* v, const forge_hyper* h, int64_t step, uint64_t seed,
                                    forge_stream_t stream) {
  return wgrad_step(OPT_ADAMW, X, dY, W, m, v, h, step, seed, stream);
}

forge_status forge_wgrad_step_sgdm(const forge_tensor* X, const forge_tensor* dY, forge_tensor* W, forge_tensor* m,
                                   const forge_hyper* h, int64_t step, uint64_t seed, forge_stream_t stream) {
  return wgrad_step(OPT_SGDM, X, dY, W, m, nullptr, h, step, seed, stream);
}

forge_status forge_wgrad_step_lion(const forge_tensor* X, const forge_tensor* dY, forge_tensor* W, forge_tensor* m,
                                   const forge_hyper* h, int64_t step, uint64_t seed, forge_stream_t stream) {
  return wgrad_step(OPT_LION, X, dY, W, m, nullptr, h, step, seed, stream);
}

forge_status forge_wgrad_step_sgd(const forge_tensor* X, const forge_tensor* dY, forge_tensor* W,
                                  const forge_hyper* h, int64_t step, uint64_t seed, forge_stream_t stream) {
  return wgrad_step(OPT_SGD, X, dY, W, nullptr, nullptr, h, step, seed, stream);
}

forge_status forge_wgrad_step_rmsprop(const forge_tensor* X, const forge_tensor* dY, forge_tensor* W, forge_tensor* v,
                                      const forge_hyper* h, int64_t step, uint64_t seed, forge_stream_t stream) {
  return wgrad_step(OPT_RMSPROP, X, dY, W, v, nullptr, h, step, seed, stream);
}

forge_status forge_wgrad_step_adagrad(const forge_tensor* X, const forge_tensor* dY, forge_tensor* W, forge_tensor* v,
                                      const forge_hyper* h, int64_t step, uint64_t seed, forge_stream_t stream) {
  return wgrad_step(OPT_ADAGRAD, X, dY, W, v, nullptr, h, step, seed, stream);
}

forge_status forge_wgrad_step_nadam(const forge_tensor* X, const forge_tensor* dY, forge_tensor* W, forge_tensor* m,
                                    forge_tensor* v, const forge_hyper* h, int64_t step, uint64_t seed,
                                    forge_stream_t stream) {
  return wgrad_step(OPT_NADAM, X, dY, W, m, v, h, step, seed, stream);
}

forge_status forge_wgrad_step_radam(const forge_tensor* X, const forge_tensor* dY, forge_tensor* W, forge_tensor* m,
                                    forge_tensor* v, const forge_hyper* h, int64_t step, uint64_t seed,
                                    forge_stream_t stream) {
  return wgrad_step(OPT_RADAM, X, dY, W, m, v, h, step, seed, stream);
}

forge_status forge_backward_step(forge_rule rule, const forge_tensor* X, const forge_tensor* dY, forge_tensor* W,
                                 forge_tensor* s0, forge_tensor* s1, forge_tensor* dX, const forge_hyper* h,
                                 int64_t step, uint64_t seed, void* workspace, size_t workspace_bytes,
                                 forge_stream_t stream) {
  if (static_cast<int>(rule) < OPT_ADAMW || static_cast<int>(rule) > OPT_RADAM)
    return fail(FORGE_ERR_INVALID_ARG, "backward_step: unknown rule %d", static_cast<int>(rule));
  return backward_step(static_cast<int>(rule), X, dY, W, s0, s1, dX, h, step, seed, workspace, workspace_bytes,
                       stream);
}

forge_status forge_dgrad(const forge_tensor* dY, const forge_tensor* W_old, forge_tensor* dX, forge_stream_t stream) {
  return dgrad_impl(dY, W_old, dX, stream);
}

forge_status forge_dgrad_ws(const forge_tensor* dY, const forge_tensor* W_old, forge_tensor* dX, void* workspace,
                            size_t workspace_bytes, forge_stream_t stream) {
  return dgrad_impl(dY, W_old, dX, stream, workspace, workspace_bytes);
}

forge_status forge_wgrad_accumulate(const forge_tensor* X, const forge_tensor* dY, forge_tensor* G_acc, int overwrite,
                                    forge_stream_t stream) {
  if (G_acc == nullptr) return fail(FORGE_ERR_INVALID_ARG, "accumulate: null G_acc");
  forge_hyper h;
  std::memset(&h, 0, sizeof(h));
  return wgrad_step(overwrite ? OPT_ACCSET : OPT_ACCUM, X, dY, G_acc, nullptr, nullptr, &h, 1, 0, stream);
}

forge_status forge_backward_accumulate(const forge_tensor* X, const forge_tensor* dY, const forge_tensor* W,
                                       forge_tensor* G_acc, forge_tensor* dX, int overwrite, uint32_t flags,
                                       void* workspace, size_t workspace_bytes, forge_stream_t stream) {
  return backward_accumulate(X, dY, W, G_acc, dX, overwrite, flags, workspace, workspace_bytes, stream);
}

forge_status forge_wgrad_step_accumulated(forge_rule rule, const forge_tensor* X, const forge_tensor* dY,
                                          const forge_tensor* G_acc, forge_tensor* W, forge_tensor* s0,
                                          forge_tensor* s1, const forge_hyper* h, int64_t step, uint64_t seed,
                                          forge_stream_t stream) {
  if (static_cast<int>(rule) < OPT_ADAMW || static_cast<int>(rule) > OPT_RADAM)
    return fail(FORGE_ERR_INVALID_ARG, "step_accumulated: unknown rule %d", static_cast<int>(rule));
  if (G_acc == nullptr) return fail(FORGE_ERR_INVALID_ARG, "step_accumulated: null G_acc");
  return wgrad_step(static_cast<int>(rule), X, dY, W, s0, s1, h, step, seed, stream, nullptr, G_acc);
}

}  // extern "C"

namespace {

forge_status dgrad_impl(const forge_tensor* dY, const forge_tensor* W_old, forge_tensor* dX, forge_stream_t stream,
                        void* ws, size_t ws_bytes, uint32_t flags) {
  if (dY == nullptr || W_old == nullptr || dX == nullptr) return fail(FORGE_ERR_INVALID_ARG, "dgrad: null argument");
  const int64_t bt = dY->rows, d_out = dY->cols, d_in = W_old->cols;
  if (bt < 0 || d_out < 0 || d_in < 0) return fail(FORGE_ERR_INVALID_ARG, "dgrad: negative size");
  if (dY->dtype != FORGE_BF16) return fail(FORGE_ERR_UNSUPPORTED, "dgrad: dY must be bf16");
  if (W_old->dtype != FORGE_BF16 && W_old->dtype != FORGE_F32)
    return fail(FORGE_ERR_UNSUPPORTED, "dgrad: W must be bf16 or f32");
  if (dX->dtype != FORGE_BF16 && dX->dtype != FORGE_F32)
    return fail(FORGE_ERR_UNSUPPORTED, "dgrad: dX must be bf16 or f32");
  forge_status st;
  if ((st = check_tensor(dY, "dY", bt, d_out, true)) != FORGE_OK) return st;
  if ((st = check_tensor(W_old, "W", d_out, d_in, true)) != FORGE_OK) return st;
  if ((st = check_tensor(dX, "dX", bt, d_in, true)) != FORGE_OK) return st;
  if (d_in % 8 != 0 || d_out % 8 != 0)
    return fail(FORGE_ERR_UNSUPPORTED, "dgrad: D_in (%lld) and D_out (%lld) must be multiples of 8",
                (long long)d_in, (long long)d_out);
  if (bt > 0x7FFFFFFF || d_in > 0x7FFFFFFF || d_out > 0x7FFFFFFF)
    return fail(FORGE_ERR_INVALID_ARG, "dgrad: dimension exceeds 2^31 - 1");
  if (bt == 0 || d_in == 0) return ok();

  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != FORGE_OK) return st;
  DgradParams p;
  std::memset(&p, 0, sizeof(p));
  p.dX = dX->data;
  p.ld_dx = dX->ld;
  p.dx_bf16 = dX->dtype == FORGE_BF16 ? 1 : 0;
  p.status = dev->status;
  p.bt = static_cast<int>(bt);
  p.d_out = static_cast<int>(d_out);
  p.d_in = static_cast<int>(d_in);
  // The plan (dgrad_plan): tile shape, and a split contraction where the
  // caller's workspace holds its partial sums.
  const bool w_bf16 = W_old->dtype == FORGE_BF16;
  const bool ws_ok = ws != nullptr && reinterpret_cast<uintptr_t>(ws) % 16 == 0;
  const int force = (flags & FORGE_FLAG_DGRAD_ALL_TOKENS) ? 2 : (flags & FORGE_FLAG_DGRAD_TOKENS_128) ? 1 : 0;
  DgradPlan g = dgrad_plan(d_out, d_in, bt, w_bf16, dev->sms, ws_ok, force);
  if (g.parts >= 2 && ws_bytes < g.bytes) g = dgrad_plan(d_out, d_in, bt, w_bf16, dev->sms, false, force);
  if (g.num_tiles == 0)
    return fail(FORGE_ERR_UNSUPPORTED, "dgrad: all-token tiles need 128 < BT <= 512 (BT = %lld)", (long long)bt);
  const bool split = g.parts >= 2;
  // dY boxes: 64 K columns x 128 token rows, 128-byte swizzle.
  if ((st = encode_2d(&p.tm_dy, dY, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, "dY")) !=
      FORGE_OK)
    return st;
  p.mb = g.mb;
  p.bn = g.bn;
  p.bk = g.bk;
  p.stg_rows = g.stg_rows;
  // All-token tiles start their stage walks at evenly spaced stages, so that
  // the tiles (which all read the same dY rows) spread over L2 (down-
  // projection, bf16 weights, BT 512: 86 -> 76 us; 128-token tiles: no gain).
  p.k_rotate = g.mb > 1 ? 1 : 0;
  p.tiles_m = g.tiles_m;
  p.tiles_n = g.tiles_n;
  p.num_tiles = g.num_tiles;
  p.num_kb = g.num_kb;
  // The W boxes must match what the kernel expects per load: bf16 weights
  // one box of 64 columns x bk rows; fp32 weights 32-column x stg_rows
  // boxes (staged in slots of stg_rows rows, bk / stg_rows per stage).
  if (w_bf16) {
    if ((st = encode_2d(&p.tm_w, W_old, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, static_cast<uint32_t>(g.bk),
                        CU_TENSOR_MAP_SWIZZLE_128B, "W")) != FORGE_OK)
      return st;
    p.w_f32 = nullptr;
  } else {
    if ((st = encode_2d(&p.tm_w, W_old, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 32, static_cast<uint32_t>(g.stg_rows),
                        CU_TENSOR_MAP_SWIZZLE_128B, "W")) != FORGE_OK)
      return st;
    p.w_f32 = static_cast<const float*>(W_old->data);
    p.ld_w32 = W_old->ld;
  }
  p.group_m = 8;
  p.timeout_ns = kTimeoutNs;
  int grid = p.num_tiles < dev->sms ? p.num_tiles : dev->sms;
  if (split) {
    p.splitk = g.parts;
    p.part = static_cast<float*>(ws);
    grid = g.num_tiles * g.parts;
  }
  cudaError_t e = launch_dgrad_tc(p, grid, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(FORGE_ERR_CUDA, "dgrad launch: %s", cudaGetErrorString(e));
  if (split) {
    DgradFixupParams f{};
    f.part = p.part;
    f.dX = p.dX;
    f.ld_dx = p.ld_dx;
    f.dx_bf16 = p.dx_bf16;
    f.bt = p.bt;
    f.d_in = p.d_in;
    f.bn = p.bn;
    f.tiles_m = p.tiles_m;
    f.tiles_n = p.tiles_n;
    f.group_m = p.group_m;
    f.num_tiles = p.num_tiles;
    f.parts = g.parts;
    f.rows = 128 * g.mb;
    e = launch_dgrad_fixup(f, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(FORGE_ERR_CUDA, "dgrad fix-up launch: %s", cudaGetErrorString(e));
  }
  return ok();
}

}  // namespace

extern "C" {

forge_status forge_sync_status(forge_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(FORGE_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
  unsigned int host[4] = {0, 0, 0, 0};
  e = cudaMemcpyFromSymbol(host, forge_device_status, sizeof(host));
  if (e != cudaSuccess) return fail(FORGE_ERR_CUDA, "reading the status word: %s", cudaGetErrorString(e));
  if (host[0] != 0) {
    const unsigned int zero[4] = {0, 0, 0, 0};
    e = cudaMemcpyToSymbol(forge_device_status, zero, sizeof(zero));
    if (e != cudaSuccess) return fail(FORGE_ERR_CUDA, "clearing the status word: %s", cudaGetErrorString(e));
    const char* what = "unknown wait";
    switch (host[0]) {
      case WAIT_OP_EMPTY: what = "operand producer waiting for a free stage"; break;
      case WAIT_OP_FULL: what = "MMA issuer waiting for an operand stage"; break;
      case WAIT_TMEM_EMPTY: what = "MMA issuer waiting for a drained accumulator"; break;
      case WAIT_ST_EMPTY: what = "state producer waiting for a free slot"; break;
      case WAIT_ST_WRITTEN: what = "state storer waiting for the epilogue"; break;
      case WAIT_TMEM_FULL: what = "epilogue waiting for an accumulator"; break;
      case WAIT_ST_FULL: what = "epilogue waiting for a state slot"; break;
      case WAIT_RED: what = "epilogue waiting for the block absmax exchange"; break;
      case WAIT_TEST_HOOK: what = "forced-timeout test hook"; break;
      case WAIT_MMA_DRAIN: what = "MMA issuer draining after an abort"; break;
      case WAIT_DRAIN: what = "producer draining after an abort"; break;
      case WAIT_WB_FULL: what = "MMA issuer waiting for the bf16 W_old tile"; break;
      case WAIT_WB_EMPTY: what = "converters waiting for the W_old buffer"; break;
      case WAIT_DX_FULL: what = "converters waiting for a dX partial"; break;
      case WAIT_DX_EMPTY: what = "MMA issuer waiting for the dX partial to be written out"; break;
      default: break;
    }
    return fail(FORGE_ERR_TIMEOUT, "device wait gave up: %s (code 0x%x)", what, host[0]);
  }
  return ok();
}

const char* forge_last_error(void) { return g_last_error.c_str(); }

const char* forge_version(void) { return "0.3.0"; }

size_t forge_workspace_bytes(int64_t d_out, int64_t d_in, int64_t bt) {
  DeviceInfo* dev = nullptr;
  if (device_info(&dev) != FORGE_OK) return 0;
  const size_t fused = dx_geometry(d_out, d_in, bt, dev->sms).bytes;
  size_t split = 0;
  for (const bool w_bf16 : {false, true}) {
    const DgradPlan g = dgrad_plan(d_out, d_in, bt, w_bf16, dev->sms, true);
    if (g.bytes > split) split = g.bytes;
  }
  return fused > split ? fused : split;
}

}  // extern "C"
