// sgemm_api.cu -- host side of the C ABI declared in include/sgemm.h:
// argument validation, the shape-keyed variant selector, the work
// decomposition (whole-tile waves and Stream-K), the TMA descriptor for B,
// the per-(device, stream) workspace cache and the device status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "sgemm.h"
#include "sgemm_internal.h"

namespace {

using gb300::Sched;
using gb300::TileConfig;
using gb300::TileShape;

// [0] = first sgemm_status_t recorded by a kernel since the last query, [1] = wait site;
// [2..3] = the snapshot a query takes of [0..1] (status_take_kernel).
__device__ uint32_t g_status_word[4];

// sgemm_debug_owner_publishes(): copied into every pipelined launch's arguments.
std::atomic<int> g_owner_publishes{0};

constexpr int64_t kInt32Max = 0x7fffffffLL;
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s: far above any legitimate wait
using gb300::kGroupM;
// Every workspace starts with a counter region of fixed size, so that a cached
// workspace reused with another layout never finds partial sums where its
// counters are: counters are zero at allocation and every call leaves them zero.
constexpr size_t kCounterBytes = 16384;
constexpr int64_t kMaxSplitTiles = kCounterBytes / 4;
// Cost-model constants of the guarded kernel and of the operand copies
// (measured on GB300).
constexpr double kGuardedTflops = 23.0;     // large products
constexpr double kGuardedStepUs = 1.6;      // one 16-deep step of a CTA (a global-load round trip)
constexpr double kGuardedCtasPerSm = 4.0;   // 256 threads x 64 registers
constexpr double kCopyBytesPerUs = 4.5e6;
// Small-product kernel: the time of one 16-deep slice of a 64 x 64 tile
// when the SM runs one CTA (latency bound: the copy ring keeps three slices
// in flight) and the time per four CTAs an SM runs (arithmetic bound); the
// fixed cost of a launch; the reduction of a split tile, a fixed part
// (publishing, the arrival counter) and a part per share (the last share
// reads every other share's 16 KB partial).  Fitted to GB300 timings with
// forced split counts from 64^3 to 1024^3 and K up to 4096.
constexpr int kSmallCtasPerSm = 4;
constexpr double kSmallSliceUs = 0.55;
constexpr double kSmallFullSliceUs = 1.9;
constexpr double kSmallFixedUs = 4.6;
constexpr double kSmallReduceUs = 1.2;
constexpr double kSmallShareUs = 0.45;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
  sgemm_status_t init_status = SGEMM_OK;
  int sms = 0;
  int ctas_per_sm[gb300::kTileConfigs] = {};
  int tf32_ctas_per_sm = 0;
  int tf32_pairs = 0;  // CTA pairs of the 2-SM TF32 kernel that run at once (0: not used)
  uint32_t* status = nullptr;
};

struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
  // A kernel gave up part-way (timeout) since this workspace was last used:
  // its arrival counters may be nonzero.  They are cleared on the owning
  // stream, in stream order, before the next call that uses the workspace.
  bool dirty = false;
};

// Compiled tile configuration behind each tile size of the variants; the
// environment variables SGEMM_TILE_LARGE / SGEMM_TILE_SMALL (a configuration
// id) override them, for tuning sweeps.
int g_cfg_large = 0;
int g_cfg_small = 3;

int env_config(const char* name, int fallback) {
  const char* v = std::getenv(name);
  if (v == nullptr || *v == 0) return fallback;
  char* end = nullptr;
  long id = std::strtol(v, &end, 10);
  return (end && *end == 0 && id >= 0 && id < gb300::kTileConfigs) ? int(id) : fallback;
}

std::mutex g_mu;
std::map<int, DeviceState> g_devices;
std::map<std::pair<int, cudaStream_t>, Workspace> g_workspaces;
// Workspaces replaced by a larger one.  They stay allocated until
// sgemm_release_workspaces(): kernels still running, or a CUDA graph captured
// while one was current, may use them.
std::vector<std::pair<int, void*>> g_retired;
EncodeTiledFn g_encode = nullptr;

// Initialises (once) and returns the state of the current device.
sgemm_status_t device_state(DeviceState** out, int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_devices.find(dev);
  if (it == g_devices.end()) {
    DeviceState st;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) {
      st.init_status = SGEMM_ERR_UNSUPPORTED;  // the library carries sm_103a code only
    } else {
      cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev);
      g_cfg_large = env_config("SGEMM_TILE_LARGE", g_cfg_large);
      g_cfg_small = env_config("SGEMM_TILE_SMALL", g_cfg_small);
      for (int c = 0; c < gb300::kTileConfigs; ++c) {
        st.ctas_per_sm[c] = gb300::tile_kernel_prepare(TileConfig(c));
        if (st.ctas_per_sm[c] <= 0) st.init_status = SGEMM_ERR_LAUNCH;
      }
      if (gb300::specialized_prepare() < 0) st.init_status = SGEMM_ERR_LAUNCH;
      st.tf32_ctas_per_sm = gb300::tf32_prepare();
      st.tf32_pairs = gb300::tf32_pair_prepare();
      if (st.tf32_pairs < 0) st.tf32_pairs = 0;
      // SGEMM_TF32_PAIRS=0 selects the single-SM TF32 kernel (for testing that path).
      const char* pairs_env = std::getenv("SGEMM_TF32_PAIRS");
      if (pairs_env != nullptr && std::strcmp(pairs_env, "0") == 0) st.tf32_pairs = 0;
      if (st.tf32_ctas_per_sm <= 0) st.init_status = SGEMM_ERR_LAUNCH;
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) {
        st.init_status = SGEMM_ERR_LAUNCH;
      } else {
        st.status = static_cast<uint32_t*>(p);
        if (cudaMemset(p, 0, sizeof(g_status_word)) != cudaSuccess) st.init_status = SGEMM_ERR_LAUNCH;
      }
      if (g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
          g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        } else {
          st.init_status = SGEMM_ERR_UNSUPPORTED;
        }
      }
    }
    cudaGetLastError();  // attribute queries must not leak a sticky error into the caller
    it = g_devices.emplace(dev, st).first;
  }
  *out = &it->second;
  if (dev_out) *dev_out = dev;
  return it->second.init_status;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const float* a, int64_t rows, int64_t cols, int64_t ld, const float* c,
              int64_t crows, int64_t ccols, int64_t ldc) {
  if (rows == 0 || cols == 0 || crows == 0 || ccols == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a);
  const uintptr_t a1 = a0 + uintptr_t(((rows - 1) * ld + cols) * 4);
  const uintptr_t c0 = reinterpret_cast<uintptr_t>(c);
  const uintptr_t c1 = c0 + uintptr_t(((crows - 1) * ldc + ccols) * 4);
  return a0 < c1 && c0 < a1;
}

// Argument checks.  A holds op(A) (M x K) or, when trans_a, op(A)^T (K x M);
// B holds op(B) (K x N) or, when trans_b, op(B)^T (N x K); row strides lda,
// ldb, ldc cover the stored rows.
sgemm_status_t validate(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda, bool trans_a,
                        const float* B, int64_t ldb, bool trans_b, const float* C, int64_t ldc) {
  if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_VALUE;
  if (M > kInt32Max || N > kInt32Max || K > kInt32Max) return SGEMM_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return SGEMM_OK;
  if (C == nullptr || ldc < N) return SGEMM_ERR_INVALID_VALUE;
  if (K == 0) return SGEMM_OK;
  const int64_t a_rows = trans_a ? K : M, a_cols = trans_a ? M : K;
  const int64_t b_rows = trans_b ? N : K, b_cols = trans_b ? K : N;
  if (A == nullptr || B == nullptr || lda < a_cols || ldb < b_cols) return SGEMM_ERR_INVALID_VALUE;
  if (overlaps(A, a_rows, a_cols, lda, C, M, N, ldc) || overlaps(B, b_rows, b_cols, ldb, C, M, N, ldc))
    return SGEMM_ERR_INVALID_VALUE;
  return SGEMM_OK;
}

sgemm_status_t validate(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                        const float* B, int64_t ldb, const float* C, int64_t ldc) {
  return validate(M, N, K, A, lda, false, B, ldb, false, C, ldc);
}

bool fast_path_ok(const float* A, int64_t lda, const float* B, int64_t ldb, const float* C,
                  int64_t ldc) {
  return aligned16(A) && aligned16(B) && aligned16(C) && lda % 4 == 0 && ldb % 4 == 0 &&
         ldc % 4 == 0;
}

bool operand_ok(const void* p, int64_t ld) { return aligned16(p) && ld % 4 == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Plan {
  int variant = -1;
  TileConfig cfg = 0;
  Sched sc{};
  int grid = 0;
  size_t partial_bytes = 0;
  // The small-product kernel's decomposition: 64 x 64 tiles, K in `splits` shares.
  int64_t small_tiles = 0, small_tiles_n = 0;
  int splits = 1, k_chunk = 0;
  size_t workspace_bytes() const { return partial_bytes ? kCounterBytes + partial_bytes : 0; }
};

// The staged variant: an operand the TMA-fed kernels cannot read in place (a
// base address that is not 16-byte aligned, or a row stride that is not a
// multiple of 4 floats) is first copied into the workspace with row stride
// round_up(cols, 4); a C of that kind is written with 4-byte stores.  The
// copies sit after the counter region and the partial tiles.
struct Staging {
  bool a = false, b = false;
  int64_t lda = 0, ldb = 0;     // row strides of the copies
  size_t a_off = 0, b_off = 0;  // byte offsets of the copies in the workspace
  size_t bytes = 0;             // workspace bytes, copies included
};

Staging make_staging(const Plan& p, int64_t M, int64_t N, int64_t K, bool stage_a, bool stage_b) {
  Staging sg;
  sg.bytes = p.workspace_bytes();
  if (!stage_a && !stage_b) return sg;
  size_t off = kCounterBytes + round_up(p.partial_bytes, 256);
  if (stage_a) {
    sg.a = true;
    sg.lda = (K + 3) / 4 * 4;
    sg.a_off = off;
    off += round_up(size_t(M) * size_t(sg.lda) * 4, 256);
  }
  if (stage_b) {
    sg.b = true;
    sg.ldb = (N + 3) / 4 * 4;
    sg.b_off = off;
    off += round_up(size_t(K) * size_t(sg.ldb) * 4, 256);
  }
  sg.bytes = off;
  return sg;
}

bool is_fast(int v) {
  return v == SGEMM_VARIANT_TILED || v == SGEMM_VARIANT_STREAMK ||
         v == SGEMM_VARIANT_TILED_SMALL || v == SGEMM_VARIANT_STREAMK_SMALL ||
         v == SGEMM_VARIANT_SMALL;
}

// Estimated duration (microseconds) of the small-product kernel for `grid`
// CTAs of `slices` 16-deep slices each, the tiles split into `splits` shares.
// Each SM works through its CTAs' slices at the arithmetic rate
// (kSmallFullSliceUs per slice of four CTAs), but no faster than one slice
// per kSmallSliceUs.
double small_cost_us(int64_t grid, int64_t slices, int64_t splits, const DeviceState& ds) {
  const double per_sm = std::ceil(double(grid) / double(ds.sms));
  double slice_us = kSmallFullSliceUs * per_sm / kSmallCtasPerSm;
  if (slice_us < kSmallSliceUs) slice_us = kSmallSliceUs;
  const double reduce = splits > 1 ? kSmallReduceUs + kSmallShareUs * double(splits) : 0.0;
  return kSmallFixedUs + double(slices) * slice_us + reduce;
}

// The small-product kernel: the number of K shares per tile (a power of two,
// at least two 16-deep slices per share) with the lowest estimated time.
bool make_small_plan(int64_t M, int64_t N, int64_t K, const DeviceState& ds, Plan* p) {
  const gb300::SmallShape ss = gb300::small_shape();
  const int64_t tiles_n = (N + ss.bn - 1) / ss.bn;
  const int64_t tiles = ((M + ss.bm - 1) / ss.bm) * tiles_n;
  const int64_t kslices = (K + ss.bk - 1) / ss.bk;
  if (tiles > kInt32Max || tiles_n > kInt32Max || kslices * ss.bk > kInt32Max) return false;
  double best = 1e300;
  int64_t best_splits = 1, best_chunk = kslices * ss.bk;
  for (int64_t want = 1; want == 1 || (want <= kslices / 2 && tiles * want <= kInt32Max);
       want *= 2) {
    const int64_t chunk_slices = (kslices + want - 1) / want;
    const int64_t splits = (kslices + chunk_slices - 1) / chunk_slices;
    if (splits > 1 && tiles > kMaxSplitTiles) break;
    const double cost = small_cost_us(tiles * splits, chunk_slices, splits, ds);
    if (cost < best * 0.999) {
      best = cost;
      best_splits = splits;
      best_chunk = chunk_slices * ss.bk;
    }
  }
  if (tiles * best_splits > kInt32Max) return false;
  p->small_tiles = tiles;
  p->small_tiles_n = tiles_n;
  p->splits = int(best_splits);
  p->k_chunk = int(best_chunk);
  p->grid = int(tiles * best_splits);
  p->partial_bytes = best_splits > 1 ? size_t(tiles * best_splits) * ss.bm * ss.bn * 4 : 0;
  return true;
}

// Work decomposition of a fast variant.
bool make_plan(int variant, int64_t M, int64_t N, int64_t K, const DeviceState& ds, Plan* p) {
  p->variant = variant;
  if (!is_fast(variant)) return true;
  if (variant == SGEMM_VARIANT_SMALL) return make_small_plan(M, N, K, ds, p);
  p->cfg = (variant == SGEMM_VARIANT_TILED_SMALL || variant == SGEMM_VARIANT_STREAMK_SMALL)
               ? g_cfg_small
               : g_cfg_large;
  const TileShape ts = gb300::tile_shape(p->cfg);
  const bool streamk = (variant == SGEMM_VARIANT_STREAMK || variant == SGEMM_VARIANT_STREAMK_SMALL);
  const int64_t resident = int64_t(ds.sms) * ds.ctas_per_sm[p->cfg];
  const gb300::LaunchPlan lp = gb300::plan_launch(M, N, K, ts.bm, ts.bn, ts.bk, resident, streamk);
  if (!lp.ok || lp.grid > kInt32Max) return false;
  if (lp.sc.sk_tiles > kMaxSplitTiles) return false;
  p->sc = lp.sc;
  p->grid = int(lp.grid);
  p->partial_bytes = size_t(lp.slots) * ts.bm * ts.bn * 4;
  return true;
}

// The size-specialized instance compiled for exactly this planned launch, or -1.
int find_specialized(const Plan& p, int64_t M, int64_t N, int64_t K, const DeviceState& ds) {
  if (p.variant != SGEMM_VARIANT_STREAMK && p.variant != SGEMM_VARIANT_STREAMK_SMALL) return -1;
  const TileShape ts = gb300::tile_shape(p.cfg);
  return gb300::find_specialized_plan(p.cfg, M, N, K, ts.bm, ts.bn, ts.bk,
                                      int64_t(ds.sms) * ds.ctas_per_sm[p.cfg], p.sc, p.grid);
}

// Estimated duration (microseconds) of a planned fast variant on this device.
// The model was fitted to measured GB300 timings of the compiled
// configurations: every CTA slot streams its k-tiles at a fixed efficiency
// of the FFMA peak (86% with 8x16 patches, 80% with 8x8), plus a fixed cost
// per launch (6 us: start-up and tail, fitted from 256^3 to 1280^3) and,
// when tiles are split, the time the last CTA of a tile spends reading the
// partial sums back.
double plan_cost_us(const Plan& p, const DeviceState& ds) {
  if (p.variant == SGEMM_VARIANT_SMALL)
    return small_cost_us(p.grid, p.k_chunk / 16, p.splits, ds);
  const TileShape ts = gb300::tile_shape(p.cfg);
  const int cps = ds.ctas_per_sm[p.cfg] > 0 ? ds.ctas_per_sm[p.cfg] : 1;
  const double flop_per_us_per_sm = 128.0 * 2.0 * 2070.0;  // FFMA lanes x 2 x max clock (MHz)
  const double eff = ts.patch_n == 16 ? 0.86 : 0.80;
  const double ktile_us = double(ts.bm) * ts.bn * ts.bk * 2.0 * cps / (flop_per_us_per_sm * eff);
  const int64_t resident = int64_t(ds.sms) * cps;
  const double ipt = p.sc.iters_per_tile;
  if (p.sc.sk_tiles == 0 && p.sc.dp_tiles == int64_t(p.sc.tiles_m) * p.sc.tiles_n &&
      p.grid == p.sc.dp_tiles) {
    // One tile per CTA: whole waves of CTA slots.
    const int64_t waves = (int64_t(p.sc.dp_tiles) + resident - 1) / resident;
    return 6.0 + double(waves) * ipt * ktile_us;
  }
  const double dp_waves = double(p.sc.dp_tiles) / double(resident);
  double iters = dp_waves * ipt;
  double fixup = 0.0;
  if (p.sc.sk_tiles > 0) {
    iters += double(p.sc.sk_base + (p.sc.sk_extra ? 1 : 0));
    // The last CTA of a split tile reads every segment's partial tile back.
    const double tile_kb = double(ts.bm) * ts.bn * 4.0 / 1024.0;
    const double segments = std::ceil(double(p.sc.sk_ctas) / double(p.sc.sk_tiles)) + 1.0;
    fixup = 0.015 * tile_kb * segments;
  }
  return 6.0 + iters * ktile_us + fixup;
}

// Estimated duration (microseconds) of the bounds-checked kernel, fitted to
// measured GB300 timings: small products are bound by the latency of its
// unpipelined 16-deep steps (one global round trip each, per wave of 64 x 64
// tiles), large ones by its arithmetic rate.
double guarded_cost_us(int64_t M, int64_t N, int64_t K, const DeviceState& ds) {
  const double tiles = double((M + 63) / 64) * double((N + 63) / 64);
  const double waves = std::ceil(tiles / (double(ds.sms) * kGuardedCtasPerSm));
  const double latency = kGuardedStepUs * double((K + 15) / 16) * waves;
  const double arithmetic = 2.0 * double(M) * double(N) * double(K) / (kGuardedTflops * 1e6);
  return 5.0 + (latency > arithmetic ? latency : arithmetic);
}

// How a fast variant receives an operand.
enum OpMode {
  kInPlace,    // read where it is (16-byte aligned, row stride a multiple of 4)
  kInPlaceMN,  // A^T read where it is as an M-major A (pipelined kernels only)
  kPack,       // copied into the workspace as is, aligned (pack_kernel)
  kTranspose,  // copied into the workspace transposed (transpose kernel)
};

// The pipelined variants read a transposed A in place when their tile
// configuration has the M-major instance (the default ones do).
bool reads_a_mn(int v) {
  if (v == SGEMM_VARIANT_TILED || v == SGEMM_VARIANT_STREAMK) return gb300::tile_shape(g_cfg_large).a_mn;
  if (v == SGEMM_VARIANT_TILED_SMALL || v == SGEMM_VARIANT_STREAMK_SMALL)
    return gb300::tile_shape(g_cfg_small).a_mn;
  return false;
}

OpMode a_mode(int v, bool trans_a, bool aligned) {
  if (!trans_a) return aligned ? kInPlace : kPack;
  return aligned && reads_a_mn(v) ? kInPlaceMN : kTranspose;
}

OpMode b_mode(bool trans_b, bool aligned) {
  if (!trans_b) return aligned ? kInPlace : kPack;
  return kTranspose;
}

bool is_copy(OpMode m) { return m == kPack || m == kTranspose; }

// Estimated cost (microseconds) of the operand copies: 8 bytes of traffic per
// element, plus a launch for the packed copies (one for both) and one per
// transposed copy.
double copies_cost_us(int64_t M, int64_t N, int64_t K, OpMode am, OpMode bm) {
  double us = 0.0;
  int launches = 0;
  bool pack = false;
  if (is_copy(am)) {
    us += 8.0 * double(M) * double(K) / kCopyBytesPerUs;
    if (am == kTranspose) ++launches; else pack = true;
  }
  if (is_copy(bm)) {
    us += 8.0 * double(K) * double(N) / kCopyBytesPerUs;
    if (bm == kTranspose) ++launches; else pack = true;
  }
  if (pack) ++launches;
  return us + 4.0 * launches;
}

// The pipelined variant with the lowest estimated time for this shape,
// operand copies included (a_ok, b_ok: the operand could be read in place).
int select_fast(int64_t M, int64_t N, int64_t K, bool trans_a, bool a_ok, bool trans_b, bool b_ok,
                const DeviceState& ds, double* cost_out) {
  int best = SGEMM_VARIANT_STREAMK;
  double best_cost = 1e300;
  const int candidates[5] = {SGEMM_VARIANT_STREAMK, SGEMM_VARIANT_STREAMK_SMALL,
                             SGEMM_VARIANT_TILED, SGEMM_VARIANT_TILED_SMALL, SGEMM_VARIANT_SMALL};
  for (int v : candidates) {
    Plan p;
    if (!make_plan(v, M, N, K, ds, &p)) continue;
    const double cost = plan_cost_us(p, ds) +
                        copies_cost_us(M, N, K, a_mode(v, trans_a, a_ok), b_mode(trans_b, b_ok));
    if (cost < best_cost * 0.999) {
      best_cost = cost;
      best = v;
    }
  }
  if (cost_out) *cost_out = best_cost;
  return best;
}

int select_fast(int64_t M, int64_t N, int64_t K, const DeviceState& ds, double* cost_out) {
  return select_fast(M, N, K, false, true, false, true, ds, cost_out);
}

// The selector: when every operand a pipelined kernel reads in place is
// aligned (a transposed B is always copied; a transposed A is read M-major
// where it is, or copied), the pipelined variant with the lowest estimated
// time; otherwise the staged variant or the bounds-checked kernel, whichever
// is estimated faster.
int select_variant(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda, bool trans_a,
                   const float* B, int64_t ldb, bool trans_b, const float* C, int64_t ldc,
                   const DeviceState& ds) {
  const bool a_ok = operand_ok(A, lda), b_ok = operand_ok(B, ldb), c_ok = operand_ok(C, ldc);
  double cost = 0.0;
  const int fast = select_fast(M, N, K, trans_a, a_ok, trans_b, b_ok, ds, &cost);
  if (c_ok && (a_ok || trans_a) && (b_ok || trans_b)) {
    Plan p;
    const OpMode am = a_mode(fast, trans_a, a_ok);
    if (am == kInPlace && !trans_b && make_plan(fast, M, N, K, ds, &p) &&
        find_specialized(p, M, N, K, ds) >= 0)
      return SGEMM_VARIANT_SPECIALIZED;
    return fast;
  }
  return cost < guarded_cost_us(M, N, K, ds) ? SGEMM_VARIANT_STAGED : SGEMM_VARIANT_GUARDED;
}

int select_variant(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda, const float* B,
                   int64_t ldb, const float* C, int64_t ldc, const DeviceState& ds) {
  return select_variant(M, N, K, A, lda, false, B, ldb, false, C, ldc, ds);
}

sgemm_status_t get_workspace_bytes(int dev, cudaStream_t stream, size_t need, void** out) {
  *out = nullptr;
  if (need == 0) return SGEMM_OK;
  std::lock_guard<std::mutex> lock(g_mu);
  Workspace& ws = g_workspaces[{dev, stream}];
  if (ws.bytes < need) {
    if (ws.ptr) {
      // Not freed here: earlier kernels on this stream, or a graph captured
      // with it, may still use the old buffer (and cudaFree would also wait
      // for the whole device).
      g_retired.emplace_back(dev, ws.ptr);
      ws.ptr = nullptr;
      ws.bytes = 0;
    }
    size_t bytes = need + need / 4;
    if (cudaMalloc(&ws.ptr, bytes) != cudaSuccess) {
      cudaGetLastError();
      ws.ptr = nullptr;
      return SGEMM_ERR_ALLOC;
    }
    // Arrival counters start at zero; every finished tile resets its own.
    if (cudaMemsetAsync(ws.ptr, 0, bytes, stream) != cudaSuccess) {
      cudaFree(ws.ptr);
      ws.ptr = nullptr;
      return SGEMM_ERR_LAUNCH;
    }
    ws.bytes = bytes;
    ws.dirty = false;
  } else if (ws.dirty) {
    // After a timeout: clear the counters behind everything already queued
    // on this stream, ahead of this call's kernels.
    if (cudaMemsetAsync(ws.ptr, 0, kCounterBytes, stream) != cudaSuccess) return SGEMM_ERR_LAUNCH;
    ws.dirty = false;
  }
  *out = ws.ptr;
  return SGEMM_OK;
}

// Tensor maps of the pipelined kernel: A (K fastest) in boxes of 16 x
// a_box_rows with the 64-byte swizzle, or, for an M-major A (a_mn: the
// storage of A^T, K x M with M fastest), boxes of BM x 16 without swizzle;
// B (N fastest) in boxes of BN x 16.
sgemm_status_t encode_operands(const TileShape& ts, int64_t M, int64_t N, int64_t K, const float* A,
                               int64_t lda, bool a_mn, const float* B, int64_t ldb,
                               CUtensorMap* tmap_a, CUtensorMap* tmap_b) {
  std::memset(tmap_a, 0, sizeof(*tmap_a));
  std::memset(tmap_b, 0, sizeof(*tmap_b));
  const cuuint32_t estr[2] = {1, 1};
  {
    const cuuint64_t dims[2] = {a_mn ? cuuint64_t(M) : cuuint64_t(K), a_mn ? cuuint64_t(K) : cuuint64_t(M)};
    const cuuint64_t strides[1] = {cuuint64_t(lda) * 4};
    const cuuint32_t box[2] = {a_mn ? cuuint32_t(ts.bm) : cuuint32_t(ts.bk),
                               a_mn ? cuuint32_t(ts.bk) : cuuint32_t(ts.a_box_rows)};
    if (g_encode(tmap_a, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(A), dims, strides,
                 box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 a_mn ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_64B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return SGEMM_ERR_LAUNCH;
  }
  {
    const cuuint64_t dims[2] = {cuuint64_t(N), cuuint64_t(K)};
    const cuuint64_t strides[1] = {cuuint64_t(ldb) * 4};
    const cuuint32_t box[2] = {cuuint32_t(ts.bn), cuuint32_t(ts.bk)};
    if (g_encode(tmap_b, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(B), dims, strides,
                 box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return SGEMM_ERR_LAUNCH;
  }
  return SGEMM_OK;
}

// One call of the product C = alpha * op(A) op(B) + beta * C in row-major
// storage (trans_a / trans_b: the operand is stored transposed).
sgemm_status_t run(int variant, int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                   int64_t lda, bool trans_a, const float* B, int64_t ldb, bool trans_b, float beta,
                   float* C, int64_t ldc, cudaStream_t stream) {
  const bool scaled = !(alpha == 1.0f && beta == 0.0f);
  sgemm_status_t st = validate(M, N, K, A, lda, trans_a, B, ldb, trans_b, C, ldc);
  if (st != SGEMM_OK) return st;
  if (variant < SGEMM_VARIANT_AUTO || variant >= SGEMM_VARIANT_COUNT) return SGEMM_ERR_INVALID_VALUE;
  DeviceState* ds = nullptr;
  int dev = 0;
  st = device_state(&ds, &dev);
  if (st != SGEMM_OK) return st;
  if (M == 0 || N == 0) return SGEMM_OK;
  if (K == 0 || alpha == 0.0f) {  // the product term vanishes: C = beta * C
    const cudaError_t e = scaled ? gb300::launch_scale(M, N, C, ldc, beta, stream)
                                 : gb300::launch_zero_fill(M, N, C, ldc, stream);
    return e == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
  }
  if (variant == SGEMM_VARIANT_AUTO)
    variant = select_variant(M, N, K, A, lda, trans_a, B, ldb, trans_b, C, ldc, *ds);
  if (variant == SGEMM_VARIANT_GUARDED) {
    return gb300::launch_guarded_kernel(M, N, K, A, lda, trans_a, B, ldb, trans_b, C, ldc,
                                        scaled ? 1 : 0, alpha, beta, stream) == cudaSuccess
               ? SGEMM_OK
               : SGEMM_ERR_LAUNCH;
  }
  const bool a_ok = operand_ok(A, lda), b_ok = operand_ok(B, ldb), c_ok = operand_ok(C, ldc);
  const bool staged = variant == SGEMM_VARIANT_STAGED;
  const bool specialized = variant == SGEMM_VARIANT_SPECIALIZED;
  if (staged || specialized)
    variant = select_fast(M, N, K, trans_a, a_ok, trans_b, b_ok, *ds, nullptr);
  const OpMode am = a_mode(variant, trans_a, a_ok), bm = b_mode(trans_b, b_ok);
  // Outside the staged variant, operands are only copied to transpose them.
  if (!staged && (am == kPack || bm == kPack || !c_ok)) return SGEMM_ERR_INVALID_VALUE;
  Plan p;
  if (!make_plan(variant, M, N, K, *ds, &p)) return SGEMM_ERR_UNSUPPORTED;
  // The compiled-in schedule serves the plain epilogue over operands read in
  // place; the selector names it for any shape it fits, so alpha / beta fall
  // back to the generic instance of the same schedule.
  int spec = -1;
  if (specialized) {
    spec = find_specialized(p, M, N, K, *ds);
    // The compiled-in instances read A K-major in place and B in place.
    if (spec < 0 || am != kInPlace || bm != kInPlace) return SGEMM_ERR_UNSUPPORTED;
    if (scaled) spec = -1;
  }
  const TileShape ts = gb300::tile_shape(p.cfg);
  const Staging sg = make_staging(p, M, N, K, is_copy(am), is_copy(bm));

  void* ws = nullptr;
  st = get_workspace_bytes(dev, stream, sg.bytes, &ws);
  if (st != SGEMM_OK) return st;
  const float* a_in = A;
  const float* b_in = B;
  int64_t lda_in = lda, ldb_in = ldb;
  gb300::PackCopy copy_a{}, copy_b{};
  if (sg.a) {
    float* a_copy = reinterpret_cast<float*>(static_cast<char*>(ws) + sg.a_off);
    if (am == kTranspose) {
      // A holds op(A)^T (K x M): its transpose is the row-major M x K op(A).
      if (gb300::launch_transpose(A, lda, a_copy, sg.lda, int(K), int(M), stream) != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    } else {
      copy_a = gb300::PackCopy{A, a_copy, M, K, lda, sg.lda};
    }
    a_in = a_copy;
    lda_in = sg.lda;
  }
  if (sg.b) {
    float* b_copy = reinterpret_cast<float*>(static_cast<char*>(ws) + sg.b_off);
    if (bm == kTranspose) {
      // B holds op(B)^T (N x K): its transpose is the row-major K x N op(B).
      if (gb300::launch_transpose(B, ldb, b_copy, sg.ldb, int(N), int(K), stream) != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    } else {
      copy_b = gb300::PackCopy{B, b_copy, K, N, ldb, sg.ldb};
    }
    b_in = b_copy;
    ldb_in = sg.ldb;
  }
  if ((am == kPack || bm == kPack) && gb300::launch_pack(copy_a, copy_b, stream) != cudaSuccess)
    return SGEMM_ERR_LAUNCH;
  if (p.variant == SGEMM_VARIANT_SMALL) {
    gb300::SmallArgs sa{};
    sa.M = int(M);
    sa.N = int(N);
    sa.K = int(K);
    sa.A = a_in;
    sa.lda = lda_in;
    sa.B = b_in;
    sa.ldb = ldb_in;
    sa.C = C;
    sa.ldc = ldc;
    sa.tiles_n = int(p.small_tiles_n);
    sa.splits = p.splits;
    sa.k_chunk = p.k_chunk;
    sa.counters = static_cast<int32_t*>(ws);
    sa.partials = ws ? reinterpret_cast<float*>(static_cast<char*>(ws) + kCounterBytes) : nullptr;
    sa.scaled = scaled ? 1 : 0;
    sa.alpha = alpha;
    sa.beta = beta;
    sa.c_scalar = c_ok ? 0 : 1;
    return gb300::launch_small_kernel(sa, p.small_tiles, stream) == cudaSuccess ? SGEMM_OK
                                                                               : SGEMM_ERR_LAUNCH;
  }
  const bool a_mn = am == kInPlaceMN;
  CUtensorMap tmap_a, tmap_b;
  st = encode_operands(ts, M, N, K, a_in, lda_in, a_mn, b_in, ldb_in, &tmap_a, &tmap_b);
  if (st != SGEMM_OK) return st;

  gb300::GemmArgs args{};
  args.M = int(M);
  args.N = int(N);
  args.K = int(K);
  args.A = a_in;
  args.lda = lda_in;
  args.C = C;
  args.ldc = ldc;
  args.counters = static_cast<int32_t*>(ws);
  args.partials = ws ? reinterpret_cast<float*>(static_cast<char*>(ws) + kCounterBytes) : nullptr;
  args.status = ds->status;
  args.wait_limit_ns = kDefaultWaitLimitNs;
  args.scaled = scaled ? 1 : 0;
  args.alpha = alpha;
  args.beta = beta;
  args.c_scalar = c_ok ? 0 : 1;
  args.a_mn = a_mn ? 1 : 0;
  args.owner_publishes = g_owner_publishes.load(std::memory_order_relaxed);
  const cudaError_t e =
      spec >= 0 ? gb300::launch_specialized(spec, tmap_a, tmap_b, args, p.sc, p.grid, stream)
                : gb300::launch_tile_kernel(p.cfg, tmap_a, tmap_b, args, p.sc, p.grid, stream);
  return e == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
}

sgemm_status_t run(int variant, int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                   int64_t lda, const float* B, int64_t ldb, float beta, float* C, int64_t ldc,
                   cudaStream_t stream) {
  return run(variant, M, N, K, alpha, A, lda, false, B, ldb, false, beta, C, ldc, stream);
}

}  // namespace

extern "C" {

sgemm_status_t sgemm(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda, const float* B,
                     int64_t ldb, float* C, int64_t ldc, cudaStream_t stream) {
  return run(SGEMM_VARIANT_AUTO, M, N, K, 1.0f, A, lda, B, ldb, 0.0f, C, ldc, stream);
}

sgemm_status_t sgemm_ex(int layout, int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                        int64_t lda, const float* B, int64_t ldb, float beta, float* C, int64_t ldc,
                        cudaStream_t stream) {
  if (layout == SGEMM_ROW_MAJOR)
    return run(SGEMM_VARIANT_AUTO, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
  if (layout != SGEMM_COL_MAJOR) return SGEMM_ERR_INVALID_VALUE;
  // Column-major C = A B is row-major C^T = B^T A^T over the same memory: the
  // column-major B (K x N, ld ldb) read row-major is B^T (N x K), and so on.
  return run(SGEMM_VARIANT_AUTO, N, M, K, alpha, B, ldb, A, lda, beta, C, ldc, stream);
}

sgemm_status_t sgemm_ex2(int layout, int trans_a, int trans_b, int64_t M, int64_t N, int64_t K,
                         float alpha, const float* A, int64_t lda, const float* B, int64_t ldb,
                         float beta, float* C, int64_t ldc, cudaStream_t stream) {
  if ((trans_a != SGEMM_OP_N && trans_a != SGEMM_OP_T) ||
      (trans_b != SGEMM_OP_N && trans_b != SGEMM_OP_T))
    return SGEMM_ERR_INVALID_VALUE;
  const bool ta = trans_a == SGEMM_OP_T, tb = trans_b == SGEMM_OP_T;
  if (layout == SGEMM_ROW_MAJOR)
    return run(SGEMM_VARIANT_AUTO, M, N, K, alpha, A, lda, ta, B, ldb, tb, beta, C, ldc, stream);
  if (layout != SGEMM_COL_MAJOR) return SGEMM_ERR_INVALID_VALUE;
  // Column-major C = op(A) op(B) is row-major C^T = op(B)^T op(A)^T over the
  // same memory.  A column-major matrix read row-major is its transpose, so
  // B's memory read row-major is op(B)^T exactly when op(B) = B (trans_b ==
  // N): each operand keeps its own flag.
  return run(SGEMM_VARIANT_AUTO, N, M, K, alpha, B, ldb, tb, A, lda, ta, beta, C, ldc, stream);
}

sgemm_status_t sgemm_variant(int variant, int64_t M, int64_t N, int64_t K, const float* A,
                             int64_t lda, const float* B, int64_t ldb, float* C, int64_t ldc,
                             cudaStream_t stream) {
  return run(variant, M, N, K, 1.0f, A, lda, B, ldb, 0.0f, C, ldc, stream);
}

int sgemm_select_variant(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                         const float* B, int64_t ldb, const float* C, int64_t ldc) {
  if (validate(M, N, K, A, lda, B, ldb, C, ldc) != SGEMM_OK) return -1;
  DeviceState* ds = nullptr;
  if (device_state(&ds, nullptr) != SGEMM_OK) return -1;
  return select_variant(M, N, K, A, lda, B, ldb, C, ldc, *ds);
}

size_t sgemm_workspace_size(int variant, int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0 || M > kInt32Max || N > kInt32Max || K > kInt32Max) return 0;
  DeviceState* ds = nullptr;
  if (device_state(&ds, nullptr) != SGEMM_OK) return 0;
  if (variant == SGEMM_VARIANT_AUTO) {
    // Aligned operands are assumed (the guarded kernel needs no workspace).
    const float* p = reinterpret_cast<const float*>(uintptr_t(256));
    variant = select_variant(M, N, K, p, (K + 3) / 4 * 4, p, (N + 3) / 4 * 4, p, (N + 3) / 4 * 4, *ds);
  }
  const bool staged = variant == SGEMM_VARIANT_STAGED;
  if (staged || variant == SGEMM_VARIANT_SPECIALIZED) variant = select_fast(M, N, K, *ds, nullptr);
  Plan p;
  if (!make_plan(variant, M, N, K, *ds, &p)) return 0;
  // The staged variant is sized for copies of both A and B.
  return make_staging(p, M, N, K, staged, staged).bytes;
}

sgemm_status_t sgemm_tf32(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                          const float* B, int64_t ldb, float* C, int64_t ldc, cudaStream_t stream) {
  sgemm_status_t st = validate(M, N, K, A, lda, B, ldb, C, ldc);
  if (st != SGEMM_OK) return st;
  DeviceState* ds = nullptr;
  int dev = 0;
  st = device_state(&ds, &dev);
  if (st != SGEMM_OK) return st;
  if (M == 0 || N == 0) return SGEMM_OK;
  if (K == 0) {
    return gb300::launch_zero_fill(M, N, C, ldc, stream) == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
  }
  // A goes to the tensor cores by TMA: an A that TMA cannot read in place is
  // first copied into the workspace (rows padded to a multiple of 4 floats).
  // A C that is not 16-byte aligned row by row is written 4 bytes at a time.
  const bool a_copy = !operand_ok(A, lda);
  const bool c_scalar = !operand_ok(C, ldc);
  // 128 x 256 x 32 tiles.  More tiles than resident CTAs: a persistent
  // Stream-K schedule (one CTA per SM) that splits the last partial wave over
  // K.  At most one wave: one tile per CTA, since reducing 128 KB partial
  // tiles then costs more than the idle SMs (measured on GB300 from 1024^3
  // to 2048^3; from 2560^3 up the split schedule wins).
  const bool pair = ds->tf32_pairs > 0;
  const int64_t resident = pair ? int64_t(ds->tf32_pairs) : int64_t(ds->sms) * ds->tf32_ctas_per_sm;
  const int bm = pair ? gb300::tf32_pair_tile_m() : gb300::tf32_tile_m();
  const int bn = pair ? gb300::tf32_pair_tile_n() : gb300::tf32_tile_n();
  const int bk = gb300::tf32_tile_k();
  const int64_t tiles = ((M + bm - 1) / bm) * ((N + bn - 1) / bn);
  const gb300::LaunchPlan lp = gb300::plan_launch(M, N, K, bm, bn, bk, resident, tiles > resident);
  if (!lp.ok || lp.grid > kInt32Max ||
      lp.sc.sk_tiles * (pair ? 2 : 1) > kMaxSplitTiles)
    return SGEMM_ERR_UNSUPPORTED;
  // Workspace: [counters][partial slots][B^T when B cannot be read in place]
  // [copy of A when A cannot be read in place].
  const size_t slot_bytes = size_t(bm) * bn * 4;
  const size_t partial_bytes = size_t(lp.slots) * slot_bytes;
  // B is read in place as an MN-major operand when TMA can address it;
  // otherwise B^T (N x K, rows padded to a multiple of 4 floats) is written
  // to the workspace and read K-major like A.
  const bool b_mn = operand_ok(B, ldb);
  const int64_t ldbt = (K + 3) / 4 * 4;
  const size_t bt_off = kCounterBytes + round_up(partial_bytes, 256);
  const int64_t lda_copy = (K + 3) / 4 * 4;
  const size_t a_off = round_up(b_mn ? kCounterBytes + partial_bytes : bt_off + size_t(N) * ldbt * 4, 256);
  size_t ws_bytes =
      b_mn ? (partial_bytes ? kCounterBytes + partial_bytes : 0) : bt_off + size_t(N) * ldbt * 4;
  if (a_copy) ws_bytes = a_off + size_t(M) * size_t(lda_copy) * 4;
  void* ws = nullptr;
  st = get_workspace_bytes(dev, stream, ws_bytes, &ws);
  if (st != SGEMM_OK) return st;
  if (a_copy) {
    float* a_dst = reinterpret_cast<float*>(static_cast<char*>(ws) + a_off);
    const gb300::PackCopy copy{A, a_dst, M, K, lda, lda_copy};
    if (gb300::launch_pack(copy, gb300::PackCopy{}, stream) != cudaSuccess) return SGEMM_ERR_LAUNCH;
    A = a_dst;
    lda = lda_copy;
  }
  const float* b_src = B;
  if (!b_mn) {
    float* Bt = reinterpret_cast<float*>(static_cast<char*>(ws) + bt_off);
    if (gb300::launch_transpose(B, ldb, Bt, ldbt, int(K), int(N), stream) != cudaSuccess)
      return SGEMM_ERR_LAUNCH;
    b_src = Bt;
    ldb = ldbt;
  }

  CUtensorMap tmap_a, tmap_b;
  std::memset(&tmap_a, 0, sizeof(tmap_a));
  std::memset(&tmap_b, 0, sizeof(tmap_b));
  const cuuint32_t estr[2] = {1, 1};
  {
    const cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(M)};
    const cuuint64_t strides[1] = {cuuint64_t(lda) * 4};
    const cuuint32_t box[2] = {cuuint32_t(gb300::tf32_tile_k()), cuuint32_t(gb300::tf32_tile_m())};
    if (g_encode(&tmap_a, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(A), dims, strides,
                 box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return SGEMM_ERR_LAUNCH;
  }
  {
    // In place: B (N fastest), boxes of 32 columns x 32 rows of k, 128-byte
    // swizzle of 32-byte atoms (what MN-major TF32 operands take).
    // Transposed: Bt (K fastest), boxes of 32 k x 256 rows, 128-byte swizzle.
    const cuuint64_t dims[2] = {b_mn ? cuuint64_t(N) : cuuint64_t(K),
                                b_mn ? cuuint64_t(K) : cuuint64_t(N)};
    const cuuint64_t strides[1] = {cuuint64_t(ldb) * 4};
    const cuuint32_t box[2] = {
        b_mn ? cuuint32_t(gb300::tf32_b_chunk()) : cuuint32_t(bk),
        b_mn ? cuuint32_t(bk) : cuuint32_t(pair ? bn / 2 : bn)};
    if (g_encode(&tmap_b, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(b_src), dims,
                 strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 b_mn ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B : CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return SGEMM_ERR_LAUNCH;
  }
  // C for the kernels' TMA stores: boxes of 32 columns x 32 rows, 128-byte swizzle.
  CUtensorMap tmap_c;
  std::memset(&tmap_c, 0, sizeof(tmap_c));
  if (!c_scalar) {
    const cuuint64_t dims[2] = {cuuint64_t(N), cuuint64_t(M)};
    const cuuint64_t strides[1] = {cuuint64_t(ldc) * 4};
    const cuuint32_t box[2] = {32, 32};
    if (g_encode(&tmap_c, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, C, dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return SGEMM_ERR_LAUNCH;
  }
  gb300::Tf32Args args{};
  args.M = int(M);
  args.N = int(N);
  args.C = C;
  args.ldc = ldc;
  args.counters = static_cast<int32_t*>(ws);
  args.partials = ws ? reinterpret_cast<float*>(static_cast<char*>(ws) + kCounterBytes) : nullptr;
  args.status = ds->status;
  args.wait_limit_ns = kDefaultWaitLimitNs;
  args.c_scalar = c_scalar ? 1 : 0;
  args.owner_publishes = g_owner_publishes.load(std::memory_order_relaxed);
  const cudaError_t e =
      pair ? gb300::launch_tf32_pair_kernel(b_mn, tmap_a, tmap_b, tmap_c, args, lp.sc, int(lp.grid),
                                             stream)
           : gb300::launch_tf32_kernel(b_mn, tmap_a, tmap_b, tmap_c, args, lp.sc, int(lp.grid), stream);
  return e == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
}

sgemm_status_t sgemm_query_device_status(cudaStream_t stream, uint32_t* detail) {
  DeviceState* ds = nullptr;
  int dev = 0;
  sgemm_status_t st = device_state(&ds, &dev);
  if (detail) *detail = 0;
  if (st != SGEMM_OK) return st;
  // Take and clear the word on `stream` (an atomic exchange on the device, so
  // kernels still running on other streams lose no record), then read it.
  uint32_t word[2] = {0, 0};
  if (gb300::launch_status_take(ds->status, stream) != cudaSuccess ||
      cudaMemcpyAsync(word, ds->status + 2, sizeof(word), cudaMemcpyDeviceToHost, stream) !=
          cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return SGEMM_ERR_LAUNCH;
  if (word[0] == SGEMM_OK) return SGEMM_OK;
  if (detail) *detail = word[1];
  // A kernel gave up part-way: its arrival counters may be left nonzero.  The
  // workspaces of this device are cleared lazily, each on its own stream just
  // before its next use, so that no kernel still running on another stream
  // sees its counters change under it.
  {
    std::lock_guard<std::mutex> lock(g_mu);
    for (auto& kv : g_workspaces)
      if (kv.first.first == dev && kv.second.ptr) kv.second.dirty = true;
  }
  return sgemm_status_t(word[0]);
}

void sgemm_release_workspaces(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int cur = 0;
  cudaGetDevice(&cur);
  auto release = [](int dev, void* ptr) {
    cudaSetDevice(dev);
    cudaDeviceSynchronize();
    cudaFree(ptr);
  };
  for (auto& kv : g_workspaces)
    if (kv.second.ptr) release(kv.first.first, kv.second.ptr);
  for (auto& r : g_retired) release(r.first, r.second);
  g_workspaces.clear();
  g_retired.clear();
  cudaSetDevice(cur);
  gb300::host_staging_release();
}

const char* sgemm_status_string(sgemm_status_t s) {
  switch (s) {
    case SGEMM_OK: return "ok";
    case SGEMM_ERR_INVALID_VALUE: return "invalid argument";
    case SGEMM_ERR_LAUNCH: return "CUDA launch or API call failed";
    case SGEMM_ERR_TIMEOUT: return "device wait exceeded its time limit";
    case SGEMM_ERR_UNSUPPORTED: return "unsupported device or size";
    case SGEMM_ERR_ALLOC: return "workspace allocation failed";
  }
  return "unknown status";
}

const char* sgemm_variant_name(int v) {
  switch (v) {
    case SGEMM_VARIANT_GUARDED: return "guarded";
    case SGEMM_VARIANT_TILED: return "tiled";
    case SGEMM_VARIANT_STREAMK: return "streamk";
    case SGEMM_VARIANT_TILED_SMALL: return "tiled_small";
    case SGEMM_VARIANT_STREAMK_SMALL: return "streamk_small";
    case SGEMM_VARIANT_STAGED: return "staged";
    case SGEMM_VARIANT_SPECIALIZED: return "specialized";
    case SGEMM_VARIANT_SMALL: return "small";
  }
  return "unknown";
}

void sgemm_debug_owner_publishes(int on) {
  g_owner_publishes.store(on ? 1 : 0, std::memory_order_relaxed);
}

sgemm_status_t sgemm_debug_expire_wait(uint64_t limit_ns, cudaStream_t stream) {
  DeviceState* ds = nullptr;
  sgemm_status_t st = device_state(&ds, nullptr);
  if (st != SGEMM_OK) return st;
  if (limit_ns > 10000000000ull) return SGEMM_ERR_INVALID_VALUE;  // keep the probe short
  return gb300::launch_expire_probe(ds->status, limit_ns, stream) == cudaSuccess ? SGEMM_OK
                                                                                 : SGEMM_ERR_LAUNCH;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free Stream-K entry point.
//
// The Stream-K schedule needs scratch memory (arrival counters and the
// partial sums of split tiles).  sgemm() takes it from a cache that calls
// cudaMalloc the first time a stream needs more.  Some callers cannot let a
// library allocate: code that must never wait on the whole device
// (cudaMalloc and cudaFree may synchronise it), code that hands out a fixed
// memory budget before any work starts, and code inside a framework whose own
// allocator owns the device memory.  sgemm_streamk_static() serves them from a fixed array in the
// library's device image instead.
namespace {

// Every GPU that loads the library holds this array until the process exits.
constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch, per device.  In host code the symbol is
// only a host-side stand-in, never a device address.
std::map<int, void*> g_static_scratch_addr;

sgemm_status_t static_scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_static_scratch_addr.find(dev);
  if (it == g_static_scratch_addr.end()) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return SGEMM_ERR_LAUNCH;
    }
    it = g_static_scratch_addr.emplace(dev, p).first;
  }
  *out = it->second;
  return SGEMM_OK;
}

}  // namespace

extern "C" sgemm_status_t sgemm_streamk_static(int64_t M, int64_t N, int64_t K, const float* A,
                                               int64_t lda, const float* B, int64_t ldb, float* C,
                                               int64_t ldc, cudaStream_t stream) {
  sgemm_status_t st = validate(M, N, K, A, lda, B, ldb, C, ldc);
  if (st != SGEMM_OK) return st;
  DeviceState* ds = nullptr;
  int dev = 0;
  st = device_state(&ds, &dev);
  if (st != SGEMM_OK) return st;
  if (M == 0 || N == 0) return SGEMM_OK;
  if (K == 0) {
    return gb300::launch_zero_fill(M, N, C, ldc, stream) == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
  }
  if (!fast_path_ok(A, lda, B, ldb, C, ldc)) return SGEMM_ERR_INVALID_VALUE;
  Plan p;
  if (!make_plan(SGEMM_VARIANT_STREAMK, M, N, K, *ds, &p)) return SGEMM_ERR_UNSUPPORTED;
  if (p.workspace_bytes() > kStaticScratchBytes) return SGEMM_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  st = static_scratch_address(dev, &scratch);
  if (st != SGEMM_OK) return st;
  const TileShape ts = gb300::tile_shape(p.cfg);

  CUtensorMap tmap_a, tmap_b;
  st = encode_operands(ts, M, N, K, A, lda, false, B, ldb, &tmap_a, &tmap_b);
  if (st != SGEMM_OK) return st;

  // The array keeps whatever the previous call left: the arrival counters of
  // this call's split tiles must start at zero.
  if (p.sc.sk_tiles > 0 &&
      cudaMemsetAsync(scratch, 0, size_t(p.sc.sk_tiles) * sizeof(int32_t), stream) != cudaSuccess)
    return SGEMM_ERR_LAUNCH;
  gb300::GemmArgs args{};
  args.M = int(M);
  args.N = int(N);
  args.K = int(K);
  args.A = A;
  args.lda = lda;
  args.C = C;
  args.ldc = ldc;
  args.counters = static_cast<int32_t*>(scratch);
  args.partials = reinterpret_cast<float*>(static_cast<char*>(scratch) + kCounterBytes);
  args.status = ds->status;
  args.wait_limit_ns = kDefaultWaitLimitNs;
  args.owner_publishes = g_owner_publishes.load(std::memory_order_relaxed);
  return gb300::launch_tile_kernel(p.cfg, tmap_a, tmap_b, args, p.sc, p.grid, stream) == cudaSuccess
             ? SGEMM_OK
             : SGEMM_ERR_LAUNCH;
}
