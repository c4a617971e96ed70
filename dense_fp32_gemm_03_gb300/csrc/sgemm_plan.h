// sgemm_plan.h -- the FFMA tile kernel's interface: its work decomposition
// (Sched, plan_launch), launch arguments and launchers, shared by the host
// API, the tile kernel and the schedule walk.  Not installed; the public
// interface is include/sgemm.h.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime_api.h>

namespace gb300 {

// Codes written to the device status word (detail) when a bounded wait expires.
enum WaitSite : uint32_t {
  kWaitNone = 0,
  kWaitTileStage = 1,   // a compute thread waiting for a B stage (TMA) to land
  kWaitDrain = 2,       // draining in-flight copies after an error
  kWaitDebugProbe = 3,  // the deliberate expiry hook
};

// Work decomposition of one launch of the tile kernel (host-computed).
//
// The output is cut into tiles_m x tiles_n tiles of BM x BN, visited in a
// grouped ("swizzled") order of `group_m` tile rows.  Tiles [0, dp_tiles) are
// computed whole, tile c + w * gridDim.x by CTA c.  The K iterations of tiles
// [dp_tiles, dp_tiles + sk_tiles) form one stream that is cut evenly over the
// first sk_ctas CTAs (Stream-K): CTA c < sk_ctas owns iterations
// [c * sk_base + min(c, sk_extra), ...) of length sk_base + (c < sk_extra).  A tile whose K range is shared by
// several CTAs is finished by whichever of them arrives last, which adds the
// partial sums in CTA order (deterministic).
struct Sched {
  int32_t tiles_m, tiles_n;
  int32_t group_m;
  int32_t iters_per_tile;  // ceil(K / BK)
  int32_t dp_tiles;
  int32_t sk_tiles;
  int32_t sk_ctas;
  int32_t sk_base, sk_extra;
};

__host__ __device__ constexpr bool same_sched(const Sched& a, const Sched& b) {
  return a.tiles_m == b.tiles_m && a.tiles_n == b.tiles_n && a.group_m == b.group_m &&
         a.iters_per_tile == b.iters_per_tile && a.dp_tiles == b.dp_tiles &&
         a.sk_tiles == b.sk_tiles && a.sk_ctas == b.sk_ctas && a.sk_base == b.sk_base &&
         a.sk_extra == b.sk_extra;
}

// Constants of the work decomposition, shared by the host planner and the
// size-specialized kernel instances (which compile the plan in).
constexpr int kGroupM = 8;      // tile rows per raster group
constexpr int kMinSkIters = 4;  // Stream-K shares shorter than this many k-tiles are not worth splitting

struct LaunchPlan {
  bool ok;        // false: a size does not fit the schedule's 32-bit fields
  Sched sc;
  int64_t grid;   // CTAs launched
  int64_t slots;  // partial-tile slots the split tiles need (0: none)
};

// The schedule of one launch over BM x BN x BK tiles.  One tile per CTA, or
// (streamk) a persistent grid of `resident` CTAs: whole tiles fill complete
// waves and the tiles of the last, partial wave are shared out over K.
__host__ __device__ constexpr LaunchPlan plan_launch(int64_t M, int64_t N, int64_t K, int bm,
                                                     int bn, int bk, int64_t resident,
                                                     bool streamk) {
  LaunchPlan p{};
  const int64_t tiles_m = (M + bm - 1) / bm, tiles_n = (N + bn - 1) / bn;
  const int64_t tiles = tiles_m * tiles_n;
  const int64_t ipt = (K + bk - 1) / bk;
  p.ok = tiles <= 0x7fffffffLL && ipt <= 0x7fffffffLL;
  if (!p.ok) return p;
  p.sc.tiles_m = int32_t(tiles_m);
  p.sc.tiles_n = int32_t(tiles_n);
  p.sc.group_m = kGroupM;
  p.sc.iters_per_tile = int32_t(ipt);
  if (!streamk || resident <= 0) {
    p.sc.dp_tiles = int32_t(tiles);
    p.grid = tiles;
    return p;
  }
  const int64_t waves = tiles / resident;
  const int64_t rem = tiles % resident;
  p.sc.dp_tiles = int32_t(waves * resident);
  p.sc.sk_tiles = int32_t(rem);
  p.grid = tiles < resident ? tiles : resident;
  if (rem > 0) {
    const int64_t total = rem * ipt;
    int64_t sk_ctas = resident;
    if (total / sk_ctas < kMinSkIters) sk_ctas = total / kMinSkIters;
    if (sk_ctas < rem) sk_ctas = rem;  // never fewer sharers than tiles
    if (sk_ctas > resident) sk_ctas = resident;
    p.sc.sk_ctas = int32_t(sk_ctas);
    p.sc.sk_base = int32_t(total / sk_ctas);
    p.sc.sk_extra = int32_t(total % sk_ctas);
    p.grid = p.sc.dp_tiles > 0 ? resident : sk_ctas;
    p.slots = rem + sk_ctas - 1;
  }
  return p;
}

struct GemmArgs {
  int32_t M, N, K;
  const float* A;
  int64_t lda;
  float* C;
  int64_t ldc;
  float* partials;      // Stream-K partial tiles (sk_tiles + gridDim.x - 1 slots), or null
  int32_t* counters;    // one arrival counter per split tile, zero on entry, zero on exit
  uint32_t* status;     // device status word: [0] = sgemm_status_t, [1] = WaitSite
  uint64_t wait_limit_ns;
  // Epilogue C = alpha * acc + beta * C when `scaled` (beta == 0 never reads C);
  // C = acc otherwise.
  int32_t scaled;
  float alpha, beta;
  // Nonzero when C is not 16-byte aligned or ldc is not a multiple of 4: every
  // access to C is then a 4-byte one (in the general epilogue, which also
  // applies alpha and beta: alpha = 1, beta = 0 leave acc unchanged).
  int32_t c_scalar;
  // Nonzero when A arrives M-major (the operand is A^T stored K x M, M
  // fastest): tmap_a then has box {BM, BK} and its copies land in the A ring
  // as the compute warps read it, with no staging and no transposition.
  int32_t a_mn;
  // Test switch: nonzero makes the CTA that owns a split tile's first
  // k-tiles publish its partial like every other sharer, so the last to arrive
  // always sums all partials from the workspace (the same additions, in CTA
  // order, as the owner's sum from its registers).
  int32_t owner_publishes;
};

// Tile configurations of the pipelined kernel (compiled instances, by id).
typedef int TileConfig;
constexpr int kTileConfigs = 6;

struct TileShape {
  int bm, bn, bk, threads, stages;
  size_t smem_bytes;
  int a_box_rows;  // rows of A per TMA copy (one producer warp's slice)
  int patch_n;     // outputs per thread along N (16 or 8)
  int ctas_per_sm; // CTAs the configuration is built to co-reside per SM
  bool a_mn;       // has an instance that reads A M-major (GemmArgs::a_mn)
};

TileShape tile_shape(TileConfig cfg);

// Sets the kernel attributes (dynamic shared memory) once per device and
// returns the resident CTAs per SM, or a negative value on error.
int tile_kernel_prepare(TileConfig cfg);

// tmap_a: A as a 2-D tensor (K fastest) with box {16, a_box_rows} and the
// 64-byte swizzle, or, when args.a_mn, A^T's storage (M fastest) with box
// {BM, 16} and no swizzle; tmap_b: B (N fastest) with box {BN, 16}, no swizzle.
cudaError_t launch_tile_kernel(TileConfig cfg, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                               const GemmArgs& args, const Sched& sched, int grid,
                               cudaStream_t stream);

// Size-specialized instances: the plain epilogue (C = A * B, 16-byte-aligned
// C) of one configuration with M, N, K and the Stream-K schedule of
// kSpecializedResident CTAs compiled in as constants.
constexpr int kSpecializedResident = 152;  // GB300: 152 SMs, one CTA each
struct SpecShape {
  TileConfig cfg;
  int64_t m, n, k;
};
// The compiled instances, by index (the kernel translation unit checks that
// its instance list matches this table).  768^3 and 1024^3 run 128 x 128
// tiles (configuration 3), 4096^3 128 x 256 (configuration 0).
constexpr SpecShape kSpecShapes[] = {{0, 4096, 4096, 4096}, {3, 1024, 1024, 1024},
                                     {3, 768, 768, 768}};
constexpr int kSpecShapeCount = int(sizeof(kSpecShapes) / sizeof(kSpecShapes[0]));

// The instance compiled for exactly this launch -- configuration `cfg` with
// BM x BN x BK tiles, the planned schedule `sc` over `grid` CTAs, `resident`
// CTAs able to run at once -- or -1.  An instance's schedule is compiled for
// kSpecializedResident CTAs, so on a device with another SM count (times
// CTAs per SM) nothing matches and the generic kernel runs.
constexpr int find_specialized_plan(TileConfig cfg, int64_t M, int64_t N,
                                         int64_t K, int bm, int bn, int bk,
                                         int64_t resident, const Sched& sc,
                                         int64_t grid) {
  if (resident != kSpecializedResident) return -1;
  for (int i = 0; i < kSpecShapeCount; ++i) {
    const SpecShape& s = kSpecShapes[i];
    if (s.cfg != cfg || s.m != M || s.n != N || s.k != K) continue;
    const LaunchPlan lp = plan_launch(M, N, K, bm, bn, bk, kSpecializedResident, true);
    if (lp.ok && same_sched(lp.sc, sc) && lp.grid == grid) return i;
  }
  return -1;
}
int specialized_count();
SpecShape specialized_shape(int i);
int specialized_prepare();  // 0, or < 0 on error
// `sched` and `grid` must be the plan the instance was compiled with.
cudaError_t launch_specialized(int i, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                               const GemmArgs& args, const Sched& sched, int grid,
                               cudaStream_t stream);

}  // namespace gb300
