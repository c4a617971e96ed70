// sgemm_internal.h -- declarations shared by the host API and the kernel translation units.
// Not installed; the public interface is include/sgemm.h.
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
};

TileShape tile_shape(TileConfig cfg);

// Sets the kernel attributes (dynamic shared memory) once per device and
// returns the resident CTAs per SM, or a negative value on error.
int tile_kernel_prepare(TileConfig cfg);

// tmap_a: A as a 2-D tensor (K fastest) with box {16, a_box_rows} and the
// 64-byte swizzle; tmap_b: B (N fastest) with box {BN, 16}, no swizzle.
cudaError_t launch_tile_kernel(TileConfig cfg, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                               const GemmArgs& args, const Sched& sched, int grid,
                               cudaStream_t stream);

// TF32 tensor-core mode (sgemm_tf32.cu): 128 x 256 output tiles, 32-deep k slices.
size_t tf32_smem_bytes();
int tf32_tile_m();
int tf32_tile_n();
int tf32_tile_k();
int tf32_prepare();  // resident CTAs per SM, or < 0 on error
// Bt (N x K, row stride ldbt, K contiguous) = B^T.
cudaError_t launch_transpose(const float* B, int64_t ldb, float* Bt, int64_t ldbt, int K, int N,
                             cudaStream_t stream);
// tmap_a: A (K fastest), box {32, 128}; tmap_bt: Bt (K fastest), box {32, 256}; both with the
// 128-byte swizzle.
cudaError_t launch_tf32_kernel(const CUtensorMap& tmap_a, const CUtensorMap& tmap_bt, int M, int N,
                               int K, float* C, int64_t ldc, int group_m, uint32_t* status,
                               uint64_t limit, cudaStream_t stream);

cudaError_t launch_guarded_kernel(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                                  const float* B, int64_t ldb, float* C, int64_t ldc, int scaled,
                                  float alpha, float beta, cudaStream_t stream);

// dst (rows x cols, row stride ld_dst, 16-byte aligned, ld_dst a multiple of
// 4) = src (any row stride and alignment).  Columns cols..ld_dst-1 of dst are
// left as they are.  rows == 0 or cols == 0: nothing to copy.
struct PackCopy {
  const float* src;
  float* dst;
  int64_t rows, cols, ld_src, ld_dst;
};
// Both copies in one launch.
cudaError_t launch_pack(const PackCopy& first, const PackCopy& second, cudaStream_t stream);

cudaError_t launch_zero_fill(int64_t M, int64_t N, float* C, int64_t ldc, cudaStream_t stream);

// C = beta * C (beta == 0: C = 0 without reading it).
cudaError_t launch_scale(int64_t M, int64_t N, float* C, int64_t ldc, float beta, cudaStream_t stream);

cudaError_t launch_expire_probe(uint32_t* status, uint64_t limit_ns, cudaStream_t stream);

}  // namespace gb300
