// sgemm_internal.h -- declarations shared by the host API and the kernel
// translation units other than the tile kernel's (whose interface is
// sgemm_plan.h, included here).  Not installed; the public interface is
// include/sgemm.h.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime_api.h>

#include "sgemm_plan.h"

namespace gb300 {

// TF32 tensor-core mode (sgemm_tf32.cu): 128 x 256 output tiles, 32-deep k slices.
size_t tf32_smem_bytes();
int tf32_tile_m();
int tf32_tile_n();
int tf32_tile_k();
int tf32_prepare();  // resident CTAs per SM, or < 0 on error
// Bt (N x K, row stride ldbt, K contiguous) = B^T.
cudaError_t launch_transpose(const float* B, int64_t ldb, float* Bt, int64_t ldbt, int K, int N,
                             cudaStream_t stream);
int tf32_b_chunk();  // columns of B per TMA box when B is read in place (MN-major)
struct Tf32Args {
  int32_t M, N;
  float* C;
  int64_t ldc;
  float* partials;    // split-tile partial sums (128 x 256 floats per slot), or null
  int32_t* counters;  // one arrival counter per split tile, zero on entry, zero on exit
  uint32_t* status;   // device status word
  uint64_t wait_limit_ns;
  int32_t c_scalar;   // C is not 16-byte aligned row by row: 4-byte stores
  int32_t owner_publishes;  // test switch: as GemmArgs::owner_publishes (sgemm_plan.h)
};
// tmap_a: A (K fastest), box {32, 128}, 128-byte swizzle.  b_mn: tmap_b is B itself (N
// fastest), box {32, 32}, 128-byte swizzle of 32-byte atoms; otherwise tmap_b is Bt (K
// fastest), box {32, 256}, 128-byte swizzle.  tmap_c: C (N fastest), box {32, 32},
// 128-byte swizzle, used unless args.c_scalar (then its contents are ignored).  `sched` is
// plan_launch over 128 x 256 x 32 tiles for `grid` persistent CTAs.
cudaError_t launch_tf32_kernel(bool b_mn, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                               const CUtensorMap& tmap_c, const Tf32Args& args, const Sched& sched,
                               int grid, cudaStream_t stream);

// CTA-pair TF32 kernel (tcgen05.mma.cta_group::2): 256 x 256 tiles per pair of SMs.  Returns
// the CTA pairs that can run at once, or <= 0 if none.
int tf32_pair_prepare();
int tf32_pair_tile_m();
int tf32_pair_tile_n();
// tmap_b and tmap_c as for launch_tf32_kernel, except that a transposed Bt is read in
// boxes {32, 128}.  `sched` is plan_launch over 256 x 256 x 32 tiles for `pairs`
// persistent pairs.  Split tiles use two counters and two partial slots (one per CTA of
// the pair) each.
cudaError_t launch_tf32_pair_kernel(bool b_mn, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                                    const CUtensorMap& tmap_c, const Tf32Args& args,
                                    const Sched& sched, int pairs, cudaStream_t stream);

// Small-product kernel (sgemm_small.cu): 64 x 64 tiles, K split into `splits`
// shares of `k_chunk` (a multiple of 16) per tile; grid = tiles x splits.
struct SmallArgs {
  int32_t M, N, K;
  const float* A;  // 16-byte aligned, lda a multiple of 4
  int64_t lda;
  const float* B;  // 16-byte aligned, ldb a multiple of 4
  int64_t ldb;
  float* C;
  int64_t ldc;
  int32_t tiles_n;
  int32_t splits;
  int32_t k_chunk;
  float* partials;    // tiles x splits slots of 64 x 64 floats when splits > 1
  int32_t* counters;  // one per tile, zero on entry and exit, when splits > 1
  int32_t scaled;     // C = alpha * acc + beta * C (beta == 0 never reads C)
  float alpha, beta;
  int32_t c_scalar;   // C accessed 4 bytes at a time
};
struct SmallShape {
  int bm, bn, bk;
};
SmallShape small_shape();
cudaError_t launch_small_kernel(const SmallArgs& args, int64_t tiles, cudaStream_t stream);

// trans_a: A holds op(A)^T (K x M, row stride lda); trans_b: B holds op(B)^T
// (N x K, row stride ldb).  Any alignment and stride.
cudaError_t launch_guarded_kernel(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                                  bool trans_a, const float* B, int64_t ldb, bool trans_b,
                                  float* C, int64_t ldc, int scaled, float alpha, float beta,
                                  cudaStream_t stream);

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

// status[2..3] = status[0..1], then status[0..1] = 0 (status has four words).
cudaError_t launch_status_take(uint32_t* status, cudaStream_t stream);

// Frees sgemm_host()'s device staging, copy streams and events (every device).
void host_staging_release();

}  // namespace gb300
