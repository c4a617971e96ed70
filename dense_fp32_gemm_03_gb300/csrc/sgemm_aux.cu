// sgemm_aux.cu -- the small kernels around the pipelined one:
//  * the bounds-checked GEMM for operands the fast kernels cannot take
//    (misaligned pointers, strides that are not multiples of 4);
//  * the copy of an operand the TMA-fed kernels cannot read in place into an
//    aligned buffer;
//  * the zero fill of C for K == 0 (the empty sum);
//  * the wait-expiry probe behind sgemm_debug_expire_wait().
#include <cuda_runtime.h>

#include "sgemm_device.cuh"
#include "sgemm_internal.h"

namespace gb300 {
namespace {

constexpr int kGBM = 64, kGBN = 64, kGBK = 16, kGThreads = 256;

// Shared-memory tiled GEMM with zero-padded loads and guarded stores ("2D
// Block Tiling: Scaling Matrix Multiplication on NVIDIA H100", section 5, the
// edge kernel), correct for every shape, stride and alignment.  Each thread
// computes a 4 x 4 patch whose rows and columns are strided by 16, so that the
// shared-memory reads of a warp fall in distinct banks or broadcast.  op(A)
// element (m, k) is read at A[m * a_m + k * a_k] and op(B) element (k, n) at
// B[k * b_k + n * b_n], so one kernel serves stored and transposed operands.
__global__ void __launch_bounds__(kGThreads)
    guarded_kernel(int64_t M, int64_t N, int64_t K, const float* __restrict__ A, int64_t a_m,
                   int64_t a_k, const float* __restrict__ B, int64_t b_k, int64_t b_n,
                   float* __restrict__ C, int64_t ldc, int64_t tiles_n, int scaled, float alpha,
                   float beta) {
  __shared__ float As[kGBK][kGBM];
  __shared__ float Bs[kGBK][kGBN];
  const int64_t tile = blockIdx.x;
  const int64_t m0 = (tile / tiles_n) * kGBM, n0 = (tile % tiles_n) * kGBN;
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
  float acc[4][4] = {};
  for (int64_t k0 = 0; k0 < K; k0 += kGBK) {
#pragma unroll
    for (int e = 0; e < kGBM * kGBK / kGThreads; ++e) {
      const int idx = tid + e * kGThreads;
      const int r = idx / kGBK, kk = idx % kGBK;
      const int64_t gm = m0 + r, gk = k0 + kk;
      As[kk][r] = (gm < M && gk < K) ? A[gm * a_m + gk * a_k] : 0.f;
    }
#pragma unroll
    for (int e = 0; e < kGBN * kGBK / kGThreads; ++e) {
      const int idx = tid + e * kGThreads;
      const int kk = idx / kGBN, c = idx % kGBN;
      const int64_t gk = k0 + kk, gn = n0 + c;
      Bs[kk][c] = (gk < K && gn < N) ? B[gk * b_k + gn * b_n] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kGBK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t gm = m0 + ty + 16 * i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t gn = n0 + tx + 16 * j;
      if (gn >= N) continue;
      float* p = C + gm * ldc + gn;
      if (!scaled)
        *p = acc[i][j];
      else
        *p = beta != 0.f ? fmaf(beta, *p, alpha * acc[i][j]) : alpha * acc[i][j];
    }
  }
}

// One warp copies one 128-column segment of one row: 4-byte loads and stores
// that are consecutive across the warp, so any source alignment and stride
// coalesce.  The source is read once, hence the streaming loads.  One launch
// serves up to two matrices (A and B): warps [0, jobs[0].rows * segs) copy
// the first, the rest the second.
constexpr int kPackSeg = 128;

struct PackJob {
  const float* src;
  float* dst;
  int64_t rows, cols, ld_src, ld_dst, segs;
};

__device__ __forceinline__ void pack_segment(const PackJob& j, int64_t w, int lane) {
  const int64_t r = w / j.segs, c0 = (w % j.segs) * kPackSeg + lane;
  const float* s = j.src + r * j.ld_src;
  float* d = j.dst + r * j.ld_dst;
  float v[kPackSeg / 32];
#pragma unroll
  for (int i = 0; i < kPackSeg / 32; ++i) v[i] = c0 + 32 * i < j.cols ? __ldcs(s + c0 + 32 * i) : 0.f;
#pragma unroll
  for (int i = 0; i < kPackSeg / 32; ++i)
    if (c0 + 32 * i < j.cols) d[c0 + 32 * i] = v[i];
}

__global__ void pack_kernel(PackJob j0, PackJob j1) {
  const int lane = threadIdx.x & 31;
  const int64_t n0 = j0.rows * j0.segs, total = n0 + j1.rows * j1.segs;
  const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
  for (int64_t w = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); w < total;
       w += warps) {
    if (w < n0)
      pack_segment(j0, w, lane);
    else
      pack_segment(j1, w - n0, lane);
  }
}

__global__ void zero_fill_kernel(int64_t M, int64_t N, float* __restrict__ C, int64_t ldc) {
  const int64_t total = M * N;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    C[(i / N) * ldc + (i % N)] = 0.f;
  }
}

// C = beta * C: the product term vanishes (K == 0 or alpha == 0).
__global__ void scale_kernel(int64_t M, int64_t N, float* __restrict__ C, int64_t ldc, float beta) {
  const int64_t total = M * N;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    float* p = C + (i / N) * ldc + (i % N);
    *p = beta != 0.f ? beta * *p : 0.f;
  }
}

// Moves the live status word (status[0..1]) into the snapshot (status[2..3])
// and clears it, atomically with respect to kernels still recording on other
// streams: an error recorded after the exchange stays for the next query.
__global__ void status_take_kernel(uint32_t* status) {
  const uint32_t code = atomicExch(status, 0u);
  status[2] = code;
  status[3] = code != 0u ? atomicExch(status + 1, 0u) : 0u;
}

// One CTA waits on a barrier that nothing completes; the bounded wait gives up
// after limit_ns and the timeout is recorded.  Nothing is in flight.
__global__ void expire_probe_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    dev::mbar_init(&bar, 1);
    dev::mbar_init_fence();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!dev::mbar_wait(&bar, 0u, limit_ns)) dev::record_status(status, 3u, kWaitDebugProbe);
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_guarded_kernel(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                                  bool trans_a, const float* B, int64_t ldb, bool trans_b,
                                  float* C, int64_t ldc, int scaled, float alpha, float beta,
                                  cudaStream_t stream) {
  const int64_t tiles_m = (M + kGBM - 1) / kGBM, tiles_n = (N + kGBN - 1) / kGBN;
  const int64_t tiles = tiles_m * tiles_n;
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int64_t a_m = trans_a ? 1 : lda, a_k = trans_a ? lda : 1;
  const int64_t b_k = trans_b ? 1 : ldb, b_n = trans_b ? ldb : 1;
  guarded_kernel<<<unsigned(tiles), kGThreads, 0, stream>>>(M, N, K, A, a_m, a_k, B, b_k, b_n, C,
                                                            ldc, tiles_n, scaled, alpha, beta);
  return cudaGetLastError();
}

cudaError_t launch_pack(const PackCopy& first, const PackCopy& second, cudaStream_t stream) {
  auto job = [](const PackCopy& c) {
    PackJob j{c.src, c.dst, c.rows, c.cols, c.ld_src, c.ld_dst, 0};
    if (c.rows > 0 && c.cols > 0) j.segs = (c.cols + kPackSeg - 1) / kPackSeg;
    else j.rows = 0;
    return j;
  };
  const PackJob j0 = job(first), j1 = job(second);
  const int64_t warps = j0.rows * j0.segs + j1.rows * j1.segs;
  if (warps == 0) return cudaSuccess;
  int64_t blocks = (warps + 7) / 8;  // 8 warps per block
  if (blocks > 65536) blocks = 65536;
  pack_kernel<<<unsigned(blocks), 256, 0, stream>>>(j0, j1);
  return cudaGetLastError();
}

cudaError_t launch_zero_fill(int64_t M, int64_t N, float* C, int64_t ldc, cudaStream_t stream) {
  const int64_t total = M * N;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  zero_fill_kernel<<<unsigned(blocks), 256, 0, stream>>>(M, N, C, ldc);
  return cudaGetLastError();
}

cudaError_t launch_scale(int64_t M, int64_t N, float* C, int64_t ldc, float beta,
                         cudaStream_t stream) {
  const int64_t total = M * N;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  scale_kernel<<<unsigned(blocks), 256, 0, stream>>>(M, N, C, ldc, beta);
  return cudaGetLastError();
}

cudaError_t launch_expire_probe(uint32_t* status, uint64_t limit_ns, cudaStream_t stream) {
  expire_probe_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_status_take(uint32_t* status, cudaStream_t stream) {
  status_take_kernel<<<1, 1, 0, stream>>>(status);
  return cudaGetLastError();
}

}  // namespace gb300
