// sgemm_aux.cu -- the small kernels around the pipelined one:
//  * the bounds-checked GEMM for operands the fast kernels cannot take
//    (misaligned pointers, strides that are not multiples of 4);
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
// shared-memory reads of a warp fall in distinct banks or broadcast.
__global__ void __launch_bounds__(kGThreads)
    guarded_kernel(int64_t M, int64_t N, int64_t K, const float* __restrict__ A, int64_t lda,
                   const float* __restrict__ B, int64_t ldb, float* __restrict__ C, int64_t ldc,
                   int64_t tiles_n, int scaled, float alpha, float beta) {
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
      As[kk][r] = (gm < M && gk < K) ? A[gm * lda + gk] : 0.f;
    }
#pragma unroll
    for (int e = 0; e < kGBN * kGBK / kGThreads; ++e) {
      const int idx = tid + e * kGThreads;
      const int kk = idx / kGBN, c = idx % kGBN;
      const int64_t gk = k0 + kk, gn = n0 + c;
      Bs[kk][c] = (gk < K && gn < N) ? B[gk * ldb + gn] : 0.f;
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
                                  const float* B, int64_t ldb, float* C, int64_t ldc, int scaled,
                                  float alpha, float beta, cudaStream_t stream) {
  const int64_t tiles_m = (M + kGBM - 1) / kGBM, tiles_n = (N + kGBN - 1) / kGBN;
  const int64_t tiles = tiles_m * tiles_n;
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
  guarded_kernel<<<unsigned(tiles), kGThreads, 0, stream>>>(M, N, K, A, lda, B, ldb, C, ldc,
                                                            tiles_n, scaled, alpha, beta);
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

}  // namespace gb300
