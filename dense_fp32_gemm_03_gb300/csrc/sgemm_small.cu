// sgemm_small.cu -- the FFMA kernel for small products.
//
// Below roughly 768^3 the pipelined kernel is bound by fixed costs: its
// 128-row tiles leave most SMs idle, and its first copies wait for the
// tensor-map descriptors.  Here a CTA of 128 threads computes a 64 x 64
// tile over one share of K ("2D Block Tiling ...", section 4: register
// outer products of 4 x 8 per thread, "Beyond Kernel 7", section "Kernel
// 6": warp tiling), with plain 128-bit loads staged through registers into
// double-buffered shared memory (the prefetch of "Beyond Kernel 7",
// section "Kernel 8").  K is split so that the grid fills the GPU; the
// shares of a tile publish their partial sums and the last to arrive adds
// them in share order, so the result is the same whoever finishes last.
#include <cuda_runtime.h>

#include "sgemm_device.cuh"
#include "sgemm_internal.h"

namespace gb300 {
namespace {

constexpr int kSmBM = 64, kSmBN = 64, kSmBK = 16, kSmThreads = 128;
constexpr int kSmVec = kSmBM * kSmBN / 4 / kSmThreads;  // float4 outputs per thread: 8

// A k-slice of A (64 rows x 16) and of B (16 x 64 columns) held in registers
// between its global loads and its shared-memory stores.
struct Slice {
  float4 a[2];
  float4 b[2];
};

// 128-bit load of row[0..3], columns col..col+3 that lie below `end`, zeros elsewhere.
__device__ __forceinline__ float4 load4(const float* row, int64_t col, int64_t end) {
  if (col + 3 < end) return __ldg(reinterpret_cast<const float4*>(row + col));
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  if (col + 0 < end) v.x = __ldg(row + col);
  if (col + 1 < end) v.y = __ldg(row + col + 1);
  if (col + 2 < end) v.z = __ldg(row + col + 2);
  return v;
}

// Loads k-slice [k0, k0 + 16) of the tile, clipped to [.., k_end) and to M, N.
// A: thread i = tid + 128 j holds rows (i mod 64), k quad (i div 64), so a warp
// touches 32 consecutive rows and the transposed stores are conflict-free.
// B: thread i holds k row (i div 16), column quad (i mod 16).
__device__ __forceinline__ void load_slice(const SmallArgs& p, int m0, int n0, int k0, int k_end,
                                           int tid, Slice& s) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int i = tid + kSmThreads * j;
    const int row = i & 63, kq = i >> 6;
    const int64_t m = int64_t(m0) + row;
    s.a[j] = m < p.M ? load4(p.A + m * p.lda, k0 + 4 * kq, k_end) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int i = tid + kSmThreads * j;
    const int kr = i >> 4, cq = i & 15;
    const int64_t k = int64_t(k0) + kr;
    s.b[j] = k < k_end ? load4(p.B + k * p.ldb, int64_t(n0) + 4 * cq, p.N)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// Shared memory: A k-major ([k][m], transposed on the way in), B as is ([k][n]).
struct SmallSmem {
  float a[2][kSmBK][kSmBM];
  float b[2][kSmBK][kSmBN];
  int last;
};

__device__ __forceinline__ void store_slice(SmallSmem& sm, int buf, int tid, const Slice& s) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int i = tid + kSmThreads * j;
    const int row = i & 63, kq = i >> 6;
    sm.a[buf][4 * kq + 0][row] = s.a[j].x;
    sm.a[buf][4 * kq + 1][row] = s.a[j].y;
    sm.a[buf][4 * kq + 2][row] = s.a[j].z;
    sm.a[buf][4 * kq + 3][row] = s.a[j].w;
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int i = tid + kSmThreads * j;
    const int kr = i >> 4, cq = i & 15;
    *reinterpret_cast<float4*>(&sm.b[buf][kr][4 * cq]) = s.b[j];
  }
}

// Grid: tiles x splits CTAs, CTA (tile, share) = (blockIdx.x / splits, blockIdx.x % splits).
// Thread (ty, tx) = (tid / 8, tid % 8) owns rows 4 ty .. 4 ty + 3 and columns
// 4 tx .. 4 tx + 3 and 32 + 4 tx .. 32 + 4 tx + 3 of the tile (column quads 32
// apart: the eight lanes of a row read 128 contiguous bytes of B).
__global__ void __launch_bounds__(kSmThreads)
    small_kernel(const SmallArgs p) {
  __shared__ __align__(16) SmallSmem sm;
  const int tid = threadIdx.x, ty = tid >> 3, tx = tid & 7;
  const int tile = blockIdx.x / p.splits, share = blockIdx.x % p.splits;
  const int m0 = (tile / p.tiles_n) * kSmBM, n0 = (tile % p.tiles_n) * kSmBN;
  const int k_begin = share * p.k_chunk;
  const int k_end = min(p.K, k_begin + p.k_chunk);
  const int nk = (k_end - k_begin + kSmBK - 1) / kSmBK;

  float2 acc[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[r][q] = make_float2(0.f, 0.f);

  Slice s;
  if (nk > 0) {
    load_slice(p, m0, n0, k_begin, k_end, tid, s);
    store_slice(sm, 0, tid, s);
  }
  __syncthreads();
  for (int kt = 0; kt < nk; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < nk) load_slice(p, m0, n0, k_begin + (kt + 1) * kSmBK, k_end, tid, s);
#pragma unroll
    for (int kk = 0; kk < kSmBK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&sm.a[buf][kk][4 * ty]);
      const float4 b0 = *reinterpret_cast<const float4*>(&sm.b[buf][kk][4 * tx]);
      const float4 b1 = *reinterpret_cast<const float4*>(&sm.b[buf][kk][32 + 4 * tx]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float2 bq[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w),
                            make_float2(b1.x, b1.y), make_float2(b1.z, b1.w)};
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int r = 0; r < 4; ++r) dev::ffma2(acc[r][q], make_float2(av[r], av[r]), bq[q]);
    }
    if (kt + 1 < nk) store_slice(sm, buf ^ 1, tid, s);
    __syncthreads();
  }

  // Output value j (0..7) of this thread: row 4 ty + (j / 2), column quad j % 2.
  auto value = [&](int j) {
    const int r = j >> 1, h = j & 1;
    return make_float4(acc[r][2 * h].x, acc[r][2 * h].y, acc[r][2 * h + 1].x, acc[r][2 * h + 1].y);
  };
  auto store = [&](int j, float4 v) {
    const int64_t row = int64_t(m0) + 4 * ty + (j >> 1);
    const int64_t col = int64_t(n0) + (j & 1) * 32 + 4 * tx;
    if (row >= p.M) return;
    float* c = p.C + row * p.ldc + col;
    const int64_t left = p.N - col;
    if (p.scaled) {
      float4 o = make_float4(p.alpha * v.x, p.alpha * v.y, p.alpha * v.z, p.alpha * v.w);
      if (p.beta != 0.f) {
        float4 old = make_float4(0.f, 0.f, 0.f, 0.f);
        if (left >= 4 && !p.c_scalar) {
          old = *reinterpret_cast<const float4*>(c);
        } else {
          if (left > 0) old.x = c[0];
          if (left > 1) old.y = c[1];
          if (left > 2) old.z = c[2];
          if (left > 3) old.w = c[3];
        }
        o.x = fmaf(p.beta, old.x, o.x);
        o.y = fmaf(p.beta, old.y, o.y);
        o.z = fmaf(p.beta, old.z, o.z);
        o.w = fmaf(p.beta, old.w, o.w);
      }
      v = o;
    }
    if (left >= 4 && !p.c_scalar) {
      *reinterpret_cast<float4*>(c) = v;
    } else {
      if (left > 0) c[0] = v.x;
      if (left > 1) c[1] = v.y;
      if (left > 2) c[2] = v.z;
      if (left > 3) c[3] = v.w;
    }
  };

  if (p.splits == 1) {
#pragma unroll
    for (int j = 0; j < kSmVec; ++j) store(j, value(j));
    return;
  }

  // Split K: publish this share's partial tile (float4 j of thread t at
  // j * 128 + t, coalesced), then the last share to arrive adds all of them
  // in share order, this one's from registers, and writes C.
  constexpr int64_t kSlotVec = int64_t(kSmBM) * kSmBN / 4;
  float4* slots = reinterpret_cast<float4*>(p.partials) + int64_t(tile) * p.splits * kSlotVec;
#pragma unroll
  for (int j = 0; j < kSmVec; ++j) __stcg(slots + share * kSlotVec + j * kSmThreads + tid, value(j));
  __threadfence();
  __syncthreads();
  if (tid == 0) sm.last = atomicAdd(p.counters + tile, 1) == p.splits - 1 ? 1 : 0;
  __syncthreads();
  if (!sm.last) return;
  __threadfence();
  float4 sum[kSmVec];
#pragma unroll 1
  for (int sh = 0; sh < p.splits; ++sh) {
    float4 v[kSmVec];
    if (sh == share) {
#pragma unroll
      for (int j = 0; j < kSmVec; ++j) v[j] = value(j);
    } else {
#pragma unroll
      for (int j = 0; j < kSmVec; ++j) v[j] = __ldcg(slots + sh * kSlotVec + j * kSmThreads + tid);
    }
    if (sh == 0) {
#pragma unroll
      for (int j = 0; j < kSmVec; ++j) sum[j] = v[j];
    } else {
#pragma unroll
      for (int j = 0; j < kSmVec; ++j) {
        sum[j].x += v[j].x;
        sum[j].y += v[j].y;
        sum[j].z += v[j].z;
        sum[j].w += v[j].w;
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kSmVec; ++j) store(j, sum[j]);
  if (tid == 0) p.counters[tile] = 0;
}

}  // namespace

SmallShape small_shape() { return SmallShape{kSmBM, kSmBN, kSmBK}; }

cudaError_t launch_small_kernel(const SmallArgs& args, int64_t tiles, cudaStream_t stream) {
  const int64_t grid = tiles * args.splits;
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  small_kernel<<<unsigned(grid), kSmThreads, 0, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace gb300
