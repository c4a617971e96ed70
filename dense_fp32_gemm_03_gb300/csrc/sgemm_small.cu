// sgemm_small.cu -- the FFMA kernel for small products.
//
// Below roughly 768^3 the pipelined kernel is bound by fixed costs: its
// 128-row tiles leave most SMs idle, and its first copies wait for the
// tensor-map descriptors.  Here a CTA of 128 threads computes a 64 x 64
// tile over one share of K ("2D Block Tiling ...", section 4: register
// outer products of 4 x 8 per thread, "Beyond Kernel 7", section "Kernel
// 6": warp tiling), fed by asynchronous 16-byte copies (cp.async) into a
// four-stage shared-memory ring (the multi-stage copy pipeline of "Beyond
// Kernel 7", section "Kernel 8").  K is split so that the grid fills the GPU; the
// shares of a tile publish their partial sums and the last to arrive adds
// them in share order, so the result is the same whoever finishes last.
#include <cuda_runtime.h>

#include "sgemm_device.cuh"
#include "sgemm_internal.h"

namespace gb300 {
namespace {

constexpr int kSmBM = 64, kSmBN = 64, kSmBK = 16, kSmThreads = 128;
constexpr int kSmVec = kSmBM * kSmBN / 4 / kSmThreads;  // float4 outputs per thread: 8

constexpr int kSmStages = 4;  // k-slices in the shared-memory ring (three in flight)

// 16-byte asynchronous copy global -> shared (cp.async, cached in L2 only).
// `bytes` < 16 copies that many bytes and fills the rest of the 16 with
// zeros; bytes == 0 reads nothing (src is then any valid address).
__device__ __forceinline__ void cp_async16(void* dst, const float* src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dev::smem_addr(dst)),
               "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// Waits until at most `n` of this thread's most recent copy groups are pending.
template <int n>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(n) : "memory");
}

// Shared memory: a ring of k-slices, A as rows ([m][k], 64 bytes a row) and
// B as is ([k][n]).  The four 16-byte k-chunks of an A row are stored in the
// order kq ^ ((row / 4) % 4): a warp reads one chunk from each of four rows
// 256 bytes apart, which would otherwise fall on the same four banks; with
// the swizzle the four chunks cover sixteen different banks.
__device__ __forceinline__ int a_chunk(int row, int kq) { return kq ^ ((row >> 2) & 3); }

struct SmallSmem {
  float a[kSmStages][kSmBM][kSmBK];
  float b[kSmStages][kSmBK][kSmBN];
  int last;
};

// Copies k-slice [k0, k0 + 16) of the tile into ring stage `st`: 16-byte
// chunks, two of A and two of B per thread, clipped to M, N and k_end (the
// copies zero-fill what lies outside).  A: thread i = tid + 128 j copies row
// i / 4, k quad i % 4 (a warp covers 8 whole rows); B: row i / 16, column
// quad i % 16 (a warp covers two rows of 64 columns).
__device__ __forceinline__ void issue_slice(const SmallArgs& p, SmallSmem& sm, int st, int m0,
                                            int n0, int k0, int k_end, int tid) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int i = tid + kSmThreads * j;
    const int row = i >> 2, kq = i & 3;
    const int64_t m = int64_t(m0) + row;
    const int k = k0 + 4 * kq;
    const int bytes = m < p.M ? 4 * max(0, min(4, k_end - k)) : 0;
    cp_async16(&sm.a[st][row][4 * a_chunk(row, kq)], bytes > 0 ? p.A + m * p.lda + k : p.A, bytes);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int i = tid + kSmThreads * j;
    const int kr = i >> 4, cq = i & 15;
    const int k = k0 + kr;
    const int64_t n = int64_t(n0) + 4 * cq;
    const int bytes = k < k_end ? int(4 * max(int64_t(0), min(int64_t(4), p.N - n))) : 0;
    cp_async16(&sm.b[st][kr][4 * cq], bytes > 0 ? p.B + int64_t(k) * p.ldb + n : p.B, bytes);
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

  // Ring of kSmStages k-slices: the copies of up to three slices are in
  // flight while one is computed, so a short K does not pay one global round
  // trip per slice.  One copy group per slice, committed even when empty so
  // that the group count stays aligned with the slice index.
#pragma unroll
  for (int st = 0; st < kSmStages - 1; ++st) {
    if (st < nk) issue_slice(p, sm, st, m0, n0, k_begin + st * kSmBK, k_end, tid);
    cp_async_commit();
  }
#pragma unroll 1
  for (int kt = 0; kt < nk; ++kt) {
    cp_async_wait<kSmStages - 2>();  // slice kt has landed (this thread's copies)
    __syncthreads();                 // ... and every thread's; slice kt - 1 is free
    const int nxt = kt + kSmStages - 1;
    if (nxt < nk) issue_slice(p, sm, nxt % kSmStages, m0, n0, k_begin + nxt * kSmBK, k_end, tid);
    cp_async_commit();
    const int st = kt % kSmStages;
#pragma unroll
    for (int k4 = 0; k4 < kSmBK / 4; ++k4) {
      // A at rows 4 ty .. 4 ty + 3, k = 4 k4 .. 4 k4 + 3 (one 128-bit load a row).
      float4 a[4];
#pragma unroll
      for (int r = 0; r < 4; ++r)
        a[r] = *reinterpret_cast<const float4*>(&sm.a[st][4 * ty + r][4 * a_chunk(4 * ty + r, k4)]);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int k = 4 * k4 + kk;
        const float4 b0 = *reinterpret_cast<const float4*>(&sm.b[st][k][4 * tx]);
        const float4 b1 = *reinterpret_cast<const float4*>(&sm.b[st][k][32 + 4 * tx]);
        const float2 bq[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w),
                              make_float2(b1.x, b1.y), make_float2(b1.z, b1.w)};
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const float av = kk == 0 ? a[r].x : kk == 1 ? a[r].y : kk == 2 ? a[r].z : a[r].w;
            dev::ffma2(acc[r][q], make_float2(av, av), bq[q]);
          }
      }
    }
  }
  cp_async_wait<0>();  // no copy is left pending when the CTA moves on

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
  // One thread releases the partial: the barrier orders every thread's stores
  // before its GPU-scope fence (cumulative), the fence before the arrival, and
  // a second fence orders the last arriver's reads below.
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    sm.last = atomicAdd(p.counters + tile, 1) == p.splits - 1 ? 1 : 0;
    __threadfence();
  }
  __syncthreads();
  if (!sm.last) return;
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
