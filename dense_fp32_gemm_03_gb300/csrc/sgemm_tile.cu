// sgemm_tile.cu -- the pipelined FP32 GEMM kernel for sm_103a.
//
// C = A * B, row-major FP32, alpha = 1, beta = 0 ("Beyond Kernel 7: Closing
// the Gap to cuBLAS on an H100 FP32 GEMM", section "The operation").  One
// kernel template serves three schedules (see Sched in sgemm_internal.h):
// one tile per CTA, persistent whole-tile waves, and Stream-K splits of K.
//
// Per CTA and output tile BM x BN:
//  * B (K x N) streams global -> shared through a STAGES-deep ring filled by
//    TMA (cp.async.bulk.tensor) and guarded by one mbarrier per stage.  The
//    ring is the multi-stage pipeline of "Beyond Kernel 7", section "Kernel 8:
//    asynchronous copies", with the bulk tensor copy engine in place of
//    per-thread cp.async.
//  * A (M x K) is read with 128-bit loads one k-tile ahead into registers
//    ("Vectorized Memory Access ...", sections 1 and 3) and written to shared
//    memory transposed, k-major ([k][m], section 4 of the same page), with
//    every value stored twice side by side so that a 128-bit shared load
//    yields ready-made operand pairs (a, a) for the paired FMA.
//  * Each thread owns an 8 x 16 patch of C (128 accumulators; the 16 x 8 /
//    8 x 16 patches of "Beyond Kernel 7", section "Kernel 10"), updated per
//    k step as a register outer product ("2D Block Tiling ...", section 4)
//    with fma.rn.f32x2: one instruction performs two FP32 FFMAs, each with
//    its own single rounding, which halves the issue slots the arithmetic
//    takes and leaves room for the shared loads and address math that bound
//    the pages' kernels (same page, "Kernel 11" and the closing roofline).
//  * Warp tiling ("Beyond Kernel 7", section "Kernel 6"): a warp covers
//    32 x 128 outputs as a 4 x 8 lane grid; within a patch the column quads
//    are strided by 32 so that the eight lanes of a row read 128 contiguous
//    bytes of B (conflict-free; "Kernel 10", strided B-column mapping) and
//    the four lanes of a column read 64 contiguous bytes of A (broadcast).
//  * Output: coalesced 128-bit row stores ("cuSgemm", Kernel 5), bounds
//    checked on edge tiles ("2D Block Tiling ...", section 5).
#include <cuda.h>
#include <cuda_runtime.h>

#include "sgemm_device.cuh"
#include "sgemm_internal.h"

namespace gb300 {
namespace {

constexpr uint32_t kStatusTimeout = 3;  // SGEMM_ERR_TIMEOUT

template <int WARPS_M, int WARPS_N, int BK_, int STAGES, int MIN_CTAS>
struct TileCfg {
  static constexpr int kTR = 4, kTC = 8;    // lane grid of a warp: rows x columns
  static constexpr int kTM = 8, kTN = 16;   // outputs per thread
  static constexpr int kWarpM = kTR * kTM;  // 32
  static constexpr int kWarpN = kTC * kTN;  // 128
  static constexpr int kWarpsM = WARPS_M;
  static constexpr int BM = WARPS_M * kWarpM;
  static constexpr int BN = WARPS_N * kWarpN;
  static constexpr int BK = BK_;
  static constexpr int S = STAGES;
  static constexpr int NT = 32 * WARPS_M * WARPS_N;
  static constexpr int kMinCtas = MIN_CTAS;
  static constexpr int kAStride = 2 * BM;  // floats per k row of the doubled, transposed A tile
  static constexpr int kABufFloats = BK * kAStride;
  static constexpr int kBStageFloats = BK * BN;
  static constexpr uint32_t kBStageBytes = kBStageFloats * 4;
  static constexpr int kAVec = BM * BK / (4 * NT);  // 128-bit A loads per thread per k-tile
  static constexpr int kOutVec = kTM * kTN / 4;     // float4 partial values per thread
  static constexpr size_t kBOff = 0;
  static constexpr size_t kAOff = S * size_t(kBStageBytes);
  static constexpr size_t kBarOff = kAOff + 2 * size_t(kABufFloats) * 4;
  static constexpr size_t kFlagOff = kBarOff + S * 8;
  static constexpr size_t kSmem = kFlagOff + 16;
  static_assert(NT % BM == 0 && (NT / BM) * kAVec * 4 == BK, "A load split must cover the tile");
  static_assert(BN <= 256 && BK <= 256, "TMA box dimensions are at most 256");
  static_assert((S & (S - 1)) == 0, "stage count must be a power of two");
};

using CfgLarge = TileCfg<4, 2, 16, 4, 1>;  // 128 x 256 tile, 256 threads, 1 CTA / SM
using CfgSmall = TileCfg<4, 1, 8, 8, 2>;   // 128 x 128 tile, 128 threads, 2 CTAs / SM

// Maps a linear tile index to (tile row, tile column) in groups of `group_m`
// tile rows, so that CTAs running together share panels of A and B in L2
// ("Beyond Kernel 7", section "A plausible optimization that didn't improve
// runtime": block swizzling with eight block-rows per group).
__device__ __forceinline__ void tile_coords(const Sched& sc, int tile, int& tm, int& tn) {
  const int per_group = sc.group_m * sc.tiles_n;
  const int g = tile / per_group;
  const int first = g * sc.group_m;
  const int rows = min(sc.tiles_m - first, sc.group_m);
  const int r = tile - g * per_group;
  tm = first + r % rows;
  tn = r / rows;
}

// CTA that owns iteration `i` of the Stream-K iteration stream.
__device__ __forceinline__ int sk_owner(const Sched& sc, int64_t i) {
  const int64_t big = int64_t(sc.sk_extra) * (sc.sk_base + 1);
  if (i < big) return int(i / (sc.sk_base + 1));
  return sc.sk_extra + int((i - big) / sc.sk_base);
}

template <class T>
__global__ void __launch_bounds__(T::NT, T::kMinCtas)
    tile_kernel(const __grid_constant__ CUtensorMap tmap_b, const GemmArgs args, const Sched sc) {
  extern __shared__ __align__(1024) unsigned char smem[];
  float* sB = reinterpret_cast<float*>(smem + T::kBOff);
  float* sA = reinterpret_cast<float*>(smem + T::kAOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + T::kBarOff);
  int& s_last = *reinterpret_cast<int*>(smem + T::kFlagOff);

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int tr = lane / T::kTC, tc = lane % T::kTC;
  const int wm = warp % T::kWarpsM, wn = warp / T::kWarpsM;
  // Compute-side shared-memory offsets (floats).
  const int a_frag = 2 * wm * T::kWarpM + 4 * tr;  // + 16 g + kAStride kk
  const int b_frag = wn * T::kWarpN + 4 * tc;      // + 32 h + BN kk
  // Load-side assignment for A: one row, kAVec consecutive 4-wide k groups.
  const int a_row = tid % T::BM;
  const int a_q0 = (tid / T::BM) * T::kAVec;

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < T::S; ++s) dev::mbar_init(&full[s], 1);
    dev::mbar_init_fence();
    dev::tma_prefetch_desc(&tmap_b);
  }
  __syncthreads();

  const int M = args.M, N = args.N, K = args.K;
  const int cta = blockIdx.x, ctas = gridDim.x;
  uint32_t it = 0;  // k-tiles this CTA has consumed: position in the stage ring

  // Work list of this CTA: whole tiles first, then its Stream-K iterations.
  int dp_next = cta;
  int64_t sk_pos = 0, sk_end = 0;
  if (sc.sk_tiles > 0 && cta < sc.sk_ctas) {
    sk_pos = int64_t(cta) * sc.sk_base + min(cta, sc.sk_extra);
    sk_end = sk_pos + sc.sk_base + (cta < sc.sk_extra ? 1 : 0);
  }

  for (;;) {
    int tile, kb, ke, t_sk = -1;
    if (dp_next < sc.dp_tiles) {
      tile = dp_next;
      kb = 0;
      ke = sc.iters_per_tile;
      dp_next += ctas;
    } else if (sk_pos < sk_end) {
      t_sk = int(sk_pos / sc.iters_per_tile);
      const int64_t tile_start = int64_t(t_sk) * sc.iters_per_tile;
      kb = int(sk_pos - tile_start);
      const int64_t left = sk_end - tile_start;
      ke = left < sc.iters_per_tile ? int(left) : sc.iters_per_tile;
      tile = sc.dp_tiles + t_sk;
      sk_pos = tile_start + ke;
    } else {
      break;
    }
    int tm, tn;
    tile_coords(sc, tile, tm, tn);
    const int m0 = tm * T::BM, n0 = tn * T::BN;
    const int nk = ke - kb;

    float2 acc[T::kTM][T::kTN / 2];
#pragma unroll
    for (int r = 0; r < T::kTM; ++r)
#pragma unroll
      for (int q = 0; q < T::kTN / 2; ++q) acc[r][q] = make_float2(0.f, 0.f);

    // ---- prologue: fill the B ring, stage the first A tile
    if (tid == 0) {
      for (int j = 0; j < T::S && j < nk; ++j) {
        const uint32_t st = (it + j) & (T::S - 1);
        dev::mbar_arrive_expect_tx(&full[st], T::kBStageBytes);
        dev::tma_load_2d(sB + st * T::kBStageFloats, &tmap_b, n0, (kb + j) * T::BK, &full[st]);
      }
    }
    const int a_grow = m0 + a_row;
    const bool a_row_ok = a_grow < M;
    const float* a_src = args.A + int64_t(a_row_ok ? a_grow : 0) * args.lda + a_q0 * 4;
    float4 areg[T::kAVec];
    auto load_a = [&](int kt) {
      const int k0 = kt * T::BK + a_q0 * 4;
#pragma unroll
      for (int v = 0; v < T::kAVec; ++v) {
        const int k = k0 + 4 * v;
        const float* p = a_src + int64_t(kt) * T::BK + 4 * v;
        if (a_row_ok && k + 4 <= K) {
          areg[v] = __ldg(reinterpret_cast<const float4*>(p));
        } else {
          areg[v].x = (a_row_ok && k + 0 < K) ? __ldg(p + 0) : 0.f;
          areg[v].y = (a_row_ok && k + 1 < K) ? __ldg(p + 1) : 0.f;
          areg[v].z = (a_row_ok && k + 2 < K) ? __ldg(p + 2) : 0.f;
          areg[v].w = (a_row_ok && k + 3 < K) ? __ldg(p + 3) : 0.f;
        }
      }
    };
    auto store_a = [&](int buf) {
      float* dst = sA + buf * T::kABufFloats + 2 * a_row;
#pragma unroll
      for (int v = 0; v < T::kAVec; ++v) {
        const int kl = (a_q0 + v) * 4;
        *reinterpret_cast<float2*>(dst + (kl + 0) * T::kAStride) = make_float2(areg[v].x, areg[v].x);
        *reinterpret_cast<float2*>(dst + (kl + 1) * T::kAStride) = make_float2(areg[v].y, areg[v].y);
        *reinterpret_cast<float2*>(dst + (kl + 2) * T::kAStride) = make_float2(areg[v].z, areg[v].z);
        *reinterpret_cast<float2*>(dst + (kl + 3) * T::kAStride) = make_float2(areg[v].w, areg[v].w);
      }
    };
    load_a(kb);
    store_a(0);
    __syncthreads();

    // ---- main loop over the k-tiles of this work unit
    for (int j = 0; j < nk; ++j) {
      const bool more = j + 1 < nk;
      if (more) load_a(kb + j + 1);
      const uint32_t pos = it + j;
      const uint32_t st = pos & (T::S - 1);
      const bool ok = dev::mbar_wait(&full[st], (pos / T::S) & 1u, args.wait_limit_ns);
      const float* a_buf = sA + (j & 1) * T::kABufFloats + a_frag;
      const float* b_buf = sB + st * T::kBStageFloats + b_frag;
#pragma unroll
      for (int kk = 0; kk < T::BK; ++kk) {
        float4 a4[T::kTM / 2], b4[T::kTN / 4];
#pragma unroll
        for (int g = 0; g < T::kTM / 2; ++g)
          a4[g] = *reinterpret_cast<const float4*>(a_buf + kk * T::kAStride + 16 * g);
#pragma unroll
        for (int h = 0; h < T::kTN / 4; ++h)
          b4[h] = *reinterpret_cast<const float4*>(b_buf + kk * T::BN + 32 * h);
#pragma unroll
        for (int g = 0; g < T::kTM / 2; ++g) {
          const float2 a_lo = make_float2(a4[g].x, a4[g].y);  // (a[m], a[m])
          const float2 a_hi = make_float2(a4[g].z, a4[g].w);  // (a[m+1], a[m+1])
#pragma unroll
          for (int h = 0; h < T::kTN / 4; ++h) {
            const float2 b_lo = make_float2(b4[h].x, b4[h].y);
            const float2 b_hi = make_float2(b4[h].z, b4[h].w);
            dev::ffma2(acc[2 * g][2 * h], a_lo, b_lo);
            dev::ffma2(acc[2 * g][2 * h + 1], a_lo, b_hi);
            dev::ffma2(acc[2 * g + 1][2 * h], a_hi, b_lo);
            dev::ffma2(acc[2 * g + 1][2 * h + 1], a_hi, b_hi);
          }
        }
      }
      if (more) store_a((j + 1) & 1);
      if (__syncthreads_or(!ok)) {
        // A stage never landed: record the timeout, let the copies still in
        // flight finish (bounded) so none lands after the CTA has exited.
        if (tid == 0) {
          for (int jj = j; jj < nk && jj < j + T::S; ++jj) {
            const uint32_t p2 = it + jj;
            dev::mbar_wait(&full[p2 & (T::S - 1)], (p2 / T::S) & 1u, args.wait_limit_ns);
          }
          dev::record_status(args.status, kStatusTimeout, kWaitTileStage);
        }
        return;
      }
      if (tid == 0 && j + T::S < nk) {
        dev::mbar_arrive_expect_tx(&full[st], T::kBStageBytes);
        dev::tma_load_2d(sB + st * T::kBStageFloats, &tmap_b, n0, (kb + j + T::S) * T::BK,
                         &full[st]);
      }
    }
    it += nk;

    // ---- epilogue
    // Thread value j (0..31) is the float4 of patch row r = j / 4, column quad h = j % 4.
    auto out_row = [&](int r) { return m0 + wm * T::kWarpM + (r >> 1) * (2 * T::kTR) + 2 * tr + (r & 1); };
    auto out_col = [&](int h) { return n0 + wn * T::kWarpN + h * (4 * T::kTC) + 4 * tc; };
    auto value = [&](int j) {
      const int r = j >> 2, h = j & 3;
      return make_float4(acc[r][2 * h].x, acc[r][2 * h].y, acc[r][2 * h + 1].x, acc[r][2 * h + 1].y);
    };
    auto store_c = [&](int j, float4 v) {
      const int row = out_row(j >> 2), col = out_col(j & 3);
      if (row >= M) return;
      float* p = args.C + int64_t(row) * args.ldc + col;
      if (col + 4 <= N) {
        *reinterpret_cast<float4*>(p) = v;
      } else {
        if (col + 0 < N) p[0] = v.x;
        if (col + 1 < N) p[1] = v.y;
        if (col + 2 < N) p[2] = v.z;
        if (col + 3 < N) p[3] = v.w;
      }
    };

    const bool whole = (kb == 0 && ke == sc.iters_per_tile);
    if (whole) {
      if (m0 + T::BM <= M && n0 + T::BN <= N) {
#pragma unroll
        for (int j = 0; j < T::kOutVec; ++j) {
          float* p = args.C + int64_t(out_row(j >> 2)) * args.ldc + out_col(j & 3);
          *reinterpret_cast<float4*>(p) = value(j);
        }
      } else {
#pragma unroll
        for (int j = 0; j < T::kOutVec; ++j) store_c(j, value(j));
      }
      continue;
    }

    // Split tile: publish this CTA's partial sums; the last CTA to arrive
    // adds all partials in CTA order and writes C.
    const int64_t t_first_iter = int64_t(t_sk) * sc.iters_per_tile;
    const int c_first = sk_owner(sc, t_first_iter);
    const int c_last = sk_owner(sc, t_first_iter + sc.iters_per_tile - 1);
    const int64_t tile_floats = int64_t(T::BM) * T::BN;
    {
      float4* mine = reinterpret_cast<float4*>(args.partials + (t_sk + cta) * tile_floats);
#pragma unroll
      for (int j = 0; j < T::kOutVec; ++j) __stcg(mine + j * T::NT + tid, value(j));
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const int arrived = atomicAdd(args.counters + t_sk, 1);
      s_last = (arrived == c_last - c_first) ? 1 : 0;
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
#pragma unroll
      for (int j = 0; j < T::kOutVec; ++j) {
        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int cc = c_first; cc <= c_last; ++cc) {
          float4 v;
          if (cc == cta) {
            v = value(j);
          } else {
            const float4* src = reinterpret_cast<const float4*>(args.partials + (t_sk + cc) * tile_floats);
            v = __ldcg(src + j * T::NT + tid);
          }
          if (cc == c_first) {
            sum = v;
          } else {
            sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
          }
        }
        store_c(j, sum);
      }
      if (tid == 0) args.counters[t_sk] = 0;
    }
    // The next unit's prologue rewrites shared memory only after its own barrier.
  }
}

template <class T>
int prepare() {
  if (cudaFuncSetAttribute(tile_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(T::kSmem)) != cudaSuccess)
    return -1;
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, tile_kernel<T>, T::NT, T::kSmem) !=
      cudaSuccess)
    return -1;
  return blocks;
}

template <class T>
TileShape shape_of() {
  return TileShape{T::BM, T::BN, T::BK, T::NT, T::S, T::kSmem};
}

}  // namespace

TileShape tile_shape(TileConfig cfg) {
  return cfg == kTileSmall ? shape_of<CfgSmall>() : shape_of<CfgLarge>();
}

int tile_kernel_prepare(TileConfig cfg) {
  return cfg == kTileSmall ? prepare<CfgSmall>() : prepare<CfgLarge>();
}

cudaError_t launch_tile_kernel(TileConfig cfg, const CUtensorMap& tmap_b, const GemmArgs& args,
                               const Sched& sched, int grid, cudaStream_t stream) {
  if (cfg == kTileSmall) {
    tile_kernel<CfgSmall><<<grid, CfgSmall::NT, CfgSmall::kSmem, stream>>>(tmap_b, args, sched);
  } else {
    tile_kernel<CfgLarge><<<grid, CfgLarge::NT, CfgLarge::kSmem, stream>>>(tmap_b, args, sched);
  }
  return cudaGetLastError();
}

}  // namespace gb300
