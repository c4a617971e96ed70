// sgemm_tf32.cu -- opt-in TF32 tensor-core GEMM for sm_103a (tcgen05).
//
// C = A * B with the products formed by the 5th-generation tensor cores in
// TF32 (inputs keep FP32's exponent and 10 fraction bits) and accumulated in
// FP32.  This is a separate mode with its own, looser tolerance: TF32 is the
// different-numerics tensor path the pages name ("Beyond Kernel 7", section
// "The operation: GEMM and the precision of the comparison"; "cuSgemm",
// Kernel 7 uses mma.sync m16n8k4 TF32 on sm_120).  It never stands in for the
// FP32 FFMA path.
//
// Structure: a persistent grid of one CTA per SM walks the same work
// decomposition as the FFMA kernel (Sched: whole 128 x 256 tiles in full
// waves, the tiles of the last partial wave split over K, Stream-K), each
// CTA its Stream-K share first (SkFirstIter).
//  * A reaches shared memory by TMA in the canonical K-major layout with the
//    128-byte swizzle that tcgen05.mma reads through its shared-memory
//    descriptors.  B, row-major (N contiguous), is read as an MN-major
//    operand: a 32-deep k-slice of its 256 columns arrives as eight 32 x 32
//    boxes (128 bytes of N by 32 rows of k, 128-byte swizzle of 32-byte
//    atoms) 4 KB apart.  Only a B that TMA cannot read in place (a
//    misaligned base or a row stride that is not a multiple of 4) is first
//    rewritten K-major (transpose_kernel) and read like A.
//  * warp 0 (one lane) streams the CTA's k-slices of A (128 x 32) and B
//    (256 x 32) into a 4-stage ring (full / empty mbarriers);
//  * warp 1 allocates 512 TMEM columns (two 128 x 256 FP32 accumulators) and
//    one lane issues tcgen05.mma.cta_group::1.kind::tf32 (M = 128, N = 256,
//    K = 8, four per k-slice) into accumulator u mod 2 for the CTA's u-th
//    unit, releasing stages with tcgen05.commit;
//  * warps 2-5 read each finished accumulator with tcgen05.ld (each warp its
//    32-lane quarter, i.e. 32 rows of C) while the MMAs of the next unit run
//    into the other one, and store C; a split tile's sharers publish their
//    partial sums and the last to arrive adds them in CTA order.
#include <cuda.h>
#include <cuda_runtime.h>

#include "sgemm_device.cuh"
#include "sgemm_internal.h"
#include "sgemm_sched.cuh"

namespace gb300 {
namespace {

// The TF32 kernels walk each CTA's (or CTA pair's) Stream-K share before its
// whole tiles.  The epilogue warps then publish and add the split tiles'
// partial sums while the tensor core computes whole tiles into the other
// accumulator.  Walked last, as the FFMA kernel does, the share leaves its
// reductions (latency-bound reads of the other sharers' partials) exposed
// after the last MMA; walked first, only one whole tile's store is.
struct SkFirstIter {
  WorkIter w;
  int dp_first;
  bool sk_phase;

  __device__ __forceinline__ void init(const Sched& sc, int cta) {
    w.init(sc, cta);
    dp_first = w.dp_next;
    w.dp_next = sc.dp_tiles;  // no whole tile until the share is done
    sk_phase = true;
  }
  __device__ __forceinline__ bool next(const Sched& sc, int ctas, Unit& u) {
    if (sk_phase) {
      if (w.next(sc, ctas, u)) return true;
      sk_phase = false;
      w.dp_next = dp_first;  // the share is exhausted: whole tiles only from here
    }
    return w.next(sc, ctas, u);
  }
};

// KCursor over SkFirstIter: the k-tiles of all units in that order.
struct SkFirstCursor {
  SkFirstIter w;
  Unit u;
  int j;
  int tm, tn;
  bool valid;

  __device__ __forceinline__ void init(const Sched& sc, int cta, int ctas) {
    w.init(sc, cta);
    j = 0;
    valid = w.next(sc, ctas, u);
    if (valid) tile_coords(sc, u.tile, tm, tn);
  }
  __device__ __forceinline__ void advance(const Sched& sc, int ctas) {
    if (++j >= u.ke - u.kb) {
      j = 0;
      valid = w.next(sc, ctas, u);
      if (valid) tile_coords(sc, u.tile, tm, tn);
    }
  }
};

constexpr int kTfBM = 128, kTfBN = 256, kTfBK = 32, kTfStages = 4, kTfThreads = 192;
constexpr uint32_t kTfAStageBytes = kTfBM * kTfBK * 4;  // 16 KB
constexpr uint32_t kTfBStageBytes = kTfBN * kTfBK * 4;  // 32 KB
constexpr uint32_t kTfTmemCols = 2 * kTfBN;             // two accumulators of 128 lanes x 256 FP32
constexpr int kTfEpiWarps = 4;                          // warps 2..5
constexpr int kTfEpiThreads = 32 * kTfEpiWarps;
constexpr int kTfBarriers = 2 * kTfStages + 5;          // full, empty, acc_full[2], acc_empty[2], drain
constexpr uint32_t kTfStagingBytes = kTfEpiWarps * 2 * 4096;  // CStager buffers of the epilogue warps
constexpr size_t kTfSmem = 1024 /* alignment slack */ + kTfStages * size_t(kTfAStageBytes + kTfBStageBytes) +
                           kTfStagingBytes + kTfBarriers * 8 + 16;
static_assert(kTfSmem <= 232448, "shared memory per CTA");
constexpr uint32_t kStatusTimeout = 3;

// Instruction descriptor of tcgen05.mma kind::tf32: FP32 accumulator, TF32 A
// and B, A K-major, B K-major (b_mn = 0) or MN-major (b_mn = 1), M = 128,
// N = 256.
__host__ __device__ constexpr uint32_t tf_idesc(uint32_t b_mn) {
  return (1u << 4)                  // D format: F32
         | (2u << 7)                // A format: TF32
         | (2u << 10)               // B format: TF32
         | (0u << 15) | (b_mn << 16)  // A K-major; B K- or MN-major
         | (uint32_t(kTfBN >> 3) << 17) | (uint32_t(kTfBM >> 4) << 24);
}
// B as an MN-major operand: 32-column (128-byte) chunks of N, one TMA box each.
constexpr int kTfBChunk = 32;
constexpr uint32_t kTfBChunkBytes = kTfBChunk * kTfBK * 4;  // 4 KB: 32 rows of k x 128 bytes

// Shared-memory matrix descriptor for a K-major operand stored as rows of 128
// bytes with the 128-byte swizzle: 8-row core groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= uint64_t((smem_addr & 0x3FFFFu) >> 4);  // start address
  d |= uint64_t(16 >> 4) << 16;                // leading byte offset (unused when swizzled)
  d |= uint64_t(1024 >> 4) << 32;              // stride byte offset between 8-row groups
  d |= uint64_t(1) << 46;                      // descriptor version for sm_100 family
  d |= uint64_t(2) << 61;                      // layout: 128-byte swizzle
  return d;
}

// Shared-memory matrix descriptor for an MN-major TF32 operand stored as
// 128-byte (32-element) chunks of MN, each chunk 32 rows of k, with the
// 128-byte swizzle of 32-byte atoms (TMA's SWIZZLE_128B_ATOM_32B; 4-row
// period).  TF32 in MN-major form takes this swizzle: with the plain 128-byte
// one the tensor core produced zeros on GB300.  The leading byte offset steps
// to the next MN chunk (4 KB), the stride byte offset to the next 4-row group
// of k (512 bytes), so one K = 8 instruction reads two groups.  Established
// on GB300 by multiplying A[m][k] = (k == m mod 8) with B[k][n] = 256 k + n,
// which shows which B element meets each (k, n).
__device__ __forceinline__ uint64_t sw128a32_mnmajor_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= uint64_t((smem_addr & 0x3FFFFu) >> 4);  // start address
  d |= uint64_t(kTfBChunkBytes >> 4) << 16;    // leading byte offset: next MN chunk
  d |= uint64_t(512 >> 4) << 32;               // stride byte offset: next 4 rows of k
  d |= uint64_t(1) << 46;                      // descriptor version for sm_100 family
  d |= uint64_t(1) << 61;                      // layout: 128-byte swizzle, 32-byte atoms
  return d;
}

template <uint32_t kIdesc>
__device__ __forceinline__ void tc_mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "n"(kIdesc), "r"(accumulate)
      : "memory");
}

// Arrives on `bar` once every tcgen05 operation this thread issued so far completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   dev::smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Stores 32 consecutive values of row `row` of C from column `col` on.
__device__ __forceinline__ void store_row32(const Tf32Args& args, int row, int col,
                                            const float (&v)[32]) {
  if (row >= args.M) return;
  float* dst = args.C + int64_t(row) * args.ldc + col;
  if (col + 32 <= args.N && !args.c_scalar) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      reinterpret_cast<float4*>(dst)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (col + i < args.N) dst[i] = v[i];
  }
}

// Stores the box at element coordinates (x = column, y = row) of a 2-D tensor
// map from shared memory as one bulk group of this thread.  Elements outside
// the tensor are not written.  x must be a multiple of 4.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int32_t x, int32_t y,
                                             const void* src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(dev::smem_addr(src))
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// One epilogue warp's stores of C through shared memory: a 32 x 32 block
// (row = lane) goes to one of two 4 KB buffers in the 128-byte swizzle that
// TMA reads (16-byte chunk j of row r at j ^ (r mod 8), so the warp's
// writes are free of bank conflicts), then out with one TMA store.  Every
// 128-byte line of C is written whole, where row-per-lane stores would touch
// 32 lines per instruction.
struct CStager {
  unsigned char* buf;  // two 4 KB buffers, 1024-byte aligned
  uint32_t n;          // blocks stored so far

  __device__ __forceinline__ void put(const CUtensorMap* map, int x, int y, const float (&v)[32],
                                      int lane) {
    unsigned char* b = buf + (n & 1u) * 4096u;
    // The store that used this buffer two blocks ago has finished reading it.
    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
    __syncwarp();
    float4* row = reinterpret_cast<float4*>(b + lane * 128);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      row[i ^ (lane & 7)] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    dev::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) tma_store_2d(map, x, y, b);
    ++n;
  }
  // Every store issued has completed (before shared memory is released).
  __device__ __forceinline__ void drain(int lane) const {
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
  }
};

// B_MN: B is read in place as an MN-major operand (tmap_b: B, N fastest, box
// 32 x 32); otherwise tmap_b holds B^T (K fastest, box 32 x 256) like A.
template <bool B_MN>
__global__ void __launch_bounds__(kTfThreads, 1)
    tf32_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                const __grid_constant__ CUtensorMap tmap_c, const Tf32Args args, const Sched sc) {
  extern __shared__ unsigned char smem_raw[];
  // Stages must sit on 1024-byte boundaries (the 128-byte swizzle period).
  const uint32_t raw = dev::smem_addr(smem_raw);
  unsigned char* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  unsigned char* sA = smem;
  unsigned char* sB = smem + kTfStages * kTfAStageBytes;
  unsigned char* sC = sB + kTfStages * kTfBStageBytes;  // epilogue staging (1024-byte aligned)
  uint64_t* full = reinterpret_cast<uint64_t*>(sC + kTfStagingBytes);
  uint64_t* empty = full + kTfStages;
  uint64_t* acc_full = empty + kTfStages;  // [2] accumulator b holds a finished unit
  uint64_t* acc_empty = acc_full + 2;      // [2] the epilogue has read accumulator b
  uint64_t* drain = acc_empty + 2;         // every MMA this CTA issued has completed
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(drain + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(drain + 1) + 1;
  int* s_last = reinterpret_cast<int*>(drain + 1) + 2;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x, ctas = gridDim.x;
  const uint64_t limit = args.wait_limit_ns;

  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dev::smem_addr(const_cast<uint32_t*>(tmem_slot))),
                 "r"(kTfTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTfStages; ++s) {
      dev::mbar_init(&full[s], 1);
      dev::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      dev::mbar_init(&acc_full[b], 1);
      dev::mbar_init(&acc_empty[b], kTfEpiWarps);  // one arrival per epilogue warp
    }
    dev::mbar_init(drain, 1);
    *s_abort = 0;
    dev::mbar_init_fence();
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  // A wait that failed: record it once and make every later wait give up at
  // once, so that all roles run to their end without waiting.
  auto fail = [&]() {
    if (!*s_abort) {
      *s_abort = 1;
      dev::record_status(args.status, kStatusTimeout, kWaitTileStage);
    }
  };

  if (warp == 0) {
    // ---- TMA producer: the CTA's k-slices, unit after unit.  The whole warp
    // walks the schedule and waits; one elected lane issues the copies.
    if (dev::elect_one()) {
      dev::tma_prefetch_desc(&tmap_a);
      dev::tma_prefetch_desc(&tmap_b);
    }
    SkFirstCursor c;
    c.init(sc, cta, ctas);
    uint32_t i = 0;
    for (; c.valid; ++i, c.advance(sc, ctas)) {
      const uint32_t s = i % kTfStages, n = i / kTfStages;
      if (n > 0 && !dev::mbar_wait_abortable(&empty[s], (n - 1) & 1u, limit, s_abort)) fail();
      if (*s_abort) break;
      const int k0 = (c.u.kb + c.j) * kTfBK, m0 = c.tm * kTfBM, n0 = c.tn * kTfBN;
      if (dev::elect_one()) {
        dev::mbar_arrive_expect_tx(&full[s], kTfAStageBytes + kTfBStageBytes);
        dev::tma_load_2d(sA + s * kTfAStageBytes, &tmap_a, k0, m0, &full[s]);
        if constexpr (B_MN) {
#pragma unroll
          for (int j = 0; j < kTfBN / kTfBChunk; ++j)
            dev::tma_load_2d(sB + s * kTfBStageBytes + j * kTfBChunkBytes, &tmap_b,
                             n0 + j * kTfBChunk, k0, &full[s]);
        } else {
          dev::tma_load_2d(sB + s * kTfBStageBytes, &tmap_b, k0, n0, &full[s]);
        }
      }
      __syncwarp();
    }
    // After a failure, let the copies already issued land (bounded) before
    // the CTA's shared memory is released.
    if (*s_abort)
      for (uint32_t k = (i > kTfStages ? i - kTfStages : 0); k < i; ++k)
        dev::mbar_wait(&full[k % kTfStages], (k / kTfStages) & 1u, limit);
  } else if (warp == 1) {
    // ---- MMA issuer: unit u accumulates into TMEM columns [256 (u mod 2), +256).
    // The whole warp walks the schedule and waits; one elected lane issues.
    SkFirstIter w;
    w.init(sc, cta);
    Unit u;
    uint32_t it = 0, ui = 0;
    while (w.next(sc, ctas, u)) {
      const uint32_t b = ui & 1u, nb = ui >> 1;
      if (nb > 0 && !dev::mbar_wait_abortable(&acc_empty[b], (nb - 1) & 1u, limit, s_abort))
        fail();
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t d = tmem + b * kTfBN;
      const int nk = u.ke - u.kb;
      for (int j = 0; j < nk; ++j, ++it) {
        const uint32_t s = it % kTfStages;
        if (!dev::mbar_wait_abortable(&full[s], (it / kTfStages) & 1u, limit, s_abort)) fail();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (dev::elect_one()) {
          if (!*s_abort) {
            const uint64_t a_desc = sw128_kmajor_desc(dev::smem_addr(sA + s * kTfAStageBytes));
            const uint32_t b_addr = dev::smem_addr(sB + s * kTfBStageBytes);
            const uint64_t b_desc =
                B_MN ? sw128a32_mnmajor_desc(b_addr) : sw128_kmajor_desc(b_addr);
            // K = 8 TF32 per instruction: 32 bytes along a K-major row, or 8
            // rows (1 KB) of an MN-major chunk.  Descriptor addresses are in
            // 16-byte units.
            constexpr uint64_t kBStep = B_MN ? 1024 / 16 : 32 / 16;
#pragma unroll
            for (int k = 0; k < kTfBK / 8; ++k)
              tc_mma_tf32<tf_idesc(B_MN ? 1u : 0u)>(d, a_desc + 2 * k, b_desc + kBStep * k,
                                                    (j | k) != 0 ? 1u : 0u);
          }
          tc_commit(&empty[s]);  // the stage is free once these MMAs have read it
        }
        __syncwarp();
      }
      if (dev::elect_one()) tc_commit(&acc_full[b]);  // the unit's accumulator is final
      __syncwarp();
      ++ui;
    }
    if (dev::elect_one()) tc_commit(drain);
    __syncwarp();
    dev::mbar_wait(drain, 0u, limit);  // nothing of this CTA is left in the tensor pipe
  } else {
    // ---- epilogue: warps 2..5 own TMEM lane quarters (warp % 4), 32 rows each
    const int q = warp & 3;
    const int row_local = 32 * q + lane;
    const int etid = threadIdx.x - 64;  // 0..127
    constexpr int64_t kSlotVec = int64_t(kTfBM) * kTfBN / 4;
    // C through shared memory and TMA where TMA can address it (CStager;
    // the block over a right edge that is not 16-byte aligned row by row).
    const bool tma_c = !args.c_scalar;
    const bool tma_edge = (args.N & 3) == 0;
    CStager stager{sC + q * 8192, 0};
    if (tma_c && lane == 0) dev::tma_prefetch_desc(&tmap_c);
    SkFirstIter w;
    w.init(sc, cta);
    Unit u;
    uint32_t ui = 0;
    while (w.next(sc, ctas, u)) {
      const uint32_t b = ui & 1u, nb = ui >> 1;
      if (!dev::mbar_wait_abortable(&acc_full[b], nb & 1u, limit, s_abort)) fail();
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      int tm, tn;
      tile_coords(sc, u.tile, tm, tn);
      const int row = tm * kTfBM + row_local, n0 = tn * kTfBN;
      const uint32_t taddr = tmem + b * kTfBN + (uint32_t(32 * q) << 16);
      const bool ok = __shfl_sync(0xffffffffu, !*s_abort ? 1 : 0, 0) != 0;  // warp-uniform
      // Row `row`, columns col .. col + 31 of C.
      auto emit = [&](int col, const float(&v)[32]) {
        if (tma_c && (tma_edge || col + 32 <= args.N))
          stager.put(&tmap_c, col, row - lane, v, lane);
        else
          store_row32(args, row, col, v);
      };
      if (u.t_sk < 0 || (u.kb == 0 && u.ke == sc.iters_per_tile)) {
#pragma unroll 1
        for (int c = 0; c < kTfBN; c += 32) {
          uint32_t r[32];
          tc_ld32(taddr + uint32_t(c), r);
          if (ok) emit(n0 + c, reinterpret_cast<const float(&)[32]>(r));
        }
      } else {
        // Split tile, as in the FFMA kernel: the sharers publish their partial
        // sums (float4 j of row r at j * 128 + r, coalesced across a warp) and
        // the last to arrive adds all of them in CTA order.  The owner of the
        // tile's first k-slices keeps its partial in TMEM: when every other
        // sharer has already arrived it is the last and publishes nothing.
        // All four epilogue warps take the same path through the named
        // barriers below, also after a timeout (whose output is invalid).
        const int64_t t_first_iter = int64_t(u.t_sk) * sc.iters_per_tile;
        const int c_first = sk_owner(sc, t_first_iter);
        const int c_last = sk_owner(sc, t_first_iter + sc.iters_per_tile - 1);
        const int others = c_last - c_first;
        const bool own_first = cta == c_first && !args.owner_publishes;
        bool last = false;
        if (own_first) {
          if (etid == 0) *s_last = dev::ld_acquire_gpu(args.counters + u.t_sk) == others ? 1 : 0;
          dev::named_barrier(1, kTfEpiThreads);
          last = *s_last != 0;
          dev::named_barrier(1, kTfEpiThreads);
        }
        if (!last) {
          float4* mine = reinterpret_cast<float4*>(args.partials) + (u.t_sk + cta) * kSlotVec + row_local;
#pragma unroll 1
          for (int c = 0; c < kTfBN; c += 32) {
            uint32_t r[32];
            tc_ld32(taddr + uint32_t(c), r);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              __stcg(mine + (c / 4 + v) * kTfBM,
                     make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                 __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3])));
          }
          // One thread releases the partial (cumulative fence after the
          // barrier); its second fence orders a last arriver's reads.
          dev::named_barrier(1, kTfEpiThreads);
          if (etid == 0) {
            __threadfence();
            *s_last = atomicAdd(args.counters + u.t_sk, 1) == others ? 1 : 0;
            __threadfence();
          }
          dev::named_barrier(1, kTfEpiThreads);
          last = *s_last != 0;
          dev::named_barrier(1, kTfEpiThreads);  // s_last may be rewritten by the next split tile
        }
        if (last) {
          const float4* base = reinterpret_cast<const float4*>(args.partials) + row_local;
          // 64 columns per step: every slot's 16 loads of a step are in flight together.
#pragma unroll 1
          for (int c = 0; c < kTfBN; c += 64) {
            float sum[64];
            if (own_first) {
              uint32_t r[32];
              tc_ld32(taddr + uint32_t(c), r);
#pragma unroll
              for (int i = 0; i < 32; ++i) sum[i] = __uint_as_float(r[i]);
              tc_ld32(taddr + uint32_t(c + 32), r);
#pragma unroll
              for (int i = 0; i < 32; ++i) sum[32 + i] = __uint_as_float(r[i]);
            } else {
              const float4* src = base + (u.t_sk + c_first) * kSlotVec + (c / 4) * kTfBM;
#pragma unroll
              for (int v = 0; v < 16; ++v) {
                const float4 x = __ldcg(src + v * kTfBM);
                sum[4 * v] = x.x;
                sum[4 * v + 1] = x.y;
                sum[4 * v + 2] = x.z;
                sum[4 * v + 3] = x.w;
              }
            }
#pragma unroll 1
            for (int cc = c_first + 1; cc <= c_last; ++cc) {
              const float4* src = base + (u.t_sk + cc) * kSlotVec + (c / 4) * kTfBM;
              float4 x[16];
#pragma unroll
              for (int v = 0; v < 16; ++v) x[v] = __ldcg(src + v * kTfBM);
#pragma unroll
              for (int v = 0; v < 16; ++v) {
                sum[4 * v] += x[v].x;
                sum[4 * v + 1] += x[v].y;
                sum[4 * v + 2] += x[v].z;
                sum[4 * v + 3] += x[v].w;
              }
            }
            emit(n0 + c, reinterpret_cast<const float(&)[32]>(sum[0]));
            emit(n0 + c + 32, reinterpret_cast<const float(&)[32]>(sum[32]));
          }
          if (etid == 0) args.counters[u.t_sk] = 0;
        }
      }
      // The accumulator may be overwritten by the unit after next.
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(&acc_empty[b]);
      ++ui;
    }
    if (tma_c) stager.drain(lane);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTfTmemCols)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// CTA-pair kernel: tcgen05.mma.cta_group::2 over 256 x 256 tiles.
//
// A cluster of two CTAs on two SMs computes one 256 x 256 tile.  Each CTA
// stages its own 128 rows of A and its own 128 columns of B per 32-deep
// k-slice (32 KB, so six stages fit); the even CTA (the leader) issues the
// M = 256, N = 256 MMAs, which read both CTAs' shared memory at the same
// offsets and leave rows [128 r, 128 r + 128) of the tile in the TMEM of CTA
// r.  Both CTAs' copies complete on the leader's full barrier; the leader's
// commits are multicast to the barriers of both CTAs; each CTA's epilogue
// reads its own TMEM and tells the leader, across the cluster, when the
// accumulator may be reused.  The work decomposition runs over CTA pairs.
constexpr int kPrBM = 256, kPrBN = 256, kPrBK = 32, kPrStages = 6;
constexpr int kPrRows = kPrBM / 2, kPrCols = kPrBN / 2;      // per CTA
constexpr uint32_t kPrAStageBytes = kPrRows * kPrBK * 4;    // 16 KB
constexpr uint32_t kPrBStageBytes = kPrCols * kPrBK * 4;    // 16 KB
// Two 256-column accumulators per CTA.  Both CTAs execute the cta_group::2
// allocation and receive the same address (measured on GB300).
constexpr uint32_t kPrTmemCols = 512;
constexpr int kPrAccBufs = int(kPrTmemCols / kPrBN);          // accumulators per CTA
constexpr int kPrBarriers = 2 * kPrStages + 2 * 2 + 1;
constexpr uint32_t kPrStagingBytes = kTfEpiWarps * 2 * 4096;  // CStager buffers of the epilogue warps
constexpr size_t kPrSmem = 1024 + kPrStages * size_t(kPrAStageBytes + kPrBStageBytes) +
                           kPrStagingBytes + kPrBarriers * 8 + 16;
static_assert(kPrSmem <= 232448, "shared memory per CTA");

__host__ __device__ constexpr uint32_t pr_idesc(uint32_t b_mn) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (0u << 15) | (b_mn << 16) |
         (uint32_t(kPrBN >> 3) << 17) | (uint32_t(kPrBM >> 4) << 24);
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of this CTA's shared-memory location `p` in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(dev::smem_addr(p)), "r"(rank));
  return d;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ void pr_tma_load(void* dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint32_t bar_cluster_addr) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dev::smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster_addr)
      : "memory");
}

template <uint32_t kIdesc>
__device__ __forceinline__ void pr_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "n"(kIdesc), "r"(accumulate)
      : "memory");
}

// Arrives on the barrier at `bar`'s offset in both CTAs of the pair once every
// tcgen05 operation this thread issued so far completed.
__device__ __forceinline__ void pr_commit_both(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(dev::smem_addr(bar)),
      "h"(uint16_t(3))
      : "memory");
}

__device__ __forceinline__ void pr_commit_own(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   dev::smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void remote_arrive(uint32_t bar_cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster_addr)
               : "memory");
}

template <bool B_MN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kTfThreads, 1)
    tf32_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                     const __grid_constant__ CUtensorMap tmap_c, const Tf32Args args, const Sched sc) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = dev::smem_addr(smem_raw);
  unsigned char* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  unsigned char* sA = smem;
  unsigned char* sB = smem + kPrStages * kPrAStageBytes;
  unsigned char* sC = sB + kPrStages * kPrBStageBytes;  // epilogue staging (1024-byte aligned)
  uint64_t* full = reinterpret_cast<uint64_t*>(sC + kPrStagingBytes);  // used in the leader
  uint64_t* empty = full + kPrStages;
  uint64_t* acc_full = empty + kPrStages;  // [2]
  uint64_t* acc_empty = acc_full + 2;      // [2], used in the leader: 4 warps x 2 CTAs arrive
  uint64_t* drain = acc_empty + 2;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(drain + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(drain + 1) + 1;
  int* s_last = reinterpret_cast<int*>(drain + 1) + 2;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, pairs = gridDim.x >> 1;
  const uint64_t limit = args.wait_limit_ns;

  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dev::smem_addr(const_cast<uint32_t*>(tmem_slot))),
                 "r"(kPrTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPrStages; ++s) {
      dev::mbar_init(&full[s], 1);
      dev::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      dev::mbar_init(&acc_full[b], 1);
      dev::mbar_init(&acc_empty[b], 2 * kTfEpiWarps);
    }
    dev::mbar_init(drain, 1);
    *s_abort = 0;
    dev::mbar_init_fence();
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  cluster_sync_all();  // the peer's barriers exist before anything signals them
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  auto fail = [&]() {
    if (!*s_abort) {
      *s_abort = 1;
      dev::record_status(args.status, kStatusTimeout, kWaitTileStage);
    }
  };

  if (warp == 0) {
    // ---- TMA producer (both CTAs): this CTA's rows of A and columns of B,
    // completing on the leader's full barrier.
    if (dev::elect_one()) {
      dev::tma_prefetch_desc(&tmap_a);
      dev::tma_prefetch_desc(&tmap_b);
    }
    SkFirstCursor c;
    c.init(sc, pair, pairs);
    uint32_t i = 0;
    for (; c.valid; ++i, c.advance(sc, pairs)) {
      const uint32_t s = i % kPrStages, n = i / kPrStages;
      if (n > 0 && !dev::mbar_wait_abortable(&empty[s], (n - 1) & 1u, limit, s_abort)) fail();
      if (*s_abort) break;
      const int k0 = (c.u.kb + c.j) * kPrBK;
      const int m0 = c.tm * kPrBM + int(rank) * kPrRows, n0 = c.tn * kPrBN + int(rank) * kPrCols;
      if (dev::elect_one()) {
        const uint32_t bar = peer_addr(&full[s], 0);
        if (leader) dev::mbar_arrive_expect_tx(&full[s], 2 * (kPrAStageBytes + kPrBStageBytes));
        pr_tma_load(sA + s * kPrAStageBytes, &tmap_a, k0, m0, bar);
        if constexpr (B_MN) {
#pragma unroll
          for (int j = 0; j < kPrCols / kTfBChunk; ++j)
            pr_tma_load(sB + s * kPrBStageBytes + j * kTfBChunkBytes, &tmap_b, n0 + j * kTfBChunk, k0,
                        bar);
        } else {
          pr_tma_load(sB + s * kPrBStageBytes, &tmap_b, k0, n0, bar);
        }
      }
      __syncwarp();
    }
    // After a failure, this CTA's last copies complete on the leader's barrier,
    // which it cannot observe: give them a bounded grace period (a copy lands
    // within microseconds) before shared memory is released.
    if (*s_abort) {
      const uint64_t t0 = dev::global_timer_ns();
      while (dev::global_timer_ns() - t0 < 100000ull) __nanosleep(1000);
    }
  } else if (warp == 1) {
    if (leader) {
      // ---- MMA issuer (leader only)
      SkFirstIter w;
      w.init(sc, pair);
      Unit u;
      uint32_t it = 0, ui = 0;
      while (w.next(sc, pairs, u)) {
        const uint32_t b = ui % kPrAccBufs, nb = ui / kPrAccBufs;
        if (nb > 0 && !dev::mbar_wait_abortable(&acc_empty[b], (nb - 1) & 1u, limit, s_abort))
          fail();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t d = tmem + b * kPrBN;
        const int nk = u.ke - u.kb;
        for (int j = 0; j < nk; ++j, ++it) {
          const uint32_t s = it % kPrStages;
          if (!dev::mbar_wait_abortable(&full[s], (it / kPrStages) & 1u, limit, s_abort)) fail();
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          if (dev::elect_one()) {
            if (!*s_abort) {
              const uint64_t a_desc = sw128_kmajor_desc(dev::smem_addr(sA + s * kPrAStageBytes));
              const uint32_t b_addr = dev::smem_addr(sB + s * kPrBStageBytes);
              const uint64_t b_desc =
                  B_MN ? sw128a32_mnmajor_desc(b_addr) : sw128_kmajor_desc(b_addr);
              constexpr uint64_t kBStep = B_MN ? 1024 / 16 : 32 / 16;
#pragma unroll
              for (int k = 0; k < kPrBK / 8; ++k)
                pr_mma<pr_idesc(B_MN ? 1u : 0u)>(d, a_desc + 2 * k, b_desc + kBStep * k,
                                                 (j | k) != 0 ? 1u : 0u);
            }
            pr_commit_both(&empty[s]);
          }
          __syncwarp();
        }
        if (dev::elect_one()) pr_commit_both(&acc_full[b]);
        __syncwarp();
        ++ui;
      }
      if (dev::elect_one()) pr_commit_own(drain);
      __syncwarp();
      dev::mbar_wait(drain, 0u, limit);
    }
  } else {
    // ---- epilogue (both CTAs): rows [128 rank, 128 rank + 128) of each tile
    const int q = warp & 3;
    const int row_local = 32 * q + lane;
    const int etid = threadIdx.x - 64;
    constexpr int64_t kHalfVec = int64_t(kPrRows) * kPrBN / 4;  // one CTA's partial, in float4
    // C aligned for TMA: stores through shared memory (CStager); otherwise
    // row by row, 4 bytes at a time.  A TMA store clips a box at the right
    // edge of C only to 16-byte granules (measured on GB300: with N not a
    // multiple of 4 it wrote the columns up to the next multiple of 4), so
    // the block holding column N - 1 of such a C is stored row by row.
    const bool tma_c = !args.c_scalar;
    const bool tma_edge = (args.N & 3) == 0;  // a TMA store may cross column N
    CStager stager{sC + q * 8192, 0};
    if (tma_c && lane == 0) dev::tma_prefetch_desc(&tmap_c);
    SkFirstIter w;
    w.init(sc, pair);
    Unit u;
    uint32_t ui = 0;
    while (w.next(sc, pairs, u)) {
      const uint32_t b = ui % kPrAccBufs, nb = ui / kPrAccBufs;
      if (!dev::mbar_wait_abortable(&acc_full[b], nb & 1u, limit, s_abort)) fail();
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      int tm, tn;
      tile_coords(sc, u.tile, tm, tn);
      const int row = tm * kPrBM + int(rank) * kPrRows + row_local, n0 = tn * kPrBN;
      const int row0 = row - lane;  // first row of this warp's 32
      const uint32_t taddr = tmem + b * kPrBN + (uint32_t(32 * q) << 16);
      const bool ok = __shfl_sync(0xffffffffu, !*s_abort ? 1 : 0, 0) != 0;  // warp-uniform
      // Row `row`, columns col .. col + 31 of C.
      auto emit = [&](int col, const float(&v)[32]) {
        if (tma_c && (tma_edge || col + 32 <= args.N))
          stager.put(&tmap_c, col, row0, v, lane);
        else
          store_row32(args, row, col, v);
      };
      if (u.t_sk < 0 || (u.kb == 0 && u.ke == sc.iters_per_tile)) {
#pragma unroll 1
        for (int c = 0; c < kPrBN; c += 32) {
          uint32_t r[32];
          tc_ld32(taddr + uint32_t(c), r);
          if (ok) emit(n0 + c, reinterpret_cast<const float(&)[32]>(r));
        }
      } else {
        // Split tile, per CTA half: counters[2 t + rank], slot 2 (t + pair) + rank.
        const int64_t t_first_iter = int64_t(u.t_sk) * sc.iters_per_tile;
        const int c_first = sk_owner(sc, t_first_iter);
        const int c_last = sk_owner(sc, t_first_iter + sc.iters_per_tile - 1);
        const int others = c_last - c_first;
        const bool own_first = pair == c_first && !args.owner_publishes;
        int32_t* counter = args.counters + 2 * u.t_sk + int(rank);
        bool last = false;
        if (own_first) {
          if (etid == 0) *s_last = dev::ld_acquire_gpu(counter) == others ? 1 : 0;
          dev::named_barrier(1, kTfEpiThreads);
          last = *s_last != 0;
          dev::named_barrier(1, kTfEpiThreads);
        }
        if (!last) {
          float4* mine = reinterpret_cast<float4*>(args.partials) +
                         (2 * (u.t_sk + pair) + int(rank)) * kHalfVec + row_local;
#pragma unroll 1
          for (int c = 0; c < kPrBN; c += 32) {
            uint32_t r[32];
            tc_ld32(taddr + uint32_t(c), r);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              __stcg(mine + (c / 4 + v) * kPrRows,
                     make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                 __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3])));
          }
          // One thread releases the partial (cumulative fence after the
          // barrier); its second fence orders a last arriver's reads.
          dev::named_barrier(1, kTfEpiThreads);
          if (etid == 0) {
            __threadfence();
            *s_last = atomicAdd(counter, 1) == others ? 1 : 0;
            __threadfence();
          }
          dev::named_barrier(1, kTfEpiThreads);
          last = *s_last != 0;
          dev::named_barrier(1, kTfEpiThreads);
        }
        if (last) {
          const float4* base = reinterpret_cast<const float4*>(args.partials) + row_local;
#pragma unroll 1
          for (int c = 0; c < kPrBN; c += 64) {
            float sum[64];
            if (own_first) {
              uint32_t r[32];
              tc_ld32(taddr + uint32_t(c), r);
#pragma unroll
              for (int k = 0; k < 32; ++k) sum[k] = __uint_as_float(r[k]);
              tc_ld32(taddr + uint32_t(c + 32), r);
#pragma unroll
              for (int k = 0; k < 32; ++k) sum[32 + k] = __uint_as_float(r[k]);
            } else {
              const float4* src =
                  base + (2 * (u.t_sk + c_first) + int(rank)) * kHalfVec + (c / 4) * kPrRows;
#pragma unroll
              for (int v = 0; v < 16; ++v) {
                const float4 x = __ldcg(src + v * kPrRows);
                sum[4 * v] = x.x;
                sum[4 * v + 1] = x.y;
                sum[4 * v + 2] = x.z;
                sum[4 * v + 3] = x.w;
              }
            }
#pragma unroll 1
            for (int cc = c_first + 1; cc <= c_last; ++cc) {
              const float4* src = base + (2 * (u.t_sk + cc) + int(rank)) * kHalfVec + (c / 4) * kPrRows;
              float4 x[16];
#pragma unroll
              for (int v = 0; v < 16; ++v) x[v] = __ldcg(src + v * kPrRows);
#pragma unroll
              for (int v = 0; v < 16; ++v) {
                sum[4 * v] += x[v].x;
                sum[4 * v + 1] += x[v].y;
                sum[4 * v + 2] += x[v].z;
                sum[4 * v + 3] += x[v].w;
              }
            }
            emit(n0 + c, reinterpret_cast<const float(&)[32]>(sum[0]));
            emit(n0 + c + 32, reinterpret_cast<const float(&)[32]>(sum[32]));
          }
          if (etid == 0) *counter = 0;
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) remote_arrive(peer_addr(&acc_empty[b], 0));
      ++ui;
    }
    if (tma_c) stager.drain(lane);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  cluster_sync_all();  // nothing of either CTA is still signalled or read by the other
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kPrTmemCols)
                 : "memory");
  }
}

// Bt[n][k] = B[k][n] through 32 x 33 shared tiles (coalesced on both sides).
__global__ void __launch_bounds__(256)
    transpose_kernel(const float* __restrict__ B, int64_t ldb, float* __restrict__ Bt,
                     int64_t ldbt, int K, int N) {
  __shared__ float tile[32][33];
  const int64_t n0 = int64_t(blockIdx.x) * 32;
  const int64_t k_tiles = (int64_t(K) + 31) / 32;
  for (int64_t ky = blockIdx.y; ky < k_tiles; ky += gridDim.y) {
    const int64_t k0 = ky * 32;
    for (int i = threadIdx.y; i < 32; i += 8) {
      const int64_t k = k0 + i, n = n0 + threadIdx.x;
      tile[i][threadIdx.x] = (k < K && n < N) ? B[k * ldb + n] : 0.f;
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += 8) {
      const int64_t n = n0 + i, k = k0 + threadIdx.x;
      if (n < N && k < K) Bt[n * ldbt + k] = tile[threadIdx.x][i];
    }
    __syncthreads();
  }
}

// Vectorized variant for 16-byte-aligned B with ldb % 4 == 0 (and Bt likewise):
// 64 x 64 tiles moved as 128-bit loads and stores.
__global__ void __launch_bounds__(256)
    transpose_vec_kernel(const float* __restrict__ B, int64_t ldb, float* __restrict__ Bt,
                         int64_t ldbt, int K, int N) {
  __shared__ float tile[64][65];
  const int64_t n0 = int64_t(blockIdx.x) * 64;
  const int64_t k_tiles = (int64_t(K) + 63) / 64;
  for (int64_t ky = blockIdx.y; ky < k_tiles; ky += gridDim.y) {
    const int64_t k0 = ky * 64;
    for (int i = threadIdx.x; i < 64 * 16; i += 256) {
      const int r = i / 16, c = 4 * (i % 16);
      const int64_t k = k0 + r, n = n0 + c;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (k < K) {
        const float* p = B + k * ldb + n;
        if (n + 3 < N) {
          v = *reinterpret_cast<const float4*>(p);
        } else {
          if (n + 0 < N) v.x = p[0];
          if (n + 1 < N) v.y = p[1];
          if (n + 2 < N) v.z = p[2];
        }
      }
      tile[r][c] = v.x;
      tile[r][c + 1] = v.y;
      tile[r][c + 2] = v.z;
      tile[r][c + 3] = v.w;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 64 * 16; i += 256) {
      const int r = i / 16, c = 4 * (i % 16);
      const int64_t n = n0 + r, k = k0 + c;
      if (n >= N) continue;
      const float4 v = make_float4(tile[c][r], tile[c + 1][r], tile[c + 2][r], tile[c + 3][r]);
      float* p = Bt + n * ldbt + k;
      if (k + 3 < K) {
        *reinterpret_cast<float4*>(p) = v;
      } else {
        if (k + 0 < K) p[0] = v.x;
        if (k + 1 < K) p[1] = v.y;
        if (k + 2 < K) p[2] = v.z;
      }
    }
    __syncthreads();
  }
}

}  // namespace

size_t tf32_smem_bytes() { return kTfSmem; }
int tf32_tile_m() { return kTfBM; }
int tf32_tile_n() { return kTfBN; }
int tf32_tile_k() { return kTfBK; }

int tf32_b_chunk() { return kTfBChunk; }

int tf32_prepare() {
  if (cudaFuncSetAttribute(tf32_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(kTfSmem)) != cudaSuccess ||
      cudaFuncSetAttribute(tf32_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(kTfSmem)) != cudaSuccess)
    return -1;
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, tf32_kernel<true>, kTfThreads,
                                                    kTfSmem) != cudaSuccess)
    return -1;
  return blocks;
}

cudaError_t launch_transpose(const float* B, int64_t ldb, float* Bt, int64_t ldbt, int K, int N,
                             cudaStream_t stream) {
  const bool vec = (reinterpret_cast<uintptr_t>(B) & 15u) == 0 && ldb % 4 == 0 &&
                   (reinterpret_cast<uintptr_t>(Bt) & 15u) == 0 && ldbt % 4 == 0;
  if (vec) {
    const int64_t k_tiles = (int64_t(K) + 63) / 64;
    const dim3 grid(unsigned((int64_t(N) + 63) / 64), unsigned(k_tiles < 65535 ? k_tiles : 65535));
    transpose_vec_kernel<<<grid, 256, 0, stream>>>(B, ldb, Bt, ldbt, K, N);
  } else {
    const int64_t k_tiles = (int64_t(K) + 31) / 32;
    const dim3 grid(unsigned((int64_t(N) + 31) / 32), unsigned(k_tiles < 65535 ? k_tiles : 65535));
    transpose_kernel<<<grid, dim3(32, 8), 0, stream>>>(B, ldb, Bt, ldbt, K, N);
  }
  return cudaGetLastError();
}

int tf32_pair_prepare() {
  if (cudaFuncSetAttribute(tf32_pair_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(kPrSmem)) != cudaSuccess ||
      cudaFuncSetAttribute(tf32_pair_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(kPrSmem)) != cudaSuccess)
    return -1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kTfThreads, 1, 1);
  cfg.dynamicSmemBytes = kPrSmem;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, tf32_pair_kernel<true>, &cfg) != cudaSuccess)
    return -1;
  return clusters;
}

int tf32_pair_tile_m() { return kPrBM; }
int tf32_pair_tile_n() { return kPrBN; }

cudaError_t launch_tf32_pair_kernel(bool b_mn, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                                    const CUtensorMap& tmap_c, const Tf32Args& args, const Sched& sched,
                                    int pairs, cudaStream_t stream) {
  if (b_mn)
    tf32_pair_kernel<true><<<2 * pairs, kTfThreads, kPrSmem, stream>>>(tmap_a, tmap_b, tmap_c, args, sched);
  else
    tf32_pair_kernel<false><<<2 * pairs, kTfThreads, kPrSmem, stream>>>(tmap_a, tmap_b, tmap_c, args, sched);
  return cudaGetLastError();
}

cudaError_t launch_tf32_kernel(bool b_mn, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                               const CUtensorMap& tmap_c, const Tf32Args& args, const Sched& sched,
                               int grid, cudaStream_t stream) {
  if (b_mn)
    tf32_kernel<true><<<grid, kTfThreads, kTfSmem, stream>>>(tmap_a, tmap_b, tmap_c, args, sched);
  else
    tf32_kernel<false><<<grid, kTfThreads, kTfSmem, stream>>>(tmap_a, tmap_b, tmap_c, args, sched);
  return cudaGetLastError();
}

}  // namespace gb300
