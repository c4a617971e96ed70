// sgemm_tile.cu -- the warp-specialized FP32 GEMM kernel for sm_103a.
//
// C = A * B, row-major FP32, alpha = 1, beta = 0 ("Beyond Kernel 7: Closing
// the Gap to cuBLAS on an H100 FP32 GEMM", section "The operation").  One
// kernel template serves three schedules (Sched in sgemm_plan.h): one
// tile per CTA, persistent whole-tile waves, and Stream-K splits of K.
//
// Roles inside a CTA:
//  * a producer warpgroup (four warps, one per SM sub-partition) moves data.
//    One lane issues TMA bulk-tensor copies (cp.async.bulk.tensor) of B tiles
//    straight into a STAGES-deep ring.  Each producer warp copies its own
//    32-row slice of every A tile into a private staging ring laid out with
//    the 64-byte swizzle, then rewrites it transposed (k-major, "Vectorized
//    Memory Access ...", section 4) so that one 128-bit shared load yields
//    four rows of A at one k.  This is the multi-stage copy pipeline of
//    "Beyond Kernel 7", section "Kernel 8", with the bulk copy engine in
//    place of per-thread cp.async; A never passes through the compute warps'
//    registers or the L1 request path.  The producers give most of their
//    registers to the consumers (setmaxnreg).
//  * the consumer warps compute.  Each thread owns an 8 x 16 (or 8 x 8)
//    patch of C ("Beyond Kernel 7", section "Kernel 10"), updated per k step
//    as a register outer product ("2D Block Tiling ...", section 4) with
//    fma.rn.f32x2: one instruction performs two FP32 FFMAs, each with its own
//    single rounding, halving the issue slots the arithmetic takes.  The A
//    operand enters as the pair (a, a); building that pair in registers
//    costs no instruction (measured: the broadcast folds into the FFMA2),
//    so A is stored once and read with half the shared-memory traffic of a
//    doubled layout.
//  Producers and consumers meet only at per-stage mbarriers ("full": the
//  stage holds data; "empty": every consumer warp is done with it), so the
//  compute loop has no block-wide barrier.
//
// Warp tiling ("Beyond Kernel 7", section "Kernel 6"): a consumer warp covers
// 32 x (8 * TN) outputs as a 4 x 8 lane grid; within a patch the column
// quads are strided by 32 so that the eight lanes of a row read 128
// contiguous bytes of B ("Kernel 10", strided B-column mapping) and the four
// lanes of a column read 64 contiguous bytes of A.  Output: coalesced
// 128-bit row stores ("cuSgemm", Kernel 5), bounds-checked on edge tiles
// ("2D Block Tiling ...", section 5).
#include <cuda.h>
#include <cuda_runtime.h>

#include <tuple>
#include <type_traits>
#include <utility>

#include "sgemm_device.cuh"
#include "sgemm_plan.h"
#include "sgemm_sched.cuh"
#include "sgemm_trace.h"

namespace gb300 {

#ifdef SGEMM_PHASE_TRACE
__device__ uint64_t* g_trace_buf;
__device__ int64_t g_trace_ctas;

// Phase records of one CTA (one writing thread per log).  The log's pointer
// and extent are loaded at set-up but first used by a record, and the times
// are read before that, so that a record never waits on those loads (they
// miss in L2 right after a flush) ahead of the phase it stamps.
struct TraceLog {
  uint64_t* buf;
  int64_t cap;
  int n, end;
  __device__ __forceinline__ void init(int first, int last) {
    buf = g_trace_buf;
    cap = g_trace_ctas;
    n = first;
    end = last;
  }
  __device__ __forceinline__ void put_at(uint64_t t, uint32_t kind, uint32_t a, uint32_t b) {
    if (buf == nullptr || int64_t(blockIdx.x) >= cap || n >= end) return;
    uint64_t* rec = buf + size_t(blockIdx.x) * kTraceSlots * 2;
    rec[2 * n] = t;
    rec[2 * n + 1] = (uint64_t(kind) << 56) | (uint64_t(a & 0xffffffu) << 32) | b;
    ++n;
  }
  __device__ __forceinline__ void put(uint32_t kind, uint32_t a, uint32_t b) {
    put_at(dev::global_timer_ns(), kind, a, b);
  }
  __device__ __forceinline__ void entry(uint64_t t) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    put_at(t, kTrEntry, smid, 0);
  }
  static __device__ __forceinline__ uint64_t now() { return dev::global_timer_ns(); }
};
#else
struct TraceLog {
  __device__ __forceinline__ void init(int, int) {}
  __device__ __forceinline__ void put(uint32_t, uint32_t, uint32_t) {}
  __device__ __forceinline__ void put_at(uint64_t, uint32_t, uint32_t, uint32_t) {}
  __device__ __forceinline__ void entry(uint64_t) {}
  static __device__ __forceinline__ uint64_t now() { return 0; }
};
#endif

namespace {

constexpr uint32_t kStatusTimeout = 3;  // SGEMM_ERR_TIMEOUT
// How long the CTA that owns a split tile's first k-tiles waits for the other
// sharers' partial sums before publishing its own (see the split-tile epilogue).
constexpr uint64_t kOwnerWaitNs = 5000;
constexpr uint32_t kPfChunk = 16384;  // bytes per bulk copy of a prefetched partial tile

template <int WARPS_M, int WARPS_N, int TN, int STAGES, int ASTAGES, bool DB, int CTAS,
          int PRODUCER_REGS = 56, bool PAIRED_COLS = false, int PF_SLOTS = 0>
struct TileCfg {
  static constexpr int kTR = 4, kTC = 8;    // lane grid of a consumer warp: rows x columns
  static constexpr int kTM = 8, kTN = TN;   // outputs per thread
  static constexpr int kWarpM = kTR * kTM;  // 32
  static constexpr int kWarpN = kTC * kTN;  // 64 or 128
  static constexpr int kWarpsM = WARPS_M;
  static constexpr int kConsumerWarps = WARPS_M * WARPS_N;
  static constexpr int kConsumers = 32 * kConsumerWarps;
  static constexpr int kProducerWarps = 4;  // one warpgroup: one warp per SM sub-partition
  static constexpr int kProducers = 32 * kProducerWarps;
  static constexpr int NT = kConsumers + kProducers;
  static constexpr int kCtasPerSm = CTAS;
  // Registers: the launch gives every thread R0; when R0 is short of what a
  // consumer needs, the producer warpgroup hands registers to the consumer
  // warpgroups (setmaxnreg), keeping the block's total.
  static constexpr int kRegsLaunch = (65536 / (CTAS * NT)) / 8 * 8;
  static constexpr bool kHandOver = kRegsLaunch < 232;
  static constexpr int kRegsProducer = PRODUCER_REGS;
  // Lane layout.  false: a quarter-warp is one lane row (one A address, eight
  // B addresses).  true: a quarter-warp is four lane rows x two lane columns,
  // each column's four lanes adjacent (four A addresses, two B addresses),
  // which costs fewer shared-memory wavefronts per k step.
  static constexpr bool kPairedCols = PAIRED_COLS;
  static constexpr int kRegsConsumer =
      kHandOver ? ((NT * kRegsLaunch - kProducers * kRegsProducer) / kConsumers) / 8 * 8
                : kRegsLaunch;
  static constexpr int BM = WARPS_M * kWarpM;
  static constexpr int BN = WARPS_N * kWarpN;
  static constexpr int BK = 16;  // one 64-byte swizzle span of A per row
  static constexpr int kRowsPerProducer = BM / kProducerWarps;  // 32
  static constexpr int S = STAGES;
  static constexpr int S2 = ASTAGES;
  static constexpr bool kDoubleBuffer = DB;
  static constexpr int kAStride = BM;  // floats per k row of the transposed A tile
  static constexpr int kAStageFloats = BK * kAStride;
  static constexpr int kBStageFloats = BK * BN;
  static constexpr int kAStagingFloats = kRowsPerProducer * BK;  // one producer warp's slot
  static constexpr uint32_t kBStageBytes = kBStageFloats * 4;
  static constexpr uint32_t kAStagingBytes = kAStagingFloats * 4;
  static constexpr int kOutVec = kTM * kTN / 4;  // float4 values per thread
  // Partial tiles of other CTAs that the producer prefetches into shared
  // memory for the split tile this CTA finishes last (0: none).
  static constexpr int kPfSlots = PF_SLOTS;
  static constexpr uint32_t kSlotBytes = uint32_t(BM) * BN * 4;
  // Shared memory: [B ring][A staging: producer warp x slot][A ring]
  // [prefetched partials][barriers][flags]
  static constexpr size_t kBOff = 0;
  static constexpr size_t kAStagingOff = kBOff + size_t(S) * kBStageBytes;
  static constexpr size_t kAOff = kAStagingOff + size_t(kProducerWarps) * S2 * kAStagingBytes;
  static constexpr size_t kPfOff = kAOff + size_t(S) * kAStageFloats * 4;
  static constexpr size_t kBarOff = kPfOff + size_t(PF_SLOTS) * kSlotBytes;
  static constexpr size_t kFlagOff = kBarOff + size_t(2 * S + kProducerWarps * S2 + 1) * 8;
  static constexpr size_t kSmem = kFlagOff + 16;
  static_assert(TN == 8 || TN == 16, "patch width");
  static_assert(ASTAGES <= STAGES, "the prologue's B tiles must fit the empty ring");
  static_assert(kRowsPerProducer == 32, "each producer lane owns one row of the A tile");
  static_assert(BM <= 256 && BN <= 256, "TMA box dimensions are at most 256");
  static_assert(kBStageBytes % 1024 == 0 && kAStagingBytes % 512 == 0,
                "stages keep the 64-byte swizzle period (512 bytes) aligned");
  static_assert(!kHandOver ||
                    kConsumers * kRegsConsumer + kProducers * kRegsProducer <= NT * kRegsLaunch,
                "register hand-over must stay within the launch allocation");
  static_assert(!kHandOver || (kRegsConsumer <= 256 && kRegsConsumer >= kRegsLaunch),
                "consumer register budget");
};

// The compiled tile configurations (index = TileConfig id).
// The 128 x 256 configurations keep six k-tiles in the ring (176 KB of
// shared memory): with four, the compute warps waited for data whenever A
// and B exceed L2 (4096^3: 3 % slower); eight left L1 too small (2.6 %).
using Cfg0 = TileCfg<4, 2, 16, 6, 4, false, 1, 56, true>;   // 128 x 256 tile, 8 + 4 warps, 8x16 patch
using Cfg1 = TileCfg<4, 2, 16, 6, 4, false, 1>;             // Cfg0, one-row quarter-warps
using Cfg2 = TileCfg<4, 2, 16, 6, 4, true, 1, 56, true>;    // Cfg1 with fragment double buffering
using Cfg3 = TileCfg<4, 2, 8, 4, 4, true, 1, 56, false, 1>; // 128 x 128 tile, 8 + 4 warps, 8x8 patch
using Cfg4 = TileCfg<4, 2, 8, 4, 4, true, 1, 56, true>;     // Cfg3, paired-column lane layout
using Cfg5 = TileCfg<4, 2, 8, 4, 4, false, 1, 56, true>;    // Cfg4 without double buffering

// Only the configurations the selector uses by default (0 and 3) carry
// instances that read A M-major; the others exist for tuning runs.
template <class T>
constexpr bool kHasAmn = std::is_same<T, Cfg0>::value || std::is_same<T, Cfg3>::value;

template <class F>
auto with_cfg(int id, F&& f) {
  switch (id) {
    case 1: return f(Cfg1{});
    case 2: return f(Cfg2{});
    case 3: return f(Cfg3{});
    case 4: return f(Cfg4{});
    case 5: return f(Cfg5{});
    default: return f(Cfg0{});
  }
}

// SCALED: the general epilogue, C = alpha * acc + beta * C with C read and
// written 4 bytes at a time when it is not 16-byte aligned row by row (a
// separate instance, so that the plain C = A * B kernel with aligned C
// carries neither).
//
// FM, FN, FK > 0: the size-specialized instance ("Beyond Kernel 7", the
// size-specialized kernel behind the confirmed 4096 result): the problem
// shape and the Stream-K schedule of kSpecializedResident CTAs are compile-
// time constants, so tile coordinates, shares and bounds fold into the code.
// The launch must pass exactly that schedule (the host checks).
template <class T, bool SCALED, bool AMN = false, int FM = 0, int FN = 0, int FK = 0>
__global__ void __launch_bounds__(T::NT, T::kCtasPerSm)
    tile_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                const GemmArgs args, const Sched sc_in) {
  const uint64_t t_entry = TraceLog::now();
  Sched sc = sc_in;
  if constexpr (FM > 0) {
    constexpr LaunchPlan kPlan =
        plan_launch(FM, FN, FK, T::BM, T::BN, T::BK, kSpecializedResident, true);
    static_assert(kPlan.ok && kPlan.grid == kSpecializedResident, "specialized schedule");
    sc = kPlan.sc;
  }
  extern __shared__ __align__(1024) unsigned char smem[];
  float* sB = reinterpret_cast<float*>(smem + T::kBOff);
  float* sAst = reinterpret_cast<float*>(smem + T::kAStagingOff);
  float* sA = reinterpret_cast<float*>(smem + T::kAOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + T::kBarOff);
  uint64_t* empty = full + T::S;
  uint64_t* astage = empty + T::S;  // [producer warp][slot]
  uint64_t* pf_full = astage + T::kProducerWarps * T::S2;  // prefetched partials landed
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + T::kFlagOff);
  int* s_last = reinterpret_cast<int*>(smem + T::kFlagOff + 4);
  volatile int* s_epi = reinterpret_cast<volatile int*>(smem + T::kFlagOff + 8);  // owner epilogue reached
  volatile int* s_pf = reinterpret_cast<volatile int*>(smem + T::kFlagOff + 12);  // partials prefetched

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  constexpr bool kEarlyFirstCopy = !AMN && FM > 0;
  const int cta = blockIdx.x, ctas = gridDim.x;
  const uint64_t limit = args.wait_limit_ns;
  TraceLog trace;

  if (tid == 0) {
    for (int s = 0; s < T::S; ++s) {
      dev::mbar_init(&full[s], T::kProducers);       // every producer thread
      dev::mbar_init(&empty[s], T::kConsumerWarps);  // one arrival per consumer warp
    }
    for (int s = 0; s < T::kProducerWarps * T::S2; ++s) dev::mbar_init(&astage[s], 1);
    dev::mbar_init(pf_full, 1);
    *s_abort = 0;
    *s_epi = 0;
    *s_pf = 0;
    dev::mbar_init_fence();
    // Size-specialized instances: the first k-tile's copies leave now, before
    // the CTA-wide barrier and the producers' register hand-over (right after
    // a cache flush they wait on DRAM, and that wait starts the pipeline); the
    // producers issue the rest.  The generic kernel would first wait here for
    // its schedule in the constant bank, which measured slower.
    if constexpr (kEarlyFirstCopy) {
      KCursor c0;
      c0.init(sc, cta, ctas);
      if (c0.valid) {
        const int k0 = c0.u.kb * T::BK;
        for (int pw = 0; pw < T::kProducerWarps; ++pw) {
          dev::mbar_arrive_expect_tx(&astage[pw * T::S2], T::kAStagingBytes);
          dev::tma_load_2d(sAst + pw * T::S2 * T::kAStagingFloats, &tmap_a, k0,
                           c0.tm * T::BM + pw * T::kRowsPerProducer, &astage[pw * T::S2]);
        }
        dev::mbar_expect_tx(&full[0], T::kBStageBytes);
        dev::tma_load_2d(sB, &tmap_b, c0.tn * T::BN, k0, &full[0]);
      }
    }
  }
  const uint64_t t_init = TraceLog::now();
  __syncthreads();
  const uint64_t t_sync = TraceLog::now();

  // A wait that failed: record it once, make every later wait of the CTA give
  // up at once, and carry on without waiting so that nothing hangs.
  auto fail = [&](uint32_t site) {
    if (!*s_abort) {
      *s_abort = 1;
      dev::record_status(args.status, kStatusTimeout, site);
    }
  };

  // The CTAs that share split tile t_sk, [c_first, c_last] in CTA order.
  auto sharers = [&](int t_sk, int& c_first, int& c_last) {
    const int64_t first_iter = int64_t(t_sk) * sc.iters_per_tile;
    c_first = sk_owner(sc, first_iter);
    c_last = sk_owner(sc, first_iter + sc.iters_per_tile - 1);
  };

  // Prefetch of the other sharers' partial tiles for the split tile this CTA
  // finishes last.  The CTA that owns a split tile's first k-tiles computes
  // them at the end of its share, and the other sharers have usually
  // published their partials by then; reading those from L2 after the last
  // k-tile was most of the hand-off's cost.  Once every other sharer has
  // arrived, producer warp 0 bulk-copies up to kPfSlots partials into shared
  // memory while the compute warps finish.  It stops polling kOwnerWaitNs
  // after the compute warps reached that epilogue (they then publish as
  // usual); it always arrives on pf_full exactly once, with the number of
  // partials copied in s_pf.
  auto prefetch_partials = [&]() {
    if constexpr (T::kPfSlots > 0) {
      if (warp != T::kConsumerWarps || lane != 0) return;
      WorkIter wl;
      wl.init(sc, cta);
      Unit lu{}, uu;
      bool any = false;
      while (wl.next(sc, ctas, uu)) {
        lu = uu;
        any = true;
      }
      if (!any || lu.t_sk < 0 || (lu.kb == 0 && lu.ke == sc.iters_per_tile)) return;
      int c_first, c_last;
      sharers(lu.t_sk, c_first, c_last);
      const int others = c_last - c_first;
      if (c_first != cta || others == 0 || args.owner_publishes) return;
      int npf = 0;
      if (!*s_abort) {
        const int32_t* cnt = args.counters + lu.t_sk;
        const uint64_t t0 = dev::global_timer_ns();
        uint64_t t_epi = 0;
        int seen = dev::ld_acquire_gpu(cnt);
        while (seen != others && !*s_abort) {
          const uint64_t t = dev::global_timer_ns();
          if (*s_epi) {
            if (t_epi == 0) t_epi = t;
            else if (t - t_epi > kOwnerWaitNs) break;
          }
          if (t - t0 > limit) break;
          __nanosleep(128);
          seen = dev::ld_acquire_gpu(cnt);
        }
        if (seen == others) {
          // The partials were written through the generic proxy; the bulk
          // copies read them through the async proxy.
          asm volatile("fence.proxy.async.global;" ::: "memory");
          npf = others < T::kPfSlots ? others : T::kPfSlots;
          *s_pf = npf;
          dev::mbar_arrive_expect_tx(pf_full, uint32_t(npf) * T::kSlotBytes);
          for (int i = 0; i < npf; ++i) {
            const unsigned char* src = reinterpret_cast<const unsigned char*>(
                args.partials + int64_t(lu.t_sk + c_first + 1 + i) * (int64_t(T::BM) * T::BN));
            unsigned char* dst = smem + T::kPfOff + size_t(i) * T::kSlotBytes;
            for (uint32_t off = 0; off < T::kSlotBytes; off += kPfChunk)
              dev::bulk_load(dst + off, src + off, kPfChunk, pf_full);
          }
        }
      }
      if (npf == 0) {
        *s_pf = 0;
        dev::mbar_arrive(pf_full);
      }
      // The CTA must not exit with copies in flight.
      if (!dev::mbar_wait(pf_full, 0, limit)) fail(kWaitTileStage);
    }
  };

  if (warp >= T::kConsumerWarps) {
    // ================================================ producer warpgroup
    if constexpr (T::kHandOver) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(T::kRegsProducer));
    // (After the register hand-over: it would wait for the trace loads.)
    if (tid == T::kConsumers) trace.init(kTraceProducerSlot0, kTraceSlots);
    const int pw = warp - T::kConsumerWarps;  // this warp owns A rows [32 pw, 32 pw + 32)
    // Producer phase times, recorded when the producer is done (see TraceLog).
    const uint64_t tp_start = TraceLog::now();
    uint64_t tp_issued = 0, tp_first_a = 0;
    auto put_producer_times = [&]() {
      if (pw == 0 && lane == 0) {
        trace.put_at(tp_start, kTrProducerStart, 0, 0);
        if (tp_issued) trace.put_at(tp_issued, kTrProducerIssued, 0, 0);
        if (tp_first_a) trace.put_at(tp_first_a, kTrFirstALanded, 0, 0);
      }
    };
    uint64_t* my_astage = astage + pw * T::S2;
    float* my_staging = sAst + pw * T::S2 * T::kAStagingFloats;
    if (lane == 0) {
      dev::tma_prefetch_desc(&tmap_a);
      if (pw == 0) dev::tma_prefetch_desc(&tmap_b);
    }
    if constexpr (AMN) {
      // A^T's storage is M-major: one copy of the BK x BM tile lands in the
      // ring exactly as the compute warps read it ([k][m]).  One lane issues
      // both tiles of a stage; every producer thread arrives on full[s].
      KCursor cur;
      cur.init(sc, cta, ctas);
      uint32_t i = 0;
      for (; cur.valid; ++i) {
        const uint32_t s = i % T::S, n = i / T::S;
        if (n > 0 && !dev::mbar_wait_abortable(&empty[s], (n - 1) & 1u, limit, s_abort))
          fail(kWaitTileStage);
        if (pw == 0 && lane == 0 && !*s_abort) {
          dev::mbar_expect_tx(&full[s], T::kBStageBytes + T::kAStageFloats * 4);
          const int k0 = (cur.u.kb + cur.j) * T::BK;
          dev::tma_load_2d(sB + s * T::kBStageFloats, &tmap_b, cur.tn * T::BN, k0, &full[s]);
          dev::tma_load_2d(sA + s * T::kAStageFloats, &tmap_a, cur.tm * T::BM, k0, &full[s]);
        }
        dev::mbar_arrive(&full[s]);
        cur.advance(sc, ctas);
      }
      if (*s_abort && pw == 0 && lane == 0)
        for (uint32_t k = (i > T::S ? i - T::S : 0); k < i; ++k)
          dev::mbar_wait(&full[k % T::S], (k / T::S) & 1u, limit);
      put_producer_times();
      prefetch_partials();
      return;
    }
    KCursor issue, proc;
    issue.init(sc, cta, ctas);
    proc.init(sc, cta, ctas);
    auto issue_a = [&](uint32_t slot) {
      dev::mbar_arrive_expect_tx(&my_astage[slot], T::kAStagingBytes);
      dev::tma_load_2d(my_staging + slot * T::kAStagingFloats, &tmap_a,
                       (issue.u.kb + issue.j) * T::BK, issue.tm * T::BM + pw * T::kRowsPerProducer,
                       &my_astage[slot]);
    };
    // The B tile of k-tile `c.j` of unit `c.u` into ring stage s.
    auto issue_b = [&](const KCursor& c, uint32_t s) {
      dev::mbar_expect_tx(&full[s], T::kBStageBytes);
      dev::tma_load_2d(sB + s * T::kBStageFloats, &tmap_b, c.tn * T::BN, (c.u.kb + c.j) * T::BK,
                       &full[s]);
    };
    // Prologue: this warp's first S2 A slices into its staging ring and, from
    // warp 0, the B tiles of the same k-tiles (their ring stages start empty),
    // each right behind its A slice so that the first stage fills as early
    // as the copies allow.  (With kEarlyFirstCopy the first k-tile's copies
    // were issued at set-up.)
    uint32_t issued = 0;
    for (int s = 0; s < T::S2 && issue.valid; ++s) {
      if (lane == 0 && (s > 0 || !kEarlyFirstCopy)) {
        issue_a(s);
        if (pw == 0) issue_b(issue, s);
      }
      ++issued;
      issue.advance(sc, ctas);
    }
    const uint32_t b_issued = issued;
    tp_issued = TraceLog::now();
    uint32_t i = 0;
    for (; proc.valid; ++i) {
      const uint32_t s = i % T::S, n = i / T::S;
      const uint32_t s2 = i % T::S2, n2 = i / T::S2;
      if (i >= b_issued) {
        if (n > 0 && !dev::mbar_wait_abortable(&empty[s], (n - 1) & 1u, limit, s_abort))
          fail(kWaitTileStage);
        if (pw == 0 && lane == 0 && !*s_abort) issue_b(proc, s);
      }
      if (!dev::mbar_wait_abortable(&my_astage[s2], n2 & 1u, limit, s_abort)) fail(kWaitTileStage);
      if (i == 0) tp_first_a = TraceLog::now();
      // Transpose this warp's 32 rows: staging [r][k] (64-byte swizzled rows:
      // 16-byte chunk q of row r sits at q ^ ((r >> 1) & 3)) -> ring [k][m].
      // Consecutive lanes write consecutive m: conflict-free 4-byte stores.
      {
        const int r = lane;                    // row within this warp's slice
        const int m = pw * T::kRowsPerProducer + r;  // row within the tile
        const float* src = my_staging + s2 * T::kAStagingFloats + r * T::BK;
        float* d = sA + s * T::kAStageFloats + m;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 v = *reinterpret_cast<const float4*>(src + (q ^ ((r >> 1) & 3)) * 4);
          d[(4 * q + 0) * T::kAStride] = v.x;
          d[(4 * q + 1) * T::kAStride] = v.y;
          d[(4 * q + 2) * T::kAStride] = v.z;
          d[(4 * q + 3) * T::kAStride] = v.w;
        }
      }
      __syncwarp();
      // The staging slot is free again: refill it with the slice S2 k-tiles ahead.
      if (issue.valid) {
        if (lane == 0 && !*s_abort) {
          dev::fence_proxy_async_smem();
          issue_a(s2);
        }
        ++issued;
        issue.advance(sc, ctas);
      }
      dev::mbar_arrive(&full[s]);
      proc.advance(sc, ctas);
    }
    // Normally every copy was consumed.  After a failure, let any copy still
    // in flight land (bounded) before the CTA's shared memory is released.
    if (*s_abort && lane == 0) {
      for (uint32_t k = i; k < issued; ++k)
        dev::mbar_wait(&my_astage[k % T::S2], (k / T::S2) & 1u, limit);
      if (pw == 0)
        for (uint32_t k = (i > T::S ? i - T::S : 0); k < i; ++k)
          dev::mbar_wait(&full[k % T::S], (k / T::S) & 1u, limit);
    }
    put_producer_times();
    prefetch_partials();
    return;
  }

  // ======================================================= consumer warps
  if constexpr (T::kHandOver) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(T::kRegsConsumer));
  if (tid == 0) trace.init(0, kTraceProducerSlot0);
  const int tr = T::kPairedCols ? (lane & 3) : lane / T::kTC;
  const int tc = T::kPairedCols ? (((lane >> 3) << 1) | ((lane >> 2) & 1)) : lane % T::kTC;
  const int wm = warp % T::kWarpsM, wn = warp / T::kWarpsM;
  const int a_frag = wm * T::kWarpM + 4 * tr;  // + 16 g + kAStride kk
  const int b_frag = wn * T::kWarpN + 4 * tc;      // + 32 h + BN kk
  const int M = FM > 0 ? FM : args.M, N = FN > 0 ? FN : args.N;

  WorkIter w;
  w.init(sc, cta);
  Unit u;
  uint32_t it = 0;  // k-tiles consumed so far: position in the stage ring
  while (w.next(sc, ctas, u)) {
    int tm, tn;
    tile_coords(sc, u.tile, tm, tn);
    const int m0 = tm * T::BM, n0 = tn * T::BN;
    const int nk = u.ke - u.kb;

    float2 acc[T::kTM][T::kTN / 2];
#pragma unroll
    for (int r = 0; r < T::kTM; ++r)
#pragma unroll
      for (int q = 0; q < T::kTN / 2; ++q) acc[r][q] = make_float2(0.f, 0.f);

    for (int j = 0; j < nk; ++j, ++it) {
      const uint32_t s = it % T::S;
      if (!dev::mbar_wait_abortable(&full[s], (it / T::S) & 1u, limit, s_abort)) fail(kWaitTileStage);
      if (it == 0 && tid == 0) trace.put(kTrFirstStage, 0, 0);
      const float* a_buf = sA + s * T::kAStageFloats + a_frag;
      const float* b_buf = sB + s * T::kBStageFloats + b_frag;
      struct Frag {
        float4 a[T::kTM / 4];  // A at rows m .. m+3 of each of the thread's row quads
        float4 b[T::kTN / 4];  // four consecutive B values per column quad
      };
      auto load_frag = [&](Frag& f, int kk) {
#pragma unroll
        for (int g = 0; g < T::kTM / 4; ++g)
          f.a[g] = *reinterpret_cast<const float4*>(a_buf + kk * T::kAStride + 16 * g);
#pragma unroll
        for (int h = 0; h < T::kTN / 4; ++h)
          f.b[h] = *reinterpret_cast<const float4*>(b_buf + kk * T::BN + 32 * h);
      };
      // B-major order: consecutive FFMA2s share one B pair and walk the rows,
      // which measured markedly faster than row-major orders on sm_103a.
      auto fma_frag = [&](const Frag& f) {
        float2 ap[T::kTM];  // (a, a) for each of the thread's rows
#pragma unroll
        for (int g = 0; g < T::kTM / 4; ++g) {
          ap[4 * g + 0] = make_float2(f.a[g].x, f.a[g].x);
          ap[4 * g + 1] = make_float2(f.a[g].y, f.a[g].y);
          ap[4 * g + 2] = make_float2(f.a[g].z, f.a[g].z);
          ap[4 * g + 3] = make_float2(f.a[g].w, f.a[g].w);
        }
#pragma unroll
        for (int h = 0; h < T::kTN / 4; ++h) {
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            const float2 bq = p ? make_float2(f.b[h].z, f.b[h].w) : make_float2(f.b[h].x, f.b[h].y);
#pragma unroll
            for (int r = 0; r < T::kTM; ++r) dev::ffma2(acc[r][2 * h + p], ap[r], bq);
          }
        }
      };
      if constexpr (T::kDoubleBuffer) {
        Frag f[2];
        load_frag(f[0], 0);
#pragma unroll
        for (int kk = 0; kk < T::BK; ++kk) {
          if (kk + 1 < T::BK) load_frag(f[(kk + 1) & 1], kk + 1);
          fma_frag(f[kk & 1]);
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < T::BK; ++kk) {
          Frag f;
          load_frag(f, kk);
          fma_frag(f);
        }
      }
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(&empty[s]);
    }

    if (tid == 0) trace.put(kTrKLoopEnd, uint32_t(u.tile), uint32_t(nk));
    // ---- epilogue
    // Thread value j is the float4 of patch row r = j / Q, column quad h = j % Q.
    constexpr int Q = T::kTN / 4;
    auto out_row = [&](int r) {
      return m0 + wm * T::kWarpM + (r >> 2) * (4 * T::kTR) + 4 * tr + (r & 3);
    };
    auto out_col = [&](int h) { return n0 + wn * T::kWarpN + h * (4 * T::kTC) + 4 * tc; };
    auto value = [&](int j) {
      const int r = j / Q, h = j % Q;
      return make_float4(acc[r][2 * h].x, acc[r][2 * h].y, acc[r][2 * h + 1].x, acc[r][2 * h + 1].y);
    };
    // A C that is not 16-byte aligned row by row is read and written 4 bytes
    // at a time; only the general (SCALED) instance carries that code.
    const bool c_vec = SCALED ? args.c_scalar == 0 : true;
    // alpha / beta epilogue: C = alpha * v + beta * C; beta == 0 never reads C.
    auto finish = [&](float4 v, const float* p, int ncols) {
      float4 r = make_float4(args.alpha * v.x, args.alpha * v.y, args.alpha * v.z, args.alpha * v.w);
      if (args.beta != 0.f) {
        float4 c;
        if (ncols >= 4 && c_vec) {
          c = *reinterpret_cast<const float4*>(p);
        } else {
          c.x = ncols > 0 ? p[0] : 0.f;
          c.y = ncols > 1 ? p[1] : 0.f;
          c.z = ncols > 2 ? p[2] : 0.f;
          c.w = ncols > 3 ? p[3] : 0.f;
        }
        r.x = fmaf(args.beta, c.x, r.x);
        r.y = fmaf(args.beta, c.y, r.y);
        r.z = fmaf(args.beta, c.z, r.z);
        r.w = fmaf(args.beta, c.w, r.w);
      }
      return r;
    };
    auto store_c = [&](int j, float4 v) {
      const int row = out_row(j / Q), col = out_col(j % Q);
      if (row >= M) return;
      float* p = args.C + int64_t(row) * args.ldc + col;
      if constexpr (SCALED) v = finish(v, p, N - col);
      if (col + 4 <= N && c_vec) {
        *reinterpret_cast<float4*>(p) = v;
      } else {
        if (col + 0 < N) p[0] = v.x;
        if (col + 1 < N) p[1] = v.y;
        if (col + 2 < N) p[2] = v.z;
        if (col + 3 < N) p[3] = v.w;
      }
    };

    if (u.t_sk < 0 || (u.kb == 0 && u.ke == sc.iters_per_tile)) {
      if (m0 + T::BM <= M && n0 + T::BN <= N && !SCALED && c_vec) {
#pragma unroll
        for (int j = 0; j < T::kOutVec; ++j) {
          float* p = args.C + int64_t(out_row(j / Q)) * args.ldc + out_col(j % Q);
          *reinterpret_cast<float4*>(p) = value(j);
        }
      } else {
#pragma unroll
        for (int j = 0; j < T::kOutVec; ++j) store_c(j, value(j));
      }
      if (tid == 0) trace.put(kTrStoreEnd, uint32_t(u.tile), 0);
      continue;
    }

    // Split tile: the CTAs that share it publish their partial sums and the
    // last to arrive adds all partials in CTA order (deterministic) and
    // writes C.  The CTA that owns the tile's first k-tiles keeps its partial
    // in registers: if it finds every other sharer already arrived it is the
    // last and publishes nothing; if it turns out last after publishing, it
    // still adds from its registers.  Either way the sum is the same
    // sequence of additions, so the result does not depend on who is last.
    int c_first, c_last;
    sharers(u.t_sk, c_first, c_last);
    const int others = c_last - c_first;
    const int64_t tile_floats = int64_t(T::BM) * T::BN;
    const bool own_first = cta == c_first && !args.owner_publishes;
    bool last = false;
    int npf = 0;  // other sharers' partials already in shared memory
    if constexpr (T::kPfSlots > 0) {
      WorkIter wp = w;
      Unit un;
      if (own_first && others > 0 && !wp.next(sc, ctas, un)) {
        // This CTA's last unit: the producer prefetches (or gives up on) the
        // other sharers' partials and always arrives on pf_full.
        if (tid == 0) *s_epi = 1;
        if (!dev::mbar_wait_abortable(pf_full, 0, limit, s_abort)) fail(kWaitTileStage);
        npf = *s_pf;
        if (npf > 0) last = true;  // every other sharer had arrived
        if (tid == 0) trace.put(kTrOwnerWait, uint32_t(u.tile), npf > 0 ? 2u : 0u);
      }
    }
    if (own_first && !last) {
      // The other sharers usually finish their parts at about the same time
      // (a sharer whose whole share lies in this tile ends with it).  Where
      // partials are prefetched, waiting a little for their arrivals costs
      // less than publishing this partial and reading it back, so poll the
      // counter for up to kOwnerWaitNs; if they are not all in by then,
      // publish as any sharer does.  The wait is bounded, so no CTA depends on
      // another being resident.  Without prefetching (128 x 256 tiles: no
      // room for a 128 KB partial) the wait measured a loss: at 4096^3 a few
      // owners waited it out behind a slower SM and then published anyway.
      if (tid == 0) {
        const int32_t* cnt = args.counters + u.t_sk;
        int seen = dev::ld_acquire_gpu(cnt);
        if (T::kPfSlots > 0 && seen != others) {
          const uint64_t t0 = dev::global_timer_ns();
          while (seen != others && dev::global_timer_ns() - t0 < kOwnerWaitNs) {
            __nanosleep(64);
            seen = dev::ld_acquire_gpu(cnt);
          }
        }
        *s_last = seen == others ? 1 : 0;
        trace.put(kTrOwnerWait, uint32_t(u.tile), seen == others ? 1u : 0u);
      }
      dev::named_barrier(1, T::kConsumers);
      last = *s_last != 0;
      dev::named_barrier(1, T::kConsumers);  // s_last is rewritten below
    }
    if (!last) {
      float4* mine = reinterpret_cast<float4*>(args.partials + (u.t_sk + cta) * tile_floats);
#pragma unroll
      for (int j = 0; j < T::kOutVec; ++j) __stcg(mine + j * T::kConsumers + tid, value(j));
      // One thread releases the whole partial: the barrier orders every
      // thread's stores before tid 0's GPU-scope fence, which is cumulative,
      // and that fence before the arrival.  (A fence in every thread, each
      // waiting for its own stores, measured 1.7 us slower at 768^3.)  The
      // fence after the arrival orders the reads of a last arriver.
      dev::named_barrier(1, T::kConsumers);
      if (tid == 0) {
        __threadfence();
        const int arrived = atomicAdd(args.counters + u.t_sk, 1);
        __threadfence();
        *s_last = (arrived == others) ? 1 : 0;
      }
      dev::named_barrier(1, T::kConsumers);
      last = *s_last != 0;
      dev::named_barrier(1, T::kConsumers);  // s_last may be rewritten by the next split tile
      if (tid == 0) trace.put(kTrPublishEnd, uint32_t(u.tile), last ? 1u : 0u);
    }
    if (last) {
      // Every other partial is in the workspace.  The reads below are ordered
      // after the other sharers' stores by the acquire that decided `last`
      // (tid 0's fence after its arrival, its acquire load of the counter, or
      // the producer's before the prefetch) and the CTA barrier or prefetch
      // barrier that followed it.
      const float4* base = reinterpret_cast<const float4*>(args.partials) + tid;
      const int64_t slot_vec = tile_floats / 4;
      if (own_first) {
        // acc += partial, CTA after CTA.  Partials in shared memory first (the
        // prefetched ones lead in CTA order), then the rest from L2 with a
        // slot's loads in flight at once -- two slots' where the registers
        // allow (the additions keep CTA order either way).
        auto add_partial = [&](const float4 (&v)[T::kOutVec]) {
#pragma unroll
          for (int j = 0; j < T::kOutVec; ++j) {
            const int r = j / Q, h = j % Q;
            acc[r][2 * h].x += v[j].x;
            acc[r][2 * h].y += v[j].y;
            acc[r][2 * h + 1].x += v[j].z;
            acc[r][2 * h + 1].y += v[j].w;
          }
        };
        int cc = c_first + 1;
#pragma unroll 1
        for (; cc <= c_last && cc - c_first - 1 < npf; ++cc) {
          float4 v[T::kOutVec];
          const float4* src = reinterpret_cast<const float4*>(
                                  smem + T::kPfOff + size_t(cc - c_first - 1) * T::kSlotBytes) +
                              tid;
#pragma unroll
          for (int j = 0; j < T::kOutVec; ++j) v[j] = src[j * T::kConsumers];
          add_partial(v);
        }
        if constexpr (T::kOutVec <= 16) {
#pragma unroll 1
          for (; cc + 1 <= c_last; cc += 2) {
            float4 v0[T::kOutVec], v1[T::kOutVec];
            const float4* src0 = base + (u.t_sk + cc) * slot_vec;
            const float4* src1 = src0 + slot_vec;
#pragma unroll
            for (int j = 0; j < T::kOutVec; ++j) v0[j] = __ldcg(src0 + j * T::kConsumers);
#pragma unroll
            for (int j = 0; j < T::kOutVec; ++j) v1[j] = __ldcg(src1 + j * T::kConsumers);
            add_partial(v0);
            add_partial(v1);
          }
        }
#pragma unroll 1
        for (; cc <= c_last; ++cc) {
          float4 v[T::kOutVec];
          const float4* src = base + (u.t_sk + cc) * slot_vec;
#pragma unroll
          for (int j = 0; j < T::kOutVec; ++j) v[j] = __ldcg(src + j * T::kConsumers);
          add_partial(v);
        }
#pragma unroll
        for (int j = 0; j < T::kOutVec; ++j) store_c(j, value(j));
      } else {
        // Sum every partial, this CTA's included, in CTA order (two slots'
        // loads in flight at once where the registers allow).
        float4 sum[T::kOutVec];
        auto add_partial = [&](const float4 (&v)[T::kOutVec]) {
#pragma unroll
          for (int j = 0; j < T::kOutVec; ++j) {
            sum[j].x += v[j].x;
            sum[j].y += v[j].y;
            sum[j].z += v[j].z;
            sum[j].w += v[j].w;
          }
        };
        {
          const float4* src = base + (u.t_sk + c_first) * slot_vec;
#pragma unroll
          for (int j = 0; j < T::kOutVec; ++j) sum[j] = __ldcg(src + j * T::kConsumers);
        }
        int cc = c_first + 1;
        if constexpr (T::kOutVec <= 16) {
#pragma unroll 1
          for (; cc + 1 <= c_last; cc += 2) {
            float4 v0[T::kOutVec], v1[T::kOutVec];
            const float4* src0 = base + (u.t_sk + cc) * slot_vec;
            const float4* src1 = src0 + slot_vec;
#pragma unroll
            for (int j = 0; j < T::kOutVec; ++j) v0[j] = __ldcg(src0 + j * T::kConsumers);
#pragma unroll
            for (int j = 0; j < T::kOutVec; ++j) v1[j] = __ldcg(src1 + j * T::kConsumers);
            add_partial(v0);
            add_partial(v1);
          }
        }
#pragma unroll 1
        for (; cc <= c_last; ++cc) {
          const float4* src = base + (u.t_sk + cc) * slot_vec;
          float4 v[T::kOutVec];
#pragma unroll
          for (int j = 0; j < T::kOutVec; ++j) v[j] = __ldcg(src + j * T::kConsumers);
          add_partial(v);
        }
#pragma unroll
        for (int j = 0; j < T::kOutVec; ++j) store_c(j, sum[j]);
      }
      if (tid == 0) {
        args.counters[u.t_sk] = 0;
        trace.put(kTrReduceEnd, uint32_t(u.tile), uint32_t(others));
      }
    }
  }
  if (tid == 0) {
    trace.entry(t_entry);
    trace.put_at(t_init, kTrBarriersReady, 0, 0);
    trace.put_at(t_sync, kTrCtaSynced, 0, 0);
    trace.put(kTrExit, 0, 0);
  }
}

template <class T>
int prepare() {
  if (cudaFuncSetAttribute(tile_kernel<T, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(T::kSmem)) != cudaSuccess ||
      cudaFuncSetAttribute(tile_kernel<T, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(T::kSmem)) != cudaSuccess)
    return -1;
  if constexpr (kHasAmn<T>) {
    if (cudaFuncSetAttribute(tile_kernel<T, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(T::kSmem)) != cudaSuccess ||
        cudaFuncSetAttribute(tile_kernel<T, true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(T::kSmem)) != cudaSuccess)
      return -1;
  }
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, tile_kernel<T, false>, T::NT,
                                                    T::kSmem) != cudaSuccess)
    return -1;
  return blocks;
}

// The size-specialized instances: configuration id and M = N = K.  The
// square sizes where the compiled-in schedule measured faster than the
// generic kernel on GB300: 768^3 and 1024^3 on 128 x 128 tiles, 4096^3 on
// 128 x 256.  At 1536^3 and 2048^3 it did not (equal, and 2 us slower).
template <int ID>
struct CfgById;
template <>
struct CfgById<0> {
  using type = Cfg0;
};
template <>
struct CfgById<3> {
  using type = Cfg3;
};

template <int ID, int M, int N, int K>
struct SpecInst {
  using T = typename CfgById<ID>::type;
  static constexpr int kId = ID;
  static constexpr int64_t kM = M, kN = N, kK = K;
  static SpecShape shape() { return SpecShape{ID, M, N, K}; }
  static bool prepare() {
    return cudaFuncSetAttribute(tile_kernel<T, false, false, M, N, K>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                int(T::kSmem)) == cudaSuccess;
  }
  static void launch(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b, const GemmArgs& args,
                     const Sched& sched, int grid, cudaStream_t stream) {
    tile_kernel<T, false, false, M, N, K><<<grid, T::NT, T::kSmem, stream>>>(tmap_a, tmap_b, args, sched);
  }
};

using SpecList = std::tuple<SpecInst<0, 4096, 4096, 4096>, SpecInst<3, 1024, 1024, 1024>,
                            SpecInst<3, 768, 768, 768>>;
constexpr int kSpecCount = int(std::tuple_size<SpecList>::value);
static_assert(kSpecCount == kSpecShapeCount, "SpecList and kSpecShapes list the same instances");
template <size_t... I>
constexpr bool spec_table_matches(std::index_sequence<I...>) {
  return ((kSpecShapes[I].cfg == std::tuple_element_t<I, SpecList>::kId &&
           kSpecShapes[I].m == std::tuple_element_t<I, SpecList>::kM &&
           kSpecShapes[I].n == std::tuple_element_t<I, SpecList>::kN &&
           kSpecShapes[I].k == std::tuple_element_t<I, SpecList>::kK) &&
          ...);
}
static_assert(spec_table_matches(std::make_index_sequence<kSpecCount>{}),
              "SpecList and kSpecShapes list the same instances in the same order");
using SpecIndex = std::make_index_sequence<std::tuple_size<SpecList>::value>;

template <size_t... I>
SpecShape spec_shape_at(int i, std::index_sequence<I...>) {
  SpecShape out{-1, 0, 0, 0};
  ((int(I) == i ? (out = std::tuple_element_t<I, SpecList>::shape(), true) : false) || ...);
  return out;
}

template <size_t... I>
bool spec_prepare_all(std::index_sequence<I...>) {
  return (std::tuple_element_t<I, SpecList>::prepare() && ...);
}

template <size_t... I>
bool spec_launch_at(int i, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                    const GemmArgs& args, const Sched& sched, int grid, cudaStream_t stream,
                    std::index_sequence<I...>) {
  return ((int(I) == i
               ? (std::tuple_element_t<I, SpecList>::launch(tmap_a, tmap_b, args, sched, grid, stream),
                  true)
               : false) ||
          ...);
}

template <class T>
TileShape shape_of() {
  return TileShape{T::BM, T::BN, T::BK, T::NT, T::S, T::kSmem, T::kRowsPerProducer, T::kTN,
                   T::kCtasPerSm, kHasAmn<T>};
}

}  // namespace

TileShape tile_shape(TileConfig cfg) {
  return with_cfg(cfg, [](auto c) { return shape_of<decltype(c)>(); });
}

int tile_kernel_prepare(TileConfig cfg) {
  return with_cfg(cfg, [](auto c) { return prepare<decltype(c)>(); });
}

int specialized_count() { return kSpecCount; }

SpecShape specialized_shape(int i) { return spec_shape_at(i, SpecIndex{}); }

int specialized_prepare() { return spec_prepare_all(SpecIndex{}) ? 0 : -1; }

cudaError_t launch_specialized(int i, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                               const GemmArgs& args, const Sched& sched, int grid,
                               cudaStream_t stream) {
  if (args.a_mn || args.scaled || args.c_scalar) return cudaErrorInvalidValue;  // plain instances only
  if (!spec_launch_at(i, tmap_a, tmap_b, args, sched, grid, stream, SpecIndex{}))
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_tile_kernel(TileConfig cfg, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                               const GemmArgs& args, const Sched& sched, int grid,
                               cudaStream_t stream) {
  return with_cfg(cfg, [&](auto c) {
    using T = decltype(c);
    const bool scaled = args.scaled || args.c_scalar;
    if (args.a_mn) {
      if constexpr (kHasAmn<T>) {
        if (scaled)
          tile_kernel<T, true, true><<<grid, T::NT, T::kSmem, stream>>>(tmap_a, tmap_b, args, sched);
        else
          tile_kernel<T, false, true><<<grid, T::NT, T::kSmem, stream>>>(tmap_a, tmap_b, args, sched);
      } else {
        return cudaErrorInvalidValue;  // the host reads tile_shape().a_mn first
      }
    } else if (scaled) {
      tile_kernel<T, true><<<grid, T::NT, T::kSmem, stream>>>(tmap_a, tmap_b, args, sched);
    } else {
      tile_kernel<T, false><<<grid, T::NT, T::kSmem, stream>>>(tmap_a, tmap_b, args, sched);
    }
    return cudaGetLastError();
  });
}

}  // namespace gb300

#ifdef SGEMM_PHASE_TRACE
extern "C" __attribute__((visibility("default"))) int sgemm_trace_configure(void* device_buffer,
                                                                           int64_t ctas) {
  uint64_t* buf = static_cast<uint64_t*>(device_buffer);
  if (buf == nullptr) ctas = 0;
  if (cudaMemcpyToSymbol(gb300::g_trace_buf, &buf, sizeof(buf)) != cudaSuccess ||
      cudaMemcpyToSymbol(gb300::g_trace_ctas, &ctas, sizeof(ctas)) != cudaSuccess)
    return 1;
  return 0;
}
#endif
