// sgemm_trace.h -- the tile kernel's optional phase trace.
//
// Compiled in only with -DSGEMM_PHASE_TRACE, into a library of its own
// (libsgemm_trace.so, built by _build.build_trace()); the product library
// carries none of it.  With it, every CTA of the tile kernel writes
// %globaltimer stamps of its phases into a device buffer that the host
// configures with sgemm_trace_configure(): up to kTraceSlots records of two
// 64-bit words per CTA, record i of CTA c at words (c * kTraceSlots + i) * 2:
//   word 0: global time in ns; word 1: kind << 56 | (a & 0xffffff) << 32 | b.
// Consumer thread 0 writes records [0, kTraceProducerSlot0), the producer
// warpgroup's first lane the rest; unused records stay as the host left
// them (zero).  dense_fp32_gemm_03_gb300/phase_trace.py reads the buffer.
#pragma once

#include <cstdint>

namespace gb300 {

enum TraceKind : uint32_t {
  kTrEntry = 1,          // kernel entry                       a = SM id
  kTrFirstStage = 2,     // the first ring stage has landed
  kTrKLoopEnd = 3,       // last k-tile of a unit computed       a = tile, b = k-tiles
  kTrStoreEnd = 4,       // whole tile stored to C               a = tile
  kTrPublishEnd = 5,     // split tile's partial published       a = tile, b = 1: then last
  kTrReduceEnd = 6,      // split tile reduced and stored        a = tile, b = partials read
  kTrExit = 7,           // consumer warps done
  kTrProducerIssued = 8, // producer: first copies issued
  kTrOwnerWait = 9,      // owner of a split tile done waiting    a = tile, b = 1: all arrived,
                         //                                       2: partials prefetched
  kTrProducerStart = 10, // producer warpgroup running (registers handed over)
  kTrFirstALanded = 11,  // producer: its first A slice is in shared memory
  kTrBarriersReady = 12, // thread 0 initialised the CTA's mbarriers
  kTrCtaSynced = 13,     // thread 0 passed the CTA barrier after that
};

constexpr int kTraceSlots = 64;
constexpr int kTraceProducerSlot0 = 56;

}  // namespace gb300

#ifdef SGEMM_PHASE_TRACE
// Points the trace at `device_buffer` (kTraceSlots * 16 bytes per CTA) for
// CTAs [0, ctas); NULL or ctas == 0 turns it off.  Returns 0, or nonzero if
// the device symbols could not be written.
extern "C" int sgemm_trace_configure(void* device_buffer, int64_t ctas);
#endif
