// sgemm_sched.cuh -- device-side walk of the work decomposition (Sched in
// sgemm_plan.h), shared by the FFMA tile kernel and the TF32 kernel.
#pragma once

#include <cstdint>

#include "sgemm_plan.h"

namespace gb300 {

// a / b for a >= 0, b > 0.  A 64-bit division is a long software sequence;
// the positions in the Stream-K iteration stream fit 31 bits for any size
// short of 2^31 k-tile iterations, where the 32-bit division suffices.
__device__ __forceinline__ int64_t div_nonneg(int64_t a, int32_t b) {
  if (a <= 0x7fffffffLL) return int64_t(uint32_t(a) / uint32_t(b));
  return a / b;
}

// One unit of work: a tile and a range [kb, ke) of its k-tiles.
struct Unit {
  int tile, kb, ke, t_sk;  // t_sk >= 0: index of a split (Stream-K) tile
};

// Walks the units of one CTA: whole tiles first, then its Stream-K share.
struct WorkIter {
  int dp_next;
  int64_t sk_pos, sk_end;

  __device__ __forceinline__ void init(const Sched& sc, int cta) {
    dp_next = cta;
    sk_pos = sk_end = 0;
    if (sc.sk_tiles > 0 && cta < sc.sk_ctas) {
      sk_pos = int64_t(cta) * sc.sk_base + min(cta, sc.sk_extra);
      sk_end = sk_pos + sc.sk_base + (cta < sc.sk_extra ? 1 : 0);
    }
  }

  __device__ __forceinline__ bool next(const Sched& sc, int ctas, Unit& u) {
    if (dp_next < sc.dp_tiles) {
      u.tile = dp_next;
      u.kb = 0;
      u.ke = sc.iters_per_tile;
      u.t_sk = -1;
      dp_next += ctas;
      return true;
    }
    if (sk_pos < sk_end) {
      u.t_sk = int(div_nonneg(sk_pos, sc.iters_per_tile));
      const int64_t start = int64_t(u.t_sk) * sc.iters_per_tile;
      u.kb = int(sk_pos - start);
      const int64_t left = sk_end - start;
      u.ke = left < sc.iters_per_tile ? int(left) : sc.iters_per_tile;
      u.tile = sc.dp_tiles + u.t_sk;
      sk_pos = start + u.ke;
      return true;
    }
    return false;
  }
};

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

// Walks the k-tiles of all units of one CTA in order.  The tile coordinates
// of the current unit are computed once per unit, not per k-tile: the
// producer issues two copies per k-tile and the divisions would otherwise
// sit on its path every time.
struct KCursor {
  WorkIter w;
  Unit u;
  int j;
  int tm, tn;  // tile row and column of u.tile
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

// CTA that owns iteration `i` of the Stream-K iteration stream.
__device__ __forceinline__ int sk_owner(const Sched& sc, int64_t i) {
  const int64_t big = int64_t(sc.sk_extra) * (sc.sk_base + 1);
  if (i < big) return int(div_nonneg(i, sc.sk_base + 1));
  return sc.sk_extra + int(div_nonneg(i - big, sc.sk_base));
}

}  // namespace gb300
