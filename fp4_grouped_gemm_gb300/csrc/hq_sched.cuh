// hq_sched.cuh -- device-side tile scheduler for dense, grouped-contiguous and
// grouped-masked GEMMs.  Every role of a CTA decodes the same tile sequence
// from a small table built once per CTA in shared memory by one warp:
//   contiguous  (cuDNN frontend "Grouped GEMM + dGLU (SM100)": groups
//               contiguous in M, padded_offsets = cumulative aligned ends):
//               sanitised offsets; m-tile -> group by binary search.
//   masked      (HALOps group_masked_gemm: masked_m valid rows per expert in
//               a [E * max_m, K] layout): per-expert clamped counts and an
//               exclusive prefix of their 128-row tile counts, so only tiles
//               that hold valid rows are ever scheduled.
//   segments    (HALOps group_contiguous_gemm: a per-row expert index, groups
//               packed without padding): a list, built by a preparatory
//               kernel, of (128-row block, expert, first row, end row) runs;
//               a block that holds rows of several experts is computed once
//               per expert and each pass writes only that expert's rows.
// Tile t covers rows [row0, row0 + 128) of one group and columns
// [n0, n0 + BN); n varies fastest.
#pragma once

#include <stdint.h>

#include "hq_ptx.cuh"

namespace hq {

enum Sched : int { kDense = 0, kContig = 1, kMasked = 2, kSegments = 3 };

constexpr int kBM = 128;
constexpr int kMaxGroups = 1024;

struct GroupSched {
  const int32_t* group_info;  // contig: padded_offsets[L]; masked: masked_m[E];
                              // segments: [count, pad x3, {row0, g, lo, hi} x count]
  int64_t a_rows;             // rows of A / out
  int64_t max_m;              // masked only
  int groups;
  int sched;
  uint32_t* status;
};

struct TileInfo {
  int g;
  int64_t row0;
  int rows_valid;  // rows [row0, row0 + rows_valid) may be written ...
  int row_lo;      // ... from row0 + row_lo on (segments only; 0 otherwise)
  int n0;
};

// Per-CTA schedule state, built once in shared memory.
struct Schedule {
  int64_t total_tiles;
  int n_tiles;
  const int32_t* tab0;  // contig: sanitised offsets; masked: tile-prefix
  const int32_t* tab1;  // masked: clamped counts
};

__device__ __forceinline__ TileInfo decode_tile(const GroupSched& p, const Schedule& s, int64_t t,
                                                int BN) {
  TileInfo ti;
  const int64_t mt = t / s.n_tiles;
  ti.n0 = static_cast<int>(t - mt * s.n_tiles) * BN;
  ti.row_lo = 0;
  if (p.sched == kSegments) {
    const int4 sg = __ldg(reinterpret_cast<const int4*>(p.group_info) + 1 + mt);
    ti.row0 = sg.x;
    ti.g = sg.y;
    ti.row_lo = sg.z;
    ti.rows_valid = sg.w;
  } else if (p.sched == kDense) {
    ti.g = 0;
    ti.row0 = mt * kBM;
    const int64_t rem = p.a_rows - ti.row0;
    ti.rows_valid = rem < kBM ? static_cast<int>(rem) : kBM;
  } else if (p.sched == kContig) {
    const int64_t r0 = mt * kBM;
    int lo = 0, hi = p.groups - 1;  // first g with off[g] > r0
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (s.tab0[mid] > r0) hi = mid; else lo = mid + 1;
    }
    ti.g = lo;
    ti.row0 = r0;
    const int64_t rem = static_cast<int64_t>(s.tab0[lo]) - r0;
    ti.rows_valid = rem < kBM ? static_cast<int>(rem) : kBM;
  } else {
    int lo = 0, hi = p.groups - 1;  // last e with prefix[e] <= mt
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s.tab0[mid] <= mt) lo = mid; else hi = mid - 1;
    }
    ti.g = lo;
    const int64_t local = mt - s.tab0[lo];
    ti.row0 = static_cast<int64_t>(lo) * p.max_m + local * kBM;
    const int64_t rem = static_cast<int64_t>(s.tab1[lo]) - local * kBM;
    ti.rows_valid = rem < kBM ? static_cast<int>(rem) : kBM;
  }
  return ti;
}

// Warp-cooperative construction of the group table (one warp, L <= 1024).
// unit: rows per scheduled m-tile of the masked layout (128, or 256 for the
// two-CTA pairs); the other layouts use 128.
__device__ inline void build_table(const GroupSched& p, int32_t* tab0, int32_t* tab1, int lane,
                            int64_t* total_mtiles, int unit = kBM) {
  if (p.sched == kDense) {
    if (lane == 0) *total_mtiles = (p.a_rows + kBM - 1) / kBM;
    return;
  }
  if (p.sched == kSegments) {
    if (lane == 0) *total_mtiles = __ldg(p.group_info);
    return;
  }
  bool bad = false;
  if (p.sched == kContig) {
    // sanitised[g] = min(prefix_max(round_down_128(off[h]), h <= g), round_down_128(a_rows))
    const int32_t row_cap = static_cast<int32_t>((p.a_rows / kBM) * kBM);
    int32_t carry = 0;
    for (int base = 0; base < p.groups; base += 32) {
      const int g = base + lane;
      int32_t v = 0;
      if (g < p.groups) {
        const int32_t raw = __ldg(p.group_info + g);
        v = raw < 0 ? 0 : (raw / kBM) * kBM;
        if (raw < 0 || raw % kBM != 0 || raw > p.a_rows) bad = true;
        if (g > 0 && raw < __ldg(p.group_info + g - 1)) bad = true;
        if (v > row_cap) v = row_cap;
      }
      v = v > carry ? v : carry;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t u = __shfl_up_sync(0xFFFFFFFFu, v, o);
        if (lane >= o && u > v) v = u;
      }
      if (g < p.groups) tab0[g] = v;
      carry = __shfl_sync(0xFFFFFFFFu, v, 31);
    }
    if (lane == 0) *total_mtiles = carry / kBM;
    if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) atomicOr(p.status, HQ_STATUS_BAD_OFFSETS);
  } else {
    int32_t carry = 0;
    for (int base = 0; base < p.groups; base += 32) {
      const int e = base + lane;
      int32_t cnt = 0;
      if (e < p.groups) {
        const int32_t raw = __ldg(p.group_info + e);
        cnt = raw;
        if (raw < 0) { cnt = 0; bad = true; }
        if (raw > p.max_m) { cnt = static_cast<int32_t>(p.max_m); bad = true; }
        tab1[e] = cnt;
      }
      const int32_t tiles = (cnt + unit - 1) / unit;
      int32_t incl = tiles;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += u;
      }
      if (e < p.groups) tab0[e] = carry + incl - tiles;  // exclusive prefix
      carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (lane == 0) *total_mtiles = carry;
    if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) atomicOr(p.status, HQ_STATUS_MASK_CLAMPED);
  }
}

}  // namespace hq
