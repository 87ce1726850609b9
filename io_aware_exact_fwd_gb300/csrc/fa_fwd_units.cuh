// Work units of the persistent forward kernel (fa_fwd.cu): a unit
// is 256 query rows (two 128-row tiles) of one head and, for the split-KV
// forward, one range of its keys.  Each persistent CTA walks a fixed list of
// units; causal units are numbered heaviest first and dealt out in zigzag passes
// so that every SM gets a similar total.
#pragma once

#include "fa_internal.h"

namespace fa {

constexpr int kTiles = 2;                       // query tiles per unit
constexpr int kRowsPerCta = kTiles * kBlockQ;   // 256 query rows

// Key range of a launch and where its results go.  The plain forward has one
// split covering all Nk = N keys.  The split-KV forward cuts the key blocks into
// nsplit ranges of kbps blocks (split s: blocks [s kbps, (s+1) kbps)), aligns
// causal queries with the last keys (query i sees key j iff j <= i + coff,
// coff = Nk - Nq), and writes each split's normalised O (fp32) and LSE to
// o_part [nsplit, BH, Nq, d] and lse_part [nsplit, BH, Nq].
struct KeySplit {
  int Nk;
  int nsplit;
  int kbps;
  int coff;
  float* o_part;
  float* lse_part;
  int tail_from;  // work items >= tail_from are shared tiles (see item_at); INT_MAX: none
};

// K/V blocks [begin, begin + count) that query tile t of unit (u, split s) attends
// to; count = 0 if the tile is past the last query row.
struct KvSpan {
  int begin, count;
};
template <bool CAUSAL>
__device__ __forceinline__ KvSpan kv_span(int u, int t, int s, int N, const KeySplit& ks) {
  const int row0 = u * kRowsPerCta + t * kBlockQ;
  if (row0 >= N) return {0, 0};
  const int nkb = (ks.Nk + kBlockK - 1) / kBlockK;
  const int b = min(s * ks.kbps, nkb);
  int e = min(b + ks.kbps, nkb);
  // The tile's last row sees keys up to its index + coff.
  if (CAUSAL) e = min(e, (min(row0 + kBlockQ - 1, N - 1) + ks.coff) / kBlockK + 1);
  return {b, max(e - b, 0)};
}

// Dequantisation scales of the FP8 variant (unused by the bf16 one): per
// 64-row tile of each head, [BH, ntiles].
struct Fp8Scales {
  const float* sq;
  const float* sk;
  const float* sv;
  int ntiles;
};

// Work unit w -> (256-row query block u, head bh, key split s).  Causal units
// are numbered heaviest first (largest u first), so the zigzag assignment below
// hands every CTA a similar total.
template <bool CAUSAL>
__device__ __forceinline__ void decode_unit(int w, int nunits, int BH, int nsplit, int& u, int& bh, int& s) {
  if (CAUSAL) {
    const int per_u = BH * nsplit;
    u = nunits - 1 - w / per_u;
    const int r = w % per_u;
    bh = r / nsplit;
    s = r % nsplit;
  } else {
    u = w % nunits;
    const int r = w / nunits;
    s = r % nsplit;
    bh = r / nsplit;
  }
}

// k-th work item of CTA c out of G persistent CTAs: pass k covers items kG .. kG+G-1,
// in increasing CTA order on even passes and decreasing on odd ones.
__device__ __forceinline__ int unit_of(int k, int c, int G) { return k * G + ((k & 1) ? (G - 1 - c) : c); }

// A work item: a whole unit (ts = -1: query tile t of the unit goes to warpgroup /
// Q slot / TMEM buffer t, each with all its keys), or one query tile ts of a unit
// shared by both warpgroups, slot t taking the tile's key blocks t, t+2, t+4, ...
// and the two partial softmaxes merged at the end.  Shared tiles fill the last
// pass when the units do not divide evenly over the CTAs (non-causal only): the
// R leftover units become 2R shared tiles on 2R <= G CTAs, so that pass takes
// about half a unit's time instead of a whole one.
struct Item {
  int u, bh, sp, ts;
};
template <bool CAUSAL, bool TAIL>
__device__ __forceinline__ bool item_at(int w, int total, int nunits, int BH, const KeySplit& ks, Item& it) {
  int wu = w;
  it.ts = -1;
  if (TAIL && w >= ks.tail_from) {  // only the kernel built for shared tiles has them
    wu = ks.tail_from + (w - ks.tail_from) / 2;
    it.ts = (w - ks.tail_from) & 1;
  }
  if (wu >= total) return false;
  decode_unit<CAUSAL>(wu, nunits, BH, ks.nsplit, it.u, it.bh, it.sp);
  return true;
}

// Query rows and key blocks of slot t for an item: rows row0 .. row0 + 127, key
// blocks begin, begin + step, ... (count of them).
struct SlotWork {
  int row0, begin, count, step;
};
template <bool CAUSAL>
__device__ __forceinline__ SlotWork slot_work(const Item& it, int t, int N, const KeySplit& ks) {
  if (it.ts < 0) {
    const KvSpan s = kv_span<CAUSAL>(it.u, t, it.sp, N, ks);
    return {it.u * kRowsPerCta + t * kBlockQ, s.begin, s.count, 1};
  }
  const KvSpan s = kv_span<CAUSAL>(it.u, it.ts, it.sp, N, ks);
  return {it.u * kRowsPerCta + it.ts * kBlockQ, s.begin + t, (s.count + 1 - t) / 2, 2};
}


}  // namespace fa
