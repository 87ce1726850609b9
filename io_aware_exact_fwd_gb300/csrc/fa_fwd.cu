// Exact attention forward, bf16 in / bf16 out, fp32 logsumexp, for sm_103a.
//
// Method ("FlashAttention-Skalierung, Multi-GPU-Training und
// Gewichtsquantisierung", section 1; "FlashAttention-2 (DE)", sections
// "Hintergrund" and "Technische Architektur und Funktionsprinzipien"): the
// N x N score matrix is never materialised.  Each CTA owns query rows of one
// head (outer loop over Q blocks, parallel over the sequence as well as over
// batch and heads) and streams the K/V blocks of that head through shared
// memory (inner loop), keeping a running row maximum m and row sum l (online
// softmax).  The single division by l happens once, after the inner loop.
//
// GB300 mapping of the pages' ideas:
//  * Persistent CTAs: one per SM, each walking a fixed list of work units
//    (256 query rows of one head); causal units are ordered heaviest first and
//    dealt out in zigzag passes so that every SM gets a similar total.  The K/V
//    stream, the TMEM buffers and the barrier phases simply continue from one
//    unit to the next, so a unit's Q load, first Q K^T and epilogue overlap the
//    neighbouring unit's main loop instead of costing a CTA launch each.
//  * TMA copies ("Asynchrone Datenübertragung (TMA)") move the Q tiles once per
//    unit and K_j, V_j through a ring of shared-memory slots guarded by
//    full/empty mbarriers.
//  * Warp specialisation ("Warp-Spezialisierung"): warp 8 issues the K/V copies,
//    warp 10 the Q copies, one thread of warp 9 issues tcgen05 MMAs, and two
//    softmax warpgroups (warps 0-3 and 4-7, one thread per query row = one TMEM
//    lane) each own one of the unit's two 128-row query tiles.  While one warpgroup exponentiates its scores the
//    tensor core runs the other tile's P V and Q K^T ("Nahtloses Interleaving von
//    Operationen" on the FlashAttention-3 page: matmul and softmax overlap).
//  * Per tile, S = Q K_j^T accumulates in TMEM; P is written back over S as packed
//    bf16 and feeds the P V MMA straight from TMEM, so P never touches shared
//    memory.  TMEM holds S_a, S_b (128 columns each) and O_a, O_b (d columns
//    each): all 512 columns at d = 128.
//  * The O accumulators stay in TMEM for the whole inner loop.  O is rescaled only
//    when a row maximum grows by more than 2^8 (the pages' single rescaling at
//    the end of the loop, taken one step further): until then exponentials are taken against the
//    stale maximum, which keeps O and l consistent and the final O/l exact.
//
// Every mbarrier wait is bounded (see fa_device.cuh); on expiry the CTA sets a
// device error word, drains its own in-flight copies, frees TMEM and exits.
#include <limits.h>
#include <math.h>

#include "fa_device.cuh"
#include "fa_fwd_units.cuh"
#include "fa_internal.h"

namespace fa {
namespace {
constexpr int kThreads = 384;                   // warps 0-7 softmax (2 groups), 8 K/V TMA, 9 MMA, 10 Q TMA, 11 spare
constexpr int kWarpLoad = 8;
constexpr int kWarpMma = 9;
constexpr int kWarpLoadQ = 10;
// Launch budget: 168 registers x 384 threads.  Softmax warpgroups take 216 each
// (128 live scores per thread), the TMA/MMA warpgroup gives back down to 72:
// 2 x 128 x 216 + 128 x 72 = 168 x 384.
constexpr uint32_t kRegsSoftmax = 216;
constexpr uint32_t kRegsControl = 72;
constexpr uint32_t kRegsNeeded = 2 * 128 * kRegsSoftmax + 128 * kRegsControl;
static_assert(kRegsNeeded <= 65536, "register split exceeds the SM register file");
constexpr uint32_t kTmemCols = 512;
// A key block is exponentiated against the running maximum without computing
// its own; the result is kept if the block's row sum is at most this bound
// (then every P <= 2^16, far from fp32 overflow even after accumulation).
constexpr float kSpeculationSumBound = 65536.0f;
// FP8 keeps a per-block maximum and moves its reference only when a block's
// maximum exceeds it by more than 8.75 (log2 units), so P <= 2^8.75 = 430.5 < 448,
// inside e4m3's range.
constexpr float kRescaleThreshold = 8.75f;
constexpr float kLn2 = 0.69314718055994530942f;

// Sites recorded in the error word when a wait expires.
enum : uint32_t {
  kSiteLoadEmpty = 0x101,
  kSiteLoadQ = 0x102,
  kSiteMmaQ = 0x201,
  kSiteMmaK = 0x202,
  kSiteMmaP = 0x203,
  kSiteMmaV = 0x204,
  kSiteSoftS = 0x301,
  kSiteSoftO = 0x302,
  kSiteEpi = 0x303,
  kSiteSoftKV = 0x304,
};

// FP8 selects the e4m3 variant: Q, K and V tiles of e4m3 codes (V transposed,
// keys contiguous), kind::f8f6f4 MMAs, per-tile dequantisation scales folded
// into the softmax, P quantised to e4m3 in TMEM, bf16 O.
template <int D, bool FP8>
struct FwdCfg {
  static constexpr int kRowBytes = D * (FP8 ? 1 : 2);       // one row of a Q, K or V tile
  static constexpr int kBoxes = (kRowBytes + 127) / 128;    // TMA boxes per row, 128 bytes wide (64 for FP8 d = 64)
  static constexpr int kBoxBytes = kBlockK * 128;           // 16 KB: 128 rows x 128 bytes
  // FP8 at d = 64: Q and K rows are 64 bytes, staged with the 64-byte swizzle.
  static constexpr bool kSw64 = kRowBytes == 64;
  static constexpr int kTileBytes = kBlockK * kRowBytes;    // one Q, K or V tile
  static constexpr int kKSteps = kRowBytes / 32;            // MMA K-steps of 32 bytes over d
  static constexpr int kOBytes = kBlockQ * D * 2;           // bf16 O staging of one query tile
  static constexpr int kOBoxes = D * 2 / 128;               // 128-byte boxes per bf16 O row
  static constexpr int kSlots = kTileBytes == 32768 ? 4 : 8;
  static constexpr int kQOff = 0;                           // Q_a, Q_b (one tile each)
  static constexpr int kOOff = kTiles * kTileBytes;         // O staging, shared by both tiles in turn
  static constexpr int kRingOff = kOOff + kOBytes;
  static constexpr int kBarOff = kRingOff + kSlots * kTileBytes;
  // q_full[2], q_empty[2], full[kSlots], empty[kSlots], s_full[2], p_full[2], o_done[2], epi[2], stg, drain,
  // shared-tile swap
  static constexpr int kNumBars = 2 + 2 + 2 * kSlots + 2 + 2 + 2 + 2 + 1 + 1 + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + slack to align the base to 1024
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  // Who waits for the K/V ring inside a whole unit.  The single MMA-issuing thread
  // paces the tensor pipe: each instruction it runs between two MMA bursts leaves
  // the pipe idle, while the softmax warpgroups wait for S more than half the time.
  // For bf16 at d = 128 the softmax warpgroups therefore check that V_j and K_{j+1}
  // have landed before signalling P, and the MMA thread waits on P alone.  With
  // FP8 or d = 64 the MMA bursts are shorter and the softmax chain is the longer
  // one, so there the MMA thread keeps those waits (measured both ways); so does
  // the split-KV build (see fwd_kernel), whose decode-shaped launches are bound by
  // HBM: there P_t V_j must not wait for K_{j+1} to land.
  static constexpr bool kRingWaitsInSoftmax = !FP8 && D == 128;
  static __device__ __forceinline__ uint32_t col_s(int t) { return 128u * static_cast<uint32_t>(t); }
  static __device__ __forceinline__ uint32_t col_o(int t) { return 256u + D * static_cast<uint32_t>(t); }
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& wc, uint32_t site) {
  const bool ok = mbar_wait(bar, parity, wc, site);
  return __all_sync(0xffffffffu, ok);
}
// The softmax warpgroups' wait for S: they wait more than half of each block, on
// the same SM sub-partitions as the MMA-issuing warp, so their polls suspend.
__device__ __forceinline__ bool warp_wait_suspend(uint64_t* bar, uint32_t parity, const WaitCtl& wc, uint32_t site) {
  const bool ok = mbar_wait_suspend(bar, parity, wc, site, 20000u);
  return __all_sync(0xffffffffu, ok);
}

// TAIL: the build for launches whose last pass is dealt out as shared tiles
// (item_at); only the non-causal, whole-key forward has one.  Every other launch
// uses the build without that code.
template <int D, bool CAUSAL, bool FP8, bool SPLIT, bool TAIL = false>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
               float* __restrict__ lse, int N, int H, int BH, int nunits, float scale_log2,
               unsigned int* err_word, unsigned long long wait_ns, int fault, Fp8Scales f8, KeySplit ks) {
  static_assert(!(SPLIT && FP8), "the split-KV variant is bf16 only");
  static_assert(!(TAIL && (CAUSAL || SPLIT)), "shared tiles only for the non-causal, whole-key forward");
  using C = FwdCfg<D, FP8>;
  constexpr bool kRingWaitsInSoftmax = C::kRingWaitsInSoftmax && !SPLIT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::kQOff;
  uint8_t* sO = smem + C::kOOff;
  uint8_t* sRing = smem + C::kRingOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* bar_q = bars;                    // [2] per tile: Q landed
  uint64_t* bar_qe = bar_q + 2;              // [2] per tile: last Q K^T of a unit done (Q slot free)
  uint64_t* bar_full = bar_qe + 2;           // [kSlots]
  uint64_t* bar_empty = bar_full + C::kSlots;
  uint64_t* bar_s = bar_empty + C::kSlots;   // [2] per tile: S ready
  uint64_t* bar_p = bar_s + 2;               // [2] per tile: P written
  uint64_t* bar_o = bar_p + 2;               // [2] per tile: last P V of a unit done
  uint64_t* bar_epi = bar_o + 2;             // [2] per tile: O staged in shared memory
  uint64_t* bar_stg = bar_epi + 2;           // O staging buffer read out by the previous store
  uint64_t* bar_drain = bar_stg + 1;
  uint64_t* bar_xm = bar_drain + 1;          // shared tile: both warpgroups stored their (m, l)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Persistent CTAs: CTA c takes units unit_of(0, c, G), unit_of(1, c, G), ...
  const int total = nunits * BH * ks.nsplit;
  const int G = static_cast<int>(gridDim.x);
  const int cta = static_cast<int>(blockIdx.x);

  if (threadIdx.x == 0) {
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(&bar_q[t], 1);
      mbar_init(&bar_qe[t], 1);
      mbar_init(&bar_s[t], 1);
      mbar_init(&bar_p[t], 4);
      mbar_init(&bar_o[t], 1);
      mbar_init(&bar_epi[t], 4);
    }
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    mbar_init(bar_stg, 1);
    mbar_init(bar_drain, 1);
    mbar_init(bar_xm, 8);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) tmem_alloc(tmem_slot, kTmemCols);
  if (warp == kWarpLoad && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_o);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, err_word, wait_ns};

  if (warp >= 8) {
   // Control warpgroup: gives registers back to the softmax warpgroups.
   regs_decrease<kRegsControl>();
   if (warp == kWarpLoad) {
    // --------------------------------------------------------- K/V TMA producer
    if (lane == 0) {
      // Ring order = MMA first-use order: K0, V0, K1, V1, ... of unit after unit.
      int issued = 0;
      bool ok = true;
      auto push = [&](const CUtensorMap* tm, int j, int bh) -> bool {
        const int slot = issued % C::kSlots;
        const uint32_t ph = (issued / C::kSlots) & 1;
        if (!mbar_wait(&bar_empty[slot], ph ^ 1, wc, kSiteLoadEmpty)) return false;
        if (fault == 1 && tm == &tm_k && j == 1) return false;  // test-only: K block 1 never arrives
        mbar_arrive_expect_tx(&bar_full[slot], C::kTileBytes);
        uint8_t* dst = sRing + slot * C::kTileBytes;
        if (FP8 && tm == &tm_v) {
          // V^T codes [d rows][keys]: one 128-key x d-row box at key offset j * 128.
          tma_load_4d(dst, tm, &bar_full[slot], j * kBlockK, 0, bh % H, bh / H);
        } else {
#pragma unroll
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_4d(dst + b * C::kBoxBytes, tm, &bar_full[slot], b * kBoxCols, j * kBlockK, bh % H, bh / H);
        }
        ++issued;
        return true;
      };
      for (int k = 0; ok; ++k) {
        Item it;
        if (!item_at<CAUSAL, TAIL>(unit_of(k, cta, G), total, nunits, BH, ks, it)) break;
        // Every block of the item once, in order: for a whole unit the blocks of its
        // longer tile (both tiles start at the split's first block), for a shared
        // tile all of the tile's blocks.
        const KvSpan a = kv_span<CAUSAL>(it.u, it.ts < 0 ? 0 : it.ts, it.sp, N, ks);
        const int n_blocks = it.ts < 0 ? max(a.count, kv_span<CAUSAL>(it.u, 1, it.sp, N, ks).count) : a.count;
        for (int j = 0; ok && j < n_blocks; ++j) {
          ok = push(&tm_k, a.begin + j, it.bh);
          if (ok) ok = push(&tm_v, a.begin + j, it.bh);
        }
      }
      if (!ok) {  // drain: the last (up to kSlots) issued copies may still be landing
        for (int t = max(0, issued - C::kSlots); t < issued; ++t)
          mbar_wait_drain(&bar_full[t % C::kSlots], (t / C::kSlots) & 1, wait_ns);
      }
    }
    __syncwarp();
   } else if (warp == kWarpLoadQ) {
    // ----------------------------------------------------------- Q TMA producer
    // Q_t of the next unit loads as soon as the current unit's last Q_t K^T MMA
    // has completed, so it overlaps that unit's last P V and epilogue.
    if (lane == 0) {
      int nload[kTiles] = {0, 0};
      bool ok = true;
      for (int k = 0; ok; ++k) {
        Item it;
        if (!item_at<CAUSAL, TAIL>(unit_of(k, cta, G), total, nunits, BH, ks, it)) break;
        for (int t = 0; ok && t < kTiles; ++t) {
          const SlotWork sw = slot_work<CAUSAL>(it, t, N, ks);  // a shared tile loads into both slots
          if (sw.count == 0) continue;
          if (nload[t] > 0 && !(ok = mbar_wait(&bar_qe[t], (nload[t] - 1) & 1, wc, kSiteLoadQ))) break;
          mbar_arrive_expect_tx(&bar_q[t], C::kTileBytes);
#pragma unroll
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_4d(sQ + t * C::kTileBytes + b * C::kBoxBytes, &tm_q, &bar_q[t], b * kBoxCols, sw.row0,
                        it.bh % H, it.bh / H);
          ++nload[t];
        }
      }
      if (!ok) {  // drain the Q copies that may still be landing
        for (int t = 0; t < kTiles; ++t)
          if (nload[t] > 0) mbar_wait_drain(&bar_q[t], (nload[t] - 1) & 1, wait_ns);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk =
          FP8 ? idesc_e4m3_f32(kBlockQ, kBlockK, 0, 0) : idesc_bf16_f32(kBlockQ, kBlockK, 0, 0);
      constexpr uint32_t idesc_pv = FP8 ? idesc_e4m3_f32(kBlockQ, D, 0, 0) : idesc_bf16_f32(kBlockQ, D, 0, 1);
      const uint32_t q_addr = smem_u32(sQ);
      const uint32_t ring_addr = smem_u32(sRing);
      int item = 0;               // ring index of the next K or V block to consume
      int nq_seen[kTiles] = {0, 0};  // Q tiles consumed so far (bar_q phase)
      int np[kTiles] = {0, 0};       // P blocks consumed so far (bar_p phase)
      bool ok = true;
      Item shared_item{0, 0, 0, -1};

      // Base descriptors; every MMA operand below is one of these advanced by a
      // compile-time byte offset (a single 32-bit add on the issuing thread).
      // K-major, SBO = 8 rows x the row (128 B, or 64 B for FP8 at d = 64).
      const uint64_t qdesc = C::kSw64 ? sdesc_sw64(q_addr) : sdesc_sw128(q_addr, 16, 1024);
      const uint64_t kdesc = C::kSw64 ? sdesc_sw64(ring_addr) : sdesc_sw128(ring_addr, 16, 1024);  // a ring slot
      // bf16: V is MN-major (LBO = one box); FP8: V^T is K-major like K.
      const uint64_t vdesc = sdesc_sw128(ring_addr, FP8 ? 16 : C::kBoxBytes, 1024);

      // S_t = Q_t K^T : both operands K-major (d contiguous), 16 d-columns per MMA.
      auto qk = [&](int t, int slot) {
        const uint64_t qd = sdesc_add(qdesc, t * C::kTileBytes);
        const uint64_t kd = sdesc_add(kdesc, slot * C::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < C::kKSteps; ++kk) {
          const uint32_t off = (kk / 4) * C::kBoxBytes + (kk % 4) * 32;
          if constexpr (FP8)
            mma_e4m3_ss(tmem + C::col_s(t), sdesc_add(qd, off), sdesc_add(kd, off), idesc_qk, kk > 0 ? 1u : 0u);
          else
            mma_bf16_ss(tmem + C::col_s(t), sdesc_add(qd, off), sdesc_add(kd, off), idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bar_s[t]);
      };
      // O_t += P_t V : A = P from TMEM (2 bf16 per column), B = V tile, MN-major
      // (d contiguous): 8 key rows per 1024-byte swizzle atom (SBO), 64 d-columns
      // per TMA box (LBO = one box).
      auto pv = [&](int t, int slot, bool accumulate) {
        const uint64_t vd = sdesc_add(vdesc, slot * C::kTileBytes);
        if constexpr (FP8) {
          // A = P (e4m3, 4 per TMEM column), 32 keys per MMA; B = V^T K-major, 32 key bytes per step.
#pragma unroll
          for (int kk = 0; kk < kBlockK / 32; ++kk)
            mma_e4m3_ts(tmem + C::col_o(t), tmem + C::col_s(t) + kk * 8, sdesc_add(vd, kk * 32), idesc_pv,
                        (accumulate || kk > 0) ? 1u : 0u);
        } else {
#pragma unroll
          for (int kk = 0; kk < kBlockK / 16; ++kk)
            mma_bf16_ts(tmem + C::col_o(t), tmem + C::col_s(t) + kk * 8, sdesc_add(vd, kk * 16 * 128), idesc_pv,
                        (accumulate || kk > 0) ? 1u : 0u);
        }
      };

      for (int k = 0; ok; ++k) {
        Item itm;
        if (!item_at<CAUSAL, TAIL>(unit_of(k, cta, G), total, nunits, BH, ks, itm)) break;
        if (TAIL && itm.ts >= 0) {  // a shared tile: always the CTA's last item (below)
          shared_item = itm;
          break;
        }
        const int u = itm.u;
        const int nq[kTiles] = {kv_span<CAUSAL>(u, 0, itm.sp, N, ks).count, kv_span<CAUSAL>(u, 1, itm.sp, N, ks).count};
        const int n_max = max(nq[0], nq[1]);
        if (n_max == 0) continue;  // an empty key split: nothing was loaded for it
        // Prologue: S_a = Q_a K_0^T, S_b = Q_b K_0^T.  S_t is free: the previous
        // unit's last P_t V MMA, which read P_t from it, was issued earlier.
        {
          const int slot = item % C::kSlots;
          ok = mbar_wait(&bar_full[slot], (item / C::kSlots) & 1, wc, kSiteMmaK);
          for (int t = 0; ok && t < kTiles; ++t) {
            if (nq[t] == 0) continue;
            ok = mbar_wait(&bar_q[t], nq_seen[t] & 1, wc, kSiteMmaQ);
            if (!ok) break;
            ++nq_seen[t];
            tc_fence_after();
            qk(t, slot);
            if (nq[t] == 1) mma_commit(&bar_qe[t]);
          }
          if (!ok) break;
          mma_commit(&bar_empty[slot]);
          ++item;
        }
        // With kRingWaitsInSoftmax, V_j and K_{j+1} are not waited for here: a
        // softmax warpgroup signals P_t only once both have landed, so the wait on
        // P_t covers them and this thread does one wait per tile and block.
        for (int j = 0; ok && j < n_max; ++j) {
          const int slot_v = item % C::kSlots;
          if constexpr (!kRingWaitsInSoftmax) {
            ok = mbar_wait(&bar_full[slot_v], (item / C::kSlots) & 1, wc, kSiteMmaV);
            if (!ok) break;
          }
          ++item;
          const bool has_next = j + 1 < n_max;
          const int slot_k = item % C::kSlots;
          const uint32_t par_k = (item / C::kSlots) & 1;
          if (has_next) ++item;
          bool k_ready = kRingWaitsInSoftmax;
          for (int t = 0; ok && t < kTiles; ++t) {
            if (j >= nq[t]) continue;
            ok = mbar_wait(&bar_p[t], np[t] & 1, wc, kSiteMmaP);
            if (!ok) break;
            ++np[t];
            tc_fence_after();
            // The first P V of a unit overwrites O_t: the softmax warpgroup read the
            // previous unit's O_t out of TMEM before it wrote this P_t.
            pv(t, slot_v, j > 0);
            if (j + 1 == nq[t]) mma_commit(&bar_o[t]);
            if (j + 1 < nq[t]) {
              if (!k_ready) {
                ok = mbar_wait(&bar_full[slot_k], par_k, wc, kSiteMmaK);
                if (!ok) break;
                tc_fence_after();
                k_ready = true;
              }
              qk(t, slot_k);
              if (j + 2 == nq[t]) mma_commit(&bar_qe[t]);
            }
          }
          if (!ok) break;
          mma_commit(&bar_empty[slot_v]);
          if (has_next) {
            if (!k_ready) {  // no tile needed K_{j+1} (cannot happen for n_max > j + 1, kept for safety)
              ok = mbar_wait(&bar_full[slot_k], par_k, wc, kSiteMmaK);
              if (!ok) break;
            }
            mma_commit(&bar_empty[slot_k]);
          }
        }
      }
      if (TAIL && ok && shared_item.ts >= 0) {
        // A shared tile: slot t takes key blocks t, t + 2, ... of the tile (Q loaded
        // into both slots).  K_j is ring item i0 + 2j and V_j item i0 + 2j + 1;
        // they are consumed slightly out of order (K_{j+2} before V_{j+1}), which
        // the ring of at least 4 slots, filled in order, always allows.
        const Item& itm = shared_item;
        const int n = kv_span<CAUSAL>(itm.u, itm.ts, itm.sp, N, ks).count;  // 0: past the last query row
        const int i0 = item;
        auto wait_item = [&](int i, uint32_t site) {
          return mbar_wait(&bar_full[i % C::kSlots], (i / C::kSlots) & 1, wc, site);
        };
        for (int t = 0; ok && t < kTiles && t < n; ++t) {  // S_t = Q K_t^T
          if (!(ok = wait_item(i0 + 2 * t, kSiteMmaK))) break;
          if (!(ok = mbar_wait(&bar_q[t], nq_seen[t] & 1, wc, kSiteMmaQ))) break;
          tc_fence_after();
          qk(t, (i0 + 2 * t) % C::kSlots);
          if (t + 2 >= n) mma_commit(&bar_qe[t]);
          mma_commit(&bar_empty[(i0 + 2 * t) % C::kSlots]);
        }
        for (int j = 0; ok && j < n; ++j) {
          const int t = j & 1;
          if (!(ok = wait_item(i0 + 2 * j + 1, kSiteMmaV))) break;
          // (np indexed by constants only: a runtime index would put it in local memory)
          if (!(ok = mbar_wait(&bar_p[t], (t ? np[1] : np[0]) & 1, wc, kSiteMmaP))) break;
          if (t) ++np[1]; else ++np[0];
          tc_fence_after();
          pv(t, (i0 + 2 * j + 1) % C::kSlots, j >= 2);  // slot t's first block (j = t) overwrites O_t
          mma_commit(&bar_empty[(i0 + 2 * j + 1) % C::kSlots]);
          if (j + 2 >= n) {
            mma_commit(&bar_o[t]);
          } else {  // S_t = Q K_{j+2}^T, the slot's next block
            if (!(ok = wait_item(i0 + 2 * j + 4, kSiteMmaK))) break;
            tc_fence_after();
            qk(t, (i0 + 2 * j + 4) % C::kSlots);
            if (j + 4 >= n) mma_commit(&bar_qe[t]);
            mma_commit(&bar_empty[(i0 + 2 * j + 4) % C::kSlots]);
          }
        }
      }
      // Every issued MMA must finish before TMEM is released.
      mma_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0, wait_ns);
    }
    __syncwarp();
   }
  } else {
    regs_increase<kRegsSoftmax>();
    // -------------------------------------------- softmax warpgroups (0-3, 4-7)
    const int t = warp >> 2;                 // query tile of this warpgroup
    const int row = threadIdx.x & 127;       // tile row == TMEM lane
    const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t col_s = C::col_s(t);
    const uint32_t col_o = C::col_o(t);
    uint32_t scnt = 0;             // S blocks consumed so far (bar_s phase)
    uint32_t oc0 = 0, oc1 = 0;     // items in which slot 0 / slot 1 had keys (bar_o, bar_epi phases)
    uint32_t nepi = 0;             // epilogues before this item's (bar_stg phase)
    int ring0 = 0;                 // K/V ring items of the whole units before this one
    bool ok = true;
    // What the merge epilogue of a shared tile needs once the item loop is left.
    struct {
      bool pending = false;
      float m = 0.f, l = 0.f, svmax = 1.f;
      int bh = 0, qrow0 = 0;
      uint32_t ph0 = 0, ph1 = 0, epi_index = 0;
    } sh;
    for (int k = 0; ok; ++k) {
      Item itm;
      if (!item_at<CAUSAL, TAIL>(unit_of(k, cta, G), total, nunits, BH, ks, itm)) break;
      const int bh = itm.bh, sp = itm.sp;
      const bool shared = itm.ts >= 0;  // both warpgroups on one tile (see item_at)
      const SlotWork sw = slot_work<CAUSAL>(itm, t, N, ks);
      const bool has0 = slot_work<CAUSAL>(itm, 0, N, ks).count > 0;
      const bool has1 = slot_work<CAUSAL>(itm, 1, N, ks).count > 0;
      const int nkt = sw.count;
      // A whole unit takes 2 n_max ring items: K_0, then V_j and K_{j+1} per block j.
      int n_max = 0, ring_unit = 0;
      if constexpr (kRingWaitsInSoftmax) {
        n_max = shared ? 0 : max(slot_work<CAUSAL>(itm, 0, N, ks).count, slot_work<CAUSAL>(itm, 1, N, ks).count);
        ring_unit = ring0;
        ring0 += 2 * n_max;
      }
      const uint32_t ph0 = oc0, ph1 = oc1;          // this item's phases of slot 0 and slot 1
      const uint32_t ph_t = t == 0 ? ph0 : ph1;     // own slot
      oc0 += has0 ? 1u : 0u;
      oc1 += has1 ? 1u : 0u;
      // Epilogues run in (item, tile) order through one staging buffer; a shared
      // tile has one.
      const uint32_t epi_index = nepi + ((!shared && t == 1 && has0) ? 1u : 0u);
      nepi += shared ? (has0 ? 1u : 0u) : (has0 ? 1u : 0u) + (has1 ? 1u : 0u);
      const int qrow0 = sw.row0;
      const int qrow = qrow0 + row;
      if (nkt == 0) {
        // No key of this split is visible to the tile: an empty partial.
        if (SPLIT && qrow < N)
          ks.lse_part[(static_cast<size_t>(sp) * BH + bh) * N + qrow] = -INFINITY;
        continue;
      }
      float m_used = -INFINITY;  // running maximum in log2 units (possibly stale, see header)
      float l = 0.f;
      // FP8: the row's Q scale joins the score scale; V scales are folded into P
      // relative to the head's largest V scale (so P stays <= 256 in e4m3) and
      // undone in the epilogue.
      float crow = scale_log2, inv_svmax = 1.f, svmax = 1.f;
      const float* skh = nullptr;
      const float* svh = nullptr;
      if constexpr (FP8) {
        const size_t hb = static_cast<size_t>(bh) * f8.ntiles;
        skh = f8.sk + hb;
        svh = f8.sv + hb;
        float mxv = 0.f;
        for (int i = lane; i < f8.ntiles; i += 32) mxv = fmaxf(mxv, svh[i]);
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) mxv = fmaxf(mxv, __shfl_xor_sync(0xffffffffu, mxv, m));
        svmax = mxv;
        inv_svmax = 1.f / mxv;
        crow = scale_log2 * (qrow < N ? f8.sq[hb + qrow / 64] : 1.f);
      }
      // FP8: the K and V tile scales of the next key block, loaded one block ahead
      // so that no global load sits between S becoming ready and the exponentials.
      float nsk[2] = {1.f, 1.f}, nsv[2] = {svmax, svmax};
      auto fetch_scales = [&](int jj) {
        if constexpr (FP8) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int kt = 2 * (sw.begin + sw.step * jj) + h;
            const bool in = jj < nkt && kt < f8.ntiles;
            nsk[h] = in ? skh[kt] : 1.f;
            nsv[h] = in ? svh[kt] : svmax;
          }
        }
      };
      fetch_scales(0);

      for (int j = 0; j < nkt; ++j, ++scnt) {
        if (!warp_wait_suspend(&bar_s[t], scnt & 1, wc, kSiteSoftS)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int kbase = (sw.begin + sw.step * j) * kBlockK;
        // Some key of the block is past Nk, or beyond what the tile's first row sees.
        const bool need_mask = (kbase + kBlockK > ks.Nk) || (CAUSAL && kbase + kBlockK - 1 > qrow0 + ks.coff);
        // Per 64-key half h: multiplier c[h] of the raw score (FP8: times that key
        // tile's K scale) and lg[h] = log2 of the V-scale fold of P (0 for bf16).
        // The tile scales are powers of two (fa_fp8_prepare), so the fold
        // fv = sV / max sV is exact and its log2 is the difference of the two
        // exponent fields.
        float ch[2] = {crow, crow}, lg[2] = {0.f, 0.f}, fv[2] = {1.f, 1.f}, inv_fv[2] = {1.f, 1.f};
        if constexpr (FP8) {
  #pragma unroll
          for (int h = 0; h < 2; ++h) {
            ch[h] = crow * nsk[h];
            fv[h] = nsv[h] * inv_svmax;
            const int lgi = static_cast<int>((__float_as_uint(nsv[h]) >> 23) & 0xFFu) -
                            static_cast<int>((__float_as_uint(svmax) >> 23) & 0xFFu);  // <= 0
            lg[h] = static_cast<float>(lgi);
            // 1 / fv = 2^-lgi, exact.  (Dividing the row sums by fv instead would take
            // the division's slow path on rows whose sums are tiny after their
            // reference moved far up.)
            inv_fv[h] = lgi >= -127 ? __uint_as_float(static_cast<uint32_t>(127 - lgi) << 23) : svmax / nsv[h];
          }
          fetch_scales(j + 1);
        }
        uint32_t r[4][32];
        auto load_and_mask = [&](int c) {
          if (need_mask) {
  #pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int key = kbase + c * 32 + i;
              if (key >= ks.Nk || (CAUSAL && key > qrow + ks.coff)) r[c][i] = __float_as_uint(-INFINITY);
            }
          }
        };
        // Row maximum of the scaled scores (scale > 0: max commutes with it), as a
        // shallow max3 tree per 32-key chunk.
        auto tile_max = [&]() -> float {
          float mc[4];
  #pragma unroll
          for (int c = 0; c < 4; ++c) {
            float a[11];
  #pragma unroll
            for (int i = 0; i < 10; ++i)
              a[i] = max3(__uint_as_float(r[c][3 * i]), __uint_as_float(r[c][3 * i + 1]), __uint_as_float(r[c][3 * i + 2]));
            a[10] = fmaxf(__uint_as_float(r[c][30]), __uint_as_float(r[c][31]));
            const float b0 = max3(a[0], a[1], a[2]), b1 = max3(a[3], a[4], a[5]), b2 = max3(a[6], a[7], a[8]);
            mc[c] = fmaxf(max3(b0, b1, b2), fmaxf(a[9], a[10]));
          }
          return fmaxf(fmaxf(mc[0], mc[1]) * ch[0], fmaxf(mc[2], mc[3]) * ch[1]);
        };
        // P = exp2(S * c - m) over chunk c, written back over the S buffer.  bf16:
        // keys 32c..32c+31 become TMEM columns 16c..16c+15 (2 per column).  FP8:
        // P * fv (the V-scale fold) as e4m3, 4 per column, keys 64h..64h+63 in
        // columns 16h..16h+15.  Returns nothing; accumulates part[h].
        float2 part[2];
        uint32_t pk8[16];
        auto exp_chunk = [&](int c) {
          const int h = c >> 1;
          const float2 c2 = make_float2(ch[h], ch[h]);
          const float2 b2 = make_float2(lg[h] - m_used, lg[h] - m_used);
          uint32_t pk[16];
  #pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 x =
                __ffma2_rn(make_float2(__uint_as_float(r[c][2 * i]), __uint_as_float(r[c][2 * i + 1])), c2, b2);
            const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            part[h] = __fadd2_rn(part[h], p);
            if constexpr (FP8)
              pk[i] = e4m3x2_bits(p.x, p.y);
            else
              pk[i] = pack_bf16x2(p.x, p.y);
          }
          if constexpr (FP8) {
  #pragma unroll
            for (int i = 0; i < 8; ++i) pk8[(c & 1) * 8 + i] = pk[2 * i] | (pk[2 * i + 1] << 16);
            if (c & 1) tmem_st16(trow + col_s + h * 16, pk8);
          } else {
            tmem_st16(trow + col_s + c * 16, pk);
          }
        };
        auto tile_sum = [&]() {
          // l counts the unscaled P: undo the V-scale fold of each half.
          return (part[0].x + part[0].y) * inv_fv[0] + (part[1].x + part[1].y) * inv_fv[1];
        };

        // O_t is rescaled (in TMEM) by alpha for rows whose reference maximum moves
        // up; O_t already holds P V up to block j-1 because Q K_j^T was issued after it.
        auto rescale_o = [&](float alpha, bool any) {
          if (!any) return;
          const float2 a2 = make_float2(alpha, alpha);
  #pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(trow + col_o + c * 32, o);
            tmem_ld_wait32(o);
  #pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), a2);
              o[i] = __float_as_uint(v.x);
              o[i + 1] = __float_as_uint(v.y);
            }
            tmem_st32(trow + col_o + c * 32, o);
          }
        };

        // FP8: O rescaled after this block's exponentials (the scores are dead by
        // then, so all of O_t's columns are loaded at once), before P_t is signalled.
        auto rescale_o_all = [&](float alpha) {
          uint32_t o[D / 32][32];
  #pragma unroll
          for (int c = 0; c < D / 32; ++c) tmem_ld32(trow + col_o + c * 32, o[c]);
  #pragma unroll
          for (int c = 0; c < D / 32; ++c) tmem_ld_wait32(o[c]);
          const float2 a2 = make_float2(alpha, alpha);
  #pragma unroll
          for (int c = 0; c < D / 32; ++c) {
  #pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[c][i]), __uint_as_float(o[c][i + 1])), a2);
              o[c][i] = __float_as_uint(v.x);
              o[c][i + 1] = __float_as_uint(v.y);
            }
            tmem_st32(trow + col_o + c * 32, o[c]);
          }
        };

        float l_tile;
        if (j == 0 || FP8) {
          // The block's own maximum first.  First block: it is the reference
          // maximum.  FP8, later blocks: the reference moves up (and O is rescaled)
          // only when the block's maximum exceeds it by more than 2^8, so every
          // folded P stays <= 256, inside e4m3's range.  (Exponentiating before
          // knowing the maximum, as bf16 does below, pays off only when blocks
          // rarely overshoot; with outliers they often overshoot e4m3's 448.)
  #pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(trow + col_s + c * 32, r[c]);
  #pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld_wait32(r[c]);
  #pragma unroll
          for (int c = 0; c < 4; ++c) load_and_mask(c);
          const float mt = tile_max();
          float alpha = 1.f;
          bool any_rescale = false;
          if (j == 0) {
            m_used = (mt == -INFINITY) ? 0.f : mt;
          } else {
            const float m_new = fmaxf(m_used, mt);
            const bool need = m_new > m_used + kRescaleThreshold;
            if (need) {
              alpha = ex2_approx(m_used - m_new);
              m_used = m_new;
            }
            l *= alpha;
            any_rescale = __any_sync(0xffffffffu, need);
          }
          part[0] = part[1] = make_float2(0.f, 0.f);
  #pragma unroll
          for (int c = 0; c < 4; ++c) exp_chunk(c);
          l_tile = tile_sum();
          if (any_rescale) rescale_o_all(alpha);  // only FP8 reaches here with j > 0
        } else {
          // bf16, later blocks: exponentiate against the running maximum without
          // looking for a new one.  This is exact as long as no P overflows, which
          // the block's row sum proves (sum <= 2^16 => every P <= 2^16); otherwise
          // the block is redone below with its own maximum.  The second half of S
          // loads while the first half is exponentiated.
          tmem_ld32(trow + col_s, r[0]);
          tmem_ld32(trow + col_s + 32, r[1]);
          tmem_ld_wait32(r[0]);
          tmem_ld_wait32(r[1]);
          tmem_ld32(trow + col_s + 64, r[2]);
          tmem_ld32(trow + col_s + 96, r[3]);
          part[0] = part[1] = make_float2(0.f, 0.f);
          load_and_mask(0);
          load_and_mask(1);
          exp_chunk(0);
          exp_chunk(1);
          tmem_ld_wait32(r[2]);
          tmem_ld_wait32(r[3]);
          load_and_mask(2);
          load_and_mask(3);
          exp_chunk(2);
          exp_chunk(3);
          l_tile = tile_sum();
          const bool bad = !(l_tile <= kSpeculationSumBound);  // also true for inf / NaN
          if (__any_sync(0xffffffffu, bad)) {
            tmem_st_wait();  // the speculative P has landed before it is overwritten
            const float m_new = fmaxf(m_used, tile_max());
            const bool need = m_new > m_used;
            float alpha = 1.f;
            if (need) {
              alpha = ex2_approx(m_used - m_new);
              m_used = m_new;
            }
            l *= alpha;
            rescale_o(alpha, __any_sync(0xffffffffu, need));
            part[0] = part[1] = make_float2(0.f, 0.f);
  #pragma unroll
            for (int c = 0; c < 4; ++c) exp_chunk(c);
            l_tile = tile_sum();
          }
        }
        l += l_tile;
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          // With kRingWaitsInSoftmax, P_t of a whole unit signals more than P: V_j
          // (ring item ring_unit + 1 + 2j), and K_{j+1} after it when there is one,
          // have landed, so the MMA thread waits on P_t alone before P_t V_j and
          // S_t = Q_t K_{j+1}^T.
          bool landed = true;
          if (kRingWaitsInSoftmax && !shared) {
            const int iv = ring_unit + 1 + 2 * j;
            landed = mbar_wait(&bar_full[iv % C::kSlots], (iv / C::kSlots) & 1, wc, kSiteSoftKV);
            if (landed && j + 1 < n_max)
              landed = mbar_wait(&bar_full[(iv + 1) % C::kSlots], ((iv + 1) / C::kSlots) & 1, wc, kSiteSoftKV);
          }
          if (landed) mbar_arrive(&bar_p[t]);
        }
        if (kRingWaitsInSoftmax && !__shfl_sync(0xffffffffu, static_cast<int>(*abort_flag == 0), 0)) {
          ok = false;  // lane 0 gave up on the ring (the CTA is aborting)
          break;
        }
      }
      if (!ok) break;

      if (TAIL && shared) {  // the merge epilogue follows the loop (always the last item)
        sh.pending = true;
        sh.m = m_used;
        sh.l = l;
        sh.svmax = svmax;
        sh.bh = bh;
        sh.qrow0 = qrow0;
        sh.ph0 = ph0;
        sh.ph1 = ph1;
        sh.epi_index = epi_index;
        break;
      }
      // ---------------------------------------------------------- epilogue
      if (!(ok = warp_wait(&bar_o[t], ph_t & 1, wc, kSiteSoftO))) break;
      tc_fence_after();
      if constexpr (SPLIT) {
        // Partial of this split: O / l in fp32 straight from TMEM, LSE in natural
        // log; a row that saw no key of the split gets LSE = -inf (O is not read).
        const bool seen = l > 0.f;
        const float inv_l = seen ? 1.f / l : 0.f;
        float4* orow = reinterpret_cast<float4*>(ks.o_part + ((static_cast<size_t>(sp) * BH + bh) * N + qrow) * D);
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(trow + col_o + c * 32, o);
          tmem_ld_wait32(o);
          if (qrow < N) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              orow[c * 8 + i] = make_float4(__uint_as_float(o[4 * i]) * inv_l, __uint_as_float(o[4 * i + 1]) * inv_l,
                                            __uint_as_float(o[4 * i + 2]) * inv_l, __uint_as_float(o[4 * i + 3]) * inv_l);
          }
        }
        tc_fence_before();
        if (qrow < N)
          ks.lse_part[(static_cast<size_t>(sp) * BH + bh) * N + qrow] = seen ? (m_used + log2f(l)) * kLn2 : -INFINITY;
        continue;
      }
      // The staging buffer is free once the previous epilogue's store has read it.
      if (epi_index > 0 && !(ok = warp_wait(bar_stg, (epi_index - 1) & 1, wc, kSiteEpi))) break;
      const float inv_l = svmax / l;  // svmax = 1 for bf16
      const float2 il2 = make_float2(inv_l, inv_l);
      // O row -> bf16 -> the staging buffer, laid out as the 128-byte-swizzled TMA box expects.
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(trow + col_o + c * 32, o);
        tmem_ld_wait32(o);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), il2);
          pk[i] = pack_bf16x2(v.x, v.y);
        }
        uint8_t* box = sO + (c / 2) * C::kBoxBytes + row * 128;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int chunk = (c % 2) * 4 + q4;
          const uint4 val = make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
          *reinterpret_cast<uint4*>(box + ((chunk ^ (row & 7)) * 16)) = val;
        }
      }
      // O_t has been read out of TMEM (tcgen05.wait::ld above); the next unit's
      // first P V may overwrite it once this warpgroup signals its next P.
      tc_fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_epi[t]);
      if (qrow < N) lse[static_cast<size_t>(bh) * N + qrow] = (m_used + log2f(l)) * kLn2;
      if (row == 0) {
        if ((ok = mbar_wait(&bar_epi[t], ph_t & 1, wc, kSiteEpi))) {
#pragma unroll
          for (int b = 0; b < C::kOBoxes; ++b)
            tma_store_4d(&tm_o, sO + b * C::kBoxBytes, b * kBoxCols, qrow0, bh % H, bh / H);
          tma_store_commit_and_wait_read();
          mbar_arrive(bar_stg);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (TAIL && ok && sh.pending) do {
      // Shared tile: slot t holds the softmax of the tile over key blocks t, t+2,
      // ... (running maximum m_t, sum l_t, O_t).  Once the other slot's last P V
      // is done too, the two warpgroups swap (m, l) through the Q buffer (every
      // Q K^T of the item has completed) and each writes half of O's columns:
      //   O = (a_0 O_0 + a_1 O_1) / (a_0 l_0 + a_1 l_1),  a_t = 2^(m_t - max(m_0, m_1)).
      // (At most one shared tile per CTA, its last item: the barrier is used once.)
      if (!(ok = warp_wait(&bar_o[t], (t == 0 ? sh.ph0 : sh.ph1) & 1, wc, kSiteSoftO))) break;
      if (!(ok = warp_wait(&bar_o[t ^ 1], (t == 0 ? sh.ph1 : sh.ph0) & 1, wc, kSiteSoftO))) break;
      tc_fence_after();
      float2* xch = reinterpret_cast<float2*>(sQ);
      xch[t * kBlockQ + row] = make_float2(sh.m, sh.l);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_xm);
      if (!(ok = warp_wait(bar_xm, 0, wc, kSiteSoftO))) break;
      const float2 other = xch[(t ^ 1) * kBlockQ + row];
      const float m0 = t == 0 ? sh.m : other.x, l0 = t == 0 ? sh.l : other.y;
      const float m1 = t == 0 ? other.x : sh.m, l1 = t == 0 ? other.y : sh.l;
      const float mm = fmaxf(m0, m1);
      const float a0 = ex2_approx(m0 - mm), a1 = ex2_approx(m1 - mm);
      const float lsum = l0 * a0 + l1 * a1;
      const float inv_l = sh.svmax / lsum;  // svmax = 1 for bf16
      if (sh.epi_index > 0 && !(ok = warp_wait(bar_stg, (sh.epi_index - 1) & 1, wc, kSiteEpi))) break;
      const float2 w0 = make_float2(a0 * inv_l, a0 * inv_l), w1 = make_float2(a1 * inv_l, a1 * inv_l);
#pragma unroll 1
      for (int cc = 0; cc < D / 64; ++cc) {
        const int c = t * (D / 64) + cc;  // 32-column chunk of O written by this warpgroup
        uint32_t o0[32], o1[32];
        tmem_ld32(trow + C::col_o(0) + c * 32, o0);
        tmem_ld32(trow + C::col_o(1) + c * 32, o1);
        tmem_ld_wait32(o0);
        tmem_ld_wait32(o1);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 v = __ffma2_rn(make_float2(__uint_as_float(o0[2 * i]), __uint_as_float(o0[2 * i + 1])), w0,
                                      __fmul2_rn(make_float2(__uint_as_float(o1[2 * i]),
                                                             __uint_as_float(o1[2 * i + 1])), w1));
          pk[i] = pack_bf16x2(v.x, v.y);
        }
        uint8_t* box = sO + (c / 2) * C::kBoxBytes + row * 128;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int chunk = (c % 2) * 4 + q4;
          const uint4 val = make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
          *reinterpret_cast<uint4*>(box + ((chunk ^ (row & 7)) * 16)) = val;
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_epi[t]);
      const int qrow = sh.qrow0 + row;
      if (t == 0 && qrow < N) lse[static_cast<size_t>(sh.bh) * N + qrow] = (mm + log2f(lsum)) * kLn2;
      if (t == 0 && row == 0) {
        if ((ok = mbar_wait(&bar_epi[0], sh.ph0 & 1, wc, kSiteEpi) &&
                  mbar_wait(&bar_epi[1], sh.ph1 & 1, wc, kSiteEpi))) {
#pragma unroll
          for (int b = 0; b < C::kOBoxes; ++b)
            tma_store_4d(&tm_o, sO + b * C::kBoxBytes, b * kBoxCols, sh.qrow0, sh.bh % H, sh.bh / H);
          tma_store_commit_and_wait_read();
          mbar_arrive(bar_stg);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    } while (false);
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool CAUSAL, bool FP8, bool SPLIT = false>
cudaError_t launch_kernel(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                          float* lse, int N, int H, int BH, float scale_log2, unsigned int* err_word,
                          const DebugKnobs& dbg, const Fp8Scales& f8, const KeySplit& ks, cudaStream_t stream) {
  using C = FwdCfg<D, FP8>;
  cudaError_t e;
  auto kern = fwd_kernel<D, CAUSAL, FP8, SPLIT>;
  const int nunits = (N + kRowsPerCta - 1) / kRowsPerCta;
  // Persistent: one CTA per SM (shared memory and TMEM admit no second), each
  // walking its share of the units.
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev))) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))) return e;
  const long long units = static_cast<long long>(nunits) * BH * ks.nsplit;
  // Non-causal, unsplit keys, at least two key blocks: if the units leave a partial
  // last pass of R <= sms / 2 units, its units are dealt out as 2R shared tiles
  // (item_at), so that pass takes about half a unit's time.  The build with shared
  // tiles runs whole units about 3 % slower (measured), so it is used only when
  // the saving, half a pass of P + 1, is large: P <= 4 full passes.
  KeySplit kse = ks;
  long long items = units;
  if constexpr (!CAUSAL && !SPLIT) {
    if (ks.nsplit == 1 && (ks.Nk + kBlockK - 1) / kBlockK >= 2) {
      const long long full = units / sms * sms, rem = units - full;
      if (rem > 0 && 2 * rem <= sms && full / sms <= 4) {
        kse.tail_from = static_cast<int>(full);
        items = full + 2 * rem;
        kern = fwd_kernel<D, CAUSAL, FP8, SPLIT, true>;
      }
    }
  }
  // Per device and idempotent; cheap enough to repeat on every launch.
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes))) return e;
  // setmaxnreg.inc can only draw on the registers the block was launched with; a
  // build that allocated fewer per thread than the split assumes would stall.
  cudaFuncAttributes fattr;
  if ((e = cudaFuncGetAttributes(&fattr, kern))) return e;
  if (static_cast<uint32_t>(fattr.numRegs) * kThreads < kRegsNeeded) return cudaErrorInvalidConfiguration;
  dim3 grid(static_cast<unsigned>(min(items, static_cast<long long>(sms))));
  kern<<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, to, lse, N, H, BH, nunits, scale_log2, err_word,
                                                   dbg.wait_limit_ns, dbg.fault, f8, kse);
  return cudaGetLastError();
}

// The plain forward: one split over all N keys, queries aligned with keys.
KeySplit whole_keys(int N) { return KeySplit{N, 1, (N + kBlockK - 1) / kBlockK, 0, nullptr, nullptr, INT_MAX}; }

template <int D, bool CAUSAL>
cudaError_t launch_fwd_impl(const FwdArgs& a, cudaStream_t stream) {
  const int BH = a.B * a.H;
  CUtensorMap tq, tk, tv, to;
  cudaError_t e;
  constexpr auto kBf16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if ((e = make_tmap_4d(&tq, a.q, kBf16, 2, D, a.N, a.H, a.B, a.sq.s, kBoxCols, kBlockQ))) return e;
  if ((e = make_tmap_4d(&tk, a.k, kBf16, 2, D, a.N, a.H, a.B, a.sk.s, kBoxCols, kBlockK))) return e;
  if ((e = make_tmap_4d(&tv, a.v, kBf16, 2, D, a.N, a.H, a.B, a.sv.s, kBoxCols, kBlockK))) return e;
  if ((e = make_tmap_4d(&to, a.o, kBf16, 2, D, a.N, a.H, a.B, a.so.s, kBoxCols, kBlockQ))) return e;
  return launch_kernel<D, CAUSAL, false>(tq, tk, tv, to, a.lse, a.N, a.H, BH, a.scale * 1.4426950408889634f,
                                         a.err_word, a.dbg, Fp8Scales{nullptr, nullptr, nullptr, 0}, whole_keys(a.N),
                                         stream);
}

template <int D, bool CAUSAL>
cudaError_t launch_splitkv_impl(const SplitKvArgs& a, cudaStream_t stream) {
  const int BH = a.B * a.H;
  CUtensorMap tq, tk, tv;
  cudaError_t e;
  constexpr auto kBf16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if ((e = make_tmap_4d(&tq, a.q, kBf16, 2, D, a.Nq, a.H, a.B, a.sq.s, kBoxCols, kBlockQ))) return e;
  if ((e = make_tmap_4d(&tk, a.k, kBf16, 2, D, a.Nk, a.H, a.B, a.sk.s, kBoxCols, kBlockK))) return e;
  if ((e = make_tmap_4d(&tv, a.v, kBf16, 2, D, a.Nk, a.H, a.B, a.sv.s, kBoxCols, kBlockK))) return e;
  const KeySplit ks{a.Nk, a.n_split, splitkv_kbps(a.Nk, a.n_split), a.Nk - a.Nq, a.o_part, a.lse_part, INT_MAX};
  // The partial epilogue stores fp32 rows itself; the O tensor map is never used.
  return launch_kernel<D, CAUSAL, false, true>(tq, tk, tv, tq, nullptr, a.Nq, a.H, BH, a.scale * 1.4426950408889634f,
                                               a.err_word, a.dbg, Fp8Scales{nullptr, nullptr, nullptr, 0}, ks, stream);
}

template <int D, bool CAUSAL>
cudaError_t launch_fwd_fp8_impl(const FwdArgs& a, const void* workspace, cudaStream_t stream) {
  const int BH = a.B * a.H;
  const Fp8Layout lay = fp8_layout(a.B, a.H, a.N, D);
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  CUtensorMap tq, tk, tv, to;
  cudaError_t e;
  constexpr auto kU8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const Strides s8 = dense_strides(a.H, a.N, D), svt = dense_strides(a.H, D, lay.npad);
  // Q and K code rows: one box of the whole row (128 bytes at d = 128, 64 at d = 64).
  constexpr auto kSwQK = D == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  if ((e = make_tmap_4d(&tq, ws + lay.off_q8, kU8, 1, D, a.N, a.H, a.B, s8.s, D, kBlockQ, kSwQK))) return e;
  if ((e = make_tmap_4d(&tk, ws + lay.off_k8, kU8, 1, D, a.N, a.H, a.B, s8.s, D, kBlockK, kSwQK))) return e;
  if ((e = make_tmap_4d(&tv, ws + lay.off_v8t, kU8, 1, lay.npad, D, a.H, a.B, svt.s, kBlockK, D))) return e;
  if ((e = make_tmap_4d(&to, a.o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, a.H, a.B, a.so.s, kBoxCols, kBlockQ)))
    return e;
  const Fp8Scales f8{reinterpret_cast<const float*>(ws + lay.off_sq), reinterpret_cast<const float*>(ws + lay.off_sk),
                     reinterpret_cast<const float*>(ws + lay.off_sv), lay.ntiles};
  // Scores of the rotated operands are d times the plain ones: fold 1/d into the scale.
  const float scale_log2 = a.scale * 1.4426950408889634f / static_cast<float>(D);
  return launch_kernel<D, CAUSAL, true>(tq, tk, tv, to, a.lse, a.N, a.H, BH, scale_log2, a.err_word, a.dbg, f8,
                                        whole_keys(a.N), stream);
}

}  // namespace

cudaError_t launch_fwd_bf16(const FwdArgs& a, cudaStream_t stream) {
  if (a.d == 64) return a.causal ? launch_fwd_impl<64, true>(a, stream) : launch_fwd_impl<64, false>(a, stream);
  return a.causal ? launch_fwd_impl<128, true>(a, stream) : launch_fwd_impl<128, false>(a, stream);
}

cudaError_t launch_fwd_fp8(const FwdArgs& a, const void* workspace, cudaStream_t stream) {
  if (a.d == 64)
    return a.causal ? launch_fwd_fp8_impl<64, true>(a, workspace, stream)
                    : launch_fwd_fp8_impl<64, false>(a, workspace, stream);
  return a.causal ? launch_fwd_fp8_impl<128, true>(a, workspace, stream)
                  : launch_fwd_fp8_impl<128, false>(a, workspace, stream);
}

int splitkv_kbps(int Nk, int n_split) {
  const int nkb = (Nk + kBlockK - 1) / kBlockK;
  return (nkb + n_split - 1) / n_split;
}

cudaError_t launch_fwd_splitkv_partial(const SplitKvArgs& a, cudaStream_t stream) {
  // One query row (causal or not: the last position sees every key) is a stream over
  // K and V; at d = 64 the CUDA-core kernel in fa_splitkv.cu takes it (decode_takes).
  if (decode_takes(a.Nq, a.d)) return launch_decode_partial(a, stream);
  if (a.d == 64) return a.causal ? launch_splitkv_impl<64, true>(a, stream) : launch_splitkv_impl<64, false>(a, stream);
  return a.causal ? launch_splitkv_impl<128, true>(a, stream) : launch_splitkv_impl<128, false>(a, stream);
}

}  // namespace fa
