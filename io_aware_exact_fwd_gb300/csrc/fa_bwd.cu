// Exact attention backward, bf16, d = 64 or 128, for sm_103a.
//
// The pages describe only the forward ("FlashAttention-2 (DE)", "Hintergrund";
// "FlashAttention-Skalierung ...", section 1).  The backward follows from the
// chain rule applied to the same definition, recomputing P from the forward's
// per-row logsumexp instead of storing the N x N matrix (the same IO-aware
// idea applied to the gradient):
//
//   P_ij  = exp(scale * q_i . k_j - LSE_i)            (0 where masked)
//   dV    = P^T dO          dP = dO V^T
//   D_i   = sum_c dO_ic O_ic = sum_j P_ij dP_ij
//   dS    = P * (dP - D)    dQ = scale * dS K          dK = scale * dS^T Q
//
// Three launches on one stream:
//  1. bwd_preprocess: D_i and LSE_i * log2(e), written as the per-query operand
//     tiles of that extra K-step (padded rows get a huge negative LSE term so their
//     P is exactly 0), and zeroing of the fp32 dQ accumulator.
//  2. bwd_main: one CTA per (128-key block, head), the K/V-outer loop order.
//     K_j, V_j stay in shared memory; Q_i, dO_i (64 query rows) and two small
//     per-query tiles stream through a TMA ring.  The per-query terms LSE_i and D_i
//     enter the tensor core instead of the compute warps: S^T and dP^T get one
//     more K-step of 16 columns whose product is -LSE_i * log2(e) / (scale log2 e)
//     (resp. -D_i) in every key row, so the accumulators hold scale^-1 log2 P
//     and dP - D directly and the compute warps read no per-query value from
//     shared memory.  Per query block, tcgen05 MMAs (issued by two or three
//     single threads, see kSplitSdp) compute
//     S^T = K Q_i^T and dP^T = V dO_i^T into TMEM (keys on TMEM lanes, so a
//     thread owns one key row; two warpgroups split the 64 query columns),
//     eight warps form P^T and dS^T in registers and write them back to TMEM
//     as bf16 (A operands of dV += P^T dO_i and dK += dS^T Q_i) and to shared
//     memory (B operand of dQ_i^T = K^T dS^T).  dQ_i^T lands over the consumed
//     P^T, dS^T; four more warps (one d-row per thread) add it into the fp32
//     accumulator with coalesced reductions.
//     TMEM: dV, dK (128 columns each), one S^T, dP^T pair (64 each, free again
//     as soon as the compute warps hold it in registers, so S^T, dP^T of the
//     next block overlap this block's math), and two 64-column buffers for
//     P^T, dS^T and then dQ^T.
//  3. bwd_dq_convert: dQ = bf16(scale * dQacc).
//
// Every MMA has M = 128 (the tcgen05 data path with one TMEM lane per row).  At
// d = 64 the dQ^T product (M = d) is padded to 128 rows: its A operand, K^T read
// MN-major in two 64-row groups, takes the second group from a zeroed 16 KB
// shared-memory box, so rows 64..127 of dQ^T come out zero and are not reduced.
// That doubles only the dQ^T product (one fifth of the backward's FLOPs).
#include <math.h>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kBkB = 128;       // keys per CTA
constexpr int kBqB = 64;        // query rows per inner step
constexpr int kThreads = 512;   // 0-7 compute, 8-11 dQ reduction, 12 TMA, 13-15 MMA issuers (15: see kSplitSdp)
constexpr int kWarpDq = 8;
constexpr int kWarpCtl = 12;
constexpr int kWarpLoad = 12;
constexpr int kWarpMma = 13;     // issues dV, dK, dQ^T (and owns the TMEM allocation)
constexpr int kWarpMmaS = 14;    // issues S^T
constexpr int kWarpMmaDP = 15;   // issues dP^T when the kernel splits that issue (kSplitSdp), else idle
constexpr int kStages = 3;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
// Launch budget 128 x 512 registers: the two compute warpgroups (one 32-query
// half of a score row each) take 160, the dQ warpgroup 120, the control
// warpgroup (TMA, MMA) gives back to 72.
constexpr uint32_t kLaunchRegs = 128;
constexpr uint32_t kRegsCompute = 160;
constexpr uint32_t kRegsDq = 120;
constexpr uint32_t kRegsControl = 72;
static_assert(128 * (2 * kRegsCompute + kRegsDq + kRegsControl) <= kLaunchRegs * kThreads, "register split");

enum : uint32_t {
  kSiteBLoad = 0x111,
  kSiteBMmaKV = 0x211,
  kSiteBMmaQ = 0x212,
  kSiteBMmaC = 0x213,
  kSiteBMmaDq = 0x214,
  kSiteBMmaSd = 0x215,
  kSiteBComp = 0x311,
  kSiteBDq = 0x312,
  kSiteBEpi = 0x313,
};

template <int D>
struct BwdCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kBoxes = D / 64;                 // 128-byte TMA boxes per bf16 row
  static constexpr int kKVBox = kBkB * 64 * 2;          // 16 KB: 128 rows x 128 B
  static constexpr int kKVTile = kBkB * D * 2;          // 32 KB (d=128), 16 KB (d=64)
  static constexpr int kQBox = kBqB * 64 * 2;           // 8 KB: 64 rows x 128 B
  static constexpr int kQTile = kBqB * D * 2;           // 16 KB (d=128), 8 KB (d=64)
  static constexpr int kStageQ = 0;
  static constexpr int kStageDO = kQTile;
  // The extra K-step's per-query tiles (64 rows x 32 bytes, 32-byte swizzle):
  // [a1 a2 a3 a1 a2 a3 a1 a2 a3 0...] with a1 + a2 + a3 = -LSE2 for S^T, then
  // [d1 d2 d3 0...] with d1 + d2 + d3 = -D for dP^T (three-term bf16 splits).
  static constexpr int kAugTile = kBqB * 32;           // 2 KB
  static constexpr int kStageAug = 2 * kQTile;
  static constexpr int kStageTx = 2 * kQTile + 2 * kAugTile;  // bytes landing per stage
  static constexpr int kStageBytes = (kStageTx + 1023) / 1024 * 1024;
  static constexpr int kDsBytes = kBkB * kBqB * 2;      // 16 KB: 128 key rows x 128 B
  // K, then (d = 64) the zero box that pads K^T to the dQ^T MMA's 128 rows, then V,
  // then the extra K-step's constant key-side tiles (128 rows x 32 bytes each):
  // [c1 c1 c1 c2 c2 c2 c3 c3 c3 0...] with c1 + c2 + c3 = 1 / (scale log2 e) for S^T
  // (so the nine products sum to (c1 + c2 + c3)(a1 + a2 + a3)), [1 1 1 0...] for dP^T.
  static constexpr int kKOff = 0;
  static constexpr int kZeroOff = kKVTile;
  static constexpr int kVOff = kKVTile + (D == 64 ? kKVBox : 0);
  static constexpr int kKAugOff = kVOff + kKVTile;
  static constexpr int kVAugOff = kKAugOff + kBkB * 32;
  static constexpr int kRingOff = kVAugOff + kBkB * 32;
  static constexpr int kDsOff = kRingOff + kStages * kStageBytes;
  static constexpr int kBarOff = kDsOff + 2 * kDsBytes;
  // kv, full[S], empty[S], sdp, sde, comp[2], dqf[2], dqe[2], dkv, epi, drain
  static constexpr int kNumBars = 1 + 2 * kStages + 1 + 1 + 2 + 2 + 2 + 1 + 1 + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
  // TMEM columns: dV, dK accumulators (D columns each); one S^T, dP^T pair (fp32,
  // read once by the compute warps, then free for the next query block); two
  // 64-column buffers that hold P^T | dS^T (bf16, 32 columns each) and then dQ^T (fp32).
  static constexpr uint32_t kColDV = 0, kColDK = 128, kColS = 256, kColDP = 320;
  static __device__ __forceinline__ uint32_t col_pdq(int b) { return 384u + 64u * b; }
  static_assert(kStageTx <= kStageBytes, "stage layout");
  static_assert(kZeroOff % 1024 == 0 && kKAugOff % 1024 == 0 && kRingOff % 1024 == 0, "operand tile alignment");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ bool warp_wait_b(uint64_t* bar, uint32_t parity, const WaitCtl& wc, uint32_t site) {
  const bool ok = mbar_wait(bar, parity, wc, site);
  return __all_sync(0xffffffffu, ok);
}
// For the compute and dQ warps' long waits (S^T, dP^T ready; dQ^T ready): their polls
// suspend instead of spinning beside the MMA-issuing warps.
__device__ __forceinline__ bool warp_wait_b_suspend(uint64_t* bar, uint32_t parity, const WaitCtl& wc, uint32_t site) {
  const bool ok = mbar_wait_suspend(bar, parity, wc, site, 20000u);
  return __all_sync(0xffffffffu, ok);
}

// Deterministic dQ: fixed-point accumulation.  Every contribution of a key block
// to dQacc[i, c] is sum_j dS_ij k_jc, and the whole sum over all key blocks obeys
//   |sum_j dS_ij k_jc| <= sum_j |dS_ij| max|k| <= 2 max_j |dP_ij| max|k|
//                      <= 2 |dO_i| max_j |v_j| max|k|
// (|dS_ij| = P_ij |dP_ij - D_i| with D_i a P-weighted mean of dP_i., and
// |dP_ij| = |dO_i . v_j| <= |dO_i| |v_j|).  With a 64-row block's largest |dO_i|,
// the head's largest |v_j| and largest |k_jc|, and a 12.5 % margin for the bf16
// rounding of P and dS, the power of two 2^S below puts every partial sum of the
// block's rows under 2^22 in magnitude.  Contributions are rounded to integers
// once (x 2^S, nearest) and added as int32: integer addition does not depend on
// order, so dQ is the same bits on every run.  2^22 keeps the float-to-int step
// a single add of 1.5 * 2^23 (the rounding is the fp32 add's).
__device__ __forceinline__ int det_shift(float dq_block_max, float vmax, float kmax) {
  const float bound = 2.25f * dq_block_max * vmax * kmax;
  if (!(bound > 0.f)) return 100;           // all-zero block (or no data): nothing to scale
  if (!(bound < 3.0e38f)) return -100;      // non-finite inputs: the result is undefined anyway
  int e;
  frexpf(bound, &e);                        // bound < 2^e
  return max(-100, min(100, 22 - e));
}
__device__ __forceinline__ float pow2f(int s) { return __int_as_float((s + 127) << 23); }  // -126 <= s <= 127

// Three-term bf16 split of x: t1 = bf16(x), t2 = bf16(x - t1), t3 = bf16(x - t1 - t2)
// (each difference exact in fp32), so t1 + t2 + t3 carries about 24 significant
// bits of x.  Returned as raw bf16 bits.
__device__ __forceinline__ void split3_bf16(float x, uint32_t (&t)[3]) {
  float r = x;
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const __nv_bfloat16 h = __float2bfloat16_rn(r);
    t[i] = static_cast<uint32_t>(__bfloat16_as_ushort(h));
    r -= __bfloat162float(h);
  }
}

// Element offset of row n of head (b, h) in a strided [B, H, N, d] tensor.
__device__ __forceinline__ size_t row_offset(const Strides& st, long long bh, int H, int n) {
  return static_cast<size_t>((bh / H) * st.s[2] + (bh % H) * st.s[1] + static_cast<long long>(n) * st.s[0]);
}

// Stage this thread's D-column fp32 accumulator row as bf16 into 128-byte-swizzled
// [128 rows][64 cols] TMA boxes (D / 64 of them).
template <int D>
__device__ __forceinline__ void stage_row_bf16(uint32_t taddr_row, uint8_t* boxes, int row, float mul) {
#pragma unroll 1
  for (int c = 0; c < D / 32; ++c) {
    uint32_t o[32];
    tmem_ld32(taddr_row + c * 32, o);
    tmem_ld_wait32(o);
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * mul, __uint_as_float(o[2 * i + 1]) * mul);
    uint8_t* box = boxes + (c / 2) * BwdCfg<D>::kKVBox + row * 128;
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const int chunk = (c % 2) * 4 + q4;
      *reinterpret_cast<uint4*>(box + ((chunk ^ (row & 7)) * 16)) =
          make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
    }
  }
}

template <int D, bool CAUSAL, bool DET>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                    const uint8_t* __restrict__ aug, float* __restrict__ dq_acc,
                    const float* __restrict__ dq_bmax, const float* __restrict__ kv_max, int N, int Npad, int H,
                    int BH, int nkb, float scale, float scale_log2, unsigned int* err_word, unsigned long long wait_ns) {
  using C = BwdCfg<D>;
  // Whether warps 14 and 15 split the S^T and dP^T issue (see the MMA issuers below).
  // Measured faster with atomic dQ at d = 128 only: the deterministic dQ warps and
  // the d = 64 kernel (where the chain is the elementwise work) do not gain from it.
  constexpr bool kSplitSdp = D == 128 && !DET;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem + C::kKOff;
  uint8_t* sV = smem + C::kVOff;
  uint8_t* sRing = smem + C::kRingOff;
  uint8_t* sDs = smem + C::kDsOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* bar_kv = bars;
  uint64_t* bar_full = bars + 1;
  uint64_t* bar_empty = bar_full + kStages;
  uint64_t* bar_sdp = bar_empty + kStages;  // S^T, dP^T ready in TMEM
  uint64_t* bar_sde = bar_sdp + 1;          // S^T, dP^T read out of TMEM
  uint64_t* bar_comp = bar_sde + 1;         // [2] P^T, dS^T written
  uint64_t* bar_dqf = bar_comp + 2;         // [2] dQ^T ready in TMEM
  uint64_t* bar_dqe = bar_dqf + 2;          // [2] dQ^T read out of TMEM
  uint64_t* bar_dkv = bar_dqe + 2;
  uint64_t* bar_epi = bar_dkv + 1;
  uint64_t* bar_drain = bar_epi + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  int kb, bh;
  if (CAUSAL) {  // key blocks near the start see the most query blocks: issue them first
    kb = static_cast<int>(blockIdx.x) / BH;
    bh = static_cast<int>(blockIdx.x) % BH;
  } else {
    kb = static_cast<int>(blockIdx.x) % nkb;
    bh = static_cast<int>(blockIdx.x) / nkb;
  }
  const int h_idx = bh % H, b_idx = bh / H;  // head and batch of the TMA coordinates
  const int nqb = (N + kBqB - 1) / kBqB;
  const int i0 = CAUSAL ? (kb * kBkB) / kBqB : 0;
  const int n = nqb - i0;  // >= 1: query row kb*128 < N exists

  if (threadIdx.x == 0) {
    mbar_init(bar_kv, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    mbar_init(bar_sdp, kSplitSdp ? 2 : 1);  // one commit per S^T / dP^T issuing thread
    mbar_init(bar_sde, 8);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_comp[b], 8);
      mbar_init(&bar_dqf[b], 1);
      mbar_init(&bar_dqe[b], 4);
    }
    mbar_init(bar_dkv, 1);
    mbar_init(bar_epi, 8);
    mbar_init(bar_drain, kSplitSdp ? 3 : 2);  // one commit per MMA-issuing thread
    *abort_flag = 0;
    fence_mbar_init();
  }
  if constexpr (D == 64) {
    // Rows 64..127 of the dQ^T MMA's A operand: zeros, read by the tensor core.
    uint4* z = reinterpret_cast<uint4*>(smem + C::kZeroOff);
    for (int i = threadIdx.x; i < C::kKVBox / 16; i += kThreads) z[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  {
    // The extra K-step's key-side tiles: one 16-byte half-row per thread (128 rows,
    // two halves, two tiles = 512 stores), at its 32-byte-swizzle position.
    const int tile = threadIdx.x >> 8, krow = (threadIdx.x >> 1) & 127, half = threadIdx.x & 1;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (tile == 0) {
      uint32_t c[3];
      split3_bf16(1.f / scale_log2, c);
      // elements 0-7: c1 c1 c1 c2 c2 c2 c3 c3; element 8: c3
      val = half == 0 ? make_uint4(c[0] | (c[0] << 16), c[0] | (c[1] << 16), c[1] | (c[1] << 16), c[2] | (c[2] << 16))
                      : make_uint4(c[2], 0u, 0u, 0u);
    } else if (half == 0) {
      val = make_uint4(0x3F803F80u, 0x3F80u, 0u, 0u);  // bf16 1.0, 1.0, 1.0
    }
    uint8_t* base = smem + (tile == 0 ? C::kKAugOff : C::kVAugOff);
    *reinterpret_cast<uint4*>(base + krow * 32 + ((half ^ ((krow >> 2) & 1)) << 4)) = val;
    fence_proxy_async_smem();
  }
  if (warp == kWarpMma) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, err_word, wait_ns};
  const uint8_t* aug_h = aug + static_cast<size_t>(bh) * (Npad / kBqB) * (2 * C::kAugTile);

  if (warp >= kWarpCtl) {
   regs_decrease<kRegsControl>();
   if (warp == kWarpLoad) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_kv, 2 * C::kKVTile);
      for (int b = 0; b < C::kBoxes; ++b) {
        tma_load_4d(sK + b * C::kKVBox, &tm_k, bar_kv, b * 64, kb * kBkB, h_idx, b_idx);
        tma_load_4d(sV + b * C::kKVBox, &tm_v, bar_kv, b * 64, kb * kBkB, h_idx, b_idx);
      }
      int issued = 0;
      for (int it = 0; it < n; ++it) {
        const int slot = it % kStages;
        if (!mbar_wait(&bar_empty[slot], ((it / kStages) & 1) ^ 1, wc, kSiteBLoad)) break;
        const int i = i0 + it;
        uint8_t* st = sRing + slot * C::kStageBytes;
        mbar_arrive_expect_tx(&bar_full[slot], C::kStageTx);
        for (int b = 0; b < C::kBoxes; ++b) {
          tma_load_4d(st + C::kStageQ + b * C::kQBox, &tm_q, &bar_full[slot], b * 64, i * kBqB, h_idx, b_idx);
          tma_load_4d(st + C::kStageDO + b * C::kQBox, &tm_do, &bar_full[slot], b * 64, i * kBqB, h_idx, b_idx);
        }
        bulk_load(st + C::kStageAug, aug_h + static_cast<size_t>(i) * (2 * C::kAugTile), 2 * C::kAugTile,
                  &bar_full[slot]);
        ++issued;
      }
      if (issued < n) {  // aborted: let the copies already in flight land
        mbar_wait_drain(bar_kv, 0, wait_ns);
        for (int t = max(0, issued - kStages); t < issued; ++t)
          mbar_wait_drain(&bar_full[t % kStages], (t / kStages) & 1, wait_ns);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma || warp == kWarpMmaS || (kSplitSdp && warp == kWarpMmaDP)) {
    // ------------------------------------------------ MMA issuers (one thread each)
    // Two threads issue MMAs so that S^T/dP^T of a later query block never waits
    // behind dV/dK/dQ^T of an earlier one (or vice versa).  Each hazard between
    // them is covered by a barrier: S^T(it), dP^T(it) overwrite the pair that the
    // compute warps have already loaded into registers (bar_sde), dV/dK/dQ^T(it)
    // start only after P^T, dS^T(it) are written (bar_comp), and the compute
    // warps write P^T, dS^T(it) only after dQ^T(it-2), which they overwrite, was
    // read out (bar_dqe).  MMAs of one thread run in issue order, so dQ^T(it)
    // lands over P^T, dS^T(it) only after dV, dK(it) consumed them.
    if (lane == 0) {
      constexpr uint32_t idesc_sdp = idesc_bf16_f32(kBkB, kBqB, 0, 0);   // keys x queries, K = d
      constexpr uint32_t idesc_dkv = idesc_bf16_f32(kBkB, D, 0, 1);      // keys x d, K = queries
      // d x queries, K = keys; M = 128 rows (at d = 64, rows 64..127 read the zero box).
      constexpr uint32_t idesc_dq = idesc_bf16_f32(128, kBqB, 1, 1);
      const uint64_t k_kmaj = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t v_kmaj = sdesc_sw128(smem_u32(sV), 16, 1024);
      const uint64_t k_mn = sdesc_sw128(smem_u32(sK), C::kKVBox, 1024);
      const uint64_t ring_kmaj = sdesc_sw128(smem_u32(sRing), 16, 1024);
      const uint64_t ring_mn = sdesc_sw128(smem_u32(sRing), C::kQBox, 1024);
      const uint64_t ds_mn = sdesc_sw128(smem_u32(sDs), 16, 1024);
      const uint64_t kaug = sdesc_sw32(smem_u32(smem + C::kKAugOff));
      const uint64_t vaug = sdesc_sw32(smem_u32(smem + C::kVAugOff));
      const uint64_t ring_aug = sdesc_sw32(smem_u32(sRing + C::kStageAug));
      bool ok = mbar_wait(bar_kv, 0, wc, kSiteBMmaKV);
      if (warp == kWarpMmaS || warp == kWarpMmaDP) {
        // S^T = K Q_i^T and dP^T = V dO_i^T for local step `it`, as soon as the
        // compute warps have read the previous pair out of TMEM.  With
        // kSplitSdp warp 14 issues S^T and warp 15 dP^T: one thread's chain of
        // N = 64 MMAs runs at about half the tensor rate, two overlap, and this
        // pair is the backward's critical path (issue, completion, the compute
        // warps' TMEM loads, bar_sde).  Otherwise warp 14 issues both.
        const bool issue_s = warp == kWarpMmaS;
        const bool issue_dp = kSplitSdp ? warp == kWarpMmaDP : warp == kWarpMmaS;
        // Ring slot, its phase and byte offset, stepped instead of recomputed (these
        // threads' instructions pace the step).
        int slot = 0;
        uint32_t ring_ph = 0, st = 0;
        for (int it = 0; ok && it < n; ++it) {
          if (!(ok = mbar_wait(&bar_full[slot], ring_ph, wc, kSiteBMmaQ))) break;
          if (it >= 1 && !(ok = mbar_wait(bar_sde, (it - 1) & 1, wc, kSiteBMmaSd))) break;
          tc_fence_after();
          if (issue_s) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t offa = (kk / 4) * C::kKVBox + (kk % 4) * 32;
              const uint32_t offb = (kk / 4) * C::kQBox + (kk % 4) * 32;
              mma_bf16_ss(tmem + C::kColS, sdesc_add(k_kmaj, offa), sdesc_add(ring_kmaj, st + C::kStageQ + offb),
                          idesc_sdp, kk > 0 ? 1u : 0u);
            }
            mma_bf16_ss(tmem + C::kColS, kaug, sdesc_add(ring_aug, st), idesc_sdp, 1u);  // - LSE2 / (scale log2 e)
          }
          if (issue_dp) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t offa = (kk / 4) * C::kKVBox + (kk % 4) * 32;
              const uint32_t offb = (kk / 4) * C::kQBox + (kk % 4) * 32;
              mma_bf16_ss(tmem + C::kColDP, sdesc_add(v_kmaj, offa), sdesc_add(ring_kmaj, st + C::kStageDO + offb),
                          idesc_sdp, kk > 0 ? 1u : 0u);
            }
            mma_bf16_ss(tmem + C::kColDP, vaug, sdesc_add(ring_aug, st + C::kAugTile), idesc_sdp, 1u);  // - D
          }
          mma_commit(bar_sdp);
          if (++slot == kStages) {
            slot = 0;
            ring_ph ^= 1u;
            st = 0;
          } else {
            st += C::kStageBytes;
          }
        }
      } else {
        int slot = 0;  // ring slot and byte offset, stepped (see the S^T / dP^T issuers)
        uint32_t st = 0;
        for (int it = 0; ok && it < n; ++it) {
          const int b = it & 1;
          if (!(ok = mbar_wait(&bar_comp[b], (it >> 1) & 1, wc, kSiteBMmaC))) break;
          tc_fence_after();
          // dV += P^T dO_i ; dK += dS^T Q_i   (A from TMEM, B MN-major: 16 query rows per MMA)
#pragma unroll
          for (int kk = 0; kk < kBqB / 16; ++kk)
            mma_bf16_ts(tmem + C::kColDV, tmem + C::col_pdq(b) + kk * 8,
                        sdesc_add(ring_mn, st + C::kStageDO + kk * 2048), idesc_dkv, (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < kBqB / 16; ++kk)
            mma_bf16_ts(tmem + C::kColDK, tmem + C::col_pdq(b) + 32 + kk * 8,
                        sdesc_add(ring_mn, st + C::kStageQ + kk * 2048), idesc_dkv, (it > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bar_empty[slot]);
          // dQ_i^T = K^T dS^T : A = K MN-major (d contiguous; the second 64-row group is K's
          // second box at d = 128, the zero box at d = 64), B = dS^T rows of 64 queries;
          // 16 keys per MMA.
#pragma unroll
          for (int kk = 0; kk < kBkB / 16; ++kk)
            mma_bf16_ss(tmem + C::col_pdq(b), sdesc_add(k_mn, kk * 2048),
                        sdesc_add(ds_mn, b * C::kDsBytes + kk * 2048), idesc_dq, kk > 0 ? 1u : 0u);
          mma_commit(&bar_dqf[b]);
          if (++slot == kStages) {
            slot = 0;
            st = 0;
          } else {
            st += C::kStageBytes;
          }
        }
        if (ok) mma_commit(bar_dkv);
      }
      // Every issued MMA of every issuing thread must finish before TMEM is released.
      mma_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0, wait_ns);
    }
    __syncwarp();
   }
  } else if (warp < kWarpDq) {
    regs_increase<kRegsCompute>();
    // ------------------------------------- P and dS (one key row per thread)
    // Warpgroup g = warp / 4 takes query columns 32g .. 32g+31 of every 64-query
    // block, so two warps share each SM sub-partition's TMEM lanes and the
    // latency of one block's softmax-gradient math is split between them.
    const int g = warp >> 2;
    const int row = threadIdx.x & 127;
    const int key = kb * kBkB + row;
    const bool key_valid = key < N;
    const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const float2 sl2 = make_float2(scale_log2, scale_log2);
    bool ok = true;
    for (int it = 0; it < n; ++it) {
      const int b = it & 1;
      const int i = i0 + it;
      if (!(ok = warp_wait_b_suspend(bar_sdp, it & 1, wc, kSiteBComp))) break;
      tc_fence_after();
      uint32_t s[32], dp[32];
      tmem_ld32(trow + C::kColS + 32 * g, s);
      tmem_ld32(trow + C::kColDP + 32 * g, dp);
      tmem_ld_wait32(s);
      tmem_ld_wait32(dp);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_sde);  // the MMA warp may now overwrite S^T, dP^T
      const bool diag = CAUSAL && (i * kBqB < kb * kBkB + kBkB);  // some query in this block precedes a key
      const int q0 = i * kBqB + 32 * g;
      uint32_t ppk[16], dpk[16];
#pragma unroll
      for (int c2 = 0; c2 < 16; ++c2) {
        const int c = 2 * c2;
        // S^T holds S - LSE2 / (scale log2 e) and dP^T holds dP - D (the extra K-step).
        const float2 x = __fmul2_rn(make_float2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), sl2);
        float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        if (!key_valid || (diag && key > q0 + c)) p.x = 0.f;
        if (!key_valid || (diag && key > q0 + c + 1)) p.y = 0.f;
        const float2 ds = __fmul2_rn(p, make_float2(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1])));
        ppk[c2] = pack_bf16x2(p.x, p.y);
        dpk[c2] = pack_bf16x2(ds.x, ds.y);
      }
      // P^T, dS^T(it) overwrite dQ^T(it-2) (TMEM) and dS^T(it-2) (shared memory).
      if (it >= 2 && !(ok = warp_wait_b(&bar_dqe[b], ((it - 2) >> 1) & 1, wc, kSiteBComp))) break;
      tc_fence_after();
      tmem_st16(trow + C::col_pdq(b) + 16 * g, ppk);
      tmem_st16(trow + C::col_pdq(b) + 32 + 16 * g, dpk);
      // dS row into shared memory, 128-byte swizzle: chunk ch holds queries 8ch..8ch+7.
      uint8_t* ds_row = sDs + b * C::kDsBytes + row * 128;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const int ch = g * 4 + c4;
        *reinterpret_cast<uint4*>(ds_row + ((ch ^ (row & 7)) * 16)) =
            make_uint4(dpk[4 * c4], dpk[4 * c4 + 1], dpk[4 * c4 + 2], dpk[4 * c4 + 3]);
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_comp[b]);
    }
    // ------------------------------- dK, dV epilogue (warpgroup 0: dV, 1: dK)
    if (ok) ok = warp_wait_b(bar_dkv, 0, wc, kSiteBEpi);
    if (ok) {
      tc_fence_after();
      if (g == 0) stage_row_bf16<D>(trow + C::kColDV, sV, row, 1.f);
      else stage_row_bf16<D>(trow + C::kColDK, sK, row, scale);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_epi);
      if (threadIdx.x == 0 && mbar_wait(bar_epi, 0, wc, kSiteBEpi)) {
        for (int bb = 0; bb < C::kBoxes; ++bb) {
          tma_store_4d(&tm_dv, sV + bb * C::kKVBox, bb * 64, kb * kBkB, h_idx, b_idx);
          tma_store_4d(&tm_dk, sK + bb * C::kKVBox, bb * 64, kb * kBkB, h_idx, b_idx);
        }
        tma_store_commit_and_wait_read();
      }
    }
    __syncwarp();
  } else {
    regs_decrease<kRegsDq>();
    // -------------------------------- dQ reduction (one d-row of dQ^T per thread)
    const int dcol = threadIdx.x - kWarpDq * 32;
    const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    for (int it = 0; it < n; ++it) {
      const int b = it & 1;
      if (!warp_wait_b_suspend(&bar_dqf[b], (it >> 1) & 1, wc, kSiteBDq)) break;
      if (D == 64 && dcol >= D) {  // the zero-padded rows of dQ^T: nothing to read or add
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_dqe[b]);
        continue;
      }
      tc_fence_after();
      uint32_t v[2][32];
      tmem_ld32(trow + C::col_pdq(b), v[0]);
      tmem_ld32(trow + C::col_pdq(b) + 32, v[1]);
      tmem_ld_wait32(v[0]);
      tmem_ld_wait32(v[1]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_dqe[b]);
      const int q0 = (i0 + it) * kBqB;
      float* dst = dq_acc + (static_cast<size_t>(bh) * N + q0) * D + dcol;
      const int lim = min(kBqB, N - q0);
      if constexpr (DET) {
        const float mul = pow2f(det_shift(dq_bmax[static_cast<size_t>(bh) * (Npad / kBqB) + i0 + it],
                                          kv_max[2 * bh], kv_max[2 * bh + 1]));
        constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23: x + kMagic rounds x to an integer in the low bits
        int* dsti = reinterpret_cast<int*>(dst);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (h * 32 + c < lim)
              atomicAdd(dsti + static_cast<size_t>(h * 32 + c) * D,
                        __float_as_int(fmaf(__uint_as_float(v[h][c]), mul, kMagic)) - 0x4B400000);
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (h * 32 + c < lim) atomicAdd(dst + static_cast<size_t>(h * 32 + c) * D, __uint_as_float(v[h][c]));
      }
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// D_i = sum_c dO_ic O_ic and LSE2_i = LSE_i * log2(e), written as row i of the
// main kernel's per-query operand tiles (64 rows x 32 bytes each, 32-byte swizzle,
// one pair per 64-row query block): [a1 a2 a3 a1 a2 a3 a1 a2 a3 0...] with
// a1 + a2 + a3 = -LSE2 and [d1 d2 d3 0...] with d1 + d2 + d3 = -D (three-term bf16
// splits).  Rows >= N get -LSE2 = -1e30 (their P is exactly 0) and D = 0.
// dQacc rows < N are zeroed.  D / 8 threads per row, 8 elements each.
template <int D, bool DET>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ o,
                                                             const __nv_bfloat16* __restrict__ dout,
                                                             const float* __restrict__ lse, uint8_t* __restrict__ aug,
                                                             float* __restrict__ dq_acc,
                                                             unsigned int* __restrict__ dq_bmax, int N, int Npad,
                                                             long long rows_pad, int H, Strides so, Strides sdo) {
  constexpr int kTpr = D / 8;          // threads per row
  constexpr int kRpb = 256 / kTpr;     // rows per block: 16 (d=128) or 32 (d=64)
  const long long r = static_cast<long long>(blockIdx.x) * kRpb + (threadIdx.x / kTpr);
  const int t = threadIdx.x % kTpr;
  // The grid is exactly rows_pad / kRpb blocks (Npad is a multiple of 64), so every
  // thread has a row and all of them reach the shuffles and the barrier below.
  const long long bh = r / Npad;
  const int nrow = static_cast<int>(r - bh * Npad);
  float acc = 0.f, nrm = 0.f;
  if (nrow < N) {
    const size_t base = (static_cast<size_t>(bh) * N + nrow) * D + t * 8;  // dense: the dQ accumulator
    const uint4 ov = *reinterpret_cast<const uint4*>(o + row_offset(so, bh, H, nrow) + t * 8);
    const uint4 gv = *reinterpret_cast<const uint4*>(dout + row_offset(sdo, bh, H, nrow) + t * 8);
    const __nv_bfloat162* op = reinterpret_cast<const __nv_bfloat162*>(&ov);
    const __nv_bfloat162* gp = reinterpret_cast<const __nv_bfloat162*>(&gv);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 a = __bfloat1622float2(op[e]);
      const float2 g = __bfloat1622float2(gp[e]);
      acc = fmaf(a.x, g.x, acc);
      acc = fmaf(a.y, g.y, acc);
      if (DET) {
        nrm = fmaf(g.x, g.x, nrm);
        nrm = fmaf(g.y, g.y, nrm);
      }
    }
    float4* z = reinterpret_cast<float4*>(dq_acc + base);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int m = kTpr / 2; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m, kTpr);
  if (t == 0) {
    uint32_t a[3], dd[3];
    split3_bf16(nrow < N ? -lse[static_cast<size_t>(bh) * N + nrow] * kLog2e : -1e30f, a);
    split3_bf16(nrow < N ? -acc : 0.f, dd);
    const int rr = nrow % kBqB;
    uint8_t* tile = aug + (static_cast<size_t>(r / kBqB)) * (2 * kBqB * 32);  // r / 64 = (bh, query block)
    const int h0 = ((rr >> 2) & 1) << 4, h1 = (1 ^ ((rr >> 2) & 1)) << 4;     // swizzled half-row positions
    // elements 0-7: a1 a2 a3 a1 a2 a3 a1 a2; element 8: a3
    *reinterpret_cast<uint4*>(tile + rr * 32 + h0) =
        make_uint4(a[0] | (a[1] << 16), a[2] | (a[0] << 16), a[1] | (a[2] << 16), a[0] | (a[1] << 16));
    *reinterpret_cast<uint4*>(tile + rr * 32 + h1) = make_uint4(a[2], 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(tile + kBqB * 32 + rr * 32 + h0) = make_uint4(dd[0] | (dd[1] << 16), dd[2], 0u, 0u);
    *reinterpret_cast<uint4*>(tile + kBqB * 32 + rr * 32 + h1) = make_uint4(0u, 0u, 0u, 0u);
  }
  if (DET) {
    // The block's rows lie in one 64-row query block (Npad and the block start are
    // multiples of kRpb, which divides 64): reduce to one atomic per block.
#pragma unroll
    for (int m = kTpr / 2; m >= 1; m >>= 1) nrm += __shfl_xor_sync(0xffffffffu, nrm, m, kTpr);
    float mx = sqrtf(nrm);  // 0 for padded rows
#pragma unroll
    for (int m = kTpr; m < 32; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
    __shared__ float red[8];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 1; w < 8; ++w) mx = fmaxf(mx, red[w]);
      const long long r_first = static_cast<long long>(blockIdx.x) * kRpb;
      const long long bh0 = r_first / Npad;
      atomicMax(dq_bmax + bh0 * (Npad / kBqB) + (r_first - bh0 * Npad) / kBqB, __float_as_uint(mx));
    }
  }
}

// Deterministic mode: per head, the largest |v_j| and the largest |k_jc| (atomicMax
// on float bits, both >= 0).  A block of 256 threads covers 256 rows of one head
// (D / 8 threads per row, 8 elements each, 256 / (D / 8) rows per pass) and issues
// one atomic per value.
constexpr int kBoundRows = 256;
template <int D>
__global__ void __launch_bounds__(256) bwd_kv_bound_kernel(const __nv_bfloat16* __restrict__ k,
                                                           const __nv_bfloat16* __restrict__ v,
                                                           unsigned int* __restrict__ kv_max, int N, int H,
                                                           Strides sk, Strides sv) {
  constexpr int kTpr = D / 8;
  constexpr int kRpp = 256 / kTpr;  // rows per pass
  const int bh = blockIdx.y;
  const int t = threadIdx.x % kTpr;
  const int r0 = blockIdx.x * kBoundRows + (threadIdx.x / kTpr);
  float km = 0.f, vm = 0.f;
  // Every thread runs all passes (the shuffles below need the whole warp); rows
  // past N contribute zeros.
#pragma unroll 1
  for (int pass = 0; pass < kBoundRows / kRpp; ++pass) {
    const int r = r0 + pass * kRpp;
    uint4 kv4 = make_uint4(0, 0, 0, 0), vv4 = make_uint4(0, 0, 0, 0);
    if (r < N) {
      kv4 = *reinterpret_cast<const uint4*>(k + row_offset(sk, bh, H, r) + t * 8);
      vv4 = *reinterpret_cast<const uint4*>(v + row_offset(sv, bh, H, r) + t * 8);
    }
    const __nv_bfloat162* kp = reinterpret_cast<const __nv_bfloat162*>(&kv4);
    const __nv_bfloat162* vp = reinterpret_cast<const __nv_bfloat162*>(&vv4);
    float vn = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 a = __bfloat1622float2(kp[e]);
      const float2 b = __bfloat1622float2(vp[e]);
      km = fmaxf(km, fmaxf(fabsf(a.x), fabsf(a.y)));
      vn = fmaf(b.x, b.x, fmaf(b.y, b.y, vn));
    }
#pragma unroll
    for (int m = kTpr / 2; m >= 1; m >>= 1) vn += __shfl_xor_sync(0xffffffffu, vn, m, kTpr);
    vm = fmaxf(vm, sqrtf(vn));
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    km = fmaxf(km, __shfl_xor_sync(0xffffffffu, km, m));
    vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, m));
  }
  __shared__ float red[2][8];
  if ((threadIdx.x & 31) == 0) {
    red[0][threadIdx.x >> 5] = vm;
    red[1][threadIdx.x >> 5] = km;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < 8; ++w) {
      vm = fmaxf(vm, red[0][w]);
      km = fmaxf(km, red[1][w]);
    }
    atomicMax(kv_max + 2 * bh, __float_as_uint(vm));
    atomicMax(kv_max + 2 * bh + 1, __float_as_uint(km));
  }
}

// dQ = bf16(scale * dQacc), 8 elements per thread.  Deterministic mode: the
// accumulator holds integers in units of 2^-S of the row block's shift S.
template <int D, bool DET>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float* __restrict__ dq_acc,
                                                             __nv_bfloat16* __restrict__ dq, float scale,
                                                             long long n8, const float* __restrict__ dq_bmax,
                                                             const float* __restrict__ kv_max, int N, int Npad, int H,
                                                             Strides sdq) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= n8) return;
  float4 a = reinterpret_cast<const float4*>(dq_acc)[2 * idx];
  float4 b = reinterpret_cast<const float4*>(dq_acc)[2 * idx + 1];
  const long long row = idx * 8 / D;  // (bh, query row) flattened
  const long long bh = row / N;
  const int qrow = static_cast<int>(row - bh * N);
  if (DET) {
    const float inv = pow2f(-det_shift(dq_bmax[bh * (Npad / kBqB) + qrow / kBqB], kv_max[2 * bh], kv_max[2 * bh + 1]));
    auto cv = [&](float x) { return static_cast<float>(__float_as_int(x)) * inv; };
    a = make_float4(cv(a.x), cv(a.y), cv(a.z), cv(a.w));
    b = make_float4(cv(b.x), cv(b.y), cv(b.z), cv(b.w));
  }
  uint4 out;
  out.x = pack_bf16x2(a.x * scale, a.y * scale);
  out.y = pack_bf16x2(a.z * scale, a.w * scale);
  out.z = pack_bf16x2(b.x * scale, b.y * scale);
  out.w = pack_bf16x2(b.z * scale, b.w * scale);
  *reinterpret_cast<uint4*>(dq + row_offset(sdq, bh, H, qrow) + (idx * 8) % D) = out;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

BwdWorkspace bwd_workspace_layout(int B, int H, int N, int d) {
  BwdWorkspace w{};
  const size_t bh = static_cast<size_t>(B) * H;
  const size_t npad = (static_cast<size_t>(N) + kBqB - 1) / kBqB * kBqB;
  w.npad = static_cast<int>(npad);
  w.off_dq = 0;
  w.off_aug = align256(bh * N * d * sizeof(float));
  w.off_dqmax = w.off_aug + align256(bh * npad * 64);  // two 32-byte operand rows per query row
  w.off_kvmax = w.off_dqmax + align256(bh * (npad / kBqB) * sizeof(float));
  w.total = w.off_kvmax + align256(bh * 2 * sizeof(float));
  return w;
}

namespace {

template <int D>
cudaError_t launch_bwd_prep_d(const BwdArgs& a, cudaStream_t stream) {
  const int BH = a.B * a.H;
  const BwdWorkspace w = bwd_workspace_layout(a.B, a.H, a.N, a.d);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  const long long rows_pad = static_cast<long long>(BH) * w.npad;
  unsigned int* dq_bmax = reinterpret_cast<unsigned int*>(ws + w.off_dqmax);
  if (a.deterministic) {
    // The block and head maxima are built with atomicMax from zero.
    cudaError_t e = cudaMemsetAsync(ws + w.off_dqmax, 0, w.total - w.off_dqmax, stream);
    if (e) return e;
    bwd_kv_bound_kernel<D><<<dim3(static_cast<unsigned>((a.N + kBoundRows - 1) / kBoundRows), BH), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(a.k), static_cast<const __nv_bfloat16*>(a.v),
        reinterpret_cast<unsigned int*>(ws + w.off_kvmax), a.N, a.H, a.sk, a.sv);
    if ((e = cudaGetLastError())) return e;
  }
  constexpr int kRpb = 256 / (D / 8);
  auto kern = a.deterministic ? bwd_preprocess_kernel<D, true> : bwd_preprocess_kernel<D, false>;
  kern<<<static_cast<unsigned>(rows_pad / kRpb), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dout), a.lse,
      ws + w.off_aug, reinterpret_cast<float*>(ws + w.off_dq), dq_bmax, a.N, w.npad, rows_pad, a.H, a.so, a.sdo);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd_main_d(const BwdArgs& a, cudaStream_t stream) {
  using C = BwdCfg<D>;
  const int BH = a.B * a.H;
  const BwdWorkspace w = bwd_workspace_layout(a.B, a.H, a.N, a.d);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  cudaError_t e;
  CUtensorMap tq, tk, tv, tdo, tdk, tdv;
  constexpr auto kBf16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if ((e = make_tmap_4d(&tq, a.q, kBf16, 2, D, a.N, a.H, a.B, a.sq.s, 64, kBqB))) return e;
  if ((e = make_tmap_4d(&tdo, a.dout, kBf16, 2, D, a.N, a.H, a.B, a.sdo.s, 64, kBqB))) return e;
  if ((e = make_tmap_4d(&tk, a.k, kBf16, 2, D, a.N, a.H, a.B, a.sk.s, 64, kBkB))) return e;
  if ((e = make_tmap_4d(&tv, a.v, kBf16, 2, D, a.N, a.H, a.B, a.sv.s, 64, kBkB))) return e;
  if ((e = make_tmap_4d(&tdk, a.dk, kBf16, 2, D, a.N, a.H, a.B, a.sdk.s, 64, kBkB))) return e;
  if ((e = make_tmap_4d(&tdv, a.dv, kBf16, 2, D, a.N, a.H, a.B, a.sdv.s, 64, kBkB))) return e;
  auto kern = a.deterministic ? (a.causal ? bwd_main_kernel<D, true, true> : bwd_main_kernel<D, false, true>)
                              : (a.causal ? bwd_main_kernel<D, true, false> : bwd_main_kernel<D, false, false>);
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes))) return e;
  // The register split assumes the block launches with kLaunchRegs per thread.
  cudaFuncAttributes fattr;
  if ((e = cudaFuncGetAttributes(&fattr, kern))) return e;
  if (static_cast<uint32_t>(fattr.numRegs) < kLaunchRegs) return cudaErrorInvalidConfiguration;
  const int nkb = (a.N + kBkB - 1) / kBkB;
  kern<<<static_cast<unsigned>(nkb * BH), kThreads, C::kSmemBytes, stream>>>(
      tq, tk, tv, tdo, tdk, tdv, ws + w.off_aug, reinterpret_cast<float*>(ws + w.off_dq),
      reinterpret_cast<const float*>(ws + w.off_dqmax), reinterpret_cast<const float*>(ws + w.off_kvmax), a.N, w.npad,
      a.H, BH, nkb, a.scale, a.scale * kLog2e, a.err_word, a.dbg.wait_limit_ns);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd_dq_d(const BwdArgs& a, cudaStream_t stream) {
  const BwdWorkspace w = bwd_workspace_layout(a.B, a.H, a.N, a.d);
  const uint8_t* ws = static_cast<const uint8_t*>(a.workspace);
  const float* dq_acc = reinterpret_cast<const float*>(ws + w.off_dq);
  const long long n8 = static_cast<long long>(a.B) * a.H * a.N * D / 8;
  auto kern = a.deterministic ? bwd_dq_convert_kernel<D, true> : bwd_dq_convert_kernel<D, false>;
  kern<<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, stream>>>(
      dq_acc, static_cast<__nv_bfloat16*>(a.dq), a.scale, n8, reinterpret_cast<const float*>(ws + w.off_dqmax),
      reinterpret_cast<const float*>(ws + w.off_kvmax), a.N, w.npad, a.H, a.sdq);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_prep(const BwdArgs& a, cudaStream_t stream) {
  return a.d == 64 ? launch_bwd_prep_d<64>(a, stream) : launch_bwd_prep_d<128>(a, stream);
}

cudaError_t launch_bwd_main(const BwdArgs& a, cudaStream_t stream) {
  return a.d == 64 ? launch_bwd_main_d<64>(a, stream) : launch_bwd_main_d<128>(a, stream);
}

cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t stream) {
  return a.d == 64 ? launch_bwd_dq_d<64>(a, stream) : launch_bwd_dq_d<128>(a, stream);
}

cudaError_t launch_bwd_bf16(const BwdArgs& a, cudaStream_t stream) {
  cudaError_t e;
  if ((e = launch_bwd_prep(a, stream))) return e;
  if ((e = launch_bwd_main(a, stream))) return e;
  return launch_bwd_dq(a, stream);
}

}  // namespace fa
