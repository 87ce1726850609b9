// Exact attention forward, bf16 in / bf16 out, fp32 logsumexp, for sm_103a.
//
// Method ("FlashAttention-Skalierung, Multi-GPU-Training und
// Gewichtsquantisierung", section 1; "FlashAttention-2 (DE)", sections
// "Hintergrund" and "Technische Architektur und Funktionsprinzipien"): the
// N x N score matrix is never materialised.  Each CTA owns one block of 128
// query rows (outer loop over Q blocks) and streams the K/V blocks of its head
// through shared memory (inner loop), keeping a running row maximum m and row
// sum l (online softmax).  The single division by l happens once, after the
// inner loop.
//
// GB300 mapping of the pages' ideas:
//  * TMA copies (asynchronous copy unit, FlashAttention-3 bullet "Asynchrone
//    Datenübertragung") move Q once and K_j, V_j through a ring of
//    shared-memory slots guarded by full/empty mbarriers.
//  * Warp specialisation (bullet "Warp-Spezialisierung"): warp 4 issues TMA,
//    one thread of warp 5 issues tcgen05 MMAs, warps 0-3 run the softmax (one
//    thread per query row = one TMEM lane), so the exponentials of block j
//    overlap the tensor-core work of blocks j-1 (P V) and j+1 (Q K^T).
//  * S = Q K_j^T accumulates in TMEM (two buffers, alternating); P is written
//    back over its own S buffer as packed bf16 and fed to the P V MMA straight
//    from TMEM, so P never touches shared memory.
//  * The O accumulator stays in TMEM for the whole inner loop.  It is rescaled
//    only when a row maximum grows by more than 2^8 ("rescale as late as
//    possible"): until then exponentials are taken against the stale maximum,
//    which keeps O and l consistent and the final O/l exact.
//
// Every mbarrier wait is bounded (see fa_device.cuh); on expiry the CTA sets a
// device error word, drains its own in-flight copies, frees TMEM and exits.
#include <math.h>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kThreads = 192;          // warps 0-3 softmax + epilogue, warp 4 TMA, warp 5 MMA
constexpr int kWarpLoad = 4;
constexpr int kWarpMma = 5;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: stale-max exponentials stay <= 256
constexpr float kLn2 = 0.69314718055994530942f;

// Sites recorded in the error word when a wait expires.
enum : uint32_t {
  kSiteLoadEmpty = 0x101,
  kSiteMmaQ = 0x201,
  kSiteMmaK = 0x202,
  kSiteMmaP = 0x203,
  kSiteMmaV = 0x204,
  kSiteSoftS = 0x301,
  kSiteSoftO = 0x302,
  kSiteEpi = 0x303,
};

template <int D>
struct FwdCfg {
  static constexpr int kBoxes = D / kBoxCols;
  static constexpr int kBoxBytes = kBlockK * kBoxCols * 2;  // 16 KB: 128 rows x 128 bytes
  static constexpr int kTileBytes = kBlockK * D * 2;        // one Q, K or V tile
  static constexpr int kSlots = D == 128 ? 5 : 8;
  static constexpr int kQOff = 0;
  static constexpr int kRingOff = kTileBytes;
  static constexpr int kBarOff = kRingOff + kSlots * kTileBytes;
  // q_full, full[kSlots], empty[kSlots], s_full[2], p_full[2], o_done[2], epi, drain
  static constexpr int kNumBars = 1 + 2 * kSlots + 2 + 2 + 2 + 1 + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + slack to align the base to 1024
  static constexpr uint32_t kColSBase = 0;  // S buffer b occupies columns [128*b, 128*b + 128)
  static constexpr uint32_t kColO = 256;
  static __device__ __forceinline__ uint32_t col_s(int b) { return kColSBase + 128u * static_cast<uint32_t>(b); }
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& wc, uint32_t site) {
  const bool ok = mbar_wait(bar, parity, wc, site);
  return __all_sync(0xffffffffu, ok);
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_bf16_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    float* __restrict__ lse, int N, int BH, int nqt, float scale_log2, unsigned int* err_word,
                    unsigned long long wait_ns, int fault) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::kQOff;
  uint8_t* sRing = smem + C::kRingOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* bar_q = bars;
  uint64_t* bar_full = bars + 1;
  uint64_t* bar_empty = bar_full + C::kSlots;
  uint64_t* bar_s = bar_empty + C::kSlots;
  uint64_t* bar_p = bar_s + 2;
  uint64_t* bar_o = bar_p + 2;
  uint64_t* bar_epi = bar_o + 2;
  uint64_t* bar_drain = bar_epi + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work unit: (query block, head).  Causal blocks are issued heaviest first.
  int qt, bh;
  if (CAUSAL) {
    qt = nqt - 1 - static_cast<int>(blockIdx.x) / BH;
    bh = static_cast<int>(blockIdx.x) % BH;
  } else {
    qt = static_cast<int>(blockIdx.x) % nqt;
    bh = static_cast<int>(blockIdx.x) / nqt;
  }
  const int nkt_all = (N + kBlockK - 1) / kBlockK;
  const int nkt = CAUSAL ? min(qt + 1, nkt_all) : nkt_all;

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_s[b], 1);
      mbar_init(&bar_p[b], 4);
      mbar_init(&bar_o[b], 1);
    }
    mbar_init(bar_epi, 4);
    mbar_init(bar_drain, 1);
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

  if (warp == kWarpLoad) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_q, C::kTileBytes);
#pragma unroll
      for (int b = 0; b < C::kBoxes; ++b) tma_load_3d(sQ + b * C::kBoxBytes, &tm_q, bar_q, b * kBoxCols, qt * kBlockQ, bh);

      // Ring order = MMA consumption order: K0, K1, V0, K2, V1, ..., K_{n-1}, V_{n-2}, V_{n-1}.
      int issued = 0;
      bool ok = true;
      auto push = [&](const CUtensorMap* tm, int j) -> bool {
        const int slot = issued % C::kSlots;
        const uint32_t ph = (issued / C::kSlots) & 1;
        if (!mbar_wait(&bar_empty[slot], ph ^ 1, wc, kSiteLoadEmpty)) return false;
        if (fault == 1 && tm == &tm_k && j == 1) return false;  // test-only: K block 1 never arrives
        mbar_arrive_expect_tx(&bar_full[slot], C::kTileBytes);
        uint8_t* dst = sRing + slot * C::kTileBytes;
#pragma unroll
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_3d(dst + b * C::kBoxBytes, tm, &bar_full[slot], b * kBoxCols, j * kBlockK, bh);
        ++issued;
        return true;
      };
      for (int j = 0; ok && j < nkt; ++j) {
        ok = push(&tm_k, j);
        if (ok && j >= 1) ok = push(&tm_v, j - 1);
      }
      if (ok) ok = push(&tm_v, nkt - 1);
      if (!ok) {
        // Drain: the last (up to kSlots) issued copies may still be landing in shared memory.
        mbar_wait_drain(bar_q, 0, wait_ns);
        for (int t = max(0, issued - C::kSlots); t < issued; ++t)
          mbar_wait_drain(&bar_full[t % C::kSlots], (t / C::kSlots) & 1, wait_ns);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(kBlockQ, kBlockK, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kBlockQ, D, 0, 1);
      const uint32_t q_addr = smem_u32(sQ);
      const uint32_t ring_addr = smem_u32(sRing);
      int t = 0;
      bool ok = mbar_wait(bar_q, 0, wc, kSiteMmaQ);
      tc_fence_after();

      // O += P_jj V_jj : A = P from TMEM (K-major, 2 bf16 per column), B = V tile,
      // MN-major (d contiguous): 8 key rows per 1024-byte swizzle atom (SBO),
      // 64 d-columns per TMA box (LBO = one box).
      auto pv = [&](int jj) -> bool {
        const int sb = jj & 1;
        if (!mbar_wait(&bar_p[sb], (jj >> 1) & 1, wc, kSiteMmaP)) return false;
        const int slot = t % C::kSlots;
        if (!mbar_wait(&bar_full[slot], (t / C::kSlots) & 1, wc, kSiteMmaV)) return false;
        tc_fence_after();
        const uint32_t vbase = ring_addr + slot * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kBlockK / 16; ++kk) {
          const uint64_t bdesc = sdesc_sw128(vbase + kk * 16 * 128, C::kBoxBytes, 1024);
          mma_bf16_ts(tmem + C::kColO, tmem + C::col_s(sb) + kk * 8, bdesc, idesc_pv, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bar_o[sb]);
        mma_commit(&bar_empty[slot]);
        ++t;
        return true;
      };

      for (int j = 0; ok && j < nkt; ++j) {
        // S_j = Q K_j^T : both operands K-major (d contiguous), 16 d-columns per MMA.
        const int slot = t % C::kSlots;
        if (!mbar_wait(&bar_full[slot], (t / C::kSlots) & 1, wc, kSiteMmaK)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t kbase = ring_addr + slot * C::kTileBytes;
        const uint32_t sb = j & 1;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * C::kBoxBytes + (kk % 4) * 32;
          mma_bf16_ss(tmem + C::col_s(sb), sdesc_sw128(q_addr + off, 16, 1024), sdesc_sw128(kbase + off, 16, 1024),
                      idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bar_s[sb]);
        mma_commit(&bar_empty[slot]);
        ++t;
        if (j >= 1) ok = pv(j - 1);
      }
      if (ok) pv(nkt - 1);
      // Every issued MMA must finish before TMEM is released.
      mma_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0, wait_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax warps (0..3)
    const int row = threadIdx.x;  // tile row == TMEM lane
    const int qrow = qt * kBlockQ + row;
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float m_used = -INFINITY;  // running maximum in log2 units (possibly stale, see header)
    float l = 0.f;
    bool ok = true;

    for (int j = 0; j < nkt; ++j) {
      const int sb = j & 1;
      if (!warp_wait(&bar_s[sb], (j >> 1) & 1, wc, kSiteSoftS)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t r[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(trow + C::col_s(sb) + c * 32, r[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_wait32(r[c]);

      const int kbase = j * kBlockK;
      const bool need_mask = (kbase + kBlockK > N) || (CAUSAL && j == qt);
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int key = kbase + c * 32 + i;
            const bool masked = key >= N || (CAUSAL && key > qrow);
            if (masked) r[c][i] = __float_as_uint(-INFINITY);
          }
      }
      // Row maximum of the raw scores (scale > 0, so scaling commutes with max).
      float mx[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float a = __uint_as_float(r[c][0]);
#pragma unroll
        for (int i = 1; i < 31; i += 2) a = max3(a, __uint_as_float(r[c][i]), __uint_as_float(r[c][i + 1]));
        mx[c] = fmaxf(a, __uint_as_float(r[c][31]));
      }
      const float rmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      const float m_tile = rmax * scale_log2;
      const float m_new = fmaxf(m_used, m_tile);

      if (j == 0) {
        m_used = (m_new == -INFINITY) ? 0.f : m_new;
      } else {
        const bool need = m_new > m_used + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          // O must hold P_{j-1} V_{j-1} before it is rescaled.
          const int pj = j - 1;
          if (!warp_wait(&bar_o[pj & 1], (pj >> 1) & 1, wc, kSiteSoftO)) {
            ok = false;
            break;
          }
          tc_fence_after();
          float alpha = 1.f;
          if (need) {
            alpha = ex2_approx(m_used - m_new);
            m_used = m_new;
          }
          l *= alpha;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(trow + C::kColO + c * 32, o);
            tmem_ld_wait32(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(trow + C::kColO + c * 32, o);
          }
          tmem_st_wait();
        }
      }

      // P = exp2(S * scale * log2(e) - m), packed to bf16 pairs over the S buffer.
      const float neg_m = -m_used;
      float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(r[c][2 * i]), scale_log2, neg_m));
          const float p1 = ex2_approx(fmaf(__uint_as_float(r[c][2 * i + 1]), scale_log2, neg_m));
          part[c] += p0 + p1;
          pk[i] = pack_bf16x2(p0, p1);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) r[c][i] = pk[i];
      }
      l += (part[0] + part[1]) + (part[2] + part[3]);
      // r[0][0..15], r[1][0..15], ... hold 64 packed columns; gather into two stores of 32.
      uint32_t st0[32], st1[32];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        st0[i] = r[0][i];
        st0[16 + i] = r[1][i];
        st1[i] = r[2][i];
        st1[16 + i] = r[3][i];
      }
      tmem_st32(trow + C::col_s(sb), st0);
      tmem_st32(trow + C::col_s(sb) + 32, st1);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_p[sb]);
    }

    // ------------------------------------------------------------ epilogue
    if (ok && nkt >= 2) ok = warp_wait(&bar_o[(nkt - 2) & 1], ((nkt - 2) >> 1) & 1, wc, kSiteSoftO);
    if (ok) ok = warp_wait(&bar_o[(nkt - 1) & 1], ((nkt - 1) >> 1) & 1, wc, kSiteSoftO);
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      // O row -> bf16 -> the Q staging area (free: every Q K^T MMA has completed),
      // laid out exactly as the 128-byte-swizzled TMA box expects.
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(trow + C::kColO + c * 32, o);
        tmem_ld_wait32(o);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
        uint8_t* box = sQ + (c / 2) * C::kBoxBytes + row * 128;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int chunk = (c % 2) * 4 + q4;
          uint4 val = make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
          *reinterpret_cast<uint4*>(box + ((chunk ^ (row & 7)) * 16)) = val;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_epi);
      if (qrow < N) lse[static_cast<size_t>(bh) * N + qrow] = (m_used + log2f(l)) * kLn2;
      if (threadIdx.x == 0 && mbar_wait(bar_epi, 0, wc, kSiteEpi)) {
#pragma unroll
        for (int b = 0; b < C::kBoxes; ++b) tma_store_3d(&tm_o, sQ + b * C::kBoxBytes, b * kBoxCols, qt * kBlockQ, bh);
        tma_store_commit_and_wait_read();
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

template <int D, bool CAUSAL>
cudaError_t launch_fwd_impl(const FwdArgs& a, cudaStream_t stream) {
  using C = FwdCfg<D>;
  const int BH = a.B * a.H;
  CUtensorMap tq, tk, tv, to;
  cudaError_t e;
  if ((e = make_tmap_3d(&tq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, kBoxCols, kBlockQ))) return e;
  if ((e = make_tmap_3d(&tk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, kBoxCols, kBlockK))) return e;
  if ((e = make_tmap_3d(&tv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, kBoxCols, kBlockK))) return e;
  if ((e = make_tmap_3d(&to, a.o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, kBoxCols, kBlockQ))) return e;
  auto kern = fwd_bf16_kernel<D, CAUSAL>;
  // Per device and idempotent; cheap enough to repeat on every launch.
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes))) return e;
  const int nqt = (a.N + kBlockQ - 1) / kBlockQ;
  const float scale_log2 = a.scale * 1.4426950408889634f;
  dim3 grid(static_cast<unsigned>(nqt * BH));
  kern<<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, to, a.lse, a.N, BH, nqt, scale_log2, a.err_word,
                                                   a.dbg.wait_limit_ns, a.dbg.fault);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_bf16(const FwdArgs& a, cudaStream_t stream) {
  if (a.d == 64) return a.causal ? launch_fwd_impl<64, true>(a, stream) : launch_fwd_impl<64, false>(a, stream);
  return a.causal ? launch_fwd_impl<128, true>(a, stream) : launch_fwd_impl<128, false>(a, stream);
}

}  // namespace fa
