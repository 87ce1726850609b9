// 4-bit-weight, 16-bit-activation matrix product (W4A16) for sm_103a.
//
// "FlashAttention-Skalierung, Multi-GPU-Training und Gewichtsquantisierung",
// section 3 ("Wie spezielle CUDA-Kernels während der Ausführung dequantisieren
// (W4A16)"): the weights stay packed in memory (eight 4-bit codes per 32-bit
// word), are taken apart in registers with shifts and masks, turned back into
// fp16 with stored scale and zero-point factors, and fed with the fp16
// activations to the tensor cores; the unpacked weights never return to memory.
//
//   Y[m, n] = sum_k X[m, k] * fp16((q[n, k] - z[k/128, n]) * s[k/128, n])
//
// Decode-sized M (<= 128 tokens) makes this a stream over the weights, so the
// bound is HBM: 0.5 byte per weight plus 3 bytes of scale and zero per 128.
//
// GB300 mapping.  A persistent CTA per SM takes work units = (128 output rows,
// K range).  Per 256-wide K chunk:
//  * warp 0 loads, by TMA, the packed 128 x 256 weight tile (16 KB), the chunk's
//    activations X[:, k0:k0+256] (four 64-column boxes, rows past M zero-filled)
//    and the two groups' scales and zero points into a ring of stages;
//  * two sets of eight dequantising warps take alternate chunks (thread = weight
//    row = TMEM lane; warpgroup g of a set takes group g of the chunk).  Each word
//    becomes four fp16 pairs: the pair's two codes are masked into the mantissa
//    of 1024.0 (bits 0-3 and 16-19) or of 64.0 (bits 4-7 and 20-23, whose weight
//    there is 1), so one shift serves the word's upper byte pair; then one exact
//    subtraction of 1024 + z or 64 + z and one multiplication by s (the only
//    rounding).  The pairs go to TMEM, two fp16 per column, as the MMA's A operand;
//  * two threads issue tcgen05.mma kind::f16, one per 128-wide group of the chunk,
//    A from TMEM (128 rows x 16 k) and B = X from shared memory (K-major, 128-byte
//    swizzle), each accumulating its share of Y^T[128 rows x M] in its own TMEM
//    columns; three A buffers let the dequantisation of the next chunks overlap
//    the MMAs of this one;
//  * after the unit's last chunk, warpgroup 0 of the set that unpacked it adds the
//    two accumulators and writes fp16 Y (one split) or fp32 partials (several),
//    coalesced along n.
// Every wait is bounded, as in the attention kernels.
#include <cuda_fp16.h>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kW4Sets = 2;       // dequantising warp sets, alternate chunks
constexpr int kW4Threads = 128 + 256 * kW4Sets;  // 0 TMA, 1-2 MMA issuers (1 owns TMEM), 3 idle, then the sets
constexpr int kW4Rows = 128;     // output rows per unit (MMA M, TMEM lanes)
constexpr int kW4Kc = 256;       // K per chunk: two groups of 128
constexpr uint32_t kW4TmemCols = 512;

enum : uint32_t {
  kSiteW4Load = 0x401,
  kSiteW4Mma = 0x402,
  kSiteW4Deq = 0x403,
  kSiteW4Epi = 0x404,
};

template <int MP>  // tokens padded to 16 or a multiple of 32 (the MMA's N)
struct W4Cfg {
  static constexpr int kWBytes = kW4Rows * 128;              // 128 rows x 32 words
  static constexpr int kXBox = MP * 128;                      // MP rows x 64 fp16
  static constexpr int kXBytes = 4 * kXBox;
  static constexpr int kSBytes = 2 * kW4Rows * 2;             // two groups x 128 fp16
  static constexpr int kZBytes = 2 * kW4Rows;                 // two groups x 128 uint8
  static constexpr int kOffX = kWBytes;
  static constexpr int kOffS = kOffX + kXBytes;
  static constexpr int kOffZ = kOffS + kSBytes;
  static constexpr int kStageTx = kOffZ + kZBytes;
  static constexpr int kStageBytes = (kStageTx + 1023) / 1024 * 1024;
  // As many stages as fit next to the barriers (more bytes in flight per SM).
  static constexpr int kStages = (220 * 1024 / kStageBytes) < 8 ? (220 * 1024 / kStageBytes) : 8;
  static constexpr int kBarOff = kStages * kStageBytes;
  // full[S], empty[S], afull[kA][2], aempty[kA], dfull, dempty, drain
  static constexpr int kA = MP <= 64 ? 3 : 2;  // A buffers in TMEM (128 columns each)
  static constexpr int kNumBars = 2 * kStages + 3 * kA + 1 + 1 + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
  // A buffers at 0, 128, ...; then one accumulator per group of the chunk (each group's MMAs
  // are issued by their own thread, so the two streams overlap in the tensor pipe).
  static constexpr uint32_t kDCols = MP < 32 ? 32 : MP;
  static constexpr uint32_t kColA = 0, kColD0 = 128 * kA, kColD1 = 128 * kA + kDCols;
  static_assert(kColD1 + kDCols <= 512, "TMEM budget");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ bool w4_warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& wc, uint32_t site) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, wc, site));
}

template <int MP>
__global__ void __launch_bounds__(kW4Threads, 1)
    w4a16_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                 const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_z,
                 __half* __restrict__ y, float* __restrict__ partials, int M, int N, int nstrips, int nsplit,
                 int kchunks, int cps, unsigned int* err_word, unsigned long long wait_ns) {
  using C = W4Cfg<MP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* bar_full = bars;
  uint64_t* bar_empty = bar_full + C::kStages;
  uint64_t* bar_afull = bar_empty + C::kStages;  // [kA][2] group g of an A buffer written
  uint64_t* bar_aempty = bar_afull + 2 * C::kA;  // [kA] A buffer consumed by both issuers' MMAs
  uint64_t* bar_dfull = bar_aempty + C::kA;      // unit's Y^T complete in TMEM
  uint64_t* bar_dempty = bar_dfull + 1;          // Y^T read out
  uint64_t* bar_drain = bar_dempty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int total = nstrips * nsplit;
  const int G = static_cast<int>(gridDim.x);
  // Unit w = strip + nstrips * split; CTA c takes w = c, c + G, ...
  auto unit_range = [&](int w, int& strip, int& c0, int& c1) {
    strip = w % nstrips;
    const int sp = w / nstrips;
    c0 = min(sp * cps, kchunks);
    c1 = min(c0 + cps, kchunks);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 8 + 2);  // the eight dequantising warps of the item's set + both issuers' commits
    }
    for (int b = 0; b < C::kA; ++b) {
      mbar_init(&bar_afull[2 * b], 4);
      mbar_init(&bar_afull[2 * b + 1], 4);
      mbar_init(&bar_aempty[b], 2);
    }
    mbar_init(bar_dfull, 2);
    mbar_init(bar_dempty, 4);
    mbar_init(bar_drain, 2);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kW4TmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, err_word, wait_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int item = 0;
      bool ok = true;
      for (int w = static_cast<int>(blockIdx.x); ok && w < total; w += G) {
        int strip, c0, c1;
        unit_range(w, strip, c0, c1);
        for (int c = c0; ok && c < c1; ++c, ++item) {
          const int slot = item % C::kStages;
          if (!(ok = mbar_wait(&bar_empty[slot], ((item / C::kStages) & 1) ^ 1, wc, kSiteW4Load))) break;
          uint8_t* st = smem + slot * C::kStageBytes;
          mbar_arrive_expect_tx(&bar_full[slot], C::kStageTx);
          tma_load_2d(st, &tm_w, &bar_full[slot], c * (kW4Kc / 8), strip * kW4Rows);
#pragma unroll
          for (int bx = 0; bx < 4; ++bx)
            tma_load_2d(st + C::kOffX + bx * C::kXBox, &tm_x, &bar_full[slot], c * kW4Kc + bx * 64, 0);
          tma_load_2d(st + C::kOffS, &tm_s, &bar_full[slot], strip * kW4Rows, 2 * c);
          tma_load_2d(st + C::kOffZ, &tm_z, &bar_full[slot], strip * kW4Rows, 2 * c);
        }
      }
      if (!ok) {  // let the copies already issued land before the CTA exits
        for (int t = max(0, item - C::kStages); t < item; ++t)
          mbar_wait_drain(&bar_full[t % C::kStages], (t / C::kStages) & 1, wait_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------- MMA issuers (thread g: group g of each chunk)
    if (lane == 0) {
      const int g = warp - 1;
      const uint32_t dcol = g == 0 ? C::kColD0 : C::kColD1;
      constexpr uint32_t idesc = idesc_f16_f32(kW4Rows, MP < 16 ? 16 : MP, 0, 0);  // rows x tokens, K-major B
      const uint64_t xdesc = sdesc_sw128(smem_u32(smem + C::kOffX), 16, 1024);
      int item = 0, units = 0;
      bool ok = true;
      for (int w = static_cast<int>(blockIdx.x); ok && w < total; w += G) {
        int strip, c0, c1;
        unit_range(w, strip, c0, c1);
        if (c1 <= c0) continue;
        for (int c = c0; ok && c < c1; ++c, ++item) {
          const int slot = item % C::kStages;
          const int b = item % C::kA;
          if (!(ok = mbar_wait(&bar_full[slot], (item / C::kStages) & 1, wc, kSiteW4Mma))) break;
          if (!(ok = mbar_wait(&bar_afull[2 * b + g], (item / C::kA) & 1, wc, kSiteW4Mma))) break;
          // The unit's first MMA overwrites Y^T: the previous unit's must be read out.
          if (c == c0 && units > 0 && !(ok = mbar_wait(bar_dempty, (units - 1) & 1, wc, kSiteW4Mma))) break;
          tc_fence_after();
          const uint32_t st = slot * C::kStageBytes;
#pragma unroll
          for (int j = 0; j < 8; ++j) {  // kind::f16; the descriptor selects fp16 operands
            const int kk = 8 * g + j;      // 16-wide K step within the chunk
            mma_bf16_ts(tmem + dcol, tmem + C::kColA + 128u * b + 8u * kk,
                        sdesc_add(xdesc, st + (kk / 4) * C::kXBox + (kk % 4) * 32), idesc,
                        (c > c0 || j > 0) ? 1u : 0u);
          }
          mma_commit(&bar_aempty[b]);
          mma_commit(&bar_empty[slot]);
        }
        if (!ok) break;
        mma_commit(bar_dfull);
        ++units;
      }
      mma_commit(bar_drain);
      mbar_wait_drain(bar_drain, 0, wait_ns);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------ dequantisation (thread = weight row)
    const int set = (warp - 4) >> 3;         // this set unpacks items with item % kW4Sets == set
    const int g = ((warp - 4) >> 2) & 1;     // group of the chunk this warpgroup unpacks
    const int r = ((warp & 3) << 5) + lane;  // row within the 128-row tile
    const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    int item = 0, units = 0;
    bool ok = true;
    for (int w = static_cast<int>(blockIdx.x); ok && w < total; w += G) {
      int strip, c0, c1;
      unit_range(w, strip, c0, c1);
      if (c1 <= c0) continue;
      for (int c = c0; ok && c < c1; ++c, ++item) {
        if (item % kW4Sets != set) continue;
        const int slot = item % C::kStages;
        const int b = item % C::kA;
        if (!(ok = w4_warp_wait(&bar_full[slot], (item / C::kStages) & 1, wc, kSiteW4Deq))) break;
        if (item >= C::kA && !(ok = w4_warp_wait(&bar_aempty[b], ((item - C::kA) / C::kA) & 1, wc, kSiteW4Deq)))
          break;
        tc_fence_after();
        const uint8_t* st = smem + slot * C::kStageBytes;
        const __half s = reinterpret_cast<const __half*>(st + C::kOffS)[g * kW4Rows + r];
        const int z = st[C::kOffZ + g * kW4Rows + r];
        const __half2 s2 = __halves2half2(s, s);
        const __half zb = __int2half_rn(1024 + z);  // exact: integers below 2048
        const __half2 zb2 = __halves2half2(zb, zb);
        const __half zs = __int2half_rn(64 + z);
        const __half2 zs2 = __halves2half2(zs, zs);
        // This warpgroup's 16 words of the row: 16-byte chunks 4g .. 4g+3 of the
        // 128-byte swizzled row.
        const uint8_t* wrow = st + r * 128;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t out[32];
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            const int chunk = 4 * g + 2 * half + ch;
            const uint4 v = *reinterpret_cast<const uint4*>(wrow + ((chunk ^ (r & 7)) * 16));
            const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                // Codes of k = 8w + 2i (bits 4i..) and 8w + 2i + 1 (bits 4i + 16..).
                // Even i: mantissa bits 0-3 of 1024.0 (value 1024 + code); odd i: bits
                // 4-7 of 64.0 (value 64 + code).  Then (code - z) exactly, then times s.
                const uint32_t src = i < 2 ? wd[e] : (wd[e] >> 8);
                const uint32_t t = (i & 1) ? ((src & 0x00F000F0u) | 0x54005400u) : ((src & 0x000F000Fu) | 0x64006400u);
                const __half2 d = __hsub2(*reinterpret_cast<const __half2*>(&t), (i & 1) ? zs2 : zb2);
                const __half2 wv = __hmul2(d, s2);
                out[(ch * 4 + e) * 4 + i] = *reinterpret_cast<const uint32_t*>(&wv);
              }
            }
          }
          tmem_st32(trow + C::kColA + 128u * b + 64u * g + 32u * half, out);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bar_afull[2 * b + g]);
          mbar_arrive(&bar_empty[slot]);
        }
      }
      if (!ok) break;
      if (g == 0 && (item - 1) % kW4Sets == set) {
        // ------------------- epilogue (warpgroup 0 of the set that unpacked the last chunk)
        if (!(ok = w4_warp_wait(bar_dfull, units & 1, wc, kSiteW4Epi))) break;
        tc_fence_after();
        const int n = strip * kW4Rows + r;
        const int sp = w / nstrips;
#pragma unroll 1
        for (int mc = 0; mc < (MP + 31) / 32; ++mc) {  // MP = 16 reads 16 unused columns too
          uint32_t v[32], v1[32];
          tmem_ld32(trow + C::kColD0 + 32u * mc, v);
          tmem_ld32(trow + C::kColD1 + 32u * mc, v1);
          tmem_ld_wait32(v);
          tmem_ld_wait32(v1);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(v1[j]));
          if (n < N) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int m = mc * 32 + j;
              if (m < M) {
                if (nsplit == 1)
                  y[static_cast<size_t>(m) * N + n] = __float2half_rn(__uint_as_float(v[j]));
                else
                  partials[(static_cast<size_t>(sp) * M + m) * N + n] = __uint_as_float(v[j]);
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_dempty);
      }
      ++units;
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kW4TmemCols);
  }
}

// ------------------------------------------------------------------------------
// One token (M = 1): the product is a matrix-vector stream, HBM-bound work that the
// tensor cores only slow down here (each M=128 x K=16 MMA covers 2048 weights and
// its dequantised A operand has to pass through TMEM; measured, that path issues
// one MMA per ~96 cycles per SM while the TMEM stores run, below the HBM rate).
// Here the dequantised weights go straight from registers into mixed-precision
// FMAs (fp16 x fp16 products, exact in fp32, summed in fp32).
//
// CTA = 8 warps x 4 rows = 32 output rows; it stages the rows' scales and zero
// points for all groups in shared memory (one coalesced pass), then each warp
// streams its 4 rows: per step, lane l takes words 4l .. 4l+3 of a 128-word block
// of every row (one 16-byte streaming load per row) and the 32 activations they
// multiply (16-byte loads, L1-resident, shared by the 4 rows).  The dequantisation
// is the tensor path's, bit for bit.  A warp reduction finishes each row.
constexpr int kGvWarps = 8;
constexpr int kGvRowsPerWarp = 4;
constexpr int kGvRows = kGvWarps * kGvRowsPerWarp;
constexpr int kGvMaxM = 1;  // measured: from M = 2 the tensor-core path is faster

__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// acc += lo(w) * lo(x) + hi(w) * hi(x): fp16 operands, fp32 product and sum.
__device__ __forceinline__ float fma2_f16_f32(uint32_t w, uint32_t x, float acc) {
  asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
      "mov.b32 {wl, wh}, %1;\n\t"
      "mov.b32 {xl, xh}, %2;\n\t"
      "fma.rn.f32.f16 %0, wl, xl, %0;\n\t"
      "fma.rn.f32.f16 %0, wh, xh, %0;\n\t}"
      : "+f"(acc)
      : "r"(w), "r"(x));
  return acc;
}

template <int MP>
__global__ void __launch_bounds__(kGvWarps * 32) w4a16_gemv_kernel(const __half* __restrict__ x,
                                                                    const uint32_t* __restrict__ wq,
                                                                    const __half* __restrict__ scales,
                                                                    const uint8_t* __restrict__ zeros,
                                                                    __half* __restrict__ y, int M, int N, int K) {
  extern __shared__ __align__(16) uint8_t gv_smem[];
  const int G = K / 128;
  __half* s_sm = reinterpret_cast<__half*>(gv_smem);  // [G][32]
  uint8_t* z_sm = gv_smem + static_cast<size_t>(G) * kGvRows * 2;  // [G][32]
  const int n0 = blockIdx.x * kGvRows;
  for (int i = threadIdx.x; i < G * kGvRows; i += blockDim.x) {
    const int g = i / kGvRows, r = i % kGvRows, n = n0 + r;
    s_sm[i] = n < N ? scales[static_cast<size_t>(g) * N + n] : __float2half(0.f);
    z_sm[i] = n < N ? zeros[static_cast<size_t>(g) * N + n] : 0;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rb = warp * kGvRowsPerWarp;  // first of this warp's rows within the CTA
  const int W = K / 8;                   // words per row (a multiple of 32)
  const uint32_t* wrow[kGvRowsPerWarp];
#pragma unroll
  for (int r = 0; r < kGvRowsPerWarp; ++r)  // rows past N (N % 32 == 16) re-read row N - 1, never stored
    wrow[r] = wq + static_cast<size_t>(min(n0 + rb + r, N - 1)) * W;
  float acc[kGvRowsPerWarp][MP];
#pragma unroll
  for (int r = 0; r < kGvRowsPerWarp; ++r)
#pragma unroll
    for (int m = 0; m < MP; ++m) acc[r][m] = 0.f;

  // Lane l's words of block j are 128 j + 4 l .. +3 (the last block of a row may be
  // short: W is a multiple of 32).  The next block's words are loaded before this
  // block's arithmetic, so every lane keeps one block of loads in flight.
  uint4 nxt[kGvRowsPerWarp];
  if (4 * lane < W) {
#pragma unroll
    for (int r = 0; r < kGvRowsPerWarp; ++r) nxt[r] = ldg_stream16(wrow[r] + 4 * lane);
  }
  for (int wi = 4 * lane; wi < W; wi += 128) {
    uint4 wv[kGvRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kGvRowsPerWarp; ++r) wv[r] = nxt[r];
    if (wi + 128 < W) {
#pragma unroll
      for (int r = 0; r < kGvRowsPerWarp; ++r) nxt[r] = ldg_stream16(wrow[r] + wi + 128);
    }
    uint32_t xv[MP][16];  // x[m][8 wi .. 8 wi + 31] as fp16 pairs
#pragma unroll
    for (int m = 0; m < MP; ++m) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 t = make_uint4(0u, 0u, 0u, 0u);
        if (m < M) t = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(m) * K + 8 * wi) + q);
        xv[m][4 * q] = t.x;
        xv[m][4 * q + 1] = t.y;
        xv[m][4 * q + 2] = t.z;
        xv[m][4 * q + 3] = t.w;
      }
    }
    const int g = wi / 16;  // the 4 words share one group of 128
#pragma unroll
    for (int r = 0; r < kGvRowsPerWarp; ++r) {
      const __half s = s_sm[g * kGvRows + rb + r];
      const int z = z_sm[g * kGvRows + rb + r];
      const __half2 s2 = __halves2half2(s, s);
      const __half zb = __int2half_rn(1024 + z), zs = __int2half_rn(64 + z);
      const __half2 zb2 = __halves2half2(zb, zb), zs2 = __halves2half2(zs, zs);
      const uint32_t wd[4] = {wv[r].x, wv[r].y, wv[r].z, wv[r].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t src = i < 2 ? wd[e] : (wd[e] >> 8);
          const uint32_t t = (i & 1) ? ((src & 0x00F000F0u) | 0x54005400u) : ((src & 0x000F000Fu) | 0x64006400u);
          const __half2 d = __hsub2(*reinterpret_cast<const __half2*>(&t), (i & 1) ? zs2 : zb2);
          const __half2 wh = __hmul2(d, s2);
          const uint32_t w2 = *reinterpret_cast<const uint32_t*>(&wh);
#pragma unroll
          for (int m = 0; m < MP; ++m) acc[r][m] = fma2_f16_f32(w2, xv[m][4 * e + i], acc[r][m]);
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kGvRowsPerWarp; ++r) {
#pragma unroll
    for (int m = 0; m < MP; ++m) {
      float v = acc[r][m];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      acc[r][m] = v;
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int r = 0; r < kGvRowsPerWarp; ++r) {
      const int n = n0 + rb + r;
#pragma unroll
      for (int m = 0; m < MP; ++m)
        if (n < N && m < M) y[static_cast<size_t>(m) * N + n] = __float2half_rn(acc[r][m]);
    }
  }
}

template <int MP>
cudaError_t launch_gemv(const W4a16Args& a, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(a.K / 128) * kGvRows * 3;
  auto kern = w4a16_gemv_kernel<MP>;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)))) return e;
  const unsigned blocks = static_cast<unsigned>((a.N + kGvRows - 1) / kGvRows);
  kern<<<blocks, kGvWarps * 32, smem, stream>>>(static_cast<const __half*>(a.x), static_cast<const uint32_t*>(a.wq),
                                               static_cast<const __half*>(a.scales),
                                               static_cast<const uint8_t*>(a.zeros), static_cast<__half*>(a.y), a.M,
                                               a.N, a.K);
  return cudaGetLastError();
}

// Y = fp16(sum_s partials[s]), in split order (the same bits on every run).
__global__ void __launch_bounds__(256) w4a16_reduce_kernel(const float* __restrict__ partials,
                                                           __half* __restrict__ y, int nsplit, long long mn) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= mn) return;
  float acc = 0.f;
  for (int s = 0; s < nsplit; ++s) acc += partials[static_cast<size_t>(s) * mn + i];
  y[i] = __float2half_rn(acc);
}

template <int MP>
cudaError_t launch_mp(const W4a16Args& a, cudaStream_t stream) {
  using C = W4Cfg<MP>;
  cudaError_t e;
  CUtensorMap tw, tx, ts, tz;
  if ((e = make_tmap_2d(&tw, a.wq, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, a.K / 8, a.N, a.K / 8, kW4Kc / 8, kW4Rows,
                        true)))
    return e;
  if ((e = make_tmap_2d(&tx, a.x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.K, a.M, a.K, 64, MP, true))) return e;
  if ((e = make_tmap_2d(&ts, a.scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.N, a.K / 128, a.N, kW4Rows, 2, false)))
    return e;
  if ((e = make_tmap_2d(&tz, a.zeros, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.N, a.K / 128, a.N, kW4Rows, 2, false)))
    return e;
  auto kern = w4a16_kernel<MP>;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes))) return e;
  const int kchunks = a.K / kW4Kc;
  const int cps = w4a16_chunks_per_split(a.K, a.n_split);
  const int nsplit = (kchunks + cps - 1) / cps;  // no empty split
  const int nstrips = (a.N + kW4Rows - 1) / kW4Rows;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev))) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))) return e;
  const int units = nstrips * nsplit;
  kern<<<static_cast<unsigned>(units < sms ? units : sms), kW4Threads, C::kSmemBytes, stream>>>(
      tw, tx, ts, tz, static_cast<__half*>(a.y), a.partials, a.M, a.N, nstrips, nsplit, kchunks, cps, a.err_word,
      a.dbg.wait_limit_ns);
  if ((e = cudaGetLastError())) return e;
  if (nsplit > 1) {
    const long long mn = static_cast<long long>(a.M) * a.N;
    w4a16_reduce_kernel<<<static_cast<unsigned>((mn + 255) / 256), 256, 0, stream>>>(
        a.partials, static_cast<__half*>(a.y), nsplit, mn);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace

int w4a16_chunks_per_split(int K, int n_split) {
  const int kchunks = K / kW4Kc;
  return (kchunks + n_split - 1) / n_split;
}

bool w4a16_uses_gemv(int M, int K) { return M <= kGvMaxM && K <= 65536; }

cudaError_t launch_w4a16(const W4a16Args& a, cudaStream_t stream) {
  if (w4a16_uses_gemv(a.M, a.K)) return launch_gemv<1>(a, stream);
  if (a.M <= 16) return launch_mp<16>(a, stream);
  if (a.M <= 32) return launch_mp<32>(a, stream);
  if (a.M <= 64) return launch_mp<64>(a, stream);
  if (a.M <= 96) return launch_mp<96>(a, stream);
  return launch_mp<128>(a, stream);
}

}  // namespace fa
