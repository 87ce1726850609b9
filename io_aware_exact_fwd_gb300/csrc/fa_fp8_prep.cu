// FP8 input preparation for sm_103a: incoherent processing and block quantisation.
//
// "FlashAttention-Skalierung, Multi-GPU-Training und Gewichtsquantisierung",
// section 1, bullet "Unterstützung geringer FP8-Präzision": FP8 tensor cores
// double raw throughput; to keep outliers from destroying precision, small tiles
// are scaled independently (block quantisation) and Q and K are multiplied by a
// random orthogonal matrix before quantising (incoherent processing).
//
// Here (one CTA per 64-row tile of one head of Q, K or V):
//  * Q and K rows are rotated by x -> (x * s) H_d, s the caller's +-1 signs (or,
//    given a 64-bit seed instead, signs from the SplitMix64 outputs, see
//    seeded_sign in fa_internal.h) and
//    H_d the Sylvester Walsh-Hadamard matrix, as a radix-2 transform with
//    butterfly spans 1, 2, ..., d/2 (each butterfly one fp32 add and one fp32
//    subtract; spans below the per-thread width in registers, the rest across
//    lanes with shuffles).  The 1/sqrt(d) normalisation of the orthogonal
//    matrix is left to the attention kernel's score scale.  V is not rotated.
//  * amax = max |x| over the tile (exact); sigma = 2^e, the smallest power of
//    two with amax <= 448 sigma (1 for an all-zero tile), inv = 2^-e; codes =
//    e4m3_rn_satfinite(x * inv), an exact scaling.  e4m3 being floating point, a
//    power-of-two scale loses no relative precision, and decode(code) * sigma is
//    exact in fp32 and bf16 (the FP8 backward's operands).
//  * Inputs may be strided (element (b, h, n, c) at b s[2] + h s[1] + n s[0] + c,
//    c contiguous); the workspace is always dense.
//  * Q and K codes are written row-major [BH, N, d]; V codes transposed,
//    [BH, d, npad] with keys contiguous (npad = N rounded up to 128, a whole
//    attention key block), so that V is a K-major operand of the P V MMA.
//    Keys >= N are zeros (a V-only block past the last tile writes zeros).
#include <cuda_bf16.h>
#include <stdint.h>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kTileRows = 64;
constexpr int kPrepThreads = 256;  // 8 warps x 8 rows each

__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %2, %1;\n\tmov.b16 %0, t;\n\t}" : "=h"(r) : "f"(lo), "f"(hi));
  return r;
}

// Load 16 consecutive elements of one row as fp32 (bf16: two 16-byte loads; fp32: four).
__device__ __forceinline__ void load16(const void* base, size_t elem0, int in_bf16, float (&x)[16]) {
  if (in_bf16) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + elem0);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 u = p[h];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[j]));
        x[8 * h + 2 * j] = f.x;
        x[8 * h + 2 * j + 1] = f.y;
      }
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem0);
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float4 f = p[h];
      x[4 * h] = f.x;
      x[4 * h + 1] = f.y;
      x[4 * h + 2] = f.z;
      x[4 * h + 3] = f.w;
    }
  }
}

// In-place unnormalised Walsh-Hadamard transform of one row spread over D/16 lanes
// of 16 consecutive elements (sl = the lane's index within its row): spans 1..8 in
// the lane, then spans 16..D/2 with the partner lane sl ^ (span / 16).
template <int D>
__device__ __forceinline__ void fwht16(float (&x)[16], int sl) {
#pragma unroll
  for (int span = 1; span < 16; span <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if ((i & span) == 0) {
        const float a = x[i], b = x[i + span];
        x[i] = a + b;
        x[i + span] = a - b;
      }
    }
  }
#pragma unroll
  for (int span = 16; span < D; span <<= 1) {
    const int m = span / 16;
    const bool upper = (sl & m) != 0;  // this lane holds the "b" half
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float other = __shfl_xor_sync(0xffffffffu, x[i], m);
      x[i] = upper ? (other - x[i]) : (x[i] + other);
    }
  }
}

// Block-wide max of a per-thread value (8 warps).
__device__ __forceinline__ float block_amax(float amax, float* s_amax, int warp, int lane) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
  if (lane == 0) s_amax[warp] = amax;
  __syncthreads();
  amax = s_amax[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) amax = fmaxf(amax, s_amax[w]);
  return amax;
}

// Power-of-two tile scale: e = the smallest integer with amax <= 448 * 2^e, read
// from amax's fp32 bits (amax = m 2^e0, m in [1, 2): e = e0 - 8, plus 1 when
// m > 1.75), clamped to [-126, 126]; e = 0 for amax = 0.  sigma = 2^e and
// inv = 2^-e are exact normal fp32 numbers.
__device__ __forceinline__ void pow2_scale(float amax, float& sigma, float& inv) {
  const uint32_t b = __float_as_uint(amax);
  const int field = static_cast<int>((b >> 23) & 0xFFu);
  int e = field == 0 ? -126 : field - 135 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  if (amax == 0.f) e = 0;
  e = max(-126, min(126, e));
  sigma = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
  inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
}

// STRIDED: inputs at the caller's strides; otherwise dense [B, H, N, d] (the
// index arithmetic of the dense build is cheaper, and this kernel is partly
// issue-bound).
template <int D, bool STRIDED>
__global__ void __launch_bounds__(kPrepThreads) fp8_prepare_kernel(const void* __restrict__ q,
                                                                   const void* __restrict__ k,
                                                                   const void* __restrict__ v, int in_bf16,
                                                                   const int8_t* __restrict__ signs, uint64_t seed,
                                                                   Fp8Layout lay, uint8_t* __restrict__ ws, int N,
                                                                   int H, Strides sq, Strides sk, Strides sv) {
  constexpr int E = D / 32;
  constexpr int kRowsPerWarp = kTileRows / 8;
  constexpr int kVtPitch = kTileRows + 4;  // 17 words per d-row: byte stores of 32 lanes hit 32 banks
  const int tile = blockIdx.x;
  const int bh = blockIdx.y;
  const int which = blockIdx.z;  // 0 = Q, 1 = K, 2 = V
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ntiles = lay.ntiles;
  __shared__ float s_amax[8];
  __shared__ __align__(16) uint8_t s_vt[D * kVtPitch];  // V codes of this tile, transposed [d][64 (+4)]

  // Element (b, h, row, c) of an input at b s[2] + h s[1] + row s[0] + c (dense:
  // (bh N + row) d + c).
  size_t head_off = static_cast<size_t>(bh) * N * D;
  int64_t row_stride = D;
  if constexpr (STRIDED) {
    const Strides& sin = which == 0 ? sq : (which == 1 ? sk : sv);
    head_off = static_cast<size_t>(bh / H) * sin.s[2] + static_cast<size_t>(bh % H) * sin.s[1];
    row_stride = sin.s[0];
  }
  float x[kRowsPerWarp][E];
  if (which == 2) {
    // ------------------------------------------------ V: no rotation, transposed out
    // Lane l holds columns l, l + 32, ... of each row (coalesced loads).
    float amax = 0.f;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int row = tile * kTileRows + warp * kRowsPerWarp + r;
#pragma unroll
      for (int m = 0; m < E; ++m) {
        float val = 0.f;
        if (row < N) {
          const size_t e = head_off + static_cast<size_t>(row) * row_stride + lane + 32 * m;
          val = in_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(v)[e]) : static_cast<const float*>(v)[e];
        }
        x[r][m] = val;
        amax = fmaxf(amax, fabsf(val));
      }
    }
    amax = block_amax(amax, s_amax, warp, lane);
    float sigma, inv;
    pow2_scale(amax, sigma, inv);
    if (threadIdx.x == 0 && tile < ntiles)
      reinterpret_cast<float*>(ws + lay.off_sv)[static_cast<size_t>(bh) * ntiles + tile] = sigma;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int lrow = warp * kRowsPerWarp + r;
#pragma unroll
      for (int m = 0; m < E; m += 2) {
        const uint16_t two = e4m3x2(__fmul_rn(x[r][m], inv), __fmul_rn(x[r][m + 1], inv));
        s_vt[(lane + 32 * m) * kVtPitch + lrow] = static_cast<uint8_t>(two & 0xff);
        s_vt[(lane + 32 * (m + 1)) * kVtPitch + lrow] = static_cast<uint8_t>(two >> 8);
      }
    }
    __syncthreads();
    // [d][64] tile -> V^T rows of 64 contiguous key bytes, 4 bytes per store.
    uint8_t* vt = ws + lay.off_v8t + static_cast<size_t>(bh) * D * lay.npad + static_cast<size_t>(tile) * kTileRows;
    for (int idx = threadIdx.x; idx < D * (kTileRows / 4); idx += kPrepThreads) {
      const int drow = idx / (kTileRows / 4);
      const int word = idx % (kTileRows / 4);
      *reinterpret_cast<uint32_t*>(vt + static_cast<size_t>(drow) * lay.npad + word * 4) =
          *reinterpret_cast<const uint32_t*>(s_vt + drow * kVtPitch + word * 4);
    }
    return;
  }

  // ------------------------------------------------------ Q, K: rotate, then quantise
  // A row is held by kL = d/16 lanes, 16 consecutive elements each (32-byte bf16 or
  // 64-byte fp32 loads, one 16-byte store of codes): butterfly spans 1..8 stay in
  // the lane, spans 16..d/2 pair lane l with lane l ^ (span / 16) of the same row.
  if (tile >= ntiles) return;  // blocks past the last tile exist only to pad V^T
  constexpr int kE = 16;
  constexpr int kL = D / kE;                            // lanes per row: 8 (d=128), 4 (d=64)
  constexpr int kRowsPerPass = 32 / kL;                 // rows a warp holds at once
  constexpr int kPasses = kRowsPerWarp / kRowsPerPass;  // 2 (d=128), 1 (d=64)
  const int sl = lane % kL, rg = lane / kL;
  float sg[kE];
#pragma unroll
  for (int i = 0; i < kE; ++i)
    sg[i] = signs ? (signs[kE * sl + i] < 0 ? -1.f : 1.f) : static_cast<float>(seeded_sign(seed, kE * sl + i));
  const void* src = which == 0 ? q : k;
  float xr[kPasses][kE];
  float amax = 0.f;
#pragma unroll
  for (int p = 0; p < kPasses; ++p) {
    const int row = tile * kTileRows + warp * kRowsPerWarp + p * kRowsPerPass + rg;
    if (row < N) {
      load16(src, head_off + static_cast<size_t>(row) * row_stride + kE * sl, in_bf16, xr[p]);
    } else {
#pragma unroll
      for (int i = 0; i < kE; ++i) xr[p][i] = 0.f;
    }
  }
#pragma unroll
  for (int p = 0; p < kPasses; ++p) {
#pragma unroll
    for (int i = 0; i < kE; ++i) xr[p][i] *= sg[i];
    fwht16<D>(xr[p], sl);
#pragma unroll
    for (int i = 0; i < kE; ++i) amax = fmaxf(amax, fabsf(xr[p][i]));
  }
  amax = block_amax(amax, s_amax, warp, lane);
  float sigma, inv;
  pow2_scale(amax, sigma, inv);
  if (threadIdx.x == 0)
    reinterpret_cast<float*>(ws + (which == 0 ? lay.off_sq : lay.off_sk))[static_cast<size_t>(bh) * ntiles + tile] =
        sigma;
#pragma unroll
  for (int p = 0; p < kPasses; ++p) {
    const int row = tile * kTileRows + warp * kRowsPerWarp + p * kRowsPerPass + rg;
    if (row >= N) continue;
    uint32_t wds[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t lo = e4m3x2(__fmul_rn(xr[p][4 * j], inv), __fmul_rn(xr[p][4 * j + 1], inv));
      const uint32_t hi = e4m3x2(__fmul_rn(xr[p][4 * j + 2], inv), __fmul_rn(xr[p][4 * j + 3], inv));
      wds[j] = lo | (hi << 16);
    }
    uint8_t* dst = ws + (which == 0 ? lay.off_q8 : lay.off_k8) + (static_cast<size_t>(bh) * N + row) * D + kE * sl;
    *reinterpret_cast<uint4*>(dst) = make_uint4(wds[0], wds[1], wds[2], wds[3]);
  }
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

Fp8Layout fp8_layout(int B, int H, int N, int d) {
  Fp8Layout l{};
  const size_t bh = static_cast<size_t>(B) * H;
  l.ntiles = (N + kTileRows - 1) / kTileRows;
  l.npad = (N + 127) / 128 * 128;
  l.off_q8 = 0;
  l.off_k8 = align256(bh * N * d);
  l.off_v8t = l.off_k8 + align256(bh * N * d);
  l.off_sq = l.off_v8t + align256(bh * d * l.npad);
  l.off_sk = l.off_sq + align256(bh * l.ntiles * 4);
  l.off_sv = l.off_sk + align256(bh * l.ntiles * 4);
  l.total = l.off_sv + align256(bh * l.ntiles * 4);
  return l;
}

cudaError_t launch_fp8_prepare(const Fp8PrepArgs& a, cudaStream_t stream) {
  const Fp8Layout lay = fp8_layout(a.B, a.H, a.N, a.d);
  dim3 grid(static_cast<unsigned>(lay.npad / kTileRows), static_cast<unsigned>(a.B * a.H), 3);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  const Strides dense = dense_strides(a.H, a.N, a.d);
  auto same = [&](const Strides& x) { return x.s[0] == dense.s[0] && x.s[1] == dense.s[1] && x.s[2] == dense.s[2]; };
  const bool strided = !(same(a.sq) && same(a.sk) && same(a.sv));
  auto go = [&](auto kern) {
    kern<<<grid, kPrepThreads, 0, stream>>>(a.q, a.k, a.v, a.in_bf16, a.signs, a.seed, lay, ws, a.N, a.H, a.sq, a.sk,
                                            a.sv);
  };
  if (a.d == 64)
    strided ? go(fp8_prepare_kernel<64, true>) : go(fp8_prepare_kernel<64, false>);
  else
    strided ? go(fp8_prepare_kernel<128, true>) : go(fp8_prepare_kernel<128, false>);
  return cudaGetLastError();
}

}  // namespace fa
