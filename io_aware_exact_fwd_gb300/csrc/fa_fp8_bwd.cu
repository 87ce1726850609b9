// Backward pass of the FP8 attention, for sm_103a.
//
// The FP8 forward ("FlashAttention-Skalierung, Multi-GPU-Training und
// Gewichtsquantisierung", section 1, bullet "Unterstützung geringer
// FP8-Präzision") computes attention on block-quantised e4m3 operands, Q and K
// first rotated by M = diag(s) H_d (unnormalised; the scores carry 1/d).  Its
// backward is taken straight through the quantisation: the textbook gradient on
// the dequantised operands Q', K', V', carried back through the rotation,
//
//   dQ = dQ' M^T = (dQ' H_d) * s,   dK = (dK' H_d) * s,   dV = dV'.
//
// Three stages on one stream:
//   1. fp8_dequant_kernel: e4m3 codes times the tile scale (one fp32 product),
//      rounded to bf16, into dense [BH, N, d] operands; V's codes are stored
//      transposed ([BH, d, Npad]) and are transposed back through shared memory.
//   2. the bf16 backward (fa_bwd.cu) on those operands with softmax scale scale/d,
//      writing dQ', dK', dV into the caller's buffers;
//   3. unrotate_kernel: dQ' and dK' rows through the fast Walsh-Hadamard
//      transform in fp32 (butterfly spans 1..d/2), times the signs, back to bf16
//      in place.
//
// Stages 1 and 3 are bound by HBM (stage 1 reads 3 N d bytes of codes and writes
// 6 N d bytes of operands per head; stage 3 reads and writes 4 N d bytes); the
// backward's tensor-core work is O(N^2 d) and dominates from a few hundred rows.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kTile = 64;            // rows per quantisation tile (the FP8 prepare's)
constexpr int kDeqThreads = 256;
constexpr int kRotThreads = 256;     // 8 rows per block, one warp per row

// Two e4m3 codes (low byte -> low half) to two fp16 values: exact, every e4m3
// value (subnormals included) is an fp16 value.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t pair16) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(pair16)));
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

// 16 codes -> 16 bf16 values bf16_rn(decode * sigma), written as two 16-byte stores.
__device__ __forceinline__ void dequant16(const uint4 c, float sigma, __nv_bfloat16* dst) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  uint32_t out[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float2 f = e4m3x2_to_float2(w[i] >> (16 * h));
      const __nv_bfloat162 b = __floats2bfloat162_rn(__fmul_rn(f.x, sigma), __fmul_rn(f.y, sigma));
      out[2 * i + h] = *reinterpret_cast<const uint32_t*>(&b);
    }
  }
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  d4[0] = make_uint4(out[0], out[1], out[2], out[3]);
  d4[1] = make_uint4(out[4], out[5], out[6], out[7]);
}

// One block per (64-row tile, head): block x = head * ntiles + tile.
template <int D>
__global__ void __launch_bounds__(kDeqThreads) fp8_dequant_kernel(const uint8_t* __restrict__ ws, Fp8Layout lay,
                                                                  __nv_bfloat16* __restrict__ qr,
                                                                  __nv_bfloat16* __restrict__ kr,
                                                                  __nv_bfloat16* __restrict__ vr, int N) {
  __shared__ __align__(16) uint8_t vt[D][kTile + 16];  // V codes of the tile, [column][row]
  const int t = static_cast<int>(blockIdx.x % lay.ntiles);
  const int bh = static_cast<int>(blockIdx.x / lay.ntiles);
  const int r0 = t * kTile;
  const int rows = min(kTile, N - r0);
  const size_t sidx = static_cast<size_t>(bh) * lay.ntiles + t;
  const float sq = reinterpret_cast<const float*>(ws + lay.off_sq)[sidx];
  const float sk = reinterpret_cast<const float*>(ws + lay.off_sk)[sidx];
  const float sv = reinterpret_cast<const float*>(ws + lay.off_sv)[sidx];

  // Q and K: the tile's rows are contiguous, rows * D bytes (a multiple of 16).
  const size_t base = (static_cast<size_t>(bh) * N + r0) * D;
  for (int i = threadIdx.x * 16; i < rows * D; i += kDeqThreads * 16) {
    dequant16(*reinterpret_cast<const uint4*>(ws + lay.off_q8 + base + i), sq, qr + base + i);
    dequant16(*reinterpret_cast<const uint4*>(ws + lay.off_k8 + base + i), sk, kr + base + i);
  }

  // V: codes of columns c, rows r0 .. r0+63 sit at v8t[bh][c][r0 ..] (Npad >= r0 + 64,
  // zero past N).  Stage [D][64] in shared memory, then read it back by rows.
  const uint8_t* v8t = ws + lay.off_v8t + static_cast<size_t>(bh) * D * lay.npad + r0;
  for (int i = threadIdx.x; i < D * (kTile / 16); i += kDeqThreads) {
    const int c = i / (kTile / 16), j = (i % (kTile / 16)) * 16;
    const uint4 v = *reinterpret_cast<const uint4*>(v8t + static_cast<size_t>(c) * lay.npad + j);
    *reinterpret_cast<uint4*>(&vt[c][j]) = v;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kTile * (D / 16); i += kDeqThreads) {
    const int r = i / (D / 16), c0 = (i % (D / 16)) * 16;
    if (r >= rows) continue;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      w[q] = static_cast<uint32_t>(vt[c0 + 4 * q][r]) | (static_cast<uint32_t>(vt[c0 + 4 * q + 1][r]) << 8) |
             (static_cast<uint32_t>(vt[c0 + 4 * q + 2][r]) << 16) | (static_cast<uint32_t>(vt[c0 + 4 * q + 3][r]) << 24);
    dequant16(make_uint4(w[0], w[1], w[2], w[3]), sv, vr + (static_cast<size_t>(bh) * N + r0 + r) * D + c0);
  }
}

// x <- bf16((x H_128) * s) per row of 128, for two tensors (blockIdx.y selects).
// Lane l holds columns 4l .. 4l+3: butterfly spans 1 and 2 stay in the lane,
// spans 4 .. 64 pair lane l with lane l ^ (span / 4).
__global__ void __launch_bounds__(kRotThreads) unrotate_kernel(__nv_bfloat16* __restrict__ x0,
                                                               __nv_bfloat16* __restrict__ x1,
                                                               const int8_t* __restrict__ signs, long long rows) {
  const long long r = static_cast<long long>(blockIdx.x) * (kRotThreads / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  __nv_bfloat16* row = (blockIdx.y == 0 ? x0 : x1) + r * 128 + 4 * lane;
  const uint2 raw = *reinterpret_cast<const uint2*>(row);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
  float v[4] = {a.x, a.y, b.x, b.y};
  // span 1
  float t0 = v[0] + v[1], t1 = v[0] - v[1], t2 = v[2] + v[3], t3 = v[2] - v[3];
  // span 2
  v[0] = t0 + t2;
  v[2] = t0 - t2;
  v[1] = t1 + t3;
  v[3] = t1 - t3;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float p = __shfl_xor_sync(0xffffffffu, v[e], m);
      v[e] = upper ? p - v[e] : v[e] + p;  // (a, b) -> (a + b, a - b), a the lower index
    }
  }
  float s[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) s[e] = signs[4 * lane + e] < 0 ? -1.f : 1.f;
  uint2 out;
  out.x = pack_bf16x2(v[0] * s[0], v[1] * s[1]);
  out.y = pack_bf16x2(v[2] * s[2], v[3] * s[3]);
  *reinterpret_cast<uint2*>(row) = out;
}

}  // namespace

cudaError_t launch_fp8_dequant(const void* fp8_ws, void* qr, void* kr, void* vr, int B, int H, int N, int d,
                               cudaStream_t stream) {
  const Fp8Layout lay = fp8_layout(B, H, N, d);
  const unsigned grid = static_cast<unsigned>(lay.ntiles) * static_cast<unsigned>(B * H);
  const auto* ws = static_cast<const uint8_t*>(fp8_ws);
  auto* q = static_cast<__nv_bfloat16*>(qr);
  auto* k = static_cast<__nv_bfloat16*>(kr);
  auto* v = static_cast<__nv_bfloat16*>(vr);
  if (d == 64)
    fp8_dequant_kernel<64><<<grid, kDeqThreads, 0, stream>>>(ws, lay, q, k, v, N);
  else
    fp8_dequant_kernel<128><<<grid, kDeqThreads, 0, stream>>>(ws, lay, q, k, v, N);
  return cudaGetLastError();
}

cudaError_t launch_fp8_unrotate(void* dq, void* dk, const int8_t* signs, long long rows, cudaStream_t stream) {
  const int per_block = kRotThreads / 32;
  const dim3 grid(static_cast<unsigned>((rows + per_block - 1) / per_block), 2);
  unrotate_kernel<<<grid, kRotThreads, 0, stream>>>(static_cast<__nv_bfloat16*>(dq), static_cast<__nv_bfloat16*>(dk),
                                                    signs, rows);
  return cudaGetLastError();
}

}  // namespace fa
