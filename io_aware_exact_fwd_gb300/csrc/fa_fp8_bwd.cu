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
//      writing dQ', dK', dV into the caller's buffers (on request the bf16 forward
//      first recomputes O and LSE from the same operands, so that the backward's
//      D = rowsum(dO * O) uses the unrounded probabilities);
//   3. unrotate_kernel: dQ' and dK' rows through the fast Walsh-Hadamard
//      transform in fp32 (butterfly spans 1..d/2), times the signs, back to bf16
//      in place (two rows per warp per pass, 16-byte accesses).
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
constexpr int kRotThreads = 256;

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

  // All of this thread's loads first (Q and K: the tile's rows are contiguous,
  // rows * D bytes, a multiple of 16; V: 16-byte pieces of the tile's d rows of
  // codes at v8t[bh][c][r0 ..], Npad >= r0 + 64, zero past N), then the arithmetic.
  constexpr int kQK = kTile * D / 16 / kDeqThreads;  // 16-byte pieces per thread: 2 (d=128), 1 (d=64)
  constexpr int kV = D * (kTile / 16) / kDeqThreads;
  const size_t base = (static_cast<size_t>(bh) * N + r0) * D;
  const uint8_t* v8t = ws + lay.off_v8t + static_cast<size_t>(bh) * D * lay.npad + r0;
  uint4 cq[kQK], ck[kQK], cv[kV];
#pragma unroll
  for (int j = 0; j < kQK; ++j) {
    const int i = (threadIdx.x + j * kDeqThreads) * 16;
    if (i < rows * D) {
      cq[j] = *reinterpret_cast<const uint4*>(ws + lay.off_q8 + base + i);
      ck[j] = *reinterpret_cast<const uint4*>(ws + lay.off_k8 + base + i);
    }
  }
#pragma unroll
  for (int j = 0; j < kV; ++j) {
    const int idx = threadIdx.x + j * kDeqThreads;
    const int c = idx / (kTile / 16), jj = (idx % (kTile / 16)) * 16;
    cv[j] = *reinterpret_cast<const uint4*>(v8t + static_cast<size_t>(c) * lay.npad + jj);
  }
#pragma unroll
  for (int j = 0; j < kV; ++j) {
    const int idx = threadIdx.x + j * kDeqThreads;
    *reinterpret_cast<uint4*>(&vt[idx / (kTile / 16)][(idx % (kTile / 16)) * 16]) = cv[j];
  }
#pragma unroll
  for (int j = 0; j < kQK; ++j) {
    const int i = (threadIdx.x + j * kDeqThreads) * 16;
    if (i < rows * D) {
      dequant16(cq[j], sq, qr + base + i);
      dequant16(ck[j], sk, kr + base + i);
    }
  }
  __syncthreads();
  // Consecutive lanes take consecutive rows of the same 16 columns, so each byte
  // load of the warp touches 8 consecutive words of one column (no bank conflict).
  for (int i = threadIdx.x; i < kTile * (D / 16); i += kDeqThreads) {
    const int r = i % kTile, c0 = (i / kTile) * 16;
    if (r >= rows) continue;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      w[q] = static_cast<uint32_t>(vt[c0 + 4 * q][r]) | (static_cast<uint32_t>(vt[c0 + 4 * q + 1][r]) << 8) |
             (static_cast<uint32_t>(vt[c0 + 4 * q + 2][r]) << 16) | (static_cast<uint32_t>(vt[c0 + 4 * q + 3][r]) << 24);
    dequant16(make_uint4(w[0], w[1], w[2], w[3]), sv, vr + (static_cast<size_t>(bh) * N + r0 + r) * D + c0);
  }
}

// x <- bf16((x H_d) * s) per row of d (64 or 128), for two tensors (blockIdx.y
// selects).  Lane l holds 8 consecutive columns of a row (one 16-byte load): a row
// spans d / 8 lanes, so a warp holds 32 / (d / 8) rows per pass; butterfly spans
// 1, 2, 4 stay in the lane and spans 8 .. d / 2 pair lane l with lane l ^ (span / 8)
// of the same row.  Each warp takes kRotPasses passes and issues all their loads
// before any arithmetic, to keep enough bytes in flight.
constexpr int kRotPasses = 4;

template <int D>
__global__ void __launch_bounds__(kRotThreads) unrotate_kernel(__nv_bfloat16* __restrict__ x0,
                                                               __nv_bfloat16* __restrict__ x1,
                                                               const int8_t* __restrict__ signs, long long rows) {
  constexpr int kLanesPerRow = D / 8;
  constexpr int kRowsPerPass = 32 / kLanesPerRow;
  const int lane = threadIdx.x & 31;
  const int sl = lane & (kLanesPerRow - 1);  // the lane's index within its row
  const long long r0 = (static_cast<long long>(blockIdx.x) * (kRotThreads / 32) + (threadIdx.x >> 5)) *
                           (kRowsPerPass * kRotPasses) + lane / kLanesPerRow;
  __nv_bfloat16* base = (blockIdx.y == 0 ? x0 : x1) + 8 * sl;
  uint4 raw[kRotPasses];
#pragma unroll
  for (int p = 0; p < kRotPasses; ++p) {
    const long long r = r0 + kRowsPerPass * p;
    raw[p] = r < rows ? *reinterpret_cast<const uint4*>(base + r * D) : make_uint4(0u, 0u, 0u, 0u);
  }
  float s[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) s[e] = signs[8 * sl + e] < 0 ? -1.f : 1.f;
#pragma unroll
  for (int p = 0; p < kRotPasses; ++p) {
    const uint32_t w[4] = {raw[p].x, raw[p].y, raw[p].z, raw[p].w};
    float v[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[j]));
      v[2 * j] = f.x;
      v[2 * j + 1] = f.y;
    }
#pragma unroll
    for (int span = 1; span < 8; span <<= 1) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if ((e & span) == 0) {
          const float a = v[e], b = v[e + span];
          v[e] = a + b;
          v[e + span] = a - b;
        }
      }
    }
#pragma unroll
    for (int m = 1; m < kLanesPerRow; m <<= 1) {
      const bool upper = (sl & m) != 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float o = __shfl_xor_sync(0xffffffffu, v[e], m);
        v[e] = upper ? o - v[e] : v[e] + o;  // (a, b) -> (a + b, a - b), a the lower index
      }
    }
    const long long r = r0 + kRowsPerPass * p;
    if (r < rows) {
      uint4 out;
      out.x = pack_bf16x2(v[0] * s[0], v[1] * s[1]);
      out.y = pack_bf16x2(v[2] * s[2], v[3] * s[3]);
      out.z = pack_bf16x2(v[4] * s[4], v[5] * s[5]);
      out.w = pack_bf16x2(v[6] * s[6], v[7] * s[7]);
      *reinterpret_cast<uint4*>(base + r * D) = out;
    }
  }
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

cudaError_t launch_fp8_unrotate(void* dq, void* dk, const int8_t* signs, long long rows, int d,
                                cudaStream_t stream) {
  auto* x0 = static_cast<__nv_bfloat16*>(dq);
  auto* x1 = static_cast<__nv_bfloat16*>(dk);
  const int per_block = (kRotThreads / 32) * (256 / d) * kRotPasses;  // rows per pass of a warp: 32 / (d / 8)
  const dim3 grid(static_cast<unsigned>((rows + per_block - 1) / per_block), 2);
  if (d == 64)
    unrotate_kernel<64><<<grid, kRotThreads, 0, stream>>>(x0, x1, signs, rows);
  else
    unrotate_kernel<128><<<grid, kRotThreads, 0, stream>>>(x0, x1, signs, rows);
  return cudaGetLastError();
}

}  // namespace fa
