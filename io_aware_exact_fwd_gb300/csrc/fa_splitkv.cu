// Exact merge of split-KV attention partials, for sm_103a.
//
// Each split s of the keys leaves, per query row, a normalised partial output
// O_s and its logsumexp LSE_s (natural log; -inf when the row saw no key of the
// split).  Because exp(LSE_s) is the row's partial softmax denominator over that
// split, the full result is
//
//   LSE = ln sum_s exp(LSE_s)          O = sum_s exp(LSE_s - LSE) O_s
//
// (the softmax definition of "FlashAttention-2 (DE)", section "Hintergrund",
// summed over key ranges; the setting is the bandwidth-bound token-by-token
// inference of "FlashAttention-Skalierung, Multi-GPU-Training und
// Gewichtsquantisierung", section 3).  Splits with LSE = -inf carry no weight and
// their O is never read.
//
// Bound: HBM.  One warp per query row: the lanes first reduce the row's LSE_s
// (max, then the sum of exp(LSE_s - max)), then walk the splits once, each lane
// accumulating d/32 consecutive elements of O (coalesced 128- or 256-byte rows).
// O may be strided (element (b, h, i, c) at b so[2] + h so[1] + i so[0] + c).
#include <cuda_bf16.h>
#include <math.h>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kMergeThreads = 256;  // 8 rows per block

template <int D>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const float* __restrict__ o_part,
                                                              const float* __restrict__ lse_part,
                                                              __nv_bfloat16* __restrict__ o, Strides so,
                                                              float* __restrict__ lse, int n_split, long long rows,
                                                              int H, int Nq) {
  constexpr int kPer = D / 32;  // elements of O per lane
  const long long r = static_cast<long long>(blockIdx.x) * (kMergeThreads / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  // Row maximum and denominator of the split LSEs (natural log units).
  float m = -INFINITY;
  for (int s = lane; s < n_split; s += 32) m = fmaxf(m, lse_part[static_cast<size_t>(s) * rows + r]);
#pragma unroll
  for (int k = 16; k >= 1; k >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, k));
  float acc[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
  if (m == -INFINITY) {  // the row saw no key at all
    if (lane == 0) lse[r] = -INFINITY;
  } else {
    float tot = 0.f;
    for (int s = 0; s < n_split; ++s) {
      const float ls = lse_part[static_cast<size_t>(s) * rows + r];  // same address in every lane: one broadcast
      if (ls == -INFINITY) continue;
      const float w = expf(ls - m);
      tot += w;
      const float* src = o_part + (static_cast<size_t>(s) * rows + r) * D + lane * kPer;
      if constexpr (kPer == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        acc[0] = fmaf(w, v.x, acc[0]);
        acc[1] = fmaf(w, v.y, acc[1]);
        acc[2] = fmaf(w, v.z, acc[2]);
        acc[3] = fmaf(w, v.w, acc[3]);
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        acc[0] = fmaf(w, v.x, acc[0]);
        acc[1] = fmaf(w, v.y, acc[1]);
      }
    }
    const float inv = 1.f / tot;
#pragma unroll
    for (int i = 0; i < kPer; ++i) acc[i] *= inv;
    if (lane == 0) lse[r] = m + logf(tot);
  }
  // Row r = (b H + h) Nq + i of the partials; O element (b, h, i, c) at the strides.
  const long long bh = r / Nq, i = r % Nq;
  __nv_bfloat16* dst = o + (bh / H) * so.s[2] + (bh % H) * so.s[1] + i * so.s[0] + lane * kPer;
  if constexpr (kPer == 4) {
    uint2 pk;
    pk.x = pack_bf16x2(acc[0], acc[1]);
    pk.y = pack_bf16x2(acc[2], acc[3]);
    *reinterpret_cast<uint2*>(dst) = pk;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0], acc[1]);
  }
}

}  // namespace

cudaError_t launch_merge_partials(const MergeArgs& a, cudaStream_t stream) {
  const long long rows = static_cast<long long>(a.BH) * a.Nq;
  const int per_block = kMergeThreads / 32;
  const unsigned blocks = static_cast<unsigned>((rows + per_block - 1) / per_block);
  auto* o = static_cast<__nv_bfloat16*>(a.o);
  if (a.d == 64)
    merge_kernel<64><<<blocks, kMergeThreads, 0, stream>>>(a.o_part, a.lse_part, o, a.so, a.lse, a.n_split, rows,
                                                          a.H, a.Nq);
  else
    merge_kernel<128><<<blocks, kMergeThreads, 0, stream>>>(a.o_part, a.lse_part, o, a.so, a.lse, a.n_split, rows,
                                                           a.H, a.Nq);
  return cudaGetLastError();
}

}  // namespace fa
