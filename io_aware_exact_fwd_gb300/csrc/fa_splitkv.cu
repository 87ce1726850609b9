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

// ------------------------------------------------------------------------------
// Split-KV partials for one query row (Nq = 1, the token-by-token decode step) on
// the CUDA cores.  With a single query the tcgen05 forward would spend a 128-row
// tile of MMAs and exponentials per key block on one useful row; here the work is
// the K/V stream itself: 2d fp32 FMAs per key against 4d bytes read.
//
// One CTA of 4 warps per (head, split); warp w takes the split's chunks of KC keys
// (32 at d = 64, 16 at d = 128, so that a chunk's rows fit in registers) w, w + 4,
// ...  Lane l holds the d/32 consecutive columns c = l d/32 .. of every row, so
// each row of K or V is one coalesced warp load; all of a chunk's loads are issued
// before its arithmetic.  Per chunk:
//  * partial dots: lane l forms q[c] k_j[c] summed over its columns for every key j;
//  * a butterfly of shuffles (widths KC/2, ..., 2, 1; at each step a lane keeps the
//    half of its values whose key index has its bit of the width and adds the
//    partner's copy of that half; for KC = 16 one more exchange adds the two
//    half-warps) leaves the full q . k_j in lane j (and j + 16);
//  * online softmax in base 2 (the scale and log2 e are folded into q): chunk
//    maximum, the running reference, p_j = 2^(s_j - m), O and the lane's row sum
//    rescaled by 2^(m_old - m);
//  * O[c] += p_j v_j[c] for the 32 keys, p_j broadcast from lane j.
// The four warps' (m, l, O) are merged through shared memory exactly as the split
// merge does; the partial is O / l in fp32 and LSE = ln 2 (m + log2 l), -inf for an
// empty split.  All arithmetic is fp32 (the inputs bf16).  Only d = 64 is built:
// at d = 128 this kernel streamed 0.90 of HBM bandwidth against the tensor-core
// kernel's 0.92, which therefore keeps that case.
template <int D, int KC>  // KC keys per chunk: 32 at d = 64, 16 at d = 128 (registers for the chunk's rows)
__global__ void __launch_bounds__(128) decode_partial_kernel(const __nv_bfloat16* __restrict__ q,
                                                             const __nv_bfloat16* __restrict__ k,
                                                             const __nv_bfloat16* __restrict__ v, Strides sq,
                                                             Strides sk, Strides sv, float* __restrict__ o_part,
                                                             float* __restrict__ lse_part, int H, int BH, int Nk,
                                                             int n_split, int kbps, float scale_log2) {
  constexpr int E = D / 32;  // columns per lane: 4 (d = 128) or 2 (d = 64)
  constexpr int kWarps = 4;
  __shared__ float s_m[kWarps], s_l[kWarps];
  __shared__ float s_o[kWarps][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x / n_split, sp = blockIdx.x % n_split;
  const int b = bh / H, h = bh % H;
  const int k0 = min(sp * kbps * 128, Nk), k1 = min((sp + 1) * kbps * 128, Nk);
  const size_t rows = static_cast<size_t>(sp) * BH + bh;  // partial row (Nq = 1)
  if (k0 >= k1) {  // an empty split: LSE = -inf, O not read by the merge
    if (threadIdx.x == 0) lse_part[rows] = -INFINITY;
    return;
  }
  const __nv_bfloat16* qh = q + b * sq.s[2] + h * sq.s[1] + E * lane;
  const __nv_bfloat16* kh = k + b * sk.s[2] + h * sk.s[1] + E * lane;
  const __nv_bfloat16* vh = v + b * sv.s[2] + h * sv.s[1] + E * lane;
  float qf[E];
#pragma unroll
  for (int e = 0; e < E; ++e) qf[e] = __bfloat162float(qh[e]) * scale_log2;
  float m = -INFINITY, lsum = 0.f, o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = 0.f;

  for (int c0 = k0 + KC * warp; c0 < k1; c0 += KC * kWarps) {
    const int nkeys = min(KC, k1 - c0);
    // The chunk's K and V rows, every load issued before any arithmetic and none
    // behind a branch (a ragged last chunk re-reads its last row; those scores are
    // masked to -inf below, so their P is 0).
    uint32_t kr[KC][E / 2], vr[KC][E / 2];
#pragma unroll
    for (int j = 0; j < KC; ++j) {
      const int jr = c0 + (j < nkeys ? j : nkeys - 1);
      const __nv_bfloat16* kp = kh + static_cast<size_t>(jr) * sk.s[0];
      const __nv_bfloat16* vp = vh + static_cast<size_t>(jr) * sv.s[0];
      if constexpr (E == 4) {
        const uint2 a = __ldg(reinterpret_cast<const uint2*>(kp)), c = __ldg(reinterpret_cast<const uint2*>(vp));
        kr[j][0] = a.x;
        kr[j][1] = a.y;
        vr[j][0] = c.x;
        vr[j][1] = c.y;
      } else {
        kr[j][0] = __ldg(reinterpret_cast<const uint32_t*>(kp));
        vr[j][0] = __ldg(reinterpret_cast<const uint32_t*>(vp));
      }
    }
    // Partial dots of the lane's columns, then the butterfly: lane j ends with q . k_j.
    float t[KC];
#pragma unroll
    for (int j = 0; j < KC; ++j) {
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < E / 2; ++e) {
        const float2 kf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kr[j][e]));
        acc = fmaf(qf[2 * e], kf.x, acc);
        acc = fmaf(qf[2 * e + 1], kf.y, acc);
      }
      t[j] = acc;
    }
#pragma unroll
    for (int w = KC / 2; w >= 1; w >>= 1) {
      const bool upper = (lane & w) != 0;
#pragma unroll
      for (int i = 0; i < w; ++i) {
        const float send = upper ? t[i] : t[i + w];
        const float keep = upper ? t[i + w] : t[i];
        t[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
      }
    }
    // 16-key chunks: lanes l and l + 16 hold the two half-warps' sums of key l % 16.
    if (KC == 16) t[0] += __shfl_xor_sync(0xffffffffu, t[0], 16);
    const int kj = lane % KC;
    const float sj = kj < nkeys ? t[0] : -INFINITY;  // score of key c0 + lane % KC (base 2)
    float cm = sj;
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, w));
    const float m_new = fmaxf(m, cm);  // finite: the chunk has at least one key
    const float alpha = ex2_approx(m - m_new);  // 0 on the first chunk (m = -inf)
    const float p = ex2_approx(sj - m_new);
    lsum = lsum * alpha + (lane < KC ? p : 0.f);  // 16-key chunks: each key once
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] *= alpha;
#pragma unroll
    for (int j = 0; j < KC; ++j) {
      const float pj = __shfl_sync(0xffffffffu, p, j);
#pragma unroll
      for (int e = 0; e < E / 2; ++e) {
        const float2 vf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vr[j][e]));
        o[2 * e] = fmaf(pj, vf.x, o[2 * e]);
        o[2 * e + 1] = fmaf(pj, vf.y, o[2 * e + 1]);
      }
    }
    m = m_new;
  }
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, w);
  if (lane == 0) {
    s_m[warp] = m;
    s_l[warp] = lsum;
  }
#pragma unroll
  for (int e = 0; e < E; ++e) s_o[warp][E * lane + e] = o[e];
  __syncthreads();
  if (warp == 0) {
    float M = s_m[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) M = fmaxf(M, s_m[w]);
    float L = 0.f, acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float a = s_m[w] == -INFINITY ? 0.f : ex2_approx(s_m[w] - M);  // a warp with no chunk weighs 0
      L += s_l[w] * a;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] += s_o[w][E * lane + e] * a;
    }
    const float inv = 1.f / L;
    float* dst = o_part + rows * D + E * lane;
#pragma unroll
    for (int e = 0; e < E; ++e) dst[e] = acc[e] * inv;
    if (lane == 0) lse_part[rows] = (M + log2f(L)) * 0.69314718055994530942f;
  }
}

}  // namespace

int decode_ctas_per_sm(int d) {
  int n = 0;
  if (d != 64 || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_partial_kernel<64, 32>, 128, 0) != cudaSuccess ||
      n < 1)
    n = 4;
  return n;
}

cudaError_t launch_decode_partial(const SplitKvArgs& a, cudaStream_t stream) {
  if (a.d != 64) return cudaErrorInvalidValue;  // d = 128 streams faster on the tensor-core kernel
  const int BH = a.B * a.H;
  const unsigned grid = static_cast<unsigned>(BH) * static_cast<unsigned>(a.n_split);
  const float scale_log2 = a.scale * 1.4426950408889634f;
  const int kbps = splitkv_kbps(a.Nk, a.n_split);
  decode_partial_kernel<64, 32><<<grid, 128, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k),
      static_cast<const __nv_bfloat16*>(a.v), a.sq, a.sk, a.sv, a.o_part, a.lse_part, a.H, BH, a.Nk, a.n_split, kbps,
      scale_log2);
  return cudaGetLastError();
}

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
