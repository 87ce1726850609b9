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
// One CTA of 4 warps per (head, split).  A row of K or V is read by L = d/8 lanes,
// 16 bytes (8 columns) each, so one warp load instruction covers R = 32/L rows
// (4 at d = 64, 2 at d = 128): lane l takes columns 8 (l mod L) .. +7 of row
// group g = l / L.  A chunk is 8 such loads per tensor, KC = 8 R keys (32 or 16);
// warp w takes the split's chunks w, w + 4, ...  Chunk row rho = 8-slot index i
// times R plus g.  All of a chunk's loads are issued before its arithmetic and
// none sits behind a branch (rows past the split re-read its last row; their
// scores are masked to -inf).  Per chunk:
//  * partial dots: for each of its 8 rows, q . k over the lane's 8 columns;
//  * a butterfly over the 8 lanes of an aligned group (widths 4, 2, 1: a lane keeps
//    the half of its values whose slot index has its bit of the width and adds the
//    partner's copy of that half; at d = 128 one more exchange adds the two 8-lane
//    halves of a row) leaves the score of slot i = l mod 8 in lane l;
//  * online softmax in base 2 (the scale and log2 e are folded into q): chunk
//    maximum, the running reference, p = 2^(s - m), O and the row sum rescaled by
//    2^(m_old - m);
//  * O[c] += p_i v_i[c] over the lane's 8 rows, p_i taken from lane g L + i.
// At the end the R row groups' O are summed with shuffles, and the four warps'
// (m, l, O) are merged through shared memory exactly as the split merge does; the
// partial is O / l in fp32 and LSE = ln 2 (m + log2 l), -inf for an empty split.
// All arithmetic is fp32 (the inputs bf16).  Only d = 64 is built: at d = 128 this
// kernel streamed 0.93 of HBM bandwidth at B = 8, H = 16, Nk = 32768 but 0.79 at
// B = 1, H = 16, Nk = 131072, against 0.92 and 0.85 for the tensor-core kernel,
// which keeps that case.
template <int D>
__global__ void __launch_bounds__(128) decode_partial_kernel(const __nv_bfloat16* __restrict__ q,
                                                             const __nv_bfloat16* __restrict__ k,
                                                             const __nv_bfloat16* __restrict__ v, Strides sq,
                                                             Strides sk, Strides sv, float* __restrict__ o_part,
                                                             float* __restrict__ lse_part, int H, int BH, int Nk,
                                                             int n_split, int kbps, float scale_log2) {
  constexpr int L = D / 8;    // lanes per row
  constexpr int R = 32 / L;   // rows per warp load
  constexpr int KC = 8 * R;   // keys per chunk
  constexpr int kWarps = 4;
  __shared__ float s_m[kWarps], s_l[kWarps];
  __shared__ __align__(16) float s_o[kWarps][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / L, cg = lane % L;  // row group, column group (columns 8 cg .. 8 cg + 7)
  const int bh = blockIdx.x / n_split, sp = blockIdx.x % n_split;
  const int b = bh / H, h = bh % H;
  const int k0 = min(sp * kbps * 128, Nk), k1 = min((sp + 1) * kbps * 128, Nk);
  const size_t rows = static_cast<size_t>(sp) * BH + bh;  // partial row (Nq = 1)
  if (k0 >= k1) {  // an empty split: LSE = -inf, O not read by the merge
    if (threadIdx.x == 0) lse_part[rows] = -INFINITY;
    return;
  }
  const __nv_bfloat16* kh = k + b * sk.s[2] + h * sk.s[1] + 8 * cg;
  const __nv_bfloat16* vh = v + b * sv.s[2] + h * sv.s[1] + 8 * cg;
  float qf[8];
  {
    const uint4 qv = *reinterpret_cast<const uint4*>(q + b * sq.s[2] + h * sq.s[1] + 8 * cg);
    const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qw[e]));
      qf[2 * e] = f.x * scale_log2;
      qf[2 * e + 1] = f.y * scale_log2;
    }
  }
  float m = -INFINITY, lsum = 0.f, o[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = 0.f;
  const bool counts = L == 8 || (lane & 8) == 0;  // d = 128: lanes l and l ^ 8 hold the same row

  for (int c0 = k0 + KC * warp; c0 < k1; c0 += KC * kWarps) {
    const int last = k1 - 1 - c0;  // chunk rows past this are re-reads of the split's last row
    uint4 kr[8], vr[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rho = min(i * R + grp, last);
      kr[i] = __ldg(reinterpret_cast<const uint4*>(kh + static_cast<size_t>(c0 + rho) * sk.s[0]));
      vr[i] = __ldg(reinterpret_cast<const uint4*>(vh + static_cast<size_t>(c0 + rho) * sv.s[0]));
    }
    float t[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t kw[4] = {kr[i].x, kr[i].y, kr[i].z, kr[i].w};
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 kf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kw[e]));
        acc = fmaf(qf[2 * e], kf.x, acc);
        acc = fmaf(qf[2 * e + 1], kf.y, acc);
      }
      t[i] = acc;
    }
#pragma unroll
    for (int w = 4; w >= 1; w >>= 1) {
      const bool upper = (lane & w) != 0;
#pragma unroll
      for (int i = 0; i < w; ++i) {
        const float send = upper ? t[i] : t[i + w];
        const float keep = upper ? t[i + w] : t[i];
        t[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
      }
    }
    if (L == 16) t[0] += __shfl_xor_sync(0xffffffffu, t[0], 8);
    const int my_rho = (lane & 7) * R + grp;  // the chunk row whose score this lane now holds
    const float sj = my_rho <= last ? t[0] : -INFINITY;
    float cm = sj;
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, w));
    const float m_new = fmaxf(m, cm);  // finite: the chunk has at least one key
    const float alpha = ex2_approx(m - m_new);  // 0 on the first chunk (m = -inf)
    const float p = ex2_approx(sj - m_new);
    lsum = lsum * alpha + (counts ? p : 0.f);
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] *= alpha;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float pi = __shfl_sync(0xffffffffu, p, grp * L + i);  // p of chunk row i R + grp
      const uint32_t vw[4] = {vr[i].x, vr[i].y, vr[i].z, vr[i].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 vf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vw[e]));
        o[2 * e] = fmaf(pi, vf.x, o[2 * e]);
        o[2 * e + 1] = fmaf(pi, vf.y, o[2 * e + 1]);
      }
    }
    m = m_new;
  }
  // Sum the R row groups' O (lanes with the same column group), then the row sums.
#pragma unroll
  for (int w = L; w < 32; w <<= 1)
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] += __shfl_xor_sync(0xffffffffu, o[e], w);
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, w);
  if (lane == 0) {
    s_m[warp] = m;
    s_l[warp] = lsum;
  }
  if (grp == 0) {
    float4* dst = reinterpret_cast<float4*>(&s_o[warp][8 * cg]);
    dst[0] = make_float4(o[0], o[1], o[2], o[3]);
    dst[1] = make_float4(o[4], o[5], o[6], o[7]);
  }
  __syncthreads();
  if (warp == 0) {
    constexpr int E = D / 32;  // output columns per lane
    float M = s_m[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) M = fmaxf(M, s_m[w]);
    float Lw = 0.f, acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float a = s_m[w] == -INFINITY ? 0.f : ex2_approx(s_m[w] - M);  // a warp with no chunk weighs 0
      Lw += s_l[w] * a;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] += s_o[w][E * lane + e] * a;
    }
    const float inv = 1.f / Lw;
    float* dst = o_part + rows * D + E * lane;
#pragma unroll
    for (int e = 0; e < E; ++e) dst[e] = acc[e] * inv;
    if (lane == 0) lse_part[rows] = (M + log2f(Lw)) * 0.69314718055994530942f;
  }
}

}  // namespace

int decode_ctas_per_sm(int d) {
  int n = 0;
  if (d != 64 || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_partial_kernel<64>, 128, 0) != cudaSuccess ||
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
  decode_partial_kernel<64><<<grid, 128, 0, stream>>>(
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
