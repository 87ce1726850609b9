// Internal interface between the C-ABI layer (fa_api.cu) and the kernel
// translation units.  Nothing here is exported from the shared library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fa {

// Tile geometry shared by every kernel: 128 query rows per MMA tile (the
// tcgen05 M=128 datapath, one TMEM lane per row) and 128 keys per K/V tile.
constexpr int kBlockQ = 128;
constexpr int kBlockK = 128;
// A TMA box of bf16 data is at most 64 elements (128 bytes) wide under the
// 128-byte swizzle, so a d=128 row is staged as two boxes.
constexpr int kBoxCols = 64;

struct DebugKnobs {
  uint64_t wait_limit_ns;   // deadline of every bounded mbarrier wait
  int fault;                // test-only fault injection (0 = none)
};

// Element strides {row, head, batch} of a [B, H, N, d]-indexed tensor whose d is
// contiguous.  The dense [B, H, N, d] layout is {d, N d, H N d}.
struct Strides {
  int64_t s[3];
};
inline Strides dense_strides(int H, int N, int d) {
  return Strides{{static_cast<int64_t>(d), static_cast<int64_t>(N) * d, static_cast<int64_t>(H) * N * d}};
}

struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  Strides sq, sk, sv, so;
  int B, H, N, d;
  int causal;
  float scale;
  unsigned int* err_word;
  DebugKnobs dbg;
};

// Forward launcher (fa_fwd.cu).  Returns a cudaError_t.
cudaError_t launch_fwd_bf16(const FwdArgs& a, cudaStream_t stream);

// Split-KV forward (fa_fwd.cu): the keys are cut into n_split ranges of
// splitkv_kbps(Nk, n_split) 128-key blocks; for each range the normalised
// partial O (fp32 [n_split, B*H, Nq, d]) and its LSE (fp32 [n_split, B*H, Nq],
// -inf where a row sees no key of the range).  Causal queries are aligned with
// the last keys (query i sees key j iff j <= i + Nk - Nq).
struct SplitKvArgs {
  const void* q;
  const void* k;
  const void* v;
  Strides sq, sk, sv;  // element strides (row, head, batch) of q, k, v
  float* o_part;
  float* lse_part;
  int B, H, Nq, Nk, d, n_split;
  int causal;
  float scale;
  unsigned int* err_word;
  DebugKnobs dbg;
};
int splitkv_kbps(int Nk, int n_split);
cudaError_t launch_fwd_splitkv_partial(const SplitKvArgs& a, cudaStream_t stream);
// The same partials for one query row on the CUDA cores (fa_splitkv.cu), taken
// where it streams K and V faster than the tensor-core kernel: Nq = 1 at d = 64.
inline bool decode_takes(int Nq, int d) { return Nq == 1 && d == 64; }
cudaError_t launch_decode_partial(const SplitKvArgs& a, cudaStream_t stream);
// CTAs of the one-row kernel (one per split and head) resident on one SM at head dim d.
int decode_ctas_per_sm(int d);

// Exact merge of split-KV partials into bf16 O [B*H, Nq, d] and fp32 LSE
// [B*H, Nq] (fa_splitkv.cu).
struct MergeArgs {
  const float* o_part;
  const float* lse_part;
  void* o;
  Strides so;  // element strides (row, head, batch) of o
  float* lse;
  int n_split, BH, H, Nq, d;
};
cudaError_t launch_merge_partials(const MergeArgs& a, cudaStream_t stream);

struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  Strides sq, sk, sv, so, sdo, sdq, sdk, sdv;
  void* workspace;
  int B, H, N, d;
  int causal;
  int deterministic;  // 1: dQ accumulates as fixed-point integers (bitwise reproducible)
  float scale;
  unsigned int* err_word;
  DebugKnobs dbg;
};

// Workspace of the backward: fp32 dQ accumulator [BH, N, d] (int32 in the
// deterministic mode), then the main kernel's per-query operand tiles (LSE * log2(e)
// and D as bf16 hi/lo pairs, 64 bytes per query row, npad = N rounded up to 64
// rows per head), then (deterministic mode) the largest |dO_i| per 64-row block
// [BH, npad / 64] and the head's largest |v_j| and |k_jc| [BH, 2].  Every region
// starts on a 256-byte boundary.
struct BwdWorkspace {
  size_t off_dq, off_aug, off_dqmax, off_kvmax, total;
  int npad;
};
BwdWorkspace bwd_workspace_layout(int B, int H, int N, int d);

// Backward launchers (fa_bwd.cu).  launch_bwd_bf16 = prep, main, dq in order on
// `stream`; each stage reads only the BwdArgs fields it needs.
cudaError_t launch_bwd_prep(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_main(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_bf16(const BwdArgs& a, cudaStream_t stream);

// Every check fa_bwd makes except those on the workspace (fa_api.cu): sizes,
// pointers, alignment and the device.  Returns an fa_status; FA_OK also for an
// empty problem.
int bwd_validate_without_workspace(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                   const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                                   int causal, float scale);

// Workspace of the FP8 path (written by fa_fp8_prepare, read by fa_fwd_fp8):
// e4m3 codes of the rotated Q and K, row-major [BH, N, d]; e4m3 codes of V
// transposed [BH, d, npad] (keys contiguous, npad = N rounded up to 128); fp32
// dequantisation scales per 64-row tile [BH, ntiles] for Q, K, V.  Every region
// starts on a 256-byte boundary.
struct Fp8Layout {
  size_t off_q8, off_k8, off_v8t, off_sq, off_sk, off_sv, total;
  int ntiles, npad;
};
Fp8Layout fp8_layout(int B, int H, int N, int d);

// FP8 forward launcher (fa_fwd.cu): reads the prepared workspace (q, k, v of
// FwdArgs unused), writes bf16 O and fp32 LSE; d = 64 or 128.
cudaError_t launch_fwd_fp8(const FwdArgs& a, const void* workspace, cudaStream_t stream);

// FP8 backward helpers (fa_fp8_bwd.cu).  launch_fp8_dequant: bf16 operands
// bf16_rn(decode(code) * tile scale) of the rotated Q, K and of V, dense [BH, N, d],
// from a prepared FP8 workspace.  launch_fp8_unrotate: rows of d (64 or 128) of dq
// and dk (dense, `rows` each) replaced in place by bf16((x H_d) * s).
cudaError_t launch_fp8_dequant(const void* fp8_ws, void* qr, void* kr, void* vr, int B, int H, int N, int d,
                               cudaStream_t stream);
cudaError_t launch_fp8_unrotate(void* dq, void* dk, const int8_t* signs, long long rows, int d,
                                cudaStream_t stream);

struct Fp8PrepArgs {
  const void* q;
  const void* k;
  const void* v;
  Strides sq, sk, sv;      // element strides (row, head, batch) of q, k, v
  int in_bf16;             // 0: fp32 inputs, 1: bf16 inputs
  const int8_t* signs;     // [d], the sign of each entry is used; NULL: signs from `seed`
  uint64_t seed;           // used when signs is NULL (see seeded_sign)
  void* workspace;
  int B, H, N, d;
};

// Output c (0-based) of SplitMix64 started at state `seed` (Steele, Lea and
// Flood, OOPSLA 2014): x = seed + (c + 1) * 0x9E3779B97F4A7C15, then the
// generator's two xor-shift-multiply rounds and a final xor-shift, all mod 2^64.
// The seeded rotation takes column c's sign from the top bit of output c
// (set: -1).  Host and device share this one definition.
__host__ __device__ inline uint64_t splitmix64_at(uint64_t seed, uint64_t c) {
  uint64_t z = seed + (c + 1) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
__host__ __device__ inline int seeded_sign(uint64_t seed, int c) {
  return (splitmix64_at(seed, static_cast<uint64_t>(c)) >> 63) ? -1 : 1;
}
cudaError_t launch_fp8_prepare(const Fp8PrepArgs& a, cudaStream_t stream);

// Encodes a 3-D tiled tensor map over a [BH, N, cols] row-major tensor with
// `elem_bytes`-byte elements, box {box_cols, box_rows, 1}, 128-byte swizzle.
// Implemented in fa_api.cu (driver entry point resolved once).
// 2-D map over a row-major matrix (row stride in elements); optional 128-byte swizzle.
cudaError_t make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int elem_bytes, int cols,
                         int rows, int64_t row_stride_elems, int box_cols, int box_rows, bool swizzle128);

// 4-bit-weight GEMM (fa_w4a16.cu): Y [M, N] = X [M, K] (fp16) times the transpose
// of W [N, K], W given as packed 4-bit codes wq [N, K/8] with fp16 scales and
// uint8 zero points [K/128, N].  n_split > 1 cuts K into that many ranges whose
// fp32 partials [n_split, M, N] land in `partials` and are summed in order.
struct W4a16Args {
  const void* x;
  const void* wq;
  const void* scales;
  const void* zeros;
  void* y;
  float* partials;
  int M, N, K, n_split;
  unsigned int* err_word;
  DebugKnobs dbg;
};
int w4a16_chunks_per_split(int K, int n_split);
// True when M (and K) select the CUDA-core matrix-vector path: one pass over K per
// output row, no split and no workspace.
bool w4a16_uses_gemv(int M, int K);
cudaError_t launch_w4a16(const W4a16Args& a, cudaStream_t stream);

cudaError_t make_tmap_4d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int elem_bytes, int cols,
                         int rows, int heads, int batch, const int64_t strides[3], int box_cols, int box_rows,
                         CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B);
cudaError_t make_tmap_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int elem_bytes,
                         int cols, int rows, int depth, int box_cols, int box_rows);

}  // namespace fa
