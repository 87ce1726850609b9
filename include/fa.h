/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention library (libfa.so).
 *
 * What it computes.  For every batch b and head h, with Q, K, V the N x d
 * matrices of that (b, h):
 *
 *     O   = softmax(scale * Q K^T  [+ causal mask]) V
 *     LSE = per-row natural-log logsumexp of the scaled (masked) scores
 *
 * exactly as standard self-attention defines it ("FlashAttention-2 (DE)",
 * section "Hintergrund: Das Attention-Problem in Transformern"), but computed
 * tile by tile with an online softmax so that the N x N score matrix is never
 * materialised ("FlashAttention-2 (DE)", same section, "IO-Awareness" and
 * "Tiling"; "FlashAttention-Skalierung, Multi-GPU-Training und
 * Gewichtsquantisierung", section 1, FlashAttention-2 bullets).  The result is
 * the standard one up to floating-point rounding: the tiling loses no accuracy
 * (lead of "FlashAttention-2 (DE)").
 *
 * Conventions shared by every call:
 *  - Tensors are dense, row-major [B, H, N, d] ("BHND": each head is one N x d
 *    matrix, d contiguous).  LSE is [B, H, N] float32.  No strides are taken.
 *  - Causal: key j is visible to query i iff j <= i (0-based, same N for
 *    queries and keys).  Masked scores are excluded (weight exactly 0).
 *  - scale must be finite and > 0 (the usual value is 1/sqrt(d)).
 *  - d must be 64 or 128.  N >= 1 is arbitrary (no multiple-of-128 rule).
 *  - All pointers are DEVICE pointers owned by the caller, on the current CUDA
 *    device, and must stay valid until the work queued on `stream` finishes.
 *    The library never allocates device memory in these calls and keeps no
 *    reference to the pointers after the call returns.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *    asynchronous with respect to the host: they validate, enqueue and return.
 *  - Every call is thread-safe.
 *  - Errors: validation happens synchronously, before anything is enqueued;
 *    a nonzero status means nothing was launched.  Errors detected by a kernel
 *    while it runs (a bounded wait that expired) are reported by the next
 *    fa_sync_check() on that device.  No C++ exception crosses this ABI.
 *  - B * H * N == 0 is a no-op returning FA_OK (pointers may then be NULL).
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fa_stream_t; /* identical to cudaStream_t */

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,  /* null pointer, negative size, causal not 0/1, scale not finite and > 0 */
  FA_ERR_UNSUPPORTED = 2,  /* d not 64/128, sizes beyond the kernel's index range, or not an sm_103 GPU */
  FA_ERR_MISALIGNED = 3,   /* a tensor pointer not 16-byte aligned (LSE: 4-byte) */
  FA_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed (launch, tensor-map encoding, ...) */
  FA_ERR_TIMEOUT = 5,      /* a kernel gave up on a bounded wait; its outputs are undefined */
  FA_ERR_WORKSPACE = 6     /* caller workspace missing or smaller than required */
} fa_status;

/* Static, human-readable text for a status code (never NULL). */
FA_API const char* fa_strerror(int status);

/* Library ABI version: (major << 16) | minor. */
FA_API int fa_version(void);

/*
 * fa_fwd -- bf16 forward pass.
 *   q, k, v : const bf16 [B, H, N, d]  (inputs)
 *   o       : bf16 [B, H, N, d]        (output, fully overwritten)
 *   lse     : float [B, H, N]          (output: ln sum_j exp(scale * q_i . k_j) over visible j)
 * Numerics: scores accumulate in fp32 on the tensor cores; P is rounded to
 * bf16 for the P V product; the running sum, the final 1/l and LSE are fp32;
 * O is rounded to bf16 once at the end.  The result is bitwise reproducible
 * run to run for the same inputs, sizes and device.
 * Returns FA_OK or an error above (synchronous validation / launch failure).
 */
FA_API int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
           int causal, float scale, fa_stream_t stream);

/*
 * fa_fwd_strided -- fa_fwd for tensors in other layouts, e.g. [B, N, H, d] as a
 * projection produces it before any transpose.  Element (b, h, n, c) of a tensor
 * lives at ptr + b*strides[2] + h*strides[1] + n*strides[0] + c (in elements; d is
 * contiguous).  A NULL strides pointer means the dense [B, H, N, d] layout
 * {d, N*d, H*N*d}.  Every stride must be positive and a multiple of 8 elements
 * (16 bytes; FA_ERR_MISALIGNED otherwise), and strides[0] >= d.  Output rows must
 * not overlap one another or any input.  LSE stays dense [B, H, N].  Results are
 * bitwise those of fa_fwd on the same values laid out densely.
 */
FA_API int fa_fwd_strided(const void* q, const int64_t* q_strides, const void* k, const int64_t* k_strides,
                          const void* v, const int64_t* v_strides, void* o, const int64_t* o_strides, float* lse,
                          int B, int H, int N, int d, int causal, float scale, fa_stream_t stream);

/*
 * fa_bwd_workspace_size -- bytes of device workspace fa_bwd (and
 * fa_bwd_deterministic) needs for these sizes (0 if the sizes are invalid or
 * unsupported).  The workspace holds an fp32 dQ accumulator [B, H, N, d], two
 * fp32 vectors of B*H*roundup(N, 64), and B*H*(roundup(N, 64)/64 + 2) floats of
 * bounds used by the deterministic variant.
 */
FA_API size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * fa_bwd -- bf16 backward pass of fa_fwd, d = 64 or 128.
 * The gradient follows from the chain rule applied to the definition above
 * (the pages give the forward only): with P = softmax(scale * Q K^T [+mask]),
 *     dV = P^T dO,  dP = dO V^T,  D_i = sum_c dO_ic O_ic,
 *     dS = P * (dP - D),  dQ = scale * dS K,  dK = scale * dS^T Q.
 * P is recomputed from `lse` (as written by fa_fwd for the same q, k, scale,
 * causal); the N x N matrices are never stored.
 *   q, k, v, o, dout : const bf16 [B, H, N, d]   (o, lse: the forward's outputs)
 *   lse              : const float [B, H, N]
 *   dq, dk, dv       : bf16 [B, H, N, d]          (outputs, fully overwritten)
 *   workspace        : device memory of at least fa_bwd_workspace_size(...)
 *                      bytes, 256-byte aligned, owned by the caller; its
 *                      contents on entry do not matter and are scratch after.
 * Numerics: fp32 accumulation on the tensor cores; P and dS are rounded to
 * bf16 as MMA operands; dQ accumulates across key blocks with fp32 atomic adds,
 * so dQ may differ in the last bits from run to run (dK, dV do not).
 * Errors: as fa_fwd; additionally FA_ERR_WORKSPACE for a missing or short
 * workspace; the workspace must be 256-byte aligned (FA_ERR_MISALIGNED otherwise).
 */
FA_API int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                  void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes, int B, int H, int N, int d,
                  int causal, float scale, fa_stream_t stream);

/*
 * fa_bwd_strided -- fa_bwd (deterministic = 0) or fa_bwd_deterministic
 * (deterministic = 1) for strided tensors, with the stride rules of
 * fa_fwd_strided for each of q, k, v, o, dout, dq, dk, dv (NULL = dense).  The
 * workspace and LSE stay dense.  Results are bitwise those of the dense call on
 * the same values (dQ of the non-deterministic mode up to its summation order).
 */
FA_API int fa_bwd_strided(const void* q, const int64_t* q_strides, const void* k, const int64_t* k_strides,
                          const void* v, const int64_t* v_strides, const void* o, const int64_t* o_strides,
                          const void* dout, const int64_t* dout_strides, const float* lse, void* dq,
                          const int64_t* dq_strides, void* dk, const int64_t* dk_strides, void* dv,
                          const int64_t* dv_strides, void* workspace, size_t ws_bytes, int B, int H, int N, int d,
                          int causal, float scale, int deterministic, fa_stream_t stream);

/*
 * fa_bwd_deterministic -- fa_bwd whose dQ is the same bits on every run.
 * The pages call the method exact and deterministic ("FlashAttention-2 (DE)",
 * section "Leistung und Effizienz").  fa_bwd's dQ sums the contributions of the
 * key blocks with fp32 atomic adds, whose order varies run to run; here each
 * contribution is rounded once to an integer multiple of 2^-S and added as int32,
 * and integer addition does not depend on order.  S is a power of two chosen per
 * 64-row query block from a bound on |dQ| that holds for any inputs:
 *     |dQacc_ic| <= 2 |dO_i| max_j |v_j| max_jc |k_jc|   (x 1.125 margin)
 * so that every partial sum stays below 2^22 in magnitude; the rounding of each
 * contribution is at most 2^-S / 2, far below the bf16 output's rounding.  dK and
 * dV are those of fa_bwd (already reproducible).  Costs one extra pass over K and
 * V for the bound.  Arguments, workspace and errors: exactly as fa_bwd.
 * Precondition: `lse` is the forward's LSE for the same q, k, scale and causal
 * (as fa_fwd writes it).  The bound above assumes that the recomputed
 * probabilities of each row sum to about 1; an LSE computed from other operands
 * breaks that assumption, and the int32 sums may then wrap without any error
 * being reported (fa_bwd would return finite but equally meaningless values).
 */
FA_API int fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                                int B, int H, int N, int d, int causal, float scale, fa_stream_t stream);

/*
 * The three stages of fa_bwd, for callers that schedule or time them one by one.
 * fa_bwd(...) is exactly fa_bwd_prep, fa_bwd_main, fa_bwd_dq in that order on
 * one stream with one workspace; arguments mean what they mean for fa_bwd.
 *
 * fa_bwd_prep: D_i = sum_c dO_ic O_ic and LSE_i * log2(e) into the workspace
 *   (rows padded to a multiple of 64: D = 0, LSE = +inf), and zeroes the fp32
 *   dQ accumulator.  Bandwidth-bound.
 * fa_bwd_main: the dK/dV-outer loop (per 128-key block: recompute P from LSE,
 *   dV += P^T dO, dP = dO V^T, dS = P (dP - D), dK += dS^T Q, dQ += dS K into
 *   the fp32 accumulator).  Writes dk, dv; needs the workspace fa_bwd_prep filled.
 * fa_bwd_dq: dq = bf16(scale * accumulator).
 */
FA_API int fa_bwd_prep(const void* o, const void* dout, const float* lse, void* workspace, size_t ws_bytes, int B,
                       int H, int N, int d, fa_stream_t stream);
FA_API int fa_bwd_main(const void* q, const void* k, const void* v, const void* dout, void* dk, void* dv,
                       void* workspace, size_t ws_bytes, int B, int H, int N, int d, int causal, float scale,
                       fa_stream_t stream);
FA_API int fa_bwd_dq(const void* workspace, size_t ws_bytes, void* dq, int B, int H, int N, int d, float scale,
                     fa_stream_t stream);

/*
 * fa_bwd_noalloc -- fa_bwd without a caller workspace; allocates nothing.
 * The pages have no counterpart to this call: it exists for callers that
 * cannot allocate device memory themselves (a plugin inside a host framework
 * that owns all device memory and gives plugins no allocator, or a
 * latency-critical loop where cudaMalloc, which may synchronise the device, is
 * not allowed).  The caller still passes every input and output exactly as for
 * fa_bwd; the scratch comes from one fixed buffer of
 * fa_bwd_noalloc_max_workspace() bytes (64 MiB) in this library's device code.
 * Limits and behaviour:
 *  - The buffer is reserved on a device when the library's device code is loaded
 *    into a context there: with lazy module loading (the CUDA default) at the
 *    first call of this entry point in that context; with eager loading
 *    (CUDA_MODULE_LOADING=EAGER) when any context is created while the library
 *    is loaded, whether or not this entry point is ever called.  It is held
 *    until that context is destroyed or the process exits.
 *  - Arguments are validated exactly as fa_bwd validates them (same statuses)
 *    before the buffer is touched; then sizes whose fa_bwd_workspace_size()
 *    exceeds the buffer are rejected with FA_ERR_WORKSPACE before anything is
 *    launched (this admits B*H*N up to about 116,000 rows at d = 128 and
 *    209,000 at d = 64).
 *  - It calls no cudaMalloc, cudaFree or other allocating routine.
 *  - Every call looks up the buffer's device address in the context current on
 *    the calling thread (a table lookup; a context replaced since, e.g. by
 *    cudaDeviceReset or a framework's own context, gets its own buffer).  The
 *    first call in a context loads the module that holds the buffer: make that
 *    first call before any stream capture.
 *  - Every call in a context shares the one buffer, which keeps the contents of
 *    the last call (the kernels initialise what must start at zero).  Calls that
 *    overlap on the GPU (e.g. on two streams at once) race on it: serialise them.
 */
FA_API int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                          const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal,
                          float scale, fa_stream_t stream);

/* Size in bytes of the fixed scratch buffer behind fa_bwd_noalloc (per device). */
FA_API size_t fa_bwd_noalloc_max_workspace(void);

/*
 * FP8 path ("FlashAttention-Skalierung, Multi-GPU-Training und
 * Gewichtsquantisierung", section 1, "Unterstützung geringer FP8-Präzision":
 * block quantisation plus multiplication of Q and K by a random orthogonal
 * matrix before quantising).
 *
 * fa_fp8_workspace_size -- bytes of device workspace the FP8 path needs (0 if
 *   the sizes are invalid).
 * fa_fp8_workspace_offsets -- byte offsets of the regions inside that workspace,
 *   written to offsets[0..7]: q8, k8, v8t, sq, sk, sv, then npad and ntiles.
 *   q8, k8: e4m3 codes [B, H, N, d] (row-major); v8t: e4m3 codes of V transposed
 *   [B, H, d, npad] (keys contiguous, npad = N rounded up to 128, padding zero);
 *   sq, sk, sv: fp32 dequantisation scales [B, H, ntiles], ntiles = ceil(N/64).
 *
 * fa_fp8_prepare -- fill the workspace from q, k, v.
 *   q, k, v   : const [B, H, N, d], fp32 (in_dtype = 0) or bf16 (in_dtype = 1)
 *   signs     : const int8 [d] on the device: the rotation's random signs s
 *               (an entry < 0 means -1, otherwise +1)
 *   For Q and K, each row x becomes y = (x * s) H_d (H_d the Sylvester
 *   Walsh-Hadamard matrix, entries +-1, so (QM)(KM)^T = d Q K^T with M = diag(s)
 *   H_d; fa_fwd_fp8 folds the 1/d into its scale).  V rows are unchanged.  Then
 *   per tile of 64 consecutive rows of one head: amax = max|y| (exact), scale =
 *   2^e with e the smallest integer such that amax <= 448 * 2^e (e clamped to
 *   [-126, 126]; scale 1 for an all-zero tile), codes = e4m3(y * 2^-e) with
 *   round-to-nearest-even and saturation (OCP E4M3, max 448), so that
 *   y ~= decode(code) * scale.  The transform is fp32 radix-2 butterflies with
 *   spans 1, 2, ..., d/2; the scaling by 2^-e is one fp32 multiply.
 *   Errors as fa_fwd; FA_ERR_WORKSPACE for a missing or short workspace;
 *   FA_ERR_INVALID_ARG for in_dtype not 0/1 or a NULL signs pointer.
 */
FA_API size_t fa_fp8_workspace_size(int B, int H, int N, int d);
FA_API int fa_fp8_workspace_offsets(int B, int H, int N, int d, size_t* offsets);
FA_API int fa_fp8_prepare(const void* q, const void* k, const void* v, int in_dtype, const int8_t* signs,
                          void* workspace, size_t ws_bytes, int B, int H, int N, int d, fa_stream_t stream);

/*
 * fa_fp8_prepare_seeded -- fa_fp8_prepare with the rotation's signs drawn from a
 * 64-bit seed instead of passed in: sign of column c = -1 if the top bit of
 * output c (0-based) of SplitMix64 started at state `seed` is set, else +1.
 * SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014): output c = mix(seed + (c + 1) * 0x9E3779B97F4A7C15)
 * with mix(z) = z3 ^ (z3 >> 31), z3 = (z2 ^ (z2 >> 27)) * 0x94D049BB133111EB,
 * z2 = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9, all modulo 2^64.  The signs are
 * computed on the device; the workspace, the codes and the errors are those of
 * fa_fp8_prepare given the same signs (fa_fp8_rotation_signs).
 *
 * fa_fp8_rotation_signs -- the d signs (+1 / -1) of that seed, written to
 * `signs`, HOST memory of d int8 (for fa_bwd_fp8, which takes the signs as a
 * device array).  Pure host code; FA_ERR_INVALID_ARG for d < 1 or NULL signs.
 */
FA_API int fa_fp8_prepare_seeded(const void* q, const void* k, const void* v, int in_dtype, uint64_t seed,
                                 void* workspace, size_t ws_bytes, int B, int H, int N, int d, fa_stream_t stream);
FA_API int fa_fp8_rotation_signs(uint64_t seed, int d, int8_t* signs);

/*
 * fa_fp8_prepare_strided -- fa_fp8_prepare for inputs in other layouts (e.g.
 * [B, N, H, d] straight from a projection), with the stride rules of
 * fa_fwd_strided for each of q, k, v (in elements of in_dtype; NULL = dense).
 * signs: as fa_fp8_prepare, or NULL to draw them from `seed` as
 * fa_fp8_prepare_seeded does (seed is ignored when signs is given).  The
 * workspace layout, the codes and the scales are bitwise those of
 * fa_fp8_prepare on the same values laid out densely.
 */
FA_API int fa_fp8_prepare_strided(const void* q, const int64_t* q_strides, const void* k, const int64_t* k_strides,
                                  const void* v, const int64_t* v_strides, int in_dtype, const int8_t* signs,
                                  uint64_t seed, void* workspace, size_t ws_bytes, int B, int H, int N, int d,
                                  fa_stream_t stream);

/*
 * fa_fwd_fp8 -- FP8 forward from a workspace filled by fa_fp8_prepare (same
 * B, H, N, d; d = 64 or 128).  Computes O = softmax(scale * Q K^T [+mask]) V and LSE
 * like fa_fwd, with both matmuls on e4m3 operands (kind::f8f6f4 tensor cores,
 * fp32 accumulation):
 *   S = (scale / d) * sQ(row tile) * sK(key tile) * (codesQ . codesK^T)
 *   (the rotation's H_d H_d^T = d I is undone by the 1/d);
 *   P = exp(S - m) is multiplied by sV(key tile) / max_tiles sV and rounded to
 *   e4m3 as the A operand of P V; O = acc * max sV / l, rounded to bf16 once.
 *   The row sum l and LSE use the unrounded P.
 *   o   : bf16 [B, H, N, d] (output)      lse : float [B, H, N] (output)
 * Errors as fa_fwd (FA_ERR_UNSUPPORTED for d not 64 or 128); FA_ERR_WORKSPACE
 * for a missing or short workspace (256-byte alignment required).
 */
FA_API int fa_fwd_fp8(const void* workspace, size_t ws_bytes, void* o, float* lse, int B, int H, int N, int d,
                      int causal, float scale, fa_stream_t stream);

/*
 * Backward pass of the FP8 attention.  The pages give FP8 for the forward only
 * (same section); its backward is taken straight through the quantisation (the
 * rounding's derivative taken as 1): the textbook gradient of attention on the
 * dequantised operands, carried back through the rotation M = diag(s) H_d:
 *   dQ = (dQ' H_d) * s,   dK = (dK' H_d) * s,   dV = dV'
 * with dQ', dK', dV' the gradients with respect to Q' = bf16(decode(q8) * sQ),
 * K' = bf16(decode(k8) * sK), V' = bf16(decode(v8) * sV) under the softmax scale
 * scale / d (the forward's).  With the power-of-two tile scales of
 * fa_fp8_prepare the bf16 rounding is exact: the backward sees the forward's
 * operand values.  The products run on bf16 tensor cores (the bf16
 * backward's kernels); the operands come from the FP8 workspace.
 *
 * fa_fp8_dequantize -- the operands alone: qr, kr, vr (bf16 [B, H, N, d], outputs,
 *   dense) = bf16_rn(fp32(decode(code)) * scale of the row's 64-row tile), one
 *   fp32 product then one rounding to nearest even.  d = 64 or 128.  Errors as
 *   fa_fwd_fp8 (FA_ERR_MISALIGNED: outputs not 16-byte aligned).
 *
 * fa_bwd_fp8_workspace_size -- bytes of workspace fa_bwd_fp8 needs (0 if invalid
 *   or unsupported): the bf16 backward's workspace, the three operands, and the
 *   recomputed forward's O and LSE.
 *
 * fa_bwd_fp8 -- dq, dk, dv (bf16 [B, H, N, d], outputs, dense) from
 *   fp8_ws     : const, filled by fa_fp8_prepare for these sizes (not modified)
 *   signs      : const int8 [d] on the device, the signs given to fa_fp8_prepare
 *   o, lse     : the forward's output and LSE (as from fa_fwd_fp8), dense; read
 *                only when recompute_forward = 0 (may be NULL otherwise)
 *   dout       : const bf16 [B, H, N, d]
 *   workspace  : device memory of fa_bwd_fp8_workspace_size(...) bytes, 256-byte
 *                aligned; overwritten
 *   scale      : the softmax scale given to fa_fwd_fp8 (of the unrotated problem)
 *   deterministic : 0 or 1, as fa_bwd_strided (1: dQ the same bits on every run)
 *   recompute_forward : 0 or 1.  The gradient needs D_i = dO_i . O_i with O from
 *                the UNROUNDED probabilities.  fa_fwd_fp8 rounds P to e4m3 for its
 *                P V product, so its O carries that error into D and from there
 *                into every dS of the row (a few percent RMS on dQ at N = 1000).
 *                With deterministic = 1 and recompute_forward = 0, `lse` must be
 *                the LSE fa_fwd_fp8 wrote for this workspace (see the
 *                precondition of fa_bwd_deterministic).
 *                1: O and LSE are recomputed by the bf16 forward on Q', K', V'
 *                (about 35 % more time); the result is the straight-through
 *                gradient to the bf16 backward's accuracy.  0: the caller's o and
 *                lse are used as given.
 * Stages on `stream`: dequantise, [bf16 forward,] the bf16 backward (prep, main,
 * dq), then the inverse rotation of dq and dk in place (fp32 butterflies, bf16
 * rounding).  d = 64 or 128.  Errors as fa_bwd, plus FA_ERR_WORKSPACE for a missing or
 * short FP8 workspace and FA_ERR_INVALID_ARG for a NULL signs pointer or a flag
 * not 0/1.
 */
FA_API int fa_fp8_dequantize(const void* fp8_ws, size_t fp8_ws_bytes, void* qr, void* kr, void* vr, int B, int H,
                             int N, int d, fa_stream_t stream);
FA_API size_t fa_bwd_fp8_workspace_size(int B, int H, int N, int d);
FA_API int fa_bwd_fp8(const void* fp8_ws, size_t fp8_ws_bytes, const int8_t* signs, const void* o, const void* dout,
                      const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes, int B, int H,
                      int N, int d, int causal, float scale, int deterministic, int recompute_forward,
                      fa_stream_t stream);

/*
 * Split-KV forward ("decode"-shaped attention: few queries, many keys) and the
 * exact merge of attention partials.  The setting is token-by-token inference,
 * which the pages call bandwidth-bound rather than compute-bound
 * ("FlashAttention-Skalierung, Multi-GPU-Training und Gewichtsquantisierung",
 * section 3); one head's keys are then too few work units to fill the GPU, so
 * the key range is cut into splits that run in parallel and are merged.
 *
 * Shapes: q [B, H, Nq, d]; k, v [B, H, Nk, d] (bf16, d contiguous; dense, or
 * strided through fa_fwd_splitkv_strided).
 * Causal (Nq <= Nk required): the queries are the LAST Nq positions, so query i
 * (0-based) sees key j iff j <= i + (Nk - Nq); with Nq == Nk this is fa_fwd's mask.
 * Split rule: keys form nkb = ceil(Nk / 128) blocks of 128; with
 * kbps = ceil(nkb / n_split), split s covers keys [128 s kbps, min(128 (s+1) kbps, Nk)).
 * Trailing splits may be empty.  1 <= n_split <= 1024.
 *
 * Partial of split s, row i (natural log):
 *   LSE_s[i] = ln sum_{j in s, visible} exp(scale q_i . k_j)   (-inf if no such j)
 *   O_s[i]   = sum_{j in s, visible} exp(scale q_i . k_j - LSE_s[i]) v_j
 * Merge: LSE = ln sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s, which is the
 * softmax over all keys (splits with LSE_s = -inf carry no weight and their O_s
 * is not read; a row with every split empty gets O = 0, LSE = -inf).
 */

/* Bytes of workspace fa_fwd_splitkv needs (fp32 partials: n_split * B*H*Nq*(d + 1)
 * floats, 256-byte aligned regions); 0 for invalid or unsupported sizes. */
FA_API size_t fa_splitkv_workspace_size(int B, int H, int Nq, int d, int n_split);

/* A split count for these sizes on the current device: the fewest splits (1..64,
 * each of at least 4 key blocks) within 2 % of the best balance of work units over
 * the SMs (for Nq == 1 at d == 64, over the SMs times the CTAs of the one-row
 * kernel resident on each); 1 when Nq > 128 and the unsplit units already cover
 * every SM.  Returns >= 1, or 0 for invalid sizes. */
FA_API int fa_splitkv_default_splits(int B, int H, int Nq, int Nk, int d);

/*
 * fa_fwd_splitkv_partial -- the partials only (the building block of a merge
 * done elsewhere, e.g. across devices holding different key ranges).
 *   o_part   : float [n_split, B, H, Nq, d]  (output; rows of empty splits unwritten)
 *   lse_part : float [n_split, B, H, Nq]     (output, every element written)
 * Numerics: as fa_fwd (fp32 scores on the tensor cores, bf16 P for P V), but O_s
 * stays fp32; for Nq == 1 at d == 64 every step is fp32 on the CUDA cores (P is
 * not rounded to bf16).  Errors: as fa_fwd; FA_ERR_INVALID_ARG also for n_split outside
 * [1, 1024], Nk < 1, or causal with Nq > Nk.  B * H * Nq == 0 is a no-op.
 */
FA_API int fa_fwd_splitkv_partial(const void* q, const void* k, const void* v, float* o_part, float* lse_part,
                                  int B, int H, int Nq, int Nk, int d, int n_split, int causal, float scale,
                                  fa_stream_t stream);

/*
 * fa_merge_partials -- exact merge of n_split partials laid out as above.
 *   o   : bf16 [B, H, Nq, d] (output)      lse : float [B, H, Nq] (output)
 * Bandwidth-bound; fp32 arithmetic; O rounded to bf16 once.
 */
FA_API int fa_merge_partials(const float* o_part, const float* lse_part, void* o, float* lse, int n_split, int B,
                             int H, int Nq, int d, fa_stream_t stream);

/*
 * fa_fwd_splitkv -- partials into `workspace`, then the merge: O and LSE of
 * softmax(scale Q K^T [+mask]) V for Nq queries against Nk keys.
 * n_split <= 0 selects fa_splitkv_default_splits(...).  The workspace (at least
 * fa_splitkv_workspace_size(B, H, Nq, d, n_split) bytes for the split count used,
 * 256-byte aligned, caller-owned) is scratch.  Errors: as the two calls above,
 * plus FA_ERR_WORKSPACE for a missing or short workspace.
 */
FA_API int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                          size_t ws_bytes, int B, int H, int Nq, int Nk, int d, int n_split, int causal, float scale,
                          fa_stream_t stream);

/*
 * fa_fwd_splitkv_strided -- fa_fwd_splitkv for q, k, v and o in other layouts,
 * with the stride rules of fa_fwd_strided (strides of q and o count Nq rows, of
 * k and v Nk rows; NULL = dense).  The partials in the workspace and LSE stay
 * dense.  Results are bitwise those of fa_fwd_splitkv on dense copies.
 */
FA_API int fa_fwd_splitkv_strided(const void* q, const int64_t* q_strides, const void* k, const int64_t* k_strides,
                                  const void* v, const int64_t* v_strides, void* o, const int64_t* o_strides,
                                  float* lse, void* workspace, size_t ws_bytes, int B, int H, int Nq, int Nk, int d,
                                  int n_split, int causal, float scale, fa_stream_t stream);

/*
 * W4A16: 4-bit weights times 16-bit activations, dequantised on the fly
 * ("FlashAttention-Skalierung, Multi-GPU-Training und Gewichtsquantisierung",
 * section 3, "Wie spezielle CUDA-Kernels während der Ausführung dequantisieren
 * (W4A16)": packed 4-bit weights are read from memory, unpacked in registers with
 * shifts and masks, given their scale and zero point, and fed as fp16 with the
 * fp16 activations to the tensor cores, never written back unpacked; for a
 * matrix-vector product the CUDA cores take that role, see Paths).
 *
 *   Y[m, n] = sum_k X[m, k] * W[n, k],   W[n, k] = fp16((q[n, k] - z[g, n]) * s[g, n]),  g = k / 128
 *
 *   x      : const fp16 [M, K] (row-major)          y : fp16 [M, N] (output)
 *   wq     : const uint32 [N, K / 8]: word w of row n holds k = 8w .. 8w+7; the code
 *            of k = 8w + 2i is bits 4i..4i+3, that of k = 8w + 2i + 1 bits
 *            4i+16..4i+19 (i = 0..3), so one shift and one mask give a pair
 *   scales : const fp16 [K / 128, N]     zeros : const uint8 [K / 128, N] (0..15)
 * Limits: 1 <= M <= 128 (decode-sized batches; the product is then bound by
 * reading the weights), N a multiple of 16, K a multiple of 256.
 * Paths: M = 1 (with K <= 65536) is a matrix-vector stream; it runs on the CUDA
 * cores (mixed-precision FMAs, fp16 products summed in fp32), one pass over K per
 * output row: n_split is ignored and no workspace is used.  Larger M runs on the
 * tensor cores (tcgen05 kind::f16, fp32 accumulation); there n_split cuts K into
 * ranges computed in parallel whose fp32 partials are summed in a fixed order
 * (the same bits on every run); n_split <= 0 selects fa_w4a16_default_splits.
 * Numerics: each weight is the fp16 rounding of (q - z) s; products accumulate in
 * fp32; Y is rounded to fp16 once.
 * Errors: FA_ERR_UNSUPPORTED for sizes outside the limits, FA_ERR_WORKSPACE when
 * a split needs fa_w4a16_workspace_size(...) bytes of workspace (256-byte
 * aligned) that were not given, FA_ERR_MISALIGNED for a tensor not 16-byte aligned.
 */
FA_API size_t fa_w4a16_workspace_size(int M, int N, int K, int n_split);
FA_API int fa_w4a16_default_splits(int M, int N, int K);
FA_API int fa_w4a16_gemm(const void* x, const void* wq, const void* scales, const void* zeros, void* y,
                         void* workspace, size_t ws_bytes, int M, int N, int K, int n_split, fa_stream_t stream);

/*
 * fa_sync_check -- synchronise `stream`, then report device-detected errors.
 * Returns FA_ERR_CUDA if the stream or a prior launch failed, FA_ERR_TIMEOUT
 * if any kernel of this library on the current device expired a bounded wait
 * since the last check (the word is then cleared), else FA_OK.
 */
FA_API int fa_sync_check(fa_stream_t stream);

/*
 * Last device error word observed by fa_sync_check on the current device:
 * 0, or 0x80000000 | site, where site names the wait that expired (role in
 * bits 8..11: 1 = TMA producer, 2 = MMA issuer, 3 = softmax/epilogue).
 */
FA_API unsigned int fa_last_error_site(void);

/*
 * Test hooks (process-wide, not thread-safe; meant for the test-suite only).
 * fa_debug_set_wait_limit_ns: deadline of every bounded in-kernel wait
 *   (default 2e9 ns).  0 restores the default.
 * fa_debug_set_fault: 0 = none; 1 = the forward kernel's TMA producer
 *   withholds K block 1 so that the MMA warp's bounded wait expires (needs
 *   N > 128).  Faults are injected on the host side of the pipeline only: no
 *   trap, no invalid address, no unbounded wait.
 */
FA_API void fa_debug_set_wait_limit_ns(unsigned long long ns);
FA_API void fa_debug_set_fault(int fault);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
