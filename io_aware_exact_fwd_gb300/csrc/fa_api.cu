// C ABI of libfa.so: argument validation, tensor-map encoding, dispatch to the
// kernels, and the device error word that bounded in-kernel waits report to.
// Declarations and the contract of every entry point: include/fa.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"

// One error word per device (a __device__ variable is instantiated on every
// device, in every context, that loads this module).  Kernels receive its
// address as a plain pointer.  That address belongs to the context that was
// current when it was looked up: a context can be replaced (cudaDeviceReset, or
// a non-primary context a host framework makes current), so it is looked up
// again on every call, with the caller's context current.
static __device__ unsigned int g_fa_error_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;

struct DeviceState {
  bool ready = false;
  int cc = 0;  // major * 10 + minor
  unsigned int last_site = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};
std::atomic<int> g_fault{0};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Per-device facts that do not change for the life of the process (compute
// capability, the tensor-map encoder) are resolved once; the error word's
// address in the current context is resolved on every call (see above) and
// returned through `err_word` when it is non-null.
int device_state(DeviceState** out, unsigned int** err_word = nullptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& s = g_dev[dev];
    if (!s.ready) {
      int major = 0, minor = 0;
      if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return FA_ERR_CUDA;
      if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return FA_ERR_CUDA;
      s.cc = major * 10 + minor;
      if (s.cc == 103 && !g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
          return FA_ERR_CUDA;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
      }
      s.ready = true;
    }
    *out = &s;
    if (s.cc != 103) return FA_ERR_UNSUPPORTED;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_fa_error_word) != cudaSuccess || !p) return FA_ERR_CUDA;
  if (err_word) *err_word = static_cast<unsigned int*>(p);
  return FA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

fa::DebugKnobs knobs() {
  fa::DebugKnobs k;
  k.wait_limit_ns = g_wait_ns.load();
  k.fault = g_fault.load();
  return k;
}

// Shared validation of the attention-shaped calls.  Returns FA_OK, a status,
// or -1 meaning "valid, but empty: nothing to do".
int validate_shape(int B, int H, int N, int d, int causal, float scale) {
  if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (B == 0 || H == 0 || N == 0) return -1;
  const long long bh = static_cast<long long>(B) * H;
  const long long nqt = (static_cast<long long>(N) + fa::kBlockQ - 1) / fa::kBlockQ;
  // Grid size (units of work) and element counts must stay inside int / TMA ranges.
  if (bh * nqt > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (bh * N > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Row, head and batch strides of a strided tensor (NULL: dense [B, H, N, d]).  Each
// must be positive and a multiple of 8 elements (16 bytes), as the tensor maps need.
int strides_or_dense(fa::Strides* out, const int64_t* s, int H, int N, int d) {
  if (!s) {
    *out = fa::dense_strides(H, N, d);
    return FA_OK;
  }
  for (int i = 0; i < 3; ++i) {
    if (s[i] <= 0 || s[i] > (int64_t(1) << 38)) return FA_ERR_INVALID_ARG;
    if (s[i] % 8 != 0) return FA_ERR_MISALIGNED;
    out->s[i] = s[i];
  }
  if (s[0] < d) return FA_ERR_INVALID_ARG;  // rows of one head may not overlap
  return FA_OK;
}

}  // namespace

namespace fa {

cudaError_t make_tmap_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int elem_bytes, int cols,
                         int rows, int depth, int box_cols, int box_rows) {
  if (!g_encode) return cudaErrorInitializationError;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(depth)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * elem_bytes,
                                 static_cast<cuuint64_t>(cols) * elem_bytes * static_cast<cuuint64_t>(rows)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int elem_bytes, int cols,
                         int rows, int64_t row_stride_elems, int box_cols, int box_rows, bool swizzle128) {
  if (!g_encode) return cudaErrorInitializationError;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t gstr[1] = {static_cast<cuuint64_t>(row_stride_elems) * elem_bytes};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, dtype, 2, const_cast<void*>(base), dims, gstr, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE,
                              swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_4d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int elem_bytes, int cols,
                         int rows, int heads, int batch, const int64_t strides[3], int box_cols, int box_rows,
                         CUtensorMapSwizzle swizzle) {
  if (!g_encode) return cudaErrorInitializationError;
  // strides: {row, head, batch} in elements; the column stride is 1.
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(batch)};
  const cuuint64_t gstr[3] = {static_cast<cuuint64_t>(strides[0]) * elem_bytes,
                              static_cast<cuuint64_t>(strides[1]) * elem_bytes,
                              static_cast<cuuint64_t>(strides[2]) * elem_bytes};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = g_encode(map, dtype, 4, const_cast<void*>(base), dims, gstr, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace fa

extern "C" {

const char* fa_strerror(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported (head dim, size or device)";
    case FA_ERR_MISALIGNED: return "misaligned pointer";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_TIMEOUT: return "kernel wait timed out";
    case FA_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

int fa_version(void) { return (0 << 16) | 1; }

int fa_fwd_strided(const void* q, const int64_t* q_strides, const void* k, const int64_t* k_strides, const void* v,
                   const int64_t* v_strides, void* o, const int64_t* o_strides, float* lse, int B, int H, int N, int d,
                   int causal, float scale, fa_stream_t stream) {
  const int vs = validate_shape(B, H, N, d, causal, scale);
  if (vs < 0) return FA_OK;
  if (vs != FA_OK) return vs;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  fa::FwdArgs a;
  int st = strides_or_dense(&a.sq, q_strides, H, N, d);
  if (st == FA_OK) st = strides_or_dense(&a.sk, k_strides, H, N, d);
  if (st == FA_OK) st = strides_or_dense(&a.sv, v_strides, H, N, d);
  if (st == FA_OK) st = strides_or_dense(&a.so, o_strides, H, N, d);
  if (st != FA_OK) return st;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return FA_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  unsigned int* ew = nullptr;
  st = device_state(&ds, &ew);
  if (st != FA_OK) return st;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.H = H;
  a.N = N;
  a.d = d;
  a.causal = causal;
  a.scale = scale;
  a.err_word = ew;
  a.dbg = knobs();
  return fa::launch_fwd_bf16(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d, int causal,
           float scale, fa_stream_t stream) {
  return fa_fwd_strided(q, nullptr, k, nullptr, v, nullptr, o, nullptr, lse, B, H, N, d, causal, scale, stream);
}

}  // extern "C"

namespace {

constexpr int kMaxSplits = 1024;

struct SplitKvLayout {
  size_t off_o, off_lse, total;
};

SplitKvLayout splitkv_layout(int B, int H, int Nq, int d, int n_split) {
  const size_t rows = static_cast<size_t>(B) * H * Nq * n_split;
  SplitKvLayout l;
  l.off_o = 0;
  l.off_lse = (rows * d * sizeof(float) + 255) & ~size_t(255);
  l.total = l.off_lse + ((rows * sizeof(float) + 255) & ~size_t(255));
  return l;
}

// Shape checks of the split-KV calls: FA_OK, a status, or -1 for "nothing to do".
int validate_splitkv(int B, int H, int Nq, int Nk, int d, int n_split, int causal, float scale) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (n_split < 1 || n_split > kMaxSplits) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (B == 0 || H == 0 || Nq == 0) return -1;
  if (Nk < 1) return FA_ERR_INVALID_ARG;
  if (causal && Nq > Nk) return FA_ERR_INVALID_ARG;
  const long long bh = static_cast<long long>(B) * H;
  const long long nunits = (static_cast<long long>(Nq) + 2 * fa::kBlockQ - 1) / (2 * fa::kBlockQ);
  if (bh * nunits * n_split > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (bh * Nq > 0x7fffffffLL || bh * Nk > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

int default_splits(int B, int H, int Nq, int Nk, int d) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                 cudaSuccess || sms < 1)
    sms = 148;
  const long long units = static_cast<long long>(B) * H * ((Nq + 2 * fa::kBlockQ - 1) / (2 * fa::kBlockQ));
  const int nkb = (Nk + fa::kBlockK - 1) / fa::kBlockK;
  // One query row runs one small CTA per (head, split), several resident per SM:
  // balance over those slots rather than over SMs.
  if (fa::decode_takes(Nq, d)) sms *= fa::decode_ctas_per_sm(d);
  // Many query rows and a full GPU: splitting would only add partials to merge.
  if (Nq > fa::kBlockQ && units >= sms) return 1;
  // Splits of at least 4 key blocks keep the per-unit Q load and epilogue small
  // next to the key stream; at most 64 keep the merge's reads small.
  const int n_max = static_cast<int>(std::min<long long>(std::max(1, nkb / 4), 64));
  // Time of the busiest SM in units of one unsplit work unit: ceil(units n / sms) / n.
  auto cost = [&](int n) { return static_cast<double>((units * n + sms - 1) / sms) / n; };
  double best = cost(1);
  for (int n = 2; n <= n_max; ++n) best = std::min(best, cost(n));
  // The fewest splits within 2 % of the best balance.
  for (int n = 1; n <= n_max; ++n)
    if (cost(n) <= best * 1.02) return n;
  return 1;
}

}  // namespace

extern "C" {

size_t fa_splitkv_workspace_size(int B, int H, int Nq, int d, int n_split) {
  if (validate_splitkv(B, H, Nq, 1, d, n_split, 0, 1.f) != FA_OK) return 0;
  return splitkv_layout(B, H, Nq, d, n_split).total;
}

int fa_splitkv_default_splits(int B, int H, int Nq, int Nk, int d) {
  if (validate_splitkv(B, H, Nq, Nk, d, 1, 0, 1.f) != FA_OK) return 0;
  return default_splits(B, H, Nq, Nk, d);
}

int fa_fwd_splitkv_partial(const void* q, const void* k, const void* v, float* o_part, float* lse_part, int B, int H,
                           int Nq, int Nk, int d, int n_split, int causal, float scale, fa_stream_t stream) {
  const int vs = validate_splitkv(B, H, Nq, Nk, d, n_split, causal, scale);
  if (vs < 0) return FA_OK;
  if (vs != FA_OK) return vs;
  if (!q || !k || !v || !o_part || !lse_part) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o_part, 16) || !aligned(lse_part, 4))
    return FA_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  unsigned int* ew = nullptr;
  const int st = device_state(&ds, &ew);
  if (st != FA_OK) return st;
  fa::SplitKvArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.sq = fa::dense_strides(H, Nq, d);
  a.sk = a.sv = fa::dense_strides(H, Nk, d);
  a.o_part = o_part;
  a.lse_part = lse_part;
  a.B = B;
  a.H = H;
  a.Nq = Nq;
  a.Nk = Nk;
  a.d = d;
  a.n_split = n_split;
  a.causal = causal;
  a.scale = scale;
  a.err_word = ew;
  a.dbg = knobs();
  return fa::launch_fwd_splitkv_partial(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK
                                                                                                   : FA_ERR_CUDA;
}

int fa_merge_partials(const float* o_part, const float* lse_part, void* o, float* lse, int n_split, int B, int H,
                      int Nq, int d, fa_stream_t stream) {
  const int vs = validate_splitkv(B, H, Nq, 1, d, n_split, 0, 1.f);
  if (vs < 0) return FA_OK;
  if (vs != FA_OK) return vs;
  if (!o_part || !lse_part || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned(o_part, 16) || !aligned(lse_part, 4) || !aligned(o, 16) || !aligned(lse, 4)) return FA_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  unsigned int* ew = nullptr;
  const int st = device_state(&ds, &ew);
  if (st != FA_OK) return st;
  fa::MergeArgs a;
  a.o_part = o_part;
  a.lse_part = lse_part;
  a.o = o;
  a.so = fa::dense_strides(H, Nq, d);
  a.lse = lse;
  a.n_split = n_split;
  a.BH = B * H;
  a.H = H;
  a.Nq = Nq;
  a.d = d;
  return fa::launch_merge_partials(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_fwd_splitkv_strided(const void* q, const int64_t* q_strides, const void* k, const int64_t* k_strides,
                           const void* v, const int64_t* v_strides, void* o, const int64_t* o_strides, float* lse,
                           void* workspace, size_t ws_bytes, int B, int H, int Nq, int Nk, int d, int n_split,
                           int causal, float scale, fa_stream_t stream) {
  if (n_split <= 0) {
    const int pre = validate_splitkv(B, H, Nq, Nk, d, 1, causal, scale);
    if (pre < 0) return FA_OK;
    if (pre != FA_OK) return pre;
    n_split = default_splits(B, H, Nq, Nk, d);
  }
  const int vs = validate_splitkv(B, H, Nq, Nk, d, n_split, causal, scale);
  if (vs < 0) return FA_OK;
  if (vs != FA_OK) return vs;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  fa::SplitKvArgs a;
  fa::MergeArgs m;
  int st = strides_or_dense(&a.sq, q_strides, H, Nq, d);
  if (st == FA_OK) st = strides_or_dense(&a.sk, k_strides, H, Nk, d);
  if (st == FA_OK) st = strides_or_dense(&a.sv, v_strides, H, Nk, d);
  if (st == FA_OK) st = strides_or_dense(&m.so, o_strides, H, Nq, d);
  if (st != FA_OK) return st;
  const SplitKvLayout lay = splitkv_layout(B, H, Nq, d, n_split);
  if (!workspace || ws_bytes < lay.total) return FA_ERR_WORKSPACE;
  if (!aligned(workspace, 256) || !aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4))
    return FA_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  unsigned int* ew = nullptr;
  st = device_state(&ds, &ew);
  if (st != FA_OK) return st;
  float* o_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + lay.off_o);
  float* lse_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + lay.off_lse);
  a.q = q;
  a.k = k;
  a.v = v;
  a.o_part = o_part;
  a.lse_part = lse_part;
  a.B = B;
  a.H = H;
  a.Nq = Nq;
  a.Nk = Nk;
  a.d = d;
  a.n_split = n_split;
  a.causal = causal;
  a.scale = scale;
  a.err_word = ew;
  a.dbg = knobs();
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (fa::launch_fwd_splitkv_partial(a, s) != cudaSuccess) return FA_ERR_CUDA;
  m.o_part = o_part;
  m.lse_part = lse_part;
  m.o = o;
  m.lse = lse;
  m.n_split = n_split;
  m.BH = B * H;
  m.H = H;
  m.Nq = Nq;
  m.d = d;
  return fa::launch_merge_partials(m, s) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace, size_t ws_bytes,
                   int B, int H, int Nq, int Nk, int d, int n_split, int causal, float scale, fa_stream_t stream) {
  return fa_fwd_splitkv_strided(q, nullptr, k, nullptr, v, nullptr, o, nullptr, lse, workspace, ws_bytes, B, H, Nq,
                                Nk, d, n_split, causal, scale, stream);
}

size_t fa_w4a16_workspace_size(int M, int N, int K, int n_split) {
  if (M < 1 || M > 128 || N < 16 || N % 16 != 0 || K < 256 || K % 256 != 0 || n_split < 1 || n_split > 1024) return 0;
  if (fa::w4a16_uses_gemv(M, K)) return 0;  // one pass over K per row: no partials
  const int cps = fa::w4a16_chunks_per_split(K, n_split);
  const int nsplit = (K / 256 + cps - 1) / cps;
  return nsplit > 1 ? static_cast<size_t>(nsplit) * M * N * sizeof(float) : 0;
}

int fa_w4a16_default_splits(int M, int N, int K) {
  if (M < 1 || M > 128 || N < 16 || N % 16 != 0 || K < 256 || K % 256 != 0) return 0;
  if (fa::w4a16_uses_gemv(M, K)) return 1;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                 cudaSuccess || sms < 1)
    sms = 148;
  const long long strips = (N + 127) / 128;
  const int kchunks = K / 256;
  // Splits of at least 4 chunks (1024 of K); the fewest within 2 % of the best
  // balance of units over the SMs (the same rule as the split-KV attention).
  const int n_max = std::max(1, std::min(kchunks / 4, 64));
  auto cost = [&](int n) {
    const int cps = (kchunks + n - 1) / n;
    const int eff = (kchunks + cps - 1) / cps;
    return static_cast<double>((strips * eff + sms - 1) / sms) * cps;
  };
  double best = cost(1);
  for (int n = 2; n <= n_max; ++n) best = std::min(best, cost(n));
  for (int n = 1; n <= n_max; ++n)
    if (cost(n) <= best * 1.02) return n;
  return 1;
}

int fa_w4a16_gemm(const void* x, const void* wq, const void* scales, const void* zeros, void* y, void* workspace,
                  size_t ws_bytes, int M, int N, int K, int n_split, fa_stream_t stream) {
  if (M < 0 || N < 0 || K < 0) return FA_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return FA_OK;
  if (M > 128 || N % 16 != 0 || K < 256 || K % 256 != 0) return FA_ERR_UNSUPPORTED;
  if (n_split <= 0) n_split = fa_w4a16_default_splits(M, N, K);
  if (n_split < 1 || n_split > 1024) return FA_ERR_INVALID_ARG;
  if (!x || !wq || !scales || !zeros || !y) return FA_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(wq, 16) || !aligned(scales, 16) || !aligned(zeros, 16) || !aligned(y, 16))
    return FA_ERR_MISALIGNED;
  const size_t need = fa_w4a16_workspace_size(M, N, K, n_split);
  if (need > 0 && (!workspace || ws_bytes < need)) return FA_ERR_WORKSPACE;
  if (need > 0 && !aligned(workspace, 256)) return FA_ERR_MISALIGNED;
  if (static_cast<long long>(N) * (K / 8) > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  DeviceState* ds = nullptr;
  unsigned int* ew = nullptr;
  const int st = device_state(&ds, &ew);
  if (st != FA_OK) return st;
  fa::W4a16Args a;
  a.x = x;
  a.wq = wq;
  a.scales = scales;
  a.zeros = zeros;
  a.y = y;
  a.partials = static_cast<float*>(workspace);
  a.M = M;
  a.N = N;
  a.K = K;
  a.n_split = n_split;
  a.err_word = ew;
  a.dbg = knobs();
  return fa::launch_w4a16(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  if (validate_shape(B, H, N, d, 0, 1.f) != FA_OK) return 0;
  return fa::bwd_workspace_layout(B, H, N, d).total;
}

}  // extern "C"

namespace {

// Which tensors a backward stage reads or writes.
enum BwdUse : unsigned {
  kUseQKV = 1u, kUseO = 2u, kUseDout = 4u, kUseLse = 8u, kUseDq = 16u, kUseDkDv = 32u,
  kNoWorkspace = 64u,  // validate everything but the workspace (its caller supplies one later)
};

// Validation shared by fa_bwd and its three stages; fills `a` on success.
int bwd_setup(fa::BwdArgs& a, unsigned use, const void* q, const void* k, const void* v, const void* o,
              const void* dout, const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
              int B, int H, int N, int d, int causal, float scale, const int64_t* const* strides = nullptr) {
  const int vs = validate_shape(B, H, N, d, causal, scale);
  if (vs < 0) return -1;
  if (vs != FA_OK) return vs;
  if (((use & kUseQKV) && (!q || !k || !v)) || ((use & kUseO) && !o) || ((use & kUseDout) && !dout) ||
      ((use & kUseLse) && !lse) || ((use & kUseDq) && !dq) || ((use & kUseDkDv) && (!dk || !dv)))
    return FA_ERR_INVALID_ARG;
  if (!(use & kNoWorkspace)) {
    if (!workspace) return FA_ERR_WORKSPACE;
    if (ws_bytes < fa::bwd_workspace_layout(B, H, N, d).total) return FA_ERR_WORKSPACE;
  }
  // strides (optional): q, k, v, o, dout, dq, dk, dv; NULL entries are dense.
  fa::Strides* dst[8] = {&a.sq, &a.sk, &a.sv, &a.so, &a.sdo, &a.sdq, &a.sdk, &a.sdv};
  for (int t = 0; t < 8; ++t) {
    const int st = strides_or_dense(dst[t], strides ? strides[t] : nullptr, H, N, d);
    if (st != FA_OK) return st;
  }
  const bool al = (!(use & kUseQKV) || (aligned(q, 16) && aligned(k, 16) && aligned(v, 16))) &&
                  (!(use & kUseO) || aligned(o, 16)) && (!(use & kUseDout) || aligned(dout, 16)) &&
                  (!(use & kUseLse) || aligned(lse, 4)) && (!(use & kUseDq) || aligned(dq, 16)) &&
                  (!(use & kUseDkDv) || (aligned(dk, 16) && aligned(dv, 16))) &&
                  ((use & kNoWorkspace) || aligned(workspace, 256));
  if (!al) return FA_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  unsigned int* ew = nullptr;
  const int st = device_state(&ds, &ew);
  if (st != FA_OK) return st;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.workspace = workspace;
  a.B = B;
  a.H = H;
  a.N = N;
  a.d = d;
  a.causal = causal;
  a.deterministic = 0;
  a.scale = scale;
  a.err_word = ew;
  a.dbg = knobs();
  return FA_OK;
}

int status_of(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

}  // namespace

namespace fa {

int bwd_validate_without_workspace(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                   const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                                   int causal, float scale) {
  BwdArgs a;
  const int st = bwd_setup(a, kUseQKV | kUseO | kUseDout | kUseLse | kUseDq | kUseDkDv | kNoWorkspace, q, k, v, o,
                           dout, lse, dq, dk, dv, nullptr, 0, B, H, N, d, causal, scale);
  return st < 0 ? FA_OK : st;
}

}  // namespace fa

extern "C" {

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse, void* dq,
           void* dk, void* dv, void* workspace, size_t ws_bytes, int B, int H, int N, int d, int causal, float scale,
           fa_stream_t stream) {
  fa::BwdArgs a;
  const int st = bwd_setup(a, kUseQKV | kUseO | kUseDout | kUseLse | kUseDq | kUseDkDv, q, k, v, o, dout, lse, dq,
                           dk, dv, workspace, ws_bytes, B, H, N, d, causal, scale);
  if (st < 0) return FA_OK;
  if (st != FA_OK) return st;
  return status_of(fa::launch_bwd_bf16(a, reinterpret_cast<cudaStream_t>(stream)));
}

int fa_bwd_strided(const void* q, const int64_t* q_strides, const void* k, const int64_t* k_strides, const void* v,
                   const int64_t* v_strides, const void* o, const int64_t* o_strides, const void* dout,
                   const int64_t* dout_strides, const float* lse, void* dq, const int64_t* dq_strides, void* dk,
                   const int64_t* dk_strides, void* dv, const int64_t* dv_strides, void* workspace, size_t ws_bytes,
                   int B, int H, int N, int d, int causal, float scale, int deterministic, fa_stream_t stream) {
  if (deterministic != 0 && deterministic != 1) return FA_ERR_INVALID_ARG;
  const int64_t* st8[8] = {q_strides, k_strides, v_strides, o_strides, dout_strides, dq_strides, dk_strides, dv_strides};
  fa::BwdArgs a;
  const int st = bwd_setup(a, kUseQKV | kUseO | kUseDout | kUseLse | kUseDq | kUseDkDv, q, k, v, o, dout, lse, dq,
                           dk, dv, workspace, ws_bytes, B, H, N, d, causal, scale, st8);
  if (st < 0) return FA_OK;
  if (st != FA_OK) return st;
  a.deterministic = deterministic;
  return status_of(fa::launch_bwd_bf16(a, reinterpret_cast<cudaStream_t>(stream)));
}

int fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const void* dout,
                         const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes, int B,
                         int H, int N, int d, int causal, float scale, fa_stream_t stream) {
  fa::BwdArgs a;
  const int st = bwd_setup(a, kUseQKV | kUseO | kUseDout | kUseLse | kUseDq | kUseDkDv, q, k, v, o, dout, lse, dq,
                           dk, dv, workspace, ws_bytes, B, H, N, d, causal, scale);
  if (st < 0) return FA_OK;
  if (st != FA_OK) return st;
  a.deterministic = 1;
  return status_of(fa::launch_bwd_bf16(a, reinterpret_cast<cudaStream_t>(stream)));
}

int fa_bwd_prep(const void* o, const void* dout, const float* lse, void* workspace, size_t ws_bytes, int B, int H,
                int N, int d, fa_stream_t stream) {
  fa::BwdArgs a;
  const int st = bwd_setup(a, kUseO | kUseDout | kUseLse, nullptr, nullptr, nullptr, o, dout, lse, nullptr, nullptr,
                           nullptr, workspace, ws_bytes, B, H, N, d, 0, 1.f);
  if (st < 0) return FA_OK;
  if (st != FA_OK) return st;
  return status_of(fa::launch_bwd_prep(a, reinterpret_cast<cudaStream_t>(stream)));
}

int fa_bwd_main(const void* q, const void* k, const void* v, const void* dout, void* dk, void* dv, void* workspace,
                size_t ws_bytes, int B, int H, int N, int d, int causal, float scale, fa_stream_t stream) {
  fa::BwdArgs a;
  const int st = bwd_setup(a, kUseQKV | kUseDout | kUseDkDv, q, k, v, nullptr, dout, nullptr, nullptr, dk, dv,
                           workspace, ws_bytes, B, H, N, d, causal, scale);
  if (st < 0) return FA_OK;
  if (st != FA_OK) return st;
  return status_of(fa::launch_bwd_main(a, reinterpret_cast<cudaStream_t>(stream)));
}

int fa_bwd_dq(const void* workspace, size_t ws_bytes, void* dq, int B, int H, int N, int d, float scale,
              fa_stream_t stream) {
  fa::BwdArgs a;
  const int st = bwd_setup(a, kUseDq, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, dq, nullptr, nullptr,
                           const_cast<void*>(workspace), ws_bytes, B, H, N, d, 0, scale);
  if (st < 0) return FA_OK;
  if (st != FA_OK) return st;
  return status_of(fa::launch_bwd_dq(a, reinterpret_cast<cudaStream_t>(stream)));
}

size_t fa_fp8_workspace_size(int B, int H, int N, int d) {
  if (validate_shape(B, H, N, d, 0, 1.f) != FA_OK) return 0;
  return fa::fp8_layout(B, H, N, d).total;
}

int fa_fp8_workspace_offsets(int B, int H, int N, int d, size_t* offsets) {
  if (!offsets) return FA_ERR_INVALID_ARG;
  const int vs = validate_shape(B, H, N, d, 0, 1.f);
  if (vs < 0) return FA_ERR_INVALID_ARG;
  if (vs != FA_OK) return vs;
  const fa::Fp8Layout l = fa::fp8_layout(B, H, N, d);
  offsets[0] = l.off_q8;
  offsets[1] = l.off_k8;
  offsets[2] = l.off_v8t;
  offsets[3] = l.off_sq;
  offsets[4] = l.off_sk;
  offsets[5] = l.off_sv;
  offsets[6] = static_cast<size_t>(l.npad);
  offsets[7] = static_cast<size_t>(l.ntiles);
  return FA_OK;
}

}  // extern "C"

namespace {

int fp8_prepare_impl(const void* q, const int64_t* q_strides, const void* k, const int64_t* k_strides, const void* v,
                     const int64_t* v_strides, int in_dtype, const int8_t* signs, uint64_t seed, void* workspace,
                     size_t ws_bytes, int B, int H, int N, int d, fa_stream_t stream) {
  const int vs = validate_shape(B, H, N, d, 0, 1.f);
  if (vs < 0) return FA_OK;
  if (vs != FA_OK) return vs;
  if (in_dtype != 0 && in_dtype != 1) return FA_ERR_INVALID_ARG;
  if (!q || !k || !v) return FA_ERR_INVALID_ARG;
  fa::Fp8PrepArgs a;
  int sst = strides_or_dense(&a.sq, q_strides, H, N, d);
  if (sst == FA_OK) sst = strides_or_dense(&a.sk, k_strides, H, N, d);
  if (sst == FA_OK) sst = strides_or_dense(&a.sv, v_strides, H, N, d);
  if (sst != FA_OK) return sst;
  if (!workspace) return FA_ERR_WORKSPACE;
  if (ws_bytes < fa::fp8_layout(B, H, N, d).total) return FA_ERR_WORKSPACE;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(workspace, 256)) return FA_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  const int st = device_state(&ds);
  if (st != FA_OK) return st;
  a.q = q;
  a.k = k;
  a.v = v;
  a.in_bf16 = in_dtype;
  a.signs = signs;
  a.seed = seed;
  a.workspace = workspace;
  a.B = B;
  a.H = H;
  a.N = N;
  a.d = d;
  return fa::launch_fp8_prepare(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

int fa_fp8_prepare(const void* q, const void* k, const void* v, int in_dtype, const int8_t* signs, void* workspace,
                   size_t ws_bytes, int B, int H, int N, int d, fa_stream_t stream) {
  if (!signs && B > 0 && H > 0 && N > 0) return FA_ERR_INVALID_ARG;
  return fp8_prepare_impl(q, nullptr, k, nullptr, v, nullptr, in_dtype, signs, 0, workspace, ws_bytes, B, H, N, d,
                          stream);
}

int fa_fp8_prepare_seeded(const void* q, const void* k, const void* v, int in_dtype, uint64_t seed, void* workspace,
                          size_t ws_bytes, int B, int H, int N, int d, fa_stream_t stream) {
  return fp8_prepare_impl(q, nullptr, k, nullptr, v, nullptr, in_dtype, nullptr, seed, workspace, ws_bytes, B, H, N,
                          d, stream);
}

int fa_fp8_prepare_strided(const void* q, const int64_t* q_strides, const void* k, const int64_t* k_strides,
                           const void* v, const int64_t* v_strides, int in_dtype, const int8_t* signs, uint64_t seed,
                           void* workspace, size_t ws_bytes, int B, int H, int N, int d, fa_stream_t stream) {
  return fp8_prepare_impl(q, q_strides, k, k_strides, v, v_strides, in_dtype, signs, seed, workspace, ws_bytes, B, H,
                          N, d, stream);
}

int fa_fp8_rotation_signs(uint64_t seed, int d, int8_t* signs) {
  if (d < 1 || !signs) return FA_ERR_INVALID_ARG;
  for (int c = 0; c < d; ++c) signs[c] = static_cast<int8_t>(fa::seeded_sign(seed, c));
  return FA_OK;
}

int fa_fwd_fp8(const void* workspace, size_t ws_bytes, void* o, float* lse, int B, int H, int N, int d, int causal,
               float scale, fa_stream_t stream) {
  const int vs = validate_shape(B, H, N, d, causal, scale);
  if (vs < 0) return FA_OK;
  if (vs != FA_OK) return vs;
  if (!o || !lse) return FA_ERR_INVALID_ARG;
  if (!workspace) return FA_ERR_WORKSPACE;
  if (ws_bytes < fa::fp8_layout(B, H, N, d).total) return FA_ERR_WORKSPACE;
  if (!aligned(o, 16) || !aligned(lse, 4) || !aligned(workspace, 256)) return FA_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  unsigned int* ew = nullptr;
  const int st = device_state(&ds, &ew);
  if (st != FA_OK) return st;
  fa::FwdArgs a{};
  a.o = o;
  a.so = fa::dense_strides(H, N, d);
  a.lse = lse;
  a.B = B;
  a.H = H;
  a.N = N;
  a.d = d;
  a.causal = causal;
  a.scale = scale;
  a.err_word = ew;
  a.dbg = knobs();
  return fa::launch_fwd_fp8(a, workspace, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK
                                                                                                  : FA_ERR_CUDA;
}

}  // extern "C"

namespace {

// Workspace of fa_bwd_fp8: the bf16 backward's workspace, then the bf16 operands
// Q', K', V' [BH, N, d], then the recomputed forward's O [BH, N, d] (bf16) and LSE
// [BH, N] (fp32); every region on a 256-byte boundary.
struct Fp8BwdLayout {
  size_t off_qr, off_kr, off_vr, off_o, off_lse, total;
};

Fp8BwdLayout fp8_bwd_layout(int B, int H, int N, int d) {
  auto a256 = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t op = a256(static_cast<size_t>(B) * H * N * d * 2);
  Fp8BwdLayout l{};
  l.off_qr = a256(fa::bwd_workspace_layout(B, H, N, d).total);
  l.off_kr = l.off_qr + op;
  l.off_vr = l.off_kr + op;
  l.off_o = l.off_vr + op;
  l.off_lse = l.off_o + op;
  l.total = l.off_lse + a256(static_cast<size_t>(B) * H * N * 4);
  return l;
}

}  // namespace

extern "C" {

int fa_fp8_dequantize(const void* fp8_ws, size_t fp8_ws_bytes, void* qr, void* kr, void* vr, int B, int H, int N,
                      int d, fa_stream_t stream) {
  const int vs = validate_shape(B, H, N, d, 0, 1.f);
  if (vs < 0) return FA_OK;
  if (vs != FA_OK) return vs;
  if (!fp8_ws) return FA_ERR_WORKSPACE;
  if (fp8_ws_bytes < fa::fp8_layout(B, H, N, d).total) return FA_ERR_WORKSPACE;
  if (!qr || !kr || !vr) return FA_ERR_INVALID_ARG;
  if (!aligned(fp8_ws, 256) || !aligned(qr, 16) || !aligned(kr, 16) || !aligned(vr, 16)) return FA_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  unsigned int* ew = nullptr;
  const int st = device_state(&ds, &ew);
  if (st != FA_OK) return st;
  return status_of(fa::launch_fp8_dequant(fp8_ws, qr, kr, vr, B, H, N, d, reinterpret_cast<cudaStream_t>(stream)));
}

size_t fa_bwd_fp8_workspace_size(int B, int H, int N, int d) {
  if (validate_shape(B, H, N, d, 0, 1.f) != FA_OK) return 0;
  return fp8_bwd_layout(B, H, N, d).total;
}

int fa_bwd_fp8(const void* fp8_ws, size_t fp8_ws_bytes, const int8_t* signs, const void* o, const void* dout,
               const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes, int B, int H, int N,
               int d, int causal, float scale, int deterministic, int recompute_forward, fa_stream_t stream) {
  if (deterministic != 0 && deterministic != 1) return FA_ERR_INVALID_ARG;
  if (recompute_forward != 0 && recompute_forward != 1) return FA_ERR_INVALID_ARG;
  const int vs = validate_shape(B, H, N, d, causal, scale);
  if (vs < 0) return FA_OK;
  if (vs != FA_OK) return vs;
  if (!fp8_ws || fp8_ws_bytes < fa::fp8_layout(B, H, N, d).total) return FA_ERR_WORKSPACE;
  if (!signs) return FA_ERR_INVALID_ARG;
  const Fp8BwdLayout l = fp8_bwd_layout(B, H, N, d);
  if (!workspace || ws_bytes < l.total) return FA_ERR_WORKSPACE;
  if (!aligned(fp8_ws, 256) || !aligned(workspace, 256)) return FA_ERR_MISALIGNED;
  char* ws = static_cast<char*>(workspace);
  void* qr = ws + l.off_qr;
  void* kr = ws + l.off_kr;
  void* vr = ws + l.off_vr;
  if (recompute_forward) {
    o = ws + l.off_o;
    lse = reinterpret_cast<const float*>(ws + l.off_lse);
  }
  // The operands carry the unnormalised rotation's factor d in Q' K'^T.
  const float op_scale = scale / static_cast<float>(d);
  fa::BwdArgs a;
  int st = bwd_setup(a, kUseQKV | kUseO | kUseDout | kUseLse | kUseDq | kUseDkDv, qr, kr, vr, o, dout, lse, dq, dk,
                     dv, workspace, ws_bytes, B, H, N, d, causal, op_scale);
  if (st < 0) return FA_OK;
  if (st != FA_OK) return st;
  a.deterministic = deterministic;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (fa::launch_fp8_dequant(fp8_ws, qr, kr, vr, B, H, N, d, s) != cudaSuccess) return FA_ERR_CUDA;
  if (recompute_forward) {
    st = fa_fwd(qr, kr, vr, const_cast<void*>(o), const_cast<float*>(lse), B, H, N, d, causal, op_scale, stream);
    if (st != FA_OK) return st;
  }
  cudaError_t e = fa::launch_bwd_bf16(a, s);
  if (e == cudaSuccess) e = fa::launch_fp8_unrotate(dq, dk, signs, static_cast<long long>(B) * H * N, d, s);
  return status_of(e);
}

int fa_sync_check(fa_stream_t stream) {
  DeviceState* ds = nullptr;
  unsigned int* ew = nullptr;
  const int st = device_state(&ds, &ew);
  if (st != FA_OK) return st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpy(&word, ew, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (word != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpy(ew, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    ds->last_site = word;
    return FA_ERR_TIMEOUT;
  }
  return FA_OK;
}

unsigned int fa_last_error_site(void) {
  DeviceState* ds = nullptr;
  if (device_state(&ds) != FA_OK || !ds) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  return ds->last_site;
}

void fa_debug_set_wait_limit_ns(unsigned long long ns) { g_wait_ns.store(ns ? ns : kDefaultWaitNs); }

void fa_debug_set_fault(int fault) { g_fault.store(fault); }

}  // extern "C"
