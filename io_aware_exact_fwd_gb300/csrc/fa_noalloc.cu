// fa_bwd_noalloc: the backward pass for callers that cannot allocate device
// memory themselves, using a fixed scratch buffer owned by this library.
//
// fa_bwd needs a caller-provided workspace (an fp32 dQ accumulator plus two
// per-row vectors).  Some callers have no way to provide one: code running as a
// plugin inside a host framework that owns all device memory and hands plugins
// no allocator, or latency-critical loops in which a cudaMalloc (which may
// synchronise the whole device) is not allowed.  For them this file keeps one
// scratch buffer per device in a file-scope __device__ array and passes its
// address to the unchanged fa_bwd.
//
// In host code the array's name is a host-side stand-in, not a device address.
// Its device address is looked up with cudaGetSymbolAddress on every call, with
// the caller's device and context current: the address belongs to the context
// that was current at the lookup, and a context can be replaced during the
// life of the process (cudaDeviceReset, or a host framework that makes its own
// context current), so a cached address could point into a context that no
// longer exists.  The lookup is a table search inside the CUDA runtime.
#include <cuda_runtime.h>

#include "fa.h"
#include "fa_internal.h"

namespace {

// Largest workspace the no-allocation path can serve: 64 MiB per device.  The
// array is part of this library's device code: it is reserved on a device when
// the module is loaded into a context there (with lazy module loading, the
// default, at the first call of this file on that device; with eager loading,
// when any context is created while the library is loaded) and held until that
// context is destroyed or the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array in the current context.
int noalloc_scratch(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FA_ERR_CUDA;
  *out = p;
  return FA_OK;
}

}  // namespace

extern "C" {

size_t fa_bwd_noalloc_max_workspace(void) { return kNoAllocScratchBytes; }

int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                   void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale,
                   fa_stream_t stream) {
  // Every argument check of fa_bwd other than the workspace comes first, so that a
  // bad call returns fa_bwd's status without touching (or loading) the scratch.
  const int st = fa::bwd_validate_without_workspace(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, causal, scale);
  if (st != FA_OK) return st;
  const size_t need = fa_bwd_workspace_size(B, H, N, d);
  if (need == 0) return FA_OK;  // sizes already validated: an empty problem
  if (need > kNoAllocScratchBytes) return FA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int sst = noalloc_scratch(&scratch);
  if (sst != FA_OK) return sst;
  return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, scratch, kNoAllocScratchBytes, B, H, N, d, causal, scale,
                stream);
}

}  // extern "C"
