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
// The array is a host-side stand-in in host code, not a device address, so its
// device address is looked up with cudaGetSymbolAddress, once per device, with
// that device current, on the first call made on that device.
#include <cuda_runtime.h>

#include <mutex>

#include "fa.h"

namespace {

// Largest workspace the no-allocation path can serve: 64 MiB per device.  Every
// GPU that loads this library holds the array until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return FA_ERR_CUDA;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return FA_OK;
}

}  // namespace

extern "C" {

size_t fa_bwd_noalloc_max_workspace(void) { return kNoAllocScratchBytes; }

int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                   void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale,
                   fa_stream_t stream) {
  const size_t need = fa_bwd_workspace_size(B, H, N, d);
  if (need == 0)  // empty, invalid or unsupported sizes: fa_bwd reports which, touching no workspace
    return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, nullptr, 0, B, H, N, d, causal, scale, stream);
  if (need > kNoAllocScratchBytes) return FA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int st = noalloc_scratch(&scratch);
  if (st != FA_OK) return st;
  return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, scratch, kNoAllocScratchBytes, B, H, N, d, causal, scale,
                stream);
}

}  // extern "C"
