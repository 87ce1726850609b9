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

struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, H, N, d;
  int causal;
  float scale;
  unsigned int* err_word;
  DebugKnobs dbg;
};

// Forward launcher (fa_fwd.cu).  Returns a cudaError_t.
cudaError_t launch_fwd_bf16(const FwdArgs& a, cudaStream_t stream);

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
  void* workspace;
  int B, H, N, d;
  int causal;
  float scale;
  unsigned int* err_word;
  DebugKnobs dbg;
};

// Workspace of the backward: fp32 dQ accumulator [BH, N, d], then D and
// LSE * log2(e), each [BH, npad] with npad = N rounded up to 64.  Every region
// starts on a 256-byte boundary.
struct BwdWorkspace {
  size_t off_dq, off_d, off_lse2, total;
  int npad;
};
BwdWorkspace bwd_workspace_layout(int B, int H, int N, int d);

// Backward launchers (fa_bwd.cu).  launch_bwd_bf16 = prep, main, dq in order on
// `stream`; each stage reads only the BwdArgs fields it needs.
cudaError_t launch_bwd_prep(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_main(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_bf16(const BwdArgs& a, cudaStream_t stream);

// Encodes a 3-D tiled tensor map over a [BH, N, cols] row-major tensor with
// `elem_bytes`-byte elements, box {box_cols, box_rows, 1}, 128-byte swizzle.
// Implemented in fa_api.cu (driver entry point resolved once).
cudaError_t make_tmap_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int elem_bytes,
                         int cols, int rows, int depth, int box_cols, int box_rows);

}  // namespace fa
