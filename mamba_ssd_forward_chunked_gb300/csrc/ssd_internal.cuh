// Shapes, workspace pointers and kernel launchers shared by the SSD forward
// translation units (host side of the library only).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <utility>

#include "ssd.h"

namespace ssd {

// Problem sizes with everything the kernels derive from them.
struct Dims {
  int B, L, H, P, G, N, Q;
  int nc;  // chunks per sequence, ceil(L / Q)
  int Lp;  // padded length nc * Q (row length of the head-major workspace arrays)
};

// Workspace regions, as device pointers.
struct Work {
  int* status;
  float* cumsum;               // [B][H][Lp]
  float* dt_t;                 // [B][H][Lp]
  void* states;                // [B][nc][H][P][N], fp32 (fp32 inputs) or bf16 (bf16 inputs)
  __nv_bfloat16* states_bf16;  // [B][nc][H][P][N] or null (fp32 problems)
  int* counter;                // one-pass kernel: tile counter
  int* flags;                  // one-pass kernel: [B][H/2] windows published
  float* hslot;                // one-pass kernel: states at run boundaries (its own layout)
  void* cbm;                   // bf16 problems: causal C B^T per (batch, 128-token window, group), or null
};

// Tensor maps built on the host for one call.
struct ChunkStateMaps {
  CUtensorMap x;   // x viewed as [B][L][H*P], box {128 B of (h,p), 32 tokens, 1}
  CUtensorMap bm;  // Bm [B][L][G][N], box {128 B of n, 1, 32 tokens, 1}
  CUtensorMap s;   // chunk states [(B*nc*H*P)][N], box {128 B of n, 128 rows} (TMA stores)
};
struct ComputeOutMaps {
  CUtensorMap cm;  // Cm [B][L][G][N], box {128 B of n, 1, 128 tokens, 1}
  CUtensorMap bm;  // Bm, same box
  CUtensorMap hp;  // entering states [(B*nc*H*P)][N], box {128 B of n, 64 rows}
  CUtensorMap x;   // x [B][L][H*P], box {128 B of p, 128 (bf16) or 32 (fp32) tokens, 1}
  CUtensorMap y;   // y [B][L][H*P], box {128 B of p, 32 tokens, 1} (TMA stores)
};

// Tensor maps of the one-pass schedule (bf16), windows of 128 tokens.
struct OnePassMaps {
  CUtensorMap x;   // x [B][L][H*P], box {64 p, 128 tokens, 1}
  CUtensorMap cm;  // Cm [B][L][G][N], box {64 n, 1, 128 tokens, 1}
  CUtensorMap bm;  // Bm, same box
  CUtensorMap m;   // causal C B^T rows [(B*nw*G*128)][128], box {64 j, 128 rows} (stores and loads)
  CUtensorMap y;   // y [B][L][H*P], box {64 p, 128 tokens, 1} (TMA stores)
};

// Launches `kernel`; as a programmatic dependent of the preceding kernel in the
// stream when `dependent` (its launch and prologue then overlap that kernel's
// tail, and it waits in griddepcontrol.wait before reading its results).
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                     bool dependent, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

cudaError_t launch_chunk_cumsum(const Dims& d, const float* dt, const float* A, const Work& w,
                                cudaStream_t stream);
// dt non-null (Q <= 256): chunk_state forms the chunk cumsum itself and writes the cumsum and
// dt_t rows (chunk_cumsum need not run); nchain >= 0 makes it the call's first kernel, which
// clears the status word and that many one-pass counters.  dt null: it reads chunk_cumsum's rows.
cudaError_t launch_chunk_state(const Dims& d, bool bf16, const ChunkStateMaps& maps, const Work& w,
                               uint64_t spin_ns, cudaStream_t stream, bool dependent = false,
                               const float* dt = nullptr, const float* A = nullptr, int nchain = -1);
// The persistent form launch_chunk_state takes for fp32 at dstate 256 with dt non-null (Q <= 256).
cudaError_t launch_chunk_state_persistent(const Dims& d, const ChunkStateMaps& maps, const Work& w, uint64_t spin_ns,
                                          cudaStream_t stream, bool dependent, const float* dt, const float* A,
                                          int nchain);
// hprev32 (bf16 problems): write the entering states in fp32 there instead of bf16 into
// w.states_bf16 (the segmented one-pass schedule)
cudaError_t launch_state_passing(const Dims& d, bool bf16, const float* init, float* final_state,
                                 const Work& w, cudaStream_t stream, bool dependent = false,
                                 float* hprev32 = nullptr);
cudaError_t launch_compute_out(const Dims& d, bool bf16, const ComputeOutMaps& maps, const float* D,
                               const void* x, void* y, const Work& w, uint64_t spin_ns, cudaStream_t stream,
                               bool dependent = false);
// first: the call's first launch, which clears the status word and the one-pass kernel's run
// counter and flags (otherwise an earlier launch of the call has)
cudaError_t launch_causal_cb(const Dims& d, const OnePassMaps& maps, const Work& w, uint64_t spin_ns,
                             cudaStream_t stream, bool first = true);
// force_R > 0: claimed runs of force_R windows whatever the shape's own choice would be
cudaError_t launch_onepass(const Dims& d, const OnePassMaps& maps, const float* dt, const float* A, const float* D,
                           const void* x, const float* init, float* final_state, const Work& w, uint64_t spin_ns,
                           cudaStream_t stream, bool dependent = false, int force_R = 0);
cudaError_t launch_timeout_probe(int* status, uint64_t limit_ns, cudaStream_t stream);

}  // namespace ssd
