// Step 1 of the SSD forward: per-chunk log-space cumsum of the decay term.
//
// "Jane Street ML Engineers Map Mamba-2 Recurrent State Computation to Tensor
// Cores with cuTile", three-kernel paragraph: chunk_cumsum computes per-token,
// per-head cumulative sums of dt*A within each chunk and stores them for the
// two kernels after it; the Blackwell paragraph moves them (and dt) from the
// strided [batch, token, head] layout to [batch, head, token] so that the
// consumers read contiguous rows with TMA or vector loads.
//
// One block per (chunk, batch, 32-head slice).  dt arrives as [B][L][H]: a
// block reads its Q x 32 slice row by row (128 contiguous bytes per token),
// transposes it through shared memory, scans each head's Q values with one
// warp (serial runs per lane + a warp-shuffle scan of the run totals) and
// writes cumsum and dt as contiguous [B][H][Lp] rows.  Tokens past L read as
// dt = 0, so the cumsum stays flat in a ragged last chunk.
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kHeadsPerBlock = 32;
constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) chunk_cumsum_kernel(Dims d, const float* __restrict__ dt,
                                                                 const float* __restrict__ A,
                                                                 float* __restrict__ cumsum,
                                                                 float* __restrict__ dt_t, int* status) {
  extern __shared__ float sm[];
  const int Q = d.Q;
  const int ld = Q + 1;  // odd row stride: the transposing writes hit distinct banks
  float* s_dt = sm;
  float* s_g = sm + kHeadsPerBlock * ld;
  const int c = blockIdx.x;
  const int h0 = blockIdx.y * kHeadsPerBlock;
  const int b = blockIdx.z;
  if (c == 0 && blockIdx.y == 0 && b == 0 && threadIdx.x == 0) *status = 0;

  for (int idx = threadIdx.x; idx < Q * kHeadsPerBlock; idx += kThreads) {
    const int t = idx / kHeadsPerBlock, hh = idx % kHeadsPerBlock;
    const int tok = c * Q + t, h = h0 + hh;
    float v = 0.f;
    if (tok < d.L && h < d.H) v = dt[(static_cast<int64_t>(b) * d.L + tok) * d.H + h];
    s_dt[hh * ld + t] = v;
  }
  __syncthreads();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = Q / 32;  // 2, 4 or 8 tokens per lane
  for (int hh = warp; hh < kHeadsPerBlock; hh += kThreads / 32) {
    const int h = h0 + hh;
    const float a_h = h < d.H ? A[h] : 0.f;
    float run[8];
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (k < per) {
        acc += s_dt[hh * ld + lane * per + k] * a_h;
        run[k] = acc;
      }
    }
    float incl = acc;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    const float excl = incl - acc;
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (k < per) s_g[hh * ld + lane * per + k] = run[k] + excl;
  }
  __syncthreads();

  for (int idx = threadIdx.x; idx < kHeadsPerBlock * Q; idx += kThreads) {
    const int hh = idx / Q, t = idx % Q;
    const int h = h0 + hh;
    if (h < d.H) {
      const int64_t o = (static_cast<int64_t>(b) * d.H + h) * d.Lp + static_cast<int64_t>(c) * Q + t;
      cumsum[o] = s_g[hh * ld + t];
      dt_t[o] = s_dt[hh * ld + t];
    }
  }
}

}  // namespace

cudaError_t launch_chunk_cumsum(const Dims& d, const float* dt, const float* A, const Work& w,
                                cudaStream_t stream) {
  const dim3 grid(d.nc, (d.H + kHeadsPerBlock - 1) / kHeadsPerBlock, d.B);
  const size_t smem = 2u * kHeadsPerBlock * (d.Q + 1) * sizeof(float);
  static size_t configured = 0;
  if (smem > configured) {  // above 48 KB (chunk_size 256) the opt-in limit must be raised
    cudaError_t e = cudaFuncSetAttribute(chunk_cumsum_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  chunk_cumsum_kernel<<<grid, kThreads, smem, stream>>>(d, dt, A, w.cumsum, w.dt_t, w.status);
  return cudaGetLastError();
}

}  // namespace ssd
