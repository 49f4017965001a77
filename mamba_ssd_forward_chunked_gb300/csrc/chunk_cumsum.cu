// Step 1 of the SSD forward: per-chunk log-space cumsum of the decay term.
//
// "Jane Street ML Engineers Map Mamba-2 Recurrent State Computation to Tensor
// Cores with cuTile", three-kernel paragraph: chunk_cumsum computes per-token,
// per-head cumulative sums of dt*A within each chunk and stores them for the
// two kernels after it; the Blackwell paragraph moves them (and dt) from the
// strided [batch, token, head] layout to [batch, head, token] so that the
// consumers read contiguous rows with TMA or vector loads.
//
// One block per (chunk, batch, 8-head slice): the work is a few MB in total, so
// the grid is made wide (many small blocks) and every load of a block is issued
// before any is used.  A block reads its Q x 8 slice of dt ([B][L][H]: 32
// contiguous bytes per token), transposes it through shared memory, scans each
// head's Q values with one warp (serial runs per lane + a warp-shuffle scan of
// the run totals) and writes cumsum and dt as contiguous [B][H][Lp] rows.
// Tokens past L read as dt = 0, so the cumsum stays flat in a ragged last chunk.
// The staged schedule's chunk_state forms the same rows itself (chunk_scan.cuh);
// this kernel serves the segmented schedule's segments and the step-by-step API.
#include "chunk_scan.cuh"
#include "ptx.cuh"
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kHeadsPerBlock = 8;
constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) chunk_cumsum_kernel(Dims d, const float* __restrict__ dt,
                                                                 const float* __restrict__ A,
                                                                 float* __restrict__ cumsum,
                                                                 float* __restrict__ dt_t, int* status,
                                                                 int* chain, int nchain) {
  __shared__ float s_dt[kHeadsPerBlock * 257];
  __shared__ float s_g[kHeadsPerBlock * 257];
  grid_dep_launch();  // the next kernel may start its prologue while this one runs
  const int blk = blockIdx.x;
  const int Q = d.Q;
  // a chunk longer than 256 tokens (the one-pass schedule's segments) goes in pieces of 256,
  // the running sum carried from piece to piece
  const int P0 = Q < 256 ? Q : 256;
  const int ld = P0 + 1;  // odd row stride: the transposing writes hit distinct banks
  const int hslices = (d.H + kHeadsPerBlock - 1) / kHeadsPerBlock;
  const int c = blk % d.nc;
  const int h0 = (blk / d.nc) % hslices * kHeadsPerBlock;
  const int b = blk / (d.nc * hslices);
  if (blk == 0) {
    if (threadIdx.x == 0) *status = 0;
    for (int k = threadIdx.x; k < nchain; k += kThreads) chain[k] = 0;  // one-pass kernel's counter and flags
  }

  const int lane = threadIdx.x & 31, hh = threadIdx.x >> 5;  // one warp per head
  const int h = h0 + hh;
  const float a_h = h < d.H ? A[h] : 0.f;
  const int per = P0 / 32;  // 2, 4 or 8 tokens per lane
  float carry = 0.f;        // sum of the chunk's earlier pieces
  // a piece's loads (P0 * 8 / 256 <= 8 per thread); the next piece's go out before this one is
  // scanned
  auto load_piece = [&](int t0, float (&v)[8]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int idx = threadIdx.x + k * kThreads;
      const int t = idx / kHeadsPerBlock, h2 = h0 + idx % kHeadsPerBlock;
      const int tok = t0 + t;
      v[k] = (t < P0 && tok < d.L && h2 < d.H) ? dt[(static_cast<int64_t>(b) * d.L + tok) * d.H + h2] : 0.f;
    }
  };
  float vn[8];
  load_piece(c * Q, vn);
  for (int t0 = c * Q; t0 < (c + 1) * Q; t0 += P0) {
    float v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = vn[k];
    if (t0 + P0 < (c + 1) * Q) load_piece(t0 + P0, vn);
    __syncthreads();  // the previous piece's shared-memory reads are done
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int idx = threadIdx.x + k * kThreads;
      const int t = idx / kHeadsPerBlock, hs = idx % kHeadsPerBlock;
      if (t < P0) s_dt[hs * ld + t] = v[k];
    }
    __syncthreads();

    float dv[8], g[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) dv[k] = k < per ? s_dt[hh * ld + lane * per + k] : 0.f;
    cumsum_piece(dv, per, a_h, carry, g);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (k < per) s_g[hh * ld + lane * per + k] = g[k];
    __syncthreads();

    for (int idx = threadIdx.x; idx < kHeadsPerBlock * P0; idx += kThreads) {
      const int hq = idx / P0, t = idx % P0;
      if (h0 + hq < d.H) {
        const int64_t o = (static_cast<int64_t>(b) * d.H + h0 + hq) * d.Lp + t0 + t;
        cumsum[o] = s_g[hq * ld + t];
        dt_t[o] = s_dt[hq * ld + t];
      }
    }
  }
}

}  // namespace

cudaError_t launch_chunk_cumsum(const Dims& d, const float* dt, const float* A, const Work& w,
                                cudaStream_t stream) {
  const int64_t ncum = static_cast<int64_t>(d.nc) * ((d.H + kHeadsPerBlock - 1) / kHeadsPerBlock) * d.B;
  if (ncum > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  chunk_cumsum_kernel<<<static_cast<unsigned>(ncum), kThreads, 0, stream>>>(
      d, dt, A, w.cumsum, w.dt_t, w.status, w.counter, 1 + d.B * (d.H / 2));
  return cudaGetLastError();
}

}  // namespace ssd
