// Per-chunk cumsum of dt*A for one head, one warp, as chunk_cumsum and
// chunk_state both form it ("Jane Street ML Engineers Map Mamba-2 Recurrent
// State Computation to Tensor Cores with cuTile", three-kernel paragraph:
// log-space cumulative sums of dt*A within each chunk).  Both kernels call the
// same function, so the values match bit for bit whichever one writes them.
#pragma once

namespace ssd {

// One piece of 32 * per tokens (per <= kMax): lane l holds v[k] = dt of token
// l * per + k.  On return g[k] = carry + the sum of dt*A over the piece's
// tokens up to and including that one, and carry has grown by the piece's
// total.  Each lane runs its tokens serially, then a warp-shuffle scan adds
// the earlier lanes' totals; the exclusive part is the previous lane's
// inclusive sum (not the inclusive sum minus the lane's own), so every G_t is
// formed from tokens <= t only and later tokens cannot change it, even by
// rounding.
template <int kMax>
__device__ __forceinline__ void cumsum_piece(const float (&v)[kMax], int per, float a, float& carry,
                                             float (&g)[kMax]) {
  const int lane = threadIdx.x & 31;
  float run[kMax];
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < kMax; ++k) {
    if (k < per) {
      acc += v[k] * a;
      run[k] = acc;
    }
  }
  float incl = acc;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float u = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += u;
  }
  float excl = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) excl = 0.f;
#pragma unroll
  for (int k = 0; k < kMax; ++k)
    if (k < per) g[k] = run[k] + excl + carry;
  carry += __shfl_sync(0xffffffffu, incl, 31);
}

}  // namespace ssd
