// Step 3 of the SSD forward: carry the state across chunks.
//
// "Jane Street ML Engineers Map Mamba-2 Recurrent State Computation to Tensor
// Cores with cuTile", jump-formula and three-kernel paragraphs: fwd_pass_state
// is a sequential loop over chunks; with decay, the state after chunk c is
// exp(sum of dt*A over the chunk) times the state before it plus the chunk's
// own contribution S_c.  Here S_c comes from the chunk_state kernel, so this
// pass is pure streaming: every (b, h, p, 4 n) lane walks the chunks in order,
// reads S_c once and writes the state entering chunk c once.
//
// Memory-bound by construction (no reuse): 16-byte vector loads and stores,
// consecutive threads on consecutive n, and a software pipeline that keeps the
// next eight chunks' loads in flight while the current eight are stored.
// fp32 problems overwrite S_c with the entering state; bf16 problems write it,
// rounded to bf16, to a separate array (the compute_out tensor cores read bf16
// operands) and leave S_c in place.
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kPrefetch = 8;

template <bool kBF16>
__global__ void __launch_bounds__(kThreads) state_passing_kernel(Dims d, const float* __restrict__ cumsum,
                                                                  float* states,
                                                                  __nv_bfloat16* __restrict__ states_bf16,
                                                                  const float* __restrict__ init,
                                                                  float* __restrict__ final_state) {
  const int64_t pn4 = static_cast<int64_t>(d.P) * d.N / 4;
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t total = static_cast<int64_t>(d.B) * d.H * pn4;
  if (gid >= total) return;
  const int64_t e4 = gid % pn4;
  const int64_t bh = gid / pn4;
  const int h = static_cast<int>(bh % d.H);
  const int64_t b = bh / d.H;

  float4 st = init ? reinterpret_cast<const float4*>(init)[bh * pn4 + e4] : make_float4(0.f, 0.f, 0.f, 0.f);
  const float* g_last = cumsum + bh * d.Lp + (d.Q - 1);  // cumsum at each chunk's last position
  const int64_t cstride = static_cast<int64_t>(d.H) * pn4;  // float4 stride between chunks
  const int64_t base = (b * d.nc * d.H + h) * pn4 + e4;     // chunk 0
  float4* s4 = reinterpret_cast<float4*>(states);

  // rounds of kPrefetch chunks; the loads of round r+1 are issued before the
  // stores of round r, so each thread always has a round of loads in flight
  float4 cur[kPrefetch], nxt[kPrefetch];
  float dcur[kPrefetch], dnxt[kPrefetch];
  auto load_round = [&](int c0, float4 (&v)[kPrefetch], float (&dk)[kPrefetch]) {
#pragma unroll
    for (int k = 0; k < kPrefetch; ++k) {
      if (c0 + k < d.nc) {
        v[k] = __ldcs(s4 + base + (c0 + k) * cstride);
        dk[k] = g_last[static_cast<int64_t>(c0 + k) * d.Q];
      }
    }
  };
  load_round(0, cur, dcur);
  for (int c0 = 0; c0 < d.nc; c0 += kPrefetch) {
    if (c0 + kPrefetch < d.nc) load_round(c0 + kPrefetch, nxt, dnxt);
#pragma unroll
    for (int k = 0; k < kPrefetch; ++k) {
      if (c0 + k < d.nc) {
        const int64_t o = base + (c0 + k) * cstride;
        if constexpr (kBF16) {
          uint2 packed;
          __nv_bfloat162 lo = __floats2bfloat162_rn(st.x, st.y);
          __nv_bfloat162 hi = __floats2bfloat162_rn(st.z, st.w);
          packed.x = *reinterpret_cast<uint32_t*>(&lo);
          packed.y = *reinterpret_cast<uint32_t*>(&hi);
          reinterpret_cast<uint2*>(states_bf16)[o] = packed;
        } else {
          s4[o] = st;
        }
        const float dk = expf(dcur[k]);
        st.x = fmaf(dk, st.x, cur[k].x);
        st.y = fmaf(dk, st.y, cur[k].y);
        st.z = fmaf(dk, st.z, cur[k].z);
        st.w = fmaf(dk, st.w, cur[k].w);
      }
    }
#pragma unroll
    for (int k = 0; k < kPrefetch; ++k) {
      cur[k] = nxt[k];
      dcur[k] = dnxt[k];
    }
  }
  if (final_state) reinterpret_cast<float4*>(final_state)[bh * pn4 + e4] = st;
}

}  // namespace

cudaError_t launch_state_passing(const Dims& d, bool bf16, const float* init, float* final_state,
                                 const Work& w, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(d.B) * d.H * d.P * d.N / 4;
  const unsigned blocks = static_cast<unsigned>((total + kThreads - 1) / kThreads);
  if (bf16)
    state_passing_kernel<true><<<blocks, kThreads, 0, stream>>>(d, w.cumsum, w.states, w.states_bf16, init,
                                                                 final_state);
  else
    state_passing_kernel<false><<<blocks, kThreads, 0, stream>>>(d, w.cumsum, w.states, nullptr, init,
                                                                  final_state);
  return cudaGetLastError();
}

}  // namespace ssd
