// Step 3 of the SSD forward: carry the state across chunks.
//
// "Jane Street ML Engineers Map Mamba-2 Recurrent State Computation to Tensor
// Cores with cuTile", jump-formula and three-kernel paragraphs: fwd_pass_state
// is a sequential loop over chunks; with decay, the state after chunk c is
// exp(sum of dt*A over the chunk) times the state before it plus the chunk's
// own contribution S_c.  Here S_c comes from the chunk_state kernel, so this
// pass is pure streaming: every (b, h, p, 4 or 8 n) lane walks the chunks in order,
// reads S_c once and writes the state entering chunk c once.
//
// Memory-bound by construction (no reuse): 16-byte vector loads and stores,
// consecutive threads on consecutive n, and a software pipeline that keeps the
// next eight chunks' loads in flight while the current eight are stored.
// fp32 problems overwrite S_c with the entering state; bf16 problems read S_c
// in bf16 and write the entering state, rounded to bf16, to a separate array
// (the compute_out tensor cores read bf16 operands).  The running state is
// always fp32.
#include "ptx.cuh"
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kPrefetch = 8;

// One thread owns kVec consecutive n of one (b, h, p) row: 4 for fp32 (float4)
// and 8 for bf16 (one 16-byte load of S and one 16-byte store of the entering
// state per chunk), so every global access is 16 bytes wide.
template <bool kBF16>
struct PassVec {
  static constexpr int kVec = kBF16 ? 8 : 4;
};

template <bool kBF16>
__global__ void __launch_bounds__(kThreads) state_passing_kernel(Dims d, const float* __restrict__ cumsum,
                                                                  void* states,
                                                                  __nv_bfloat16* __restrict__ states_bf16,
                                                                  const float* __restrict__ init,
                                                                  float* __restrict__ final_state,
                                                                  float* __restrict__ hprev32) {
  constexpr int kVec = PassVec<kBF16>::kVec;
  grid_dep_wait();  // chunk_state's results are visible from here on
  grid_dep_launch();
  const int64_t pnv = static_cast<int64_t>(d.P) * d.N / kVec;  // vectors per (b, h)
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t total = static_cast<int64_t>(d.B) * d.H * pnv;
  if (gid >= total) return;
  const int64_t ev = gid % pnv;
  const int64_t bh = gid / pnv;
  const int h = static_cast<int>(bh % d.H);
  const int64_t b = bh / d.H;

  float st[kVec];
#pragma unroll
  for (int e = 0; e < kVec; ++e) st[e] = init ? init[(bh * pnv + ev) * kVec + e] : 0.f;
  const float* g_last = cumsum + bh * d.Lp + (d.Q - 1);  // cumsum at each chunk's last position
  const int64_t cstride = static_cast<int64_t>(d.H) * pnv;  // vector stride between chunks
  const int64_t base = (b * d.nc * d.H + h) * pnv + ev;     // chunk 0
  uint4* sv = reinterpret_cast<uint4*>(states);             // 16 bytes: 4 fp32 or 8 bf16

  // rounds of kPrefetch chunks; the loads of round r+1 are issued before the
  // stores of round r, so each thread always has a round of loads in flight
  uint4 cur[kPrefetch], nxt[kPrefetch];
  float dcur[kPrefetch], dnxt[kPrefetch];
  auto load_round = [&](int c0, uint4 (&v)[kPrefetch], float (&dk)[kPrefetch]) {
#pragma unroll
    for (int k = 0; k < kPrefetch; ++k) {
      if (c0 + k < d.nc) {
        v[k] = __ldcs(sv + base + (c0 + k) * cstride);
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
        const uint32_t w[4] = {cur[k].x, cur[k].y, cur[k].z, cur[k].w};
        float s_c[kVec];
        if constexpr (kBF16) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            s_c[2 * e] = __uint_as_float(w[e] << 16);
            s_c[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
          }
          if (hprev32) {  // the entering state in fp32 (the segmented one-pass schedule)
            reinterpret_cast<float4*>(hprev32)[2 * o] = make_float4(st[0], st[1], st[2], st[3]);
            reinterpret_cast<float4*>(hprev32)[2 * o + 1] = make_float4(st[4], st[5], st[6], st[7]);
          } else {
            uint4 packed;
            uint32_t* pk = &packed.x;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              __nv_bfloat162 v2 = __floats2bfloat162_rn(st[2 * e], st[2 * e + 1]);
              pk[e] = *reinterpret_cast<uint32_t*>(&v2);
            }
            reinterpret_cast<uint4*>(states_bf16)[o] = packed;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) s_c[e] = __uint_as_float(w[e]);
          sv[o] = make_uint4(__float_as_uint(st[0]), __float_as_uint(st[1]), __float_as_uint(st[2]),
                             __float_as_uint(st[3]));
        }
        const float dk = expf(dcur[k]);
#pragma unroll
        for (int e = 0; e < kVec; ++e) st[e] = fmaf(dk, st[e], s_c[e]);
      }
    }
#pragma unroll
    for (int k = 0; k < kPrefetch; ++k) {
      cur[k] = nxt[k];
      dcur[k] = dnxt[k];
    }
  }
  if (final_state) {
#pragma unroll
    for (int e = 0; e < kVec; e += 4)
      reinterpret_cast<float4*>(final_state)[((bh * pnv + ev) * kVec + e) / 4] =
          make_float4(st[e], st[e + 1], st[e + 2], st[e + 3]);
  }
}

}  // namespace

cudaError_t launch_state_passing(const Dims& d, bool bf16, const float* init, float* final_state,
                                 const Work& w, cudaStream_t stream, bool dependent, float* hprev32) {
  const int64_t total = static_cast<int64_t>(d.B) * d.H * d.P * d.N / (bf16 ? 8 : 4);
  const unsigned blocks = static_cast<unsigned>((total + kThreads - 1) / kThreads);
  const float* cs = w.cumsum;
  if (bf16)
    return launch_k(state_passing_kernel<true>, dim3(blocks), dim3(kThreads), 0, stream, dependent, d, cs, w.states,
                    w.states_bf16, init, final_state, hprev32);
  return launch_k(state_passing_kernel<false>, dim3(blocks), dim3(kThreads), 0, stream, dependent, d, cs, w.states,
                  static_cast<__nv_bfloat16*>(nullptr), init, final_state, static_cast<float*>(nullptr));
}

}  // namespace ssd
