// Step 1 of the one-pass schedule: the causally masked interaction operand of
// every 128-token window, once per (batch, window, group).
//
// "Jane Street ML Engineers Map Mamba-2 Recurrent State Computation to Tensor
// Cores with cuTile", compute_out paragraph: the Q x Q matrix C B^T is built
// once by a matrix product, the positions above the diagonal are selected to
// zero, and the result multiplies the (decay-scaled) X.  Every head of a group
// reads the same Bm and Cm rows, so the masked product is the same for all of
// them: with the decay moved into per-token scales of X and of the output row
// (the one-pass kernel's rescaled form), the operand the tensor cores need is
//
//     M[i][j] = (c_i . b_j)  for j <= i,   0 for j > i        (i, j in the window)
//
// rounded to bf16.  This kernel writes M as plain row-major [i][j] rows, one
// 128 x 128 block per (batch, window, group), so that the one-pass kernel
// loads it with TMA straight into the K-major operand layout; all heads of the
// group (and both heads of every pair) then share it instead of recomputing
// C B^T per head pair.
//
// One CTA of four warps per block: TMA brings the window's C and B rows, one
// thread issues the tcgen05.mma C B^T (fp32 accumulator in tensor memory),
// each thread then owns one row i, applies the causal select in registers and
// packs bf16 pairs into a 128-byte-swizzled staging tile that two TMA stores
// write out.  Block 0 also clears the device status word and the one-pass
// kernel's run counter and per-pair flags.  Every wait is bounded.
#include "ptx.cuh"
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 128;
constexpr int kWin = 128;
constexpr uint32_t kAtom = 16384;  // 64 bf16 columns x 128 rows

__global__ void __launch_bounds__(kThreads) causal_cb_kernel(const __grid_constant__ CUtensorMap cmap,
                                                             const __grid_constant__ CUtensorMap bmap,
                                                             const __grid_constant__ CUtensorMap mmap, Dims d,
                                                             int nwin, int* status, int clear_status, int* chain,
                                                             int nchain, uint64_t spin_ns) {
  grid_dep_launch();  // the one-pass kernel may start its prologue now
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int natom = d.N / 64;
  uint8_t* sC = smem;
  uint8_t* sB = sC + natom * kAtom;
  uint8_t* sM = sB + natom * kAtom;  // two atoms: columns j in [0, 64) and [64, 128)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sM + 2 * kAtom);
  uint32_t* holder = reinterpret_cast<uint32_t*>(bars + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x;
  const int g = unit % d.G;
  const int w = (unit / d.G) % nwin;
  const int b = unit / (d.G * nwin);

  if (unit == 0) {
    if (threadIdx.x == 0 && clear_status) *status = 0;
    for (int k = threadIdx.x; k < nchain; k += kThreads) chain[k] = 0;
  }
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(holder, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *holder;
  bool ok = true;

  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bars[0], 2u * natom * kAtom);
    for (int a = 0; a < natom; ++a) {
      tma_load_4d(sC + a * kAtom, &cmap, &bars[0], a * 64, g, w * kWin, b);
      tma_load_4d(sB + a * kAtom, &bmap, &bars[0], a * 64, g, w * kWin, b);
    }
    if (!mbar_wait(&bars[0], 0, spin_ns)) {
      ok = false;
    } else {
      tc_fence_after();
      // C B^T: A = C (rows i, K = dstate), B = Bm rows (N = j, K = dstate), both K-major
      const uint32_t idesc = idesc_f32acc(1, 128, 128, 0, 0);
      const uint32_t c0 = smem_u32(sC), b0 = smem_u32(sB);
      for (int k = 0; k < d.N / 16; ++k)
        mma_ss<false>(tmem, sdesc_sw128(c0 + (k >> 2) * kAtom + (k & 3) * 32, 16, 1024),
                      sdesc_sw128(b0 + (k >> 2) * kAtom + (k & 3) * 32, 16, 1024), idesc, k != 0 ? 1u : 0u);
      mma_commit(&bars[1]);
    }
  }
  ok = __syncthreads_and(ok ? 1 : 0) != 0;
  if (ok && !mbar_wait(&bars[1], 0, spin_ns)) ok = false;
  ok = __syncthreads_and(ok ? 1 : 0) != 0;
  if (ok) {
    tc_fence_after();
    const int i = threadIdx.x;  // the row this thread owns (TMEM lane)
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
#pragma unroll 1
    for (int s = 0; s < 4; ++s) {  // 32-column strips of the 128 columns j
      uint32_t v[32];
      tmem_ld32(tmem + lane_base + 32 * s, v);
      tmem_ld_wait();
      uint8_t* row = sM + (s >> 1) * kAtom + i * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // 16-byte chunks of 8 columns
        uint4 o;
        uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = 32 * s + 8 * c + 2 * e;
          const float lo = j <= i ? __uint_as_float(v[8 * c + 2 * e]) : 0.f;
          const float hi = j + 1 <= i ? __uint_as_float(v[8 * c + 2 * e + 1]) : 0.f;
          ow[e] = pack_bf16x2(lo, hi);
        }
        const int cc = (s & 1) * 4 + c;
        *reinterpret_cast<uint4*>(row + ((cc ^ (i & 7)) << 4)) = o;
      }
    }
    fence_proxy_async_smem();
  }
  __syncthreads();
  if (ok && threadIdx.x == 0) {
    tma_store_2d(&mmap, sM, 0, unit * kWin);
    tma_store_2d(&mmap, sM + kAtom, 64, unit * kWin);
    tma_store_commit();
    tma_store_wait_all();
  }
  if (!ok && threadIdx.x == 0) atomicExch(status, static_cast<int>(SSD_ERR_DEVICE_TIMEOUT));
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
  (void)lane;
}

}  // namespace

size_t causal_cb_smem_bytes(const Dims& d) { return 1024 + 2 * (d.N / 64) * kAtom + 2 * kAtom + 64; }

cudaError_t launch_causal_cb(const Dims& d, const OnePassMaps& maps, const Work& w, uint64_t spin_ns,
                             cudaStream_t stream, bool first) {
  const int nwin = (d.L + kWin - 1) / kWin;
  const int64_t units = static_cast<int64_t>(d.B) * nwin * d.G;
  if (units <= 0 || units > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  const size_t smem = causal_cb_smem_bytes(d);
  cudaError_t e =
      cudaFuncSetAttribute(causal_cb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_k(causal_cb_kernel, dim3(static_cast<unsigned>(units)), dim3(kThreads), smem, stream, false,
                  maps.cm, maps.bm, maps.m, d, nwin, w.status, first ? 1 : 0, w.counter, first ? 1 + d.B * (d.H / 2) : 0,
                  spin_ns);
}

}  // namespace ssd
