// Step 2 of the one-pass schedule: chunk state, state passing and output in
// one persistent kernel (bf16 inputs, fp32 accumulation), every window of 128
// tokens of a (batch, head pair) in flight behind the one before it.
//
// What it computes ("Jane Street ML Engineers Map Mamba-2 Recurrent State
// Computation to Tensor Cores with cuTile", jump-formula, three-kernel and
// compute_out paragraphs).  For a window of S = 128 tokens of head h, with G
// the cumulative sum of dt*A from the window start (G_i includes token i) and
// h_in the state entering the window:
//
//     y_i   = sum_{j<=i} (c_i . b_j) e^{G_i - G_j} dt_j x_j + e^{G_i} c_i h_in^T + D x_i
//     h_out = e^{G_S} h_in + sum_j e^{G_S - G_j} dt_j x_j b_j^T
//
// i.e. the jump formula with decay applied window by window; any split into
// windows gives the recurrence's result.
//
// Rescaled form (window start as reference).  With r_i = e^{G_i} (<= 1) and
// X^_j = e^{-G_j} dt_j x_j:
//
//     y_i   = r_i [ sum_{j<=i} M_ij X^_j + c_i h_in^T ] + D x_i,   M_ij = (c_i . b_j) [j <= i]
//     h_out = e^{G_S} (h_in + X^^T B)
//
// M is the causal select of C B^T alone: the same for every head of a group,
// so the causal_cb kernel computes it once per (batch, window, group) and this
// kernel loads it.  The intra product and the carried-state product share one
// fp32 accumulator, and y_i at token i reads G only up to token i (the masked
// entries of M are exact zeros), so y is causal to the last bit.  The form
// needs e^{-G_S} within fp32 range: it is used while the window's decay -G_S
// stays below 2^100 on both heads of the pair.  Otherwise the window takes an
// exact path: X is scaled against the window END instead
// (X~_j = e^{G_S - G_j} dt_j x_j <= dt_j x_j), the intra product is not run,
// and the epilogue sums (c_i . b_j) e^{G_i - G_j} dt_j x_j on CUDA cores with
// one exponential per element (exponent <= 0).
//
// The state.  Thread (head, p) of the state pass owns row (head, p) of the
// pair's running state, and the window's state product X^^T B (resp. X~^T B)
// comes from the tensor core with lane = (head, p) and columns = dstate.
//  - dstate <= 128 (product buffers): the row lives in the thread's registers
//    (fp32).  S(n) writes the window's product fresh into tensor-memory buffer
//    n % 2; the pass reads it, h_out = e^{G_S} (h_in + X^^T B) (resp.
//    e^{G_S} h_in + X~^T B), frees the buffer and writes the bf16 copy O of
//    h_out that the next window's carried-state product reads.  S(n + 1) waits
//    for nothing of the pass of window n, so the only hand-off between windows
//    is O.
//  - dstate 256 (state in tensor memory): the row does not fit in registers,
//    so the state is an fp32 accumulator in tensor memory.  Before a window's
//    state product it holds pi * h_in (pi = 1 on the rescaled form, e^{G_S} on
//    the exact one), the product is accumulated onto it, and the pass reads it
//    back, scales it by mu (e^{G_S}, resp. 1) to get h_out, writes pi' * h_out
//    back and hands it over; only then does it write O.  The serial chain
//    between windows is one state product and the tensor-memory half of one
//    pass.
//
// Runs and chaining.  Windows go out in runs (consecutive windows of one
// sequence, i.e. one (batch, head pair)), either claimed from a global counter
// or split statically between the CTAs (see the schedule warp below).  A run's
// last window publishes its state (fp32, L2-resident workspace slot) and a
// per-pair flag; the next run's first window waits for the flag (bounded) and
// loads it.  A sequence's first window reads init_state (or zero) and its last
// writes final_state.
//
// GB300 mapping, per CTA (one per SM, 512 threads, persistent):
//   warp 2       the schedule: publishes the CTA's windows in an 8-deep ring.
//   warp 0       TMA: a ring of 32 KB stages holding, per window in the order
//                the tensor core uses them, B, M (the causal operand) and C
//                (C before M at dstate 256).
//   warp 1       owns tensor memory and issues every tcgen05.mma from one
//                thread, per window n: the state product S(n) once X^ is
//                scaled (and its product buffer read, resp. the state handed
//                over), then the intra product M X^ and, once O(n) is written,
//                the carried product C O(n)^T (at dstate 256 the carried
//                product first, since the pass writes O for the first 128
//                columns before the hand-off).
//   warp 3       TMA for the head pair's X window (three buffers; two at
//                dstate 256): stores window n - 3's y out of a buffer, then
//                loads window n's X into it.
//   warps 4-7    the state pass: thread = state row (head, p).
//   warps 8-15   one warpgroup per head, thread = token row: the window's
//                cumsum (warp-shuffle scan of dt*A), the X scaling (in place)
//                with D x_i / r_i put into the output accumulator as its
//                starting value, and the epilogue of the window before
//                (y = r_i acc written over X).
// The control warps give registers to the state pass and the head warpgroups
// (setmaxnreg).  Tensor memory: two output accumulators (columns [0, 256)) and
// two product buffers of 128 columns, resp. the state (columns [256, 512)).
// The kernel is compiled per dstate (64, 128, 256).  Every wait is bounded; on expiry the
// CTA records SSD_ERR_DEVICE_TIMEOUT, waits for its own copies and exits.
#include "ptx.cuh"
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 512;
constexpr int kWin = 128;
constexpr int kInfoRing = 8;
constexpr float kSpan = 100.f;  // log2 bound of the window decay for the rescaled form
constexpr uint32_t kStage = 32768, kAtom = 16384, kXBytes = 32768;
constexpr uint32_t kColY = 0, kColH = 256, kTmemCols = 512;

// Register split between the warpgroups (setmaxnreg): the CTA is launched with
// kRegLaunch per thread; the control warpgroup (one active lane per warp) gives
// registers up, the state warpgroup, which holds the running state row (dstate
// <= 128) or a window's bf16 state copy across the hand-off (dstate 256), and
// the two head warpgroups take them.
// The split must stay within the launch's pool (an increase that cannot be met
// waits without end), which the host checks against the compiled register count
// before every launch.
constexpr uint32_t kRegLaunch = 128, kRegCtl = 48, kRegState = 176, kRegHead = 144;
static_assert(128 * (kRegCtl + kRegState + 2 * kRegHead) <= kThreads * kRegLaunch, "register split above the pool");

// Asynchronous prefetch of a contiguous global range into L2 (16-byte aligned, size a
// multiple of 16).
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

template <uint32_t kRegs>
__device__ __forceinline__ void regs_release() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs));
}
template <uint32_t kRegs>
__device__ __forceinline__ void regs_acquire() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs));
}

struct WinInfo {
  int b, pair, w;  // batch, head pair, window index in the sequence
  int flags;       // bit 0: first window of its run, bit 1: last, bit 2: no more windows
};
// Per-window scalars the head warpgroups publish (slot n % 2, with the X buffer).
struct Scal {
  float alpha[2];  // e^{G_S} per head
  int fast[2];     // rescaled form valid for the head
};

struct OPSmem {
  uint32_t ring, xbuf, obuf, info, scal, scan, bars, holder, total;
  int stages, nob, nxb;
};

// Shared memory: three stages of 32 KB (M; B and C in ceil(N/128) stages each),
// X buffers of 32 KB (three up to dstate 128, two at 256), the carried-state
// operand O (bf16 [2*P rows][N] in 64-column atoms), and the small control data.
__host__ __device__ inline OPSmem op_layout(int N) {
  OPSmem s{};
  const uint32_t obytes = static_cast<uint32_t>(N / 64) * kAtom;
  s.nob = 1;
  s.nxb = N <= 128 ? 3 : 2;
  s.stages = 3;
  s.ring = 0;
  s.xbuf = s.ring + s.stages * kStage;
  s.obuf = s.xbuf + s.nxb * kXBytes;
  s.info = s.obuf + s.nob * obytes;
  s.scal = s.info + kInfoRing * sizeof(WinInfo);
  s.scan = s.scal + 3 * sizeof(Scal);
  s.bars = s.scan + 2 * 2 * 4 * sizeof(float);
  s.holder = s.bars + 48 * 8;
  s.total = s.holder + 16;
  return s;
}

// Scaled pair, clamped below bf16's largest finite value: an overflowing
// product must not become inf, which the causal select's zeros would turn
// into NaN in rows that never see that token.
__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t v, float s) {
  constexpr float kMax = 3.38e38f;
  return pack_bf16x2(fminf(fmaxf(bf16_lo(v) * s, -kMax), kMax), fminf(fmaxf(bf16_hi(v) * s, -kMax), kMax));
}

// Inclusive sum over the 128 threads of a warpgroup in token order; each
// result adds only values of threads at or before it.  `total` is the sum of
// all 128, formed the same way by every thread (and equal to thread 127's
// result).  `ws` holds four floats of the warpgroup.
__device__ __forceinline__ float wg_scan(float v, float* ws, uint32_t bar, int lane, int wq, float& total) {
  float incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float u = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += u;
  }
  if (lane == 31) ws[wq] = incl;
  named_bar_sync(bar, 128);
  float pre = 0.f, tot = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (k < wq) pre += ws[k];
    tot += ws[k];
  }
  total = tot;
  return wq == 0 ? incl : pre + incl;
}

// Exact epilogue of a window off the rescaled form, for token row i of head h:
// the accumulator at `tacc` (64 columns) holds c_i h_in^T (carried state,
// unscaled), and
//   y_i = e^{G_i} acc + sum_{j<=i} M_ij e^{G_i - G_j} dt_j x_j + D x_i
// with M read from the causal_cb output, x and dt from global memory and G
// summed again along the row.  Rare (a window decaying by more than 2^100)
// and slow; done in two halves of 32 columns to keep its registers few (it is
// inlined: a call would make the compiler keep the hot loop's values in local
// memory around it).
__device__ __forceinline__ void exact_epilogue(const Dims& d, int b, int h, int t0, int i, float gi, float Ah,
                                               float Dh, const __nv_bfloat16* __restrict__ Mrow,
                                               const __nv_bfloat16* __restrict__ xg, const float* __restrict__ dtg,
                                               uint32_t tacc, uint8_t* xr) {
  const float ei = fast_exp2(gi);
  const bool in_seq = t0 + i < d.L;
  const uint4* xi = reinterpret_cast<const uint4*>(xg + ((static_cast<int64_t>(b) * d.L + t0 + i) * d.H + h) * d.P);
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    uint32_t ya[32];
    tmem_ld32(tacc + 32 * half, ya);
    tmem_ld_wait();
    float acc[32];
#pragma unroll
    for (int q = 0; q < 32; ++q) acc[q] = 0.f;
    float G = 0.f;
    for (int j = 0; j <= i && t0 + j < d.L; ++j) {
      const float dtj = dtg[(static_cast<int64_t>(b) * d.L + t0 + j) * d.H + h];
      G += dtj * Ah;
      const float coef = __bfloat162float(Mrow[j]) * fast_exp2(fminf(gi - G * kLog2e, 0.f)) * dtj;
      const uint4* xj =
          reinterpret_cast<const uint4*>(xg + ((static_cast<int64_t>(b) * d.L + t0 + j) * d.H + h) * d.P) + 4 * half;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 xv = __ldg(xj + c);
        const uint32_t* xw = reinterpret_cast<const uint32_t*>(&xv);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[8 * c + 2 * e] = fmaf(coef, bf16_lo(xw[e]), acc[8 * c + 2 * e]);
          acc[8 * c + 2 * e + 1] = fmaf(coef, bf16_hi(xw[e]), acc[8 * c + 2 * e + 1]);
        }
      }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 xv = in_seq ? __ldg(xi + 4 * half + c) : make_uint4(0, 0, 0, 0);
      const uint32_t* xw = reinterpret_cast<const uint32_t*>(&xv);
      uint4 v;
      uint32_t* vw = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int pi = 8 * c + 2 * e;
        vw[e] = pack_bf16x2(fmaf(Dh, bf16_lo(xw[e]), fmaf(ei, __uint_as_float(ya[pi]), acc[pi])),
                            fmaf(Dh, bf16_hi(xw[e]), fmaf(ei, __uint_as_float(ya[pi + 1]), acc[pi + 1])));
      }
      const int cc = 4 * half + c;
      *reinterpret_cast<uint4*>(xr + ((cc ^ (i & 7)) << 4)) = v;
    }
  }
}

// A head-warpgroup thread's view of one window.
struct Ctx {
  int b, pair, w;
  float g;   // log2 cumsum at this token (window start = 0)
  float dt;  // dt at this token (0 past the sequence)
  float a;   // A_h
  float dd;  // D_h
  int fastH; // rescaled form valid for this head
};

template <int kN>
__global__ void __launch_bounds__(kThreads, 1)
    ssd_onepass_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap cmap,
                       const __grid_constant__ CUtensorMap bmap, const __grid_constant__ CUtensorMap mmap,
                       const __grid_constant__ CUtensorMap ymap, Dims d, int R, const float* __restrict__ dtg,
                       const float* __restrict__ Avec, const float* __restrict__ Dvec,
                       const __nv_bfloat16* __restrict__ Mg, const float* init, float* final_state, float* hslot,
                       int* flags, int* counter, const __nv_bfloat16* __restrict__ xg, int* status,
                       uint64_t spin_ns) {
  constexpr bool kPB = kN <= 128;  // product buffers (else the state accumulated in tensor memory)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const OPSmem Ls = op_layout(d.N);
  const int natom = d.N / 64;           // 64-column atoms of dstate
  const int nhalf = (d.N + 127) / 128;  // 128-column halves (stages) of B and C
  const int nxb = Ls.nxb;
  const int hp = d.H / 2;
  const int nw = (d.L + kWin - 1) / kWin;
  // Window n of this CTA uses X buffer (and scalar slot) n % nxb and output accumulator n % 2.
  auto xs = [&](int n) { return n % nxb; };
  auto xph = [&](int n) { return static_cast<uint32_t>((n / nxb) & 1); };
  auto yph = [](int n) { return static_cast<uint32_t>((n >> 1) & 1); };
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Ls.bars);
  uint64_t* full = bars;          // [3] ring stage landed
  uint64_t* empty = bars + 3;     // [3] ring stage consumed (MMA commit)
  uint64_t* xfull = bars + 6;     // [3] X window landed
  // [3] X scaled and window scalars published (256); with product buffers also the pass's read
  // of the product two windows back (+128), so the state product's buffer is free
  uint64_t* xready = bars + 9;
  uint64_t* ystaged = bars + 12;  // [3] y written into the X buffer (256: both head warpgroups)
  uint64_t* tfull = bars + 15;    // [8] window ring
  uint64_t* tempty = bars + 23;   // [8] (14 warps read each entry)
  uint64_t* sready = bars + 31;   // [2] state in tensor memory: pi h_in of the window in place (128)
  uint64_t* dfull = bars + 33;    // [2] state product done (X^ of the window read)
  // [2] carried-state product done: O free; with product buffers (carried product last) also
  // the output accumulator complete
  uint64_t* cdone = bars + 35;
  uint64_t* oready = bars + 39;   // [2] O (bf16 h_in) of the window in place (128)
  uint64_t* ydone = bars + 41;    // [2] state in tensor memory: output accumulator complete
  WinInfo* info = reinterpret_cast<WinInfo*>(smem + Ls.info);
  Scal* scal = reinterpret_cast<Scal*>(smem + Ls.scal);
  float* scanws = reinterpret_cast<float*>(smem + Ls.scan);  // [2 heads][2 windows][4]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Ls.holder);
  // The CTA's number of windows, once the schedule knows it (INT_MAX until then): the tensor-core
  // thread reads it instead of the window ring.
  volatile int* nwin_s = reinterpret_cast<volatile int*>(smem + Ls.holder + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 3; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&xfull[s], 1);
      mbar_init(&xready[s], kPB ? 384 : 256);
      mbar_init(&ystaged[s], 256);
    }
    for (int s = 0; s < kInfoRing; ++s) {
      mbar_init(&tfull[s], 1);
      mbar_init(&tempty[s], 14);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sready[s], 128);
      mbar_init(&oready[s], 128);
      mbar_init(&ydone[s], 1);
      mbar_init(&dfull[s], 1);
      mbar_init(&cdone[s], 1);
    }
    *nwin_s = 0x7fffffff;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&xmap);
    tma_prefetch_desc(&cmap);
    tma_prefetch_desc(&bmap);
    tma_prefetch_desc(&mmap);
    tma_prefetch_desc(&ymap);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  // No griddepcontrol.wait here: what the pre-pass writes (the causal blocks, the cleared
  // status word, counter and flags) is waited for by each role just before its first use, so
  // the first X windows and init_state prefetches go out while the pre-pass finishes.
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  bool ok = true;

  // the window ring entry n, read by a whole warp; lane 0 frees the entry
  auto read_info = [&](int n, WinInfo& I) -> bool {
    const int ts = n % kInfoRing;
    bool good = true;
    if (lane == 0) good = mbar_wait_short(&tfull[ts], (n / kInfoRing) & 1, spin_ns);
    good = __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
    if (!good) return false;
    I = info[ts];
    __syncwarp();
    if (lane == 0) mbar_arrive(&tempty[ts]);
    return true;
  };
  // the same, for a warp of which only lane 0 runs
  auto read_info1 = [&](int n, WinInfo& I) -> bool {
    const int ts = n % kInfoRing;
    if (!mbar_wait_short(&tfull[ts], (n / kInfoRing) & 1, spin_ns)) return false;
    I = info[ts];
    mbar_arrive(&tempty[ts]);
    return true;
  };

  if (warp < 4) {
  regs_release<kRegCtl>();
  if (warp == 2) {
    // ------------------------------------------------------------ schedule
    // Windows go out in runs: consecutive windows of one sequence (batch, head pair).  Two
    // schedules (R = run length, 0 for the static one):
    //  - claims: runs of R windows taken from a global counter in run-major order (all first
    //    runs, then all second runs, ...), so a run's predecessor was claimed earlier by a
    //    running CTA; a faster CTA takes more runs.
    //  - static: the CTA's share of the list of all windows, sequence by sequence,
    //    [c T / P, (c + 1) T / P) for T windows and P CTAs, as runs in this order: the first
    //    windows of the sequence that crosses the share's end (published for the next CTA),
    //    the whole sequences inside, and the rest of the sequence that crosses the share's
    //    start (resumed from the previous CTA).  With P at most the number of sequences a share
    //    holds at least one sequence's windows, so the previous CTA, which starts with that
    //    sequence's first windows, has published them before this CTA gets to the rest.  Every
    //    CTA gets the same number of windows (+-1), where claims of R windows may leave some
    //    CTAs a whole run more than others.  The list orders sequences by (pair within its
    //    group, batch, group), so the CTAs c + k P / Q run a group's Q pairs side by side.
    if (lane == 0) {
      int n = 0;
      bool good = true;
      // windows [w0, w1) of sequence (b, pair) into the ring; flags bit 0 / 1 = first / last
      // of the run, bit 2 = end marker
      auto put = [&](int b, int pair, int w0, int w1, int fl) {
        // a sequence's first window starts from init_state: bring the pair's block into L2
        // now, while the window waits in the ring behind the ones before it
        if (w0 == 0 && fl == 0 && init)
          prefetch_l2_bulk(init + (static_cast<int64_t>(b) * d.H + 2 * pair) * d.P * d.N,
                           static_cast<uint32_t>(2 * d.P * d.N * sizeof(float)));
        for (int w = w0; good && w < w1; ++w, ++n) {
          const int ts = n % kInfoRing;
          if (n >= kInfoRing && !mbar_wait_short(&tempty[ts], ((n / kInfoRing) - 1) & 1, spin_ns)) {
            good = false;
            break;
          }
          WinInfo I;
          I.b = b;
          I.pair = pair;
          I.w = w;
          I.flags = fl | (w == w0 ? 1 : 0) | (w == w1 - 1 ? 2 : 0);
          info[ts] = I;
          mbar_arrive(&tfull[ts]);
        }
      };
      if (R > 0) {
        grid_dep_wait();  // the counter is cleared by the pre-pass
        const int nruns = ((nw + R - 1) / R) * d.B * hp;
        for (;;) {
          const int run = atomicAdd(counter, 1);
          if (run >= nruns || !good) break;
          const int w0 = run / hp / d.B * R;
          put((run / hp) % d.B, run % hp, w0, min(nw, w0 + R), 0);
        }
      } else {
        const int64_t total = static_cast<int64_t>(d.B) * hp * nw;
        const int64_t lo = static_cast<int64_t>(blockIdx.x) * total / gridDim.x;
        const int64_t hi = static_cast<int64_t>(blockIdx.x + 1) * total / gridDim.x;
        const int s_lo = static_cast<int>(lo / nw), w_lo = static_cast<int>(lo % nw);
        const int s_hi = static_cast<int>(hi / nw), w_hi = static_cast<int>(hi % nw);
        const int Q = hp / d.G, nbg = d.B * d.G;  // pairs per group; (batch, group) combinations
        const int head = w_hi > 0 ? 1 : 0, tail = w_lo > 0 ? 1 : 0;
        const int first_full = s_lo + tail, nfull = s_hi - first_full;
        for (int k = 0; good && k < head + nfull + tail; ++k) {
          // run k: windows [w0, w1) of list entry sq
          const int sq = k < head ? s_hi : k < head + nfull ? first_full + k - head : s_lo;
          const int w0 = k < head + nfull ? 0 : w_lo, w1 = k < head ? w_hi : nw;
          const int q = sq / nbg, bg = sq % nbg;
          put(bg / d.G, (bg % d.G) * Q + q, w0, w1, 0);
        }
      }
      *nwin_s = n;         // for the tensor-core thread
      put(0, 0, 0, 1, 4);  // the end marker
      ok = good;
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ X loads and y stores
    // Window n's X goes into buffer n % nxb once window n - nxb's y has left it.
    if (lane == 0) {
      int hb[3] = {0, 0, 0}, ht[3] = {0, 0, 0}, hh0[3] = {0, 0, 0};  // batch, t0, h0 of each buffer's window
      auto store = [&](int k) -> bool {  // window k's y, written over its X
        const int sb = xs(k);
        if (!mbar_wait_short(&ystaged[sb], xph(k), spin_ns)) return false;
        uint8_t* xb = smem + Ls.xbuf + sb * kXBytes;
        tma_store_3d(&ymap, xb, hh0[sb] * d.P, ht[sb], hb[sb]);
        tma_store_3d(&ymap, xb + kWin * 128, (hh0[sb] + 1) * d.P, ht[sb], hb[sb]);
        tma_store_commit();
        return true;
      };
      int n = 0;
      for (; ok; ++n) {
        WinInfo I;
        if (!read_info1(n, I)) {
          ok = false;
          break;
        }
        if (I.flags & 4) break;
        const int sb = xs(n);
        if (n >= nxb) {
          if (!store(n - nxb)) {
            ok = false;
            break;
          }
          tma_store_wait_read();
        }
        hb[sb] = I.b;
        ht[sb] = I.w * kWin;
        hh0[sb] = 2 * I.pair;
        uint8_t* xb = smem + Ls.xbuf + sb * kXBytes;
        mbar_arrive_expect_tx(&xfull[sb], kXBytes);
        tma_load_3d(xb, &xmap, &xfull[sb], hh0[sb] * d.P, ht[sb], I.b);
        tma_load_3d(xb + kWin * 128, &xmap, &xfull[sb], (hh0[sb] + 1) * d.P, ht[sb], I.b);
      }
      // the last windows' y
      for (int k = max(0, n - nxb); ok && k < n; ++k)
        if (!store(k)) ok = false;
      tma_store_wait_all();
      // on a timeout: wait (bounded) for the X copies still in flight before the CTA exits
      if (!ok)
        for (int k = max(0, n - nxb); k <= n; ++k) mbar_wait_short(&xfull[xs(k)], xph(k), spin_ns);
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producer: the ring
    // Per window, in the order the tensor core consumes them: B (state product) by 128-column
    // halves, then M (intra product) and C (carried-state product, by halves); at dstate 256
    // C comes before M.
    if (lane == 0) {
      int it = 0;
      for (int n = 0; ok; ++n) {
        WinInfo I;
        if (!read_info1(n, I)) {
          ok = false;
          break;
        }
        if (I.flags & 4) break;
        const int h0 = 2 * I.pair, g = h0 / (d.H / d.G), t0 = I.w * kWin;
        const int nitems = 1 + 2 * nhalf;
        for (int q = 0; q < nitems && ok; ++q, ++it) {
          const int s = it % Ls.stages, rnd = it / Ls.stages;
          // With product buffers each item has its own stage, and B's and C's are free once the
          // state (resp. carried) product of the window before has completed, which dfull (cdone)
          // already signals; M's stage, and every stage at dstate 256, has its own commit (empty).
          bool free_stage = true;
          if (rnd > 0) {
            if (kPB && q == 0)
              free_stage = mbar_wait_short(&dfull[(n - 1) & 1], yph(n - 1), spin_ns);
            else if (kPB && q == 2)
              free_stage = mbar_wait_short(&cdone[(n - 1) & 1], yph(n - 1), spin_ns);
            else
              free_stage = mbar_wait_short(&empty[s], (rnd - 1) & 1, spin_ns);
          }
          if (!free_stage) {
            ok = false;
            break;
          }
          uint8_t* st = smem + Ls.ring + s * kStage;
          const int qm = d.N > 128 ? 2 * nhalf : nhalf;  // M after C at dstate 256, before it otherwise
          if (q == qm) {
            if (n == 0) grid_dep_wait();  // the causal blocks come from the pre-pass
            mbar_arrive_expect_tx(&full[s], 2 * kAtom);
            const int row = ((I.b * nw + I.w) * d.G + g) * kWin;
            tma_load_2d(st, &mmap, &full[s], 0, row);
            tma_load_2d(st + kAtom, &mmap, &full[s], 64, row);
          } else {
            const bool isC = q >= nhalf && q != qm;
            const int hf = !isC ? q : q - nhalf - (q > qm ? 1 : 0);
            const int na = min(2, natom - 2 * hf);
            mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(na) * kAtom);
            for (int a = 0; a < na; ++a)
              tma_load_4d(st + a * kAtom, isC ? &cmap : &bmap, &full[s], hf * 128 + a * 64, g, t0, I.b);
          }
        }
      }
      // on a timeout: wait (bounded) for the copies still in flight before the CTA exits
      if (!ok)
        for (int k = max(0, it - Ls.stages); k < it; ++k) mbar_wait_short(&full[k % Ls.stages], (k / Ls.stages) & 1, spin_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Per window n: the state product S(n) as soon as the state is in place (the serial chain
    // between windows is S(n) and the pass over its result), then the intra product and,
    // once O(n) is in place, the carried-state product C O(n)^T; both run during the pass.
    if (lane == 0) {
      const uint32_t id_st = idesc_f32acc(1, 128, d.N < 128 ? d.N : 128, 1, 1);  // X^ pair^T x B (MN / MN)
      const uint32_t id_in = idesc_f32acc(1, 128, 128, 0, 1);  // M (K-major) x X^ pair (MN-major)
      const uint32_t id_yo = idesc_f32acc(1, 128, 128, 0, 0);  // C x O (both K-major)
      const uint32_t xlbo = kWin * 128;                         // head stride in the X buffer
      const uint32_t ob = smem_u32(smem + Ls.obuf);
      const bool c_first = d.N > 128;  // carried product before the intra product (see below)
      int it = 0;
      auto stage = [&](int i) -> uint32_t {
        const int s = i % Ls.stages;
        if (!mbar_wait_short(&full[s], (i / Ls.stages) & 1, spin_ns)) return 0u;
        return smem_u32(smem + Ls.ring + s * kStage);
      };
      auto release = [&](int i) { mma_commit(&empty[i % Ls.stages]); };
      for (int n = 0; ok; ++n) {
        const int yb = n & 1;
        // S(n) once X^ is scaled: into product buffer n % 2 (xready(n) also says that the pass
        // has read window n - 2's product from it), or accumulated onto the state once pi h_in
        // is in place (sready).  Window n exists unless the schedule has published fewer
        // windows; that count is read only while xready(n) is still open.
        bool have = true;
        if (!mbar_try_wait_short(&xready[xs(n)], xph(n))) {
          const uint64_t t0w = globaltimer_ns();
          for (;;) {
            if (mbar_try_wait_short(&xready[xs(n)], xph(n))) break;
            if (n >= *nwin_s) {
              have = false;
              break;
            }
            if (globaltimer_ns() - t0w > spin_ns) {
              ok = false;
              break;
            }
          }
        }
        if (!ok || !have) break;
        if (!kPB && !mbar_wait_short(&sready[yb], yph(n), spin_ns)) {
          ok = false;
          break;
        }
        const bool fast = scal[xs(n)].fast[0] && scal[xs(n)].fast[1];
        const uint32_t xb = smem_u32(smem + Ls.xbuf + xs(n) * kXBytes);
        for (int hf = 0; hf < nhalf && ok; ++hf) {
          const uint32_t sb = stage(it);
          if (!sb) {
            ok = false;
            break;
          }
          tc_fence_after();
          // 16 tokens per MMA: both MN-major operands advance by 16 rows (2048 bytes)
          const uint64_t da = sdesc_sw128(xb, xlbo, 1024), db = sdesc_sw128(sb, kAtom, 1024);
          const uint32_t dst = tmem + kColH + 128 * (kPB ? yb : hf);
#pragma unroll 1
          for (int k = 0; k < kWin / 16; ++k)
            mma_ss<false>(dst, da + k * (2048 >> 4), db + k * (2048 >> 4), id_st, (kPB && k == 0) ? 0u : 1u);
          if constexpr (!kPB) release(it);  // product buffers: dfull frees B's stage
          ++it;
        }
        if (!ok) break;
        mma_commit(&dfull[yb]);
        // The intra and carried products into output accumulator n % 2.  Window n - 2's output
        // has been drained from it: the head warpgroups' epilogue of window n - 2 comes before
        // their X scaling of window n, which xready(n) waited for.  Up to dstate 128 the intra
        // product goes first; at dstate 256 the carried product does, so that O(n) is free
        // early: the pass writes O for the first 128 columns before it hands the state over.
        auto intra = [&]() -> bool {
          const uint32_t sm = stage(it);
          if (!sm) return false;
          tc_fence_after();
          if (fast) {
            // 16 tokens j per MMA: M (K-major, 64-column atoms) advances 32 bytes within an atom,
            // X^ (MN-major) by 16 rows
            const uint64_t da = sdesc_sw128(sm, 16, 1024), db = sdesc_sw128(xb, xlbo, 1024);
#pragma unroll 1
            for (int k = 0; k < kWin / 16; ++k)
              mma_ss<false>(tmem + kColY + 128 * yb, da + (k >> 2) * (kAtom >> 4) + (k & 3) * 2, db + k * (2048 >> 4),
                            id_in, 1u);
          }
          release(it++);
          return true;
        };
        // carried state: output += C O(n)^T over dstate, once O(n) is in place
        auto carried = [&]() -> bool {
          if (!mbar_wait_short(&oready[yb], yph(n), spin_ns)) return false;
          for (int hf = 0; hf < nhalf; ++hf) {
            const uint32_t sc = stage(it);
            if (!sc) return false;
            tc_fence_after();
            // 16 dstate columns per MMA: C and O (both K-major, 64-column atoms) advance 32 bytes
            // within an atom
            const int na = min(2, natom - 2 * hf);
            const uint64_t da = sdesc_sw128(sc, 16, 1024), db = sdesc_sw128(ob + 2 * hf * kAtom, 16, 1024);
#pragma unroll 1
            for (int k = 0; k < 4 * na; ++k) {
              const uint32_t off = (k >> 2) * (kAtom >> 4) + (k & 3) * 2;
              mma_ss<false>(tmem + kColY + 128 * yb, da + off, db + off, id_yo, (fast || hf != 0 || k != 0) ? 1u : 0u);
            }
            if constexpr (!kPB) release(it);  // product buffers: cdone frees C's stage
            ++it;
          }
          mma_commit(&cdone[yb]);
          return true;
        };
        if (c_first ? !(carried() && intra()) : !(intra() && carried())) {
          ok = false;
          break;
        }
        if constexpr (!kPB) mma_commit(&ydone[yb]);  // product buffers: cdone, the last commit
      }
    }
  }
  } else if (warp < 8) {
    regs_acquire<kRegState>();
    if constexpr (kPB) {
      // windows 0 and 1 have no product two windows back to read
      mbar_arrive(&xready[xs(0)]);
      mbar_arrive(&xready[xs(1)]);
    }
    grid_dep_wait();  // the flags are cleared by the pre-pass
    // ------------------------------------------------------------ state pass
    const int et = threadIdx.x - 128;  // TMEM lane = state row (head hd, p)
    const int quad = warp & 3;
    const int hd = et >> 6, p = et & 63;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tH = tmem + lane_base + kColH;
    constexpr uint32_t bar_s = 1;
    uint8_t* orow = smem + Ls.obuf + et * 128;  // this row of O in each 64-column atom
    // O as bf16 chunks of one 32-column strip
    auto put_o = [&](int n0, const uint32_t* hb) {
      const float* h = reinterpret_cast<const float*>(hb);
      uint8_t* oat = orow + (n0 >> 6) * kAtom;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint4 o;
        o.x = pack_bf16x2(h[8 * c], h[8 * c + 1]);
        o.y = pack_bf16x2(h[8 * c + 2], h[8 * c + 3]);
        o.z = pack_bf16x2(h[8 * c + 4], h[8 * c + 5]);
        o.w = pack_bf16x2(h[8 * c + 6], h[8 * c + 7]);
        const int cc = ((n0 & 63) >> 3) + c;
        *reinterpret_cast<uint4*>(oat + ((cc ^ (et & 7)) << 4)) = o;
      }
    };
    // before writing O for window m: the carried product of window m - 1 is done
    auto o_free = [&](int m) -> bool { return m < 1 || mbar_wait_short(&cdone[(m - 1) & 1], yph(m - 1), spin_ns); };
    // the window's scalars: alpha = e^{G_S} and the rescaled-form flag of this head
    float alpha = 1.f;
    bool fastH = true;
    if constexpr (kPB) {
    // Product buffers (dstate <= 128).  The running state row h (head, p) stays in registers;
    // S(n) writes X^^T B (X~^T B) fresh into tensor-memory buffer n % 2, and the pass adds it:
    //   h_out = e^{G_S} (h_in + X^^T B)   (rescaled form),   e^{G_S} h_in + X~^T B   (exact).
    // The pass frees the buffer as soon as it has read it, so S(n + 1) never waits for the pass
    // of window n: the only hand-off left between windows is O, the bf16 copy of h that the
    // next window's carried product reads.
    float hs[kN];
    // O = h in bf16 for the columns [0, N)
    auto put_all_o = [&]() {
#pragma unroll
      for (int c = 0; c < kN / 8; ++c) {  // 16-byte chunk c: columns 8c .. 8c + 7
        uint4 o;
        o.x = pack_bf16x2(hs[8 * c], hs[8 * c + 1]);
        o.y = pack_bf16x2(hs[8 * c + 2], hs[8 * c + 3]);
        o.z = pack_bf16x2(hs[8 * c + 4], hs[8 * c + 5]);
        o.w = pack_bf16x2(hs[8 * c + 6], hs[8 * c + 7]);
        *reinterpret_cast<uint4*>(orow + (c >> 3) * kAtom + (((c & 7) ^ (et & 7)) << 4)) = o;
      }
    };
    for (int n = 0; ok; ++n) {
      WinInfo I;
      if (named_bar_or(bar_s, 128, !read_info(n, I))) {
        ok = false;
        break;
      }
      if (I.flags & 4) break;
      const int yb = n & 1;
      const bool first = I.flags & 1, last = I.flags & 2;
      const int h = 2 * I.pair + hd;
      const int64_t hrow = ((static_cast<int64_t>(I.b) * d.H + h) * d.P + p) * d.N;  // [B][H][P][N]
      float4* slot = reinterpret_cast<float4*>(hslot + (static_cast<int64_t>(I.b) * hp + I.pair) * 128 * d.N) + et;
      const bool seq_first = I.w == 0, seq_last = I.w == nw - 1;
      if (first) {
        // the state entering the run: the predecessor's slot (float4 k of the row at
        // slot[k * 128]), init_state (prefetched into L2 when the run was published) or zero;
        // O = h_in
        bool bad = !mbar_wait_short(&xready[xs(n)], xph(n), spin_ns) || !o_free(n);
        if (!seq_first && et == 0) bad = bad || !wait_flag_geq(flags + I.b * hp + I.pair, I.w, spin_ns);
        if (named_bar_or(bar_s, 128, bad)) {
          ok = false;
          break;
        }
        alpha = scal[xs(n)].alpha[hd];
        fastH = scal[xs(n)].fast[hd] != 0;
        const float* hin = seq_first ? (init ? init + hrow : nullptr) : nullptr;
        if (seq_first && !hin) {
#pragma unroll
          for (int q = 0; q < kN; ++q) hs[q] = 0.f;
        } else {
          const float4* src0 = seq_first ? reinterpret_cast<const float4*>(hin) : slot;
          const int stride = seq_first ? 1 : 128;
#pragma unroll
          for (int k = 0; k < kN / 4; ++k) {
            const float4 h4 = __ldcg(src0 + k * stride);
            hs[4 * k] = h4.x;
            hs[4 * k + 1] = h4.y;
            hs[4 * k + 2] = h4.z;
            hs[4 * k + 3] = h4.w;
          }
        }
        put_all_o();
        fence_proxy_async_smem();
        mbar_arrive(&oready[yb]);
      }
      // the pass: h_out from h_in and window n's product, in 32-column strips
      if (named_bar_or(bar_s, 128, !mbar_wait_short(&dfull[yb], yph(n), spin_ns))) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        const float beta = fastH ? alpha : 1.f;
        const uint32_t tP = tmem + lane_base + kColH + 128 * yb;
#pragma unroll
        for (int n0 = 0; n0 < kN; n0 += 32) {  // two 16-column loads in flight
          uint32_t v[16], u[16];
          tmem_ld16(tP + n0, v);
          tmem_ld16(tP + n0 + 16, u);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 16; ++q) hs[n0 + q] = fmaf(alpha, hs[n0 + q], beta * __uint_as_float(v[q]));
#pragma unroll
          for (int q = 0; q < 16; ++q) hs[n0 + 16 + q] = fmaf(alpha, hs[n0 + 16 + q], beta * __uint_as_float(u[q]));
        }
      }
      tc_fence_before();
      mbar_arrive(&xready[xs(n + 2)]);  // product buffer n % 2 is free for S(n + 2)
      if (last) {
        // publish: the slot for the run that continues this sequence, or final_state
        if (!seq_last) {
#pragma unroll
          for (int k = 0; k < kN / 4; ++k)
            __stcg(slot + k * 128, make_float4(hs[4 * k], hs[4 * k + 1], hs[4 * k + 2], hs[4 * k + 3]));
          __threadfence();
          named_bar_sync(bar_s, 128);
          if (et == 0) st_release_gpu(flags + I.b * hp + I.pair, I.w + 1);
        } else if (final_state) {
#pragma unroll
          for (int k = 0; k < kN / 4; ++k)
            reinterpret_cast<float4*>(final_state + hrow)[k] =
                make_float4(hs[4 * k], hs[4 * k + 1], hs[4 * k + 2], hs[4 * k + 3]);
        }
      } else {
        // the next window's scalars, then O(n + 1) = h_out once the carried product of window
        // n has read O(n)
        if (named_bar_or(bar_s, 128,
                         !mbar_wait_short(&xready[xs(n + 1)], xph(n + 1), spin_ns) || !o_free(n + 1))) {
          ok = false;
          break;
        }
        alpha = scal[xs(n + 1)].alpha[hd];
        fastH = scal[xs(n + 1)].fast[hd] != 0;
        put_all_o();
        fence_proxy_async_smem();
        mbar_arrive(&oready[(n + 1) & 1]);
      }
    }
    } else {
    for (int n = 0; ok; ++n) {
      WinInfo I;
      if (named_bar_or(bar_s, 128, !read_info(n, I))) {
        ok = false;
        break;
      }
      if (I.flags & 4) break;
      const int yb = n & 1;
      const bool first = I.flags & 1, last = I.flags & 2;
      const int h = 2 * I.pair + hd;
      const int64_t hrow = ((static_cast<int64_t>(I.b) * d.H + h) * d.P + p) * d.N;  // [B][H][P][N]
      float4* slot = reinterpret_cast<float4*>(hslot + (static_cast<int64_t>(I.b) * hp + I.pair) * 128 * d.N) + et;
      const bool seq_first = I.w == 0, seq_last = I.w == nw - 1;
      if (first) {
        // the state entering the run: predecessor's slot, init_state or zero, put in place
        // as pi * h_in with O = h_in
        bool bad = !mbar_wait_short(&xready[xs(n)], xph(n), spin_ns) || !o_free(n);
        if (!seq_first && et == 0) bad = bad || !wait_flag_geq(flags + I.b * hp + I.pair, I.w, spin_ns);
        if (named_bar_or(bar_s, 128, bad)) {
          ok = false;
          break;
        }
        alpha = scal[xs(n)].alpha[hd];
        fastH = scal[xs(n)].fast[hd] != 0;
        const float* hin = seq_first ? (init ? init + hrow : nullptr) : nullptr;
        const float pre = fastH ? 1.f : alpha;
        // The entering state: the predecessor's slot ([16-column group][row] float4s),
        // init_state (the row's columns in order, prefetched into L2 when the schedule
        // published the run) or zero.  A rolled loop over 64 columns: 16 loads in flight per
        // L2 round trip, and little code, since this path runs once per run and its code is
        // never in the instruction cache.
        const bool zero = seq_first && !hin;
        const float4* src0 = seq_first ? reinterpret_cast<const float4*>(hin) : slot;
        const int step = seq_first ? 8 : 8 * 128, stride = seq_first ? 1 : 128;
#pragma unroll 1
        for (int n0 = 0; n0 < d.N; n0 += 64) {
          uint32_t hb[64];
          if (zero) {
#pragma unroll
            for (int q = 0; q < 64; ++q) hb[q] = 0u;
          } else {
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const float4 h4 = __ldcg(src0 + (n0 >> 5) * step + (q >> 3) * step + (q & 7) * stride);
              hb[4 * q] = __float_as_uint(h4.x);
              hb[4 * q + 1] = __float_as_uint(h4.y);
              hb[4 * q + 2] = __float_as_uint(h4.z);
              hb[4 * q + 3] = __float_as_uint(h4.w);
            }
          }
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t* hh = hb + 32 * half;
            put_o(n0 + 32 * half, hh);  // O = h_in
#pragma unroll
            for (int q = 0; q < 32; ++q) hh[q] = __float_as_uint(pre * __uint_as_float(hh[q]));
            tmem_st32(tH + n0 + 32 * half, *reinterpret_cast<uint32_t(*)[32]>(hh));
          }
        }
        tmem_st_wait();
        tc_fence_before();
        fence_proxy_async_smem();
        mbar_arrive(&sready[yb]);
        mbar_arrive(&oready[yb]);
      }
      // The pass over window n's state, h_out = mu * (pi h_in + X^T B), as soon as the state
      // product is done.  The state for the next window goes back into tensor memory first and
      // is handed over (sready); the bf16 copy O of the last (up to 128) columns, which only
      // the carried product reads, is kept in registers and written after the hand-off, once
      // the carried product of window n has read O(n).  At dstate 256 the first 128 columns
      // write O inside the loop.
      {
        if (named_bar_or(bar_s, 128, !mbar_wait_short(&dfull[yb], yph(n), spin_ns))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float mu = fastH ? alpha : 1.f;
        const int ndef0 = d.N > 128 ? d.N - 128 : 0;  // first column of the deferred O block
        bool ofree = last;                            // O(n + 1) may be written (no O after a run's last window)
        // one 32-column strip scaled: h = mu * v; on a run's last window, publish it
        auto scale_publish = [&](int n0, uint32_t (&v)[32]) {
#pragma unroll
          for (int q = 0; q < 32; ++q) v[q] = __float_as_uint(mu * __uint_as_float(v[q]));
          if (!last) return;
          const float* hv = reinterpret_cast<const float*>(v);
          if (!seq_last) {  // for the run that continues this sequence
#pragma unroll
            for (int q = 0; q < 8; ++q)
              __stcg(slot + ((n0 >> 5) * 8 + q) * 128, make_float4(hv[4 * q], hv[4 * q + 1], hv[4 * q + 2], hv[4 * q + 3]));
          } else if (final_state) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              reinterpret_cast<float4*>(final_state + hrow + n0)[q] =
                  make_float4(hv[4 * q], hv[4 * q + 1], hv[4 * q + 2], hv[4 * q + 3]);
          }
        };
        // strips in pairs, both loads in flight at once: tensor-memory loads issued while the
        // MMAs run take a few hundred ns each, so fewer round trips matter more than overlap
        // (65,536-token sweep point L2048-N128: 512 against 530 us for one load in flight)
        uint32_t va[32], vb[32];
#pragma unroll 1
        for (int n0 = 0; n0 < ndef0; n0 += 64) {  // dstate 256: columns 0..127
          tmem_ld32(tH + n0, va);
          tmem_ld32(tH + n0 + 32, vb);
          tmem_ld_wait();
          scale_publish(n0, va);
          scale_publish(n0 + 32, vb);
          if (!last) {
            tmem_st32(tH + n0, va);
            tmem_st32(tH + n0 + 32, vb);
            if (!ofree) {
              if (named_bar_or(bar_s, 128, !o_free(n + 1))) {
                ok = false;
                break;
              }
              ofree = true;
            }
            put_o(n0, va);
            put_o(n0 + 32, vb);
          }
        }
        if (!ok) break;
        uint32_t pk[64];  // bf16 pairs of the deferred columns ndef0 .. ndef0 + 127
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int n0 = ndef0 + 64 * k;
          if (n0 < d.N) {
            tmem_ld32(tH + n0, va);
            tmem_ld32(tH + n0 + 32, vb);
            tmem_ld_wait();
            scale_publish(n0, va);
            scale_publish(n0 + 32, vb);
            if (!last) {
              tmem_st32(tH + n0, va);
              tmem_st32(tH + n0 + 32, vb);
#pragma unroll
              for (int q = 0; q < 16; ++q) {
                pk[32 * k + q] = pack_bf16x2(__uint_as_float(va[2 * q]), __uint_as_float(va[2 * q + 1]));
                pk[32 * k + 16 + q] = pack_bf16x2(__uint_as_float(vb[2 * q]), __uint_as_float(vb[2 * q + 1]));
              }
            }
          }
        }
        if (!last) {
          tmem_st_wait();
          // the next window's scalars (its X scaled); on the exact form the state it
          // accumulates onto is e^{G_S} h_in, so rescale (rare)
          if (named_bar_or(bar_s, 128, !mbar_wait_short(&xready[xs(n + 1)], xph(n + 1), spin_ns))) {
            ok = false;
            break;
          }
          alpha = scal[xs(n + 1)].alpha[hd];
          fastH = scal[xs(n + 1)].fast[hd] != 0;
          if (!fastH) {
#pragma unroll 1
            for (int n0 = 0; n0 < d.N; n0 += 32) {
              tmem_ld32(tH + n0, va);
              tmem_ld_wait();
#pragma unroll
              for (int q = 0; q < 32; ++q) va[q] = __float_as_uint(alpha * __uint_as_float(va[q]));
              tmem_st32(tH + n0, va);
            }
            tmem_st_wait();
          }
          tc_fence_before();
          mbar_arrive(&sready[(n + 1) & 1]);
          // O(n + 1) = h_out in bf16, once the carried product of window n has read O(n)
          if (!ofree && named_bar_or(bar_s, 128, !o_free(n + 1))) {
            ok = false;
            break;
          }
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int n0 = ndef0 + 64 * k;
            if (n0 < d.N) {
              uint8_t* oat = orow + (n0 >> 6) * kAtom;
#pragma unroll
              for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(oat + ((c ^ (et & 7)) << 4)) =
                    make_uint4(pk[32 * k + 4 * c], pk[32 * k + 4 * c + 1], pk[32 * k + 4 * c + 2], pk[32 * k + 4 * c + 3]);
            }
          }
          fence_proxy_async_smem();
          mbar_arrive(&oready[(n + 1) & 1]);
        } else {
          tc_fence_before();
          if (!seq_last) {
            __threadfence();
            named_bar_sync(bar_s, 128);
            if (et == 0) st_release_gpu(flags + I.b * hp + I.pair, I.w + 1);
          }
        }
      }
    }
    }
  } else {
    regs_acquire<kRegHead>();
    // ------------------------------------------------------------ head warpgroups: cumsum, X scaling, epilogue
    const int hh = (warp - 8) >> 2;  // head of the pair
    const int et = threadIdx.x - 256 - 128 * hh;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // token row = TMEM lane of the output
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t bar_h = 2 + hh;

    // window n from the ring, and this token's dt load issued (used a window later).
    // False at the end.
    auto fetch = [&](int n, Ctx& c) -> bool {
      WinInfo I;
      if (named_bar_or(bar_h, 128, !read_info(n, I))) {
        ok = false;
        return false;
      }
      c.b = I.b;
      c.pair = I.pair;
      c.w = I.w;
      if (I.flags & 4) return false;
      const int t = I.w * kWin + r;
      c.dt = t < d.L ? __ldg(dtg + (static_cast<int64_t>(I.b) * d.L + t) * d.H + 2 * I.pair + hh) : 0.f;
      c.a = __ldg(Avec + 2 * I.pair + hh);
      c.dd = __ldg(Dvec + 2 * I.pair + hh);
      return true;
    };
    // window n's cumsum, scalars and this head's X scaled in place
    auto prepare = [&](int n, Ctx& c) -> bool {
      float total;
      const float G = wg_scan(c.dt * c.a, scanws + (hh * 2 + (n & 1)) * 4, bar_h, lane, quad, total);
      c.g = G * kLog2e;
      const float gS = total * kLog2e;
      c.fastH = -gS <= kSpan;  // G is non-increasing, so the window's decay bounds every exponent
      const int sb = xs(n);
      // the X buffer has landed, so window n - nxb (same buffer and scalar slot) has been
      // stored: its readers of the slot are all done
      if (named_bar_or(bar_h, 128, !mbar_wait_short(&xfull[sb], xph(n), spin_ns))) {
        ok = false;
        return false;
      }
      if (et == 0) {
        scal[sb].alpha[hh] = fast_exp2(gS);
        scal[sb].fast[hh] = c.fastH;
      }
      // X^ (window start as reference) or X~ (window end) for this head, in place; the
      // row's eight 16-byte chunks are all loaded before any is written back
      const float wfac = fast_exp2(c.fastH ? -c.g : gS - c.g) * c.dt;
      uint4* row = reinterpret_cast<uint4*>(smem + Ls.xbuf + sb * kXBytes + hh * kWin * 128 + r * 128);
      uint4 xv[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) xv[k] = row[k ^ (r & 7)];  // the warp's 32 rows spread over all banks
      // The output accumulator's starting value on the rescaled form: D x_i / r_i, so that the
      // epilogue's r_i * acc already holds D x_i (window n - 2's output in these columns was
      // drained by this warpgroup's epilogue).  On the exact form the carried product
      // overwrites it, and the epilogue adds D x_i itself.
      {
        const float sx = c.fastH ? c.dd * fast_exp2(-c.g) : 0.f;
        const uint32_t ty = tmem + lane_base + kColY + 128 * (n & 1) + 64 * hh;
#pragma unroll
        for (int qt = 0; qt < 4; ++qt) {  // 16 columns at a time
          uint32_t v[16];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const uint32_t* xw = reinterpret_cast<const uint32_t*>(&xv[2 * qt + k]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              v[8 * k + 2 * e] = __float_as_uint(sx * bf16_lo(xw[e]));
              v[8 * k + 2 * e + 1] = __float_as_uint(sx * bf16_hi(xw[e]));
            }
          }
          tmem_st16(ty + 16 * qt, v);
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        xv[k].x = scale_bf16x2(xv[k].x, wfac);
        xv[k].y = scale_bf16x2(xv[k].y, wfac);
        xv[k].z = scale_bf16x2(xv[k].z, wfac);
        xv[k].w = scale_bf16x2(xv[k].w, wfac);
        row[k ^ (r & 7)] = xv[k];
      }
      tmem_st_wait();
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(&xready[sb]);
      return true;
    };

    // Per iteration: the epilogue of window n, then window n + 2's cumsum and X scaling (its
    // output accumulator is the one the epilogue just drained), so that a window's scaled X and
    // scalars are ready a window before the state pass of the window ahead of it asks for them.
    Ctx cur, nxt, nn, n3;
    bool more = fetch(0, cur) && prepare(0, cur);
    bool more1 = more && fetch(1, nxt) && prepare(1, nxt);
    bool more2 = more1 && fetch(2, nn);
    for (int n = 0; ok && more; ++n) {
      if (!ok) break;
      const int yb = n & 1, sb = xs(n);
      const int h = 2 * cur.pair + hh;
      const int t0 = cur.w * kWin;
      // y = r_i * acc + D x_i, written over X^ in the X buffer once the window's last product
      // is done (tcgen05 operations complete in order, so the state product, which reads X^
      // too, is done as well); warp 3 stores it
      if (named_bar_or(bar_h, 128, !mbar_wait_short(&xready[sb], xph(n), spin_ns) ||
                                       !mbar_wait_short(kPB ? &cdone[yb] : &ydone[yb], yph(n), spin_ns))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool fast = scal[sb].fast[0] && scal[sb].fast[1];
      const float Dh = cur.dd;
      uint8_t* xr = smem + Ls.xbuf + sb * kXBytes + hh * kWin * 128 + r * 128;
      const uint32_t tacc = tmem + lane_base + kColY + 128 * yb + 64 * hh;
      if (fast) {
        uint32_t ya[64];
        tmem_ld32(tacc, *reinterpret_cast<uint32_t(*)[32]>(ya));
        tmem_ld32(tacc + 32, *reinterpret_cast<uint32_t(*)[32]>(ya + 32));
        tmem_ld_wait();
        tc_fence_before();
        // y_i = r_i * acc: the accumulator started at D x_i / r_i (see prepare)
        const float ri = fast_exp2(cur.g);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          uint4 v;
          uint32_t* vw = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int pi = 8 * k + 2 * e;
            vw[e] = pack_bf16x2(ri * __uint_as_float(ya[pi]), ri * __uint_as_float(ya[pi + 1]));
          }
          *reinterpret_cast<uint4*>(xr + ((k ^ (r & 7)) << 4)) = v;
        }
      } else {
        const int g = (2 * cur.pair) / (d.H / d.G);
        const __nv_bfloat16* Mrow = Mg + ((static_cast<int64_t>(cur.b) * nw + cur.w) * d.G + g) * kWin * kWin +
                                    static_cast<int64_t>(r) * kWin;
        grid_dep_wait();  // the causal blocks come from the pre-pass
        exact_epilogue(d, cur.b, h, t0, r, cur.g, cur.a, Dh, Mrow, xg, dtg, tacc, xr);
        tc_fence_before();
      }
      fence_proxy_async_smem();
      mbar_arrive(&ystaged[sb]);
      if (more2 && !prepare(n + 2, nn)) break;
      const bool more3 = more2 && fetch(n + 3, n3);
      if (!ok) break;
      cur = nxt;
      nxt = nn;
      nn = n3;
      more = more1;
      more1 = more2;
      more2 = more3;
    }
  }

  if (!ok) {
    grid_dep_wait();  // the status word is cleared by the pre-pass
    atomicExch(status, static_cast<int>(SSD_ERR_DEVICE_TIMEOUT));
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t onepass_smem_bytes(const Dims& d) { return op_layout(d.N).total + 1024; }

int onepass_runs(const Dims& d, int R) {
  const int nw = (d.L + kWin - 1) / kWin;
  return ((nw + R - 1) / R) * d.B * (d.H / 2);
}

// The schedule from the shape: claims of R windows (the longest of 16, 8 and 4 that
// still gives every multiprocessor at least four runs; longer runs hand the state
// between CTAs less often), unless those runs spread unevenly -- the busiest CTA more
// than 10 % above the mean -- in which case the static split (0) runs.  Measured on
// GB300 (bf16):
//  - 2.7B layer (160 sequences of 32 windows): claims of 2 / 4 / 8 / 16 windows ran
//    0.259 / 0.203 / 0.192 / 0.199 ms, and 8 windows leave some CTAs 5 runs against a
//    mean of 4.2; the static split ran 0.166 ms.
//  - 65,536-token sweep points with many whole sequences per CTA (L2048 and L8192 at
//    N64-256, L512): claims ran 0.49-0.83 ms, the static split 0.46-0.97 ms (slower
//    on all but one: per-CTA speeds differ by about 10 %, which claims absorb).
int onepass_run_length(const Dims& d, int sms) {
  int R = 4;
  for (int r : {16, 8})
    if (onepass_runs(d, r) >= 4 * sms) {
      R = r;
      break;
    }
  const int runs = onepass_runs(d, R);
  const int per_cta = (runs + sms - 1) / sms;  // the busiest CTA's runs
  return static_cast<double>(per_cta) * sms > 1.1 * runs ? 0 : R;
}

// One CTA per multiprocessor; the static split takes at most one per sequence (each
// CTA's share must hold a whole sequence's windows), claims at most one per run.
int onepass_grid(const Dims& d, int sms, int R) {
  const int units = R > 0 ? onepass_runs(d, R) : d.B * (d.H / 2);
  return units < sms ? units : sms;
}

cudaError_t launch_onepass(const Dims& d, const OnePassMaps& maps, const float* dt, const float* A, const float* D,
                           const void* x, const float* init, float* final_state, const Work& w, uint64_t spin_ns,
                           cudaStream_t stream, bool dependent, int force_R) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const size_t smem = onepass_smem_bytes(d);
  // product buffers up to dstate 128 (two of them and two output accumulators fill tensor
  // memory); the state accumulated in tensor memory at dstate 256
  const auto kern = d.N == 64 ? ssd_onepass_kernel<64> : d.N == 128 ? ssd_onepass_kernel<128> : ssd_onepass_kernel<256>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // the register split assumes the compiled count; any other count is refused here
  cudaFuncAttributes fa{};
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != static_cast<int>(kRegLaunch)) return cudaErrorInvalidConfiguration;
  const int R = force_R > 0 ? force_R : onepass_run_length(d, sms);
  const int grid = onepass_grid(d, sms, R);
  return launch_k(kern, dim3(grid), dim3(kThreads), smem, stream, dependent, maps.x, maps.cm, maps.bm,
                  maps.m, maps.y, d, R, dt, A, D, static_cast<const __nv_bfloat16*>(w.cbm), init, final_state,
                  w.hslot, w.flags, w.counter, static_cast<const __nv_bfloat16*>(x), w.status, spin_ns);
}

}  // namespace ssd
