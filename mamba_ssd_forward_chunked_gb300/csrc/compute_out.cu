// Step 4 of the SSD forward: the fused output kernel.
//
// "Jane Street ML Engineers Map Mamba-2 Recurrent State Computation to Tensor
// Cores with cuTile", compute_out paragraph: one tiled kernel sums three terms
// -- the carried-state term, the decayed and causally masked interaction
// matrix C B^T o exp(G - G^T), and the D*x skip -- without writing the
// chunk_size x chunk_size matrix to global memory; the mask is an index
// comparison, never a tensor, and the positive exponents above the diagonal
// are zeroed before they can overflow.  Blackwell paragraph: the MMA's A
// operand may live in tensor memory while B must come from shared memory, so
// the register-computed (fused) operand is routed to the A side.
//
// Work unit ("tile"): batch b, chunk c, 128-row block t of the chunk (rows i),
// and a PAIR of heads (h0, h1) of one group.  Both heads read the same C and B,
// so C B^T is computed once per tile and shared.  Columns j run over 128-wide
// blocks jb <= t.  Per head h:
//
//     Y_h   = C_t hprev_h^T                                  (K = dstate)
//     Y_h  *= exp(G_i)            (row scale, in tensor memory)
//     CB    = C_t B_jb^T                                     (K = dstate, shared)
//     M_h   = CB o [j <= i] exp(G_i - G_j) dt_j              (registers -> TMEM)
//     Y_h  += M_h X_h,jb                                     (A = M_h from TMEM)
//     y_i   = Y_h[i] + D_h x_i
//
// Tensor memory (512 columns): [0,128) CB (fp32), [128,192) Y_h0, [192,256)
// Y_h1, [256,384) M_h0, [384,512) M_h1 (TF32: 128 columns; bf16: packed pairs
// in the first 64).  In the first column block CB and both carried-state terms
// are one N = 256 product per K step: the stage holds B_jb's rows and then the
// pair's entering-state rows back to back, and CB, Y_h0, Y_h1 are adjacent
// columns.  The exponentials are factored so that every factor
// is <= 1: for a 32-column strip entirely left of row i,
// exp(G_i - G_j) = exp(G_i - G_e) exp(G_e - G_j) with e the strip's last
// column; only the 32 x 32 blocks on the diagonal take one exp per element,
// behind the causal select.
//
// GB300 mapping: a persistent grid (one CTA per SM, the CTA's tensor memory is
// the whole 512 columns) walks the tiles with the head pair fastest, so the
// CTAs running at one time share C and B tiles in L2.  Warp 0 issues TMA into
// two rings, in the order the MMA warp consumes them: per column block, the
// dstate slices of {C, B, the two entering states} (48 KB stages) and the two
// heads' X blocks (a ring of its own, so X blocks are fetched up to two column
// blocks ahead); the next tile's loads stream in while this one computes.  Warp 1
// owns tensor memory and issues every MMA from one thread; warps 2-3 only fill
// the control warpgroup, which gives its registers to the head warpgroups
// (setmaxnreg: the TF32 head code spilled at the launch count).
// Warps 4-7 and 8-11 are two warpgroups, one per head of the pair: each scales
// its carried-state accumulator, builds its masked matrix from the shared CB,
// and writes its head's output rows, so the two heads' elementwise work runs
// side by side.  A warpgroup loads the next tile's per-column data into
// registers one tile ahead, takes exponentials as 2^x of the cumsum scaled by
// log2(e), and keeps the last X block of its head until the epilogue: it reads
// x_i (for D*x) from it, overwrites it with y in the same swizzled layout and
// writes y out with TMA tensor stores, so no global load or scattered store
// sits on its critical path.  X is the intra product's MN-major B operand in both
// precisions: bf16 as one 64-p box in the 128-byte swizzle, fp32 as two 32-p boxes in
// the 128-byte swizzle of 32-byte atoms (the layout the tensor core reads an MN-major
// TF32 operand in; TMA writes it).  Every wait is bounded; on expiry the CTA
// records SSD_ERR_DEVICE_TIMEOUT, stops, frees its tensor memory and exits.
#include "ptx.cuh"
#include "ssd_internal.cuh"

namespace ssd {
namespace {

template <typename T>
struct OutCfg {
  static constexpr bool kTF32 = sizeof(T) == 4;
  static constexpr int kAtom = 128 / static_cast<int>(sizeof(T));  // elements per 128-B row
  static constexpr int kStages = 3;                                                // dstate-slice ring
  static constexpr int kStageBytes = 48 * 1024;
  static constexpr int kOffC = 0, kOffB = 16384, kOffH0 = 32768, kOffH1 = 40960;  // K-slice stage
  static constexpr int kXBytes = kTF32 ? 32768 : 16384;                            // X stage: 128 tokens x 64 p
  static constexpr int kXStages = kTF32 ? 2 : 4;                                   // X ring
  static constexpr int kKStepX = kTF32 ? 8 : 16;                                   // tokens per intra MMA
  static constexpr int kThreads = 384;
  static constexpr uint32_t kColCB = 0, kColY0 = 128, kColM0 = 256, kTmemCols = 512;
  static constexpr int kWgFloats = 3 * 256;  // per warpgroup: cumsum, dt, strip factors for 256 columns
};

static_assert(OutCfg<float>::kOffH0 == OutCfg<float>::kOffB + 128 * 128 &&
                  OutCfg<float>::kOffH1 == OutCfg<float>::kOffH0 + 64 * 128 &&
                  OutCfg<float>::kColY0 == OutCfg<float>::kColCB + 128,
              "B_jb's and the entering states' slices, and CB and Y, must be adjacent (one N = 256 product)");

constexpr float kSpan = 100.f;  // rescaled form: log2 bound on the diagonal block's decay

// Register split (setmaxnreg): 384 threads launch with kRegLaunch each (12 warps, three per
// sub-partition); the control warpgroup (TMA and MMA warps, two idle) gives registers up and
// the two head warpgroups take them.  The split must stay within the launch's pool (an
// increase that cannot be met waits without end); the host checks the compiled count.
constexpr uint32_t kRegLaunch = 168, kRegCtl = 88, kRegHead = 200;
static_assert(128 * (kRegCtl + 2 * kRegHead) <= 384 * kRegLaunch, "register split above the pool");
template <uint32_t kRegs>
__device__ __forceinline__ void regs_release() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs));
}
template <uint32_t kRegs>
__device__ __forceinline__ void regs_acquire() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs));
}

// Rescaled operands are clamped to finite values: an overflowing product must
// not become inf, which the causal select's zeros would turn into NaN in rows
// that never see that token.
__device__ __forceinline__ float clamp_finite(float v) { return fminf(fmaxf(v, -3.4e38f), 3.4e38f); }
__device__ __forceinline__ uint32_t scale_bf16x2_clamped(uint32_t v, float s) {
  constexpr float kMax = 3.38e38f;  // below bf16's largest finite value, so rounding cannot reach inf
  return pack_bf16x2(fminf(fmaxf(bf16_lo(v) * s, -kMax), kMax), fminf(fmaxf(bf16_hi(v) * s, -kMax), kMax));
}

struct OutSmem {
  uint32_t ring, xring, wg, bars, holder, total;
};

template <typename T>
__host__ __device__ constexpr OutSmem out_smem_layout() {
  using C = OutCfg<T>;
  OutSmem s{};
  s.ring = 0;
  s.xring = C::kStages * C::kStageBytes;
  s.wg = s.xring + C::kXStages * C::kXBytes;
  s.bars = s.wg + 2 * C::kWgFloats * 4;
  s.holder = s.bars + 32 * 8;
  s.total = s.holder + 16;
  return s;
}

struct TileId {
  int b, c, t, h0;
};

__device__ __forceinline__ TileId decode_tile(int tile, const Dims& d, int ntile) {
  const int hp = d.H / 2;
  TileId id;
  id.h0 = 2 * (tile % hp);
  int rest = tile / hp;
  id.t = rest % ntile;
  rest /= ntile;
  id.c = rest % d.nc;
  id.b = rest / d.nc;
  return id;
}

// One 32-column strip of the masked, decayed matrix for row i, in place:
// v holds C_i . B_j for j = j0 .. j0 + 31 on entry and is written to the
// tensor-memory A operand at `dst` (TF32: one column per element; bf16: packed
// pairs).  gs is the cumsum in log2 units, vref[j] = 2^(gs[e] - gs[j]) dt_j
// for e the last column of j's strip.
template <bool kTF32>
__device__ __forceinline__ void mask_strip(uint32_t (&v)[32], int j0, int i, float Gi, const float* gs,
                                           const float* dts, const float* vref, uint32_t dst) {
  if (j0 + 31 < i) {  // strip strictly left of the diagonal (warp-uniform)
    const float u = fast_exp2(Gi - gs[j0 + 31]);
#pragma unroll
    for (int q = 0; q < 32; ++q) v[q] = __float_as_uint(__uint_as_float(v[q]) * u * vref[j0 + q]);
  } else if (j0 > i) {  // strip strictly right of the diagonal (warp-uniform)
#pragma unroll
    for (int q = 0; q < 32; ++q) v[q] = 0u;
  } else {  // the 32 x 32 block on the diagonal: select, then exp (exponent <= 0)
#pragma unroll
    for (int q = 0; q < 32; ++q) {
      const int j = j0 + q;
      v[q] = j <= i ? __float_as_uint(__uint_as_float(v[q]) * fast_exp2(Gi - gs[j]) * dts[j]) : 0u;
    }
  }
  if constexpr (kTF32) {
#pragma unroll
    for (int q = 0; q < 32; ++q) v[q] = __float_as_uint(round_tf32(__uint_as_float(v[q])));
    tmem_st32(dst, v);
  } else {
    uint32_t o[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) o[q] = pack_bf16x2(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1]));
    tmem_st16(dst, o);
  }
}

// Rescaled form (see the kernel comment): the masked operand is the causal
// select of C B^T alone.  One 32-column strip for row i, stored at `dst`.
template <bool kTF32>
__device__ __forceinline__ void causal_strip(uint32_t (&v)[32], int j0, int i, uint32_t dst) {
  if (j0 > i) {  // strictly right of the diagonal (warp-uniform)
#pragma unroll
    for (int q = 0; q < 32; ++q) v[q] = 0u;
  } else if (j0 + 31 > i) {  // the diagonal block
#pragma unroll
    for (int q = 0; q < 32; ++q) v[q] = j0 + q <= i ? v[q] : 0u;
  }
  if constexpr (kTF32) {
    tmem_st32(dst, v);
  } else {
    uint32_t o[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) o[q] = pack_bf16x2(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1]));
    tmem_st16(dst, o);
  }
}

// 16-byte piece k (values 4k .. 4k + 3) of row r of a 32-p fp32 box: in the
// 32-byte-atom swizzle, 32-byte chunk k / 2 of the row sits at (k / 2) ^ (r % 4).
__device__ __forceinline__ int a32_piece(int k, int r) { return (((k >> 1) ^ (r & 3)) << 1) | (k & 1); }

// Copies token r's raw x row (64 values, or zeros) over its rescaled copy in
// the X block, in the layout the epilogue reads: TF32 row r of the two 32-p
// boxes (32-byte-atom swizzle), bf16 row r (128-byte swizzle).  Only thread r
// touches these bytes.
template <bool kTF32, typename T>
__device__ __noinline__ void restore_x_row(uint8_t* xy, int r, const T* src) {
  if constexpr (kTF32) {
    for (int half = 0; half < 2; ++half) {
      float4* row = reinterpret_cast<float4*>(xy + half * 16384 + r * 128);
      for (int k = 0; k < 8; ++k) {
        const int q = 32 * half + 4 * k;
        row[a32_piece(k, r)] = src ? make_float4(static_cast<float>(src[q]), static_cast<float>(src[q + 1]),
                                                 static_cast<float>(src[q + 2]), static_cast<float>(src[q + 3]))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  } else {
    for (int k = 0; k < 8; ++k)
      *reinterpret_cast<uint4*>(xy + r * 128 + ((k ^ (r & 7)) << 4)) =
          src ? reinterpret_cast<const uint4*>(src)[k] : make_uint4(0, 0, 0, 0);
  }
}

template <typename T>
__global__ void __launch_bounds__(OutCfg<T>::kThreads, 1)
    compute_out_kernel(const __grid_constant__ CUtensorMap cmap, const __grid_constant__ CUtensorMap bmap,
                       const __grid_constant__ CUtensorMap hmap, const __grid_constant__ CUtensorMap xmap,
                       const __grid_constant__ CUtensorMap ymap, Dims d,
                       const float* __restrict__ cumsum, const float* __restrict__ dt_t,
                       const float* __restrict__ Dvec, const T* __restrict__ xg, int* status, uint64_t spin_ns) {
  using C = OutCfg<T>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr OutSmem L = out_smem_layout<T>();
  const int Q = d.Q;
  const int ntile = Q >= 128 ? Q / 128 : 1;
  const int ntiles = d.B * d.nc * ntile * (d.H / 2);
  const int NB = d.N / C::kAtom;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* full = bars;                  // [kStages]
  uint64_t* empty = bars + C::kStages;    // [kStages]
  uint64_t* xfullb = bars + 2 * C::kStages;    // [kXStages]
  uint64_t* xempty = xfullb + C::kXStages;      // [kXStages]
  uint64_t* cbfull = xempty + C::kXStages;
  uint64_t* mready = cbfull + 1;          // [2]
  uint64_t* mfree = cbfull + 3;           // [2]
  uint64_t* yfull = cbfull + 5;
  uint64_t* yfree = cbfull + 6;           // [2]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L.holder);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < C::kXStages; ++s) {
      mbar_init(&xfullb[s], 1);
      mbar_init(&xempty[s], 1 + 128);  // the MMA commit and the head's warpgroup
    }
    mbar_init(cbfull, 1);
    mbar_init(&mready[0], 128);
    mbar_init(&mready[1], 128);
    mbar_init(&mfree[0], 1);
    mbar_init(&mfree[1], 1);
    mbar_init(yfull, 1);
    mbar_init(&yfree[0], 128);
    mbar_init(&yfree[1], 128);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&cmap);
    tma_prefetch_desc(&bmap);
    tma_prefetch_desc(&hmap);
    tma_prefetch_desc(&xmap);
    tma_prefetch_desc(&ymap);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, C::kTmemCols);
    tmem_relinquish();
  }
  grid_dep_wait();  // the entering states (and the cumsum) are visible from here on
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  bool ok = true;

  if (warp < 4) {
  regs_release<kRegCtl>();
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int it = 0, xit = 0;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
        const TileId id = decode_tile(tile, d, ntile);
        const int g = id.h0 / (d.H / d.G);
        const int hrow0 = ((id.b * d.nc + id.c) * d.H + id.h0) * d.P;
        for (int jb = 0; jb <= id.t && ok; ++jb) {
          for (int nb = 0; nb < NB + 2; ++nb) {
            const bool kslice = nb < NB;
            const int ring_n = kslice ? C::kStages : C::kXStages;
            const int cnt = kslice ? it++ : xit++;
            const int s = cnt % ring_n, r = cnt / ring_n;
            uint64_t* emp = kslice ? &empty[s] : &xempty[s];
            if (r > 0 && !mbar_wait(emp, (r - 1) & 1, spin_ns)) {
              ok = false;
              break;
            }
            uint8_t* st = kslice ? smem + L.ring + s * C::kStageBytes : smem + L.xring + s * C::kXBytes;
            if (kslice) {  // dstate slice: C, B (and the entering states at jb = 0)
              mbar_arrive_expect_tx(&full[s], 32768u + (jb == 0 ? 16384u : 0u));
              tma_load_4d(st + C::kOffC, &cmap, &full[s], nb * C::kAtom, g, id.c * Q + id.t * 128, id.b);
              tma_load_4d(st + C::kOffB, &bmap, &full[s], nb * C::kAtom, g, id.c * Q + jb * 128, id.b);
              if (jb == 0) {
                tma_load_2d(st + C::kOffH0, &hmap, &full[s], nb * C::kAtom, hrow0);
                tma_load_2d(st + C::kOffH1, &hmap, &full[s], nb * C::kAtom, hrow0 + d.P);
              }
            } else {  // X block of one head: 128 tokens x 64 p
              const int h = id.h0 + (nb - NB);
              mbar_arrive_expect_tx(&xfullb[s], static_cast<uint32_t>(C::kXBytes));
              if constexpr (C::kTF32) {
                // two 128-token boxes of 32 p, 16 KB apart (the operand's column blocks)
                for (int hf = 0; hf < 2; ++hf)
                  tma_load_3d(st + hf * 16384, &xmap, &xfullb[s], h * d.P + hf * 32, id.c * Q + jb * 128, id.b);
              } else {
                tma_load_3d(st, &xmap, &xfullb[s], h * d.P, id.c * Q + jb * 128, id.b);
              }
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t fmt = C::kTF32 ? 2u : 1u;
      // first column block: C [B_jb; h_h0; h_h1]^T -> [CB | Y_h0 | Y_h1] in one product
      const uint32_t id_cby = idesc_f32acc(fmt, 128, 256, 0, 0);
      const uint32_t id_cb = idesc_f32acc(fmt, 128, 128, 0, 0);
      const uint32_t id_yint = idesc_f32acc(fmt, 128, 64, 0, 1u);
      int it = 0, xit = 0, ntd = 0, nm = 0;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++ntd) {
        const TileId id = decode_tile(tile, d, ntile);
        for (int jb = 0; jb <= id.t && ok; ++jb) {
          if (jb == 0 && ntd > 0) {  // both heads drained Y of the previous tile
            if (!mbar_wait(&yfree[0], (ntd - 1) & 1, spin_ns) || !mbar_wait(&yfree[1], (ntd - 1) & 1, spin_ns)) {
              ok = false;
              break;
            }
          }
          for (int nb = 0; nb < NB; ++nb, ++it) {
            const int s = it % C::kStages, r = it / C::kStages;
            if (!mbar_wait(&full[s], r & 1, spin_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t st = smem_u32(smem + L.ring + s * C::kStageBytes);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              // K-major, 128-B swizzle: a K step is 32 B along the row; SBO = 1024 B
              const uint64_t ad = sdesc_sw128(st + C::kOffC + k * 32, 16, 1024);
              const uint32_t acc = (nb | k) != 0 ? 1u : 0u;
              mma_ss<C::kTF32>(tmem + C::kColCB, ad, sdesc_sw128(st + C::kOffB + k * 32, 16, 1024),
                               jb == 0 ? id_cby : id_cb, acc);
            }
            mma_commit(&empty[s]);
          }
          if (!ok) break;
          mma_commit(cbfull);
          for (int hh = 0; hh < 2; ++hh, ++xit) {
            const int s = xit % C::kXStages, r = xit / C::kXStages;
            if (!mbar_wait(&xfullb[s], r & 1, spin_ns) || !mbar_wait(&mready[hh], nm & 1, spin_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t xb = smem_u32(smem + L.xring + s * C::kXBytes);
#pragma unroll 4
            for (int k = 0; k < 128 / C::kKStepX; ++k) {
              uint64_t xd;
              if constexpr (C::kTF32) {
                // X, MN-major: a K step is 8 token rows of 128 B; LBO = the second 32-p box,
                // SBO = 4-row groups
                xd = sdesc_sw128_a32(xb + k * 1024, 16384, 512);
              } else {
                xd = sdesc_sw128(xb + k * C::kKStepX * 128, 16384, 1024);  // X, MN-major (one 64-p atom)
              }
              mma_ts<C::kTF32>(tmem + C::kColY0 + 64 * hh, tmem + C::kColM0 + 128 * hh + k * 8, xd, id_yint, 1u);
            }
            mma_commit(&xempty[s]);
            mma_commit(&mfree[hh]);
          }
          ++nm;
        }
        if (ok) mma_commit(yfull);
      }
    }
  }
  } else {
    regs_acquire<kRegHead>();
    // ------------------------------------------------------------ one warpgroup per head
    const int hh = (warp - 4) >> 2;
    const int et = threadIdx.x - 128 - 128 * hh;  // 0..127
    const uint32_t bar_id = 1 + hh;
    float* gs = reinterpret_cast<float*>(smem + L.wg) + hh * C::kWgFloats;  // cumsum in log2 units
    float* dts = gs + 256;
    float* vref = gs + 512;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // TMEM lane = row of the tile
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t colM = C::kColM0 + 128 * hh, colY = C::kColY0 + 64 * hh;
    // per-tile column data (columns et and et + 128) and D_h, loaded one tile ahead
    float pg[2], pd[2], pD = 0.f, pm[2], pl[2];
    auto prefetch = [&](int tile) {
      const TileId id = decode_tile(tile, d, ntile);
      const int h = id.h0 + hh;
      const int64_t grow = (static_cast<int64_t>(id.b) * d.H + h) * d.Lp + static_cast<int64_t>(id.c) * Q;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int j = et + 128 * k;
        pg[k] = cumsum[grow + (j < Q ? j : Q - 1)];
        pd[k] = j < Q ? dt_t[grow + j] : 0.f;
        // both heads of the pair: cumsum at the tile's first row (the reference token) and at
        // the last column of its diagonal block
        const int64_t prow = (static_cast<int64_t>(id.b) * d.H + id.h0 + k) * d.Lp + static_cast<int64_t>(id.c) * Q;
        const int last = id.t * 128 + 127 < Q ? id.t * 128 + 127 : Q - 1;
        pm[k] = cumsum[prow + id.t * 128];
        pl[k] = cumsum[prow + last];
      }
      pD = Dvec[h];
    };
    // per-tile scalars of this warpgroup's head, set up from the prefetched column data
    struct TileVars {
      float Dh, gm, Gi, dti;
      bool fast;
    };
    // writes the tile's gs / dts / vref and issues the next tile's prefetch; runs while the
    // previous tile's last products are on the tensor core (its epilogue needs none of them)
    auto setup = [&](int tile) -> TileVars {
      const TileId id = decode_tile(tile, d, ntile);
      const int i = id.t * 128 + r;  // row within the chunk
      const int ncol = 128 * (id.t + 1);
      named_bar_sync(bar_id, 128);  // the previous tile's readers of gs / dts / vref are done
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int j = et + 128 * k;
        if (j < ncol) {
          gs[j] = pg[k] * kLog2e;
          dts[j] = pd[k];
        }
      }
      TileVars v;
      v.Dh = pD;
      // rescaled form for the whole pair while the diagonal block's decay stays within 2^kSpan
      // (G is non-increasing: every other factor of the form is <= 1)
      v.fast = true;
#pragma unroll
      for (int k = 0; k < 2; ++k) v.fast = v.fast && ((pm[k] - pl[k]) * kLog2e <= kSpan);
      v.gm = pm[hh] * kLog2e;  // this head's reference, log2 units
      if (tile + static_cast<int>(gridDim.x) < ntiles) prefetch(tile + gridDim.x);  // in flight during this tile
      named_bar_sync(bar_id, 128);
      // fast: vref[j] = 2^(G_m - G_j) dt_j, the row scale of X; exact form: strip factors
      for (int j = et; j < ncol; j += 128)
        vref[j] = fast_exp2((v.fast ? v.gm : gs[j | 31]) - gs[j]) * dts[j];
      named_bar_sync(bar_id, 128);
      v.Gi = gs[i];
      v.dti = i < 256 ? dts[i] : 0.f;
      return v;
    };
    TileVars nxt{};
    if (static_cast<int>(blockIdx.x) < ntiles) {
      prefetch(blockIdx.x);
      nxt = setup(blockIdx.x);
    }
    int xit = 0, ncb = 0, nm = 0, ntd = 0;
    const uint8_t* xlast = nullptr;  // X block (this head, last column block) read by the epilogue
    int xs_last = 0;
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++ntd) {
      const TileId id = decode_tile(tile, d, ntile);
      const int h = id.h0 + hh;
      const int i = id.t * 128 + r;  // row within the chunk
      const TileVars cur = nxt;
      const float Dh = cur.Dh, gm = cur.gm, Gi = cur.Gi;
      const bool fast = cur.fast;

      for (int jb = 0; jb <= id.t; ++jb) {
        if (!mbar_wait(cbfull, ncb & 1, spin_ns)) {
          ok = false;
          break;
        }
        ++ncb;
        tc_fence_after();
        const int xs = xit + hh;  // X-ring stage holding this head's X block
        xit += 2;
        uint8_t* xb = smem + L.xring + (xs % C::kXStages) * C::kXBytes;
        if (jb == 0) {  // carried-state term: scale row i by exp(G_i) (rescaled form: by exp(G_m))
          const float eGi = fast_exp2(fast ? gm : Gi);
          uint32_t v0[32], v1[32];
          tmem_ld32(tmem + lane_base + colY, v0);
          tmem_ld32(tmem + lane_base + colY + 32, v1);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            v0[q] = __float_as_uint(__uint_as_float(v0[q]) * eGi);
            v1[q] = __float_as_uint(__uint_as_float(v1[q]) * eGi);
          }
          tmem_st32(tmem + lane_base + colY, v0);
          tmem_st32(tmem + lane_base + colY + 32, v1);
        }
        if (nm > 0 && !mbar_wait(&mfree[hh], (nm - 1) & 1, spin_ns)) {  // M_h no longer read
          ok = false;
          break;
        }
        if (fast) {  // rescaled form: X^ = 2^(G_m - G_j) dt_j x_j, rows scaled in place (row et = token et)
          if (!mbar_wait(&xfullb[xs % C::kXStages], (xs / C::kXStages) & 1, spin_ns)) {
            ok = false;
            break;
          }
          const float wj = vref[jb * 128 + et];
          if constexpr (C::kTF32) {
            // 128 bytes of the row in each of the two 32-p boxes; the chunk order is rotated per
            // row so that a warp's accesses spread over all banks (the scale is the same for all)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              float4* row = reinterpret_cast<float4*>(xb + hf * 16384 + et * 128);
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                float4* cp = row + (k ^ (et & 7));
                float4 v = *cp;
                v.x = clamp_finite(v.x * wj);
                v.y = clamp_finite(v.y * wj);
                v.z = clamp_finite(v.z * wj);
                v.w = clamp_finite(v.w * wj);
                *cp = v;
              }
            }
          } else {
            uint4* row = reinterpret_cast<uint4*>(xb + et * 128);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              uint4* cp = row + (k ^ (et & 7));  // swizzle-ordered steps: the warp spreads over all banks
              uint4 v = *cp;
              v.x = scale_bf16x2_clamped(v.x, wj);
              v.y = scale_bf16x2_clamped(v.y, wj);
              v.z = scale_bf16x2_clamped(v.z, wj);
              v.w = scale_bf16x2_clamped(v.w, wj);
              *cp = v;
            }
          }
          fence_proxy_async_smem();
        }
        // masked matrix, four 32-column strips; two TMEM loads in flight so the
        // next strip's load overlaps this strip's arithmetic
        if (fast) {
          uint32_t va[32], vb[32];
          tmem_ld32(tmem + lane_base + C::kColCB, va);
          tmem_ld32(tmem + lane_base + C::kColCB + 32, vb);
          tmem_ld_wait();
          causal_strip<C::kTF32>(va, jb * 128, i, tmem + lane_base + colM);
          tmem_ld32(tmem + lane_base + C::kColCB + 64, va);
          causal_strip<C::kTF32>(vb, jb * 128 + 32, i, tmem + lane_base + colM + (C::kTF32 ? 32 : 16));
          tmem_ld_wait();
          tmem_ld32(tmem + lane_base + C::kColCB + 96, vb);
          causal_strip<C::kTF32>(va, jb * 128 + 64, i, tmem + lane_base + colM + (C::kTF32 ? 64 : 32));
          tmem_ld_wait();
          causal_strip<C::kTF32>(vb, jb * 128 + 96, i, tmem + lane_base + colM + (C::kTF32 ? 96 : 48));
        } else {
          uint32_t va[32], vb[32];
          tmem_ld32(tmem + lane_base + C::kColCB, va);
          tmem_ld32(tmem + lane_base + C::kColCB + 32, vb);
          tmem_ld_wait();
          mask_strip<C::kTF32>(va, jb * 128, i, Gi, gs, dts, vref, tmem + lane_base + colM);
          tmem_ld32(tmem + lane_base + C::kColCB + 64, va);
          mask_strip<C::kTF32>(vb, jb * 128 + 32, i, Gi, gs, dts, vref, tmem + lane_base + colM + (C::kTF32 ? 32 : 16));
          tmem_ld_wait();
          tmem_ld32(tmem + lane_base + C::kColCB + 96, vb);
          mask_strip<C::kTF32>(va, jb * 128 + 64, i, Gi, gs, dts, vref, tmem + lane_base + colM + (C::kTF32 ? 64 : 32));
          tmem_ld_wait();
          mask_strip<C::kTF32>(vb, jb * 128 + 96, i, Gi, gs, dts, vref, tmem + lane_base + colM + (C::kTF32 ? 96 : 48));
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&mready[hh]);
        ++nm;
        // this warpgroup's share of releasing the X block; the last one is kept for D*x
        if (!mbar_wait(&xfullb[xs % C::kXStages], (xs / C::kXStages) & 1, spin_ns)) {
          ok = false;
          break;
        }
        if (jb < id.t) {
          mbar_arrive(&xempty[xs % C::kXStages]);
        } else {
          xlast = xb;
          xs_last = xs % C::kXStages;
        }
      }
      if (!ok) break;
      if (tile + static_cast<int>(gridDim.x) < ntiles) nxt = setup(tile + gridDim.x);

      // epilogue: y_i = Y_h[i] + D_h x_i, written over x in the X block and
      // stored with TMA (rows past Q are not stored; TMA clips rows past L)
      if (!mbar_wait(yfull, ntd & 1, spin_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t yall[2][32];
      tmem_ld32(tmem + lane_base + colY, yall[0]);
      tmem_ld32(tmem + lane_base + colY + 32, yall[1]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&yfree[hh]);  // Y_h may be overwritten by the next tile's MMAs
      uint8_t* xy = const_cast<uint8_t*>(xlast);
      // rescaled form: y_i = r_i (acc + (D / dt_i) X^_i) with r_i = 2^(G_i - G_m), while X^_i = w_i x_i
      // is well inside the normal range; otherwise x_i is copied back over X^_i from global memory
      float ry = 1.f, kx = Dh;
      if (fast) {
        const float dti = cur.dti;
        const float wi = fast_exp2(gm - Gi) * dti;
        ry = fast_exp2(Gi - gm);
        if (wi >= 0x1p-80f) {
          kx = Dh / dti;
        } else {
          kx = Dh / ry;
          const int tok = id.c * Q + i;
          const bool in_seq = i < Q && tok < d.L;
          restore_x_row<C::kTF32>(xy, r, in_seq ? xg + ((static_cast<int64_t>(id.b) * d.L + tok) * d.H + h) * d.P
                                                : nullptr);
        }
      }
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint32_t (&yv)[32] = yall[half];
        if constexpr (C::kTF32) {
          // row r of box `half` holds x_r's 32 values (32-byte-atom swizzle); y_r goes in place
          float4* row = reinterpret_cast<float4*>(xy + half * 16384 + r * 128);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            float4* px = row + a32_piece(k, r);
            const float4 xv = *px;
            const int q = 4 * k;
            *px = make_float4(ry * fmaf(kx, xv.x, __uint_as_float(yv[q])), ry * fmaf(kx, xv.y, __uint_as_float(yv[q + 1])),
                              ry * fmaf(kx, xv.z, __uint_as_float(yv[q + 2])),
                              ry * fmaf(kx, xv.w, __uint_as_float(yv[q + 3])));
          }
        } else {
          // MN-major rows: token r is row r, p in 16-B chunks of 8 (in place)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4* px = reinterpret_cast<uint4*>(xy + r * 128 + (((half * 4 + k) ^ (r & 7)) << 4));
            const uint4 xv = *px;
            const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int q = 8 * k + 2 * e;
              o[e] = pack_bf16x2(ry * fmaf(kx, bf16_lo(xw[e]), __uint_as_float(yv[q])),
                                 ry * fmaf(kx, bf16_hi(xw[e]), __uint_as_float(yv[q + 1])));
            }
            *px = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(bar_id, 128);
      if (et == 0) {
        const int nbox = Q >= 128 ? 4 : Q / 32;  // 32-token boxes of valid rows
        const int tok0 = id.c * Q + id.t * 128;
        for (int sb = 0; sb < nbox; ++sb) {
          if constexpr (C::kTF32) {
            tma_store_3d(&ymap, xy + sb * 4096, h * d.P, tok0 + 32 * sb, id.b);
            tma_store_3d(&ymap, xy + 16384 + sb * 4096, h * d.P + 32, tok0 + 32 * sb, id.b);
          } else {
            tma_store_3d(&ymap, xy + sb * 4096, h * d.P, tok0 + 32 * sb, id.b);
          }
        }
        tma_store_commit();
        tma_store_wait_read();  // the X block may be refilled once the stores have read it
      }
      mbar_arrive(&xempty[xs_last]);
    }
  }
  if (!ok) atomicExch(status, static_cast<int>(SSD_ERR_DEVICE_TIMEOUT));
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");  // this thread's TMA stores are complete
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
  }
  return n;
}

template <typename T>
cudaError_t launch_impl(const Dims& d, const ComputeOutMaps& maps, const float* D, const void* x, void* y,
                        const Work& w, uint64_t spin_ns, cudaStream_t stream, bool dependent) {
  using C = OutCfg<T>;
  const size_t smem = 1024 + out_smem_layout<T>().total;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(compute_out_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    // the register split assumes the compiled count; any other count is refused here
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, compute_out_kernel<T>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != static_cast<int>(kRegLaunch)) return cudaErrorInvalidConfiguration;
    configured = true;
  }
  const int ntile = d.Q >= 128 ? d.Q / 128 : 1;
  const long long ntiles = static_cast<long long>(d.B) * d.nc * ntile * (d.H / 2);
  const int grid = static_cast<int>(ntiles < sm_count() ? ntiles : sm_count());
  (void)y;  // written through maps.y
  // the D*x term reads x from the X blocks in shared memory; x itself only for rows whose rescaled copy is tiny
  return launch_k(compute_out_kernel<T>, dim3(grid), dim3(C::kThreads), smem, stream, dependent, maps.cm, maps.bm,
                  maps.hp, maps.x, maps.y, d, static_cast<const float*>(w.cumsum), static_cast<const float*>(w.dt_t), D,
                  static_cast<const T*>(x), w.status, spin_ns);
}

}  // namespace

cudaError_t launch_compute_out(const Dims& d, bool bf16, const ComputeOutMaps& maps, const float* D, const void* x,
                               void* y, const Work& w, uint64_t spin_ns, cudaStream_t stream, bool dependent) {
  return bf16 ? launch_impl<__nv_bfloat16>(d, maps, D, x, y, w, spin_ns, stream, dependent)
              : launch_impl<float>(d, maps, D, x, y, w, spin_ns, stream, dependent);
}

}  // namespace ssd
