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
// Per (batch b, chunk c, head h, 128-row tile t of the chunk), rows i in the
// tile, columns j in 128-wide blocks jb <= t:
//
//     Y_off   = C_t hprev^T                          (K = dstate)
//     CB_jb   = C_t B_jb^T                           (K = dstate)
//     M_jb    = CB_jb o [j <= i] exp(G_i - G_j) dt_j (registers, -> TMEM)
//     Y_intra = sum_jb M_jb X_jb                     (A = M from TMEM, K = 128)
//     y_i     = exp(G_i) Y_off_i + Y_intra_i + D_h x_i
//
// Tensor memory (256 columns): [0,64) Y_off, [64,128) Y_intra, [128,256) CB,
// overwritten in place by M (packed bf16 pairs in the bf16 path).  The
// exponentials are factored so that every factor is <= 1: for a 32-column
// strip entirely left of row i, exp(G_i - G_j) = exp(G_i - G_e) exp(G_e - G_j)
// with e the strip's last column (one exp per row and strip plus a per-column
// table); only the 32 x 32 blocks on the diagonal take one exp per element,
// behind the causal select.
//
// TF32 (fp32 inputs) needs K-major shared-memory operands.  The C, B and state
// tiles already have dstate (the K of their products) along the rows; the X
// tiles of the intra-chunk product (K = tokens) arrive as 32 x 32 boxes that
// the epilogue warps transpose in place before the first use.  bf16 reads X
// MN-major directly.
//
// Warp roles (192 threads): warp 0 TMA, warp 1 TMEM owner + MMA issuer,
// warps 2-5 mask pass and epilogue (TMEM lane quadrant = warp % 4).  C, B and
// the entering state stream through a 2-slot ring in 128-byte K-slices; the
// X tiles the intra-chunk product needs are loaded once.  Bounded waits.
#include "ptx.cuh"
#include "ssd_internal.cuh"
#include "tile_transpose.cuh"

namespace ssd {
namespace {

template <typename T>
struct OutCfg {
  static constexpr bool kTF32 = sizeof(T) == 4;
  static constexpr int kAtom = 128 / static_cast<int>(sizeof(T));  // elements per 128-B row
  static constexpr int kRows = 128;                                 // tile rows / block columns
  static constexpr int kCBox = kRows * 128;                         // 128 rows x 128 B
  static constexpr int kHBox = 64 * 128;                            // 64 state rows x 128 B
  static constexpr int kSlot = 2 * kCBox + kHBox;
  static constexpr int kXBoxes = 64 / kAtom;                        // x tile: 64 p = 1 or 2 atoms
  static constexpr int kXTile = kXBoxes * kCBox;                    // 128 tokens x 64 p
  static constexpr int kKStepMN = kTF32 ? 8 : 16;                  // tokens per MMA (intra product)
  static constexpr int kStages = 2;
  static constexpr int kThreads = 192;
  static constexpr uint32_t kColYoff = 0, kColYint = 64, kColCB = 128, kTmemCols = 256;
};

struct OutSmem {
  uint32_t slots, xt, gs, dts, vref, bars, holder, total;
};

template <typename T>
__host__ __device__ inline OutSmem out_smem_layout(int ntile) {
  using C = OutCfg<T>;
  OutSmem s{};
  s.slots = 0;
  s.xt = s.slots + C::kStages * C::kSlot;
  s.gs = s.xt + ntile * C::kXTile;
  s.dts = s.gs + ntile * 128 * 4;
  s.vref = s.dts + ntile * 128 * 4;
  s.bars = s.vref + ntile * 128 * 4;
  s.holder = s.bars + (2 * C::kStages + 6) * 8;
  s.total = s.holder + 16;
  return s;
}

template <typename T>
__global__ void __launch_bounds__(OutCfg<T>::kThreads, 1)
    compute_out_kernel(const __grid_constant__ CUtensorMap cmap, const __grid_constant__ CUtensorMap bmap,
                       const __grid_constant__ CUtensorMap hmap, const __grid_constant__ CUtensorMap xmap, Dims d,
                       const float* __restrict__ cumsum, const float* __restrict__ dt_t,
                       const float* __restrict__ Dvec, T* __restrict__ y, int* status, uint64_t spin_ns) {
  using C = OutCfg<T>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int Q = d.Q;
  const int ntile = Q >= 128 ? Q / 128 : 1;
  const int t = blockIdx.x % ntile;
  const int h = blockIdx.x / ntile;
  const int c = blockIdx.y, b = blockIdx.z;
  const int g = h / (d.H / d.G);
  const int i0 = t * 128;
  const int njb = t + 1;
  const int NB = d.N / C::kAtom;
  const OutSmem L = out_smem_layout<T>(ntile);
  float* gs = reinterpret_cast<float*>(smem + L.gs);
  float* dts = reinterpret_cast<float*>(smem + L.dts);
  float* vref = reinterpret_cast<float*>(smem + L.vref);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::kStages;
  uint64_t* xfull = bars + 2 * C::kStages;
  uint64_t* cbfull = xfull + 1;
  uint64_t* mready = xfull + 2;
  uint64_t* mfree = xfull + 3;
  uint64_t* yfull = xfull + 4;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L.holder);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(xfull, 1);
    mbar_init(cbfull, 1);
    mbar_init(mready, 128);
    mbar_init(mfree, 1);
    mbar_init(yfull, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&cmap);
    tma_prefetch_desc(&bmap);
    tma_prefetch_desc(&hmap);
    tma_prefetch_desc(&xmap);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  bool ok = true;

  if (warp == 0) {
    if (lane == 0) {
      uint8_t* xt = smem + L.xt;
      mbar_arrive_expect_tx(xfull, static_cast<uint32_t>(njb * C::kXTile));
      for (int jb = 0; jb < njb; ++jb) {
        if constexpr (C::kTF32) {
          // 32-token x 32-p boxes; box (s, half) at s * 8 KB + half * 4 KB so that,
          // once transposed, each 32-token K block is one 64-row K-major tile
          for (int sb = 0; sb < 4; ++sb)
            for (int hf = 0; hf < 2; ++hf)
              tma_load_3d(xt + jb * C::kXTile + sb * 8192 + hf * 4096, &xmap, xfull, h * d.P + hf * 32,
                          c * Q + jb * 128 + sb * 32, b);
        } else {
          tma_load_3d(xt + jb * C::kXTile, &xmap, xfull, h * d.P, c * Q + jb * 128, b);
        }
      }
      const int hrow = ((b * d.nc + c) * d.H + h) * d.P;
      int it = 0;
      for (int jb = 0; jb < njb && ok; ++jb) {
        for (int nb = 0; nb < NB; ++nb, ++it) {
          const int s = it % C::kStages, r = it / C::kStages;
          if (r > 0 && !mbar_wait(&empty[s], (r - 1) & 1, spin_ns)) {
            ok = false;
            break;
          }
          uint8_t* slot = smem + L.slots + s * C::kSlot;
          mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(2 * C::kCBox + (jb == 0 ? C::kHBox : 0)));
          tma_load_4d(slot, &cmap, &full[s], nb * C::kAtom, g, c * Q + i0, b);
          tma_load_4d(slot + C::kCBox, &bmap, &full[s], nb * C::kAtom, g, c * Q + jb * 128, b);
          if (jb == 0) tma_load_2d(slot + 2 * C::kCBox, &hmap, &full[s], nb * C::kAtom, hrow);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t fmt = C::kTF32 ? 2u : 1u;
      const uint32_t id_yoff = idesc_f32acc(fmt, 128, 64, 0, 0);
      const uint32_t id_cb = idesc_f32acc(fmt, 128, 128, 0, 0);
      const uint32_t id_yint = idesc_f32acc(fmt, 128, 64, 0, C::kTF32 ? 0u : 1u);
      const uint32_t xt = smem_u32(smem + L.xt);
      int it = 0;
      for (int jb = 0; jb < njb && ok; ++jb) {
        if (jb > 0 && !mbar_wait(mfree, (jb - 1) & 1, spin_ns)) {
          ok = false;
          break;
        }
        for (int nb = 0; nb < NB; ++nb, ++it) {
          const int s = it % C::kStages, r = it / C::kStages;
          if (!mbar_wait(&full[s], r & 1, spin_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t slot = smem_u32(smem + L.slots + s * C::kSlot);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            // K-major, 128-B swizzle: K advances 32 B inside the atom row;
            // SBO = 1024 B between 8-row groups; LBO unused.
            const uint64_t ad = sdesc_sw128(slot + k * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(slot + C::kCBox + k * 32, 16, 1024);
            const uint32_t acc = (nb | k) != 0 ? 1u : 0u;
            if (jb == 0) {
              const uint64_t hd = sdesc_sw128(slot + 2 * C::kCBox + k * 32, 16, 1024);
              mma_ss<C::kTF32>(tmem + C::kColYoff, ad, hd, id_yoff, acc);
            }
            mma_ss<C::kTF32>(tmem + C::kColCB, ad, bd, id_cb, acc);
          }
          mma_commit(&empty[s]);
        }
        if (!ok) break;
        mma_commit(cbfull);
        if (!mbar_wait(mready, jb & 1, spin_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (jb == 0 && !mbar_wait(xfull, 0, spin_ns)) {
          ok = false;
          break;
        }
        const uint32_t xb = xt + jb * C::kXTile;
#pragma unroll 4
        for (int k = 0; k < 128 / C::kKStepMN; ++k) {
          uint64_t xd;
          if constexpr (C::kTF32) {
            // B = X^T block, K-major: 64 p-rows of 32 tokens per 8 KB block;
            // a K step of 8 tokens is 32 B along the row.
            xd = sdesc_sw128(xb + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024);
          } else {
            // B = X block, MN-major (p contiguous, one 128-B atom = 64 p):
            // SBO = 1024 B between 8-token groups.
            xd = sdesc_sw128(xb + k * C::kKStepMN * 128, C::kCBox, 1024);
          }
          mma_ts<C::kTF32>(tmem + C::kColYint, tmem + C::kColCB + k * 8, xd, id_yint, (jb | k) != 0 ? 1u : 0u);
        }
        mma_commit(mfree);
      }
      mma_commit(yfull);
    }
  } else {
    const int et = threadIdx.x - 64;
    const int64_t grow = (static_cast<int64_t>(b) * d.H + h) * d.Lp + static_cast<int64_t>(c) * Q;
    const int ncol = 128 * ntile;
    for (int j = et; j < ncol; j += 128) {
      const bool in = j < Q;
      gs[j] = cumsum[grow + (in ? j : Q - 1)];
      dts[j] = in ? dt_t[grow + j] : 0.f;
    }
    named_bar_sync(1, 128);
    for (int j = et; j < ncol; j += 128) vref[j] = expf(gs[j | 31] - gs[j]) * dts[j];
    named_bar_sync(1, 128);
    if constexpr (C::kTF32) {
      // flip the X boxes to K-major before the first intra-chunk product
      if (!mbar_wait(xfull, 0, spin_ns)) ok = false;
      uint8_t* xt = smem + L.xt;
      const int m = et & 63;
      for (int box0 = 0; box0 < njb * 8; box0 += 2) {
        uint8_t* bp = xt + (box0 + (et >> 6)) * 4096;
        float4 v[4];
        box_read_4x4(bp, m, v);
        named_bar_sync(1, 128);
        box_write_4x4_transposed(bp, m, v);
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 128);  // the D*x epilogue below reads other threads' writes
    }

    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // TMEM lane = tile row
    const int i = i0 + r;            // row within the chunk
    const float Gi = gs[i];
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;

    for (int jb = 0; jb < njb; ++jb) {
      if (!mbar_wait(cbfull, jb & 1, spin_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        const int j0 = jb * 128 + cc * 32;
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + C::kColCB + cc * 32, v);
        tmem_ld_wait();
        float m[32];
        if (j0 + 31 < i) {  // strip strictly left of the diagonal (warp-uniform)
          const float u = expf(Gi - gs[j0 + 31]);
#pragma unroll
          for (int q = 0; q < 32; ++q) m[q] = __uint_as_float(v[q]) * u * vref[j0 + q];
        } else if (j0 > i) {  // strip strictly right of the diagonal (warp-uniform)
#pragma unroll
          for (int q = 0; q < 32; ++q) m[q] = 0.f;
        } else {  // the 32 x 32 block on the diagonal: select, then exp (exponent <= 0)
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            const int j = j0 + q;
            m[q] = j <= i ? __uint_as_float(v[q]) * expf(Gi - gs[j]) * dts[j] : 0.f;
          }
        }
        if constexpr (C::kTF32) {
          uint32_t o[32];
#pragma unroll
          for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(round_tf32(m[q]));
          tmem_st32(tmem + lane_base + C::kColCB + cc * 32, o);
        } else {
          uint32_t o[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) o[q] = pack_bf16x2(m[2 * q], m[2 * q + 1]);
          tmem_st16(tmem + lane_base + C::kColCB + cc * 16, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(mready);
    }

    if (ok && !mbar_wait(yfull, 0, spin_ns)) ok = false;
    tc_fence_after();
    const bool valid = (i < Q) && (c * Q + i < d.L);
    const float eGi = expf(Gi);
    const float Dh = Dvec[h];
    const uint8_t* xrow_base = smem + L.xt + t * C::kXTile;
    T* yrow = y + ((static_cast<int64_t>(b) * d.L + static_cast<int64_t>(c) * Q + i) * d.H + h) * d.P;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      uint32_t yo[32], yi[32];
      tmem_ld32(tmem + lane_base + C::kColYoff + half * 32, yo);
      tmem_ld32(tmem + lane_base + C::kColYint + half * 32, yi);
      tmem_ld_wait();
      float out[32];
      // x_i[p] for p = 32*half .. +31 from the x tile of this row block
      if constexpr (C::kTF32) {
        // transposed boxes: token r lives in K block r / 32, p in box half p / 32
        const uint8_t* bx = xrow_base + (r >> 5) * 8192 + half * 4096;
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          const float xf = *reinterpret_cast<const float*>(bx + box_t_offset(r & 31, q));
          out[q] = fmaf(eGi, __uint_as_float(yo[q]), __uint_as_float(yi[q])) + Dh * xf;
        }
      } else {
        // MN-major rows: token r is row r, p in 16-B chunks of 8
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int chunk = half * 4 + k;
          const uint4 xv = *reinterpret_cast<const uint4*>(xrow_base + r * 128 + ((chunk ^ (r & 7)) << 4));
          const float xf[8] = {bf16_lo(xv.x), bf16_hi(xv.x), bf16_lo(xv.y), bf16_hi(xv.y),
                               bf16_lo(xv.z), bf16_hi(xv.z), bf16_lo(xv.w), bf16_hi(xv.w)};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int q = k * 8 + e;
            out[q] = fmaf(eGi, __uint_as_float(yo[q]), __uint_as_float(yi[q])) + Dh * xf[e];
          }
        }
      }
      if (valid) {
        if constexpr (C::kTF32) {
          float4* o4 = reinterpret_cast<float4*>(yrow + half * 32);
#pragma unroll
          for (int k = 0; k < 8; ++k) o4[k] = make_float4(out[4 * k], out[4 * k + 1], out[4 * k + 2], out[4 * k + 3]);
        } else {
          uint4* o4 = reinterpret_cast<uint4*>(yrow + half * 32);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            o4[k] = make_uint4(pack_bf16x2(out[8 * k], out[8 * k + 1]), pack_bf16x2(out[8 * k + 2], out[8 * k + 3]),
                               pack_bf16x2(out[8 * k + 4], out[8 * k + 5]),
                               pack_bf16x2(out[8 * k + 6], out[8 * k + 7]));
        }
      }
    }
  }
  if (!ok) atomicExch(status, static_cast<int>(SSD_ERR_DEVICE_TIMEOUT));
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <typename T>
cudaError_t launch_impl(const Dims& d, const ComputeOutMaps& maps, const float* D, void* y, const Work& w,
                        uint64_t spin_ns, cudaStream_t stream) {
  using C = OutCfg<T>;
  const int ntile = d.Q >= 128 ? d.Q / 128 : 1;
  const size_t smem = 1024 + out_smem_layout<T>(ntile).total;
  static size_t configured = 0;
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(compute_out_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  const dim3 grid(ntile * d.H, d.nc, d.B);
  compute_out_kernel<T><<<grid, C::kThreads, smem, stream>>>(maps.cm, maps.bm, maps.hp, maps.x, d, w.cumsum,
                                                             w.dt_t, D, static_cast<T*>(y), w.status, spin_ns);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_compute_out(const Dims& d, bool bf16, const ComputeOutMaps& maps, const float* D, void* y,
                               const Work& w, uint64_t spin_ns, cudaStream_t stream) {
  return bf16 ? launch_impl<__nv_bfloat16>(d, maps, D, y, w, spin_ns, stream)
              : launch_impl<float>(d, maps, D, y, w, spin_ns, stream);
}

}  // namespace ssd
