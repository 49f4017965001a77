// Step 2 of the SSD forward: each chunk's contribution to the state, on the
// fifth-generation tensor cores.
//
// "Jane Street ML Engineers Map Mamba-2 Recurrent State Computation to Tensor
// Cores with cuTile", jump-formula paragraph: without decay the state jumps by
// B X^T over a chunk, one matrix product; with decay the rows are first
// multiplied by exponentials of log-space sums, which keeps it one product.
// Per (batch b, chunk c, head h):
//
//     S_c[p][n] = sum_j w_j x_j[p] b_j[n],   w_j = exp(G_last - G_j) * dt_j  (<= dt_j)
//
// GB300 mapping.  One CTA per (b, c, pair of heads of one group).  The MMA is
// D[M = 128][N = dstate] = X~^T B: M stacks the two heads' 64 p-rows (x keeps
// (h, p) contiguous, so one TMA box row covers both), K runs over the chunk's
// tokens, and the group's B tile is the shared N-side operand.  Both operands
// come straight from the token-major global layouts, so both are MN-major in
// shared memory (128-byte swizzle, TMA-written).  S_c leaves through shared
// memory and TMA stores, in fp32 for fp32 inputs and in bf16 for bf16 inputs
// (its rounding, 2^-9 relative, is far inside the bf16 tolerance and halves
// the bytes this kernel writes and the state pass reads).  The head-dependent token
// weights w_j are applied in shared memory, in place, between the TMA landing
// and the MMA -- a row of a 128-byte swizzle atom is one token of one head, so
// the swizzle never moves data across rows.  The fp32 accumulator lives in
// tensor memory (dstate columns) and is drained by tcgen05.ld.
//
// fp32 inputs run the MMA as TF32.  An MN-major TF32 operand is read in the
// 128-byte swizzle of 32-byte atoms, so the fp32 tensor maps write that layout
// and both operands stay MN-major, as in bf16; the x boxes are scaled (and
// rounded to TF32) in place.
//
// Warp roles (192 threads): warp 0 issues TMA, warp 1 owns TMEM and issues
// the MMAs (one thread), warps 2-5 compute the weights, transform each stage
// and write S_c.  On the staged schedule the weights start from the chunk's
// cumsum of dt*A, which warps 2 and 3 form here (one head each, the scan of
// chunk_scan.cuh) and write to the workspace for the kernels after this one,
// so that schedule has no chunk_cumsum launch.  A ring of 2-4 stages (as many as fit 96 KB; mbarriers full ->
// scaled -> empty) pipelines the 32-token stages.  All waits are bounded
// (device-timeout status, no hang).
#include "chunk_scan.cuh"
#include "ptx.cuh"
#include "ssd_internal.cuh"

namespace ssd {
namespace {

template <typename T>
struct StateCfg {
  static constexpr bool kTF32 = sizeof(T) == 4;
  static constexpr int kAtom = 128 / static_cast<int>(sizeof(T));  // elements per 128-B row
  static constexpr int kTokens = 32;                                // tokens per stage
  static constexpr int kKStep = kTF32 ? 8 : 16;                     // K of one MMA
  static constexpr int kBox = kTokens * 128;                        // one TMA box, bytes
  static constexpr int kABoxes = 128 / kAtom;                       // boxes spanning M = 128
  static constexpr int kABytes = kABoxes * kBox;
  static constexpr int kMaxStages = 4;
  static constexpr int kRingBytes = 96 * 1024;  // two CTAs per SM: each keeps its ring within 96 KB
  static constexpr int kThreads = 192;
};

__host__ __device__ inline uint32_t state_stage_bytes(int N, int atom, int box, int abytes) {
  return static_cast<uint32_t>(abytes + (N / atom) * box);
}

// Stages that fit the ring budget (2..4).
__host__ __device__ inline int state_stages(uint32_t stage_bytes, int ring_bytes, int max_stages) {
  const int n = ring_bytes / static_cast<int>(stage_bytes);
  return n < 2 ? 2 : (n > max_stages ? max_stages : n);
}

template <typename T>
__global__ void __launch_bounds__(StateCfg<T>::kThreads, 2)
    chunk_state_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap bmap,
                       const __grid_constant__ CUtensorMap smap, Dims d, float* __restrict__ cumsum,
                       float* __restrict__ dt_t, const float* __restrict__ dt, const float* __restrict__ A,
                       int* chain, int nchain, int* status, uint64_t spin_ns) {
  using C = StateCfg<T>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int N = d.N, Q = d.Q;
  const int h0 = blockIdx.x * 2;
  const int c = blockIdx.y, b = blockIdx.z;
  const int g = h0 / (d.H / d.G);
  const int bBoxes = N / C::kAtom;
  const uint32_t stage_bytes = state_stage_bytes(N, C::kAtom, C::kBox, C::kABytes);
  const int NS = state_stages(stage_bytes, C::kRingBytes, C::kMaxStages);
  float* w_s = reinterpret_cast<float*>(smem + NS * stage_bytes);  // [2][Q]
  uint64_t* bars = reinterpret_cast<uint64_t*>(w_s + 2 * Q);
  uint64_t* full = bars;
  uint64_t* scaled = bars + NS;
  uint64_t* empty = bars + 2 * NS;
  uint64_t* accum = bars + 3 * NS;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(accum + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nstages = Q / C::kTokens;
  const uint32_t tmem_cols = static_cast<uint32_t>(N);  // the accumulator

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&scaled[s], 128);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accum, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&xmap);
    tma_prefetch_desc(&bmap);
    tma_prefetch_desc(&smap);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, tmem_cols);
    tmem_relinquish();
  }
  grid_dep_wait();  // the kernel before (chunk_cumsum, when it ran) is complete from here on
  grid_dep_launch();
  // As the call's first kernel (dt non-null, nchain >= 0), CTA (0, 0, 0) clears the status
  // word and the first `nchain` one-pass counters.
  if (dt && nchain >= 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) {
    if (threadIdx.x == 0) *status = 0;
    for (int k = threadIdx.x; k < nchain; k += C::kThreads) chain[k] = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  bool ok = true;

  if (warp == 0) {
    if (lane == 0) {
      for (int it = 0; it < nstages; ++it) {
        const int s = it % NS, r = it / NS;
        if (r > 0 && !mbar_wait(&empty[s], (r - 1) & 1, spin_ns)) {
          ok = false;
          break;
        }
        uint8_t* sa = smem + s * stage_bytes;
        uint8_t* sb = sa + C::kABytes;
        mbar_arrive_expect_tx(&full[s], stage_bytes);
        const int tok = c * Q + it * C::kTokens;
        for (int k = 0; k < C::kABoxes; ++k)
          tma_load_3d(sa + k * C::kBox, &xmap, &full[s], h0 * d.P + k * C::kAtom, tok, b);
        for (int k = 0; k < bBoxes; ++k)
          tma_load_4d(sb + k * C::kBox, &bmap, &full[s], k * C::kAtom, g, tok, b);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // both operands MN-major
      const uint32_t idesc = idesc_f32acc(C::kTF32 ? 2u : 1u, 128u, static_cast<uint32_t>(N), 1u, 1u);
      for (int it = 0; it < nstages; ++it) {
        const int s = it % NS, r = it / NS;
        if (!mbar_wait(&scaled[s], r & 1, spin_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + s * stage_bytes);
        const uint32_t sb = sa + C::kABytes;
#pragma unroll
        for (int k = 0; k < C::kTokens / C::kKStep; ++k) {
          uint64_t ad, bd;
          if constexpr (C::kTF32) {
            // MN-major, 128-B swizzle of 32-B atoms: a K step is 8 token rows (1 KB);
            // LBO = stride between 32-element column blocks (one TMA box), SBO = 4-row groups.
            ad = sdesc_sw128_a32(sa + k * 1024, C::kBox, 512);
            bd = sdesc_sw128_a32(sb + k * 1024, C::kBox, 512);
          } else {
            // MN-major, 128-B swizzle: LBO = stride between 128-B atom columns
            // (one TMA box), SBO = stride between 8-row groups along K.
            ad = sdesc_sw128(sa + k * C::kKStep * 128, C::kBox, 1024);
            bd = sdesc_sw128(sb + k * C::kKStep * 128, C::kBox, 1024);
          }
          mma_ss<C::kTF32>(tmem, ad, bd, idesc, (it | k) != 0 ? 1u : 0u);
        }
        mma_commit(&empty[s]);
      }
      mma_commit(accum);
    }
  } else {
    // token weights w_j = exp(G_last - G_j) * dt_j for both heads (exponent <= 0), while the
    // producer's first loads are in flight
    if (dt) {
      // The chunk's cumsum formed here (dt non-null; one piece, Q <= 256): one warp per head of
      // the pair, the rows written for state_passing and compute_out exactly as chunk_cumsum
      // writes them.
      if (warp == 2 || warp == 3) {
        const int hl = warp - 2, h = h0 + hl;
        const int per = Q / 32;  // 2, 4 or 8 tokens per lane
        const int64_t row = (static_cast<int64_t>(b) * d.H + h) * d.Lp + static_cast<int64_t>(c) * Q;
        float v[8], gv[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int tok = c * Q + lane * per + k;
          v[k] = (k < per && tok < d.L) ? dt[(static_cast<int64_t>(b) * d.L + tok) * d.H + h] : 0.f;
        }
        float carry = 0.f;
        cumsum_piece(v, per, A[h], carry, gv);
        // the chunk's last value (per is 2, 4 or 8; constant indices keep gv in registers)
        const float gl = per == 2 ? gv[1] : per == 4 ? gv[3] : gv[7];
        const float glast = __shfl_sync(0xffffffffu, gl, 31);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (k < per) {
            const int j = lane * per + k;
            cumsum[row + j] = gv[k];
            dt_t[row + j] = v[k];
            w_s[hl * Q + j] = expf(glast - gv[k]) * v[k];
          }
        }
      }
    } else {
      // chunk_cumsum's rows, read-only here (non-coherent loads, several in flight)
#pragma unroll 4
      for (int idx = threadIdx.x - 64; idx < 2 * Q; idx += 128) {
        const int hl = idx / Q, j = idx % Q;
        const int64_t row = (static_cast<int64_t>(b) * d.H + h0 + hl) * d.Lp + static_cast<int64_t>(c) * Q;
        w_s[idx] = expf(__ldg(cumsum + row + Q - 1) - __ldg(cumsum + row + j)) * __ldg(dt_t + row + j);
      }
    }
    named_bar_sync(1, 128);  // w_s complete for the four scaling warps
    const int et = threadIdx.x - 64;
    for (int it = 0; it < nstages; ++it) {
      const int s = it % NS, r = it / NS;
      if (!mbar_wait(&full[s], r & 1, spin_ns)) {
        ok = false;
        break;
      }
      uint8_t* sa = smem + s * stage_bytes;
      if constexpr (C::kTF32) {
        // x scaled in place: thread = token row (et % 32) of A box et / 32 (32 p of one head);
        // the row's 16-byte chunks go in a per-row rotated order so that a warp's accesses
        // spread over all banks (one scale for the whole row)
        const int box = et >> 5, row = et & 31;
        const float w = w_s[(box >> 1) * Q + it * C::kTokens + row];
        float4* rp = reinterpret_cast<float4*>(sa + box * C::kBox + row * 128);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          float4* cp = rp + (k ^ (row & 7));
          float4 v = *cp;
          v.x = round_tf32(v.x * w);
          v.y = round_tf32(v.y * w);
          v.z = round_tf32(v.z * w);
          v.w = round_tf32(v.w * w);
          *cp = v;
        }
      } else {
        constexpr int kChunks = C::kABytes / 16;
#pragma unroll 4
        for (int q = et; q < kChunks; q += 128) {
          const int box = q / (C::kTokens * 8);
          const int row = (q >> 3) % C::kTokens;
          const int hl = box / (C::kABoxes / 2);
          const float w = w_s[hl * Q + it * C::kTokens + row];
          uint4* p = reinterpret_cast<uint4*>(sa + q * 16);
          uint4 v = *p;
          v.x = pack_bf16x2(bf16_lo(v.x) * w, bf16_hi(v.x) * w);
          v.y = pack_bf16x2(bf16_lo(v.y) * w, bf16_hi(v.y) * w);
          v.z = pack_bf16x2(bf16_lo(v.z) * w, bf16_hi(v.z) * w);
          v.w = pack_bf16x2(bf16_lo(v.w) * w, bf16_hi(v.w) * w);
          *p = v;
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&scaled[s]);
    }
    if (ok && !mbar_wait(accum, 0, spin_ns)) ok = false;
    tc_fence_after();
    // drain: TMEM lane = 64 * (head within the pair) + p, column = n.  Rows go
    // to shared memory (the pipeline stages are idle now) in the 128-B swizzled
    // box layout of the states tensor map -- fp32, or bf16 for bf16 inputs --
    // and leave with TMA tensor stores, so the writes are whole lines.
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    constexpr int kSAtom = C::kAtom;  // states elements per 128-B box row (same dtype as the inputs)
    uint8_t* stage = smem;
    auto put = [&](int n0, const uint32_t (&v)[32]) {
      uint8_t* box = stage + (n0 / kSAtom) * (128 * 128) + row * 128;
      if constexpr (C::kTF32) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          *reinterpret_cast<uint4*>(box + ((k ^ (row & 7)) << 4)) = make_uint4(v[4 * k], v[4 * k + 1], v[4 * k + 2],
                                                                                 v[4 * k + 3]);
      } else {
        const int c0 = ((n0 / 32) & 1) * 4;  // 32 bf16 fill half of a 128-B row
#pragma unroll
        for (int k = 0; k < 4; ++k)
          *reinterpret_cast<uint4*>(box + (((c0 + k) ^ (row & 7)) << 4)) =
              make_uint4(pack_bf16x2(__uint_as_float(v[8 * k]), __uint_as_float(v[8 * k + 1])),
                         pack_bf16x2(__uint_as_float(v[8 * k + 2]), __uint_as_float(v[8 * k + 3])),
                         pack_bf16x2(__uint_as_float(v[8 * k + 4]), __uint_as_float(v[8 * k + 5])),
                         pack_bf16x2(__uint_as_float(v[8 * k + 6]), __uint_as_float(v[8 * k + 7])));
      }
    };
    // in rounds of as many 16 KB boxes as the (now idle) ring holds; a round's
    // stores have read the boxes before the next round overwrites them
    const int nbox = N / kSAtom;
    const int per_round = static_cast<int>(NS * stage_bytes / (128 * 128)) < nbox
                              ? static_cast<int>(NS * stage_bytes / (128 * 128)) : nbox;
    const int cols_round = per_round * kSAtom;  // a multiple of 64
    for (int c0 = 0; c0 < N; c0 += cols_round) {
      const int c1 = c0 + cols_round < N ? c0 + cols_round : N;
      for (int n0 = c0; n0 < c1; n0 += 64) {
        uint32_t va[32], vb[32];
        tmem_ld32(lane_addr + static_cast<uint32_t>(n0), va);
        tmem_ld32(lane_addr + static_cast<uint32_t>(n0 + 32), vb);
        tmem_ld_wait();
        put(n0 - c0, va);
        put(n0 - c0 + 32, vb);
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (threadIdx.x == 64) {
        const int row0 = ((b * d.nc + c) * d.H + h0) * d.P;
        for (int k = 0; k < (c1 - c0) / kSAtom; ++k)
          tma_store_2d(&smap, stage + k * (128 * 128), c0 + k * kSAtom, row0);
        tma_store_commit();
        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      }
      named_bar_sync(1, 128);
    }
    if (threadIdx.x == 64) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
  if (!ok) atomicExch(status, static_cast<int>(SSD_ERR_DEVICE_TIMEOUT));
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

template <typename T>
cudaError_t launch_impl(const Dims& d, const ChunkStateMaps& maps, const Work& w, uint64_t spin_ns,
                        cudaStream_t stream, bool dependent, const float* dt, const float* A, int nchain) {
  using C = StateCfg<T>;
  const uint32_t stage_bytes = state_stage_bytes(d.N, C::kAtom, C::kBox, C::kABytes);
  const int ns = state_stages(stage_bytes, C::kRingBytes, C::kMaxStages);
  const size_t smem = 1024 + ns * stage_bytes + 2 * d.Q * sizeof(float) + (3 * ns + 1) * sizeof(uint64_t) + 16;
  static size_t configured = 0;
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(chunk_state_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  const dim3 grid(d.H / 2, d.nc, d.B);
  if (dt && d.Q > 256) return cudaErrorInvalidValue;  // the in-kernel cumsum takes one piece
  return launch_k(chunk_state_kernel<T>, grid, dim3(C::kThreads), smem, stream, dependent, maps.x, maps.bm, maps.s, d,
                  w.cumsum, w.dt_t, dt, A, w.counter, nchain, w.status, spin_ns);
}

}  // namespace

cudaError_t launch_chunk_state(const Dims& d, bool bf16, const ChunkStateMaps& maps, const Work& w,
                               uint64_t spin_ns, cudaStream_t stream, bool dependent, const float* dt,
                               const float* A, int nchain) {
  // fp32 at dstate 256 with the cumsum formed in-kernel: one persistent CTA per SM walking its
  // units with two accumulators (chunk_state_persistent.cu)
  if (!bf16 && d.N == 256 && dt && d.Q <= 256)
    return launch_chunk_state_persistent(d, maps, w, spin_ns, stream, dependent, dt, A, nchain);
  return bf16 ? launch_impl<__nv_bfloat16>(d, maps, w, spin_ns, stream, dependent, dt, A, nchain)
              : launch_impl<float>(d, maps, w, spin_ns, stream, dependent, dt, A, nchain);
}

}  // namespace ssd
