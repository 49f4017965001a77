// Step 2 of the SSD forward, persistent form for fp32 inputs at dstate 256.
//
// Same computation as chunk_state.cu ("Jane Street ML Engineers Map Mamba-2
// Recurrent State Computation to Tensor Cores with cuTile", jump-formula
// paragraph): per (batch b, chunk c, head pair), S_c[p][n] = sum_j w_j x_j[p]
// b_j[n] with w_j = exp(G_last - G_j) dt_j, one TF32 MMA chain D[M = 128 (h, p)]
// [N = 256] per unit, both operands MN-major in the 128-byte swizzle of 32-byte
// atoms, straight from TMA.
//
// At dstate 256 one unit's accumulator takes 256 tensor-memory columns, and a
// CTA per unit pays its start-up (barriers, tensor memory, the token weights,
// the first TMA round trip) and its accumulator drain around only eight
// 32-token stages.  Here one CTA per SM walks its units (unit = blockIdx.x +
// k * gridDim.x) with two accumulators (all 512 columns), so the TMA ring
// streams from one unit into the next and a unit's drain runs beside the next
// unit's products:
//
//   warp 0      TMA: x (4 boxes of 32 (h, p)) and Bm (8 boxes of 32 n) per stage
//   warp 1      tensor memory; the MMAs (one thread), unit k into accumulator k % 2
//   warps 2-5   scale each stage's x rows by w_j in place (rounded to TF32)
//   warps 6-9   the token weights of the next unit (its chunk cumsum, written
//               to the workspace as chunk_cumsum would), then the drain of the
//               finished accumulator through two 16 KB staging boxes and TMA
//               stores of the states
//
// Barriers: full/scaled/empty per ring stage; accfull/accfree per accumulator;
// wready/wfree per weight buffer.  Every wait is bounded; on expiry the CTA
// records SSD_ERR_DEVICE_TIMEOUT, waits (bounded) for its copies in flight,
// frees its tensor memory and exits.
#include "chunk_scan.cuh"
#include "ptx.cuh"
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kTokens = 32;                 // tokens per stage
constexpr int kAtom = 32;                   // fp32 values per 128-byte row
constexpr int kBox = kTokens * 128;         // one TMA box: 32 rows of 128 B
constexpr int kN = 256;                     // dstate
constexpr int kABoxes = 128 / kAtom;        // (head, p) columns of a pair: 4 boxes
constexpr int kBBoxes = kN / kAtom;         // 8 boxes
constexpr int kStage = (kABoxes + kBBoxes) * kBox;  // 48 KB
constexpr int kStages = 3;
constexpr int kStaging = 2 * 128 * 128;     // two 16 KB boxes of 128 state rows x 32 n
constexpr int kThreads = 320;
constexpr uint32_t kDrainBar = 2;           // named barrier of the drain warps

struct PersistSmem {
  uint32_t ring, staging, w, bars, holder, total;
};

__host__ __device__ constexpr PersistSmem persist_layout(int Q) {
  PersistSmem s{};
  s.ring = 0;
  s.staging = kStages * kStage;
  s.w = s.staging + kStaging;
  s.bars = s.w + static_cast<uint32_t>(2 * 2 * Q * 4);  // two buffers of [2 heads][Q]
  s.holder = s.bars + (3 * kStages + 8) * 8;
  s.total = s.holder + 16;
  return s;
}

__global__ void __launch_bounds__(kThreads, 1)
    chunk_state_persistent_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap bmap,
                                  const __grid_constant__ CUtensorMap smap, Dims d, float* __restrict__ cumsum,
                                  float* __restrict__ dt_t, const float* __restrict__ dt, const float* __restrict__ A,
                                  int* chain, int nchain, int* status, uint64_t spin_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int Q = d.Q;
  const PersistSmem L = persist_layout(Q);
  float* w_s = reinterpret_cast<float*>(smem + L.w);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* full = bars;
  uint64_t* scaled = bars + kStages;
  uint64_t* empty = bars + 2 * kStages;
  uint64_t* accfull = bars + 3 * kStages;  // [2]
  uint64_t* accfree = accfull + 2;         // [2]
  uint64_t* wready = accfull + 4;          // [2]
  uint64_t* wfree = accfull + 6;           // [2]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L.holder);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hp = d.H / 2;
  const int units = hp * d.nc * d.B;
  const int nstage = Q / kTokens;  // stages per unit
  const int nmine = units > static_cast<int>(blockIdx.x)
                        ? (units - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) / gridDim.x
                        : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&scaled[s], 128);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&accfull[a], 1);
      mbar_init(&accfree[a], 128);
      mbar_init(&wready[a], 128);
      mbar_init(&wfree[a], 128);
    }
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&xmap);
    tma_prefetch_desc(&bmap);
    tma_prefetch_desc(&smap);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  grid_dep_wait();
  grid_dep_launch();
  // as the call's first kernel: clear the status word and the one-pass counters
  if (nchain >= 0 && blockIdx.x == 0) {
    if (threadIdx.x == 0) *status = 0;
    for (int k = threadIdx.x; k < nchain; k += kThreads) chain[k] = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  bool ok = true;

  // unit k of this CTA: (batch, chunk, head pair)
  auto unit = [&](int k, int& b, int& c, int& h0) {
    int u = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
    h0 = 2 * (u % hp);
    u /= hp;
    c = u % d.nc;
    b = u / d.nc;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int it = 0;
      for (int k = 0; k < nmine && ok; ++k) {
        int b, c, h0;
        unit(k, b, c, h0);
        const int g = h0 / (d.H / d.G);
        for (int st = 0; st < nstage; ++st, ++it) {
          const int s = it % kStages, r = it / kStages;
          if (r > 0 && !mbar_wait(&empty[s], (r - 1) & 1, spin_ns)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + L.ring + s * kStage;
          uint8_t* sb = sa + kABoxes * kBox;
          mbar_arrive_expect_tx(&full[s], kStage);
          const int tok = c * Q + st * kTokens;
          for (int j = 0; j < kABoxes; ++j) tma_load_3d(sa + j * kBox, &xmap, &full[s], h0 * d.P + j * kAtom, tok, b);
          for (int j = 0; j < kBBoxes; ++j) tma_load_4d(sb + j * kBox, &bmap, &full[s], j * kAtom, g, tok, b);
        }
      }
      if (!ok) {  // wait (bounded) for the copies still in flight before the CTA exits
        for (int i = max(0, it - kStages); i < it; ++i) mbar_wait(&full[i % kStages], (i / kStages) & 1, spin_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f32acc(2u, 128u, static_cast<uint32_t>(kN), 1u, 1u);  // both MN-major
      int it = 0;
      for (int k = 0; k < nmine && ok; ++k) {
        const int a = k & 1;
        if (k >= 2 && !mbar_wait(&accfree[a], ((k >> 1) - 1) & 1, spin_ns)) {  // unit k - 2 drained
          ok = false;
          break;
        }
        tc_fence_after();
        for (int st = 0; st < nstage; ++st, ++it) {
          const int s = it % kStages, r = it / kStages;
          if (!mbar_wait(&scaled[s], r & 1, spin_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + L.ring + s * kStage);
          const uint32_t sb = sa + kABoxes * kBox;
#pragma unroll
          for (int kk = 0; kk < kTokens / 8; ++kk) {
            // a K step is 8 token rows (1 KB); LBO = one box (the next 32 columns), SBO = 4 rows
            const uint64_t ad = sdesc_sw128_a32(sa + kk * 1024, kBox, 512);
            const uint64_t bd = sdesc_sw128_a32(sb + kk * 1024, kBox, 512);
            mma_ss<true>(tmem + static_cast<uint32_t>(a * kN), ad, bd, idesc, (st | kk) != 0 ? 1u : 0u);
          }
          mma_commit(&empty[s]);
        }
        if (!ok) break;
        mma_commit(&accfull[a]);
      }
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ x scaling
    const int et = threadIdx.x - 64;  // one token row of one A box per stage
    const int box = et >> 5, row = et & 31;
    int it = 0;
    for (int k = 0; k < nmine && ok; ++k) {
      const int wb = k & 1;
      if (!mbar_wait(&wready[wb], (k >> 1) & 1, spin_ns)) {
        ok = false;
        break;
      }
      const float* w = w_s + wb * 2 * Q + (box >> 1) * Q;
      for (int st = 0; st < nstage; ++st, ++it) {
        const int s = it % kStages, r = it / kStages;
        if (!mbar_wait(&full[s], r & 1, spin_ns)) {
          ok = false;
          break;
        }
        const float wj = w[st * kTokens + row];
        float4* rp = reinterpret_cast<float4*>(smem + L.ring + s * kStage + box * kBox + row * 128);
#pragma unroll
        for (int q = 0; q < 8; ++q) {  // chunk order rotated per row: a warp's accesses hit all banks
          float4* cp = rp + (q ^ (row & 7));
          float4 v = *cp;
          v.x = round_tf32(v.x * wj);
          v.y = round_tf32(v.y * wj);
          v.z = round_tf32(v.z * wj);
          v.w = round_tf32(v.w * wj);
          *cp = v;
        }
        fence_proxy_async_smem();
        mbar_arrive(&scaled[s]);
      }
      if (!ok) break;
      mbar_arrive(&wfree[wb]);  // this unit's weights are no longer read
    }
  } else {
    // ------------------------------------------------------------ weights and drain
    const int dt_idx = threadIdx.x - 192;
    const int quad = warp & 3;  // tensor-memory lane quadrant of this warp
    const int row = quad * 32 + lane;
    uint8_t* staging = smem + L.staging;
    // the token weights of unit k into buffer k % 2: warps 6 and 7 scan one head each, write the
    // cumsum and dt_t rows for the kernels after this one, and store w_j
    // (the drain warps decide every wait together, so that none of them is left at a named barrier)
    auto weights = [&](int k) -> bool {
      const int wb = k & 1;
      const bool good = k < 2 || mbar_wait(&wfree[wb], ((k >> 1) - 1) & 1, spin_ns);
      if (named_bar_or(kDrainBar, 128, !good)) return false;
      if (warp < 8) {
        int b, c, h0;
        unit(k, b, c, h0);
        const int hl = warp - 6, h = h0 + hl;
        const int per = Q / 32;  // 2, 4 or 8 tokens per lane
        const int64_t grow = (static_cast<int64_t>(b) * d.H + h) * d.Lp + static_cast<int64_t>(c) * Q;
        float v[8], gv[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int tok = c * Q + lane * per + q;
          v[q] = (q < per && tok < d.L) ? dt[(static_cast<int64_t>(b) * d.L + tok) * d.H + h] : 0.f;
        }
        float carry = 0.f;
        cumsum_piece(v, per, A[h], carry, gv);
        const float gl = per == 2 ? gv[1] : per == 4 ? gv[3] : gv[7];
        const float glast = __shfl_sync(0xffffffffu, gl, 31);
        float* w = w_s + wb * 2 * Q + hl * Q;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (q < per) {
            const int j = lane * per + q;
            cumsum[grow + j] = gv[q];
            dt_t[grow + j] = v[q];
            w[j] = expf(glast - gv[q]) * v[q];
          }
        }
      }
      mbar_arrive(&wready[wb]);
      return true;
    };
    if (nmine > 0 && !weights(0)) ok = false;
    for (int k = 0; k < nmine && ok; ++k) {
      if (k + 1 < nmine && !weights(k + 1)) {
        ok = false;
        break;
      }
      const int a = k & 1;
      const bool good = mbar_wait(&accfull[a], (k >> 1) & 1, spin_ns);
      if (named_bar_or(kDrainBar, 128, !good)) {
        ok = false;
        break;
      }
      tc_fence_after();
      int b, c, h0;
      unit(k, b, c, h0);
      const int row0 = ((b * d.nc + c) * d.H + h0) * d.P;
      const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(a * kN);
      // rounds of 64 columns: two staging boxes, each 128 rows of 32 n (128-byte swizzle)
      for (int n0 = 0; n0 < kN; n0 += 64) {
        if (dt_idx == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");  // staging free
        named_bar_sync(kDrainBar, 128);
        uint32_t va[32], vb[32];
        tmem_ld32(lane_addr + static_cast<uint32_t>(n0), va);
        tmem_ld32(lane_addr + static_cast<uint32_t>(n0 + 32), vb);
        tmem_ld_wait();
        if (n0 + 64 == kN) {  // every column read: the accumulator may take unit k + 2
          tc_fence_before();
          mbar_arrive(&accfree[a]);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          *reinterpret_cast<uint4*>(staging + row * 128 + ((q ^ (row & 7)) << 4)) =
              make_uint4(va[4 * q], va[4 * q + 1], va[4 * q + 2], va[4 * q + 3]);
          *reinterpret_cast<uint4*>(staging + 16384 + row * 128 + ((q ^ (row & 7)) << 4)) =
              make_uint4(vb[4 * q], vb[4 * q + 1], vb[4 * q + 2], vb[4 * q + 3]);
        }
        fence_proxy_async_smem();
        named_bar_sync(kDrainBar, 128);
        if (dt_idx == 0) {
          tma_store_2d(&smap, staging, n0, row0);
          tma_store_2d(&smap, staging + 16384, n0 + 32, row0);
          tma_store_commit();
        }
      }
    }
    if (dt_idx == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
  if (!ok) atomicExch(status, static_cast<int>(SSD_ERR_DEVICE_TIMEOUT));
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

int persistent_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) cache[dev] = n;
  }
  return cache[dev];
}

}  // namespace

cudaError_t launch_chunk_state_persistent(const Dims& d, const ChunkStateMaps& maps, const Work& w, uint64_t spin_ns,
                                          cudaStream_t stream, bool dependent, const float* dt, const float* A,
                                          int nchain) {
  if (d.N != kN || d.Q > 256 || d.Q < 64 || !dt || !A) return cudaErrorInvalidValue;
  const size_t smem = 1024 + persist_layout(d.Q).total;
  static size_t configured = 0;
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(chunk_state_persistent_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  const long long units = static_cast<long long>(d.H / 2) * d.nc * d.B;
  const int sms = persistent_sm_count();
  const int grid = static_cast<int>(units < sms ? units : sms);
  if (grid <= 0) return cudaErrorInvalidConfiguration;
  return launch_k(chunk_state_persistent_kernel, dim3(grid), dim3(kThreads), smem, stream, dependent, maps.x, maps.bm,
                  maps.s, d, w.cumsum, w.dt_t, dt, A, w.counter, nchain, w.status, spin_ns);
}

}  // namespace ssd
