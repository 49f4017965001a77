// Host side of the C ABI declared in include/ssd.h: argument checks, workspace
// carving, TMA tensor-map encoding and the four launches on the caller's
// stream.  Nothing here allocates device memory or synchronises (except
// ssd_fwd_check, which reads the 4-byte status word).
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr size_t kAlign = 1024;
inline size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

uint64_t spin_limit_ns() {
  static uint64_t v = [] {
    const char* s = std::getenv("SSD_SPIN_LIMIT_MS");
    uint64_t ms = 2000;
    if (s && *s) {
      char* end = nullptr;
      unsigned long long x = std::strtoull(s, &end, 10);
      if (end != s && x > 0) ms = x;
    }
    return ms * 1000000ull;
  }();
  return v;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Tiled map with a 128-byte swizzle (16-byte chunks, or 32-byte chunks for the MN-major TF32
// operands), zero fill outside the tensor.
bool encode(CUtensorMap* m, bool bf16, int rank, const void* base, const uint64_t* dims,
            const uint64_t* strides_bytes, const uint32_t* box,
            CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto fn = encode_fn();
  if (!fn) return false;
  const uint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                  static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims, strides_bytes, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

Dims make_dims(const ssd_shape& s) {
  Dims d{};
  d.B = static_cast<int>(s.batch);
  d.L = static_cast<int>(s.seqlen);
  d.H = s.nheads;
  d.P = s.headdim;
  d.G = s.ngroups;
  d.N = s.dstate;
  d.Q = s.chunk_size;
  d.nc = static_cast<int>((s.seqlen + s.chunk_size - 1) / s.chunk_size);
  d.Lp = d.nc * d.Q;
  return d;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

bool empty_problem(const ssd_shape& s) { return s.batch == 0 || s.seqlen == 0; }

ssd_status layout_of(const ssd_shape* shape, ssd_workspace_layout* out) {
  ssd_status st = ssd_validate_shape(shape);
  if (st != SSD_OK) return st;
  const ssd_shape& s = *shape;
  const int64_t nc = (s.seqlen + s.chunk_size - 1) / s.chunk_size;
  const size_t lp = static_cast<size_t>(nc) * s.chunk_size;
  const size_t heads = static_cast<size_t>(s.batch) * s.nheads;
  const size_t nstate = static_cast<size_t>(s.batch) * nc * s.nheads * s.headdim * s.dstate;
  ssd_workspace_layout L{};
  size_t off = 0;
  L.status = off;
  off = align_up(off + 256);
  L.cumsum = off;
  off = align_up(off + heads * lp * sizeof(float));
  L.dt_t = off;
  off = align_up(off + heads * lp * sizeof(float));
  L.states = off;
  off = align_up(off + nstate * (s.dtype == SSD_BF16 ? sizeof(__nv_bfloat16) : sizeof(float)));
  L.states_bf16 = off;
  if (s.dtype == SSD_BF16) off = align_up(off + nstate * sizeof(__nv_bfloat16));
  L.chain = off;
  off = align_up(off + (1 + heads / 2) * sizeof(int));
  L.hslot = off;
  off = align_up(off + heads * s.headdim * s.dstate * sizeof(float));
  L.cbm = off;
  if (s.dtype == SSD_BF16) {
    const size_t nwin = static_cast<size_t>((s.seqlen + 127) / 128);
    off = align_up(off + static_cast<size_t>(s.batch) * nwin * s.ngroups * 128 * 128 * sizeof(__nv_bfloat16));
  }
  L.total = off;
  *out = L;
  return SSD_OK;
}

Work carve(void* ws, const ssd_workspace_layout& L, bool bf16) {
  uint8_t* p = static_cast<uint8_t*>(ws);
  Work w{};
  w.status = reinterpret_cast<int*>(p + L.status);
  w.cumsum = reinterpret_cast<float*>(p + L.cumsum);
  w.dt_t = reinterpret_cast<float*>(p + L.dt_t);
  w.states = p + L.states;
  w.states_bf16 = bf16 ? reinterpret_cast<__nv_bfloat16*>(p + L.states_bf16) : nullptr;
  w.counter = reinterpret_cast<int*>(p + L.chain);
  w.flags = w.counter + 1;
  w.hslot = reinterpret_cast<float*>(p + L.hslot);
  w.cbm = bf16 ? static_cast<void*>(p + L.cbm) : nullptr;
  return w;
}

ssd_status check_workspace(const ssd_shape* shape, void* ws, size_t bytes, ssd_workspace_layout* L) {
  ssd_status st = layout_of(shape, L);
  if (st != SSD_OK) return st;
  if (!ws || !aligned16(ws)) return SSD_ERR_INVALID_ARG;
  if (bytes < L->total) return SSD_ERR_WORKSPACE;
  return SSD_OK;
}

ssd_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA; }

size_t esize(const ssd_shape& s) { return s.dtype == SSD_BF16 ? 2 : 4; }

bool build_state_maps(const ssd_shape& s, const void* x, const void* Bm, const void* states, ChunkStateMaps* m) {
  const bool bf16 = s.dtype == SSD_BF16;
  const uint64_t es = esize(s);
  const uint32_t atom = static_cast<uint32_t>(128 / es);
  const uint64_t hp = static_cast<uint64_t>(s.nheads) * s.headdim;
  // the MMA operands (x, Bm) are MN-major: fp32 tiles in the 32-byte-atom swizzle TF32 needs
  const CUtensorMapSwizzle sw = bf16 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B;
  {
    const uint64_t dims[3] = {hp, static_cast<uint64_t>(s.seqlen), static_cast<uint64_t>(s.batch)};
    const uint64_t str[2] = {hp * es, hp * es * s.seqlen};
    const uint32_t box[3] = {atom, 32, 1};
    if (!encode(&m->x, bf16, 3, x, dims, str, box, sw)) return false;
  }
  {
    const uint64_t gn = static_cast<uint64_t>(s.ngroups) * s.dstate;
    const uint64_t dims[4] = {static_cast<uint64_t>(s.dstate), static_cast<uint64_t>(s.ngroups),
                              static_cast<uint64_t>(s.seqlen), static_cast<uint64_t>(s.batch)};
    const uint64_t str[3] = {s.dstate * es, gn * es, gn * es * s.seqlen};
    const uint32_t box[4] = {atom, 1, 32, 1};
    if (!encode(&m->bm, bf16, 4, Bm, dims, str, box, sw)) return false;
  }
  {
    const int64_t nc = (s.seqlen + s.chunk_size - 1) / s.chunk_size;
    const uint64_t rows = static_cast<uint64_t>(s.batch) * nc * s.nheads * s.headdim;
    const uint64_t dims[2] = {static_cast<uint64_t>(s.dstate), rows};
    const uint64_t str[1] = {s.dstate * es};
    const uint32_t box[2] = {atom, 128};
    if (!encode(&m->s, bf16, 2, states, dims, str, box)) return false;
  }
  return true;
}

bool build_out_maps(const ssd_shape& s, const void* x, const void* Bm, const void* Cm, const void* hp_states,
                    const void* y, ComputeOutMaps* m) {
  const bool bf16 = s.dtype == SSD_BF16;
  const uint64_t es = esize(s);
  const uint32_t atom = static_cast<uint32_t>(128 / es);
  const uint64_t gn = static_cast<uint64_t>(s.ngroups) * s.dstate;
  const uint64_t dims4[4] = {static_cast<uint64_t>(s.dstate), static_cast<uint64_t>(s.ngroups),
                             static_cast<uint64_t>(s.seqlen), static_cast<uint64_t>(s.batch)};
  const uint64_t str4[3] = {s.dstate * es, gn * es, gn * es * s.seqlen};
  const uint32_t box4[4] = {atom, 1, 128, 1};
  if (!encode(&m->cm, bf16, 4, Cm, dims4, str4, box4)) return false;
  if (!encode(&m->bm, bf16, 4, Bm, dims4, str4, box4)) return false;
  const int64_t nc = (s.seqlen + s.chunk_size - 1) / s.chunk_size;
  {
    const uint64_t rows = static_cast<uint64_t>(s.batch) * nc * s.nheads * s.headdim;
    const uint64_t dims[2] = {static_cast<uint64_t>(s.dstate), rows};
    const uint64_t str[1] = {s.dstate * es};
    const uint32_t box[2] = {atom, 64};
    if (!encode(&m->hp, bf16, 2, hp_states, dims, str, box)) return false;
  }
  {
    const uint64_t hp = static_cast<uint64_t>(s.nheads) * s.headdim;
    const uint64_t dims[3] = {hp, static_cast<uint64_t>(s.seqlen), static_cast<uint64_t>(s.batch)};
    const uint64_t str[2] = {hp * es, hp * es * s.seqlen};
    // one 128-token box per 128-byte column of the block (bf16: 64 p, fp32: 32 p); fp32 tiles
    // take the 32-byte-atom swizzle, the layout of an MN-major TF32 operand
    const CUtensorMapSwizzle sw = bf16 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B;
    const uint32_t box[3] = {atom, 128u, 1};
    if (!encode(&m->x, bf16, 3, x, dims, str, box, sw)) return false;
    const uint32_t ybox[3] = {atom, 32u, 1};
    if (!encode(&m->y, bf16, 3, y, dims, str, ybox, sw)) return false;
  }
  return true;
}

// Multiprocessors of the current device (cached per device).
int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) cache[dev] = n;
  }
  return cache[dev];
}

// The one-pass schedule pays a chain of windows per (batch, head pair); it wins
// once there are enough sequences to fill the multiprocessors (measured on
// GB300, bf16: every 65,536-token sweep point with at least 152 head-pair
// sequences, dstate 64 to 256 -- at dstate 256 0.71-0.83 ms against 1.29-1.60
// ms staged; with 64 sequences of 256 windows the staged schedule is faster,
// 1.02 against 1.42 ms).  Without a device (no multiprocessor count) the
// answer is the staged schedule.
bool use_fused(const ssd_shape& s) {
  if (s.dtype != SSD_BF16) return false;
  const int sms = sm_count();
  return sms > 0 && s.batch * (s.nheads / 2) >= sms;
}

// Windows per segment of the segmented one-pass schedule, or 0 where it does not apply.  With
// fewer head-pair sequences than multiprocessors but long sequences (bf16), the staged kernels
// first carry the state across segments of 2048 (or 1024) tokens -- chunk_cumsum, chunk_state
// and state_passing with the segment as their chunk -- and the one-pass kernel then runs every
// segment as an independent run from its entering state, so every multiprocessor has work.
// It applies when the segments divide the sequence and give at least two per multiprocessor
// over all pairs.  Measured on GB300 with 64 sequences of 32768 tokens: segments of 1024, 2048
// and 4096 tokens ran 0.61-1.12, 0.62-1.12 and 0.68-1.18 ms.
int segment_windows(const ssd_shape& s) {
  if (s.dtype != SSD_BF16 || use_fused(s)) return 0;
  const int sms = sm_count();
  if (sms <= 0) return 0;
  const int64_t pairs = static_cast<int64_t>(s.batch) * (s.nheads / 2);
  for (int r : {16, 8}) {
    const int64_t q = 128 * r;
    if (s.seqlen % q == 0 && pairs * (s.seqlen / q) >= 2 * static_cast<int64_t>(sms)) return r;
  }
  return 0;
}

// 0 staged, 1 one-pass, 2 segmented one-pass
int schedule_of(const ssd_shape& s) { return use_fused(s) ? 1 : segment_windows(s) > 0 ? 2 : 0; }

ssd_status fwd_impl(int path, int first, int end, const ssd_shape* shape, const void* x, const float* dt,
                    const float* A, const void* Bm, const void* Cm, const float* D, const float* init_state, void* y,
                    float* final_state, void* workspace, size_t workspace_bytes, ssd_stream_t stream);

bool build_onepass_maps(const ssd_shape& s, const void* x, const void* Bm, const void* Cm, const void* y,
                        const void* cbm, OnePassMaps* m) {
  const uint64_t es = 2;
  const uint64_t gn = static_cast<uint64_t>(s.ngroups) * s.dstate;
  const uint64_t dims4[4] = {static_cast<uint64_t>(s.dstate), static_cast<uint64_t>(s.ngroups),
                             static_cast<uint64_t>(s.seqlen), static_cast<uint64_t>(s.batch)};
  const uint64_t str4[3] = {s.dstate * es, gn * es, gn * es * s.seqlen};
  const uint32_t box4[4] = {64, 1, 128, 1};
  if (!encode(&m->cm, true, 4, Cm, dims4, str4, box4)) return false;
  if (!encode(&m->bm, true, 4, Bm, dims4, str4, box4)) return false;
  const uint64_t hp = static_cast<uint64_t>(s.nheads) * s.headdim;
  const uint64_t dims[3] = {hp, static_cast<uint64_t>(s.seqlen), static_cast<uint64_t>(s.batch)};
  const uint64_t str[2] = {hp * es, hp * es * s.seqlen};
  const uint32_t box[3] = {64, 128, 1};
  if (!encode(&m->x, true, 3, x, dims, str, box)) return false;
  if (!encode(&m->y, true, 3, y, dims, str, box)) return false;
  const uint64_t nwin = static_cast<uint64_t>((s.seqlen + 127) / 128);
  const uint64_t mdims[2] = {128, static_cast<uint64_t>(s.batch) * nwin * s.ngroups * 128};
  const uint64_t mstr[1] = {128 * es};
  const uint32_t mbox[2] = {64, 128};
  return encode(&m->m, true, 2, cbm, mdims, mstr, mbox);
}

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" {

const char* ssd_status_string(ssd_status s) {
  switch (s) {
    case SSD_OK: return "SSD_OK";
    case SSD_ERR_INVALID_ARG: return "SSD_ERR_INVALID_ARG: null, misaligned or negative argument";
    case SSD_ERR_UNSUPPORTED: return "SSD_ERR_UNSUPPORTED: shape outside the supported set";
    case SSD_ERR_WORKSPACE: return "SSD_ERR_WORKSPACE: workspace smaller than ssd_fwd_workspace_size()";
    case SSD_ERR_CUDA: return "SSD_ERR_CUDA: a CUDA launch or runtime call failed";
    case SSD_ERR_DEVICE_TIMEOUT: return "SSD_ERR_DEVICE_TIMEOUT: a bounded wait inside a kernel ran out";
  }
  return "unknown ssd_status";
}

ssd_status ssd_validate_shape(const ssd_shape* s) {
  if (!s) return SSD_ERR_INVALID_ARG;
  if (s->batch < 0 || s->seqlen < 0 || s->nheads <= 0 || s->headdim <= 0 || s->ngroups <= 0 || s->dstate <= 0 ||
      s->chunk_size <= 0)
    return SSD_ERR_INVALID_ARG;
  if (s->dtype != SSD_F32 && s->dtype != SSD_BF16) return SSD_ERR_UNSUPPORTED;
  if (s->headdim != 64) return SSD_ERR_UNSUPPORTED;
  if (s->dstate != 64 && s->dstate != 128 && s->dstate != 256) return SSD_ERR_UNSUPPORTED;
  if (s->chunk_size != 64 && s->chunk_size != 128 && s->chunk_size != 256) return SSD_ERR_UNSUPPORTED;
  if (s->nheads % s->ngroups != 0 || (s->nheads / s->ngroups) % 2 != 0) return SSD_ERR_UNSUPPORTED;
  // every index that reaches a TMA coordinate or a grid dimension fits int32 / grid limits
  const int64_t nc = (s->seqlen + s->chunk_size - 1) / s->chunk_size;
  if (s->seqlen > (int64_t(1) << 30) || s->batch > 65535 || nc > 65535) return SSD_ERR_UNSUPPORTED;
  if (s->batch * nc * s->nheads * int64_t(s->headdim) >= (int64_t(1) << 31)) return SSD_ERR_UNSUPPORTED;
  if (s->batch * s->seqlen * int64_t(s->nheads) >= (int64_t(1) << 31)) return SSD_ERR_UNSUPPORTED;
  return SSD_OK;
}

ssd_status ssd_fwd_workspace_layout(const ssd_shape* shape, ssd_workspace_layout* out) {
  if (!out) return SSD_ERR_INVALID_ARG;
  return layout_of(shape, out);
}

size_t ssd_fwd_workspace_size(const ssd_shape* shape) {
  ssd_workspace_layout L;
  return layout_of(shape, &L) == SSD_OK ? L.total : 0;
}

int ssd_fwd_kernel_count(const ssd_shape* shape) {
  if (ssd_validate_shape(shape) != SSD_OK || empty_problem(*shape)) return 0;
  const int sched = schedule_of(*shape);
  return sched == 1 ? 2 : sched == 2 ? 5 : 3;
}

ssd_status ssd_chunk_cumsum(const ssd_shape* shape, const float* dt, const float* A, void* workspace,
                            size_t workspace_bytes, ssd_stream_t stream) {
  ssd_workspace_layout L;
  ssd_status st = check_workspace(shape, workspace, workspace_bytes, &L);
  if (st != SSD_OK) return st;
  if (empty_problem(*shape)) return SSD_OK;
  if (!dt || !A || !aligned4(dt) || !aligned4(A)) return SSD_ERR_INVALID_ARG;
  Work w = carve(workspace, L, shape->dtype == SSD_BF16);
  return from_cuda(launch_chunk_cumsum(make_dims(*shape), dt, A, w, reinterpret_cast<cudaStream_t>(stream)));
}

ssd_status ssd_chunk_state(const ssd_shape* shape, const void* x, const void* Bm, void* workspace,
                           size_t workspace_bytes, ssd_stream_t stream) {
  ssd_workspace_layout L;
  ssd_status st = check_workspace(shape, workspace, workspace_bytes, &L);
  if (st != SSD_OK) return st;
  if (empty_problem(*shape)) return SSD_OK;
  if (!x || !Bm || !aligned16(x) || !aligned16(Bm)) return SSD_ERR_INVALID_ARG;
  const bool bf16 = shape->dtype == SSD_BF16;
  Work w = carve(workspace, L, bf16);
  ChunkStateMaps maps;
  if (!build_state_maps(*shape, x, Bm, w.states, &maps)) return SSD_ERR_CUDA;
  const Dims d = make_dims(*shape);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_chunk_state(d, bf16, maps, w, spin_limit_ns(), cs);
  return from_cuda(e);
}

ssd_status ssd_state_passing(const ssd_shape* shape, const float* init_state, float* final_state,
                             void* workspace, size_t workspace_bytes, ssd_stream_t stream) {
  ssd_workspace_layout L;
  ssd_status st = check_workspace(shape, workspace, workspace_bytes, &L);
  if (st != SSD_OK) return st;
  if ((init_state && !aligned16(init_state)) || (final_state && !aligned16(final_state)))
    return SSD_ERR_INVALID_ARG;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (empty_problem(*shape)) {
    // no tokens: the final state is the initial one (or zero)
    if (!final_state || shape->batch == 0) return SSD_OK;
    const size_t bytes = static_cast<size_t>(shape->batch) * shape->nheads * shape->headdim * shape->dstate * 4;
    return from_cuda(init_state ? cudaMemcpyAsync(final_state, init_state, bytes, cudaMemcpyDeviceToDevice, cs)
                                : cudaMemsetAsync(final_state, 0, bytes, cs));
  }
  const bool bf16 = shape->dtype == SSD_BF16;
  Work w = carve(workspace, L, bf16);
  return from_cuda(launch_state_passing(make_dims(*shape), bf16, init_state, final_state, w, cs));
}

ssd_status ssd_compute_out(const ssd_shape* shape, const void* x, const void* Bm, const void* Cm, const float* D,
                           void* y, void* workspace, size_t workspace_bytes, ssd_stream_t stream) {
  ssd_workspace_layout L;
  ssd_status st = check_workspace(shape, workspace, workspace_bytes, &L);
  if (st != SSD_OK) return st;
  if (empty_problem(*shape)) return SSD_OK;
  if (!x || !Bm || !Cm || !D || !y || !aligned16(x) || !aligned16(Bm) || !aligned16(Cm) || !aligned16(y) ||
      !aligned4(D))
    return SSD_ERR_INVALID_ARG;
  const bool bf16 = shape->dtype == SSD_BF16;
  Work w = carve(workspace, L, bf16);
  ComputeOutMaps maps;
  const void* hp = bf16 ? static_cast<const void*>(w.states_bf16) : static_cast<const void*>(w.states);
  if (!build_out_maps(*shape, x, Bm, Cm, hp, y, &maps)) return SSD_ERR_CUDA;
  return from_cuda(launch_compute_out(make_dims(*shape), bf16, maps, D, x, y, w, spin_limit_ns(),
                                      reinterpret_cast<cudaStream_t>(stream)));
}

ssd_status ssd_fwd(const ssd_shape* shape, const void* x, const float* dt, const float* A, const void* Bm,
                   const void* Cm, const float* D, const float* init_state, void* y, float* final_state,
                   void* workspace, size_t workspace_bytes, ssd_stream_t stream) {
  const int path = shape && ssd_validate_shape(shape) == SSD_OK ? schedule_of(*shape) : 0;
  return fwd_impl(path, 0, 1 << 30, shape, x, dt, A, Bm, Cm, D, init_state, y, final_state, workspace,
                  workspace_bytes, stream);
}

ssd_status ssd_fwd_range(const ssd_shape* shape, const void* x, const float* dt, const float* A, const void* Bm,
                         const void* Cm, const float* D, const float* init_state, void* y, float* final_state,
                         void* workspace, size_t workspace_bytes, int first_launch, int end_launch,
                         ssd_stream_t stream) {
  if (first_launch < 0 || end_launch < first_launch) return SSD_ERR_INVALID_ARG;
  const int path = shape && ssd_validate_shape(shape) == SSD_OK ? schedule_of(*shape) : 0;
  return fwd_impl(path, first_launch, end_launch, shape, x, dt, A, Bm, Cm, D, init_state, y, final_state, workspace,
                  workspace_bytes, stream);
}

ssd_status ssd_causal_cb(const ssd_shape* shape, const void* Bm, const void* Cm, void* workspace,
                         size_t workspace_bytes, ssd_stream_t stream) {
  ssd_workspace_layout L;
  ssd_status st = check_workspace(shape, workspace, workspace_bytes, &L);
  if (st != SSD_OK) return st;
  if (shape->dtype != SSD_BF16) return SSD_ERR_UNSUPPORTED;
  if (empty_problem(*shape)) return SSD_OK;
  if (!Bm || !Cm || !aligned16(Bm) || !aligned16(Cm)) return SSD_ERR_INVALID_ARG;
  Work w = carve(workspace, L, true);
  OnePassMaps maps;
  // x and y are not read by this step: Cm stands in as a valid base for their (unused) maps
  if (!build_onepass_maps(*shape, Cm, Bm, Cm, Cm, w.cbm, &maps)) return SSD_ERR_CUDA;
  return from_cuda(launch_causal_cb(make_dims(*shape), maps, w, spin_limit_ns(), reinterpret_cast<cudaStream_t>(stream)));
}

ssd_status ssd_fused_pass(const ssd_shape* shape, const void* x, const float* dt, const float* A, const void* Bm,
                          const void* Cm, const float* D, const float* init_state, void* y, float* final_state,
                          void* workspace, size_t workspace_bytes, ssd_stream_t stream) {
  ssd_workspace_layout L;
  ssd_status st = check_workspace(shape, workspace, workspace_bytes, &L);
  if (st != SSD_OK) return st;
  if (shape->dtype != SSD_BF16) return SSD_ERR_UNSUPPORTED;
  if ((init_state && !aligned16(init_state)) || (final_state && !aligned16(final_state)))
    return SSD_ERR_INVALID_ARG;
  if (empty_problem(*shape)) return SSD_OK;
  if (!x || !dt || !A || !Bm || !Cm || !D || !y || !aligned16(x) || !aligned16(Bm) || !aligned16(Cm) ||
      !aligned16(y) || !aligned4(dt) || !aligned4(A) || !aligned4(D))
    return SSD_ERR_INVALID_ARG;
  Work w = carve(workspace, L, true);
  OnePassMaps maps;
  if (!build_onepass_maps(*shape, x, Bm, Cm, y, w.cbm, &maps)) return SSD_ERR_CUDA;
  return from_cuda(launch_onepass(make_dims(*shape), maps, dt, A, D, x, init_state, final_state, w, spin_limit_ns(),
                                  reinterpret_cast<cudaStream_t>(stream)));
}

ssd_status ssd_fwd_fused(const ssd_shape* shape, const void* x, const float* dt, const float* A, const void* Bm,
                         const void* Cm, const float* D, const float* init_state, void* y, float* final_state,
                         void* workspace, size_t workspace_bytes, ssd_stream_t stream) {
  if (shape && ssd_validate_shape(shape) == SSD_OK && shape->dtype != SSD_BF16) return SSD_ERR_UNSUPPORTED;
  return fwd_impl(1, 0, 1 << 30, shape, x, dt, A, Bm, Cm, D, init_state, y, final_state, workspace, workspace_bytes,
                  stream);
}

}  // extern "C"

namespace ssd {
namespace {

// path: 0 staged, 1 one-pass, 2 segmented one-pass.  Enqueues the schedule's launches with index in
// [first, end); a launch is a programmatic dependent only of a launch of the
// same call (the first one enqueued here is an ordinary stream-ordered launch).
ssd_status fwd_impl(int path, int first, int end, const ssd_shape* shape, const void* x, const float* dt,
                    const float* A, const void* Bm, const void* Cm, const float* D, const float* init_state, void* y,
                    float* final_state, void* workspace, size_t workspace_bytes, ssd_stream_t stream) {
  ssd_workspace_layout L;
  ssd_status st = check_workspace(shape, workspace, workspace_bytes, &L);
  if (st != SSD_OK) return st;
  if (!empty_problem(*shape)) {
    if (!x || !dt || !A || !Bm || !Cm || !D || !y) return SSD_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(Bm) || !aligned16(Cm) || !aligned16(y) || !aligned4(dt) || !aligned4(A) ||
        !aligned4(D))
      return SSD_ERR_INVALID_ARG;
  }
  if ((init_state && !aligned16(init_state)) || (final_state && !aligned16(final_state)))
    return SSD_ERR_INVALID_ARG;
  if (empty_problem(*shape))
    return first == 0 && end > 0 ? ssd_state_passing(shape, init_state, final_state, workspace, workspace_bytes, stream)
                                 : SSD_OK;
  // build every tensor map before the first launch, so an encoding failure enqueues nothing
  const bool bf16 = shape->dtype == SSD_BF16;
  Work w = carve(workspace, L, bf16);
  const Dims d = make_dims(*shape);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  int k = 0;  // index of the next launch of the schedule
  auto step = [&](auto&& launch) {
    if (e == cudaSuccess && k >= first && k < end) e = launch(k > first);
    ++k;
  };
  if (path == 1) {
    OnePassMaps omaps;
    if (!build_onepass_maps(*shape, x, Bm, Cm, y, w.cbm, &omaps)) return SSD_ERR_CUDA;
    const uint64_t spin = spin_limit_ns();
    step([&](bool) { return launch_causal_cb(d, omaps, w, spin, cs); });
    step([&](bool dep) {
      return launch_onepass(d, omaps, dt, A, D, x, init_state, final_state, w, spin, cs, dep);
    });
    return from_cuda(e);
  }
  if (path == 2) {
    // The staged state kernels, with the segment as their chunk, leave every segment's entering
    // state (fp32, [B][segment][H][P][N]) and the final state.  A sequence's segments lie back
    // to back in x, dt, Bm, Cm and y, so they are also a batch of B * segments sequences of one
    // segment each; the one-pass pair runs that batch, each sequence as one claimed run from its
    // entering state.
    const int R = segment_windows(*shape);
    ssd_shape ss = *shape;
    ss.chunk_size = 128 * R;
    const Dims ds = make_dims(ss);
    ssd_shape sv = *shape;
    sv.batch = shape->batch * ds.nc;
    sv.seqlen = 128 * R;
    const Dims dv = make_dims(sv);
    ChunkStateMaps smaps;
    OnePassMaps vmaps;
    if (!build_state_maps(ss, x, Bm, w.states, &smaps) || !build_onepass_maps(sv, x, Bm, Cm, y, w.cbm, &vmaps))
      return SSD_ERR_CUDA;
    // in the region sized for the chunks' bf16 entering states (at least twice as many chunks)
    float* seg_init = reinterpret_cast<float*>(w.states_bf16);
    const uint64_t spin = spin_limit_ns();
    step([&](bool) { return launch_chunk_cumsum(ds, dt, A, w, cs); });
    step([&](bool dep) { return launch_chunk_state(ds, true, smaps, w, spin, cs, dep); });
    step([&](bool) { return launch_state_passing(ds, true, init_state, final_state, w, cs, false, seg_init); });
    step([&](bool) { return launch_causal_cb(dv, vmaps, w, spin, cs, false); });
    step([&](bool dep) {
      return launch_onepass(dv, vmaps, dt, A, D, x, seg_init, nullptr, w, spin, cs, dep, R);
    });
    return from_cuda(e);
  }
  ChunkStateMaps smaps;
  ComputeOutMaps omaps;
  const void* hp = bf16 ? static_cast<const void*>(w.states_bf16) : static_cast<const void*>(w.states);
  if (!build_state_maps(*shape, x, Bm, w.states, &smaps) || !build_out_maps(*shape, x, Bm, Cm, hp, y, &omaps))
    return SSD_ERR_CUDA;
  const uint64_t spin = spin_limit_ns();
  // chunk_state forms each chunk's cumsum itself (no chunk_cumsum launch) and, as the first
  // kernel, clears the status word and the one-pass counters.  compute_out is a programmatic dependent of the kernel
  // before it (its launch and prologue overlap that kernel's tail).  state_passing is one only
  // while chunk_state runs in a single wave (two CTAs per SM): launched early beside a later
  // wave, its blocks slowed long sequences (16k tokens x dstate 256: 0.397 against 0.381 ms),
  // while on a one-wave problem the early launch saves about 1 us (370M layer: 0.0897 against
  // 0.0908 ms).
  const bool one_wave = static_cast<int64_t>(d.B) * d.nc * (d.H / 2) <= 2 * static_cast<int64_t>(sm_count());
  step([&](bool dep) { return launch_chunk_state(d, bf16, smaps, w, spin, cs, dep, dt, A, 1 + d.B * (d.H / 2)); });
  step([&](bool dep) { return launch_state_passing(d, bf16, init_state, final_state, w, cs, one_wave && dep); });
  step([&](bool dep) { return launch_compute_out(d, bf16, omaps, D, x, y, w, spin, cs, dep); });
  return from_cuda(e);
}

}  // namespace
}  // namespace ssd

extern "C" {

ssd_status ssd_fwd_check(const void* workspace) {
  if (!workspace) return SSD_ERR_INVALID_ARG;
  int v = 0;
  if (cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SSD_ERR_CUDA;
  return v == 0 ? SSD_OK : static_cast<ssd_status>(v);
}

ssd_status ssd_debug_timeout_probe(void* workspace, uint32_t limit_us, ssd_stream_t stream) {
  if (!workspace || !aligned4(workspace) || limit_us == 0 || limit_us > 10u * 1000u * 1000u)
    return SSD_ERR_INVALID_ARG;
  return from_cuda(launch_timeout_probe(static_cast<int*>(workspace), static_cast<uint64_t>(limit_us) * 1000ull,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
