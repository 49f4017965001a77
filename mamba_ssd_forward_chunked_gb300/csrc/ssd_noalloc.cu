// ssd_fwd_static_scratch: the forward pass for callers that cannot allocate
// device memory.
//
// Some hosts of this library may not call cudaMalloc at all: plugins inside a
// runtime that owns every byte of device memory through its own pool, serving
// processes that forbid allocation after start-up (an allocation can stall the
// device and can fail under memory pressure at the worst moment), and code
// that runs where a new allocation is not allowed.  For them this file keeps
// the forward pass's workspace in a fixed array in the library's own device
// data, so the caller passes only inputs and outputs.
//
// The array is kSsdStaticScratchBytes (SSD_STATIC_SCRATCH_BYTES) long and
// lives on every GPU that loads this library until the process exits.
// Problems whose workspace (ssd_fwd_workspace_size) is larger are rejected.
// All calls share the one array, so calls whose GPU work overlaps in time (on
// different streams, or from different threads without ordering) race on it.
#include <mutex>

#include "ssd_internal.cuh"

namespace {

constexpr size_t kSsdStaticScratchBytes = SSD_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Device-side scratch.  In host code this name is only a host-side stand-in:
// its device address must come from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_ssd_static_scratch[kSsdStaticScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device (set-up once per device).
ssd_status scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSD_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ssd_static_scratch) != cudaSuccess || p == nullptr) return SSD_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SSD_OK;
}

}  // namespace

extern "C" ssd_status ssd_fwd_static_scratch(const ssd_shape* shape, const void* x, const float* dt,
                                             const float* A, const void* Bm, const void* Cm, const float* D,
                                             const float* init_state, void* y, float* final_state,
                                             ssd_stream_t stream) {
  ssd_status st = ssd_validate_shape(shape);
  if (st != SSD_OK) return st;
  const size_t need = ssd_fwd_workspace_size(shape);
  if (need > kSsdStaticScratchBytes) return SSD_ERR_WORKSPACE;
  void* scratch = nullptr;
  st = scratch_on_current_device(&scratch);
  if (st != SSD_OK) return st;
  // Nothing is enqueued here: ssd_fwd checks every pointer first, and for a
  // non-empty problem its first kernel clears the status word and the one-pass
  // counters, so the previous call's contents of the array never leak into this one.
  return ssd_fwd(shape, x, dt, A, Bm, Cm, D, init_state, y, final_state, scratch, kSsdStaticScratchBytes, stream);
}
