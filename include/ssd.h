/*
 * ssd.h -- C ABI of the GB300 (sm_103a) Mamba-2 chunked SSD forward library.
 *
 * The operation (source: "Jane Street ML Engineers Map Mamba-2 Recurrent State
 * Computation to Tensor Cores with cuTile", paragraphs on the fixed-size
 * recurrent state, the jump formula and the three-kernel decomposition): for
 * every batch b and head h, with head h reading group g = h / (nheads/ngroups)
 * of Bm and Cm and the state h_t a headdim x dstate matrix,
 *
 *     h_t = exp(dt_t * A_h) * h_{t-1} + dt_t * x_t b_t^T        (h_{-1} = init_state or 0)
 *     y_t = h_t c_t + D_h * x_t                                  final_state = h_{L-1}
 *
 * computed chunk by chunk (chunk_size tokens) in four kernels: a log-space
 * cumsum of dt*A per chunk, each chunk's state contribution on the tensor
 * cores, a sequential pass over chunks that carries the state (the jump
 * formula with decay), and a fused output kernel (carried-state term, causally
 * masked decayed interaction matrix, D*x skip).
 *
 * Conventions shared by every entry point below:
 *  - Pointers are caller-owned DEVICE memory (CUDA global memory of the current
 *    device), row-major and contiguous, never freed or kept by the library.
 *  - Layouts: x, y [batch][seqlen][nheads][headdim]; dt [batch][seqlen][nheads];
 *    A, D [nheads]; Bm, Cm [batch][seqlen][ngroups][dstate];
 *    init_state, final_state [batch][nheads][headdim][dstate].
 *  - dtype: x, Bm, Cm and y are fp32 (SSD_F32: TF32 tensor-core products with
 *    fp32 accumulation) or bf16 (SSD_BF16: bf16 products, fp32 accumulation,
 *    y rounded to nearest even).  dt, A, D, init_state and final_state are
 *    always fp32.  dt is used as given (post-activation, positive).
 *  - Work is enqueued on `stream` (0 = legacy default stream) and is
 *    asynchronous: no call synchronises.  Calls that share a workspace must be
 *    ordered on one stream.
 *  - Argument errors are reported before anything is enqueued.  CUDA launch
 *    errors return SSD_ERR_CUDA.  Waits inside the kernels are bounded; a wait
 *    that runs out records SSD_ERR_DEVICE_TIMEOUT in the workspace status word,
 *    which ssd_fwd_check() reads after the caller synchronises.  The library
 *    never aborts the process.
 *  - Supported shapes: headdim == 64; dstate in {64, 128, 256};
 *    chunk_size in {64, 128, 256}; nheads % ngroups == 0 and (nheads/ngroups)
 *    even; x, Bm, Cm, y and the workspace 16-byte aligned.  Anything else
 *    returns SSD_ERR_UNSUPPORTED (shape) or SSD_ERR_INVALID_ARG (pointer,
 *    negative size).  batch == 0 or seqlen == 0 is valid (empty input).
 */
#ifndef SSD_GB300_H_
#define SSD_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* ssd_stream_t; /* same handle as cudaStream_t */

typedef enum {
  SSD_OK = 0,
  SSD_ERR_INVALID_ARG = 1,
  SSD_ERR_UNSUPPORTED = 2,
  SSD_ERR_WORKSPACE = 3,
  SSD_ERR_CUDA = 4,
  SSD_ERR_DEVICE_TIMEOUT = 5
} ssd_status;

typedef enum { SSD_F32 = 0, SSD_BF16 = 1 } ssd_dtype;

typedef struct {
  int64_t batch;      /* B >= 0 */
  int64_t seqlen;     /* L >= 0; need not be a multiple of chunk_size */
  int32_t nheads;     /* H */
  int32_t headdim;    /* P (64) */
  int32_t ngroups;    /* G, divides H */
  int32_t dstate;     /* N */
  int32_t chunk_size; /* Q */
  int32_t dtype;      /* ssd_dtype of x, Bm, Cm, y */
} ssd_shape;

/* Byte offsets of the workspace regions (each 1024-byte aligned).  The
 * workspace is caller-owned scratch; its contents between calls are
 * intermediate results exposed for testing:
 *   status      int32 device status word (0 = OK)
 *   cumsum      fp32 [B][H][nc*Q]  inclusive cumsum of dt*A within each chunk
 *   dt_t        fp32 [B][H][nc*Q]  dt transposed to head-major order (0 past L)
 *   states      [B][nc][H][P][N] chunk states S_c, fp32 for SSD_F32 and bf16
 *               for SSD_BF16; after the state pass, for SSD_F32 the state
 *               entering each chunk (in place)
 *   states_bf16 bf16 [B][nc][H][P][N]  (SSD_BF16 only) state entering each
 *               chunk, rounded to bf16 for the output kernel's tensor cores
 *   chain       int32 [1 + B*H/2]  one-pass kernel: tile counter, then per
 *               (batch, head pair) the number of windows whose state is
 *               published (cleared by the call's first kernel)
 *   hslot       fp32, B*H*P*N values  one-pass kernel: the state handed from
 *               one run of windows to the next, per head pair in a layout of
 *               its own ([N/32][8][2*P rows][4]: a warp's 16-byte accesses are
 *               consecutive)
 *   cbm         (SSD_BF16 only) bf16 [B][nw][G][128][128], nw = ceil(seqlen/128):
 *               for every 128-token window and group the causal select of
 *               C B^T, M[i][j] = c_i . b_j for j <= i and 0 above the
 *               diagonal (one-pass schedule, written by its first step)
 * nc = ceil(seqlen / chunk_size), Lp = nc * chunk_size. */
typedef struct {
  size_t status;
  size_t cumsum;
  size_t dt_t;
  size_t states;
  size_t states_bf16;
  size_t chain;
  size_t hslot;
  size_t cbm;
  size_t total;
} ssd_workspace_layout;

/* Human-readable name of a status code (static storage; never NULL). */
const char* ssd_status_string(ssd_status s);

/* Checks the shape (see "Supported shapes") without touching memory. */
ssd_status ssd_validate_shape(const ssd_shape* shape);

/* Workspace regions for `shape`; returns SSD_OK or the shape error. */
ssd_status ssd_fwd_workspace_layout(const ssd_shape* shape, ssd_workspace_layout* out);

/* Bytes of device workspace ssd_fwd needs for `shape` (0 if the shape is
 * invalid or unsupported). */
size_t ssd_fwd_workspace_size(const ssd_shape* shape);

/* The whole forward pass, enqueued on `stream`.  Three schedules give the
 * recurrence's result (see the steps below for the formulas):
 *  - one-pass (ssd_fwd_fused; SSD_BF16 only): ssd_causal_cb, then one
 *    persistent kernel (ssd_fused_pass) that runs every 128-token window of a
 *    (batch, head pair): the window's cumulative decay, its state product on
 *    the tensor core accumulated onto the running state, the carried-state
 *    and intra-window products and y; the state moves between windows in
 *    tensor memory and between runs of windows through the workspace (or
 *    final_state).  x is read once and the states never reach HBM.
 *  - staged: chunk_state (which forms each chunk's cumsum itself, exactly as
 *    chunk_cumsum does, and writes the cumsum and dt_t rows), state_passing and
 *    compute_out.
 *  - segmented one-pass (SSD_BF16 only): chunk_cumsum, chunk_state and
 *    state_passing with segments of 2048 (or 1024) tokens as their chunk,
 *    which leaves every segment's entering state (fp32) in the workspace and
 *    writes final_state, then the one-pass pair on the sequences' segments
 *    taken as a batch of one-segment sequences, each from its entering state.
 * ssd_fwd takes the one-pass schedule for SSD_BF16 when there are at least as
 * many (batch, head pair) sequences as multiprocessors (below that the chain
 * of windows, not bandwidth, bounds the one-pass kernel); below that, the
 * segmented one when the segments divide the sequence and give at least two
 * per multiprocessor over all pairs; otherwise the staged one (always for
 * SSD_F32).  The one-pass schedules work in windows of 128
 * tokens whatever chunk_size is; the result is the recurrence's either way.
 * init_state may be NULL (zero initial state); final_state
 * may be NULL (not written; the workspace holds the running state instead).
 * When given, final_state is also the running state's storage during the
 * call, so it must not overlap the inputs (it may equal init_state).  The
 * workspace must hold ssd_fwd_workspace_size(shape) bytes. */
ssd_status ssd_fwd(const ssd_shape* shape, const void* x, const float* dt, const float* A,
                   const void* Bm, const void* Cm, const float* D, const float* init_state, void* y,
                   float* final_state, void* workspace, size_t workspace_bytes, ssd_stream_t stream);

/* ssd_fwd forced onto the one-pass schedule (same arguments and contract).
 * SSD_ERR_UNSUPPORTED unless shape->dtype is SSD_BF16. */
ssd_status ssd_fwd_fused(const ssd_shape* shape, const void* x, const float* dt, const float* A,
                         const void* Bm, const void* Cm, const float* D, const float* init_state, void* y,
                         float* final_state, void* workspace, size_t workspace_bytes, ssd_stream_t stream);

/* Step 1 of the one-pass schedule alone ("Jane Street ML Engineers Map Mamba-2
 * Recurrent State Computation to Tensor Cores with cuTile", compute_out
 * paragraph: C B^T by one matrix product, causal mask made in registers):
 * writes the workspace's cbm region, the causal select of C B^T in bf16 for
 * every (batch, 128-token window, group), shared by every head of the group;
 * also clears the status word and the one-pass run counter and flags.
 * SSD_BF16 only (SSD_ERR_UNSUPPORTED otherwise). */
ssd_status ssd_causal_cb(const ssd_shape* shape, const void* Bm, const void* Cm, void* workspace,
                         size_t workspace_bytes, ssd_stream_t stream);

/* Step 2 of the one-pass schedule alone (ssd_fwd_fused is ssd_causal_cb
 * followed by this call): the persistent kernel described under ssd_fwd.
 * Needs step 1.  SSD_BF16 only (SSD_ERR_UNSUPPORTED otherwise); arguments as
 * for ssd_fwd. */
ssd_status ssd_fused_pass(const ssd_shape* shape, const void* x, const float* dt, const float* A, const void* Bm,
                          const void* Cm, const float* D, const float* init_state, void* y, float* final_state,
                          void* workspace, size_t workspace_bytes, ssd_stream_t stream);

/* The launches ssd_fwd makes for `shape`, numbered 0 .. ssd_fwd_kernel_count()-1
 * in the order ssd_fwd enqueues them, restricted to those with index in
 * [first_launch, end_launch): the same kernels with the same arguments, so
 * that calls covering consecutive ranges on one stream compute exactly what
 * one ssd_fwd call computes.  Inside one call a launch overlaps the tail of
 * the launch before it as in ssd_fwd; the first launch of a call waits for
 * the work already on the stream.  Used to time the schedule's kernels one by
 * one with events between the calls.  Arguments as for ssd_fwd;
 * SSD_ERR_INVALID_ARG if first_launch < 0 or end_launch < first_launch. */
ssd_status ssd_fwd_range(const ssd_shape* shape, const void* x, const float* dt, const float* A,
                         const void* Bm, const void* Cm, const float* D, const float* init_state, void* y,
                         float* final_state, void* workspace, size_t workspace_bytes, int first_launch,
                         int end_launch, ssd_stream_t stream);

/* After the caller has synchronised the stream of a call that used
 * `workspace`: SSD_OK, or SSD_ERR_DEVICE_TIMEOUT if a bounded wait inside a
 * kernel ran out (its outputs are then invalid).  Blocking 4-byte read. */
ssd_status ssd_fwd_check(const void* workspace);

/* --- The four steps, callable one by one (for SSD_F32, ssd_fwd computes
 * exactly what these four calls in order compute -- its chunk_state launch
 * forms the step-1 rows itself; for SSD_BF16 the four calls in order give the
 * same result as ssd_fwd through the staged path).  Each reads and writes the
 * workspace regions named. ---- */

/* Step 1 (page 1, chunk_cumsum): cumsum[b][h][cQ+i] = sum_{k<=i} dt*A over the
 * chunk, dt_t = dt transposed; tokens past seqlen contribute 0.  Also clears
 * the status word. */
ssd_status ssd_chunk_cumsum(const ssd_shape* shape, const float* dt, const float* A, void* workspace,
                            size_t workspace_bytes, ssd_stream_t stream);

/* Step 2 (page 1, jump formula with decay; fwd_pass_state's per-chunk MMA):
 * states[b][c][h][p][n] = sum_{j in chunk c} exp(G_last - G_j) dt_j x_j[p] b_j[n]
 * on the tensor cores (tcgen05, accumulator in tensor memory, operands staged
 * by TMA).  Needs step 1. */
ssd_status ssd_chunk_state(const ssd_shape* shape, const void* x, const void* Bm, void* workspace,
                           size_t workspace_bytes, ssd_stream_t stream);

/* Step 3 (page 1, fwd_pass_state's sequential loop over chunks): with
 * h = init_state (or 0), for c = 0..nc-1: entering_c = h;
 * h = exp(G_last_c) h + S_c.  Writes the entering states (see the layout) and
 * final_state = h (if not NULL).  Needs steps 1-2. */
ssd_status ssd_state_passing(const ssd_shape* shape, const float* init_state, float* final_state,
                             void* workspace, size_t workspace_bytes, ssd_stream_t stream);

/* Step 4 (page 1, compute_out): y_i = exp(G_i) C_i h_entering^T
 *   + sum_{j<=i in chunk} (C_i . B_j) exp(G_i - G_j) dt_j x_j + D_h x_i,
 * one fused tile kernel on the tensor cores; the causal mask is made in
 * registers and the chunk_size x chunk_size matrix never reaches global
 * memory.  Needs steps 1-3. */
ssd_status ssd_compute_out(const ssd_shape* shape, const void* x, const void* Bm, const void* Cm,
                           const float* D, void* y, void* workspace, size_t workspace_bytes,
                           ssd_stream_t stream);

/* Test hook for the failure path: enqueues one block that waits, for at most
 * `limit_us` microseconds, on a barrier nothing arrives at, then records
 * SSD_ERR_DEVICE_TIMEOUT in the workspace status word and exits (no trap, no
 * hang).  The workspace needs at least 4 bytes. */
ssd_status ssd_debug_timeout_probe(void* workspace, uint32_t limit_us, ssd_stream_t stream);

/* Number of kernels ssd_fwd enqueues for `shape` (0 for an empty input): 2
 * on the one-pass schedule, 5 on the segmented one and 3 on the staged one. */
int ssd_fwd_kernel_count(const ssd_shape* shape);

/* Bytes of the device array that ssd_fwd_static_scratch uses as its workspace. */
#define SSD_STATIC_SCRATCH_BYTES ((size_t)32 << 20)

/* ssd_fwd for callers that may not allocate device memory.  The pages describe
 * no counterpart: this is a service of the library, not a step of the method.
 *
 * Who needs it: code that runs inside a host which owns all device memory
 * (a plugin of another runtime with its own pool), serving processes that
 * allow no allocation after start-up, and any caller for whom a cudaMalloc
 * on the hot path is not allowed or too risky (it can stall the device and
 * can fail under memory pressure).  Such a caller passes only the inputs and
 * outputs of ssd_fwd; the workspace is a fixed array of
 * SSD_STATIC_SCRATCH_BYTES in the library's own device data, which every GPU
 * that loads the library holds until the process exits.  The call itself
 * allocates nothing.  Under lazy module loading (the CUDA default) the
 * array's memory is committed when the library's device code first loads on
 * a device, which is at the latest this entry point's first call there; make
 * that first call at start-up (where an out-of-memory error can still be
 * handled) and before any stream capture.
 *
 * Arguments, layouts, dtypes and supported shapes are those of ssd_fwd.
 * Returns SSD_ERR_WORKSPACE, before enqueuing anything, when
 * ssd_fwd_workspace_size(shape) is larger than SSD_STATIC_SCRATCH_BYTES.
 * The first call on a device also looks up the array's device address
 * (cudaGetSymbolAddress) for that device; this set-up is one more reason to
 * make it before any stream capture.  Argument errors are returned before
 * anything is enqueued.
 * A non-empty call's first kernel clears the status word and the one-pass
 * counters before the rest of the array is overwritten; the array keeps the
 * last call's intermediate results.
 * All calls share the one array: calls whose GPU work can overlap in time
 * (different streams, or threads without ordering between them) race and
 * give wrong results.  A device-timeout status (see ssd_fwd_check) is left in
 * the array and cannot be read through this entry point. */
ssd_status ssd_fwd_static_scratch(const ssd_shape* shape, const void* x, const float* dt, const float* A,
                                  const void* Bm, const void* Cm, const float* D, const float* init_state,
                                  void* y, float* final_state, ssd_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SSD_GB300_H_ */
