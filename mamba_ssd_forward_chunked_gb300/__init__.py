"""Mamba-2 chunked SSD forward on GB300 (sm_103a): Python binding.

Every step of the forward pass runs in the CUDA library ``libssd_gb300.so``
(C ABI in ``include/ssd.h``).  This module only marshals arguments: it checks
tensor dtypes and layouts, allocates outputs and the workspace with PyTorch
when the caller does not pass them, and calls the C entry points of the same
names on the current PyTorch CUDA stream.  There is no CPU fallback: importing
the package fails if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssd_gb300.so")

SSD_F32, SSD_BF16 = 0, 1
STATUS = {0: "SSD_OK", 1: "SSD_ERR_INVALID_ARG", 2: "SSD_ERR_UNSUPPORTED", 3: "SSD_ERR_WORKSPACE",
          4: "SSD_ERR_CUDA", 5: "SSD_ERR_DEVICE_TIMEOUT"}

# Every entry point include/ssd.h declares.
EXPORTS = ("ssd_status_string", "ssd_validate_shape", "ssd_fwd_workspace_layout", "ssd_fwd_workspace_size",
           "ssd_fwd", "ssd_fwd_check", "ssd_chunk_cumsum", "ssd_chunk_state", "ssd_state_passing",
           "ssd_compute_out", "ssd_debug_timeout_probe", "ssd_fwd_kernel_count", "ssd_fwd_static_scratch",
           "ssd_fwd_fused", "ssd_fused_pass", "ssd_fwd_range", "ssd_causal_cb")

# Size of the library's own workspace array used by ssd_fwd_static_scratch.
SSD_STATIC_SCRATCH_BYTES = 32 << 20


class ssd_shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("nheads", ctypes.c_int32),
                ("headdim", ctypes.c_int32), ("ngroups", ctypes.c_int32), ("dstate", ctypes.c_int32),
                ("chunk_size", ctypes.c_int32), ("dtype", ctypes.c_int32)]

    def __repr__(self):
        return ("ssd_shape(B=%d, L=%d, H=%d, P=%d, G=%d, N=%d, Q=%d, dtype=%s)" %
                (self.batch, self.seqlen, self.nheads, self.headdim, self.ngroups, self.dstate,
                 self.chunk_size, "bf16" if self.dtype == SSD_BF16 else "f32"))


class ssd_workspace_layout(ctypes.Structure):
    _fields_ = [("status", ctypes.c_size_t), ("cumsum", ctypes.c_size_t), ("dt_t", ctypes.c_size_t),
                ("states", ctypes.c_size_t), ("states_bf16", ctypes.c_size_t), ("chain", ctypes.c_size_t),
                ("hslot", ctypes.c_size_t), ("cbm", ctypes.c_size_t),
                ("total", ctypes.c_size_t)]


class SSDError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python mamba_ssd_forward_chunked_gb300/build_ext.py` "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    P, c_int, sz, vp = ctypes.POINTER, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
    sp = P(ssd_shape)
    lib.ssd_status_string.restype = ctypes.c_char_p
    lib.ssd_status_string.argtypes = [c_int]
    lib.ssd_validate_shape.restype = c_int
    lib.ssd_validate_shape.argtypes = [sp]
    lib.ssd_fwd_workspace_layout.restype = c_int
    lib.ssd_fwd_workspace_layout.argtypes = [sp, P(ssd_workspace_layout)]
    lib.ssd_fwd_workspace_size.restype = sz
    lib.ssd_fwd_workspace_size.argtypes = [sp]
    lib.ssd_fwd_kernel_count.restype = c_int
    lib.ssd_fwd_kernel_count.argtypes = [sp]
    lib.ssd_fwd.restype = c_int
    lib.ssd_fwd.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.ssd_fwd_fused.restype = c_int
    lib.ssd_fwd_fused.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.ssd_fwd_range.restype = c_int
    lib.ssd_fwd_range.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, c_int, c_int, vp]
    lib.ssd_fused_pass.restype = c_int
    lib.ssd_fused_pass.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.ssd_causal_cb.restype = c_int
    lib.ssd_causal_cb.argtypes = [sp, vp, vp, vp, sz, vp]
    lib.ssd_fwd_check.restype = c_int
    lib.ssd_fwd_check.argtypes = [vp]
    lib.ssd_chunk_cumsum.restype = c_int
    lib.ssd_chunk_cumsum.argtypes = [sp, vp, vp, vp, sz, vp]
    lib.ssd_chunk_state.restype = c_int
    lib.ssd_chunk_state.argtypes = [sp, vp, vp, vp, sz, vp]
    lib.ssd_state_passing.restype = c_int
    lib.ssd_state_passing.argtypes = [sp, vp, vp, vp, sz, vp]
    lib.ssd_compute_out.restype = c_int
    lib.ssd_compute_out.argtypes = [sp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.ssd_debug_timeout_probe.restype = c_int
    lib.ssd_debug_timeout_probe.argtypes = [vp, ctypes.c_uint32, vp]
    lib.ssd_fwd_static_scratch.restype = c_int
    lib.ssd_fwd_static_scratch.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    return lib


lib = _load()


# ------------------------------------------------------------------ helpers

def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(code: int, where: str) -> None:
    if code != 0:
        raise SSDError(code, where)


def make_shape(batch: int, seqlen: int, nheads: int, headdim: int, ngroups: int, dstate: int,
               chunk_size: int, dtype) -> ssd_shape:
    """Build an ssd_shape; ``dtype`` is torch.float32 / torch.bfloat16 or SSD_F32 / SSD_BF16."""
    if isinstance(dtype, torch.dtype):
        if dtype == torch.float32:
            dtype = SSD_F32
        elif dtype == torch.bfloat16:
            dtype = SSD_BF16
        else:
            raise SSDError(2, f"dtype {dtype}")
    return ssd_shape(batch, seqlen, nheads, headdim, ngroups, dstate, chunk_size, dtype)


def shape_of(x: torch.Tensor, Bm: torch.Tensor, chunk_size: int) -> ssd_shape:
    B, L, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    return make_shape(B, L, H, P, G, N, chunk_size, x.dtype)


def ssd_validate_shape(shape: ssd_shape) -> int:
    return lib.ssd_validate_shape(ctypes.byref(shape))


def ssd_status_string(code: int) -> str:
    return lib.ssd_status_string(code).decode()


def ssd_fwd_workspace_size(shape: ssd_shape) -> int:
    return lib.ssd_fwd_workspace_size(ctypes.byref(shape))


def ssd_fwd_kernel_count(shape: ssd_shape) -> int:
    return lib.ssd_fwd_kernel_count(ctypes.byref(shape))


def ssd_fwd_workspace_layout(shape: ssd_shape) -> Dict[str, int]:
    L = ssd_workspace_layout()
    _check(lib.ssd_fwd_workspace_layout(ctypes.byref(shape), ctypes.byref(L)), "ssd_fwd_workspace_layout")
    return {k: getattr(L, k) for k, _ in ssd_workspace_layout._fields_}


def new_workspace(shape: ssd_shape, device="cuda") -> torch.Tensor:
    n = ssd_fwd_workspace_size(shape)
    if n == 0:
        _check(ssd_validate_shape(shape) or 2, "ssd_fwd_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def workspace_views(shape: ssd_shape, ws: torch.Tensor) -> Dict[str, torch.Tensor]:
    """Typed views of the workspace regions (intermediate results, for tests)."""
    L = ssd_fwd_workspace_layout(shape)
    B, H, P, N, Q = shape.batch, shape.nheads, shape.headdim, shape.dstate, shape.chunk_size
    nc = -(-shape.seqlen // Q)
    Lp = nc * Q

    def view(off, count, dt, dims):
        nbytes = count * torch.tensor([], dtype=dt).element_size()
        return ws[off:off + nbytes].view(dt).view(*dims)
    out = {
        "status": view(L["status"], 1, torch.int32, (1,)),
        "cumsum": view(L["cumsum"], B * H * Lp, torch.float32, (B, H, Lp)),
        "dt_t": view(L["dt_t"], B * H * Lp, torch.float32, (B, H, Lp)),
        "states": view(L["states"], B * nc * H * P * N,
                       torch.bfloat16 if shape.dtype == SSD_BF16 else torch.float32, (B, nc, H, P, N)),
    }
    if shape.dtype == SSD_BF16:
        out["states_bf16"] = view(L["states_bf16"], B * nc * H * P * N, torch.bfloat16, (B, nc, H, P, N))
    out["chain"] = view(L["chain"], 1 + B * (H // 2), torch.int32, (1 + B * (H // 2),))
    out["hslot"] = view(L["hslot"], B * H * P * N, torch.float32, (B * H * P * N,))
    G = shape.ngroups
    if shape.dtype == SSD_BF16:  # causal C B^T per (batch, 128-token window, group)
        nw = -(-shape.seqlen // 128)
        out["cbm"] = view(L["cbm"], B * nw * G * 128 * 128, torch.bfloat16, (B, nw, G, 128, 128))
    return out


def expected_layouts(shape: ssd_shape) -> Dict[str, Tuple[Tuple[int, ...], Tuple[torch.dtype, ...]]]:
    """Shape and dtype every tensor argument must have for ``shape`` (the
    layouts include/ssd.h states): x, y [B,L,H,P] and Bm, Cm [B,L,G,N] in the
    problem dtype; dt [B,L,H], A and D [H], init_state and final_state
    [B,H,P,N] in fp32; the workspace a flat byte buffer."""
    B, L, H, P, G, N = shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.ngroups, shape.dstate
    io = torch.bfloat16 if shape.dtype == SSD_BF16 else torch.float32
    f32 = (torch.float32,)
    return {"x": ((B, L, H, P), (io,)), "y": ((B, L, H, P), (io,)), "Bm": ((B, L, G, N), (io,)),
            "Cm": ((B, L, G, N), (io,)), "dt": ((B, L, H), f32), "A": ((H,), f32), "D": ((H,), f32),
            "init_state": ((B, H, P, N), f32), "final_state": ((B, H, P, N), f32)}


def check_tensors(shape: ssd_shape, device: Optional[torch.device] = None, require_cuda: bool = True,
                  **tensors) -> torch.device:
    """Checks every tensor argument of a call before anything reaches the C
    library: each given tensor (None means "not passed") must live on the same
    CUDA device, be contiguous and have exactly the shape and dtype of
    ``expected_layouts(shape)``; ``workspace`` must be a byte tensor of at least
    ssd_fwd_workspace_size(shape) bytes.  A host tensor or a short buffer would
    otherwise become a device pointer or a tensor map the kernels read or write
    past its end.  Raises SSDError (code 1, or 2 for an unsupported dtype);
    returns the device.  ``require_cuda=False`` is for tests without a GPU."""
    want = expected_layouts(shape)
    for name, t in tensors.items():
        if t is None:
            continue
        if not isinstance(t, torch.Tensor):
            raise SSDError(1, f"{name} must be a torch.Tensor")
        if require_cuda and not t.is_cuda:
            raise SSDError(1, f"{name} must be a contiguous CUDA tensor (got {t.device})")
        if device is None:
            device = t.device
        elif t.device != device:
            raise SSDError(1, f"{name} is on {t.device}, the other arguments on {device}")
        if not t.is_contiguous():
            raise SSDError(1, f"{name} must be a contiguous CUDA tensor")
        if name == "workspace":
            need = ssd_fwd_workspace_size(shape)
            if t.dtype != torch.uint8 or t.dim() != 1:
                raise SSDError(1, "workspace must be a 1-D uint8 tensor")
            if t.numel() < need:
                raise SSDError(3, f"workspace holds {t.numel()} bytes, the shape needs {need}")
            continue
        dims, dtypes = want[name]
        if t.dtype not in dtypes:
            code = 2 if name in ("x", "Bm", "Cm", "y") else 1
            raise SSDError(code, f"{name} has dtype {t.dtype}, expected {dtypes[0]}")
        if tuple(t.shape) != dims:
            raise SSDError(1, f"{name} has shape {tuple(t.shape)}, expected {dims}")
    return device


def _shape_from(x, Bm, chunk_size: int) -> ssd_shape:
    for name, t in (("x", x), ("Bm", Bm)):
        if not isinstance(t, torch.Tensor) or t.dim() != 4:
            raise SSDError(1, f"{name} must be a 4-D tensor")
    if x.dtype not in (torch.float32, torch.bfloat16):
        raise SSDError(2, "x, Bm and Cm must share dtype float32 or bfloat16")
    return shape_of(x, Bm, chunk_size)


# ------------------------------------------------------------------ entry points

def ssd_fwd(x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor, Bm: torch.Tensor, Cm: torch.Tensor,
            D: torch.Tensor, chunk_size: int, init_state: Optional[torch.Tensor] = None,
            y: Optional[torch.Tensor] = None, final_state: Optional[torch.Tensor] = None,
            workspace: Optional[torch.Tensor] = None, stream=None,
            want_final_state: bool = True, schedule: str = "auto") -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """The whole forward pass.  Returns (y, final_state).  ``schedule``:
    "auto" (C: ssd_fwd, which picks the schedule from the shape) or "fused"
    (C: ssd_fwd_fused, the one-pass kernel; bf16 only)."""
    if schedule not in ("auto", "fused"):
        raise ValueError("schedule must be 'auto' or 'fused'")
    shape = _shape_from(x, Bm, chunk_size)
    check_tensors(shape, x=x, dt=dt, A=A, Bm=Bm, Cm=Cm, D=D, init_state=init_state, y=y, final_state=final_state,
                  workspace=workspace)
    B, L, H, P = x.shape
    N = Bm.shape[3]
    if y is None:
        y = torch.empty_like(x)
    if final_state is None and want_final_state:
        final_state = torch.empty(B, H, P, N, dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = new_workspace(shape, x.device)
    fn = lib.ssd_fwd if schedule == "auto" else lib.ssd_fwd_fused
    code = fn(ctypes.byref(shape), _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm), _ptr(D),
              _ptr(init_state), _ptr(y), _ptr(final_state), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(code, "ssd_fwd" if schedule == "auto" else "ssd_fwd_fused")
    return y, final_state


def ssd_fwd_range(x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor, Bm: torch.Tensor, Cm: torch.Tensor,
                  D: torch.Tensor, chunk_size: int, first_launch: int, end_launch: int,
                  init_state: Optional[torch.Tensor] = None, y: Optional[torch.Tensor] = None,
                  final_state: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                  stream=None) -> None:
    """Launches [first_launch, end_launch) of the ones ssd_fwd makes for this
    shape, with all of ssd_fwd's arguments (C: ssd_fwd_range).  The caller
    passes the outputs and the workspace, which consecutive ranges share."""
    shape = _shape_from(x, Bm, chunk_size)
    check_tensors(shape, x=x, dt=dt, A=A, Bm=Bm, Cm=Cm, D=D, init_state=init_state, y=y, final_state=final_state,
                  workspace=workspace)
    if y is None or workspace is None:
        raise SSDError(1, "ssd_fwd_range needs y and the workspace")
    _check(lib.ssd_fwd_range(ctypes.byref(shape), _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm), _ptr(D),
                             _ptr(init_state), _ptr(y), _ptr(final_state), _ptr(workspace), workspace.numel(),
                             int(first_launch), int(end_launch), _stream(stream)), "ssd_fwd_range")


def ssd_fwd_check(workspace: torch.Tensor) -> int:
    """Device status word after the caller synchronised (C: ssd_fwd_check)."""
    return lib.ssd_fwd_check(_ptr(workspace))


def ssd_causal_cb(shape: ssd_shape, Bm: torch.Tensor, Cm: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    """Step 1 of the one-pass schedule: the causal C B^T blocks (C: ssd_causal_cb)."""
    check_tensors(shape, Bm=Bm, Cm=Cm, workspace=workspace)
    _check(lib.ssd_causal_cb(ctypes.byref(shape), _ptr(Bm), _ptr(Cm), _ptr(workspace), workspace.numel(),
                             _stream(stream)), "ssd_causal_cb")


def ssd_fused_pass(shape: ssd_shape, x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor, Bm: torch.Tensor,
                   Cm: torch.Tensor, D: torch.Tensor, init_state: Optional[torch.Tensor], y: torch.Tensor,
                   final_state: Optional[torch.Tensor], workspace: torch.Tensor, stream=None) -> None:
    """Step 2 of the one-pass schedule, after ssd_causal_cb (C: ssd_fused_pass)."""
    check_tensors(shape, x=x, dt=dt, A=A, Bm=Bm, Cm=Cm, D=D, init_state=init_state, y=y, final_state=final_state,
                  workspace=workspace)
    _check(lib.ssd_fused_pass(ctypes.byref(shape), _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm), _ptr(D),
                              _ptr(init_state), _ptr(y), _ptr(final_state), _ptr(workspace), workspace.numel(),
                              _stream(stream)), "ssd_fused_pass")


def ssd_chunk_cumsum(shape: ssd_shape, dt: torch.Tensor, A: torch.Tensor, workspace: torch.Tensor,
                     stream=None) -> None:
    check_tensors(shape, dt=dt, A=A, workspace=workspace)
    _check(lib.ssd_chunk_cumsum(ctypes.byref(shape), _ptr(dt), _ptr(A), _ptr(workspace), workspace.numel(),
                                _stream(stream)), "ssd_chunk_cumsum")


def ssd_chunk_state(shape: ssd_shape, x: torch.Tensor, Bm: torch.Tensor, workspace: torch.Tensor,
                    stream=None) -> None:
    check_tensors(shape, x=x, Bm=Bm, workspace=workspace)
    _check(lib.ssd_chunk_state(ctypes.byref(shape), _ptr(x), _ptr(Bm), _ptr(workspace), workspace.numel(),
                               _stream(stream)), "ssd_chunk_state")


def ssd_state_passing(shape: ssd_shape, init_state: Optional[torch.Tensor], final_state: Optional[torch.Tensor],
                      workspace: torch.Tensor, stream=None) -> None:
    check_tensors(shape, init_state=init_state, final_state=final_state, workspace=workspace)
    _check(lib.ssd_state_passing(ctypes.byref(shape), _ptr(init_state), _ptr(final_state), _ptr(workspace),
                                 workspace.numel(), _stream(stream)), "ssd_state_passing")


def ssd_compute_out(shape: ssd_shape, x: torch.Tensor, Bm: torch.Tensor, Cm: torch.Tensor, D: torch.Tensor,
                    y: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    check_tensors(shape, x=x, Bm=Bm, Cm=Cm, D=D, y=y, workspace=workspace)
    _check(lib.ssd_compute_out(ctypes.byref(shape), _ptr(x), _ptr(Bm), _ptr(Cm), _ptr(D), _ptr(y),
                               _ptr(workspace), workspace.numel(), _stream(stream)), "ssd_compute_out")


def ssd_debug_timeout_probe(workspace: torch.Tensor, limit_us: int, stream=None) -> None:
    _check(lib.ssd_debug_timeout_probe(_ptr(workspace), int(limit_us), _stream(stream)), "ssd_debug_timeout_probe")


_copy_streams_by_device = {}


def _copy_streams(dev: torch.device):
    """Two side streams per device (host-to-device copies, device-to-host copies), created once."""
    key = dev.index
    pair = _copy_streams_by_device.get(key)
    if pair is None:
        pair = (torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev))
        _copy_streams_by_device[key] = pair
    return pair


def host_slices(batch: int, seqlen: int, chunk_size: int, pieces: int):
    """The slices ssd_fwd_host pipelines over, as (b0, b1, l0, l1): up to ``pieces`` batch ranges,
    or, for one sequence, up to ``pieces`` segments whose boundaries are chunk boundaries.
    Together they cover [0, batch) x [0, seqlen) once, in the order they run."""
    pieces = max(1, int(pieces))
    if batch > 1 or pieces == 1:  # batch ranges (segments of several sequences cost more host time than they save)
        n = min(batch, pieces)
        cuts = [(batch * k) // n for k in range(n + 1)]
        return [(cuts[k], cuts[k + 1], 0, seqlen) for k in range(n)]
    nc = -(-seqlen // chunk_size)  # one sequence: segments of whole chunks
    n = min(nc, pieces)
    cuts = [min(seqlen, ((nc * k) // n) * chunk_size) for k in range(n + 1)]
    return [(0, 1, cuts[k], cuts[k + 1]) for k in range(n)]


def ssd_fwd_host(x, dt, A, Bm, Cm, D, chunk_size: int, init_state=None, device="cuda",
                 out_y=None, out_final=None, workspace=None, stream=None, pieces: Optional[int] = None):
    """End-to-end call from host memory: copies the inputs to the device,
    runs ssd_fwd and copies y and the final state back into (pinned) host
    tensors.  Inputs are CPU tensors (pinned for asynchronous copies).
    Returns (y_host, final_host); synchronise the stream before reading them.

    The call is pipelined over ``pieces`` slices (default: one per ~16 MB
    moved, at most 4): slice k + 1's inputs are copied in on one side stream
    while slice k runs on ``stream`` and slice k - 1's outputs are copied out
    on another, so the two copy directions and the kernels overlap.  Slices are
    batch ranges (independent problems); a batch of one is cut along the
    sequence at chunk boundaries instead, each segment starting from the
    previous one's final state (the recurrence resumed, so the chunking is
    unchanged).  Everything is ordered after the work already on ``stream``
    and before the work queued on it later.  Each slice picks its schedule
    from its own shape (as ssd_fwd does)."""
    dev = torch.device(device)
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    st = torch.cuda.current_stream(dev) if stream is None else stream
    B, L, H, P = x.shape
    N = Bm.shape[3]
    if pieces is None:
        # about one slice per 16 MB of copies, at most four (measured with L2 flushed between
        # calls: 370M layer, 74 MB moved: 0.413 ms in two slices against 0.491 in one; 2.7B
        # layer, 370 MB: 1.55 ms in four against 2.14 in one); small problems stay in one
        moved = sum(t.numel() * t.element_size() for t in (x, dt, Bm, Cm)) * 2
        pieces = max(1, min(4, moved // (16 << 20)))
    slices = host_slices(B, L, chunk_size, pieces)
    seq_split = slices[0][3] - slices[0][2] < L
    if out_y is None:
        out_y = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    if out_final is None:
        out_final = torch.empty((B, H, P, N), dtype=torch.float32, pin_memory=True)
    # device buffers (allocated for `st`, which every side stream is ordered against)
    with torch.cuda.stream(st):
        xd, dtd, Bd, Cd = (torch.empty(t.shape, dtype=t.dtype, device=dev) for t in (x, dt, Bm, Cm))
        Ad, Dd = torch.empty(A.shape, dtype=A.dtype, device=dev), torch.empty(D.shape, dtype=D.dtype, device=dev)
        hd = torch.empty(init_state.shape, dtype=init_state.dtype, device=dev) if init_state is not None else None
        yd = torch.empty(x.shape, dtype=x.dtype, device=dev)
        fd = torch.empty((2 if seq_split else 1, B, H, P, N), dtype=torch.float32, device=dev)  # [ping-pong]
        if workspace is None:
            bmax = max(b1 - b0 for b0, b1, _, _ in slices)
            lmax = max(l1 - l0 for _, _, l0, l1 in slices)
            workspace = new_workspace(shape_of(xd[:bmax, :lmax], Bd[:bmax, :lmax], chunk_size), dev)
    cin, cout = _copy_streams(dev)
    cin.wait_stream(st)
    cout.wait_stream(st)
    ev_in = []
    with torch.cuda.stream(cin):
        Ad.copy_(A, non_blocking=True)
        Dd.copy_(D, non_blocking=True)
        if hd is not None:
            hd.copy_(init_state, non_blocking=True)
        for b0, b1, l0, l1 in slices:
            for dst, src in ((xd, x), (dtd, dt), (Bd, Bm), (Cd, Cm)):
                dst[b0:b1, l0:l1].copy_(src[b0:b1, l0:l1], non_blocking=True)
            e = torch.cuda.Event()
            e.record(cin)
            ev_in.append(e)
    for k, (b0, b1, l0, l1) in enumerate(slices):
        st.wait_event(ev_in[k])
        seg = k if seq_split else 0  # segment index within the (single) sequence
        if seq_split:  # a segment resumes from its sequence's previous segment's final state
            h_in = (hd[b0:b1] if hd is not None else None) if seg == 0 else fd[(seg - 1) % 2, b0:b1]
            fin = fd[seg % 2, b0:b1]
        else:
            h_in = hd[b0:b1] if hd is not None else None
            fin = fd[0, b0:b1]
        ssd_fwd(xd[b0:b1, l0:l1], dtd[b0:b1, l0:l1], Ad, Bd[b0:b1, l0:l1], Cd[b0:b1, l0:l1], Dd, chunk_size,
                init_state=h_in, y=yd[b0:b1, l0:l1], final_state=fin, workspace=workspace, stream=st)
        e = torch.cuda.Event()
        e.record(st)
        cout.wait_event(e)
        with torch.cuda.stream(cout):
            out_y[b0:b1, l0:l1].copy_(yd[b0:b1, l0:l1], non_blocking=True)
            if not seq_split or l1 == L:  # a sequence's last slice holds its final state
                out_final[b0:b1].copy_(fin, non_blocking=True)
    st.wait_stream(cout)
    return out_y, out_final


def ssd_fwd_static_scratch(x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor, Bm: torch.Tensor,
                           Cm: torch.Tensor, D: torch.Tensor, chunk_size: int, y: torch.Tensor,
                           final_state: Optional[torch.Tensor] = None,
                           init_state: Optional[torch.Tensor] = None, stream=None) -> None:
    """The forward pass without a workspace argument (C: ssd_fwd_static_scratch).

    For callers that may not allocate device memory: the caller provides the
    inputs and the outputs ``y`` / ``final_state``; the workspace is the
    library's fixed SSD_STATIC_SCRATCH_BYTES device array, shared by every
    call (calls whose GPU work overlaps race).  Nothing is allocated here.
    """
    shape = _shape_from(x, Bm, chunk_size)
    check_tensors(shape, x=x, dt=dt, A=A, Bm=Bm, Cm=Cm, D=D, init_state=init_state, y=y, final_state=final_state)
    if y is None:
        raise SSDError(1, "y is required")
    code = lib.ssd_fwd_static_scratch(ctypes.byref(shape), _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm),
                                      _ptr(D), _ptr(init_state), _ptr(y), _ptr(final_state), _stream(stream))
    _check(code, "ssd_fwd_static_scratch")
