"""C ABI checks that need no GPU: the library builds and loads, exports every
entry point include/ssd.h declares, and its host-side argument logic (shape
validation, workspace sizing and layout, argument errors) behaves as the header
documents.  No call here reaches a CUDA kernel."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssd.h")


@pytest.fixture(scope="module")
def ext():
    import __graft_entry__
    __graft_entry__.build()
    import mamba_ssd_forward_chunked_gb300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssd_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    names = declared_functions()
    for n in ("ssd_fwd", "ssd_fwd_workspace_size", "ssd_fwd_check", "ssd_status_string", "ssd_chunk_cumsum",
              "ssd_chunk_state", "ssd_state_passing", "ssd_compute_out"):
        assert n in names


def test_library_exports_every_declared_symbol(ext):
    lib = ctypes.CDLL(ext.LIB_PATH)
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in include/ssd.h but not exported"
    assert set(declared_functions()) == set(ext.EXPORTS)


def test_status_strings(ext):
    for code in range(6):
        assert ext.ssd_status_string(code).startswith(ext.STATUS[code])


def shape(ext, **kw):
    base = dict(batch=2, seqlen=2048, nheads=32, headdim=64, ngroups=1, dstate=128, chunk_size=256, dtype=ext.SSD_F32)
    base.update(kw)
    return ext.make_shape(**base)


def test_validate_shape(ext):
    assert ext.ssd_validate_shape(shape(ext)) == 0
    assert ext.ssd_validate_shape(shape(ext, dtype=ext.SSD_BF16, nheads=80)) == 0
    for bad in (dict(headdim=32), dict(dstate=96), dict(chunk_size=100), dict(chunk_size=512),
                dict(nheads=3, ngroups=1), dict(nheads=8, ngroups=3), dict(dtype=7)):
        assert ext.ssd_validate_shape(shape(ext, **bad)) == 2, bad
    for bad in (dict(batch=-1), dict(seqlen=-5), dict(nheads=0), dict(chunk_size=0)):
        assert ext.ssd_validate_shape(shape(ext, **bad)) == 1, bad
    assert ext.ssd_validate_shape(shape(ext, batch=0)) == 0
    assert ext.ssd_validate_shape(shape(ext, seqlen=0)) == 0


def test_workspace_layout(ext):
    for dt in (ext.SSD_F32, ext.SSD_BF16):
        for L in (1, 255, 256, 2048, 2049):
            s = shape(ext, seqlen=L, dtype=dt)
            lay = ext.ssd_fwd_workspace_layout(s)
            nc = -(-L // 256)
            Lp = nc * 256
            assert all(v % 1024 == 0 for v in lay.values())
            assert lay["dt_t"] - lay["cumsum"] >= 2 * 32 * Lp * 4
            es = 2 if dt == ext.SSD_BF16 else 4
            assert lay["states_bf16"] - lay["states"] >= 2 * nc * 32 * 64 * 128 * es
            extra = 2 * nc * 32 * 64 * 128 * 2 if dt == ext.SSD_BF16 else 0
            assert lay["total"] >= lay["states_bf16"] + extra
            assert lay["cbm"] >= lay["hslot"] + 2 * 32 * 64 * 128 * 4
            # bf16: the causal C B^T block of every (batch, 128-token window, group)
            cbm = 2 * (-(-L // 128)) * 1 * 128 * 128 * 2 if dt == ext.SSD_BF16 else 0
            assert lay["total"] - lay["cbm"] >= cbm
            assert ext.ssd_fwd_workspace_size(s) == lay["total"]
    assert ext.ssd_fwd_workspace_size(shape(ext, dstate=100)) == 0


def test_argument_errors_before_any_launch(ext):
    s = shape(ext)
    need = ext.ssd_fwd_workspace_size(s)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: every case fails its checks first
    lib = ext.lib
    by = ctypes.byref
    # workspace too small
    assert lib.ssd_fwd(by(s), fake, fake, fake, fake, fake, fake, None, fake, None, fake, need - 1, None) == 3
    # null input
    assert lib.ssd_fwd(by(s), None, fake, fake, fake, fake, fake, None, fake, None, fake, need, None) == 1
    # misaligned x
    odd = ctypes.c_void_p((1 << 20) + 4)
    assert lib.ssd_fwd(by(s), odd, fake, fake, fake, fake, fake, None, fake, None, fake, need, None) == 1
    # null / misaligned workspace
    assert lib.ssd_fwd(by(s), fake, fake, fake, fake, fake, fake, None, fake, None, None, need, None) == 1
    assert lib.ssd_fwd(by(s), fake, fake, fake, fake, fake, fake, None, fake, None, odd, need, None) == 1
    # unsupported shape
    bad = shape(ext, dstate=96)
    assert lib.ssd_fwd(by(bad), fake, fake, fake, fake, fake, fake, None, fake, None, fake, need, None) == 2
    assert lib.ssd_fwd_check(None) == 1
    # launch ranges: a negative start or an inverted range, then the same checks as ssd_fwd
    for a, b in ((-1, 1), (2, 1)):
        assert lib.ssd_fwd_range(by(s), fake, fake, fake, fake, fake, fake, None, fake, None, fake, need, a, b,
                                 None) == 1
    assert lib.ssd_fwd_range(by(s), None, fake, fake, fake, fake, fake, None, fake, None, fake, need, 0, 1,
                             None) == 1
    assert lib.ssd_fwd_range(by(s), fake, fake, fake, fake, fake, fake, None, fake, None, fake, need - 1, 0, 1,
                             None) == 3
    assert lib.ssd_debug_timeout_probe(None, 10, None) == 1
    assert lib.ssd_debug_timeout_probe(fake, 0, None) == 1


def test_empty_batch_needs_no_device(ext):
    s = shape(ext, batch=0)
    ws = ctypes.c_void_p(1 << 20)
    n = ext.ssd_fwd_workspace_size(s)
    assert ext.lib.ssd_fwd(ctypes.byref(s), None, None, None, None, None, None, None, None, None, ws, n, None) == 0
    assert ext.ssd_fwd_kernel_count(s) == 0
    assert ext.ssd_fwd_kernel_count(shape(ext)) == 3  # fp32 staged: chunk_state forms the cumsum
    assert ext.ssd_fwd_kernel_count(shape(ext, dtype=ext.SSD_BF16, dstate=256)) == 3  # bf16 staged


def test_workspace_views_are_disjoint_and_inside(ext):
    """The typed views the tests read (workspace_views) lie inside the workspace
    and never share a byte, for both dtypes and a ragged length."""
    import torch
    for dt in (ext.SSD_F32, ext.SSD_BF16):
        for L, G in ((300, 1), (2048, 2)):
            s = shape(ext, seqlen=L, dtype=dt, ngroups=G)
            ws = torch.zeros(ext.ssd_fwd_workspace_size(s), dtype=torch.uint8)
            base = ws.data_ptr()
            spans = []
            for name, v in ext.workspace_views(s, ws).items():
                lo = v.data_ptr() - base
                hi = lo + v.numel() * v.element_size()
                assert 0 <= lo < hi <= ws.numel(), name
                spans.append((lo, hi, name))
            spans.sort()
            for (a0, a1, na), (b0, b1, nb) in zip(spans, spans[1:]):
                assert a1 <= b0, (na, nb)
            assert ("cbm" in dict((n, 1) for _, _, n in spans)) == (dt == ext.SSD_BF16)


def test_step_entry_points_reject_bad_arguments_before_any_launch(ext):
    """Every step entry point checks its workspace, pointers and alignment (and
    the one-pass ones the dtype) before touching the device; the static-scratch
    entry point rejects a problem whose workspace exceeds its array.  All the
    pointers are fake and never dereferenced."""
    lib, by = ext.lib, ctypes.byref
    fake, odd4, odd2 = ctypes.c_void_p(1 << 20), ctypes.c_void_p((1 << 20) + 4), ctypes.c_void_p((1 << 20) + 2)
    for dt in (ext.SSD_F32, ext.SSD_BF16):
        s = shape(ext, dtype=dt)
        need = ext.ssd_fwd_workspace_size(s)
        # workspace: too small, missing, misaligned
        for call in (lambda w, n: lib.ssd_chunk_cumsum(by(s), fake, fake, w, n, None),
                     lambda w, n: lib.ssd_chunk_state(by(s), fake, fake, w, n, None),
                     lambda w, n: lib.ssd_state_passing(by(s), None, None, w, n, None),
                     lambda w, n: lib.ssd_compute_out(by(s), fake, fake, fake, fake, fake, w, n, None)):
            assert call(fake, need - 1) == 3
            assert call(None, need) == 1
            assert call(odd4, need) == 1
        assert lib.ssd_chunk_cumsum(by(s), None, fake, fake, need, None) == 1
        assert lib.ssd_chunk_cumsum(by(s), fake, odd2, fake, need, None) == 1
        assert lib.ssd_chunk_state(by(s), None, fake, fake, need, None) == 1
        assert lib.ssd_chunk_state(by(s), fake, odd4, fake, need, None) == 1
        assert lib.ssd_state_passing(by(s), odd4, None, fake, need, None) == 1
        assert lib.ssd_state_passing(by(s), None, odd4, fake, need, None) == 1
        assert lib.ssd_compute_out(by(s), fake, fake, fake, fake, None, fake, need, None) == 1
        assert lib.ssd_compute_out(by(s), fake, fake, odd4, fake, fake, fake, need, None) == 1
        assert lib.ssd_compute_out(by(s), fake, fake, fake, odd2, fake, fake, need, None) == 1
        if dt == ext.SSD_F32:  # the one-pass schedule is bf16 only
            assert lib.ssd_fused_pass(by(s), fake, fake, fake, fake, fake, fake, None, fake, None, fake, need,
                                      None) == 2
            assert lib.ssd_fwd_fused(by(s), fake, fake, fake, fake, fake, fake, None, fake, None, fake, need,
                                     None) == 2
            assert lib.ssd_causal_cb(by(s), fake, fake, fake, need, None) == 2
        else:
            assert lib.ssd_fused_pass(by(s), None, fake, fake, fake, fake, fake, None, fake, None, fake, need,
                                      None) == 1
            assert lib.ssd_fused_pass(by(s), fake, fake, fake, fake, fake, fake, odd4, fake, None, fake, need,
                                      None) == 1
            assert lib.ssd_fused_pass(by(s), fake, odd2, fake, fake, fake, fake, None, fake, None, fake, need,
                                      None) == 1
            assert lib.ssd_causal_cb(by(s), None, fake, fake, need, None) == 1
            assert lib.ssd_causal_cb(by(s), fake, odd4, fake, need, None) == 1
            assert lib.ssd_causal_cb(by(s), fake, fake, fake, need - 1, None) == 3
    big = shape(ext, batch=4, seqlen=4096, nheads=80, dtype=ext.SSD_BF16)
    assert ext.ssd_fwd_workspace_size(big) > (32 << 20)
    assert lib.ssd_fwd_static_scratch(by(big), fake, fake, fake, fake, fake, fake, None, fake, None, None) == 3
    assert lib.ssd_fwd_static_scratch(by(shape(ext, dstate=96)), fake, fake, fake, fake, fake, fake, None, fake,
                                      None, None) == 2


def test_binding_refuses_host_tensors(ext):
    """The Python entry points run only on the GPU path: host (CPU) tensors are
    rejected with an error, never computed some other way."""
    import torch
    x = torch.zeros(1, 64, 2, 64)
    dt, A, D = torch.zeros(1, 64, 2), torch.zeros(2), torch.zeros(2)
    Bm = Cm = torch.zeros(1, 64, 1, 64)
    with pytest.raises(ext.SSDError) as e:
        ext.ssd_fwd(x, dt, A, Bm, Cm, D, 64)
    assert e.value.code == 1 and "CUDA" in str(e.value)


def test_binding_checks_every_tensor_argument(ext):
    """Every tensor a call passes is checked against the shape before the C
    library sees it: device (host tensors and mixed devices), dtype, exact
    shape, contiguity and the workspace's size.  A host output, a short Cm or
    an undersized buffer would otherwise reach the kernels as a bad pointer."""
    import torch
    s = ext.make_shape(2, 64, 4, 64, 1, 64, 64, ext.SSD_F32)
    lay = ext.expected_layouts(s)
    good = {k: torch.zeros(dims, dtype=dts[0]) for k, (dims, dts) in lay.items()}
    ws = torch.zeros(ext.ssd_fwd_workspace_size(s), dtype=torch.uint8)
    # the full argument set passes (no GPU: the CUDA requirement is lifted for the test)
    ext.check_tensors(s, require_cuda=False, workspace=ws, **good)

    def rejects(code, **bad):
        args = dict(good, workspace=ws)
        args.update(bad)
        with pytest.raises(ext.SSDError) as e:
            ext.check_tensors(s, require_cuda=False, **args)
        assert e.value.code == code, (bad.keys(), e.value)

    rejects(1, Cm=torch.zeros(2, 63, 1, 64))                      # short Cm
    rejects(1, dt=torch.zeros(2, 64, 3))                          # dt for fewer heads
    rejects(1, D=torch.zeros(5))                                  # D for more heads
    rejects(1, final_state=torch.zeros(2, 4, 64, 32))             # undersized final state
    rejects(1, init_state=torch.zeros(2, 4, 64, 64, dtype=torch.float64))
    rejects(2, y=torch.zeros(2, 64, 4, 64, dtype=torch.bfloat16))  # y in another dtype than x
    rejects(1, y=torch.zeros(2, 64, 64, 4).transpose(2, 3))       # right shape, not contiguous
    rejects(3, workspace=ws[:-1])                                 # workspace one byte short
    rejects(1, workspace=torch.zeros(ws.numel() // 4, dtype=torch.int32))
    rejects(1, y=torch.zeros(2, 64, 4, 64, device="meta"))        # another device than the rest
    # with the CUDA requirement (the default), any host tensor is refused, outputs included
    for name in ("y", "final_state", "init_state", "workspace"):
        t = ws if name == "workspace" else good[name]
        with pytest.raises(ext.SSDError) as e:
            ext.check_tensors(s, **{name: t})
        assert e.value.code == 1 and "CUDA" in str(e.value)
