"""The C ABI on a host without a GPU: the library loads, exports every entry point
include/vg.h declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

from self_speculative_sparse_gb300 import binding as vb
from self_speculative_sparse_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return vb.load()


def declared_functions():
    txt = open(os.path.join(ROOT, "include", "vg.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(vg_[a-z_0-9]+)\s*\(", txt)))


def test_every_declared_entry_point_is_exported(lib):
    names = declared_functions()
    assert "vg_verify_attn" in names and "vg_iteration" in names and len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(vb.ENTRY_POINTS)
    assert lib.vg_version() >= 100


def test_library_needs_no_cuda_driver_to_load():
    # The runtime is linked statically; loading resolves no libcuda/libcudart symbol.
    out = os.popen(f"ldd {build.LIB}").read()
    assert "libcudart" not in out and "libcuda.so" not in out


class Buf:
    """A fake 16-byte-aligned device address (never dereferenced by these tests)."""

    def __init__(self, addr=0x10000):
        self.addr = addr

    def data_ptr(self):
        return self.addr


A = Buf(0x10000)
MIS = Buf(0x10004)  # misaligned


def dims(**kw):
    base = dict(B=1, H_q=8, H_kv=2, d=64, gamma=3, max_len=512, scale=0.0)
    base.update(kw)
    return vb.vg_dims(**base)


def cache(K=A, capacity=1024):
    return vb.vg_kv_cache(K.data_ptr(), A.data_ptr(), A.data_ptr(), capacity)


def verify(lib, d=None, c=None, q=A, kn=A, vn=A, plen=A, m0=0x9, m1=0, s0=A, s1=None, stride=512, out=A):
    d = d or dims()
    c = c or cache()
    return lib.vg_verify_attn(ctypes.byref(d), ctypes.byref(c), vb.ptr(q), vb.ptr(kn), vb.ptr(vn), vb.ptr(plen), m0,
                              m1, vb.ptr(s0), vb.ptr(s1), stride, vb.ptr(out), vb.ptr(A), 1 << 30, None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), vb.VG_ERR_UNSUPPORTED_SHAPE),
    (dict(H_q=9), vb.VG_ERR_INVALID_ARG),
    (dict(H_q=64, H_kv=2), vb.VG_ERR_UNSUPPORTED_SHAPE),        # group of 32
    (dict(H_q=64, H_kv=4, gamma=4), vb.VG_ERR_UNSUPPORTED_SHAPE),  # G * (gamma+1) = 80 rows
    (dict(gamma=16), vb.VG_ERR_UNSUPPORTED_SHAPE),
    (dict(B=0), vb.VG_ERR_UNSUPPORTED_SHAPE),
    (dict(max_len=-1), vb.VG_ERR_INVALID_ARG),
    (dict(scale=float("nan")), vb.VG_ERR_INVALID_ARG),
])
def test_verify_rejects_bad_dims(lib, kw, code):
    assert verify(lib, d=dims(**kw)) == code
    assert lib.vg_last_error().decode()


def test_verify_rejects_bad_arguments(lib):
    assert verify(lib, q=None) == vb.VG_ERR_INVALID_ARG
    assert verify(lib, q=MIS) == vb.VG_ERR_INVALID_ARG
    assert verify(lib, vn=None) == vb.VG_ERR_INVALID_ARG          # k_new without v_new
    assert verify(lib, m0=1 << 4) == vb.VG_ERR_INVALID_ARG         # row 4 > gamma = 3
    assert verify(lib, s0=None) == vb.VG_ERR_INVALID_ARG           # mask without its scores
    assert verify(lib, m0=0, s0=A) == vb.VG_ERR_INVALID_ARG        # scores without a mask
    assert verify(lib, stride=100) == vb.VG_ERR_INVALID_ARG        # score_stride < max_len
    assert verify(lib, c=cache(K=MIS)) == vb.VG_ERR_INVALID_ARG
    assert verify(lib, c=cache(capacity=0)) == vb.VG_ERR_INVALID_ARG


def test_valid_verify_call_without_a_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert verify(lib) == vb.VG_ERR_CUDA
    assert lib.vg_workspace_size(ctypes.byref(dims()), 16) == 0


def test_topk_rejects_bad_arguments(lib):
    def call(k=4, max_len=100, B=1, stride=100, scores=A):
        return lib.vg_topk_select(vb.ptr(scores), stride, vb.ptr(A), B, max_len, k, vb.ptr(A), vb.ptr(A), None, 0,
                                  None, None)
    assert call(k=0) == vb.VG_ERR_INVALID_ARG
    assert call(max_len=262145, stride=262145) == vb.VG_ERR_UNSUPPORTED_SHAPE
    assert call(B=0) == vb.VG_ERR_UNSUPPORTED_SHAPE
    assert call(stride=50) == vb.VG_ERR_INVALID_ARG
    assert call(scores=None) == vb.VG_ERR_INVALID_ARG
    assert call(scores=MIS) == vb.VG_ERR_INVALID_ARG


def test_draft_rejects_bad_arguments(lib):
    def call(k_stride=16, tail_len=A, kn=A, vn=A, q=A, noalloc=False, flags=0):
        d, c = dims(), cache()
        if noalloc:
            return lib.vg_sparse_draft_attn_noalloc(ctypes.byref(d), ctypes.byref(c), vb.ptr(q), vb.ptr(kn),
                                                    vb.ptr(vn), vb.ptr(A), vb.ptr(A), k_stride, vb.ptr(A),
                                                    vb.ptr(tail_len), vb.ptr(A), None, None)
        return lib.vg_sparse_draft_attn(ctypes.byref(d), ctypes.byref(c), vb.ptr(q), vb.ptr(kn), vb.ptr(vn),
                                        vb.ptr(A), vb.ptr(A), k_stride, vb.ptr(A), vb.ptr(tail_len), flags,
                                        vb.ptr(A), vb.ptr(A), 1 << 30, None, None)
    for noalloc in (False, True):
        assert call(k_stride=0, noalloc=noalloc) == vb.VG_ERR_INVALID_ARG
        assert call(tail_len=None, noalloc=noalloc) == vb.VG_ERR_INVALID_ARG
        assert call(vn=None, noalloc=noalloc) == vb.VG_ERR_INVALID_ARG
        assert call(q=MIS, noalloc=noalloc) == vb.VG_ERR_INVALID_ARG
    assert call(flags=2) == vb.VG_ERR_INVALID_ARG                      # unknown flag bit


def test_iteration_rejects_bad_arguments(lib):
    d, c = dims(), cache()
    ins = vb.vg_iter_inputs(A.addr, A.addr, A.addr, A.addr, A.addr, A.addr, A.addr)
    outs = vb.vg_iter_outputs(A.addr, A.addr, None, 512, A.addr, A.addr, None, None, A.addr)

    def call(k=16, m0=0x9, m1=0, o=outs):
        return lib.vg_iteration(ctypes.byref(d), ctypes.byref(c), ctypes.byref(ins), k, m0, m1, ctypes.byref(o),
                                vb.ptr(A), 1 << 30, None, None)
    assert call(k=0) == vb.VG_ERR_INVALID_ARG
    assert call(m0=0) == vb.VG_ERR_INVALID_ARG
    assert call(m1=0x2) == vb.VG_ERR_INVALID_ARG                   # mask1 without scores1
    bad = vb.vg_iter_outputs(A.addr, A.addr, None, 512, A.addr, A.addr, A.addr, None, A.addr)
    assert call(o=bad) == vb.VG_ERR_INVALID_ARG                    # idx1 without count1
    assert lib.vg_iteration(None, ctypes.byref(c), ctypes.byref(ins), 16, 1, 0, ctypes.byref(outs), None, 0,
                            None, None) == vb.VG_ERR_INVALID_ARG


def test_iteration_plan_validates_like_the_call_and_leaves_no_handle(lib):
    d, c = dims(), cache()
    ins = vb.vg_iter_inputs(A.addr, A.addr, A.addr, A.addr, A.addr, A.addr, A.addr)
    outs = vb.vg_iter_outputs(A.addr, A.addr, None, 512, A.addr, A.addr, None, None, A.addr)

    def create(k=16, m0=0x9, m1=0, o=outs, dm=d):
        h = ctypes.c_void_p(0x1234)
        code = lib.vg_iteration_plan_create(ctypes.byref(dm) if dm is not None else None, ctypes.byref(c),
                                            ctypes.byref(ins), k, m0, m1, ctypes.byref(o), vb.ptr(A), 1 << 30,
                                            None, ctypes.byref(h))
        return code, h.value
    for kw in (dict(k=0), dict(m0=0), dict(m1=0x2), dict(dm=None), dict(dm=dims(d=80))):
        code, h = create(**kw)
        assert code in (vb.VG_ERR_INVALID_ARG, vb.VG_ERR_UNSUPPORTED_SHAPE), kw
        assert h is None, kw                                          # *plan = NULL on error
    assert lib.vg_iteration_plan_create(ctypes.byref(d), ctypes.byref(c), ctypes.byref(ins), 16, 1, 0,
                                        ctypes.byref(outs), vb.ptr(A), 1 << 30, None, None) == vb.VG_ERR_INVALID_ARG
    assert lib.vg_iteration_plan_launch(None, None) == vb.VG_ERR_INVALID_ARG
    assert lib.vg_iteration_plan_destroy(None) == vb.VG_OK


def test_workspace_size_rejects_bad_dims(lib):
    assert lib.vg_workspace_size(ctypes.byref(dims(d=80)), 16) == 0
    assert lib.vg_workspace_size(ctypes.byref(dims()), 0) == 0


def test_lost_wait_self_test_validates_its_arguments_on_the_host(lib):
    # checked before any CUDA call, so this runs without a device
    for limit in (0, 1000001):
        assert lib.vg_selftest_lost_wait(limit, Buf().addr, None, None) == vb.VG_ERR_INVALID_ARG
    assert lib.vg_selftest_lost_wait(1000, None, None, None) == vb.VG_ERR_INVALID_ARG
    assert lib.vg_selftest_lost_wait(1000, Buf().addr + 2, None, None) == vb.VG_ERR_INVALID_ARG
    assert lib.vg_selftest_lost_wait(1000, Buf().addr, Buf().addr + 4, None) == vb.VG_ERR_INVALID_ARG


@pytest.mark.parametrize("H_kv", [9, 12, 14, 16])
def test_draft_pages_above_1024_elements_are_refused_before_any_device_query(lib, H_kv):
    """One token's K and V pages of every KV head are staged whole; at d = 128 more than
    8 KV heads exceed that.  The draft call, its no-allocation form and the iteration
    (and a plan of it) refuse such a shape on the host, before any CUDA call, so on a
    machine without a GPU the answer is VG_ERR_UNSUPPORTED_SHAPE, not VG_ERR_CUDA."""
    d, c = dims(B=1, H_q=H_kv, H_kv=H_kv, d=128, gamma=1, max_len=64), cache()
    code = lib.vg_sparse_draft_attn(ctypes.byref(d), ctypes.byref(c), vb.ptr(A), vb.ptr(A), vb.ptr(A), vb.ptr(A),
                                    vb.ptr(A), 8, vb.ptr(A), vb.ptr(A), 0, vb.ptr(A), vb.ptr(A), 1 << 30, None, None)
    assert code == vb.VG_ERR_UNSUPPORTED_SHAPE
    code = lib.vg_sparse_draft_attn_noalloc(ctypes.byref(d), ctypes.byref(c), vb.ptr(A), vb.ptr(A), vb.ptr(A),
                                            vb.ptr(A), vb.ptr(A), 8, vb.ptr(A), vb.ptr(A), vb.ptr(A), None, None)
    assert code == vb.VG_ERR_UNSUPPORTED_SHAPE
    ins = vb.vg_iter_inputs(A.addr, A.addr, A.addr, A.addr, A.addr, A.addr, A.addr)
    outs = vb.vg_iter_outputs(A.addr, A.addr, None, 64, A.addr, A.addr, None, None, A.addr)
    assert lib.vg_iteration(ctypes.byref(d), ctypes.byref(c), ctypes.byref(ins), 8, 0x3, 0, ctypes.byref(outs),
                            vb.ptr(A), 1 << 30, None, None) == vb.VG_ERR_UNSUPPORTED_SHAPE
    h = ctypes.c_void_p(0x1234)
    assert lib.vg_iteration_plan_create(ctypes.byref(d), ctypes.byref(c), ctypes.byref(ins), 8, 0x3, 0,
                                        ctypes.byref(outs), vb.ptr(A), 1 << 30, None,
                                        ctypes.byref(h)) == vb.VG_ERR_UNSUPPORTED_SHAPE
    assert h.value is None
    assert "1024" in lib.vg_last_error().decode()
