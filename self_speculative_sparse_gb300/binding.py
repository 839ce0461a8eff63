"""Thin ctypes binding of the C ABI in include/vg.h (argument marshalling only).

Each ``vg_*`` function here has the name and argument order of the C entry point.
Tensor arguments may be torch tensors (their device pointer is passed), raw
integer addresses, or None for NULL.  Every step of the computation runs in
libvg.so's CUDA kernels; nothing here computes.  If the library is missing the
functions raise — there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libvg.so")

VG_OK = 0
VG_ERR_INVALID_ARG = -1
VG_ERR_UNSUPPORTED_SHAPE = -2
VG_ERR_WORKSPACE = -3
VG_ERR_CUDA = -4
VG_ERR_DEVICE_TIMEOUT = -5
VG_ERR_DEVICE_BOUNDS = -6

ENTRY_POINTS = ("vg_verify_attn", "vg_topk_select", "vg_window_select", "vg_sparse_draft_attn", "vg_iteration",
                "vg_iteration_plan_create", "vg_iteration_plan_launch", "vg_iteration_plan_destroy",
                "vg_sparse_draft_attn_noalloc", "vg_workspace_size", "vg_sparse_draft_launches",
                "vg_accept", "vg_accept_workspace_size",
                "vg_last_error", "vg_version", "vg_selftest_lost_wait")


class VgError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"vg status {status}: {message}")
        self.status = status


class vg_dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H_q", ctypes.c_int32), ("H_kv", ctypes.c_int32),
                ("d", ctypes.c_int32), ("gamma", ctypes.c_int32), ("max_len", ctypes.c_int32),
                ("scale", ctypes.c_float)]


class vg_kv_cache(ctypes.Structure):
    _fields_ = [("K", ctypes.c_void_p), ("V", ctypes.c_void_p), ("seq_offset", ctypes.c_void_p),
                ("capacity_slots", ctypes.c_int64), ("page_table", ctypes.c_void_p), ("page_size", ctypes.c_int32),
                ("pages_per_seq", ctypes.c_int32)]


class vg_iter_inputs(ctypes.Structure):
    _fields_ = [("q_verify", ctypes.c_void_p), ("k_verify", ctypes.c_void_p), ("v_verify", ctypes.c_void_p),
                ("q_draft", ctypes.c_void_p), ("k_draft", ctypes.c_void_p), ("v_draft", ctypes.c_void_p),
                ("prefix_len", ctypes.c_void_p)]


class vg_iter_outputs(ctypes.Structure):
    _fields_ = [("out_verify", ctypes.c_void_p), ("scores0", ctypes.c_void_p), ("scores1", ctypes.c_void_p),
                ("score_stride", ctypes.c_int64), ("idx", ctypes.c_void_p), ("count", ctypes.c_void_p),
                ("idx1", ctypes.c_void_p), ("count1", ctypes.c_void_p), ("out_draft", ctypes.c_void_p)]


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libvg.so (built by ``self_speculative_sparse_gb300.build``) and declare its prototypes."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with self_speculative_sparse_gb300.build.build()")
    L = ctypes.CDLL(p)
    vp, i32, i64, u32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_size_t
    L.vg_verify_attn.argtypes = [ctypes.POINTER(vg_dims), ctypes.POINTER(vg_kv_cache), vp, vp, vp, vp, u32, u32,
                                 vp, vp, i64, vp, vp, sz, vp, vp]
    L.vg_verify_attn.restype = i32
    L.vg_topk_select.argtypes = [vp, i64, vp, i32, i32, i32, vp, vp, vp, sz, vp, vp]
    L.vg_topk_select.restype = i32
    L.vg_window_select.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp]
    L.vg_window_select.restype = i32
    L.vg_sparse_draft_attn.argtypes = [ctypes.POINTER(vg_dims), ctypes.POINTER(vg_kv_cache), vp, vp, vp, vp, vp,
                                       i32, vp, vp, u32, vp, vp, sz, vp, vp]
    L.vg_sparse_draft_attn.restype = i32
    L.vg_sparse_draft_attn_noalloc.argtypes = [ctypes.POINTER(vg_dims), ctypes.POINTER(vg_kv_cache), vp, vp, vp,
                                               vp, vp, i32, vp, vp, vp, vp, vp]
    L.vg_sparse_draft_attn_noalloc.restype = i32
    L.vg_iteration.argtypes = [ctypes.POINTER(vg_dims), ctypes.POINTER(vg_kv_cache), ctypes.POINTER(vg_iter_inputs),
                               i32, u32, u32, ctypes.POINTER(vg_iter_outputs), vp, sz, vp, vp]
    L.vg_iteration.restype = i32
    L.vg_iteration_plan_create.argtypes = [ctypes.POINTER(vg_dims), ctypes.POINTER(vg_kv_cache),
                                           ctypes.POINTER(vg_iter_inputs), i32, u32, u32,
                                           ctypes.POINTER(vg_iter_outputs), vp, sz, vp, ctypes.POINTER(vp)]
    L.vg_iteration_plan_create.restype = i32
    L.vg_iteration_plan_launch.argtypes = [vp, vp]
    L.vg_iteration_plan_launch.restype = i32
    L.vg_iteration_plan_destroy.argtypes = [vp]
    L.vg_iteration_plan_destroy.restype = i32
    L.vg_workspace_size.argtypes = [ctypes.POINTER(vg_dims), i32]
    L.vg_workspace_size.restype = sz
    L.vg_accept_workspace_size.argtypes = [i32, i32, i32]
    L.vg_accept_workspace_size.restype = sz
    L.vg_accept.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp, u32, vp, vp, vp, vp, sz, vp, vp]
    L.vg_accept.restype = i32
    L.vg_sparse_draft_launches.argtypes = [ctypes.POINTER(vg_dims), i32, i32]
    L.vg_sparse_draft_launches.restype = i32
    L.vg_last_error.argtypes = []
    L.vg_last_error.restype = ctypes.c_char_p
    L.vg_version.argtypes = []
    L.vg_version.restype = i32
    L.vg_selftest_lost_wait.argtypes = [u32, vp, vp, vp]
    L.vg_selftest_lost_wait.restype = i32
    if path is None:
        _lib = L
    return L


def ptr(x) -> int | None:
    """Device (or host) address of a tensor-like argument; None stays NULL."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(st: int) -> None:
    if st != VG_OK:
        raise VgError(st, load().vg_last_error().decode())


def make_dims(B, H_q, H_kv, d, gamma, max_len, scale=0.0) -> vg_dims:
    return vg_dims(B, H_q, H_kv, d, gamma, max_len, scale)


def make_cache(K, V, seq_offset, capacity_slots: int | None = None, page_table=None, page_size: int = 0) -> vg_kv_cache:
    """The cache struct: a slot pool located by seq_offset, or pages through page_table
    (int32 [B][pages_per_seq] tensor)."""
    cap = capacity_slots if capacity_slots is not None else K.shape[0]
    if page_table is None:
        return vg_kv_cache(ptr(K), ptr(V), ptr(seq_offset), cap, None, 0, 0)
    return vg_kv_cache(ptr(K), ptr(V), ptr(seq_offset), cap, ptr(page_table), page_size, page_table.shape[1])


def vg_sparse_draft_launches(dims: vg_dims, k_stride: int, tail_len_max: int = 0) -> int:
    """Kernels one vg_sparse_draft_attn call enqueues (1 or 2) for these dimensions."""
    n = load().vg_sparse_draft_launches(ctypes.byref(dims), k_stride, tail_len_max)
    if n == 0:
        raise VgError(VG_ERR_INVALID_ARG, load().vg_last_error().decode())
    return n


def vg_workspace_size(dims: vg_dims, k: int) -> int:
    n = load().vg_workspace_size(ctypes.byref(dims), k)
    if n == 0:
        raise VgError(VG_ERR_INVALID_ARG, load().vg_last_error().decode())
    return n


def vg_verify_attn(dims, cache, q, k_new, v_new, prefix_len, row_mask0, row_mask1, scores0, scores1,
                   score_stride, out, ws, ws_bytes=None, dev_status=None, stream=None) -> None:
    wsb = ws_bytes if ws_bytes is not None else (ws.numel() * ws.element_size() if ws is not None else 0)
    _check(load().vg_verify_attn(ctypes.byref(dims), ctypes.byref(cache), ptr(q), ptr(k_new), ptr(v_new),
                                 ptr(prefix_len), row_mask0, row_mask1, ptr(scores0), ptr(scores1),
                                 score_stride, ptr(out), ptr(ws), wsb, ptr(dev_status), _stream(stream)))


def vg_topk_select(scores, score_stride, len_, B, max_len, k, idx, count, ws=None, ws_bytes=0,
                   dev_status=None, stream=None) -> None:
    _check(load().vg_topk_select(ptr(scores), score_stride, ptr(len_), B, max_len, k, ptr(idx), ptr(count),
                                 ptr(ws), ws_bytes, ptr(dev_status), _stream(stream)))


def vg_window_select(len_, B, max_len, k, idx, count, dev_status=None, stream=None) -> None:
    """The last min(k, len) positions of each sequence (the sliding-window baseline)."""
    _check(load().vg_window_select(ptr(len_), B, max_len, k, ptr(idx), ptr(count), ptr(dev_status), _stream(stream)))


VG_ACCEPT_GREEDY = 0
VG_ACCEPT_SAMPLE = 1


def vg_accept_workspace_size(B: int, gamma: int, V: int) -> int:
    n = load().vg_accept_workspace_size(B, gamma, V)
    if n == 0:
        raise VgError(VG_ERR_UNSUPPORTED_SHAPE, load().vg_last_error().decode())
    return n


def vg_accept(B, gamma, V, p_logits, q_logits, draft_tokens, u_accept, u_resample, mode, n_accept, next_token,
              advance_len, ws, ws_bytes=None, dev_status=None, stream=None) -> None:
    """Acceptance of the draft chain (greedy or speculative sampling) on given logits."""
    wsb = ws_bytes if ws_bytes is not None else (ws.numel() * ws.element_size() if ws is not None else 0)
    _check(load().vg_accept(B, gamma, V, ptr(p_logits), ptr(q_logits), ptr(draft_tokens), ptr(u_accept),
                            ptr(u_resample), mode, ptr(n_accept), ptr(next_token), ptr(advance_len), ptr(ws), wsb,
                            ptr(dev_status), _stream(stream)))


VG_DRAFT_SELECTION_SETTLED = 1


def vg_sparse_draft_attn(dims, cache, q, k_new, v_new, idx, count, k_stride, tail_start, tail_len, out, ws,
                         ws_bytes=None, dev_status=None, stream=None, flags: int = 0) -> None:
    wsb = ws_bytes if ws_bytes is not None else (ws.numel() * ws.element_size() if ws is not None else 0)
    _check(load().vg_sparse_draft_attn(ctypes.byref(dims), ctypes.byref(cache), ptr(q), ptr(k_new), ptr(v_new),
                                       ptr(idx), ptr(count), k_stride, ptr(tail_start), ptr(tail_len), flags,
                                       ptr(out), ptr(ws), wsb, ptr(dev_status), _stream(stream)))


def vg_iteration(dims, cache, inputs: vg_iter_inputs, k, row_mask0, row_mask1, outputs: vg_iter_outputs, ws,
                 ws_bytes=None, dev_status=None, stream=None) -> None:
    wsb = ws_bytes if ws_bytes is not None else (ws.numel() * ws.element_size() if ws is not None else 0)
    _check(load().vg_iteration(ctypes.byref(dims), ctypes.byref(cache), ctypes.byref(inputs), k, row_mask0,
                               row_mask1, ctypes.byref(outputs), ptr(ws), wsb, ptr(dev_status), _stream(stream)))


def vg_iteration_plan_create(dims, cache, inputs: vg_iter_inputs, k, row_mask0, row_mask1,
                             outputs: vg_iter_outputs, ws, ws_bytes=None, dev_status=None) -> int:
    """Capture vg_iteration for these arguments; returns the plan handle (destroy it)."""
    wsb = ws_bytes if ws_bytes is not None else (ws.numel() * ws.element_size() if ws is not None else 0)
    h = ctypes.c_void_p()
    _check(load().vg_iteration_plan_create(ctypes.byref(dims), ctypes.byref(cache), ctypes.byref(inputs), k,
                                           row_mask0, row_mask1, ctypes.byref(outputs), ptr(ws), wsb,
                                           ptr(dev_status), ctypes.byref(h)))
    return h.value


def vg_iteration_plan_launch(plan: int, stream=None) -> None:
    _check(load().vg_iteration_plan_launch(plan, _stream(stream)))


def vg_iteration_plan_destroy(plan: int | None) -> None:
    _check(load().vg_iteration_plan_destroy(plan))


def vg_sparse_draft_attn_noalloc(dims, cache, q, k_new, v_new, idx, count, k_stride, tail_start, tail_len, out,
                                 dev_status=None, stream=None) -> None:
    """vg_sparse_draft_attn with the library's built-in scratch area instead of a workspace."""
    _check(load().vg_sparse_draft_attn_noalloc(ctypes.byref(dims), ctypes.byref(cache), ptr(q), ptr(k_new),
                                               ptr(v_new), ptr(idx), ptr(count), k_stride, ptr(tail_start),
                                               ptr(tail_len), ptr(out), ptr(dev_status), _stream(stream)))


def vg_selftest_lost_wait(limit_us, dev_status, elapsed_ns=None, stream=None) -> None:
    """Self-test of the bounded waits: a wait that nothing completes gives up after limit_us."""
    _check(load().vg_selftest_lost_wait(limit_us, ptr(dev_status), ptr(elapsed_ns), _stream(stream)))
