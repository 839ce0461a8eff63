"""Device-resident state of one Vegas layer and the calls that run on it.

``LayerState`` owns the torch tensors the C ABI works on: the token-granular KV
slot pool, per-sequence offsets and lengths, the iteration's inputs, output
buffers, the workspace and the device status word.  Its methods only marshal
arguments to libvg.so (via ``binding``); PyTorch serves as the allocator and the
stream provider.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as vb


def bf16_tensor(a: np.ndarray, device) -> torch.Tensor:
    """bf16 bit patterns (numpy uint16) -> a torch.bfloat16 tensor on `device`."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """torch.bfloat16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class LayerState:
    """One layer's cache, inputs and outputs on the GPU.

    pool: the dict produced by ``Workload.layer_pool`` (host arrays)."""

    def __init__(self, w, pool: dict, device="cuda", k: int | None = None, mask0: int | None = None,
                 mask1: int | None = None, max_len: int | None = None):
        self.w = w
        self.device = torch.device(device)
        dev = self.device
        self.B, self.Hq, self.Hkv, self.d, self.gamma = w.B, w.Hq, w.Hkv, w.d, w.gamma
        self.k = w.k if k is None else k
        self.max_len = int(pool["prefix_len"].max()) if max_len is None else max_len
        self.mask0 = w.row_mask(w.select_rows) if mask0 is None else mask0
        self.mask1 = w.row_mask(w.extra_rows) if mask1 is None else mask1
        self.K = bf16_tensor(pool["K"], dev)
        self.V = bf16_tensor(pool["V"], dev)
        self.seq_offset = torch.from_numpy(pool["seq_offset"].astype(np.int64)).to(dev)
        self.prefix_len = torch.from_numpy(pool["prefix_len"].astype(np.int32)).to(dev)
        self.q_verify = bf16_tensor(pool["q_verify"], dev)
        self.k_new = bf16_tensor(pool["k_new"], dev)
        self.v_new = bf16_tensor(pool["v_new"], dev)
        self.q_draft = bf16_tensor(pool["q_draft"], dev)
        self.k_draft = bf16_tensor(pool["k_draft"], dev)
        self.v_draft = bf16_tensor(pool["v_draft"], dev)
        self.dims = vb.make_dims(self.B, self.Hq, self.Hkv, self.d, self.gamma, self.max_len)
        if "page_table" in pool:  # a paged layout of the same layer (seq_offset then unused)
            self.page_table = torch.from_numpy(pool["page_table"].astype(np.int32)).to(dev)
            self.cache = vb.make_cache(self.K, self.V, None, page_table=self.page_table,
                                       page_size=int(pool["page_size"]))
        else:
            self.page_table = None
            self.cache = vb.make_cache(self.K, self.V, self.seq_offset)
        R = self.gamma + 1
        self.score_stride = max(4, (self.max_len + 3) // 4 * 4)
        self.out_verify = torch.empty(self.B, R, self.Hq, self.d, dtype=torch.bfloat16, device=dev)
        self.scores0 = torch.zeros(self.B, self.score_stride, dtype=torch.float32, device=dev)
        self.scores1 = (torch.zeros(self.B, self.score_stride, dtype=torch.float32, device=dev)
                        if self.mask1 else None)
        self.idx = torch.empty(self.B, self.k, dtype=torch.int32, device=dev)
        self.count = torch.empty(self.B, dtype=torch.int32, device=dev)
        self.idx1 = torch.empty(self.B, self.k, dtype=torch.int32, device=dev) if self.mask1 else None
        self.count1 = torch.empty(self.B, dtype=torch.int32, device=dev) if self.mask1 else None
        self.out_draft = torch.empty(max(self.gamma, 1), self.B, self.Hq, self.d, dtype=torch.bfloat16, device=dev)
        self.ws_bytes = vb.vg_workspace_size(self.dims, self.k)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    # --------------------------------------------------------------- calls
    def _iter_args(self, select_extra: bool):
        ins = vb.vg_iter_inputs(vb.ptr(self.q_verify), vb.ptr(self.k_new), vb.ptr(self.v_new), vb.ptr(self.q_draft),
                                vb.ptr(self.k_draft), vb.ptr(self.v_draft), vb.ptr(self.prefix_len))
        outs = vb.vg_iter_outputs(vb.ptr(self.out_verify), vb.ptr(self.scores0), vb.ptr(self.scores1),
                                  self.score_stride, vb.ptr(self.idx), vb.ptr(self.count),
                                  vb.ptr(self.idx1) if select_extra else None,
                                  vb.ptr(self.count1) if select_extra else None, vb.ptr(self.out_draft))
        return ins, outs

    def iteration(self, stream=None, select_extra: bool = True) -> None:
        """verify -> select -> gamma draft steps, one C call."""
        ins, outs = self._iter_args(select_extra)
        vb.vg_iteration(self.dims, self.cache, ins, self.k, self.mask0, self.mask1, outs, self.ws,
                        dev_status=self.status, stream=stream)

    def plan(self, select_extra: bool = True) -> "IterationPlan":
        """The iteration on this state's current buffers, captured once (vg_iteration_plan_*)."""
        ins, outs = self._iter_args(select_extra)
        h = vb.vg_iteration_plan_create(self.dims, self.cache, ins, self.k, self.mask0, self.mask1, outs, self.ws,
                                        dev_status=self.status)
        return IterationPlan(h, [v for v in vars(self).values() if isinstance(v, torch.Tensor)])

    def verify(self, stream=None, append: bool = True) -> None:
        vb.vg_verify_attn(self.dims, self.cache, self.q_verify, self.k_new if append else None,
                          self.v_new if append else None, self.prefix_len, self.mask0, self.mask1, self.scores0,
                          self.scores1, self.score_stride, self.out_verify, self.ws, dev_status=self.status,
                          stream=stream)

    def select(self, stream=None, which: int = 0) -> None:
        sc, idx, cnt = (self.scores0, self.idx, self.count) if which == 0 else (self.scores1, self.idx1, self.count1)
        vb.vg_topk_select(sc, self.score_stride, self.prefix_len, self.B, self.max_len, self.k, idx, cnt,
                          dev_status=self.status, stream=stream)

    def draft_step(self, s: int, tail_len: torch.Tensor, stream=None, settled: bool | None = None) -> None:
        """Draft step s: attend idx U [n_b, n_b + s], appending draft token s at n_b + s.

        settled (default: s > 0): the selection was made before the kernel preceding this
        call, as it is for every step of a draft phase after the first."""
        settled = s > 0 if settled is None else settled
        vb.vg_sparse_draft_attn(self.dims, self.cache, self.q_draft[s], self.k_draft[s], self.v_draft[s], self.idx,
                                self.count, self.k, self.prefix_len, tail_len, self.out_draft[s], self.ws,
                                dev_status=self.status, stream=stream,
                                flags=vb.VG_DRAFT_SELECTION_SETTLED if settled else 0)

    def launches_per_iteration(self, select_extra: bool = False, tail_from_device: bool = False) -> int:
        """Kernels one iteration enqueues: the verify kernel and its combine, one selection
        (two with select_extra), and each draft step's kernels (vg_iteration gives step s a
        host-known tail of s + 1; the per-step calls here pass a device tail array)."""
        draft = sum(vb.vg_sparse_draft_launches(self.dims, self.k, 0 if tail_from_device else s + 1)
                    for s in range(self.gamma))
        return 2 + (2 if select_extra and self.mask1 else 1) + draft

    def check_status(self) -> int:
        return int(self.status.item())


class IterationPlan:
    """An owned vg_iteration_plan.  It holds the tensors it was captured on, so they stay
    allocated at the same addresses for as long as the plan lives."""

    def __init__(self, handle: int, tensors: list):
        self.handle = handle
        self._tensors = tensors

    def launch(self, stream=None) -> None:
        if not self.handle:
            raise RuntimeError("the plan was closed")
        vb.vg_iteration_plan_launch(self.handle, stream)

    def close(self) -> None:
        if self.handle:
            vb.vg_iteration_plan_destroy(self.handle)
            self.handle = None
        self._tensors = []

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
