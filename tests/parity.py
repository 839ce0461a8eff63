"""Helpers shared by the GPU parity tests: tolerances and per-sequence oracle checks.

Tolerances (fixed for the hot path):
  attention outputs  |gpu - oracle| <= 2e-3 + 1e-2 * |oracle|   (element-wise)
  aggregated scores  |gpu - oracle| <= 1e-3 * max_i |oracle_i|   (per sequence)
  top-k indices      bit-exact against the oracle's selection run on the GPU's own
                     scores (the decision is taken in the kernel's fp32)
"""
from __future__ import annotations

import numpy as np

import oracle
from oracle import widen_bf16

ATOL, RTOL = 2e-3, 1e-2
SCORE_REL = 1e-3


def bf16_to_f64(t) -> np.ndarray:
    """torch bf16 tensor (any device) -> float64 numpy (exact)."""
    import torch
    bits = t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return widen_bf16(bits)


def assert_attn_close(gpu: np.ndarray, ref: np.ndarray, what: str) -> None:
    err = np.abs(gpu - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; worst at {i}: "
                             f"gpu={gpu[i]!r} oracle={ref[i]!r}")


def assert_scores_close(gpu: np.ndarray, ref: np.ndarray, what: str) -> None:
    if ref.size == 0:
        return
    tol = SCORE_REL * np.abs(ref).max()
    err = np.abs(gpu - ref)
    if (err > tol).any():
        i = int(np.argmax(err))
        raise AssertionError(f"{what}: max |err| {err.max():.4g} > {tol:.4g} at {i} (gpu={gpu[i]}, oracle={ref[i]})")


def assert_topk_exact(gpu_idx: np.ndarray, gpu_count: int, gpu_scores_f32: np.ndarray, k: int, n: int,
                      what: str) -> np.ndarray:
    want = oracle.select_topk(gpu_scores_f32.astype(np.float64), k)
    cnt = min(k, n)
    assert gpu_count == cnt, f"{what}: count {gpu_count} != {cnt}"
    assert np.array_equal(gpu_idx[:cnt], want), f"{what}: selected set differs from the oracle's on the same scores"
    assert (gpu_idx[cnt:] == -1).all(), f"{what}: unused slots not -1"
    return want


def token_slots(pool: dict, b: int, count: int) -> np.ndarray:
    """Physical cache slots of tokens 0..count-1 of sequence b: the slot pool from
    seq_offset[b] on, or the pages of a paged layout."""
    if "page_table" in pool:
        return oracle.paged_slots(pool["page_table"][b], int(pool["page_size"]), count)
    o = int(pool["seq_offset"][b])
    return np.arange(o, o + count)


def check_iteration(w, pool: dict, st, rows0, rows1, check_draft: bool = True,
                    seqs=None) -> dict:
    """Compare one vg_iteration on the GPU with the oracle, sequence by sequence."""
    import torch
    torch.cuda.synchronize()
    out_v = bf16_to_f64(st.out_verify)
    sc0 = st.scores0.cpu().numpy()
    sc1 = st.scores1.cpu().numpy() if st.scores1 is not None else None
    idx = st.idx.cpu().numpy()
    cnt = st.count.cpu().numpy()
    idx1 = st.idx1.cpu().numpy() if st.idx1 is not None else None
    cnt1 = st.count1.cpu().numpy() if st.count1 is not None else None
    out_d = bf16_to_f64(st.out_draft)
    Kc = bf16_to_f64(st.K)
    Vc = bf16_to_f64(st.V)
    stats = {"overlap": []}
    for b in (range(w.B) if seqs is None else seqs):
        n = int(pool["prefix_len"][b])
        sl = token_slots(pool, b, n + w.R)
        K = widen_bf16(pool["K"][sl[:n]])
        V = widen_bf16(pool["V"][sl[:n]])
        q = widen_bf16(pool["q_verify"][b])
        kn, vn = widen_bf16(pool["k_new"][b]), widen_bf16(pool["v_new"][b])
        ref = oracle.verify_attention(q, K, V, kn, vn)
        assert_attn_close(out_v[b], ref, f"verify out seq {b}")
        s0 = oracle.aggregated_scores(q, K, rows0)
        assert_scores_close(sc0[b, :n], s0, f"scores0 seq {b}")
        T = assert_topk_exact(idx[b], int(cnt[b]), sc0[b, :n], st.k, n, f"top-k seq {b}")
        if rows1 is not None:
            s1 = oracle.aggregated_scores(q, K, rows1)
            assert_scores_close(sc1[b, :n], s1, f"scores1 seq {b}")
            if idx1 is not None:
                T1 = assert_topk_exact(idx1[b], int(cnt1[b]), sc1[b, :n], st.k, n, f"top-k(1) seq {b}")
                stats["overlap"].append(oracle.selection_overlap(T, T1, min(st.k, n)) if n else 1.0)
        if check_draft and w.gamma > 0:
            qd = widen_bf16(pool["q_draft"][:, b])
            kd = widen_bf16(pool["k_draft"][:, b])
            vd = widen_bf16(pool["v_draft"][:, b])
            for s in range(w.gamma):
                ref_d = oracle.draft_step(qd[s], K, V, T, kd[:s + 1], vd[:s + 1])
                assert_attn_close(out_d[s, b], ref_d, f"draft step {s} seq {b}")
            # the cache now holds draft tokens at n..n+gamma-1 and verify row gamma at n+gamma
            assert np.array_equal(Kc[sl[n:n + w.gamma]], kd), f"draft K append seq {b}"
            assert np.array_equal(Vc[sl[n:n + w.gamma]], vd), f"draft V append seq {b}"
        assert np.array_equal(Kc[sl[n + w.gamma]], kn[w.gamma]), f"verify K append seq {b}"
        assert np.array_equal(Vc[sl[n + w.gamma]], vn[w.gamma]), f"verify V append seq {b}"
        assert np.array_equal(Kc[sl[:n]], K), f"prefix K modified seq {b}"
    return stats
