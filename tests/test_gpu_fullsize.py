"""Full-size parity: every workload at its full size, through the same C ABI calls
the benchmark times, checked against the oracle.

At these sizes the oracle cannot redo a whole iteration in seconds, so each
sequence is checked on what it can compute one piece at a time:
  - aggregated scores at every prefix position (the oracle's grouped form: one
    n x d product per KV head), both masks;
  - the selection, bit-exact against the oracle's top-k on the GPU's own scores;
  - verify outputs on sampled (row, head) pairs, always including rows 0 and gamma,
    each recomputed over the whole prefix and the causal verify keys;
  - draft outputs on sampled (step, head) pairs, always including the first and
    the last step, recomputed over the selected entries and the draft tail;
  - the cache appends (draft tokens at n..n+gamma-1, verify row gamma at n+gamma),
    bit-exact, and an untouched prefix.
The multi-layer workload runs every layer, one at a time.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import synth  # noqa: E402
from oracle import widen_bf16  # noqa: E402
from tests.parity import assert_attn_close, assert_scores_close, assert_topk_exact, bf16_to_f64  # noqa: E402

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from self_speculative_sparse_gb300 import build
    build.build()


def _row(q, keys, vals, scale):
    o, _, _ = oracle.softmax_attention(q[None, :], keys, vals, scale)
    return o[0]


def check_layer(w, pool, st, layer, rng, rows_v=4, rows_d=4):
    """Compare one full-size vg_iteration of one layer with the oracle (sampled)."""
    torch.cuda.synchronize()
    assert st.check_status() == 0, f"layer {layer}: device status {st.check_status()}"
    scale = 1.0 / np.sqrt(w.d)
    G = w.Hq // w.Hkv
    R = w.gamma + 1
    rows0 = w.rows(w.select_rows)
    rows1 = w.rows(w.extra_rows) if w.extra_rows else None
    out_v = st.out_verify.cpu()
    out_d = st.out_draft.cpu()
    sc0 = st.scores0.cpu().numpy()
    sc1 = st.scores1.cpu().numpy() if st.scores1 is not None else None
    idx = st.idx.cpu().numpy()
    cnt = st.count.cpu().numpy()
    overlaps = []
    for b in range(w.B):
        o, n = int(pool["seq_offset"][b]), int(pool["prefix_len"][b])
        K = widen_bf16(pool["K"][o:o + n])  # all heads: the scores need them
        Vg = {}  # value heads, widened when a sampled row needs them

        def V_of(g):
            if g not in Vg:
                Vg[g] = widen_bf16(pool["V"][o:o + n, g])
            return Vg[g]
        q = widen_bf16(pool["q_verify"][b])
        kn, vn = widen_bf16(pool["k_new"][b]), widen_bf16(pool["v_new"][b])
        what = f"layer {layer} seq {b} (n={n})"
        # scores at every position, and the selection on the GPU's own scores
        s0 = oracle.aggregated_scores_grouped(q, K, rows0)
        assert_scores_close(sc0[b, :n], s0, f"scores0 {what}")
        T = assert_topk_exact(idx[b], int(cnt[b]), sc0[b, :n], st.k, n, f"top-k {what}")
        if rows1 is not None:
            s1 = oracle.aggregated_scores_grouped(q, K, rows1)
            assert_scores_close(sc1[b, :n], s1, f"scores1 {what}")
            overlaps.append(oracle.selection_overlap(T, oracle.select_topk(sc1[b, :n].astype(np.float64), st.k),
                                                     min(st.k, n)))
        # verify outputs on sampled rows (rows 0 and gamma always)
        ts = sorted(set([0, w.gamma] + list(rng.integers(0, R, size=max(0, rows_v - 2)))))
        for t in ts:
            for h in sorted(set(rng.integers(0, w.Hq, size=2))):
                g = h // G
                keys = np.concatenate([K[:, g], kn[:t + 1, g]])
                vals = np.concatenate([V_of(g), vn[:t + 1, g]])
                ref = _row(q[t, h], keys, vals, scale)
                got = bf16_to_f64(out_v[b, t, h])
                assert_attn_close(got, ref, f"verify out {what} row {t} head {h}")
        # draft outputs on sampled steps (first and last always)
        if w.gamma > 0:
            qd = widen_bf16(pool["q_draft"][:, b])
            kd = widen_bf16(pool["k_draft"][:, b])
            vd = widen_bf16(pool["v_draft"][:, b])
            ss = sorted(set([0, w.gamma - 1] + list(rng.integers(0, w.gamma, size=max(0, rows_d - 2)))))
            for s in ss:
                for h in sorted(set(rng.integers(0, w.Hq, size=2))):
                    g = h // G
                    keys = np.concatenate([K[T, g], kd[:s + 1, g]])
                    vals = np.concatenate([V_of(g)[T], vd[:s + 1, g]])
                    ref = _row(qd[s, h], keys, vals, scale)
                    got = bf16_to_f64(out_d[s, b, h])
                    assert_attn_close(got, ref, f"draft step {s} {what} head {h}")
        # the appended slots, and sampled prefix slots, bit for bit
        Kt = st.K[o + n:o + n + R].view(torch.int16).cpu().numpy().view(np.uint16)
        Vt = st.V[o + n:o + n + R].view(torch.int16).cpu().numpy().view(np.uint16)
        if w.gamma > 0:
            assert np.array_equal(Kt[:w.gamma], pool["k_draft"][:, b]), f"draft K append {what}"
            assert np.array_equal(Vt[:w.gamma], pool["v_draft"][:, b]), f"draft V append {what}"
        assert np.array_equal(Kt[w.gamma], pool["k_new"][b, w.gamma]), f"verify K append {what}"
        assert np.array_equal(Vt[w.gamma], pool["v_new"][b, w.gamma]), f"verify V append {what}"
        slots = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, size=62)])) + o
        sel = torch.from_numpy(slots).to(st.K.device)
        Kp = st.K.index_select(0, sel).view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(Kp, pool["K"][slots]), f"prefix K modified {what}"
    return overlaps


@pytest.mark.parametrize("name", ["llama8b", "long70b", "batched"])
def test_full_size_workload_matches_oracle_on_samples(name):
    from self_speculative_sparse_gb300.runtime import LayerState
    w = W[name]
    pool = w.layer_pool(0)
    st = LayerState(w, pool)
    st.ws.fill_(0x7F)  # garbage workspace
    st.iteration()
    overlaps = check_layer(w, pool, st, 0, np.random.default_rng(7))
    if w.extra_rows:  # both selections came out of the same pass
        assert len(overlaps) == w.B and all(0.0 <= x <= 1.0 for x in overlaps)


def test_full_size_multilayer_loop_matches_oracle_on_samples():
    """32 layers, B=8 ragged prefixes in [4096, 65536]: every layer's iteration."""
    from self_speculative_sparse_gb300.runtime import LayerState
    w = W["loop32"]
    rng = np.random.default_rng(11)
    lengths = w.lengths(0)
    assert lengths.min() >= 4096 and lengths.max() <= 65536 and len(set(lengths.tolist())) > 1
    for layer in range(w.layers):
        pool = w.layer_pool(layer)
        assert np.array_equal(pool["prefix_len"], lengths)  # the ragged lengths are fixed across layers
        st = LayerState(w, pool)
        st.iteration()
        check_layer(w, pool, st, layer, rng, rows_v=2, rows_d=2)
        del st


@pytest.mark.parametrize("name,layer,reps", [("loop32", 6, 40), ("batched", 0, 40)])
def test_full_size_repeats_are_bit_identical(name, layer, reps):
    """The same call on the same inputs gives the same bits, every time.

    Every CTA of the verify kernel runs some 200+ tiles here, with warps whose lanes
    hold no rows in use beside the ones that do: a missing wait between them shows up
    as one lane quadrant's partial differing from run to run.  The whole iteration
    (verify, both selections, the draft steps) is repeated as well."""
    from self_speculative_sparse_gb300.runtime import LayerState
    w = W[name]
    st = LayerState(w, w.layer_pool(layer))
    ref = None
    for r in range(reps):
        st.verify()
        torch.cuda.synchronize()
        assert st.check_status() == 0
        cur = (st.out_verify.view(torch.int16).clone(), st.scores0.clone())
        if ref is None:
            ref = cur
        else:
            assert torch.equal(cur[0], ref[0]), f"verify output differs on repeat {r}"
            assert torch.equal(cur[1], ref[1]), f"scores differ on repeat {r}"
    st.iteration()
    torch.cuda.synchronize()
    iref = (st.out_verify.view(torch.int16).clone(), st.idx.clone(), st.out_draft.view(torch.int16).clone())
    assert torch.equal(iref[0], ref[0])
    for r in range(reps // 4):
        st.iteration()
        torch.cuda.synchronize()
        assert st.check_status() == 0
        assert torch.equal(st.out_verify.view(torch.int16), iref[0]), f"iteration {r}: verify output differs"
        assert torch.equal(st.idx, iref[1]), f"iteration {r}: selection differs"
        assert torch.equal(st.out_draft.view(torch.int16), iref[2]), f"iteration {r}: draft output differs"
