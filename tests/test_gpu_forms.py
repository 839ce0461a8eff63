"""GPU parity of the verify call's other forms, and of rows whose weight sits on a few keys.

* The verify call with no score mask (row_mask0 = row_mask1 = 0): full attention
  only, the form the score-emission cost study times.  With no score rows the MMA
  row count can drop (G * (gamma+1) = 64 rows run as M = 64 instead of M = 128).
* The verify call with only the second mask (row_mask0 = 0, row_mask1 != 0): the
  score rows then belong to mask 1.
* Long prefixes (several thousand keys, so the verify kernel carries P as bf16
  alone) where every query row puts almost all of its weight on three keys with
  different values: the case where rounding the attention weights matters most.
  Verification must still be exact attention (Vegas §5, lossless quality), within
  the output tolerance.

Everything goes through the C ABI and is compared with the fp64 oracle.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import synth  # noqa: E402
from synth import Workload, scaled  # noqa: E402
from tests.parity import assert_attn_close, assert_scores_close, bf16_to_f64, check_iteration  # noqa: E402

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from self_speculative_sparse_gb300 import build
    build.build()


FORM_CASES = {
    "tiny": W["tiny"],
    "llama8b_n1000": scaled(W["llama8b"], n=1000),
    "ragged_b6": scaled(W["loop32"], B=6, layers=1, ragged=(1, 1500)),
    # 64 query rows: M = 64 without score rows, M = 128 with them
    "g16_m64": Workload("g16", B=2, Hq=16, Hkv=1, d=128, gamma=3, k=100, n=777, seed=77),
    "g16_m64_d64": Workload("g16d64", B=2, Hq=16, Hkv=1, d=64, gamma=3, k=100, n=777, seed=84),
    "long70b_n2100": scaled(W["long70b"], n=2100),
}


def _verify_call(st, m0, m1, sc0, sc1):
    from self_speculative_sparse_gb300 import binding as vb
    vb.vg_verify_attn(st.dims, st.cache, st.q_verify, st.k_new, st.v_new, st.prefix_len, m0, m1, sc0, sc1,
                      st.score_stride, st.out_verify, st.ws, dev_status=st.status)


def _check_verify(w, pool, st, rows1=None, sc1=None):
    out_v = bf16_to_f64(st.out_verify)
    Kc, Vc = bf16_to_f64(st.K), bf16_to_f64(st.V)
    for b in range(w.B):
        o, n = int(pool["seq_offset"][b]), int(pool["prefix_len"][b])
        K, V = oracle.widen_bf16(pool["K"][o:o + n]), oracle.widen_bf16(pool["V"][o:o + n])
        q = oracle.widen_bf16(pool["q_verify"][b])
        kn, vn = oracle.widen_bf16(pool["k_new"][b]), oracle.widen_bf16(pool["v_new"][b])
        assert_attn_close(out_v[b], oracle.verify_attention(q, K, V, kn, vn), f"verify out seq {b}")
        if rows1 is not None:
            assert_scores_close(sc1[b, :n], oracle.aggregated_scores(q, K, rows1), f"scores1 seq {b}")
        # the verify rows were appended
        assert np.array_equal(Kc[o + n:o + n + w.R], kn) and np.array_equal(Vc[o + n:o + n + w.R], vn), b


@pytest.mark.parametrize("name", list(FORM_CASES))
def test_verify_without_scores_matches_oracle(name):
    from self_speculative_sparse_gb300.runtime import LayerState
    w = FORM_CASES[name]
    pool = w.layer_pool(0)
    st = LayerState(w, pool)
    st.ws.fill_(0xFF)
    sentinel = st.scores0.clone()
    _verify_call(st, 0, 0, None, None)
    torch.cuda.synchronize()
    assert st.check_status() == 0
    _check_verify(w, pool, st)
    assert torch.equal(st.scores0, sentinel)  # no mask: no scores written anywhere


@pytest.mark.parametrize("rows", ["c2", "all"])
@pytest.mark.parametrize("name", list(FORM_CASES))
def test_verify_with_only_the_second_mask_matches_oracle(name, rows):
    from self_speculative_sparse_gb300.runtime import LayerState
    w = FORM_CASES[name]
    pool = w.layer_pool(0)
    st = LayerState(w, pool)
    st.ws.fill_(0x7F)
    sc1 = torch.full_like(st.scores0, 123.0)
    _verify_call(st, 0, w.row_mask(rows), None, sc1)
    torch.cuda.synchronize()
    assert st.check_status() == 0
    sc1h = sc1.cpu().numpy()
    _check_verify(w, pool, st, rows1=w.rows(rows), sc1=sc1h)
    n = pool["prefix_len"]
    for b in range(w.B):  # positions past the prefix are left as they were
        assert (sc1h[b, int(n[b]):] == 123.0).all()


# ------------------------------------------------------------------ peaked long rows
def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bit patterns, round to nearest even (input construction only)."""
    f = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (f + 0x7FFF + ((f >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def peaked_pool(w: Workload, hot_scale=(50.0, 48.5, 47.0), q_shift=8.0, seed=4242) -> dict:
    """The workload's pool with three 'hot' prefix keys per sequence, c_i * u for a
    seeded unit direction u, and every query (verify and draft) shifted by q_shift * u.
    Each hot key's logit is then about c_i * q_shift / sqrt(d) (35 for the defaults at d = 128)
    above the others', so every query row puts almost all of its weight on the three
    hot keys, whose values differ."""
    pool = w.layer_pool(0)
    rng = np.random.default_rng(seed)
    n = pool["prefix_len"]
    off = pool["seq_offset"]
    K = pool["K"].copy()
    qv = oracle.widen_bf16(pool["q_verify"])
    qd = oracle.widen_bf16(pool["q_draft"])
    for b in range(w.B):
        u = rng.standard_normal(w.d)
        u /= np.linalg.norm(u)
        nb = int(n[b])
        hot = rng.choice(np.arange(1, nb - 1), size=len(hot_scale), replace=False)
        for c, p in zip(hot_scale, hot):
            K[int(off[b]) + int(p)] = _to_bf16_bits(np.tile(c * u, (w.Hkv, 1)))
        qv[b] += q_shift * u
        qd[:, b] += q_shift * u
    pool = dict(pool)
    pool["K"] = K
    pool["q_verify"] = _to_bf16_bits(qv)
    pool["q_draft"] = _to_bf16_bits(qd)
    return pool


PEAKED = {
    # several thousand keys per sequence: runs far longer than the kernel's short-run limit
    "llama8b_shape_n4096_6000": Workload("pk8b", B=3, Hq=32, Hkv=8, d=128, gamma=7, k=256, n=None,
                                          ragged=(4096, 6000), seed=91),
    "long70b_shape_n9000": Workload("pk70", B=1, Hq=64, Hkv=8, d=128, gamma=5, k=512, n=9000, seed=92),
    "d64_n5000": Workload("pk64", B=2, Hq=8, Hkv=2, d=64, gamma=3, k=64, n=5000, seed=93),
}


def _weight_on_hot_keys(w, pool) -> float:
    """Smallest share of a verify row's weight on its three largest keys (oracle, fp64)."""
    worst = 1.0
    for b in range(w.B):
        o, n = int(pool["seq_offset"][b]), int(pool["prefix_len"][b])
        K = oracle.widen_bf16(pool["K"][o:o + n])
        q = oracle.widen_bf16(pool["q_verify"][b])
        L = oracle.verify_logits(q, K)
        p = np.exp(L - L.max(axis=-1, keepdims=True))
        p /= p.sum(axis=-1, keepdims=True)
        worst = min(worst, float(np.sort(p, axis=-1)[..., -3:].sum(axis=-1).min()))
    return worst


@pytest.mark.parametrize("name", list(PEAKED))
def test_long_rows_with_weight_on_three_keys_match_oracle(name):
    from self_speculative_sparse_gb300.runtime import LayerState
    w = PEAKED[name]
    pool = peaked_pool(w)
    assert _weight_on_hot_keys(w, pool) > 0.9  # the input is what the test claims
    st = LayerState(w, pool)
    st.ws.fill_(0xFF)
    st.iteration()
    torch.cuda.synchronize()
    assert st.check_status() == 0
    rows1 = w.rows(w.extra_rows) if w.extra_rows else None
    check_iteration(w, pool, st, w.rows(w.select_rows), rows1)
