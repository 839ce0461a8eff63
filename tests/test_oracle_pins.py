"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each pin checks the oracle against something the Vegas page or plain mathematics
fixes: a hand-worked example of the selection objective (Vegas §2.A), exhaustive
search over all subsets for the argmax, a library attention routine (PyTorch's
scaled_dot_product_attention in float64) on a special case, closed forms of
softmax attention, an algebraic identity of the aggregated logits, and symmetries
(GQA head repetition, permutation of the prefix, k = n sparse equals dense).

The mutation tests at the end plant plausible mistakes *in the oracle* (on the CPU)
and check that at least one pin catches each.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import vegas as ov

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(20260202)


def _rand(*shape):
    return rng.standard_normal(shape)


# ------------------------------------------------------------ worked example
def test_hand_worked_example_scores_and_selection():
    with open(os.path.join(GOLDEN, "hand_worked_example.json")) as f:
        ex = json.load(f)
    K = np.array(ex["K_prefix"], dtype=np.float64)
    q = np.array(ex["q_verify"], dtype=np.float64)
    s_all = oracle.aggregated_scores(q, K, [0, 1], ex["scale"])
    s_r0 = oracle.aggregated_scores(q, K, [0], ex["scale"])
    assert s_all.tolist() == ex["scores_all_rows"]
    assert s_r0.tolist() == ex["scores_row0"]
    # scale omitted -> 1/sqrt(d) = 1/2 for d = 4
    assert oracle.aggregated_scores(q, K, [0, 1]).tolist() == ex["scores_all_rows"]
    for k, want in ex["topk_all_rows"].items():
        assert oracle.select_topk(s_all, int(k)).tolist() == want
    for k, want in ex["topk_row0"].items():
        assert oracle.select_topk(s_r0, int(k)).tolist() == want


def test_hand_worked_example_verify_closed_form():
    with open(os.path.join(GOLDEN, "hand_worked_example.json")) as f:
        ex = json.load(f)
    cf = ex["verify_closed_form"]
    K = np.array(ex["K_prefix"], dtype=np.float64)
    V = np.array(cf["V_prefix"], dtype=np.float64)
    q = np.array(ex["q_verify"], dtype=np.float64)
    kn = np.array(cf["k_new"], dtype=np.float64)
    vn = np.array(cf["v_new"], dtype=np.float64)
    O = oracle.verify_attention(q, K, V, kn, vn, ex["scale"])
    e = math.e
    want = np.array([2.0, 2.0, 2.0, 1.0 + e]) / (4.0 + e)
    np.testing.assert_allclose(O[cf["row"], cf["head"]], want, rtol=0, atol=1e-15)


# ------------------------------------------------------------ argmax by brute force
def _brute_force_best(s, k):
    n = len(s)
    m = min(k, n)
    best, best_set = None, None
    for c in itertools.combinations(range(n), m):       # lexicographic order
        tot = sum(s[i] for i in c)
        if best is None or tot > best:
            best, best_set = tot, c
    return list(best_set)


@pytest.mark.parametrize("trial", range(60))
def test_topk_is_the_lexicographically_first_maximiser(trial):
    n = int(rng.integers(1, 13))
    k = int(rng.integers(0, 5))
    # few distinct integer values -> many exact ties; sums stay exact
    s = rng.integers(-3, 4, size=n).astype(np.float64)
    if trial % 3 == 0:
        s[s == 0] = -0.0                                  # -0.0 must tie with +0.0
        s[::2] = np.where(s[::2] == -0.0, 0.0, s[::2])
    got = oracle.select_topk(s, k).tolist()
    assert got == _brute_force_best(list(s + 0.0), k)
    assert got == sorted(got) and len(got) == min(k, n)


def test_topk_k_at_least_n_selects_everything():
    s = _rand(7)
    assert oracle.select_topk(s, 7).tolist() == list(range(7))
    assert oracle.select_topk(s, 100).tolist() == list(range(7))
    assert oracle.select_topk(s, 0).tolist() == []
    assert oracle.select_topk(np.zeros(0), 3).tolist() == []


# ------------------------------------------------------------ library special case
def _sdpa_verify(q, K, V, kn, vn, scale):
    torch = pytest.importorskip("torch")
    R, Hq, d = q.shape
    n, Hkv, _ = K.shape
    G = Hq // Hkv
    keys = np.concatenate([K, kn], axis=0)               # [n+R][Hkv][d]
    vals = np.concatenate([V, vn], axis=0)
    Q = torch.tensor(q).permute(1, 0, 2)                 # [Hq][R][d]
    Kt = torch.tensor(keys).permute(1, 0, 2).repeat_interleave(G, dim=0)
    Vt = torch.tensor(vals).permute(1, 0, 2).repeat_interleave(G, dim=0)
    mask = torch.zeros(R, n + R, dtype=torch.bool)
    mask[:, :n] = True
    for t in range(R):
        mask[t, n:n + t + 1] = True
    o = torch.nn.functional.scaled_dot_product_attention(Q, Kt, Vt, attn_mask=mask, scale=scale)
    return o.permute(1, 0, 2).numpy()


@pytest.mark.parametrize("R,Hq,Hkv,d,n", [(4, 8, 2, 16, 9), (1, 4, 4, 8, 3), (3, 6, 1, 8, 0), (8, 8, 2, 32, 33)])
def test_verify_matches_library_sdpa_fp64(R, Hq, Hkv, d, n):
    q, K, V = _rand(R, Hq, d), _rand(n, Hkv, d), _rand(n, Hkv, d)
    kn, vn = _rand(R, Hkv, d), _rand(R, Hkv, d)
    scale = 1.0 / math.sqrt(d)
    got = oracle.verify_attention(q, K, V, kn, vn)
    want = _sdpa_verify(q, K, V, kn, vn, scale)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_draft_matches_library_sdpa_fp64():
    torch = pytest.importorskip("torch")
    Hq, Hkv, d, m = 8, 2, 16, 11
    q, Ks, Vs = _rand(Hq, d), _rand(m, Hkv, d), _rand(m, Hkv, d)
    got = oracle.sparse_draft_attention(q, Ks, Vs)
    G = Hq // Hkv
    Q = torch.tensor(q)[:, None, :]
    Kt = torch.tensor(Ks).permute(1, 0, 2).repeat_interleave(G, dim=0)
    Vt = torch.tensor(Vs).permute(1, 0, 2).repeat_interleave(G, dim=0)
    want = torch.nn.functional.scaled_dot_product_attention(Q, Kt, Vt)[:, 0, :].numpy()
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


# ------------------------------------------------------------ closed forms
def test_identical_keys_give_the_mean_value():
    R, Hq, Hkv, d, n = 4, 4, 2, 8, 6
    k = _rand(d)
    K = np.broadcast_to(k, (n, Hkv, d)).copy()
    kn = np.broadcast_to(k, (R, Hkv, d)).copy()
    V, vn, q = _rand(n, Hkv, d), _rand(R, Hkv, d), _rand(R, Hq, d)
    O = oracle.verify_attention(q, K, V, kn, vn)
    for t in range(R):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            want = np.concatenate([V[:, g], vn[:t + 1, g]]).mean(axis=0)
            np.testing.assert_allclose(O[t, h], want, atol=1e-13)


def test_dominant_key_returns_its_value():
    Hq, Hkv, d, m = 4, 1, 8, 9
    q = np.zeros((Hq, d))
    q[:, 0] = 1.0
    Ks = np.zeros((m, Hkv, d))
    Ks[5, 0, 0] = 1e3 * math.sqrt(d)                      # logit +1e3 against 0
    Vs = _rand(m, Hkv, d)
    O = oracle.sparse_draft_attention(q, Ks, Vs)
    for h in range(Hq):
        np.testing.assert_allclose(O[h], Vs[5, 0], atol=1e-14)


def test_single_entry_returns_exactly_that_value():
    Hq, Hkv, d = 4, 2, 8
    q = _rand(Hq, d)
    Ks, Vs = _rand(1, Hkv, d), _rand(1, Hkv, d)
    O = oracle.sparse_draft_attention(q, Ks, Vs)
    for h in range(Hq):
        assert np.array_equal(O[h], Vs[0, h // 2])
    # verify with an empty prefix: row 0 attends only its own new key
    R = 3
    qv, kn, vn = _rand(R, Hq, d), _rand(R, Hkv, d), _rand(R, Hkv, d)
    Ov = oracle.verify_attention(qv, np.zeros((0, Hkv, d)), np.zeros((0, Hkv, d)), kn, vn)
    for h in range(Hq):
        assert np.array_equal(Ov[0, h], vn[0, h // 2])


def test_softmax_rows_sum_to_one():
    q, K, V = _rand(5, 16), _rand(40, 16), _rand(40, 16)
    allowed = rng.random((5, 40)) < 0.6
    allowed[:, 0] = True
    _, p, _ = oracle.softmax_attention(q * 7.0, K, V, 0.25, allowed)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(p[~allowed] == 0.0) and np.all(p >= 0.0)


# ------------------------------------------------------------ identities and symmetries
def _linearity_scores(q, K, rows, scale):
    """s_i = scale * Σ_g K[i,g,:] . Qsum_g, Qsum_g = Σ_{t in rows} Σ_{h in group g} q[t,h,:]."""
    R, Hq, d = q.shape
    n, Hkv, _ = K.shape
    G = Hq // Hkv
    s = np.zeros(n)
    for g in range(Hkv):
        qsum = np.zeros(d)
        for t in rows:
            for j in range(G):
                qsum += q[t, g * G + j]
        s += K[:, g, :] @ qsum
    return s * scale


@pytest.mark.parametrize("rows", [[0, 3], [0, 1, 2, 3], [2]])
def test_scores_linearity_identity(rows):
    R, Hq, Hkv, d, n = 4, 8, 2, 16, 50
    q, K = _rand(R, Hq, d), _rand(n, Hkv, d)
    a = oracle.aggregated_scores(q, K, rows)
    b = _linearity_scores(q, K, rows, 1.0 / math.sqrt(d))
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12 * np.abs(b).max())
    # the oracle's grouped form (used at full size) is the same identity
    c = oracle.aggregated_scores_grouped(q, K, rows)
    np.testing.assert_allclose(c, a, rtol=1e-12, atol=1e-12 * np.abs(a).max())


def test_collect2_equals_all_rows_when_gamma_is_one():
    q, K = _rand(2, 8, 16), _rand(30, 2, 16)
    assert np.array_equal(oracle.aggregated_scores(q, K, [0, 1]), oracle.aggregated_scores(q, K, range(2)))


def test_gqa_equals_repeated_kv_heads():
    R, Hq, Hkv, d, n = 3, 8, 2, 16, 20
    q, K, V = _rand(R, Hq, d), _rand(n, Hkv, d), _rand(n, Hkv, d)
    kn, vn = _rand(R, Hkv, d), _rand(R, Hkv, d)
    G = Hq // Hkv
    rep = lambda x: np.repeat(x, G, axis=1)               # noqa: E731  KV head g -> heads gG..gG+G-1
    O1 = oracle.verify_attention(q, K, V, kn, vn)
    O2 = oracle.verify_attention(q, rep(K), rep(V), rep(kn), rep(vn))
    np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-14)
    s1 = oracle.aggregated_scores(q, K, [0, 2])
    s2 = oracle.aggregated_scores(q, rep(K), [0, 2])
    np.testing.assert_allclose(s1, s2, rtol=1e-14, atol=1e-13)


def test_prefix_permutation_invariance():
    R, Hq, Hkv, d, n = 4, 8, 2, 16, 25
    q, K, V = _rand(R, Hq, d), _rand(n, Hkv, d), _rand(n, Hkv, d)
    kn, vn = _rand(R, Hkv, d), _rand(R, Hkv, d)
    perm = rng.permutation(n)
    O1 = oracle.verify_attention(q, K, V, kn, vn)
    O2 = oracle.verify_attention(q, K[perm], V[perm], kn, vn)
    np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-13)
    s1 = oracle.aggregated_scores(q, K, [0, 3])
    s2 = oracle.aggregated_scores(q, K[perm], [0, 3])
    np.testing.assert_allclose(s2, s1[perm], rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("t", [0, 2, 4])
def test_sparse_with_full_selection_equals_dense_verify(t):
    R, Hq, Hkv, d, n = 5, 8, 2, 16, 30
    q, K, V = _rand(R, Hq, d), _rand(n, Hkv, d), _rand(n, Hkv, d)
    kn, vn = _rand(R, Hkv, d), _rand(R, Hkv, d)
    dense = oracle.verify_attention(q, K, V, kn, vn)[t]
    sparse = oracle.draft_step(q[t], K, V, np.arange(n), kn[:t + 1], vn[:t + 1])
    np.testing.assert_allclose(sparse, dense, rtol=0, atol=1e-13)


def test_selection_maximises_the_objective_on_random_scores():
    q, K = _rand(4, 8, 16), _rand(14, 2, 16)
    s = oracle.aggregated_scores(q, K, [0, 3])
    T = oracle.select_topk(s, 3)
    best = max(sum(s[list(c)]) for c in itertools.combinations(range(14), 3))
    assert abs(s[T].sum() - best) <= 1e-12 * abs(best)


def test_iteration_composes_the_steps():
    R, Hq, Hkv, d, n, gamma, k = 4, 8, 2, 16, 40, 3, 7
    q, K, V = _rand(R, Hq, d), _rand(n, Hkv, d), _rand(n, Hkv, d)
    kn, vn = _rand(R, Hkv, d), _rand(R, Hkv, d)
    qd, kd, vd = _rand(gamma, Hq, d), _rand(gamma, Hkv, d), _rand(gamma, Hkv, d)
    it = oracle.iteration(q, K, V, kn, vn, qd, kd, vd, k, [0, gamma], list(range(R)))
    T = oracle.select_topk(oracle.aggregated_scores(q, K, [0, gamma]), k)
    assert it["idx"].tolist() == T.tolist()
    for s in range(gamma):
        Ks = np.concatenate([K[T], kd[:s + 1]])
        Vs = np.concatenate([V[T], vd[:s + 1]])
        np.testing.assert_array_equal(it["out_draft"][s], oracle.sparse_draft_attention(qd[s], Ks, Vs))


def test_widen_bf16_exact():
    bits = np.array([0x3F80, 0xBF80, 0x0000, 0x8000, 0x4049, 0x7F7F], dtype=np.uint16)
    got = oracle.widen_bf16(bits)
    assert got[0] == 1.0 and got[1] == -1.0 and got[2] == 0.0 and got[3] == 0.0
    assert got[4] == 3.140625
    assert got[5] == float(np.float32(3.3895313892515355e38))


# ------------------------------------------------------------ selection overlap
# Vegas §2.B (Collect-2-Query, observation): the entries selected from different
# rows of the draft chain largely coincide.  The overlap of two size-k selections is
# the fraction of one selection that the other also holds, |A ∩ B| / k.
def test_overlap_hand_computed_cases():
    a = np.array([0, 2, 4, 6])
    b = np.array([2, 3, 4, 5])
    assert oracle.selection_overlap(a, b, 4) == 0.5                       # {2, 4} of 4
    assert oracle.selection_overlap(a, a, 4) == 1.0
    assert oracle.selection_overlap(a, np.array([1, 3, 5, 7]), 4) == 0.0  # disjoint
    assert oracle.selection_overlap(np.array([9]), np.array([9]), 1) == 1.0
    assert oracle.selection_overlap(np.array([], dtype=np.int64), np.array([], dtype=np.int64), 0) == 1.0


def test_overlap_against_set_intersection_and_symmetry():
    r = np.random.default_rng(17)
    for _ in range(200):
        n = int(r.integers(1, 40))
        k = int(r.integers(1, n + 1))
        a = np.sort(r.choice(n, size=k, replace=False))
        b = np.sort(r.choice(n, size=k, replace=False))
        want = len(set(a.tolist()) & set(b.tolist())) / k
        assert oracle.selection_overlap(a, b, k) == want
        assert oracle.selection_overlap(b, a, k) == want


def test_overlap_of_selections_with_k_at_least_n_is_one():
    # both masks select every prefix entry when k >= n, whatever their scores
    q, K = _rand(4, 8, 16), _rand(9, 2, 16)
    ta = oracle.select_topk(oracle.aggregated_scores(q, K, [0, 3]), 20)
    tb = oracle.select_topk(oracle.aggregated_scores(q, K, [0, 1, 2, 3]), 20)
    assert oracle.selection_overlap(ta, tb, min(20, 9)) == 1.0


# ------------------------------------------------------------ sliding window
# Vegas §1 (problem statement): the query-agnostic comparison policy, a sliding window
# of the most recent entries.
def test_window_hand_cases():
    assert oracle.select_window(10, 3).tolist() == [7, 8, 9]
    assert oracle.select_window(2, 5).tolist() == [0, 1]
    assert oracle.select_window(0, 4).tolist() == []
    assert oracle.select_window(6, 6).tolist() == [0, 1, 2, 3, 4, 5]


def test_window_is_the_topk_of_a_recency_score():
    # with scores that grow with the position, the score-based selection (the argmax of
    # Vegas §2.A, checked by exhaustive search above) picks exactly the window
    r = np.random.default_rng(23)
    for _ in range(50):
        n, k = int(r.integers(1, 60)), int(r.integers(1, 70))
        s = np.cumsum(r.uniform(0.01, 1.0, size=n))
        assert oracle.select_topk(s, k).tolist() == oracle.select_window(n, k).tolist()


# ------------------------------------------------------------ paged cache
def test_paged_slots_hand_case():
    # pages of 2 tokens, sequence in pages 3 then 0
    assert oracle.paged_slots(np.array([3, 0]), 2, 4).tolist() == [6, 7, 0, 1]
    assert oracle.paged_slots(np.array([3, 0]), 2, 3).tolist() == [6, 7, 0]


def test_page_size_one_takes_the_table_as_token_slots():
    # Vegas §3: with pages of one token, the page indices are the token slots themselves
    t = np.array([9, 2, 5, 7])
    assert oracle.paged_slots(t, 1, 4).tolist() == t.tolist()


def test_identity_table_is_the_flat_pool():
    for P in (1, 8, 16, 64):
        o = 5 * P
        n = 3 * P + 7
        table = np.arange(o // P, o // P + (n + P - 1) // P)
        assert oracle.paged_slots(table, P, n).tolist() == list(range(o, o + n))


# ------------------------------------------------------------ planted mistakes
def _pin_errors(mod):
    """Discrepancies of the pins above for a (possibly mutated) oracle module."""
    r = np.random.default_rng(5)
    R, Hq, Hkv, d, n = 4, 8, 2, 16, 12
    q, K, V = r.standard_normal((R, Hq, d)), r.standard_normal((n, Hkv, d)), r.standard_normal((n, Hkv, d))
    kn, vn = r.standard_normal((R, Hkv, d)), r.standard_normal((R, Hkv, d))
    errs = {}
    errs["sdpa"] = np.abs(mod.verify_attention(q, K, V, kn, vn) - _sdpa_verify(q, K, V, kn, vn, 0.25)).max()
    s = mod.aggregated_scores(q, K, [0, 3])
    errs["linearity"] = np.abs(s - _linearity_scores(q, K, [0, 3], 0.25)).max()
    with open(os.path.join(GOLDEN, "hand_worked_example.json")) as f:
        ex = json.load(f)
    sa = mod.aggregated_scores(np.array(ex["q_verify"], float), np.array(ex["K_prefix"], float), [0, 1])
    errs["worked"] = np.abs(sa - np.array(ex["scores_all_rows"])).max()
    bad = 0
    for _ in range(30):
        m = int(r.integers(1, 10))
        sc = r.integers(-2, 3, size=m).astype(float)
        kk = int(r.integers(0, 4))
        bad += mod.select_topk(sc, kk).tolist() != _brute_force_best(list(sc), kk)
    errs["brute"] = bad
    dense = mod.verify_attention(q, K, V, kn, vn)[2]
    sparse = mod.draft_step(q[2], K, V, np.arange(n), kn[:3], vn[:3])
    errs["k_eq_n"] = np.abs(dense - sparse).max()
    errs["overlap"] = abs(mod.selection_overlap(np.array([0, 2, 4, 6]), np.array([2, 3, 4, 5]), 4) - 0.5)
    errs["paged"] = int(mod.paged_slots(np.array([3, 0]), 2, 4).tolist() != [6, 7, 0, 1])
    errs["window"] = int(mod.select_window(10, 3).tolist() != [7, 8, 9]) + int(
        mod.select_topk(np.arange(1.0, 13.0), 5).tolist() != mod.select_window(12, 5).tolist())
    return errs


def _caught(errs):
    return (errs["sdpa"] > 1e-9 or errs["linearity"] > 1e-9 or errs["worked"] > 1e-9
            or errs["brute"] > 0 or errs["k_eq_n"] > 1e-9 or errs["overlap"] > 0 or errs["window"] > 0
            or errs["paged"] > 0)


def test_unmutated_oracle_passes_every_pin():
    assert not _caught(_pin_errors(ov))


MUTANTS = {
    "head map h % H_kv": ("verify_logits", "_heads", None),
    "drop the scale in logits": ("verify_logits", None, None),
    "causal mask off by one": ("verify_attention", None, None),
    "ties to the higher index": ("select_topk", None, None),
    "select the smallest": ("select_topk", None, None),
    "scores skip the last row": ("aggregated_scores", None, None),
    "draft drops the current token": ("draft_step", None, None),
    "overlap over the union (Jaccard)": ("selection_overlap", None, None),
    "overlap over the larger total": ("selection_overlap", None, None),
    "window one position early": ("select_window", None, None),
    "window at the start": ("select_window", None, None),
    "page rows transposed": ("paged_slots", None, None),
}


def _mutant(name):
    import types
    m = types.ModuleType("mutant")
    m.__dict__.update({k: getattr(ov, k) for k in dir(ov) if not k.startswith("__")})
    # rebind every oracle function to the mutant's namespace, so that a planted
    # mistake in one helper reaches every function that calls it
    for k, f in list(m.__dict__.items()):
        if isinstance(f, types.FunctionType) and f.__module__ == ov.__name__:
            setattr(m, k, types.FunctionType(f.__code__, m.__dict__, k, f.__defaults__))
    if name == "head map h % H_kv":
        def _heads(Hq, Hkv):
            return Hq // Hkv, [h % Hkv for h in range(Hq)]
        m._heads = _heads
    elif name == "drop the scale in logits":
        def verify_logits(q, K, scale=None):
            return ov.verify_logits(q, K, 1.0)
        m.verify_logits = verify_logits
    elif name == "causal mask off by one":
        def verify_attention(q, K, V, k_new, v_new, scale=None):
            R = q.shape[0]
            kn2 = np.concatenate([k_new[1:], k_new[-1:]])   # row t sees key t+1 instead of t
            vn2 = np.concatenate([v_new[1:], v_new[-1:]])
            return ov.verify_attention(q, K, V, kn2, vn2, scale) if R > 1 else ov.verify_attention(q, K, V, k_new, v_new, scale)
        m.verify_attention = verify_attention
    elif name == "ties to the higher index":
        def select_topk(s, k):
            s = np.asarray(s, float) + 0.0
            n = len(s)
            order = np.lexsort((-np.arange(n), -s))
            return np.sort(order[:min(k, n)])
        m.select_topk = select_topk
    elif name == "select the smallest":
        def select_topk(s, k):
            s = np.asarray(s, float) + 0.0
            n = len(s)
            order = np.lexsort((np.arange(n), s))
            return np.sort(order[:min(k, n)])
        m.select_topk = select_topk
    elif name == "scores skip the last row":
        def aggregated_scores(q, K, rows, scale=None):
            rows = sorted(set(rows))
            return ov.aggregated_scores(q, K, rows[:-1] if len(rows) > 1 else rows, scale)
        m.aggregated_scores = aggregated_scores
    elif name == "draft drops the current token":
        def draft_step(q, K, V, idx, tail_K, tail_V, scale=None):
            return ov.draft_step(q, K, V, idx, tail_K[:-1], tail_V[:-1], scale)
        m.draft_step = draft_step
    elif name == "overlap over the union (Jaccard)":
        def selection_overlap(a, b, k):
            u = np.union1d(a, b)
            return len(np.intersect1d(a, b)) / float(len(u)) if len(u) else 1.0
        m.selection_overlap = selection_overlap
    elif name == "overlap over the larger total":
        def selection_overlap(a, b, k):
            return len(np.intersect1d(a, b)) / float(len(a) + len(b)) if k > 0 else 1.0
        m.selection_overlap = selection_overlap
    elif name == "window one position early":
        def select_window(n, k):
            m_ = min(k, n)
            return np.arange(max(0, n - m_ - 1), max(0, n - 1), dtype=np.int64)
        m.select_window = select_window
    elif name == "window at the start":
        def select_window(n, k):
            return np.arange(0, min(k, n), dtype=np.int64)
        m.select_window = select_window
    elif name == "page rows transposed":
        def paged_slots(table_row, page_size, n):
            i = np.arange(n, dtype=np.int64)
            return np.asarray(table_row, dtype=np.int64)[i % len(table_row)] * page_size + i // len(table_row)
        m.paged_slots = paged_slots
    return m


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistake_is_caught(name):
    assert _caught(_pin_errors(_mutant(name))), name
