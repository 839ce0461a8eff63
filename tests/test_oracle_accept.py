"""Pins of the oracle's acceptance step (Vegas §2 step 1, verification accepts or
rejects the draft tokens; Vegas §5, lossless: the output follows the target model).

The acceptance rule is the standard one of speculative decoding; the pins check the
oracle against hand-worked cases and, above all, against the property the page claims
for it: whatever the draft distribution, the first committed token is distributed as the
target's.  The planted mistakes at the end must each break a pin.
"""
import types

import numpy as np
import pytest

import oracle
from oracle import vegas as ov


def test_inverse_cdf_hand_cases():
    w = np.array([1.0, 0.0, 3.0])  # cumulative 1, 1, 4 (total 4)
    assert oracle.sample_inverse_cdf(w, 0.0) == 0
    assert oracle.sample_inverse_cdf(w, 0.1) == 0     # 0.4 < 1
    assert oracle.sample_inverse_cdf(w, 0.2499) == 0
    assert oracle.sample_inverse_cdf(w, 0.25) == 2    # 1.0 is not > 1: the zero-weight token is skipped
    assert oracle.sample_inverse_cdf(w, 0.9) == 2
    assert oracle.sample_inverse_cdf(np.array([0.0, 0.0, 2.0, 2.0]), 0.5) == 3


def test_argmax_ties_go_to_the_lowest_position():
    assert oracle.argmax_lowest(np.array([1.0, 3.0, 3.0, 2.0])) == 1
    assert oracle.argmax_lowest(np.array([-1.0, -1.0])) == 0


def test_greedy_hand_case():
    V = 10
    p = np.zeros((4, V))
    for t, best in enumerate([5, 2, 7, 1]):
        p[t, best] = 3.0
    assert oracle.accept_greedy(p, np.array([5, 2, 9])) == (2, 7)   # third draft differs: next = argmax row 2
    assert oracle.accept_greedy(p, np.array([5, 2, 7])) == (3, 1)   # all accepted: the bonus row
    assert oracle.accept_greedy(p, np.array([4, 2, 7])) == (0, 5)


def test_sampling_with_equal_distributions_accepts_everything():
    r = np.random.default_rng(1)
    p = r.normal(size=(4, 7))
    u = np.array([0.999, 0.5, 0.0])
    a, nxt = oracle.accept_sample(p, p[:3], np.array([1, 2, 3]), u, 0.3)
    assert a == 3
    assert nxt == oracle.sample_inverse_cdf(oracle.softmax(p[3]), 0.3)


def test_sampling_accepts_with_probability_p_over_q():
    # the draft is sure of its token (q(x) ~ 1); the target gives it 0.3
    V = 4
    p = np.log(np.array([[0.3, 0.2, 0.25, 0.25], [0.25, 0.25, 0.25, 0.25]]))
    q = np.array([[40.0, 0.0, 0.0, 0.0]])
    assert oracle.accept_sample(p, q, np.array([0]), np.array([0.29]), 0.5)[0] == 1
    a, nxt = oracle.accept_sample(p, q, np.array([0]), np.array([0.31]), 0.5)
    assert a == 0
    # the excess max(0, p - q) is (0, 0.2, 0.25, 0.25): u_res 0.5 lands on token 2
    assert nxt == 2


def test_next_prefix_length():
    assert oracle.next_prefix_len(100, 0) == 101
    assert oracle.next_prefix_len(100, 6) == 107


def _first_token_distribution(mod, p_logits, q_logits, n_accept=20000, n_resample=2000):
    """Distribution of the first committed token under the oracle's rule: the draft token
    integrated over q_0, the acceptance uniform over a stratified grid, and, for a
    rejection, the resampling uniform over another (deterministic, no random draws)."""
    V = p_logits.shape[1]
    gamma = q_logits.shape[0]
    q0 = mod.softmax(q_logits[0])
    ua_grid = (np.arange(n_accept) + 0.5) / n_accept
    ur_grid = (np.arange(n_resample) + 0.5) / n_resample
    dist = np.zeros(V)
    for x0 in range(V):
        x = np.full(gamma, x0)
        acc = np.mean([mod.accept_sample(p_logits, q_logits, x, np.full(gamma, ua), 0.0)[0] >= 1 for ua in ua_grid])
        dist[x0] += q0[x0] * acc
        if acc < 1.0:  # a rejected draft: the resampled token, over the resampling uniform
            u_rej = np.full(gamma, ua_grid[-1])
            for ur in ur_grid:
                a, nxt = mod.accept_sample(p_logits, q_logits, x, u_rej, ur)
                assert a == 0
                dist[nxt] += q0[x0] * (1.0 - acc) / n_resample
    return dist


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_speculative_sampling_is_lossless(seed):
    """Vegas §5: the first committed token follows the target's distribution p_0, for
    any draft distribution q_0."""
    r = np.random.default_rng(100 + seed)
    V = 5
    p = r.normal(scale=1.5, size=(2, V))
    q = r.normal(scale=1.5, size=(1, V))
    dist = _first_token_distribution(ov, p, q)
    np.testing.assert_allclose(dist, oracle.softmax(p[0]), atol=2e-3)


# ------------------------------------------------------------ planted mistakes
def _mutant(name):
    m = types.ModuleType("mutant")
    m.__dict__.update({k: getattr(ov, k) for k in dir(ov) if not k.startswith("__")})
    for k, f in list(m.__dict__.items()):
        if isinstance(f, types.FunctionType) and f.__module__ == ov.__name__:
            setattr(m, k, types.FunctionType(f.__code__, m.__dict__, k, f.__defaults__))
    if name == "ratio inverted":
        def accept_sample(p_logits, q_logits, x, u, u_res):
            gamma = len(x)
            for t in range(gamma):
                p, q = ov.softmax(p_logits[t]), ov.softmax(q_logits[t])
                if not (u[t] * p[int(x[t])] < q[int(x[t])]):
                    return t, ov.sample_inverse_cdf(np.maximum(0.0, p - q) + 1e-300, u_res)
            return gamma, ov.sample_inverse_cdf(ov.softmax(p_logits[gamma]), u_res)
        m.accept_sample = accept_sample
    elif name == "resample from p":
        def accept_sample(p_logits, q_logits, x, u, u_res):
            gamma = len(x)
            for t in range(gamma):
                p, q = ov.softmax(p_logits[t]), ov.softmax(q_logits[t])
                if not (u[t] * q[int(x[t])] < p[int(x[t])]):
                    return t, ov.sample_inverse_cdf(p, u_res)
            return gamma, ov.sample_inverse_cdf(ov.softmax(p_logits[gamma]), u_res)
        m.accept_sample = accept_sample
    elif name == "inverse CDF takes zero-weight tokens":
        def sample_inverse_cdf(w, u):
            c = np.cumsum(np.asarray(w, dtype=np.float64))
            return int(np.searchsorted(c, u * c[-1], side="left"))
        m.sample_inverse_cdf = sample_inverse_cdf
    elif name == "argmax ties to the highest":
        def argmax_lowest(v):
            v = np.asarray(v)
            return int(np.flatnonzero(v == v.max())[-1])
        m.argmax_lowest = argmax_lowest
    elif name == "frontier without the verified row":
        m.next_prefix_len = lambda n, a: n + a
    return m


def _pins_fail(mod) -> bool:
    try:
        w = np.array([1.0, 0.0, 3.0])
        if mod.sample_inverse_cdf(w, 0.25) != 2:
            return True
        if mod.argmax_lowest(np.array([1.0, 3.0, 3.0, 2.0])) != 1:
            return True
        if mod.next_prefix_len(100, 6) != 107:
            return True
        r = np.random.default_rng(100)
        p = r.normal(scale=1.5, size=(2, 5))
        q = r.normal(scale=1.5, size=(1, 5))
        return not np.allclose(_first_token_distribution(mod, p, q), mod.softmax(p[0]), atol=2e-3)
    except Exception:
        return True


def test_unmutated_accept_oracle_passes():
    assert not _pins_fail(ov)


@pytest.mark.parametrize("name", ["ratio inverted", "resample from p", "inverse CDF takes zero-weight tokens",
                                  "argmax ties to the highest", "frontier without the verified row"])
def test_planted_accept_mistake_is_caught(name):
    assert _pins_fail(_mutant(name)), name
