"""GPU parity of the acceptance step (vg_accept) against the fp64 oracle.

Vegas §2 step 1 (verification accepts or rejects the drafts) and §5 (lossless).  The
decisions are integers that floating point decides: the kernel works in fp32, the oracle
in fp64.  The test inputs keep every decision clear of its boundary (each acceptance
uniform at least 1e-4 away, relatively, from p/q; the draw's target at least 1e-4 of the
total away from any running-sum boundary), so both must take the same decisions; the
counts, tokens and prefix-length updates are then compared exactly.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import synth  # noqa: E402

pytestmark = pytest.mark.gpu

MARGIN = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from self_speculative_sparse_gb300 import build
    build.build()


def _clear_of_boundaries(inp, rng):
    """Move the uniforms away from the decisions' boundaries (input construction)."""
    p, q, x, u, u_res = (inp[k] for k in ("p_logits", "q_logits", "x", "u", "u_res"))
    B, gamma = x.shape
    for b in range(B):
        a = gamma
        for t in range(gamma):
            pt = oracle.softmax(p[b, t])[x[b, t]]
            qt = oracle.softmax(q[b, t])[x[b, t]]
            ratio = pt / qt
            while abs(float(u[b, t]) - ratio) <= MARGIN * max(ratio, 1e-30):
                u[b, t] = np.float32(rng.uniform())
            if not (float(u[b, t]) * qt < pt):
                a = t
                break
        if a < gamma:
            w = np.maximum(0.0, oracle.softmax(p[b, a]) - oracle.softmax(q[b, a]))
        else:
            w = oracle.softmax(p[b, gamma])
        c = np.cumsum(w)
        while True:
            tgt = float(u_res[b]) * c[-1]
            j = np.searchsorted(c, tgt)
            near = min(abs(c[min(j, len(c) - 1)] - tgt), abs(c[max(j - 1, 0)] - tgt))
            if near > MARGIN * c[-1]:
                break
            u_res[b] = np.float32(rng.uniform())
    return inp


def _run(inp, mode, advance=None):
    from self_speculative_sparse_gb300 import binding as vb
    p = torch.from_numpy(inp["p_logits"]).cuda()
    q = torch.from_numpy(inp["q_logits"]).cuda()
    x = torch.from_numpy(inp["x"]).cuda()
    u = torch.from_numpy(inp["u"]).cuda()
    ur = torch.from_numpy(inp["u_res"]).cuda()
    B, gamma = inp["x"].shape
    V = inp["p_logits"].shape[-1]
    na = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    nt = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    adv = None if advance is None else torch.from_numpy(np.asarray(advance, dtype=np.int32)).cuda()
    ws = torch.empty(vb.vg_accept_workspace_size(B, gamma, V), dtype=torch.uint8, device="cuda").fill_(0xFF)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sample = mode == "sample"
    vb.vg_accept(B, gamma, V, p, q if sample else None, x, u if sample else None, ur if sample else None,
                 vb.VG_ACCEPT_SAMPLE if sample else vb.VG_ACCEPT_GREEDY, na, nt, adv, ws, dev_status=status)
    torch.cuda.synchronize()
    return (na.cpu().numpy(), nt.cpu().numpy(), None if adv is None else adv.cpu().numpy(),
            int(status.item()))


CASES = [  # (B, gamma, V, seed)
    (4, 3, 1000, 1),
    (8, 6, 32000, 2),
    (3, 0, 5000, 3),          # no drafts: only the next token
    (5, 7, 4099, 4),          # V not a multiple of 4 (scalar loads)
    (8, 6, 151936, 5),        # a Qwen3-sized vocabulary at the full-iteration batch
]


@pytest.mark.parametrize("B,gamma,V,seed", CASES)
def test_sampling_matches_oracle(B, gamma, V, seed):
    rng = np.random.default_rng(1000 + seed)
    inp = _clear_of_boundaries(synth.accept_inputs(B, gamma, V, seed), rng)
    n0 = np.arange(B, dtype=np.int32) * 100 + 50
    na, nt, adv, st = _run(inp, "sample", advance=n0)
    assert st == 0
    for b in range(B):
        a, nxt = oracle.accept_sample(inp["p_logits"][b].astype(np.float64), inp["q_logits"][b].astype(np.float64),
                                      inp["x"][b], inp["u"][b].astype(np.float64), float(inp["u_res"][b]))
        assert (int(na[b]), int(nt[b])) == (a, nxt), b
        assert int(adv[b]) == oracle.next_prefix_len(int(n0[b]), a)


@pytest.mark.parametrize("B,gamma,V,seed", CASES)
def test_greedy_matches_oracle(B, gamma, V, seed):
    inp = synth.accept_inputs(B, gamma, V, seed)
    # drafts that agree with the target's most likely token for a chosen number of steps
    r = np.random.default_rng(seed)
    for b in range(B):
        keep = int(r.integers(0, gamma + 1)) if gamma else 0
        for t in range(gamma):
            best = oracle.argmax_lowest(inp["p_logits"][b, t])
            inp["x"][b, t] = best if t < keep else (best + 1 + int(r.integers(0, V - 1))) % V
    na, nt, _, st = _run(inp, "greedy")
    assert st == 0
    for b in range(B):
        assert (int(na[b]), int(nt[b])) == oracle.accept_greedy(inp["p_logits"][b], inp["x"][b]), b


def test_equal_distributions_accept_every_draft():
    inp = synth.accept_inputs(4, 5, 2000, 9)
    inp["q_logits"][:] = inp["p_logits"][:, :5]
    inp["u"][:] = np.float32(0.999)
    inp = _clear_of_boundaries(inp, np.random.default_rng(5))
    na, nt, _, st = _run(inp, "sample")
    assert st == 0 and (na == 5).all()
    for b in range(4):
        assert int(nt[b]) == oracle.sample_inverse_cdf(oracle.softmax(inp["p_logits"][b, 5].astype(np.float64)),
                                                       float(inp["u_res"][b]))


def test_a_draft_token_outside_the_vocabulary_is_rejected_and_reported():
    from self_speculative_sparse_gb300 import binding as vb
    inp = synth.accept_inputs(2, 3, 1000, 11)
    inp["x"][1, 0] = 1000  # == V
    na, nt, _, st = _run(inp, "greedy")
    assert st == vb.VG_ERR_DEVICE_BOUNDS
    assert int(na[1]) == 0 and int(nt[1]) == oracle.argmax_lowest(inp["p_logits"][1, 0])
