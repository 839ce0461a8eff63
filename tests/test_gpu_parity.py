"""GPU parity of the CUDA path (through the C ABI) against the fp64 CPU oracle.

Small cases that the oracle finishes in seconds but that still span several
tiles, ragged tails, empty and one-entry prefixes, every m-tile count of the
verify kernel (G*(gamma+1) = 16, 28, 32, 48, 64), both head dims (both MMA row counts
at each), gamma = 0 and k >= n.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import synth  # noqa: E402
from synth import Workload, scaled  # noqa: E402
from tests.parity import bf16_to_f64, check_iteration, assert_attn_close  # noqa: E402

import oracle  # noqa: E402

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from self_speculative_sparse_gb300 import build
    build.build()


CASES = {
    "tiny": W["tiny"],
    "llama8b_n1000": scaled(W["llama8b"], n=1000),
    "batched_b3_n700": scaled(W["batched"], B=3, n=700),
    "long70b_n2100": scaled(W["long70b"], n=2100),
    "ragged_b6": scaled(W["loop32"], B=6, layers=1, ragged=(1, 1500)),
    "g16_m64": Workload("g16", B=2, Hq=16, Hkv=1, d=128, gamma=3, k=100, n=777, seed=77),
    "g16_m64_d64": Workload("g16d64", B=2, Hq=16, Hkv=1, d=64, gamma=3, k=100, n=777, seed=84),
    "mha_d64_gamma0": Workload("mha", B=2, Hq=4, Hkv=4, d=64, gamma=0, k=33, n=200, seed=78),
    "k_over_n": Workload("kbig", B=2, Hq=8, Hkv=2, d=64, gamma=2, k=300, n=250, seed=79),
    "short_prefix": Workload("short", B=3, Hq=8, Hkv=4, d=128, gamma=5, k=8, n=None, ragged=(0, 70), seed=80),
    # more than 32 sequences: the per-warp loops over sequences take several rounds
    # (narrow combine: few (sequence, KV head) rows; wide: many)
    "many_seqs_narrow": Workload("b40", B=40, Hq=2, Hkv=1, d=64, gamma=3, k=20, n=None, ragged=(1, 200), seed=81),
    "many_seqs_wide": Workload("b48", B=48, Hq=32, Hkv=8, d=128, gamma=3, k=16, n=None, ragged=(1, 150), seed=82),
    # 16 KV heads at d = 64: the draft kernel's 16-consumer-warp form
    "hkv16_d64": Workload("h16", B=3, Hq=32, Hkv=16, d=64, gamma=3, k=40, n=None, ragged=(1, 400), seed=86),
    # many (sequence, KV head) rows at d = 64: the wide verify combine at that head dim
    "many_seqs_wide_d64": Workload("w64", B=80, Hq=8, Hkv=4, d=64, gamma=3, k=8, n=None, ragged=(1, 100),
                                   seed=87),
    # short prefixes whose weight sits on two sinks (same key, different values) and a
    # few heavy hitters: rounding P to bf16 alone puts one output element past the
    # tolerance here (1.02 of it, against 0.32 with P's low part)
    "two_sinks_short": Workload("sinks2", B=24, Hq=16, Hkv=4, d=128, gamma=3, k=6, n=None, ragged=(2, 90),
                                scheme="heavy", heavy_frac=0.02, sinks=2, u_per_seq=True, seed=85),
    # at least 64 entries a draft CTA: the draft kernel's three-stage ring, in its
    # packed (at most 8 query heads a KV head), unpacked and 16-warp forms
    "deep_ring_d128": Workload("deep128", B=12, Hq=32, Hkv=8, d=128, gamma=3, k=1000, n=None, ragged=(1001, 1300),
                               seed=88),
    "deep_ring_g16": Workload("deep16", B=12, Hq=16, Hkv=1, d=128, gamma=3, k=1000, n=None, ragged=(1001, 1300),
                              seed=89),
    "deep_ring_hkv16_d64": Workload("deep64", B=12, Hq=32, Hkv=16, d=64, gamma=3, k=1000, n=None,
                                    ragged=(1001, 1300), seed=90),
    # more sequences than draft CTAs, each a few entries: a CTA holds whole sequences and
    # finishes them itself (bf16 output and the token's append in the draft kernel)
    "complete_in_cta": Workload("b304", B=304, Hq=8, Hkv=2, d=64, gamma=3, k=8, n=None, ragged=(9, 60), seed=92),
    # ... and with a split that leaves some sequences whole in a CTA and cuts others
    "mixed_complete": Workload("b200", B=200, Hq=8, Hkv=2, d=64, gamma=3, k=8, n=None, ragged=(9, 60), seed=93),
}


@pytest.mark.parametrize("fill", [0x7F, 0xFF], ids=["ws_huge", "ws_nan"])
@pytest.mark.parametrize("name", list(CASES))
def test_iteration_matches_oracle(name, fill):
    from self_speculative_sparse_gb300.runtime import LayerState
    w = CASES[name]
    pool = w.layer_pool(0)
    st = LayerState(w, pool)
    # garbage workspace: results must not depend on its contents, finite (0x7F: 3.4e38)
    # or not (0xFF: NaN), also where a split leaves CTAs without work between the
    # ones that hold a (sequence, KV head)
    st.ws.fill_(fill)
    st.iteration()
    torch.cuda.synchronize()
    assert st.check_status() == 0, f"device status {st.check_status()}"
    rows1 = w.rows(w.extra_rows) if w.extra_rows else None
    check_iteration(w, pool, st, w.rows(w.select_rows), rows1)


def test_iteration_is_deterministic():
    from self_speculative_sparse_gb300.runtime import LayerState
    w = CASES["batched_b3_n700"]
    pool = w.layer_pool(0)
    a = LayerState(w, pool)
    a.iteration()
    b = LayerState(w, pool)
    b.iteration()
    torch.cuda.synchronize()
    for name in ("out_verify", "scores0", "scores1", "idx", "out_draft"):
        x, y = getattr(a, name), getattr(b, name)
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x,
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y), name


def test_plan_launches_match_the_call_bit_for_bit():
    """vg_iteration_plan_*: the captured iteration gives vg_iteration's results, launch
    after launch, and reads its buffers at launch time (new inputs, new results)."""
    from self_speculative_sparse_gb300.runtime import LayerState
    w = CASES["batched_b3_n700"]  # two masks: both selections run
    pool = w.layer_pool(0)
    names = ("out_verify", "scores0", "scores1", "idx", "count", "idx1", "count1", "out_draft")

    def bits(t):
        return t.view(torch.int16) if t.dtype == torch.bfloat16 else t

    a, b = LayerState(w, pool), LayerState(w, pool)
    with b.plan() as plan:
        for rnd in range(3):
            if rnd == 2:  # new inputs in the same buffers
                for st in (a, b):
                    st.q_verify.copy_(-st.q_verify)
                    st.q_draft.copy_(st.q_draft.flip(-1))
            a.iteration()
            for nm in names:
                getattr(b, nm).view(torch.uint8).fill_(0xA5)
            plan.launch()
            torch.cuda.synchronize()
            for nm in names:
                assert torch.equal(bits(getattr(a, nm)), bits(getattr(b, nm))), (rnd, nm)
    assert a.check_status() == 0 and b.check_status() == 0


def test_iteration_refuses_an_unstageable_draft_shape_before_enqueueing_anything():
    """16 KV heads at d = 128 leave no room to stage a token's pages for the draft: the
    call (and a plan) must refuse before the verify and selection are enqueued."""
    import ctypes
    from self_speculative_sparse_gb300 import binding as vb
    B, Hq, Hkv, d, gamma, n, k = 1, 16, 16, 128, 1, 64, 8
    R, dev = gamma + 1, "cuda"
    dims = vb.vg_dims(B=B, H_q=Hq, H_kv=Hkv, d=d, gamma=gamma, max_len=n, scale=0.0)
    slots = n + R + 16
    K = torch.zeros(slots, Hkv, d, dtype=torch.bfloat16, device=dev)
    V = torch.zeros_like(K)
    off = torch.zeros(B, dtype=torch.int64, device=dev)
    cache = vb.vg_kv_cache(vb.ptr(K), vb.ptr(V), vb.ptr(off), slots)
    bf = dict(dtype=torch.bfloat16, device=dev)
    q, kn, vn = torch.zeros(B, R, Hq, d, **bf), torch.zeros(B, R, Hkv, d, **bf), torch.zeros(B, R, Hkv, d, **bf)
    qd, kd, vd = torch.zeros(gamma, B, Hq, d, **bf), torch.zeros(gamma, B, Hkv, d, **bf), torch.zeros(gamma, B, Hkv, d, **bf)
    plen = torch.full((B,), n, dtype=torch.int32, device=dev)
    scores = torch.full((B, n), 7.0, device=dev)
    out = torch.full((B, R, Hq, d), 3.0, **bf)
    idx = torch.full((B, k), 5, dtype=torch.int32, device=dev)
    cnt = torch.full((B,), 5, dtype=torch.int32, device=dev)
    outd = torch.full((gamma, B, Hq, d), 3.0, **bf)
    wsb = vb.vg_workspace_size(dims, k)
    assert wsb > 0
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    ins = vb.vg_iter_inputs(vb.ptr(q), vb.ptr(kn), vb.ptr(vn), vb.ptr(qd), vb.ptr(kd), vb.ptr(vd), vb.ptr(plen))
    outs = vb.vg_iter_outputs(vb.ptr(out), vb.ptr(scores), None, n, vb.ptr(idx), vb.ptr(cnt), None, None,
                              vb.ptr(outd))
    lib = vb.load()
    mask = 1 | (1 << gamma)
    code = lib.vg_iteration(ctypes.byref(dims), ctypes.byref(cache), ctypes.byref(ins), k, mask, 0,
                            ctypes.byref(outs), vb.ptr(ws), wsb, None, None)
    h = ctypes.c_void_p(0x1234)
    code_plan = lib.vg_iteration_plan_create(ctypes.byref(dims), ctypes.byref(cache), ctypes.byref(ins), k, mask,
                                             0, ctypes.byref(outs), vb.ptr(ws), wsb, None, ctypes.byref(h))
    torch.cuda.synchronize()
    assert code == vb.VG_ERR_UNSUPPORTED_SHAPE and code_plan == vb.VG_ERR_UNSUPPORTED_SHAPE
    assert h.value is None
    assert bool((scores == 7.0).all()) and bool((out.float() == 3.0).all()) and bool((outd.float() == 3.0).all())
    assert bool((idx == 5).all()) and bool((cnt == 5).all()) and bool((K == 0).all())


def test_draft_over_the_whole_prefix_equals_verify_row_zero():
    """Two kernels against each other: with k >= n the selection is the whole prefix, and
    a draft token equal to verify row 0 (same q, k, v) attends exactly what that row
    attends - the prefix and itself.  Each path is within the oracle tolerance, so they
    agree within twice that."""
    from self_speculative_sparse_gb300.runtime import LayerState
    w = Workload("xk", B=3, Hq=8, Hkv=2, d=128, gamma=1, k=2048, n=None, ragged=(1, 1500), seed=88)
    st = LayerState(w, w.layer_pool(0))
    st.q_draft[0].copy_(st.q_verify[:, 0])
    st.k_draft[0].copy_(st.k_new[:, 0])
    st.v_draft[0].copy_(st.v_new[:, 0])
    st.iteration(select_extra=False)
    torch.cuda.synchronize()
    assert st.check_status() == 0
    n = st.prefix_len.cpu().numpy()
    assert np.array_equal(st.count.cpu().numpy(), n)          # everything selected
    a = st.out_draft[0].float().cpu().numpy()
    b = st.out_verify[:, 0].float().cpu().numpy()
    lim = 4e-3 + 2e-2 * np.abs(b)
    assert np.all(np.abs(a - b) <= lim), float(np.max(np.abs(a - b) - lim))


def test_verify_reads_new_rows_from_cache_when_not_given():
    from self_speculative_sparse_gb300.runtime import LayerState
    w = CASES["llama8b_n1000"]
    pool = w.layer_pool(0)
    st = LayerState(w, pool)
    st.verify(append=True)
    torch.cuda.synchronize()
    first = st.out_verify.clone()
    s_first = st.scores0.clone()
    st.out_verify.zero_()
    st.verify(append=False)       # the rows are now in the cache
    torch.cuda.synchronize()
    assert torch.equal(first.view(torch.int16), st.out_verify.view(torch.int16))
    assert torch.equal(s_first, st.scores0)


def test_topk_ties_signed_zero_and_edges():
    from self_speculative_sparse_gb300 import binding as vb
    rng = np.random.default_rng(3)
    lens = [0, 1, 5, 1000, 40000, 70000, 50000]
    B, L = len(lens), max(lens)
    sc = np.zeros((B, L), dtype=np.float32)
    for b, n in enumerate(lens):
        v = rng.integers(-4, 5, size=n).astype(np.float32)          # heavy ties
        v[v == 0] = np.where(rng.random((v == 0).sum()) < 0.5, -0.0, 0.0)
        if b == 4:
            v = rng.standard_normal(n).astype(np.float32) * 1e3     # spread values
        if b == 6:  # a few equal scores in each 16-bit key class: the candidates exchanged
            v = np.round(rng.standard_normal(n) * 1e3).astype(np.float32)   # after two passes tie
        sc[b, :n] = v
    dev = torch.from_numpy(sc).cuda()
    lt = torch.tensor(lens, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for k in (1, 3, 64, 5000, 100000):
        idx = torch.full((B, k), 7, dtype=torch.int32, device="cuda")
        cnt = torch.full((B,), 7, dtype=torch.int32, device="cuda")
        vb.vg_topk_select(dev, L, lt, B, L, k, idx, cnt, dev_status=status)
        torch.cuda.synchronize()
        gi, gc = idx.cpu().numpy(), cnt.cpu().numpy()
        for b, n in enumerate(lens):
            want = oracle.select_topk(sc[b, :n].astype(np.float64), k)
            m = min(k, n)
            assert gc[b] == m, (k, b)
            assert np.array_equal(gi[b, :m], want), (k, b)
            assert (gi[b, m:] == -1).all(), (k, b)
    assert int(status.item()) == 0


def test_device_bounds_are_reported_not_faulted():
    from self_speculative_sparse_gb300.runtime import LayerState
    from self_speculative_sparse_gb300 import binding as vb
    w = Workload("bad", B=2, Hq=8, Hkv=2, d=64, gamma=2, k=16, n=100, seed=81)
    pool = w.layer_pool(0)
    st = LayerState(w, pool)
    st.prefix_len[1] = 100000          # beyond max_len and beyond the cache
    st.verify()
    torch.cuda.synchronize()
    assert st.check_status() == vb.VG_ERR_DEVICE_BOUNDS
    # sequence 0 is unaffected
    K = oracle.widen_bf16(pool["K"][:100])
    V = oracle.widen_bf16(pool["V"][:100])
    ref = oracle.verify_attention(oracle.widen_bf16(pool["q_verify"][0]), K, V,
                                  oracle.widen_bf16(pool["k_new"][0]), oracle.widen_bf16(pool["v_new"][0]))
    assert_attn_close(bf16_to_f64(st.out_verify)[0], ref, "seq 0 after a bad seq 1")
    # a draft index outside [0, tail_start) is skipped and reported
    st2 = LayerState(w, pool)
    st2.iteration()
    torch.cuda.synchronize()
    assert st2.check_status() == 0
    st2.idx[0, 0] = 99999
    st2.status.zero_()
    tl = torch.full((w.B,), 1, dtype=torch.int32, device="cuda")
    st2.draft_step(0, tl)
    torch.cuda.synchronize()
    assert st2.check_status() == vb.VG_ERR_DEVICE_BOUNDS
    assert torch.isfinite(st2.out_draft[0].float()).all()


def test_topk_repeated_runs_are_identical_and_exact():
    """Many launches of the multi-CTA selection on one input: a race would show."""
    from self_speculative_sparse_gb300 import binding as vb
    rng = np.random.default_rng(11)
    lens = [32768, 32768, 20000]
    B, L = len(lens), max(lens)
    sc = (rng.standard_normal((B, L)) * 10).astype(np.float32)
    sc[1, ::7] = 3.0                                                  # a block of exact ties
    dev = torch.from_numpy(sc).cuda()
    lt = torch.tensor(lens, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    k = 2048
    want = [oracle.select_topk(sc[b, :n].astype(np.float64), k) for b, n in enumerate(lens)]
    idx = torch.empty((B, k), dtype=torch.int32, device="cuda")
    cnt = torch.empty((B,), dtype=torch.int32, device="cuda")
    for rep in range(50):
        idx.fill_(123456)
        vb.vg_topk_select(dev, L, lt, B, L, k, idx, cnt, dev_status=status)
        torch.cuda.synchronize()
        gi = idx.cpu().numpy()
        for b in range(B):
            assert np.array_equal(gi[b], want[b]), (rep, b)
    assert int(status.item()) == 0


def test_graph_replay_rotation_keeps_status_clean():
    """The benchmark's flow: CUDA-graph replays of verify/select/draft over rotating
    cache copies, with the public draft entry point and a device tail-length array."""
    from self_speculative_sparse_gb300.runtime import LayerState
    w = scaled(W["llama8b"], n=4000, k=512)
    pool = w.layer_pool(0)
    ncopy = 3
    states = [LayerState(w, pool) for _ in range(ncopy)]
    tl = [torch.full((w.B,), s + 1, dtype=torch.int32, device="cuda") for s in range(w.gamma)]

    def draft_phase(st):
        for s in range(w.gamma):
            st.draft_step(s, tl[s])

    for st in states:
        st.iteration(select_extra=False)
    torch.cuda.synchronize()
    graphs = []
    for c in range(ncopy):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            a, b = states[c], states[(c + 1) % ncopy]
            a.verify()
            a.select()
            draft_phase(b)
        graphs.append(g)
    for i in range(60):
        graphs[i % ncopy].replay()
    torch.cuda.synchronize()
    assert [st.check_status() for st in states] == [0] * ncopy
    check_iteration(w, pool, states[0], w.rows(w.select_rows), None)


def test_a_lost_wait_reports_a_timeout_and_the_gpu_stays_usable():
    """The failure path of the bounded waits, made to run out on purpose (no fault, no
    hang): a wait that nothing completes gives up after its limit and reports
    VG_ERR_DEVICE_TIMEOUT; the CTA's abort flag makes the other wait give up at once
    (not after its own 2 s); the next call works as usual."""
    from self_speculative_sparse_gb300 import binding as vb
    from self_speculative_sparse_gb300.runtime import LayerState
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(1, dtype=torch.int64, device="cuda")
    vb.vg_selftest_lost_wait(20000, status, elapsed)
    torch.cuda.synchronize()
    assert int(status.item()) == vb.VG_ERR_DEVICE_TIMEOUT
    ns = int(elapsed.item())
    assert 20e6 <= ns < 500e6, ns
    w = CASES["tiny"]
    pool = w.layer_pool(0)
    st = LayerState(w, pool)
    st.iteration()
    torch.cuda.synchronize()
    assert st.check_status() == 0
    check_iteration(w, pool, st, w.rows(w.select_rows), w.rows(w.extra_rows) if w.extra_rows else None)


def test_window_selection_matches_oracle():
    """The sliding-window comparison policy (Vegas §1): bit-exact against the oracle,
    with prefixes shorter than, equal to and longer than k, empty, and several CTAs of k."""
    from self_speculative_sparse_gb300 import binding as vb
    lens = [0, 1, 5, 300, 301, 999, 70000]
    B, L = len(lens), max(lens)
    lt = torch.tensor(lens, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for k in (1, 300, 700):
        idx = torch.full((B, k), 7, dtype=torch.int32, device="cuda")
        cnt = torch.full((B,), 7, dtype=torch.int32, device="cuda")
        vb.vg_window_select(lt, B, L, k, idx, cnt, dev_status=status)
        torch.cuda.synchronize()
        gi, gc = idx.cpu().numpy(), cnt.cpu().numpy()
        for b, n in enumerate(lens):
            want = oracle.select_window(n, k)
            assert gc[b] == len(want), (k, b)
            assert np.array_equal(gi[b, :len(want)], want), (k, b)
            assert (gi[b, len(want):] == -1).all(), (k, b)
    assert int(status.item()) == 0


@pytest.mark.parametrize("name", ["llama8b_n1000", "ragged_b6", "deep_ring_d128", "complete_in_cta"])
def test_settled_draft_steps_equal_plain_ones(name):
    """VG_DRAFT_SELECTION_SETTLED only moves the gather of the selected entries ahead of
    the dependency wait: the steps' outputs and appends are bit-identical to those of
    calls without the flag (and those match the oracle through the iteration tests)."""
    from self_speculative_sparse_gb300.runtime import LayerState
    w = CASES[name]
    pool = w.layer_pool(0)
    tl = [torch.full((w.B,), s + 1, dtype=torch.int32, device="cuda") for s in range(w.gamma)]
    outs = []
    for settled in (False, True):
        st = LayerState(w, pool)
        st.verify()
        st.select()
        for s in range(w.gamma):
            st.draft_step(s, tl[s], settled=settled and s > 0)
        torch.cuda.synchronize()
        assert st.check_status() == 0
        outs.append((st.out_draft.view(torch.int16).clone(), st.K.view(torch.int16).clone(),
                     st.V.view(torch.int16).clone()))
    for x, y, nm in zip(outs[0], outs[1], ("draft outputs", "K cache", "V cache")):
        assert torch.equal(x, y), nm


def test_draft_launch_count():
    """vg_sparse_draft_launches: 1 when each sequence's entries fall to a single CTA of the
    step's grid (that CTA finishes it), else 2 (a second kernel merges the partials)."""
    from self_speculative_sparse_gb300 import binding as vb
    dims = lambda B: vb.make_dims(B=B, H_q=8, H_kv=2, d=64, gamma=3, max_len=4096)
    # one sequence of 2048 + 4 entries over many CTAs: merged by a second kernel
    assert vb.vg_sparse_draft_launches(dims(1), 2048, 4) == 2
    # 256 sequences of 4 + 4 entries: a small step, CTAs of two whole chunks (32
    # entries), so every CTA holds four whole sequences and finishes them
    assert vb.vg_sparse_draft_launches(dims(256), 4, 4) == 1
