"""GPU parity of the paged KV cache (a vLLM-style block table; Vegas §3 runs the draft
as a paged attention whose pages are tokens).

The same layers are laid out in pages scattered over the pool by a seeded permutation:
* a whole iteration (verify, selection, draft steps) with pages of 8, 16, 32, 64 and 128
  tokens matches the oracle, including the appends landing in the right physical slots,
  also with prefixes long enough that each verify CTA streams tens of tiles;
* it matches the slot-pool layout of the same data bit for bit (the layout changes the
  addressing, not the arithmetic);
* the draft step alone reads pages of one token (the page indices are token slots);
* page sizes the verify pass cannot box are refused before anything is enqueued.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import synth  # noqa: E402
from synth import Workload, scaled  # noqa: E402
from tests.parity import assert_attn_close, bf16_to_f64, check_iteration, token_slots  # noqa: E402

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
    "ragged_b6": scaled(W["loop32"], B=6, layers=1, ragged=(1, 1500)),
    "batched_b3_n700": scaled(W["batched"], B=3, n=700),
    "g16_m64_d64": Workload("g16d64", B=2, Hq=16, Hkv=1, d=64, gamma=3, k=100, n=777, seed=84),
    # at least 64 entries a draft CTA: the draft kernel's three-stage ring through pages
    "deep_ring_d128": Workload("deep128", B=12, Hq=32, Hkv=8, d=128, gamma=3, k=1000, n=None, ragged=(1001, 1300),
                               seed=88),
}


@pytest.mark.parametrize("P", [8, 16, 32, 64, 128])
@pytest.mark.parametrize("name", list(CASES))
def test_paged_iteration_matches_oracle_and_the_slot_pool(name, P):
    _paged_matches(CASES[name], P)


# Long prefixes: each verify CTA streams some 60-70 tiles, so its producer goes through
# several batches of page-table words (32 tiles a batch at 64-token pages, 8 at 16).
LONG = Workload("paged_long", B=4, Hq=32, Hkv=8, d=128, gamma=6, k=512, n=None, ragged=(15000, 22000), seed=91)


@pytest.mark.parametrize("P", [16, 64])
def test_paged_long_prefixes_match_oracle_and_the_slot_pool(P):
    _paged_matches(LONG, P)


def _paged_matches(w, P):
    from self_speculative_sparse_gb300.runtime import LayerState
    flat = w.layer_pool(0)
    paged = synth.to_paged(w, flat, P, seed=P)
    a = LayerState(w, flat)
    b = LayerState(w, paged)
    assert b.page_table is not None
    b.ws.fill_(0xFF)
    a.iteration()
    b.iteration()
    torch.cuda.synchronize()
    assert a.check_status() == 0 and b.check_status() == 0
    rows1 = w.rows(w.extra_rows) if w.extra_rows else None
    check_iteration(w, paged, b, w.rows(w.select_rows), rows1)
    for nm in ("out_verify", "scores0", "idx", "count", "out_draft"):
        x, y = getattr(a, nm), getattr(b, nm)
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x,
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y), nm


def test_draft_reads_pages_of_one_token():
    """Page size one (Vegas §3): every token its own page anywhere in the pool.  The
    selection is the oracle's on the oracle's scores; the draft step must match the
    oracle's and append the draft token into its page."""
    from self_speculative_sparse_gb300 import binding as vb
    from self_speculative_sparse_gb300.runtime import LayerState
    w = scaled(W["loop32"], B=4, layers=1, ragged=(50, 900), k=64)
    flat = w.layer_pool(0)
    paged = synth.to_paged(w, flat, 1, seed=3)
    st = LayerState(w, paged)
    n = paged["prefix_len"]
    idx = np.full((w.B, w.k), -1, dtype=np.int32)
    cnt = np.zeros(w.B, dtype=np.int32)
    for b in range(w.B):
        sl = token_slots(paged, b, int(n[b]))
        K = oracle.widen_bf16(paged["K"][sl])
        T = oracle.select_topk(oracle.aggregated_scores(oracle.widen_bf16(paged["q_verify"][b]), K,
                                                        w.rows("c2")), w.k)
        idx[b, :len(T)] = T
        cnt[b] = len(T)
    st.idx.copy_(torch.from_numpy(idx))
    st.count.copy_(torch.from_numpy(cnt))
    tl = torch.full((w.B,), 1, dtype=torch.int32, device="cuda")
    st.draft_step(0, tl)
    torch.cuda.synchronize()
    assert st.check_status() == 0
    Kc, Vc = bf16_to_f64(st.K), bf16_to_f64(st.V)
    out = bf16_to_f64(st.out_draft[0])
    for b in range(w.B):
        nb = int(n[b])
        sl = token_slots(paged, b, nb + 1)
        K = oracle.widen_bf16(paged["K"][sl[:nb]])
        V = oracle.widen_bf16(paged["V"][sl[:nb]])
        kd, vd = oracle.widen_bf16(paged["k_draft"][0, b]), oracle.widen_bf16(paged["v_draft"][0, b])
        ref = oracle.draft_step(oracle.widen_bf16(paged["q_draft"][0, b]), K, V, idx[b, :cnt[b]], kd[None], vd[None])
        assert_attn_close(out[b], ref, f"page-size-one draft seq {b}")
        assert np.array_equal(Kc[sl[nb]], kd) and np.array_equal(Vc[sl[nb]], vd)  # the append, in its page


@pytest.mark.parametrize("P", [1, 4, 24])
def test_verify_refuses_page_sizes_it_cannot_box(P):
    from self_speculative_sparse_gb300 import binding as vb
    from self_speculative_sparse_gb300.runtime import LayerState
    w = CASES["tiny"]
    paged = synth.to_paged(w, w.layer_pool(0), P, seed=1)
    st = LayerState(w, paged)
    sentinel = st.out_verify.clone()
    with pytest.raises(vb.VgError) as e:
        st.verify()
    assert e.value.status == vb.VG_ERR_UNSUPPORTED_SHAPE
    with pytest.raises(vb.VgError) as e:
        st.iteration()
    assert e.value.status == vb.VG_ERR_UNSUPPORTED_SHAPE
    torch.cuda.synchronize()
    assert torch.equal(st.out_verify.view(torch.int16), sentinel.view(torch.int16))
