"""The draft step for callers that cannot allocate device memory.

Some hosts cannot hand the library device memory while decoding: calling
cudaMalloc there can synchronise the device and stall other streams, or the host
simply has no workspace to offer.  vg_sparse_draft_attn_noalloc serves them from a
scratch area built into the library.  These tests call it through the C ABI, twice
in a row, and compare each result with vg_sparse_draft_attn (the workspace entry
point) on the same inputs: both run the same kernels in the same order, so the
outputs must agree bit for bit.  They also check that dimensions too large for the
built-in area are refused before anything runs.
"""
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from self_speculative_sparse_gb300 import build
    build.build()


def test_noalloc_draft_step_matches_the_workspace_entry_point_twice():
    import synth
    from self_speculative_sparse_gb300 import binding as vb
    from self_speculative_sparse_gb300.runtime import LayerState

    w = synth.scaled(synth.WORKLOADS["llama8b"], B=2, n=3000, k=256)
    st = LayerState(w, w.layer_pool(0))
    st.iteration(select_extra=False)
    torch.cuda.synchronize()
    assert st.check_status() == 0
    for s in range(2):  # two calls in a row: the built-in area is reused
        tl = torch.full((w.B,), s + 1, dtype=torch.int32, device="cuda")
        ref = torch.empty_like(st.out_draft[s])
        got = torch.full_like(ref, float("nan"))
        vb.vg_sparse_draft_attn(st.dims, st.cache, st.q_draft[s], st.k_draft[s], st.v_draft[s], st.idx, st.count,
                                st.k, st.prefix_len, tl, ref, st.ws, dev_status=st.status)
        vb.vg_sparse_draft_attn_noalloc(st.dims, st.cache, st.q_draft[s], st.k_draft[s], st.v_draft[s], st.idx,
                                        st.count, st.k, st.prefix_len, tl, got, dev_status=st.status)
        torch.cuda.synchronize()
        assert st.check_status() == 0
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), f"no-allocation draft step, call {s + 1}"


def test_noalloc_refuses_dimensions_beyond_its_scratch():
    from self_speculative_sparse_gb300 import binding as vb

    t = torch.zeros(1024, dtype=torch.int64, device="cuda")
    dims = vb.make_dims(1024, 128, 8, 128, 3, 4096)  # draft scratch far above the built-in 8 MiB
    cache = vb.make_cache(t, t, t, capacity_slots=16)
    with pytest.raises(vb.VgError) as e:
        vb.vg_sparse_draft_attn_noalloc(dims, cache, t, None, None, t, t, 16, t, t, t)
    assert e.value.status == vb.VG_ERR_WORKSPACE
    assert "built-in" in str(e.value)
