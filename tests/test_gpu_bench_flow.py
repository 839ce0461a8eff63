"""The benchmark's multi-layer step inside a CUDA graph runs every call it times.

bench.py times the 32-layer workload as one captured graph of its step: every layer's
verify, each layer's selection on a second stream beside the next layers' verification,
then each draft step over every layer.  A fork that missed the capture would leave the
selections out of the graph (they would run once, at capture time), and the step would
be timed without them.  Here the selections' outputs are cleared before a replay and
must come back equal to those of the calls made in order.
"""
import importlib.util
import os

import pytest

torch = pytest.importorskip("torch")

import synth  # noqa: E402

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from self_speculative_sparse_gb300 import build
    build.build()


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return b


def test_captured_multilayer_step_runs_every_selection_and_draft_step():
    bench = _bench()
    w = synth.scaled(synth.WORKLOADS["loop32"], layers=3)
    S = bench.Setup(w, 0)
    for st in S.states:  # the calls in order: the reference outputs
        st.verify()
        st.select()
    for s in range(w.gamma):
        for st in S.states:
            st.draft_step(s, S.tl[s])
    torch.cuda.synchronize()
    ref = [(st.idx.clone(), st.count.clone(), st.out_draft.view(torch.int16).clone()) for st in S.states]
    g = bench.capture(lambda: S.step(0))
    for st in S.states:
        st.idx.fill_(-5)
        st.count.fill_(-5)
        st.out_draft.zero_()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    S.check("graph replay")
    for layer, st in enumerate(S.states):
        assert torch.equal(st.idx, ref[layer][0]), f"layer {layer}: selection missing from the graph"
        assert torch.equal(st.count, ref[layer][1]), f"layer {layer}: selection count"
        assert torch.equal(st.out_draft.view(torch.int16), ref[layer][2]), f"layer {layer}: draft outputs"
