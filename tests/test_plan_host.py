"""IterationPlan, the owner of a vg_iteration_plan handle, on the host: it frees the
handle exactly once, refuses launches after that, and keeps the tensors the plan was
captured on alive until then.  The C calls are replaced by recording fakes, so this
runs without a GPU (the captured graph itself is checked on the GPU, against
vg_iteration, in the parity tests)."""
import gc

import pytest

torch = pytest.importorskip("torch")

from self_speculative_sparse_gb300 import runtime  # noqa: E402


class FakeBinding:
    def __init__(self):
        self.launched, self.destroyed = [], []

    def vg_iteration_plan_launch(self, plan, stream=None):
        self.launched.append((plan, stream))

    def vg_iteration_plan_destroy(self, plan):
        self.destroyed.append(plan)


@pytest.fixture
def fake(monkeypatch):
    fb = FakeBinding()
    monkeypatch.setattr(runtime.vb, "vg_iteration_plan_launch", fb.vg_iteration_plan_launch)
    monkeypatch.setattr(runtime.vb, "vg_iteration_plan_destroy", fb.vg_iteration_plan_destroy)
    return fb


def test_close_frees_the_handle_once_and_later_launches_raise(fake):
    plan = runtime.IterationPlan(0xBEEF, [torch.zeros(4)])
    plan.launch()
    plan.launch(stream="s1")
    assert fake.launched == [(0xBEEF, None), (0xBEEF, "s1")]
    plan.close()
    plan.close()
    assert fake.destroyed == [0xBEEF]
    with pytest.raises(RuntimeError):
        plan.launch()


def test_context_manager_closes_and_releases_the_tensors(fake):
    t = torch.zeros(8)
    with runtime.IterationPlan(7, [t]) as plan:
        assert plan._tensors[0] is t
    assert fake.destroyed == [7]
    assert plan.handle is None and plan._tensors == []


def test_the_plan_keeps_its_tensors_alive_until_closed(fake):
    import weakref
    t = torch.zeros(16)
    ref = weakref.ref(t)
    plan = runtime.IterationPlan(9, [t])
    del t
    gc.collect()
    assert ref() is not None  # still held by the plan: its buffers must not move
    plan.close()
    gc.collect()
    assert ref() is None


def test_garbage_collection_destroys_an_unclosed_plan(fake):
    plan = runtime.IterationPlan(11, [])
    del plan
    gc.collect()
    assert fake.destroyed == [11]
