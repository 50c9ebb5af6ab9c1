"""Allocation failures injected on the host (no GPU fault): the library's device allocations go
through an allocator hook (s1_set_allocator) that fails the n-th request. For every n in one
model's life (creation, prefill, decide), the failing call returns S1_ERR_OOM, every block
allocated before it is released once the caller closes what it holds, and a model that saw the
failure still prefills and decides with the same results afterwards."""
import ctypes as C

import numpy as np
import pytest

from prefill_only_decision_gb300 import configs, synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from prefill_only_decision_gb300 import binding
    binding.lib()
    return binding


class FailingAllocator:
    """Device blocks from PyTorch's caching allocator; request number `fail_at` gets NULL."""

    def __init__(self, B):
        self.live = {}
        self.count = 0
        self.fail_at = None

        def alloc(n, _ctx):
            self.count += 1
            if self.fail_at is not None and self.count == self.fail_at:
                return None
            p = torch.cuda.caching_allocator_alloc(int(n))
            self.live[p] = int(n)
            return p

        def free(p, _ctx):
            if p and self.live.pop(p, None) is not None:
                torch.cuda.caching_allocator_delete(p)

        self._a, self._f = B._ALLOC_T(alloc), B._FREE_T(free)   # kept alive while installed
        B.check(B.lib().s1_set_allocator(C.cast(self._a, C.c_void_p), C.cast(self._f, C.c_void_p), None))

    def reset(self, fail_at=None):
        self.count = 0
        self.fail_at = fail_at


def _results(res):
    return [(r["probs"].copy(), r["hidden"].copy()) for r in res]


def test_every_allocation_failure_returns_oom_and_leaks_nothing(B):
    W = synth.make_weights(configs.TINY)
    req = synth.make_requests(configs.TINY)[0]
    fa = FailingAllocator(B)
    try:
        # a full life without failures: the number of allocations it makes, and its results
        m = B.Model(W)
        st = m.prefill(req.tokens)
        ref = _results(m.decide(st, req.questions))
        st.close()
        m.close()
        total = fa.count
        assert total >= 4 and not fa.live
        for n in range(1, total + 1):
            fa.reset(fail_at=n)
            m = st = None
            failed = False
            where = "create"
            try:
                m = B.Model(W)
                where = "prefill"
                st = m.prefill(req.tokens)
                where = "decide"
                m.decide(st, req.questions)
            except B.S1Error as e:
                assert e.code == B.S1_ERR_OOM, (n, str(e))
                failed = True
                where += f" ({e})"
            assert failed, n   # the n-th request is made in every life
            if m is not None:
                # the model is still usable: the same prefill and decide give the same results
                fa.reset()
                try:
                    if st is not None:
                        st.close()
                    st = m.prefill(req.tokens)
                    got = _results(m.decide(st, req.questions))
                    for (p, h), (rp, rh) in zip(got, ref):
                        msg = f"allocation {n} of {total}: {where}"
                        np.testing.assert_allclose(p, rp, rtol=0, atol=1e-6, err_msg=msg)
                        np.testing.assert_allclose(h, rh, rtol=1e-6, atol=1e-6, err_msg=msg)
                finally:
                    if st is not None:
                        st.close()
                    m.close()
            assert not fa.live, (n, fa.live)
    finally:
        B.use_default_allocator()


def test_model_frees_through_the_allocator_it_was_created_with(B):
    """Hooks installed after a model's creation do not apply to it: a model and its snapshot
    created under one allocator give every block back to that allocator when they are closed
    after the default allocator has been restored (no block freed through cudaFree)."""
    W = synth.make_weights(configs.TINY)
    req = synth.make_requests(configs.TINY)[0]
    fa = FailingAllocator(B)
    m = st = None
    try:
        m = B.Model(W)
        st = m.prefill(req.tokens)
        m.decide(st, req.questions)
        assert fa.live
    finally:
        B.use_default_allocator()
    try:
        m.decide(st, req.questions + req.questions)   # may grow scratch: through the model's hooks
    finally:
        st.close()
        m.close()
    assert not fa.live, fa.live
