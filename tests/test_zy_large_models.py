"""Parity of the 4B, 4B-multimodal and 27B models (C ABI, GPU) against the fp32 oracle.

The oracle's results for these configurations take CPU minutes to an hour to compute, so they
are stored (tests/golden/large_*.npz, written by tests/golden/make_large_goldens.py from the
oracle and the seeded generators alone) and the GPU results are compared with them under the
full tolerance contract (`parity.compare`). A teacher-forced per-layer check
(`parity.layerwise`) runs the f16-policy oracle's layer on the GPU's own layer inputs, so a
kernel error in any layer shows up undiluted by depth. Collected after the fast tests.
"""
import os

import numpy as np
import pytest

from parity import compare, golden_results, layerwise
from prefill_only_decision_gb300 import configs, synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
torch = pytest.importorskip("torch")
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from prefill_only_decision_gb300 import binding
    binding.lib()
    return binding


def _sweep_subset(reqs):
    """Request 0 (the nominal prefix) and the shortest, median and longest of the sweep: the
    same choice as the golden writer's, recomputed from the same seeded requests."""
    lens = np.array([len(r.tokens) for r in reqs])
    order = np.argsort(lens, kind="stable")
    pick = []
    for i in (0, int(order[0]), int(order[len(order) // 2]), int(order[-1])):
        if i not in pick:
            pick.append(i)
    return pick


def test_4b_two_call_and_fused_vs_oracle(B):
    """The 4B request (1024-token prefix, 3 x 48-token questions): the two-call path (prefix
    snapshot, then the questions over it) and the one-sweep call, each against the oracle; then
    the per-layer check on the one-sweep call."""
    cfg = configs.QWEN4B
    ref = golden_results(os.path.join(GOLDEN, "large_4b.npz"))[0]
    W = synth.make_weights(cfg)
    req = synth.make_requests(cfg)[0]
    m = B.Model(W)
    try:
        st = m.prefill(req.tokens)
        two = m.decide(st, req.questions)
        st.close()
        fused, _ = m.prefill_decide(req)
    finally:
        m.close()
    compare(two, ref, req.questions, "4b two-call")
    compare(fused, ref, req.questions, "4b one-sweep")
    layerwise(B, torch, W, req, "4b")


def test_4b_multimodal_batch_vs_oracle(B):
    """Batch of 8 requests (1024 given embedding rows + 256 tokens, 32 questions of 40 tokens
    each) in one batched prefill and one batched decide; request 0's 32 questions against the
    oracle, and the one-sweep batch call against the two-call results."""
    cfg = configs.QWEN4B_MM
    ref = golden_results(os.path.join(GOLDEN, "large_4b_mm.npz"))[0]
    W = synth.make_weights(cfg)
    reqs = synth.make_requests(cfg)
    m = B.Model(W)
    try:
        states = m.prefill_batch(reqs)
        assert all(s.rows == 1280 for s in states)
        gpu = m.decide_batch(states, [r.questions for r in reqs])
        for s in states:
            s.close()
        fused, _ = m.prefill_decide_batch(reqs[:2])
    finally:
        m.close()
    compare(gpu[0], ref, reqs[0].questions, "4b-mm request 0")
    compare(fused[0], ref, reqs[0].questions, "4b-mm one-sweep request 0")
    for r, g in zip(reqs, gpu):
        for q, x in zip(r.questions, g):
            assert abs(float(x["probs"].sum()) - 1) < 1e-5 and 0 <= x["expected_score"] <= len(q.option_ids) - 1


def test_27b_sweep_subset_vs_oracle(B):
    """27B-class model: request 0 (P = 1536) and the shortest, median and longest prefix of the
    seeded 74-request sweep, each prefilled and decided on the GPU and compared with the oracle;
    the per-layer check runs on the shortest request at the first and last four layers."""
    cfg = configs.QWEN27B
    gold = golden_results(os.path.join(GOLDEN, "large_27b.npz"))
    reqs = synth.make_requests(cfg)
    pick = _sweep_subset(reqs)
    assert sorted(pick) == sorted(gold), (pick, sorted(gold))
    W = synth.make_weights(cfg)
    m = B.Model(W)
    try:
        for i in pick:
            st = m.prefill(reqs[i].tokens)
            gpu = m.decide(st, reqs[i].questions)
            st.close()
            compare(gpu, gold[i], reqs[i].questions, f"27b request {i} P={len(reqs[i].tokens)}")
    finally:
        m.close()
    i = min(pick, key=lambda k: len(reqs[k].tokens))
    L = cfg.shape.n_layers
    layerwise(B, torch, W, reqs[i], f"27b request {i}", layers=[0, 1, 2, 3, L - 4, L - 3, L - 2, L - 1])
