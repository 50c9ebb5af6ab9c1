"""End-to-end parity of the decision path (C ABI, GPU) against the oracle, plus the
boundary's behaviour: errors, state reuse, isolation and ordering of questions.

Every result is held to the tolerance contract of the method's acceptance bar against the plain
fp32 oracle (LoRA unmerged, fp32 everywhere): per-option probabilities within 2e-2 absolute,
expected score within 5e-2, last-layer hidden state within 3e-2 relative L2, identical argmax
wherever the oracle's top-2 margin exceeds 0.05 (`parity.compare`). The 4B, 4B-multimodal and
27B models are checked in test_zy_large_models.py against stored oracle results."""
import numpy as np
import pytest

from oracle import model as om
from parity import compare, layerwise
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


@pytest.fixture(scope="module")
def tiny(B, tiny_weights):
    m = B.Model(tiny_weights)
    yield m
    m.close()


def test_small_layerwise(B):
    """Per-layer parity of the small model (8 layers, LoRA) on one request's fused sweep."""
    cfg = configs.SMALL
    W = synth.make_weights(cfg)
    layerwise(B, torch, W, synth.make_requests(cfg, n_requests=1)[0], "small")


def test_tiny_vs_oracle_unbranched(tiny, tiny_weights, tiny_requests):
    r = tiny_requests[0]
    ref = om.Oracle(tiny_weights, np.float32).decide(r, branched=False)
    st = tiny.prefill(r.tokens)
    assert st.rows == len(r.tokens)
    gpu = tiny.decide(st, r.questions)
    compare(gpu, ref, r.questions, "tiny")


@pytest.mark.skipif(bool(__import__("os").environ.get("S1_TEST_NO_TC")), reason="tensor-core path disabled")
def test_tiny_simt_gemm_path_agrees(tiny, tiny_weights, tiny_requests):
    r = tiny_requests[0]
    st = tiny.prefill(r.tokens)
    a = tiny.decide(st, r.questions)
    tiny.set_gemm_impl(1)
    try:
        st2 = tiny.prefill(r.tokens)
        b = tiny.decide(st2, r.questions)
    finally:
        tiny.set_gemm_impl(0)
    for x, y in zip(a, b):
        assert np.abs(x["probs"] - y["probs"]).max() < 2e-3
        assert np.linalg.norm(x["hidden"] - y["hidden"]) / np.linalg.norm(y["hidden"]) < 5e-3


def test_tiny_state_reuse_and_permutation_bitexact(tiny, tiny_requests):
    r = tiny_requests[0]
    st = tiny.prefill(r.tokens)
    a = tiny.decide(st, r.questions)
    b = tiny.decide(st, r.questions)
    perm = [2, 0, 1]
    c = tiny.decide(st, [r.questions[i] for i in perm])
    for i in range(3):
        np.testing.assert_array_equal(a[i]["probs"], b[i]["probs"])
        np.testing.assert_array_equal(a[i]["hidden"], b[i]["hidden"])
    for k, i in enumerate(perm):
        np.testing.assert_array_equal(a[i]["probs"], c[k]["probs"])
        np.testing.assert_array_equal(a[i]["hidden"], c[k]["hidden"])


def test_tiny_isolation_add_remove(tiny, tiny_requests):
    r = tiny_requests[0]
    st = tiny.prefill(r.tokens)
    a = tiny.decide(st, r.questions)
    one = tiny.decide(st, r.questions[1:2])
    g = np.random.default_rng(11)
    extra = [synth.random_question(g, 4096, configs.CHOICE, 37, 5) for _ in range(4)]
    many = tiny.decide(st, extra[:2] + [r.questions[1]] + extra[2:])
    np.testing.assert_allclose(one[0]["probs"], a[1]["probs"], atol=1e-5)
    np.testing.assert_allclose(many[2]["probs"], a[1]["probs"], atol=1e-5)


def test_tiny_edge_cases_vs_oracle(tiny, tiny_weights):
    """Ragged suffixes (1, 7, 64, 65, 130 rows), a one-option choice, P = 1 and a long prefix."""
    o = om.Oracle(tiny_weights, np.float32)
    g = np.random.default_rng(7)
    qs = [synth.random_question(g, 4096, configs.CHOICE, 1, 1),
          synth.random_question(g, 4096, configs.SCORE, 7, 9),
          synth.random_question(g, 4096, configs.NOUL, 64, 2),
          synth.random_question(g, 4096, configs.CHOICE, 65, 26),
          synth.random_question(g, 4096, configs.SCORE, 130, 2)]
    for P in (1, 200):
        toks = g.integers(16, 4096, size=P).astype(np.int32)
        st = tiny.prefill(toks)
        gpu = tiny.decide(st, qs)
        _, caches, PP = o.prefill(toks)
        ref = o.decide_branched(caches, PP, qs)
        compare(gpu, ref, qs, f"edge P={P}")
        assert gpu[0]["confidence"] == 1.0 and gpu[0]["probs"][0] == 1.0


def test_tiny_async_device_api_matches(tiny, tiny_requests, B):
    r = tiny_requests[0]
    st_h = tiny.prefill(r.tokens)
    ref = tiny.decide(st_h, r.questions)
    st = tiny.state_create(len(r.tokens))
    dt = torch.from_numpy(r.tokens).cuda()
    tiny.prefill_async(st, dt.data_ptr(), len(r.tokens))
    dev = []
    for q in r.questions:
        s, o = torch.from_numpy(q.suffix).cuda(), torch.from_numpy(q.option_ids).cuda()
        dev.append(synth.Question(q.type, s, o))
    import ctypes as C
    arr = (B.Question * len(dev))()
    for j, q in enumerate(dev):
        arr[j] = B.Question(q.type, C.cast(C.c_void_p(q.suffix.data_ptr()), C.POINTER(C.c_int32)), q.suffix.numel(),
                            C.cast(C.c_void_p(q.option_ids.data_ptr()), C.POINTER(C.c_int32)), q.option_ids.numel())
    n_opt = sum(len(q.option_ids) for q in r.questions)
    probs = torch.zeros(n_opt, dtype=torch.float32, device="cuda")
    stats = torch.zeros((3, 8), dtype=torch.float32, device="cuda")
    hid = torch.zeros((3, 256), dtype=torch.float32, device="cuda")
    tiny.decide_async(st, arr, 3, probs.data_ptr(), stats.data_ptr(), hid.data_ptr())
    tiny.sync()
    p = probs.cpu().numpy()
    off = 0
    for j, q in enumerate(r.questions):
        np.testing.assert_array_equal(p[off:off + len(q.option_ids)], ref[j]["probs"])
        np.testing.assert_array_equal(hid[j].cpu().numpy(), ref[j]["hidden"])
        assert int(stats[j, 0].item()) == ref[j]["argmax"]
        off += len(q.option_ids)


def test_boundary_errors(tiny, tiny_requests, B):
    r = tiny_requests[0]
    st = tiny.prefill(r.tokens)
    bad_id = synth.Question(configs.CHOICE, np.array([5, 4096], np.int32), np.array([20, 21], np.int32))
    bad_noul = synth.Question(configs.NOUL, np.array([5], np.int32), np.array([20, 21, 22], np.int32))
    bad_score = synth.Question(configs.SCORE, np.array([5], np.int32), np.array([20], np.int32))
    empty = synth.Question(configs.CHOICE, np.array([], np.int32), np.array([20], np.int32))
    for q in (bad_id, bad_noul, bad_score, empty):
        with pytest.raises(B.S1Error) as e:
            tiny.decide(st, [q])
        assert e.value.code == B.S1_ERR_INVALID_ARG
    with pytest.raises(B.S1Error) as e:
        tiny.prefill(np.array([1, 2, -3], np.int32))
    assert e.value.code == B.S1_ERR_INVALID_ARG
    with pytest.raises(B.S1Error) as e:
        tiny.prefill(np.zeros(40000, np.int32))
    assert e.value.code == B.S1_ERR_BUDGET
    # the model still works after rejected calls, and a destroyed state is refused
    good = tiny.decide(st, r.questions[:1])
    assert abs(float(good[0]["probs"].sum()) - 1) < 1e-5
    dead = B.State(tiny, st.h)
    st.h = None
    B.lib().s1_state_destroy(dead.h)
    with pytest.raises(B.S1Error) as e:
        tiny.decide(dead, r.questions[:1])
    assert e.value.code == B.S1_ERR_INVALID_HANDLE
    dead.h = None


def test_small_batch_vs_oracle(B):
    cfg = configs.SMALL
    W = synth.make_weights(cfg)
    reqs = synth.make_requests(cfg)
    m = B.Model(W)
    try:
        states = m.prefill_batch(reqs)
        gpu = m.decide_batch(states, [r.questions for r in reqs])
        o = om.Oracle(W, np.float32)
        refs = {}
        for i in (0, 5, 15):
            refs[i] = o.decide(reqs[i], branched=True)
            compare(gpu[i], refs[i], reqs[i].questions, f"small req {i}")
        # three requests (12 single-chunk questions x 8 heads: each head's value columns are
        # split over 2 CTAs in the output kernel)
        three = m.decide_batch(states[:3], [r.questions for r in reqs[:3]])
        compare(three[0], refs[0], reqs[0].questions, "small 3-request batch")
        # batched and one-at-a-time calls agree
        one = m.decide(m.prefill(reqs[5].tokens), reqs[5].questions)
        for a, b in zip(one, gpu[5]):
            assert np.abs(a["probs"] - b["probs"]).max() < 2e-3   # different M -> different GEMM split plan
    finally:
        m.close()


def test_norm_fused_into_splitk_reduction_bitexact(B, monkeypatch):
    """Decide calls (few rows: residual-add GEMMs split over K) form the following RMSNorm
    inside the split-K reduction; results are bit-identical to the separate norm launches and
    the call launches fewer kernels."""
    cfg = configs.SMALL
    W = synth.make_weights(cfg)
    req = synth.make_requests(cfg)[0]
    out = {}
    for fuse in ("1", "0"):
        monkeypatch.setenv("S1_NORM_FUSE", fuse)
        m = B.Model(W)
        try:
            st = m.prefill(req.tokens)
            m.decide(st, req.questions)              # first use of each GEMM shape
            n0 = m.counters()["launches"]
            res = m.decide(st, req.questions)
            out[fuse] = (res, m.counters()["launches"] - n0)
        finally:
            m.close()
    (a, la), (b, lb) = out["1"], out["0"]
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x["probs"], y["probs"])
        np.testing.assert_array_equal(x["hidden"], y["hidden"])
    # every norm that follows a K-split residual-add GEMM rides on its reduction: the MLP norm
    # after the out-projection, and the next layer's input norm after the down-projection (the
    # planner's split choice for these shapes, host logic)
    sh = cfg.shape
    R = sum(len(q.suffix) for q in req.questions)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    k_o = sh.la_heads * sh.la_dv
    split = lambda N, K: B.gemm_plan(R, N, K, 2, sms, False)["splits"] > 1
    fused = sh.n_layers * int(split(sh.d_model, k_o)) + (sh.n_layers - 1) * int(split(sh.d_model, sh.ffn))
    assert sh.fa_q_heads * sh.fa_head_dim == k_o
    assert fused > 0 and lb - la == fused, (la, lb, fused)


# -- one sweep over prefix + questions ---------------------------------------------------------
def test_tiny_fused_vs_oracle_and_two_call(tiny, tiny_weights, tiny_requests):
    r = tiny_requests[0]
    ref = om.Oracle(tiny_weights, np.float32).decide(r, branched=False)
    fused, st = tiny.prefill_decide(r, keep_state=True)
    compare(fused, ref, r.questions, "tiny fused")
    # the returned snapshot serves further decisions, and agrees with the two-call path
    again = tiny.decide(st, r.questions)
    two = tiny.decide(tiny.prefill(r.tokens), r.questions)
    for a, b, c in zip(fused, again, two):
        assert np.abs(a["probs"] - b["probs"]).max() < 2e-3
        assert np.abs(b["probs"] - c["probs"]).max() < 2e-3   # prefix GEMMs ran at a different M


def test_tiny_fused_edge_cases(tiny, tiny_weights):
    o = om.Oracle(tiny_weights, np.float32)
    g = np.random.default_rng(8)
    qs = [synth.random_question(g, 4096, configs.CHOICE, 1, 1), synth.random_question(g, 4096, configs.NOUL, 65, 2),
          synth.random_question(g, 4096, configs.SCORE, 130, 5)]
    for P in (1, 64, 129):
        toks = g.integers(16, 4096, size=P).astype(np.int32)
        req = synth.Request(toks, None, qs)
        gpu, _ = tiny.prefill_decide(req)
        _, caches, PP = o.prefill(toks)
        compare(gpu, o.decide_branched(caches, PP, qs), qs, f"fused edge P={P}")


def test_small_fused_batch_vs_oracle(B):
    cfg = configs.SMALL
    W = synth.make_weights(cfg)
    reqs = synth.make_requests(cfg)
    m = B.Model(W)
    try:
        gpu, _ = m.prefill_decide_batch(reqs)
    finally:
        m.close()
    o = om.Oracle(W, np.float32)
    for i in (0, 9, 15):
        compare(gpu[i], o.decide(reqs[i], branched=True), reqs[i].questions, f"small fused {i}")


# -- full-vocabulary option log-probabilities --------------------------------------------------
def test_tiny_lm_logprobs_vs_oracle(tiny, tiny_weights, tiny_requests):
    r = tiny_requests[0]
    st = tiny.prefill(r.tokens)
    gpu = tiny.decide(st, r.questions, want_lm=True)
    fused, _ = tiny.prefill_decide(r, want_lm=True)
    o = om.Oracle(tiny_weights, np.float32)
    ref = o.decide(r, branched=True)
    from scipy.special import logsumexp
    for g, f, rr, q in zip(gpu, fused, ref, r.questions):
        lp_ref, _ = o.option_lm_logprobs(rr["hidden"], q.option_ids)
        assert np.abs(g["lm_logprobs"] - lp_ref).max() < 5e-2
        assert np.abs(f["lm_logprobs"] - lp_ref).max() < 5e-2
        # renormalised over the options they give back the option probabilities
        np.testing.assert_allclose(np.exp(g["lm_logprobs"] - logsumexp(g["lm_logprobs"])), g["probs"], atol=1e-4)
        assert np.all(g["lm_logprobs"] < 0)


@pytest.mark.parametrize("vocab_pass", ["tensor", "simt"])
def test_small_lm_logprobs_vs_oracle_on_gpu_hidden(B, vocab_pass, monkeypatch):
    """The full-vocabulary pass on its own: 16 requests x 4 questions = 64 readout rows of the
    small model (V = 32000, bf16 embedding, so E is the same on both sides) in one batched
    call; the oracle's option_lm_logprobs applied to the GPU's own last hidden rows must match
    the GPU's log-probabilities to 2e-3. The tensor-core pass rounds the normalised rows to f16
    (relative 2^-11 per element: about 2e-4 on z at d = 1024); the CUDA-core pass is fp32."""
    if vocab_pass == "simt":
        monkeypatch.setenv("S1_VOCAB", "simt")
    else:
        monkeypatch.delenv("S1_VOCAB", raising=False)
    cfg = configs.SMALL
    W = synth.make_weights(cfg)
    reqs = synth.make_requests(cfg)
    m = B.Model(W)
    try:
        gpu, _ = m.prefill_decide_batch(reqs, want_lm=True)
    finally:
        m.close()
    o = om.Oracle(W, np.float64)
    worst = 0.0
    for r, res in zip(reqs, gpu):
        for q, g in zip(r.questions, res):
            lp_ref, _ = o.option_lm_logprobs(g["hidden"].astype(np.float64), q.option_ids)
            worst = max(worst, float(np.abs(g["lm_logprobs"] - lp_ref).max()))
    print(f"small lm_logprobs ({vocab_pass}): max |d| {worst:.2e} over 64 questions")
    assert worst < 2e-3


@pytest.mark.parametrize("vocab_pass", ["tensor", "simt"])
def test_tiny_lm_logprobs_many_rows(B, tiny_weights, tiny_requests, vocab_pass, monkeypatch):
    """150 questions over one prefix (150 readout rows: two 128-row tiles of the tensor-core
    pass, the second ragged) against the oracle on the GPU's own hidden rows."""
    if vocab_pass == "simt":
        monkeypatch.setenv("S1_VOCAB", "simt")
    else:
        monkeypatch.delenv("S1_VOCAB", raising=False)
    r = tiny_requests[0]
    qs = [q for _ in range(50) for q in r.questions]
    m = B.Model(tiny_weights)
    try:
        st = m.prefill(r.tokens)
        gpu = m.decide(st, qs, want_lm=True)
        st.close()
    finally:
        m.close()
    o = om.Oracle(tiny_weights, np.float64)
    worst = 0.0
    for q, g in zip(qs, gpu):
        lp_ref, _ = o.option_lm_logprobs(g["hidden"].astype(np.float64), q.option_ids)
        worst = max(worst, float(np.abs(g["lm_logprobs"] - lp_ref).max()))
    # identical questions give identical rows, wherever they sit among the 150
    for i in range(3, len(qs)):
        assert np.array_equal(gpu[i]["lm_logprobs"], gpu[i % 3]["lm_logprobs"])
    print(f"tiny lm_logprobs x150 ({vocab_pass}): max |d| {worst:.2e}")
    assert worst < 2e-3


def test_lm_logprobs_survive_chunk_state_growth(B, tiny_weights, tiny_requests):
    """Full-vocabulary log-probabilities stay correct after a longer prefix has grown the
    model's per-chunk state buffer between two calls (the buffers are reallocated separately)."""
    m = B.Model(tiny_weights)
    try:
        r = tiny_requests[0]
        first = m.decide(m.prefill(r.tokens), r.questions, want_lm=True)
        long_tokens = np.concatenate([r.tokens] * 8)            # many more chunks than before
        m.decide(m.prefill(long_tokens), r.questions, want_lm=True)
        again = m.decide(m.prefill(r.tokens), r.questions, want_lm=True)
        for a, b in zip(first, again):
            assert np.array_equal(a["lm_logprobs"], b["lm_logprobs"])
            assert np.array_equal(a["probs"], b["probs"])
    finally:
        m.close()


def test_graphs_replay_matches_eager(B, tiny_weights):
    """With CUDA graphs on, repeated stream-ordered one-sweep calls (the second captured, the
    rest replayed) give the eager call's results bit for bit, and a replay reads ids rewritten in
    the same device buffers (results follow the new ids)."""
    import ctypes as C
    s = torch.cuda.Stream()
    m = B.Model(tiny_weights, stream=s.cuda_stream)
    try:
        r0, r1 = synth.make_requests(configs.TINY, n_requests=2)
        assert len(r0.tokens) == len(r1.tokens)
        assert [(q.type, len(q.suffix), len(q.option_ids)) for q in r0.questions] == \
               [(q.type, len(q.suffix), len(q.option_ids)) for q in r1.questions]
        dt = torch.from_numpy(r0.tokens.copy()).cuda()
        qd = [(torch.from_numpy(q.suffix.copy()).cuda(), torch.from_numpy(q.option_ids.copy()).cuda(), q.type)
              for q in r0.questions]
        arr = (B.Question * len(qd))()
        for j, (su, op, t) in enumerate(qd):
            arr[j] = B.Question(t, C.cast(C.c_void_p(su.data_ptr()), C.POINTER(C.c_int32)), su.numel(),
                                C.cast(C.c_void_p(op.data_ptr()), C.POINTER(C.c_int32)), op.numel())
        n_opt = sum(len(q.option_ids) for q in r0.questions)
        probs = torch.zeros(n_opt, dtype=torch.float32, device="cuda")
        stats = torch.zeros((len(qd), 8), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        st = m.state_create(len(r0.tokens))

        def run():
            m.prefill_decide_async(st, dt.data_ptr(), len(r0.tokens), arr, len(qd), probs.data_ptr(), stats.data_ptr())
            m.sync()
            return probs.cpu().numpy().copy(), stats.cpu().numpy().copy()

        eager = run()                      # graphs off
        m.set_graphs(True)
        outs = [run() for _ in range(4)]   # eager, capture, replay, replay
        for p, sstat in outs:
            np.testing.assert_array_equal(p, eager[0])
            np.testing.assert_array_equal(sstat, eager[1])
        # new ids in the same buffers: the replay follows them and matches a graph-free call
        dt.copy_(torch.from_numpy(r1.tokens))
        for (su, op, _), q in zip(qd, r1.questions):
            su.copy_(torch.from_numpy(q.suffix))
            op.copy_(torch.from_numpy(q.option_ids))
        torch.cuda.synchronize()
        replay = run()
        m.set_graphs(False)
        fresh = run()
        np.testing.assert_array_equal(replay[0], fresh[0])
        np.testing.assert_array_equal(replay[1], fresh[1])
        assert not np.array_equal(replay[0], eager[0])
    finally:
        m.close()


@pytest.mark.gpu
def test_graphs_two_call_path(B, tiny_weights):
    """With CUDA graphs on, the stream-ordered prefill and decide calls (each captured on its
    second occurrence, then replayed) give the eager calls' results bit for bit; replays follow
    ids rewritten in the same device buffers, and a decide after a shorter prefill (another
    prefix length) does not replay the longer prefix's graph."""
    import ctypes as C
    s = torch.cuda.Stream()
    m = B.Model(tiny_weights, stream=s.cuda_stream)
    try:
        r0, r1 = synth.make_requests(configs.TINY, n_requests=2)
        P = len(r0.tokens)
        assert len(r1.tokens) == P
        dt = torch.from_numpy(r0.tokens.copy()).cuda()
        qd = [(torch.from_numpy(q.suffix.copy()).cuda(), torch.from_numpy(q.option_ids.copy()).cuda(), q.type)
              for q in r0.questions]
        arr = (B.Question * len(qd))()
        for j, (su, op, t) in enumerate(qd):
            arr[j] = B.Question(t, C.cast(C.c_void_p(su.data_ptr()), C.POINTER(C.c_int32)), su.numel(),
                                C.cast(C.c_void_p(op.data_ptr()), C.POINTER(C.c_int32)), op.numel())
        n_opt = sum(len(q.option_ids) for q in r0.questions)
        probs = torch.zeros(n_opt, dtype=torch.float32, device="cuda")
        stats = torch.zeros((len(qd), 8), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        st = m.state_create(P)

        def run(n=P):
            m.prefill_async(st, dt.data_ptr(), n)
            m.decide_async(st, arr, len(qd), probs.data_ptr(), stats.data_ptr())
            m.sync()
            return probs.cpu().numpy().copy(), stats.cpu().numpy().copy()

        eager = run()
        eager_short = run(P - 3)
        m.set_graphs(True)
        outs = [run() for _ in range(4)]     # eager, capture, replay, replay
        for p, sstat in outs:
            np.testing.assert_array_equal(p, eager[0])
            np.testing.assert_array_equal(sstat, eager[1])
        for _ in range(3):                   # another prefix length: its own graphs
            p, sstat = run(P - 3)
            np.testing.assert_array_equal(p, eager_short[0])
            np.testing.assert_array_equal(sstat, eager_short[1])
        dt.copy_(torch.from_numpy(r1.tokens))
        for (su, op, _), q in zip(qd, r1.questions):
            su.copy_(torch.from_numpy(q.suffix))
            op.copy_(torch.from_numpy(q.option_ids))
        torch.cuda.synchronize()
        replay = run()
        m.set_graphs(False)
        fresh = run()
        np.testing.assert_array_equal(replay[0], fresh[0])
        np.testing.assert_array_equal(replay[1], fresh[1])
        assert not np.array_equal(replay[0], eager[0])
    finally:
        m.close()


# -- the gated delta rule's short convolution (its history continues the snapshot) -------------
def _conv_config(base, width=4):
    import dataclasses
    shape = dataclasses.replace(base.shape, conv_width=width)
    return configs.Config(base.name + "-conv", base.seed + 100, shape, base.work)


def test_tiny_conv_vs_oracle(B):
    """Tiny model with a width-4 short convolution: the two-call path against the plain
    unbranched oracle, then the one-sweep call with suffixes shorter than the history (1 and 2
    rows), a 130-row suffix and prefixes of 1, 2 and 200 rows against the branched oracle."""
    cfg = _conv_config(configs.TINY)
    W = synth.make_weights(cfg)
    req = synth.make_requests(cfg)[0]
    o = om.Oracle(W, np.float32)
    m = B.Model(W)
    try:
        st = m.prefill(req.tokens)
        compare(m.decide(st, req.questions), o.decide(req, branched=False), req.questions, "tiny conv")
        g = np.random.default_rng(9)
        qs = [synth.random_question(g, 4096, configs.CHOICE, 1, 3), synth.random_question(g, 4096, configs.NOUL, 2, 2),
              synth.random_question(g, 4096, configs.SCORE, 130, 5)]
        for P in (1, 2, 200):
            toks = g.integers(16, 4096, size=P).astype(np.int32)
            _, caches, PP = o.prefill(toks)
            ref = o.decide_branched(caches, PP, qs)
            fused, st2 = m.prefill_decide(synth.Request(toks, None, qs), keep_state=True)
            compare(fused, ref, qs, f"tiny conv fused P={P}")
            # the kept snapshot carries the convolution history into later questions
            compare(m.decide(st2, qs), ref, qs, f"tiny conv decide over snapshot P={P}")
    finally:
        m.close()


def test_small_conv_batch_vs_oracle(B):
    """Small model (8 layers, LoRA) with a width-4 short convolution: batched prefill and decide,
    and the batched one-sweep call, against the oracle on three requests."""
    cfg = _conv_config(configs.SMALL)
    W = synth.make_weights(cfg)
    reqs = synth.make_requests(cfg, n_requests=4)
    m = B.Model(W)
    try:
        states = m.prefill_batch(reqs)
        gpu = m.decide_batch(states, [r.questions for r in reqs])
        fused, _ = m.prefill_decide_batch(reqs)
    finally:
        m.close()
    o = om.Oracle(W, np.float32)
    for i in (0, 3):
        ref = o.decide(reqs[i], branched=True)
        compare(gpu[i], ref, reqs[i].questions, f"small conv {i}")
        compare(fused[i], ref, reqs[i].questions, f"small conv fused {i}")


def test_batch_async_one_sweep_matches_blocking_call(B):
    """s1_prefill_decide_batch_async (device ids, stream-ordered, into states from
    s1_state_create) gives the blocking s1_prefill_decide_batch's results bit for bit, also when
    replayed as a CUDA graph."""
    import ctypes as C
    cfg = configs.SMALL
    W = synth.make_weights(cfg)
    reqs = synth.make_requests(cfg, n_requests=3)
    s = torch.cuda.Stream()
    m = B.Model(W, stream=s.cuda_stream)
    try:
        ref, _ = m.prefill_decide_batch(reqs)
        states = [m.state_create(len(r.tokens)) for r in reqs]
        keep, qarrs = [], []
        for r in reqs:
            dq = [(torch.from_numpy(q.suffix.copy()).cuda(), torch.from_numpy(q.option_ids.copy()).cuda(), q.type)
                  for q in r.questions]
            keep += dq
            arr = (B.Question * len(dq))()
            for j, (su, op, t) in enumerate(dq):
                arr[j] = B.Question(t, C.cast(C.c_void_p(su.data_ptr()), C.POINTER(C.c_int32)), su.numel(),
                                    C.cast(C.c_void_p(op.data_ptr()), C.POINTER(C.c_int32)), op.numel())
            qarrs.append(arr)
        toks = [torch.from_numpy(r.tokens.copy()).cuda() for r in reqs]
        n_opt = sum(len(q.option_ids) for r in reqs for q in r.questions)
        n_q = [len(r.questions) for r in reqs]
        probs = torch.zeros(n_opt, dtype=torch.float32, device="cuda")
        stats = torch.zeros((sum(n_q), 8), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        m.set_graphs(True)
        for rep in range(3):   # eager, capture, replay
            m.prefill_decide_batch_async(states, [t.data_ptr() for t in toks], [len(r.tokens) for r in reqs], qarrs,
                                         n_q, probs.data_ptr(), stats.data_ptr())
            m.sync()
            p = probs.cpu().numpy()
            off = 0
            for r, res in zip(reqs, ref):
                for q, x in zip(r.questions, res):
                    np.testing.assert_array_equal(p[off:off + len(q.option_ids)], x["probs"])
                    off += len(q.option_ids)
        m.set_graphs(False)
        assert all(st.rows == len(r.tokens) for st, r in zip(states, reqs))
    finally:
        m.close()
