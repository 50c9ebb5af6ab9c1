"""Host-side prefix split of whole per-question token streams (no GPU): the result is checked
against a brute-force longest common prefix."""
import numpy as np
import pytest

from prefill_only_decision_gb300 import build


@pytest.fixture(scope="module")
def B():
    build.build()
    from prefill_only_decision_gb300 import binding
    return binding


def brute(streams, min_suffix, align):
    cap = min(len(s) for s in streams) - min_suffix
    P = 0
    while P < cap and all(s[P] == streams[0][P] for s in streams):
        P += 1
    if align > 1:
        P -= P % align
    return P


def test_split_random(B):
    g = np.random.default_rng(0)
    for trial in range(200):
        n = int(g.integers(1, 6))
        base = g.integers(0, 5, size=int(g.integers(1, 300)))
        streams = []
        for _ in range(n):
            cut = int(g.integers(0, len(base) + 1))
            tail = g.integers(0, 5, size=int(g.integers(1, 40)))
            streams.append(np.concatenate([base[:cut], tail]).astype(np.int32))
        for ms, al in ((1, 0), (1, 64), (3, 16)):
            if min(len(s) for s in streams) < ms:
                continue
            assert B.split_prefix(streams, ms, al) == brute(streams, ms, al)


def test_split_keeps_a_suffix_and_rejects_bad_input(B):
    same = [np.arange(10, dtype=np.int32)] * 3
    assert B.split_prefix(same) == 9            # identical streams: one token left for each suffix
    assert B.split_prefix(same, 1, 4) == 8
    with pytest.raises(B.S1Error):
        B.split_prefix(same, min_suffix=11)
    with pytest.raises(B.S1Error):
        B.split_prefix([], 1, 0)
