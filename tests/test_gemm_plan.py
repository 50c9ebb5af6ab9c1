"""The GEMM planner (host logic, no GPU): every plan it picks over a sweep of shapes launches
only well-formed work — tiles cover the output exactly once, every K split gets at least one
k-block (and at least four when K is split), split-K partials fit the workspace, SwiGLU tiles
hold whole gate/up groups, no weight tile is shared across a cluster — and the few-row decide
shapes get the K-split plans the launch profiles show."""
import pytest

from prefill_only_decision_gb300 import build

BM, BK, SMS = 128, 64, 152
SINGLE = {128, 144, 176, 192, 208, 256}
PAIR = {128, 176, 192, 208, 256}
EPI_F32, EPI_BF16, EPI_RESADD, EPI_SWIGLU = 0, 1, 2, 3


@pytest.fixture(scope="module")
def plan():
    build.build()
    from prefill_only_decision_gb300 import binding

    def run(M, N, K, epi, pair=0, sms=SMS):
        try:
            return 0, binding.gemm_plan(M, N, K, epi, sms, bool(pair))
        except binding.S1Error as e:
            return e.code, None

    return run


MS = [1, 16, 63, 64, 65, 127, 128, 129, 144, 255, 256, 300, 512, 777, 1024, 1168, 1600, 2048, 4096, 10240]
NS = [32, 96, 256, 1056, 2560, 3072, 5120, 6176, 7168, 12352, 18432, 34816]
KS = [64, 128, 1024, 2560, 4096, 5120, 9216, 17408]


@pytest.mark.parametrize("epi", [EPI_F32, EPI_BF16, EPI_RESADD, EPI_SWIGLU])
def test_single_cta_plans_are_well_formed(plan, epi):
    ws_cap = 2 * SMS * BM * 256
    for M in MS:
        for N in NS:
            for K in KS:
                rc, p = plan(M, N, K, epi)
                assert rc == 0, (M, N, K, epi)
                bn, cm, kb = p["bn"], p["cm"], K // BK
                # 176/208: autotuner or pinned only, except in the few-row (<= 2 m tiles) model
                assert p["pair"] == 0 and bn in (SINGLE if M <= 2 * BM else SINGLE - {176, 208}), p
                assert p["m_tiles"] == -(-M // BM) and p["n_tiles"] == -(-N // bn), (M, N, K, p)
                assert cm == 1, p
                if epi == EPI_SWIGLU:
                    assert bn % 32 == 0, p
                s, kbp = p["splits"], p["kbp"]
                assert s >= 1 and s * kbp >= kb and (s - 1) * kbp < kb, (M, N, K, p)
                if s > 1:
                    assert kbp >= 4 and s * p["m_tiles"] * BM * N <= ws_cap, (M, N, K, p)
                else:
                    assert kbp == kb


@pytest.mark.parametrize("epi", [EPI_F32, EPI_RESADD, EPI_SWIGLU])
def test_pair_plans_are_well_formed(plan, epi):
    for M in MS:
        for N in NS:
            for K in (64, 2560, 9216):
                rc, p = plan(M, N, K, epi, pair=1)
                assert rc == 0
                bn = p["bn"]
                assert p["pair"] == 1 and bn in PAIR and p["splits"] == 1 and p["kbp"] == K // BK, p
                assert p["m_tiles"] == 2 * -(-M // (2 * BM)) and p["n_tiles"] == -(-N // bn), (M, N, p)
                if epi == EPI_SWIGLU:
                    assert bn % 32 == 0, p


def test_decide_shapes_split_k(plan):
    """64 rows (one question of the 27B-class model): the weight-streaming projections get the
    plans that measured fastest (cold caches, reduction included) in a sweep of tile widths
    128..256 and splits 1..8 — K split where few n tiles would leave SMs idle, none where about
    two thirds of the SMs already stream a tile each — and fill at most one wave."""
    # down / out-projections (residual add), GDN in-projection, attention q/k/v
    for (N, K, epi, bn, splits) in [(5120, 17408, EPI_RESADD, 144, 4), (5120, 4096, EPI_RESADD, 128, 3),
                                    (12352, 5120, EPI_F32, 128, 1), (7168, 5120, EPI_F32, 144, 3)]:
        rc, p = plan(64, N, K, epi)
        assert rc == 0 and (p["bn"], p["splits"]) == (bn, splits), (N, K, p)
        assert p["n_tiles"] * p["splits"] <= SMS < p["n_tiles"] * (p["splits"] + 1), p   # one wave, filled


def test_bad_arguments(plan):
    for args in [(0, 256, 64, 0), (64, 100, 64, 0), (64, 256, 100, 0), (64, 256, 64, 4), (64, 256, 64, -1)]:
        assert plan(*args)[0] != 0, args
    assert plan(64, 256, 64, 0, sms=0)[0] != 0
