"""Kernel-level parity on the GPU, through the C ABI (s1_ops.h), against the oracle's
definitions evaluated on the CPU in float64 on the same (f16-rounded) inputs: every tensor-core
operand of the library is f16."""
import os

import numpy as np
import pytest

from oracle import gdn as ogdn
from oracle import model as om
from prefill_only_decision_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from prefill_only_decision_gb300 import binding
    binding.lib()
    return binding


def f16_round(a):
    """Round to the nearest f16 value (ties to even), returned as float32."""
    return np.asarray(a, np.float32).astype(np.float16).astype(np.float32)


def to_dev_f16(a):
    return torch.from_numpy(np.asarray(a, np.float32).astype(np.float16)).cuda()


def from_dev_f16(t):
    return t.float().cpu().numpy()


def swiglu_pack(Wg, Wu):
    """Interleave gate/up rows in blocks of 16 (the library's packed MLP layout)."""
    F, d = Wg.shape
    P = np.empty((2 * F, d), Wg.dtype)
    for b in range(F // 16):
        P[32 * b: 32 * b + 16] = Wg[16 * b: 16 * b + 16]
        P[32 * b + 16: 32 * b + 32] = Wu[16 * b: 16 * b + 16]
    return P


GEMM_SHAPES = [(1, 32, 64), (100, 160, 128), (128, 256, 256), (300, 544, 320), (1024, 2560, 2560),
               (144, 2560, 9216), (1024, 6176, 2560), (144, 18432, 2560), (77, 2048, 1024),
               (1168, 2560, 9216), (1168, 3072, 2560), (257, 1056, 1024)]


_NO_TC = pytest.mark.skipif(bool(os.environ.get("S1_TEST_NO_TC")), reason="tensor-core path disabled")
IMPLS = [pytest.param(0, id="tc", marks=_NO_TC),
         pytest.param(2, id="tc_pair", marks=_NO_TC),     # CTA-pair tiles (tcgen05 cta_group::2)
         pytest.param(3, id="tc_single", marks=_NO_TC),   # single-CTA tiles
         pytest.param(1, id="simt")]


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
@pytest.mark.parametrize("epi", [0, 1, 2])
def test_gemm(B, impl, M, N, K, epi):
    if impl == 1 and M * N * K > 2e9:
        pytest.skip("SIMT reference only on small shapes")
    g = np.random.default_rng(M * 7 + N * 3 + K + epi)
    X = f16_round(g.standard_normal((M, K)))
    W = f16_round(g.standard_normal((N, K)) * 0.05)
    ref = X.astype(np.float64) @ W.astype(np.float64).T
    dX, dW = to_dev_f16(X), to_dev_f16(W)
    if epi == 1:
        out = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    else:
        base = g.standard_normal((M, N)).astype(np.float32) if epi == 2 else np.zeros((M, N), np.float32)
        out = torch.from_numpy(base).cuda()
        ref = ref + base
    B.op_gemm(dX.data_ptr(), dW.data_ptr(), M, N, K, epi, out.data_ptr(), N, impl)
    got = from_dev_f16(out) if epi == 1 else out.cpu().numpy()
    scale = np.sqrt(K) * 0.05
    tol = 1e-5 * scale + (np.abs(ref) * 2.0 ** -10 if epi == 1 else 0)
    err = np.abs(got - ref)
    assert np.all(err <= tol + 1e-4 * scale), (err.max(), np.unravel_index(err.argmax(), err.shape))


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("M,F,K", [(5, 64, 64), (200, 768, 256), (1024, 9216, 2560), (144, 9216, 2560),
                                   (1168, 9216, 2560)])
def test_gemm_swiglu(B, impl, M, F, K):
    if impl == 1 and M * F * K > 2e9:
        pytest.skip("SIMT reference only on small shapes")
    g = np.random.default_rng(M + F + K)
    X = f16_round(g.standard_normal((M, K)))
    Wg = f16_round(g.standard_normal((F, K)) * 0.03)
    Wu = f16_round(g.standard_normal((F, K)) * 0.03)
    Xd = X.astype(np.float64)
    gt, up = Xd @ Wg.T.astype(np.float64), Xd @ Wu.T.astype(np.float64)
    ref = om.silu(gt) * up
    out = torch.zeros((M, F), dtype=torch.float16, device="cuda")
    dX, dW = to_dev_f16(X), to_dev_f16(swiglu_pack(Wg, Wu))   # keep the device buffers alive
    B.op_gemm(dX.data_ptr(), dW.data_ptr(), M, 2 * F, K, 3, out.data_ptr(), F, impl)
    got = from_dev_f16(out)
    err = np.abs(got - ref)
    assert np.all(err <= np.abs(ref) * 2.0 ** -10 + 1e-4), err.max()


@pytest.mark.skipif(bool(os.environ.get("S1_TEST_NO_TC")), reason="tensor-core path disabled")
def test_gemm_row_invariance(B):
    """Rows computed at different M agree (same K order per row)."""
    g = np.random.default_rng(5)
    K, N = 2560, 2560
    X = f16_round(g.standard_normal((1168, K)))
    W = f16_round(g.standard_normal((N, K)) * 0.05)
    dX, dW = to_dev_f16(X), to_dev_f16(W)
    outs = []
    for M in (64, 1168):
        o = torch.zeros((M, N), dtype=torch.float32, device="cuda")
        B.op_gemm(dX.data_ptr(), dW.data_ptr(), M, N, K, 0, o.data_ptr(), N, 0)
        outs.append(o.cpu().numpy())
    err = np.abs(outs[0] - outs[1][:64])
    assert err.max() <= 1e-5 * np.abs(outs[1][:64]).max()


@_NO_TC
@pytest.mark.parametrize("M,N,K", [(1168, 2560, 2048), (300, 18432, 256)])
def test_gemm_pair_matches_single(B, M, N, K):
    """CTA-pair and single-CTA tiles accumulate every output over K in the same order."""
    g = np.random.default_rng(M + N + K)
    dX = to_dev_f16(f16_round(g.standard_normal((M, K))))
    dW = to_dev_f16(f16_round(g.standard_normal((N, K)) * 0.05))
    outs = []
    for impl in (2, 3):
        o = torch.zeros((M, N), dtype=torch.float32, device="cuda")
        B.op_gemm(dX.data_ptr(), dW.data_ptr(), M, N, K, 0, o.data_ptr(), N, impl)
        outs.append(o.cpu().numpy())
    err = np.abs(outs[0] - outs[1])
    print(f"[pair vs single {M}x{N}x{K}] max |diff| {err.max():.3e}, identical: {bool((err == 0).all())}")
    assert err.max() <= 1e-6 * np.abs(outs[1]).max()


def test_rmsnorm(B):
    g = np.random.default_rng(1)
    x = (g.standard_normal((37, 2560)) * 3).astype(np.float32)
    w = (1 + 0.1 * g.standard_normal(2560)).astype(np.float32)
    out = torch.zeros((37, 2560), dtype=torch.float16, device="cuda")
    dx, dw = torch.from_numpy(x).cuda(), torch.from_numpy(w).cuda()
    B.op_rmsnorm(dx.data_ptr(), dw.data_ptr(), 37, 2560, 1e-6, out.data_ptr())
    ref = om.rmsnorm(x.astype(np.float64), w.astype(np.float64), 1e-6)
    np.testing.assert_allclose(from_dev_f16(out), ref, rtol=2.0 ** -10, atol=1e-6)


def _gdn_inputs(R, H, D, seed):
    g = np.random.default_rng(seed)
    ld = 3 * H * D + 2 * H
    proj = g.standard_normal((R, ld)).astype(np.float32)
    return proj


# (chunks x heads) picks how many CTAs share a head's value columns in the output kernel: 4 below
# about half the SM count, 2 below the SM count (16 heads x 5 chunks), else 1 (16 x 10); the
# state pass keeps two chunk tiles in flight (two CTAs per SM) once its CTAs (sequences x heads x
# D / 16) exceed the SM count (the last two shapes: 384 and 192 CTAs of several chunk steps)
@pytest.mark.parametrize("H,D,lens,with_s0", [(2, 64, [1, 63, 64, 65], False), (4, 128, [130], True),
                                              (16, 128, [48, 48, 48], True), (3, 128, [200, 7], False),
                                              (16, 128, [320], True), (16, 64, [640], False),
                                              (16, 128, [200, 300, 130], True), (16, 64, [300, 300, 300], False)])
def test_gdn_scan(B, H, D, lens, with_s0):
    R = int(sum(lens))
    proj = _gdn_inputs(R, H, D, R + H)
    row0 = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int32)
    g = np.random.default_rng(3)
    S0 = (0.3 * g.standard_normal((len(lens), H, D, D))).astype(np.float32) if with_s0 else None
    dproj = torch.from_numpy(proj.copy()).cuda()
    dS0 = torch.from_numpy(S0).cuda() if with_s0 else None
    dSo = torch.zeros((len(lens), H, D, D), dtype=torch.float32, device="cuda")
    out = torch.zeros((R, H * D), dtype=torch.float16, device="cuda")
    B.op_gdn(dproj.data_ptr(), R, H, D, D, 1e-6, row0, lens, dS0.data_ptr() if with_s0 else 0, dSo.data_ptr(),
             out.data_ptr())
    got = from_dev_f16(out)
    gotS = dSo.cpu().numpy()
    P = proj.astype(np.float64)
    HD = H * D
    for s, (r0, n) in enumerate(zip(row0, lens)):
        rows = P[r0:r0 + n]
        q = ogdn.l2norm(rows[:, :HD].reshape(n, H, D), 1e-6)
        k = ogdn.l2norm(rows[:, HD:2 * HD].reshape(n, H, D), 1e-6)
        v = rows[:, 2 * HD:3 * HD].reshape(n, H, D)
        al, be = ogdn.gates(rows[:, 3 * HD:3 * HD + H], rows[:, 3 * HD + H:])
        s0 = S0[s].astype(np.float64) if with_s0 else np.zeros((H, D, D))
        o, S = ogdn.recurrent(q, k, v, al, be, s0)
        o = o.reshape(n, HD)
        # (the chunked form's products take TF32 inputs: its error, not the f16 output rounding,
        # sets this bound)
        assert np.abs(got[r0:r0 + n] - o).max() <= 2.0 ** -8 * np.abs(o).max() + 1e-4
        # state products run on TF32 inputs (10-bit mantissa) with fp32 accumulation
        np.testing.assert_allclose(gotS[s], S, atol=3e-3 * max(1.0, np.abs(S).max()))


# shapes: a causal prefix, ragged sequences, questions over a 1024-row snapshot, a snapshot whose
# rows end mid-tile, and few query tiles over long key ranges (key tiles split over a cluster)
# (the suffix-over-prefix shapes with few query tiles split their key ranges over clusters of
# 2 or 4 CTAs: 40 x 8 x 128 over 1536 cached rows is the 27B decide's attention layer)
ATTN_SHAPES = [(4, 2, 64, 0, [96]), (16, 4, 128, 0, [300, 17]), (16, 4, 128, 1024, [48, 48, 48]),
               (8, 2, 128, 77, [1, 5, 33]), (8, 2, 128, 1536, [64]), (40, 8, 128, 600, [64, 130]),
               (4, 2, 64, 300, [200]), (40, 8, 128, 1536, [64]), (48, 8, 64, 1100, [64])]


@pytest.mark.parametrize("kernel", ["tcgen05", "sync"])
@pytest.mark.parametrize("Hq,Hkv,hd,P,lens", ATTN_SHAPES)
def test_attention(B, Hq, Hkv, hd, P, lens, kernel, monkeypatch):
    """Both attention kernels (tcgen05 / TMEM / TMA, and the mma.sync one kept for debugging)
    against softmax(QK^T)V by brute force."""
    if kernel == "sync":
        monkeypatch.setenv("S1_ATTN", "sync")
    g = np.random.default_rng(P + Hq)
    R = int(sum(lens))
    q = f16_round(g.standard_normal((R, Hq, hd)))
    kn = f16_round(g.standard_normal((R, Hkv, hd)))
    vn = f16_round(g.standard_normal((R, Hkv, hd)))
    kc = f16_round(g.standard_normal((P, Hkv, hd)))
    vc = f16_round(g.standard_normal((P, Hkv, hd)))
    row0 = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int32)
    kv = to_dev_f16(np.stack([kc, vc])) if P else None
    out = torch.zeros((R, Hq * hd), dtype=torch.float16, device="cuda")
    dq, dk, dv = to_dev_f16(q), to_dev_f16(kn), to_dev_f16(vn)
    B.op_attention(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), kv.data_ptr() if P else 0, P, row0, lens, Hq, Hkv,
                   hd, out.data_ptr())
    got = from_dev_f16(out).reshape(R, Hq, hd)
    for r0, n in zip(row0, lens):
        K = np.concatenate([kc, kn[r0:r0 + n]]).astype(np.float64)
        V = np.concatenate([vc, vn[r0:r0 + n]]).astype(np.float64)
        ref = om.attention(q[r0:r0 + n].astype(np.float64), K, V, P + np.arange(n), np.arange(P + n))
        assert np.abs(got[r0:r0 + n] - ref).max() <= 2.0 ** -9 * np.abs(ref).max() + 2e-3


@_NO_TC
@pytest.mark.parametrize("bn", [256, 208, 192, 176, 144, 128])
@pytest.mark.parametrize("impl", [2, 3])
@pytest.mark.parametrize("M,N,K,epi", [(1168, 2560, 2048, 2), (300, 6176, 256, 0), (77, 3072, 512, 1)])
def test_gemm_tile_widths(B, bn, impl, M, N, K, epi, monkeypatch):
    """Every tile width of the single-CTA and CTA-pair kernels (S1_GEMM_BN pins the planner's choice)."""
    if impl == 2 and bn == 144:
        pytest.skip("no CTA-pair kernel of width 144")
    monkeypatch.setenv("S1_GEMM_BN", str(bn))
    g = np.random.default_rng(M + N + K + bn)
    X = f16_round(g.standard_normal((M, K)))
    W = f16_round(g.standard_normal((N, K)) * 0.05)
    ref = X.astype(np.float64) @ W.astype(np.float64).T
    dX, dW = to_dev_f16(X), to_dev_f16(W)
    if epi == 1:
        out = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    else:
        base = g.standard_normal((M, N)).astype(np.float32) if epi == 2 else np.zeros((M, N), np.float32)
        out = torch.from_numpy(base).cuda()
        ref = ref + base
    B.op_gemm(dX.data_ptr(), dW.data_ptr(), M, N, K, epi, out.data_ptr(), N, impl)
    got = from_dev_f16(out) if epi == 1 else out.cpu().numpy()
    scale = np.sqrt(K) * 0.05
    tol = 1e-5 * scale + (np.abs(ref) * 2.0 ** -10 if epi == 1 else 0)
    err = np.abs(got - ref)
    assert np.all(err <= tol + 1e-4 * scale), (bn, impl, err.max())
