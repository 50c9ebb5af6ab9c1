"""The GEMM entry point that allocates nothing (s1_op_gemm_noalloc).

It is meant for callers that cannot call cudaMalloc at call time (memory owned by another
framework, real-time loops that must not allocate, fixed memory budgets): its split-K
partials and error word live in fixed device arrays inside the library. These checks call it
through the C ABI and compare it with the allocating entry point s1_op_gemm, on two calls in a
row (the shared arrays keep the previous call's contents). Collected last on purpose.
"""
import ctypes as C

import numpy as np
import pytest


pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from prefill_only_decision_gb300 import binding
    lib = binding.lib()
    f = lib.s1_op_gemm_noalloc
    f.restype = C.c_int
    f.argtypes = [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_int32,
                  C.c_void_p]
    return lib


def _f16(a):
    return torch.from_numpy(np.asarray(a, np.float32).astype(np.float16)).cuda()


# (M, N, K, epilogue): includes split-K plans (small M) and the SwiGLU / residual epilogues
SHAPES = [(144, 2560, 9216, 2), (144, 2560, 2560, 0), (1024, 2560, 2560, 0), (100, 544, 320, 1),
          (144, 18432, 2560, 3), (64, 1024, 1024, 2)]


@pytest.mark.parametrize("M,N,K,epi", SHAPES)
def test_noalloc_gemm_matches_allocating_entry_point(L, M, N, K, epi):
    from prefill_only_decision_gb300 import binding
    g = np.random.default_rng(M + N + K + epi)
    X = _f16(g.standard_normal((M, K)))
    W = _f16(0.05 * g.standard_normal((N, K)))
    ncol = N // 2 if epi == 3 else N
    dt = torch.float16 if epi in (1, 3) else torch.float32
    base = torch.from_numpy(g.standard_normal((M, ncol)).astype(np.float32)).cuda() if epi == 2 else None

    def fresh():
        return base.clone() if base is not None else torch.zeros((M, ncol), dtype=dt, device="cuda")

    ref = fresh()
    binding.op_gemm(X.data_ptr(), W.data_ptr(), M, N, K, epi, ref.data_ptr(), ncol, 0)
    torch.cuda.synchronize()
    refn = ref.float().cpu().numpy()
    scale = np.sqrt(K) * 0.05
    tol = 1e-4 * scale + (np.abs(refn) * 2.0 ** -10 if epi in (1, 3) else 0)

    def call(out):
        rc = L.s1_op_gemm_noalloc(C.c_void_p(X.data_ptr()), C.c_void_p(W.data_ptr()), M, N, K, epi,
                                  C.c_void_p(out.data_ptr()), ncol, None)
        assert rc == 0, L.s1_last_error()

    call(fresh())                 # first call on this device: looks up the arrays' addresses
    outs = [fresh(), fresh()]     # every output buffer exists before device memory is read
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for out in outs:              # two calls in a row: the fixed scratch keeps the previous call's contents
        call(out)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0, "the call changed the device's free memory"
    for out in outs:
        got = out.float().cpu().numpy()
        assert np.all(np.abs(got - refn) <= tol), np.abs(got - refn).max()


def _oversized_shape(sms):
    """A shape whose planned split-K partials exceed the fixed array on a GPU of `sms` SMs (the
    planner is host logic, so the search needs no device work), or None."""
    from prefill_only_decision_gb300 import binding
    cap = binding.S1_NOALLOC_WS_FLOATS
    for N in (256, 512, 1024, 2048):
        for mt in range(1, 4 * sms):
            M = 128 * mt
            p = binding.gemm_plan(M, N, 8192, 0, sms, False)
            if p["splits"] > 1 and p["splits"] * p["m_tiles"] * 128 * N > cap:
                return M, N, 8192
    return None


def test_noalloc_gemm_rejects_oversized_scratch(L):
    """A plan whose split-K partials exceed the fixed array is refused before any device work."""
    from prefill_only_decision_gb300 import binding
    shp = _oversized_shape(torch.cuda.get_device_properties(0).multi_processor_count)
    if shp is None:
        pytest.skip("no split-K plan on this GPU needs more scratch than the fixed array holds")
    M, N, K = shp
    X = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    W = torch.zeros((N, K), dtype=torch.float16, device="cuda")
    out = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    rc = L.s1_op_gemm_noalloc(C.c_void_p(X.data_ptr()), C.c_void_p(W.data_ptr()), M, N, K, 0,
                              C.c_void_p(out.data_ptr()), N, None)
    assert rc == binding.S1_ERR_BUDGET
    assert b"split-K scratch" in L.s1_last_error()
    assert torch.all(out == 7.0)
    # bad arguments are refused as well
    rc = L.s1_op_gemm_noalloc(C.c_void_p(X.data_ptr()), C.c_void_p(W.data_ptr()), M, 30, K, 0,
                              C.c_void_p(out.data_ptr()), N, None)
    assert rc == binding.S1_ERR_INVALID_ARG
