"""The C-ABI library builds, loads and exports every symbol include/*.h declares; host-side
validation paths that return before any device work (CPU only, no GPU needed)."""
import ctypes as C
import os
import re

import numpy as np
import pytest

from prefill_only_decision_gb300 import build, configs, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    from prefill_only_decision_gb300 import binding
    return binding.lib()


def declared_functions():
    names = set()
    for h in ("s1.h", "s1_ops.h"):
        txt = open(os.path.join(ROOT, "include", h)).read()
        txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?(?:int|void|char|int32_t)\s*\*?\s*(s1_\w+)\s*\(", txt, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 20, names
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing


def test_version_and_error_strings(L):
    assert b"sm_103a" in L.s1_version()
    assert isinstance(L.s1_last_error(), bytes)


def test_allocator_hooks_must_pair(L):
    from prefill_only_decision_gb300 import binding
    rc = L.s1_set_allocator(C.c_void_p(1), None, None)
    assert rc == binding.S1_ERR_INVALID_ARG
    assert b"both" in L.s1_last_error()
    assert L.s1_set_allocator(None, None, None) == 0


def _shape(**kw):
    from prefill_only_decision_gb300 import binding
    s = configs.TINY.shape
    full = np.array(s.layer_is_full, dtype=np.uint8)
    d = dict(vocab=s.vocab, d_model=s.d_model, n_layers=s.n_layers, ffn=s.ffn, la_heads=s.la_heads, la_dk=s.la_dk,
             la_dv=s.la_dv, fa_q_heads=s.fa_q_heads, fa_kv_heads=s.fa_kv_heads, fa_head_dim=s.fa_head_dim,
             rope_theta=1e6, rms_eps=1e-6, l2_eps=1e-6, lora_rank=0, lora_alpha=0.0, weight_dtype=0, max_rows=0)
    d.update(kw)
    sh = binding.Shape(**{k: v for k, v in d.items()})
    sh.layer_is_full = full.ctypes.data_as(C.POINTER(C.c_uint8))
    return sh, full


@pytest.mark.parametrize("bad,code", [
    (dict(d_model=200), 1),            # not a multiple of 64
    (dict(ffn=-1), 1),
    (dict(weight_dtype=7), 1),
    (dict(la_dk=64, la_dv=128), 7),    # unsupported head geometry
    (dict(fa_q_heads=3, fa_kv_heads=2), 7),
    (dict(la_dk=96, la_dv=96), 7),
])
def test_shape_validation_before_device_work(L, bad, code):
    from prefill_only_decision_gb300 import binding
    sh, keep = _shape(**bad)
    w = binding.Weights(None, None, None, None, None)
    h = C.c_void_p()
    rc = L.s1_model_create(C.byref(sh), C.byref(w), C.byref(h))
    assert rc == code, L.s1_last_error()
    assert not h.value


def test_invalid_handles_rejected(L):
    from prefill_only_decision_gb300 import binding
    assert L.s1_state_rows(None) == -1
    assert L.s1_sync(None) == binding.S1_ERR_INVALID_HANDLE
    assert L.s1_set_stream(None, None) == binding.S1_ERR_INVALID_HANDLE
    junk = (C.c_uint32 * 64)()
    assert L.s1_sync(C.cast(junk, C.c_void_p)) == binding.S1_ERR_INVALID_HANDLE
    L.s1_state_destroy(None)
    L.s1_model_destroy(None)


def test_ops_argument_validation(L):
    from prefill_only_decision_gb300 import binding
    assert L.s1_op_gemm(None, None, 4, 30, 64, 0, None, 30, 1, None) == binding.S1_ERR_INVALID_ARG   # N % 32
    assert L.s1_op_gemm(None, None, 4, 32, 60, 0, None, 32, 1, None) == binding.S1_ERR_INVALID_ARG   # K % 64
    assert L.s1_op_rmsnorm(None, None, 4, 30, 1e-6, None, None) == binding.S1_ERR_INVALID_ARG


def test_short_convolution_width_is_validated(L):
    """The gated delta-rule short convolution takes widths 0 (none) to 8; a wider one is refused
    with INVALID_ARG before any device work."""
    from prefill_only_decision_gb300 import binding
    shape = configs.ModelShape(vocab=300, d_model=64, n_layers=4, ffn=64, la_heads=1, la_dk=64, la_dv=64,
                               fa_q_heads=1, fa_kv_heads=1, fa_head_dim=64, bf16_weights=False, conv_width=9)
    W = synth.make_weights(configs.Config("conv", 0, shape, configs.TINY.work))
    with pytest.raises(binding.S1Error) as e:
        binding.Model(W)
    assert e.value.code == binding.S1_ERR_INVALID_ARG
