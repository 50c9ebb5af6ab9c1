"""ctypes binding of libs1.so: argument marshalling only, every step runs in the library.

Loads the in-tree library (built by `prefill_only_decision_gb300.build`); a missing library
is an error, there is no other implementation to fall back on.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import List, Optional, Sequence

import numpy as np

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libs1.so")

S1_OK, S1_ERR_INVALID_ARG, S1_ERR_INVALID_HANDLE, S1_ERR_OOM, S1_ERR_BUDGET, S1_ERR_CUDA, \
    S1_ERR_DEVICE_TIMEOUT, S1_ERR_UNSUPPORTED = range(8)
S1_F32, S1_BF16 = 0, 1
S1_NOALLOC_WS_FLOATS = 4 * 1024 * 1024   # fixed split-K scratch of s1_op_gemm_noalloc (include/s1_ops.h)
S1_STAT_COUNT = 8
PROF_NCLASS = 8
PROF_NAMES = ["gemm", "gdn", "attn", "norm", "other"]


class S1Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"s1 error {code}: {msg}")
        self.code = code


class Shape(C.Structure):
    _fields_ = [("vocab", C.c_int32), ("d_model", C.c_int32), ("n_layers", C.c_int32), ("ffn", C.c_int32),
                ("la_heads", C.c_int32), ("la_dk", C.c_int32), ("la_dv", C.c_int32),
                ("fa_q_heads", C.c_int32), ("fa_kv_heads", C.c_int32), ("fa_head_dim", C.c_int32),
                ("layer_is_full", C.POINTER(C.c_uint8)),
                ("rope_theta", C.c_float), ("rms_eps", C.c_float), ("l2_eps", C.c_float),
                ("lora_rank", C.c_int32), ("lora_alpha", C.c_float), ("weight_dtype", C.c_int32),
                ("max_rows", C.c_int32), ("conv_width", C.c_int32)]


class Weights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("final_norm", C.c_void_p), ("layer", C.POINTER(C.c_void_p)),
                ("lora_a", C.POINTER(C.c_void_p)), ("lora_b", C.POINTER(C.c_void_p))]


class Question(C.Structure):
    _fields_ = [("type", C.c_int32), ("suffix", C.POINTER(C.c_int32)), ("n_suffix", C.c_int32),
                ("option_ids", C.POINTER(C.c_int32)), ("n_options", C.c_int32)]


class Result(C.Structure):
    _fields_ = [("probs", C.POINTER(C.c_float)), ("argmax", C.c_int32), ("expected_score", C.c_float),
                ("yes_prob", C.c_float), ("answer_confidence", C.c_float), ("confidence", C.c_float),
                ("entropy_confidence", C.c_float), ("lm_logprobs", C.POINTER(C.c_float))]


_lib = None


def lib():
    """Load libs1.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m prefill_only_decision_gb300.build`")
    L = C.CDLL(LIB_PATH)
    vp, i32, f32 = C.c_void_p, C.c_int32, C.c_float
    P = C.POINTER
    sig = {
        "s1_model_create": (C.c_int, [P(Shape), P(Weights), P(vp)]),
        "s1_model_destroy": (None, [vp]),
        "s1_set_stream": (C.c_int, [vp, vp]),
        "s1_set_allocator": (C.c_int, [vp, vp, vp]),
        "s1_prefill_state": (C.c_int, [vp, P(i32), i32, vp, i32, P(vp)]),
        "s1_prefill_state_batch": (C.c_int, [vp, i32, P(P(i32)), P(i32), P(vp), P(i32), P(vp)]),
        "s1_state_destroy": (None, [vp]),
        "s1_state_rows": (C.c_int, [vp]),
        "s1_decide": (C.c_int, [vp, vp, P(Question), i32, P(Result), P(f32)]),
        "s1_decide_batch": (C.c_int, [vp, i32, P(vp), P(P(Question)), P(i32), P(P(Result)), P(P(f32))]),
        "s1_state_create": (C.c_int, [vp, i32, P(vp)]),
        "s1_prefill_async": (C.c_int, [vp, vp, vp, i32, vp, i32]),
        "s1_decide_async": (C.c_int, [vp, vp, P(Question), i32, vp, vp, vp]),
        "s1_sync": (C.c_int, [vp]),
        "s1_prefill_decide": (C.c_int, [vp, P(i32), i32, vp, i32, P(Question), i32, P(Result), P(f32), P(vp)]),
        "s1_prefill_decide_batch": (C.c_int, [vp, i32, P(P(i32)), P(i32), P(vp), P(i32), P(P(Question)), P(i32),
                                              P(P(Result)), P(P(f32)), P(vp)]),
        "s1_prefill_decide_async": (C.c_int, [vp, vp, vp, i32, vp, i32, P(Question), i32, vp, vp, vp]),
        "s1_prefill_decide_batch_async": (C.c_int, [vp, i32, P(vp), P(vp), P(i32), P(vp), P(i32), P(vp), P(i32),
                                                    vp, vp, vp]),
        "s1_last_error": (C.c_char_p, []),
        "s1_version": (C.c_char_p, []),
        "s1_op_gemm": (C.c_int, [vp, vp, i32, i32, i32, i32, vp, i32, i32, vp]),
        "s1_op_gdn": (C.c_int, [vp, i32, i32, i32, i32, f32, i32, P(i32), P(i32), vp, vp, vp, vp]),
        "s1_op_attention": (C.c_int, [vp, vp, vp, vp, i32, i32, P(i32), P(i32), i32, i32, i32, vp, vp]),
        "s1_op_rmsnorm": (C.c_int, [vp, vp, i32, i32, f32, vp, vp]),
        "s1_profile": (C.c_int, [vp, C.c_int]),
        "s1_profile_read": (C.c_int, [vp, P(C.c_double), P(C.c_double), P(C.c_double), P(C.c_long)]),
        "s1_set_gemm_impl": (C.c_int, [vp, C.c_int]),
        "s1_set_layer_trace": (C.c_int, [vp, vp, C.c_longlong]),
        "s1_set_graphs": (C.c_int, [vp, C.c_int]),
        "s1_counters": (C.c_int, [vp, P(C.c_longlong), P(C.c_longlong), P(C.c_longlong)]),
        "s1_split_prefix": (C.c_int, [P(P(i32)), P(i32), i32, i32, i32, P(i32)]),
        "s1_gemm_plan": (C.c_int, [i32, i32, i32, i32, i32, i32, P(i32)]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def check(rc: int):
    if rc != S1_OK:
        raise S1Error(rc, lib().s1_last_error().decode(errors="replace"))


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _iptr(a: np.ndarray):
    return a.ctypes.data_as(C.POINTER(C.c_int32))


def make_questions(questions) -> tuple:
    """Questions (objects with .type, .suffix, .option_ids) -> (ctypes array, keep-alive list)."""
    keep = []
    arr = (Question * len(questions))()
    for j, q in enumerate(questions):
        s, o = _i32(q.suffix), _i32(q.option_ids)
        keep += [s, o]
        arr[j] = Question(int(q.type), _iptr(s), len(s), _iptr(o), len(o))
    return arr, keep


class Model:
    """A model in device memory (weights copied and LoRA merged at creation)."""

    def __init__(self, weights, max_rows: int = 0, stream: Optional[int] = None):
        L = lib()
        sh = weights.shape
        self.shape = sh
        full = np.asarray(sh.layer_is_full, dtype=np.uint8)
        self._full = full
        c_shape = Shape(sh.vocab, sh.d_model, sh.n_layers, sh.ffn, sh.la_heads, sh.la_dk, sh.la_dv,
                        sh.fa_q_heads, sh.fa_kv_heads, sh.fa_head_dim,
                        full.ctypes.data_as(C.POINTER(C.c_uint8)), sh.rope_theta, sh.rms_eps, sh.l2_eps,
                        sh.lora_rank, sh.lora_alpha, S1_BF16 if sh.bf16_weights else S1_F32, max_rows,
                        int(getattr(sh, "conv_width", 0)))
        keep = []

        def ptr(a):
            a = np.ascontiguousarray(a)
            keep.append(a)
            return a.ctypes.data

        layer_ptrs = []
        for tl in weights.layers:
            layer_ptrs += [ptr(t) for t in tl]
        lp = (C.c_void_p * len(layer_ptrs))(*layer_ptrs)
        la = lb = None
        if sh.lora_rank > 0:
            a_ptrs, b_ptrs = [], []
            for l in range(sh.n_layers):
                for j in range(7):
                    A, B = weights.lora_a[l][j], weights.lora_b[l][j]
                    a_ptrs.append(ptr(A) if A is not None else None)
                    b_ptrs.append(ptr(B) if B is not None else None)
            la = (C.c_void_p * len(a_ptrs))(*a_ptrs)
            lb = (C.c_void_p * len(b_ptrs))(*b_ptrs)
        w = Weights(ptr(weights.embed), ptr(weights.final_norm), lp, la, lb)
        h = C.c_void_p()
        check(L.s1_model_create(C.byref(c_shape), C.byref(w), C.byref(h)))
        self.h = h
        del keep
        if stream is not None:
            check(L.s1_set_stream(self.h, C.c_void_p(stream)))

    def close(self):
        if getattr(self, "h", None):
            lib().s1_model_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_stream(self, stream: int):
        check(lib().s1_set_stream(self.h, C.c_void_p(stream)))

    # -- blocking API (host buffers) -------------------------------------------------------
    def prefill(self, tokens, embeds: Optional[np.ndarray] = None) -> "State":
        t = _i32(tokens)
        e = None if embeds is None else np.ascontiguousarray(embeds, dtype=np.uint16)
        st = C.c_void_p()
        check(lib().s1_prefill_state(self.h, _iptr(t), len(t), None if e is None else e.ctypes.data,
                                     0 if e is None else e.shape[0], C.byref(st)))
        return State(self, st)

    def prefill_batch(self, requests) -> List["State"]:
        n = len(requests)
        toks = [_i32(r.tokens) for r in requests]
        embs = [None if r.embeds is None else np.ascontiguousarray(r.embeds, dtype=np.uint16) for r in requests]
        tp = (C.POINTER(C.c_int32) * n)(*[_iptr(t) for t in toks])
        nt = (C.c_int32 * n)(*[len(t) for t in toks])
        ep = (C.c_void_p * n)(*[None if e is None else e.ctypes.data for e in embs])
        ne = (C.c_int32 * n)(*[0 if e is None else e.shape[0] for e in embs])
        out = (C.c_void_p * n)()
        check(lib().s1_prefill_state_batch(self.h, n, tp, nt, ep, ne, out))
        return [State(self, C.c_void_p(out[i])) for i in range(n)]

    def decide(self, state: "State", questions, want_hidden: bool = True, want_lm: bool = False):
        res = self.decide_batch([state], [questions], want_hidden, want_lm)
        return res[0]

    def decide_batch(self, states, question_lists, want_hidden: bool = True, want_lm: bool = False):
        n = len(states)
        keep, qarrs, rarrs, probs, hids = self._result_arrays(question_lists, want_hidden, want_lm)
        sp = (C.c_void_p * n)(*[s.h.value for s in states])
        qp = (C.POINTER(Question) * n)(*[C.cast(q, C.POINTER(Question)) for q in qarrs])
        nq = (C.c_int32 * n)(*[len(qs) for qs in question_lists])
        rp = (C.POINTER(Result) * n)(*[C.cast(r, C.POINTER(Result)) for r in rarrs])
        hp = (C.POINTER(C.c_float) * n)(*[h.ctypes.data_as(C.POINTER(C.c_float)) if h is not None else None
                                           for h in hids]) if want_hidden else None
        check(lib().s1_decide_batch(self.h, n, sp, qp, nq, rp, hp))
        return self._unpack(question_lists, rarrs, probs, hids, want_hidden)

    def _result_arrays(self, question_lists, want_hidden, want_lm=False):
        keep, qarrs, rarrs, probs, hids = [], [], [], [], []
        for qs in question_lists:
            qa, k = make_questions(qs)
            keep += k
            qarrs.append(qa)
            ra = (Result * len(qs))()
            pl = []
            for j, q in enumerate(qs):
                p = np.zeros(len(q.option_ids), dtype=np.float32)
                pl.append(p)
                ra[j].probs = p.ctypes.data_as(C.POINTER(C.c_float))
                if want_lm:
                    lmv = np.zeros(len(q.option_ids), dtype=np.float32)
                    keep.append(lmv)
                    ra[j].lm_logprobs = lmv.ctypes.data_as(C.POINTER(C.c_float))
            probs.append(pl)
            rarrs.append(ra)
            hids.append(np.zeros((len(qs), self.shape.d_model), dtype=np.float32) if want_hidden else None)
        return keep, qarrs, rarrs, probs, hids

    @staticmethod
    def _unpack(question_lists, rarrs, probs, hids, want_hidden):
        out = []
        for r in range(len(question_lists)):
            lst = []
            for j in range(len(question_lists[r])):
                x = rarrs[r][j]
                n = len(question_lists[r][j].option_ids)
                lm = np.ctypeslib.as_array(x.lm_logprobs, shape=(n,)).copy() if x.lm_logprobs else None
                lst.append({"probs": probs[r][j], "argmax": x.argmax, "expected_score": x.expected_score,
                            "yes_prob": x.yes_prob, "answer_confidence": x.answer_confidence,
                            "confidence": x.confidence, "entropy_confidence": x.entropy_confidence,
                            "hidden": hids[r][j] if want_hidden else None, "lm_logprobs": lm})
            out.append(lst)
        return out

    def prefill_decide(self, request, want_hidden: bool = True, keep_state: bool = False, want_lm: bool = False):
        """One sweep over prefix + questions (s1_prefill_decide). Returns (results, state or None)."""
        res, sts = self.prefill_decide_batch([request], want_hidden, keep_state, want_lm)
        return res[0], (sts[0] if sts else None)

    def prefill_decide_batch(self, requests, want_hidden: bool = True, keep_state: bool = False,
                             want_lm: bool = False):
        n = len(requests)
        toks = [_i32(r.tokens) for r in requests]
        embs = [None if r.embeds is None else np.ascontiguousarray(r.embeds, dtype=np.uint16) for r in requests]
        qls = [r.questions for r in requests]
        keep, qarrs, rarrs, probs, hids = self._result_arrays(qls, want_hidden, want_lm)
        tp = (C.POINTER(C.c_int32) * n)(*[_iptr(t) for t in toks])
        nt = (C.c_int32 * n)(*[len(t) for t in toks])
        ep = (C.c_void_p * n)(*[None if e is None else e.ctypes.data for e in embs])
        ne = (C.c_int32 * n)(*[0 if e is None else e.shape[0] for e in embs])
        qp = (C.POINTER(Question) * n)(*[C.cast(q, C.POINTER(Question)) for q in qarrs])
        nq = (C.c_int32 * n)(*[len(q) for q in qls])
        rp = (C.POINTER(Result) * n)(*[C.cast(r, C.POINTER(Result)) for r in rarrs])
        hp = (C.POINTER(C.c_float) * n)(*[h.ctypes.data_as(C.POINTER(C.c_float)) for h in hids]) if want_hidden else None
        so = (C.c_void_p * n)() if keep_state else None
        check(lib().s1_prefill_decide_batch(self.h, n, tp, nt, ep, ne, qp, nq, rp, hp, so))
        states = [State(self, C.c_void_p(so[i])) for i in range(n)] if keep_state else None
        return self._unpack(qls, rarrs, probs, hids, want_hidden), states

    def prefill_decide_async(self, state: "State", d_tokens: int, n_tokens: int, qarr, n_q: int, d_probs: int,
                             d_stats: int, d_hidden: int = 0, d_embeds: int = 0, n_embeds: int = 0):
        check(lib().s1_prefill_decide_async(self.h, state.h, C.c_void_p(d_tokens), n_tokens,
                                            C.c_void_p(d_embeds) if d_embeds else None, n_embeds, qarr, n_q,
                                            C.c_void_p(d_probs), C.c_void_p(d_stats),
                                            C.c_void_p(d_hidden) if d_hidden else None))

    def prefill_decide_batch_async(self, states, d_tokens, n_tokens, qarrs, n_q, d_probs: int, d_stats: int,
                                   d_hidden: int = 0, d_embeds=None, n_embeds=None):
        """s1_prefill_decide_batch_async: per request a state, a device id pointer and count, a
        Question array with device ids (and optional device embedding rows)."""
        n = len(states)
        S = (C.c_void_p * n)(*[s.h for s in states])
        T = (C.c_void_p * n)(*[C.c_void_p(p) for p in d_tokens])
        NT = (C.c_int32 * n)(*n_tokens)
        Q = (C.c_void_p * n)(*[C.cast(q, C.c_void_p) for q in qarrs])
        NQ = (C.c_int32 * n)(*n_q)
        E = (C.c_void_p * n)(*[C.c_void_p(p) if p else None for p in d_embeds]) if d_embeds else None
        NE = (C.c_int32 * n)(*n_embeds) if n_embeds else None
        check(lib().s1_prefill_decide_batch_async(self.h, n, S, T, NT, E, NE, Q, NQ, C.c_void_p(d_probs),
                                                  C.c_void_p(d_stats), C.c_void_p(d_hidden) if d_hidden else None))

    # -- stream-ordered API (device pointers) -----------------------------------------------
    def state_create(self, capacity_rows: int) -> "State":
        st = C.c_void_p()
        check(lib().s1_state_create(self.h, capacity_rows, C.byref(st)))
        return State(self, st)

    def prefill_async(self, state: "State", d_tokens: int, n_tokens: int, d_embeds: int = 0, n_embeds: int = 0):
        check(lib().s1_prefill_async(self.h, state.h, C.c_void_p(d_tokens), n_tokens,
                                     C.c_void_p(d_embeds) if d_embeds else None, n_embeds))

    def decide_async(self, state: "State", qarr, n_q: int, d_probs: int, d_stats: int, d_hidden: int = 0):
        check(lib().s1_decide_async(self.h, state.h, qarr, n_q, C.c_void_p(d_probs), C.c_void_p(d_stats),
                                    C.c_void_p(d_hidden) if d_hidden else None))

    def sync(self):
        check(lib().s1_sync(self.h))

    # -- instrumentation ---------------------------------------------------------------------
    def profile(self, enable: bool):
        check(lib().s1_profile(self.h, 1 if enable else 0))

    def profile_read(self):
        ms = (C.c_double * PROF_NCLASS)()
        fl = (C.c_double * PROF_NCLASS)()
        by = (C.c_double * PROF_NCLASS)()
        ct = (C.c_long * PROF_NCLASS)()
        check(lib().s1_profile_read(self.h, ms, fl, by, ct))
        return {name: {"ms": ms[i], "flops": fl[i], "bytes": by[i], "count": ct[i]}
                for i, name in enumerate(PROF_NAMES)}

    def counters(self):
        a, b, c = C.c_longlong(), C.c_longlong(), C.c_longlong()
        check(lib().s1_counters(self.h, C.byref(a), C.byref(b), C.byref(c)))
        return {"launches": a.value, "h2d_bytes": b.value, "d2h_bytes": c.value}

    def set_gemm_impl(self, impl: int):
        check(lib().s1_set_gemm_impl(self.h, impl))

    def set_graphs(self, enable: bool):
        """CUDA graphs for the stream-ordered calls (prefill_async, decide_async,
        prefill_decide_async) whose signature repeats (s1_set_graphs)."""
        check(lib().s1_set_graphs(self.h, 1 if enable else 0))

    def set_layer_trace(self, ptr: int, capacity_floats: int):
        """Record the fp32 residual stream after the embedding and after every layer of each
        forward into the device buffer at `ptr` ([n_layers + 1, R, d]); ptr 0 clears."""
        check(lib().s1_set_layer_trace(self.h, C.c_void_p(ptr) if ptr else None, int(capacity_floats)))


class State:
    def __init__(self, model: Model, h):
        self.model = model
        self.h = h

    @property
    def rows(self) -> int:
        return lib().s1_state_rows(self.h)

    def close(self):
        if getattr(self, "h", None):
            lib().s1_state_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def split_prefix(streams, min_suffix: int = 1, align: int = 0) -> int:
    """Length of the shared prefix of whole per-question token streams (s1_split_prefix)."""
    arrs = [_i32(s) for s in streams]
    sp = (C.POINTER(C.c_int32) * len(arrs))(*[_iptr(a) for a in arrs])
    ln = (C.c_int32 * len(arrs))(*[len(a) for a in arrs])
    out = C.c_int32()
    check(lib().s1_split_prefix(sp, ln, len(arrs), min_suffix, align, C.byref(out)))
    return out.value


_ALLOC_T = C.CFUNCTYPE(C.c_void_p, C.c_size_t, C.c_void_p)
_FREE_T = C.CFUNCTYPE(None, C.c_void_p, C.c_void_p)
_hooks = []


def use_torch_allocator():
    """Route the library's device allocations through PyTorch's caching allocator (call
    before creating a model; blocks are tied to the current stream)."""
    import torch

    def _alloc(n, _ctx):
        try:
            return torch.cuda.caching_allocator_alloc(int(n))
        except Exception:
            return None

    def _free(p, _ctx):
        if p:
            torch.cuda.caching_allocator_delete(p)

    a, f = _ALLOC_T(_alloc), _FREE_T(_free)
    _hooks[:] = [a, f]
    check(lib().s1_set_allocator(C.cast(a, C.c_void_p), C.cast(f, C.c_void_p), None))


def use_default_allocator():
    check(lib().s1_set_allocator(None, None, None))
    _hooks.clear()


# -- kernel-level ops on device pointers (integers) ------------------------------------------
def op_gemm(X: int, W: int, M: int, N: int, K: int, epi: int, out: int, ldo: int, impl: int = 0, stream: int = 0):
    check(lib().s1_op_gemm(C.c_void_p(X), C.c_void_p(W), M, N, K, epi, C.c_void_p(out), ldo, impl,
                           C.c_void_p(stream) if stream else None))


def op_gdn(proj: int, R: int, H: int, dk: int, dv: int, eps: float, row0: Sequence[int], lens: Sequence[int],
           S0: int, S_out: int, out: int, stream: int = 0):
    r0, ln = _i32(row0), _i32(lens)
    check(lib().s1_op_gdn(C.c_void_p(proj), R, H, dk, dv, eps, len(r0), _iptr(r0), _iptr(ln),
                          C.c_void_p(S0) if S0 else None, C.c_void_p(S_out) if S_out else None, C.c_void_p(out),
                          C.c_void_p(stream) if stream else None))


def op_attention(q: int, k_new: int, v_new: int, kv_cache: int, P: int, row0, lens, Hq: int, Hkv: int, hd: int,
                 out: int, stream: int = 0):
    r0, ln = _i32(row0), _i32(lens)
    check(lib().s1_op_attention(C.c_void_p(q), C.c_void_p(k_new), C.c_void_p(v_new),
                                C.c_void_p(kv_cache) if kv_cache else None, P, len(r0), _iptr(r0), _iptr(ln),
                                Hq, Hkv, hd, C.c_void_p(out), C.c_void_p(stream) if stream else None))


def gemm_plan(M: int, N: int, K: int, epi: int, num_sms: int, pair: bool = False) -> dict:
    """The planner's heuristic GEMM plan (s1_gemm_plan; host logic, no GPU needed)."""
    out = (C.c_int32 * 7)()
    check(lib().s1_gemm_plan(M, N, K, epi, num_sms, 1 if pair else 0, out))
    return dict(zip(("bn", "cm", "pair", "splits", "kbp", "m_tiles", "n_tiles"), list(out)))


def op_rmsnorm(x: int, w: int, R: int, d: int, eps: float, out: int, stream: int = 0):
    check(lib().s1_op_rmsnorm(C.c_void_p(x), C.c_void_p(w), R, d, eps, C.c_void_p(out),
                              C.c_void_p(stream) if stream else None))
