"""Shared parity checks of the GPU decision path against the oracle (helpers, not tests).

The tolerance contract of the method's acceptance bar, held against the plain fp32 oracle (LoRA
unmerged, fp32 everywhere): per-option probabilities within 2e-2 absolute, expected score
within 5e-2, last-layer hidden state within 3e-2 relative L2, identical argmax wherever the
oracle's top-2 margin exceeds 0.05.
"""
import numpy as np

from oracle import model as om
from prefill_only_decision_gb300 import configs

P_TOL, E_TOL, H_TOL, MARGIN = 2e-2, 5e-2, 3e-2, 0.05
LAYER_TOL = 1e-2


def compare(gpu, ref, qs, tag=""):
    """Assert the tolerance contract for one list of results (GPU vs the fp32 oracle), plus the
    readout's own invariants; returns the worst errors."""
    worst = dict(p=0.0, e=0.0, h=0.0)
    for j, (g, r, q) in enumerate(zip(gpu, ref, qs)):
        p_err = float(np.abs(g["probs"] - r["probs"]).max())
        e_err = abs(float(g["expected_score"]) - float(r["expected_score"]))
        assert p_err <= P_TOL, (tag, j, p_err)
        assert e_err <= E_TOL, (tag, j, e_err)
        srt = np.sort(r["probs"])[::-1]
        if len(srt) == 1 or srt[0] - srt[1] > MARGIN:
            assert g["argmax"] == int(r["argmax"]), (tag, j, g["probs"], r["probs"])
        if g.get("hidden") is not None:
            h_err = float(np.linalg.norm(g["hidden"] - r["hidden"]) / np.linalg.norm(r["hidden"]))
            assert h_err <= H_TOL, (tag, j, h_err)
            worst["h"] = max(worst["h"], h_err)
        assert abs(float(np.sum(g["probs"])) - 1) < 1e-5
        assert 0 <= g["expected_score"] <= len(q.option_ids) - 1 + 1e-6
        conf = g["answer_confidence"] if q.type == configs.NOUL else g["entropy_confidence"]
        assert abs(g["confidence"] - conf) < 1e-6
        assert abs(g["confidence"] - float(r["confidence"])) <= 5e-2
        worst["p"] = max(worst["p"], p_err)
        worst["e"] = max(worst["e"], e_err)
    print(f"[parity {tag}] max |dp| {worst['p']:.2e}  max |dE| {worst['e']:.2e}  max hidden rel L2 {worst['h']:.2e}")
    return worst


def layerwise(B, torch, W, req, tag, layers=None, tol=LAYER_TOL):
    """Teacher-forced per-layer parity on one fused sweep: the GPU's residual stream entering
    each layer goes through the policy oracle's layer (the GPU's rounding points: f16 merged
    weights and matrix inputs, fp32 accumulation, state and head; the prefix rows, then each
    question's rows continuing from the prefix's layer state), and the result is held against
    the GPU's stream after that layer (rel L2 per row block). Independent of depth: an error in
    any layer's kernels shows up in that layer, not amplified by the layers after it.
    `layers`: the layer indices checked (default: all)."""
    s = W.shape
    P = req.prefix_rows
    n_rows = P + sum(len(q.suffix) for q in req.questions)
    L, d = s.n_layers, s.d_model
    buf = torch.zeros(((L + 1) * n_rows * d,), dtype=torch.float32, device="cuda")
    m = B.Model(W)
    try:
        m.set_layer_trace(buf.data_ptr(), buf.numel())
        m.prefill_decide(req)
        m.set_layer_trace(0, 0)
    finally:
        m.close()
    X = buf.view(L + 1, n_rows, d).cpu().numpy()
    del buf
    o = om.Oracle(W, np.float32, precision="f16")
    rel = lambda a, b: float(np.linalg.norm(a - b) / np.linalg.norm(b))
    worst = 0.0
    for l in (range(L) if layers is None else layers):
        xp, cache = o.layer(l, X[l, :P], np.arange(P), None)
        errs = [rel(xp, X[l + 1, :P])]
        r = P
        for q in req.questions:
            n = len(q.suffix)
            xq, _ = o.layer(l, X[l, r:r + n], P + np.arange(n), cache)
            errs.append(rel(xq, X[l + 1, r:r + n]))
            r += n
        worst = max(worst, max(errs))
        assert max(errs) <= tol, (tag, l, errs)
    print(f"[layerwise {tag}] {L if layers is None else len(layers)} layers, worst per-layer rel L2 {worst:.2e}")
    return worst


def golden_results(path):
    """Per-request lists of the oracle's stored per-question results (tests/golden/large_*.npz,
    written by tests/golden/make_large_goldens.py)."""
    z = np.load(path)
    out = {}
    for i in z["requests"].tolist():
        res = []
        j = 0
        while f"q{i}_{j}_probs" in z:
            res.append({k: z[f"q{i}_{j}_{k}"] for k in ("probs", "logits", "expected_score", "argmax",
                                                         "answer_confidence", "confidence",
                                                         "entropy_confidence", "hidden")})
            j += 1
        out[i] = res
    return out
