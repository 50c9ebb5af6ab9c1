"""Write the oracle's expected results for the large configurations (4B, 4B multimodal, 27B).

    python tests/golden/make_large_goldens.py [4b] [4b_mm] [27b]

The plain fp32 oracle (LoRA unmerged, fp32 everywhere) runs on the seeded synthetic weights and
requests of each configuration and its per-question results are stored in
tests/golden/large_<config>.npz. Only `oracle/` and the seeded input generators are used: no
value here comes from the CUDA path. The GPU tests of these configurations compare against the
stored values, so that they do not spend many CPU minutes re-running the oracle.

What is stored per configuration:
  * 4b: its one request (1024-token prefix, 3 questions of 48 tokens).
  * 4b_mm: request 0 of the batch of 8 (1024 given embedding rows + 256 tokens, all 32
    questions of 40 tokens).
  * 27b: four requests of the 74-request sweep: request 0 (P = 1536) and the shortest, median
    and longest prefix among the 74.
Each question's results are prefixed q<request>_<question>_: probs, logits, expected_score,
argmax, answer_confidence, confidence, entropy_confidence, hidden (the last layer's output at
the readout row, before the final norm).
"""
from __future__ import annotations

import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle import model as om  # noqa: E402
from prefill_only_decision_gb300 import configs, synth  # noqa: E402

KEYS = ("probs", "logits", "expected_score", "argmax", "answer_confidence", "confidence", "entropy_confidence",
        "hidden")


def sweep_subset(reqs):
    """Request 0 (the nominal prefix) and the shortest, median and longest prefix of the sweep."""
    lens = np.array([len(r.tokens) for r in reqs])
    order = np.argsort(lens, kind="stable")
    pick = [0, int(order[0]), int(order[len(order) // 2]), int(order[-1])]
    out = []
    for i in pick:
        if i not in out:
            out.append(i)
    return out


def plan(name):
    """(config, request indices, question indices per request) stored for `name`."""
    cfg = configs.CONFIGS[name]
    if name == "27b":
        reqs = synth.make_requests(cfg)
        return cfg, reqs, sweep_subset(reqs)
    reqs = synth.make_requests(cfg, n_requests=1)
    return cfg, reqs, [0]


def run(name):
    cfg, reqs, idx = plan(name)
    t0 = time.time()
    W = synth.make_weights(cfg)
    print(f"[{name}] weights in {time.time() - t0:.0f} s", flush=True)
    o = om.Oracle(W, np.float32)
    out = {"config": np.array(name), "seed": np.array(cfg.seed), "requests": np.array(idx, dtype=np.int32)}
    for i in idx:
        r = reqs[i]
        t0 = time.time()
        res = o.decide(r, branched=True)
        out[f"r{i}_prefix_rows"] = np.array(r.prefix_rows, dtype=np.int32)
        for j, x in enumerate(res):
            for k in KEYS:
                out[f"q{i}_{j}_{k}"] = np.asarray(x[k], dtype=np.float64 if k not in ("hidden", "probs", "logits")
                                                  else np.float32)
        print(f"[{name}] request {i} (P = {r.prefix_rows}, {len(res)} questions) in {time.time() - t0:.0f} s",
              flush=True)
    path = os.path.join(HERE, f"large_{name}.npz")
    np.savez_compressed(path, **out)
    print(f"[{name}] wrote {path}", flush=True)


if __name__ == "__main__":
    for n in (sys.argv[1:] or ["4b", "4b_mm", "27b"]):
        run(n)
