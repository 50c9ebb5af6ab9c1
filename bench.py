"""Benchmark: prefill-only decisions on the 4B-class hybrid decoder (1 GB300).

One step = one request of the workload: prefill a 1024-token state prefix, then decide 3
questions (choice over 3 labels, score over 4 levels, noul) with 48-token suffixes branched
from the prefix snapshot -> 3 decisions per step. Weights are seeded random-init of the
4B-class shape (bf16 weights, rank-32 LoRA merged at load into f16 tensor-core operands); inputs
are seeded synthetic token ids.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 4b] [--impl ours|reference]

value  = decisions/s measured on the device (CUDA events on the library's stream) with the
         request's ids already in device memory (stream-ordered API);
e2e    = decisions/s through the blocking public API (host ids in, host results out,
         host<->device copies inside the timed region), with its p50 latency;
roofline = the tensor-core GEMM (the dominant kernel) against the measured dense 16-bit peak
         (cuBLAS bf16 burst; f16 runs at the same nominal tensor-core rate), plus the whole step;
cpu_baseline = the oracle (numpy, fp32) on a bounded sample of the same workload.
`--impl reference` times the oracle alone (the reference arm of this comparison).
Under torchrun (N > 1) every rank runs an independent replica ("replicas only").
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# The reference arm (the oracle on the host cores) runs on rank 0 alone: its BLAS gets every
# core the process may use, also under torchrun (which sets OMP_NUM_THREADS=1 for its ranks).
# Set before numpy is imported, which reads these once.
def _impl_arg(argv):
    for i, a in enumerate(argv):
        if a == "--impl" and i + 1 < len(argv):
            return argv[i + 1]
        if a.startswith("--impl="):
            return a.split("=", 1)[1]
    return None


if _impl_arg(sys.argv) == "reference":
    for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[_v] = str(len(os.sched_getaffinity(0)))

import numpy as np  # noqa: E402

FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per tensor-core GEMM launch, averaged
# over one step's GEMM launches in an ncu capture of this bench's timed step (caches not flushed
# between launches), per workload; a workload whose kernels changed since their capture has no
# entry (the field reads null).
GEMM_DRAM_BYTES_PER_LAUNCH = {"4b": 77264930}


def tensor_peak(peaks, ms_timed):
    """The bf16 peak a GEMM timed inside `ms_timed` ms of back-to-back steps is held to: the burst
    figure for a short region at full clocks, the sustained (power-capped loop) figure once the
    region lasts a quarter second or more. f16 operands run at bf16's nominal dense rate (x 1)."""
    if ms_timed >= 250.0:
        return peaks["bf16_tflops_sustained"], f"{peaks['source']} bf16 sustained x 1 (f16 operands)"
    return peaks["bf16_tflops"], f"{peaks['source']} bf16 burst x 1 (f16 operands)"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            out = {"source": "measured"}
            for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                v = d.get(k)
                if isinstance(v, dict):
                    v = v.get("value")
                out[k] = float(v) if v is not None else FALLBACK[k]
            return out
        except Exception:
            pass
    return dict(FALLBACK, source="fallback")


class ClockSampler:
    """nvidia-smi sampling (every 50 ms) of clocks and throttle reasons; summary() keeps the samples
    taken between mark_start() and mark_end() (the timed region)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            deadline = time.time() + 5.0      # sampling is running before the timed region starts
            while not self.lines and time.time() < deadline and self.proc.poll() is None:
                time.sleep(0.02)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines = self.lines
        if self.t0 is not None and self.t1 is not None:
            inside = [x for x in lines if self.t0 <= x[0] <= self.t1 + 0.05]
            lines = inside if inside else lines[-1:]
        for _, ln in lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    from prefill_only_decision_gb300 import replicas
    return replicas.world()


def time_oracle(cfg, W, req, budget_s: float = 25.0):
    """The oracle (as it stands) on a bounded sample: whole questions of the request, each
    the plain unbranched forward over prefix + suffix, until ~budget_s of CPU time. Returns the
    rate, and the sample's wall time in `seconds`."""
    from oracle import model as om
    o = om.Oracle(W, np.float32)
    t0 = time.perf_counter()
    n = 0
    for q in req.questions:
        o.decide_unbranched(req.tokens, req.embeds, [q])
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0))
    rows = req.prefix_rows + int(np.mean([len(q.suffix) for q in req.questions]))
    return {"value": n / dt, "unit": "decisions/s", "cores": cores, "kind": "oracle", "seconds": dt,
            "sample": f"{n} question(s) of request 0, each a full unbranched forward over ~{rows} rows "
                      f"(numpy fp32, {cores} host threads), {dt:.1f} s"}


def run_reference(args, cfg):
    ws, rank, _ = dist_setup()
    if rank != 0:
        return 0
    from prefill_only_decision_gb300 import synth
    W = synth.make_weights(cfg)
    req = synth.make_requests(cfg)[0]
    runs = []
    for _ in range(args.warmup + args.steps):
        runs.append(time_oracle(cfg, W, req, budget_s=float(os.environ.get("S1_REF_BUDGET", "10"))))
    timed = runs[args.warmup:] if args.steps else runs[-1:]
    v = float(np.mean([r["value"] for r in timed]))
    step_ms = 1000.0 * float(np.mean([r["seconds"] for r in timed]))   # wall time of one timed step
    cb = dict(timed[-1])
    cb["value"] = v
    line = {"impl": "reference", "metric": "decisions/s", "value": v, "unit": "decisions/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": cfg.name + " (oracle sample)", "prefix_rows": req.prefix_rows,
                       "questions": len(req.questions), "suffix_len": len(req.questions[0].suffix)},
            "cpu_baseline": cb,
            "e2e": {"value": v, "unit": "decisions/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_kernel(args):
    """Time one kernel-level entry point (s1_ops.h) in isolation: `--kernel gemm --shape M,N,K[,epi]`,
    `--kernel gdn --shape R,H,D[,nseq]` or `--kernel attn --shape P,len,nseq,Hq,Hkv,hd`."""
    import torch
    from prefill_only_decision_gb300 import binding as B
    dims = [int(x) for x in args.shape.split(";")[0].split(",")]
    g = torch.Generator(device="cuda").manual_seed(0)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if args.kernel == "gemm":
        # several shapes may be given as "M,N,K,epi[,impl[,bn,splits]];..." (one measurement pass
        # under ncu); impl as s1_op_gemm's: 0 planner's choice, 2 CTA-pair tiles, 3 single-CTA
        # tiles; bn / splits > 0 pin the single-CTA planner's tile width / K split for that entry
        shapes = [[int(x) for x in sh.split(",")] for sh in args.shape.split(";")]
        res = []
        for sh in shapes:
            M, N, K = sh[:3]
            epi = sh[3] if len(sh) > 3 else 0
            impl = sh[4] if len(sh) > 4 else 0
            for var, val in (("S1_GEMM_BN", sh[5] if len(sh) > 5 else 0), ("S1_GEMM_SPLITS", sh[6] if len(sh) > 6 else 0)):
                if val > 0:
                    os.environ[var] = str(val)
                else:
                    os.environ.pop(var, None)
            X = torch.randn((M, K), device="cuda", generator=g).to(torch.float16)
            W = (0.02 * torch.randn((N, K), device="cuda", generator=g)).to(torch.float16)
            out = torch.zeros((M, N // 2 if epi == 3 else N), device="cuda",
                              dtype=torch.float16 if epi in (1, 3) else torch.float32)
            call = lambda: B.op_gemm(X.data_ptr(), W.data_ptr(), M, N, K, epi, out.data_ptr(), out.shape[1], impl)
            for _ in range(max(1, args.warmup)):
                call()
            torch.cuda.synchronize()
            ts = []
            for _ in range(max(1, args.steps)):
                ev0.record()
                call()
                ev1.record()
                torch.cuda.synchronize()
                ts.append(ev0.elapsed_time(ev1))
            ms = float(np.median(ts))
            res.append({"shape": sh, "us_median": round(1e3 * ms, 2),
                        "tflops": round(2.0 * M * N * K / (ms / 1e3) / 1e12, 1)})
        torch.cuda.synchronize()
        print(json.dumps({"kernel": "gemm", "runs": res,
                          "note": "CUDA events around each op call (one launch; inputs L2-resident after the first call)"}))
        return 0
    elif args.kernel == "gdn":
        R, H, D = dims[:3]
        nseq = dims[3] if len(dims) > 3 else 1
        ld = 3 * H * D + 2 * H
        proj = torch.randn((R, ld), device="cuda", generator=g)
        out = torch.zeros((R, H * D), device="cuda", dtype=torch.float16)
        lens = [R // nseq] * nseq
        lens[-1] += R - sum(lens)
        row0 = list(np.cumsum([0] + lens[:-1]))
        fn = lambda: B.op_gdn(proj.data_ptr(), R, H, D, D, 1e-6, row0, lens, 0, 0, out.data_ptr())
        work, unit = 6.0 * R * H * D * D, "GFLOP/s (recurrence count)"
    else:
        P, L, nseq, Hq, Hkv, hd = dims[:6]
        R = L * nseq
        q = torch.randn((R, Hq, hd), device="cuda", generator=g).to(torch.float16)
        kn = torch.randn((R, Hkv, hd), device="cuda", generator=g).to(torch.float16)
        vn = torch.randn((R, Hkv, hd), device="cuda", generator=g).to(torch.float16)
        kv = torch.randn((2, max(P, 1), Hkv, hd), device="cuda", generator=g).to(torch.float16)
        out = torch.zeros((R, Hq * hd), device="cuda", dtype=torch.float16)
        row0 = [i * L for i in range(nseq)]
        fn = lambda: B.op_attention(q.data_ptr(), kn.data_ptr(), vn.data_ptr(), kv.data_ptr() if P else 0, P, row0,
                                    [L] * nseq, Hq, Hkv, hd, out.data_ptr())
        keys = sum(P + i + 1 for i in range(L)) * nseq
        work, unit = 4.0 * hd * Hq * keys, "TFLOP/s"
    for _ in range(max(1, args.warmup)):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(max(1, args.steps)):
        ev0.record()
        fn()
        ev1.record()
        torch.cuda.synchronize()
        ts.append(ev0.elapsed_time(ev1))
    ms = float(np.median(ts))
    scale = 1e12 if unit.startswith("TFLOP") else 1e9
    print(json.dumps({"kernel": args.kernel, "shape": dims, "ms_median": ms, "ms_min": float(min(ts)),
                      "achieved": work / (ms / 1e3) / scale, "unit": unit,
                      "note": "op-level call (includes its small temporaries and one synchronisation)"}))
    return 0


def run_batch(args, cfg, torch, ws, rank, local):
    """A batch workload (the small model's 16 requests, the 4B multimodal batch of 8): one step =
    one s1_prefill_decide_batch_async over every request of the batch (each prefix and its
    questions in one layer sweep), ids and embedding rows resident in device memory; e2e = the
    blocking s1_prefill_decide_batch with host buffers."""
    import ctypes as C
    from prefill_only_decision_gb300 import binding, replicas, synth
    W = synth.make_weights(cfg)
    reqs = synth.make_requests(cfg)
    stream = torch.cuda.Stream()
    binding.use_torch_allocator()
    model = binding.Model(W, stream=stream.cuda_stream)
    if not args.no_graphs:
        model.set_graphs(True)
    states = [model.state_create(r.prefix_rows) for r in reqs]
    toks = [torch.from_numpy(r.tokens).cuda() for r in reqs]
    embs = [torch.from_numpy(r.embeds.view(np.int16)).cuda() if r.embeds is not None else None for r in reqs]
    keep, qarrs = [], []
    for r in reqs:
        dq = [(torch.from_numpy(q.suffix).cuda(), torch.from_numpy(q.option_ids).cuda(), q.type) for q in r.questions]
        keep += dq
        arr = (binding.Question * len(dq))()
        for j, (su, op, t) in enumerate(dq):
            arr[j] = binding.Question(t, C.cast(C.c_void_p(su.data_ptr()), C.POINTER(C.c_int32)), su.numel(),
                                      C.cast(C.c_void_p(op.data_ptr()), C.POINTER(C.c_int32)), op.numel())
        qarrs.append(arr)
    n_q = [len(r.questions) for r in reqs]
    n_opt = sum(len(q.option_ids) for r in reqs for q in r.questions)
    d_probs = torch.zeros(n_opt, dtype=torch.float32, device="cuda")
    d_stats = torch.zeros((sum(n_q), 8), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    dec = sum(n_q)

    def step():
        model.prefill_decide_batch_async(states, [t.data_ptr() for t in toks], [len(r.tokens) for r in reqs], qarrs,
                                         n_q, d_probs.data_ptr(), d_stats.data_ptr(), 0,
                                         [e.data_ptr() if e is not None else 0 for e in embs],
                                         [0 if r.embeds is None else r.embeds.shape[0] for r in reqs])

    def barrier():
        torch.cuda.synchronize()
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(max(3, args.warmup)):
        step()
    model.sync()
    launches0 = model.counters()["launches"]
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nvtx = os.environ.get("S1_NVTX") == "1"     # lets ncu --nvtx-include "timed/" select the timed steps
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        clk.mark_start()
        if nvtx:
            torch.cuda.nvtx.range_push("timed")
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        if nvtx:
            torch.cuda.nvtx.range_pop()
        barrier()
        clk.mark_end()
    ms_total = replicas.max_over_ranks(e0.elapsed_time(e1), device="cuda")
    launches = (model.counters()["launches"] - launches0) // max(1, args.steps)
    ms_step = ms_total / max(1, args.steps)
    value = ws * dec * args.steps / (ms_total / 1000.0)
    model.profile(True)
    for _ in range(args.steps):
        step()
    prof = model.profile_read()
    model.profile(False)
    peaks = load_peaks()
    g = prof["gemm"]
    peak, peak_source = tensor_peak(peaks, ms_total)
    achieved = g["flops"] / (g["ms"] / 1000.0) / 1e12 if g["ms"] > 0 else 0.0
    total_prof_ms = sum(v["ms"] for v in prof.values())
    step_flops = g["flops"] / max(1, args.steps)
    roofline = {"bound": "tensor", "kernel": "gemm_kernel / gemm_pair_kernel (tcgen05, all projections)",
                "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak if peak else None,
                "traffic": GEMM_DRAM_BYTES_PER_LAUNCH.get(cfg.name),
                "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum, "
                                "mean over the timed step's GEMM launches, warm caches)",
                "algorithmic_bytes_per_launch": g["bytes"] / max(1, g["count"]),
                "peak_source": peak_source,
                "share_of_step": g["ms"] / total_prof_ms if total_prof_ms else None,
                "launches_per_step": g["count"] / max(1, args.steps), "flops_per_step": step_flops,
                "step_achieved": step_flops / (ms_step / 1000.0) / 1e12,
                "step_frac": step_flops / (ms_step / 1000.0) / 1e12 / peak if peak else None}
    model.sync()
    c0 = model.counters()
    lat = []
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        a = time.perf_counter()
        model.prefill_decide_batch(reqs, want_hidden=False)
        lat.append((time.perf_counter() - a) * 1000.0)
    barrier()
    e2e_s = time.perf_counter() - t0
    c1 = model.counters()
    e2e = {"value": ws * dec * args.steps / e2e_s, "unit": "decisions/s",
           "h2d_bytes_per_step": (c1["h2d_bytes"] - c0["h2d_bytes"]) // max(1, args.steps),
           "d2h_bytes_per_step": (c1["d2h_bytes"] - c0["d2h_bytes"]) // max(1, args.steps),
           "p50_ms": float(np.median(lat)), "p95_ms": float(np.percentile(lat, 95))}
    r0 = reqs[0]
    line = {"metric": "decisions/s", "value": value, "unit": "decisions/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic (seeded random-init weights and token ids)",
            "p50_ms": e2e["p50_ms"],
            "config": {"workload": f"{cfg.name}: batch of {len(reqs)} requests, each a {r0.prefix_rows}-row state "
                                   f"prefix + {len(r0.questions)} x {len(r0.questions[0].suffix)}-token questions",
                       "model": cfg.name, "decisions_per_step": dec, "parallelism": f"replicas x{ws}",
                       "cuda_graphs": not args.no_graphs, "path": "fused batch (s1_prefill_decide_batch_async)",
                       "class_ms_per_step": {k: round(v["ms"] / max(1, args.steps), 4) for k, v in prof.items()}},
            "roofline": roofline, "clocks": clk.summary(), "gpu_launches": int(launches), "e2e": e2e}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = time_oracle(cfg, W, r0, budget_s=float(os.environ.get("S1_CPU_BUDGET", "25")))
    if rank == 0:
        print(json.dumps(line), flush=True)
    for s_ in states:
        s_.close()
    model.close()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="4b")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel", choices=["gemm", "gdn", "attn"], help="time one kernel entry point alone")
    ap.add_argument("--path", default="fused", choices=["fused", "two-call"],
                    help="fused: s1_prefill_decide (one sweep); two-call: s1_prefill_state + s1_decide")
    ap.add_argument("--shape", default="1024,18432,2560,3")
    ap.add_argument("--no-graphs", action="store_true", help="no CUDA graphs for the stream-ordered one-sweep call")
    args = ap.parse_args()
    if args.kernel:
        return run_kernel(args)
    from prefill_only_decision_gb300 import configs
    cfg = configs.CONFIGS[args.config]
    if args.impl == "reference":
        return run_reference(args, cfg)

    import ctypes as C
    import torch

    ws, rank, local = dist_setup()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if cfg.work.n_requests > 1 and cfg.name != "27b":
        rc = run_batch(args, cfg, torch, ws, rank, local)
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return rc
    from prefill_only_decision_gb300 import binding, synth

    W = synth.make_weights(cfg)
    reqs = synth.make_requests(cfg)
    req = reqs[0]
    # a stream of its own (CUDA graphs cannot capture the legacy default stream)
    stream = torch.cuda.Stream()
    binding.use_torch_allocator()
    model = binding.Model(W, stream=stream.cuda_stream)
    if not args.no_graphs:
        model.set_graphs(True)   # repeated stream-ordered calls replay a captured graph
    n_q = len(req.questions)
    P = req.prefix_rows

    # ---- stream-ordered path, ids resident in device memory --------------------------------
    st = model.state_create(P)
    d_tok = torch.from_numpy(req.tokens).cuda()
    d_emb = torch.from_numpy(req.embeds.view(np.int16)).cuda() if req.embeds is not None else None
    dq = []
    for q in req.questions:
        dq.append((torch.from_numpy(q.suffix).cuda(), torch.from_numpy(q.option_ids).cuda(), q.type))
    qarr = (binding.Question * n_q)()
    for j, (s, o, t) in enumerate(dq):
        qarr[j] = binding.Question(t, C.cast(C.c_void_p(s.data_ptr()), C.POINTER(C.c_int32)), s.numel(),
                                   C.cast(C.c_void_p(o.data_ptr()), C.POINTER(C.c_int32)), o.numel())
    n_opt = sum(len(q.option_ids) for q in req.questions)
    d_probs = torch.zeros(n_opt, dtype=torch.float32, device="cuda")
    d_stats = torch.zeros((n_q, 8), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()   # inputs made on the default stream are ready for the model's stream

    def step_two_call():
        model.prefill_async(st, d_tok.data_ptr(), len(req.tokens), d_emb.data_ptr() if d_emb is not None else 0,
                            0 if d_emb is None else d_emb.shape[0])
        model.decide_async(st, qarr, n_q, d_probs.data_ptr(), d_stats.data_ptr(), 0)

    def step_fused():
        model.prefill_decide_async(st, d_tok.data_ptr(), len(req.tokens), qarr, n_q, d_probs.data_ptr(),
                                   d_stats.data_ptr(), 0, d_emb.data_ptr() if d_emb is not None else 0,
                                   0 if d_emb is None else d_emb.shape[0])

    step = step_fused if args.path == "fused" else step_two_call

    def barrier():
        torch.cuda.synchronize()
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(max(3, args.warmup)):
        step()
    model.sync()
    # the two-call path with an event between its phases, and one fused step (outside the timed loop)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for _ in range(2):
        step_two_call()
    ev[0].record(stream)
    model.prefill_async(st, d_tok.data_ptr(), len(req.tokens), d_emb.data_ptr() if d_emb is not None else 0,
                        0 if d_emb is None else d_emb.shape[0])
    ev[1].record(stream)
    model.decide_async(st, qarr, n_q, d_probs.data_ptr(), d_stats.data_ptr(), 0)
    ev[2].record(stream)
    step_fused()
    ev[3].record(stream)
    model.sync()
    t_prefill, t_decide, t_fused = ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2]), ev[2].elapsed_time(ev[3])

    # ---- decide phase alone (questions over the cached prefix): the weight-streaming regime ----
    # every projection weight is read once per call while only the questions' rows are computed,
    # so its roofline is HBM bandwidth over the model's weight bytes (bf16, LoRA merged)
    weight_bytes = sum(a.size * 2 for layer in W.layers for a in layer if a is not None and a.ndim == 2)
    dts = []
    nvtx_dec = os.environ.get("S1_NVTX") == "1"   # lets ncu --nvtx-include "decide/" select these calls
    for _ in range(15):
        if nvtx_dec:
            torch.cuda.nvtx.range_push("decide")
        ev[1].record(stream)
        model.decide_async(st, qarr, n_q, d_probs.data_ptr(), d_stats.data_ptr(), 0)
        ev[2].record(stream)
        if nvtx_dec:
            torch.cuda.nvtx.range_pop()
        model.sync()
        dts.append(ev[1].elapsed_time(ev[2]))
    t_dec = float(np.median(dts))
    hbm_peak = load_peaks()["hbm_gbs"]
    decide_rows = sum(len(q.suffix) for q in req.questions)
    decide_roofline = {"bound": "hbm", "phase": f"s1_decide_async: {n_q} question(s), {decide_rows} rows over "
                                                 f"the cached {P}-row prefix",
                       "weight_bytes": int(weight_bytes), "ms": t_dec,
                       "achieved": weight_bytes / (t_dec / 1000.0) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                       "frac": weight_bytes / (t_dec / 1000.0) / 1e9 / hbm_peak,
                       "peak_source": load_peaks()["source"] + " HBM copy"}

    launches0 = model.counters()["launches"]
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nvtx = os.environ.get("S1_NVTX") == "1"     # lets ncu --nvtx-include "timed/" select the timed steps
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        clk.mark_start()
        if nvtx:
            torch.cuda.nvtx.range_push("timed")
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        if nvtx:
            torch.cuda.nvtx.range_pop()
        barrier()
        torch.cuda.synchronize()
        clk.mark_end()
    ms_total = e0.elapsed_time(e1)
    launches = (model.counters()["launches"] - launches0) // max(1, args.steps)
    model.sync()
    from prefill_only_decision_gb300 import replicas
    ms_total = replicas.max_over_ranks(ms_total, device="cuda")
    ms_step = ms_total / max(1, args.steps)
    value = ws * n_q * args.steps / (ms_total / 1000.0)

    # ---- roofline of the dominant kernel (tensor-core GEMM), profiled over the same steps ----
    model.profile(True)
    for _ in range(args.steps):
        step()
    prof = model.profile_read()
    model.profile(False)
    peaks = load_peaks()
    g = prof["gemm"]
    achieved = g["flops"] / (g["ms"] / 1000.0) / 1e12 if g["ms"] > 0 else 0.0
    peak, peak_source = tensor_peak(peaks, ms_total)
    total_prof_ms = sum(v["ms"] for v in prof.values())
    step_flops = g["flops"] / max(1, args.steps)
    traffic = GEMM_DRAM_BYTES_PER_LAUNCH.get(cfg.name)
    roofline = {"bound": "tensor", "kernel": "gemm_kernel / gemm_pair_kernel (tcgen05, all projections)",
                "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak if peak else None,
                "traffic": traffic,
                "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum, "
                                "mean over the timed step's GEMM launches, warm caches)",
                "algorithmic_bytes_per_launch": g["bytes"] / max(1, g["count"]),
                "peak_source": peak_source,
                "share_of_step": g["ms"] / total_prof_ms if total_prof_ms else None,
                "launches_per_step": g["count"] / max(1, args.steps),
                "flops_per_step": step_flops,
                "step_achieved": step_flops / (ms_step / 1000.0) / 1e12,
                "step_frac": step_flops / (ms_step / 1000.0) / 1e12 / peak if peak else None}
    phase_split = {k: round(v["ms"] / max(1, args.steps), 4) for k, v in prof.items()}

    # ---- end to end through the blocking public API (host buffers) ---------------------------
    model.sync()
    c0 = model.counters()
    lat = []
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        a = time.perf_counter()
        if args.path == "fused":
            model.prefill_decide(req, want_hidden=False)
        else:
            s2 = model.prefill(req.tokens, req.embeds)
            model.decide(s2, req.questions, want_hidden=False)
            s2.close()
        lat.append((time.perf_counter() - a) * 1000.0)
    barrier()
    e2e_s = time.perf_counter() - t0
    c1 = model.counters()
    e2e = {"value": ws * n_q * args.steps / e2e_s, "unit": "decisions/s",
           "h2d_bytes_per_step": (c1["h2d_bytes"] - c0["h2d_bytes"]) // max(1, args.steps),
           "d2h_bytes_per_step": (c1["d2h_bytes"] - c0["d2h_bytes"]) // max(1, args.steps),
           "p50_ms": float(np.median(lat)), "p95_ms": float(np.percentile(lat, 95))}

    line = {"metric": "decisions/s", "value": value, "unit": "decisions/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic (seeded random-init weights and token ids)",
            "p50_ms": e2e["p50_ms"],
            "config": {"workload": f"{cfg.name}: 1 request, {P}-row state prefix + {n_q} x "
                                   f"{len(req.questions[0].suffix)}-token questions",
                       "model": "4B-class hybrid decoder (24 gated delta-rule + 8 GQA layers, d 2560, "
                                "FFN 9216, LoRA r32 merged)" if cfg.name.startswith("4b") else cfg.name,
                       "decisions_per_step": n_q, "parallelism": f"replicas x{ws}",
                       "cuda_graphs": not args.no_graphs,
                       "l2": "inputs larger than L2 (weights read every step)",
                       "path": args.path + (" (s1_prefill_decide_async)" if args.path == "fused"
                                            else " (s1_prefill_async + s1_decide_async)"),
                       "one_step_ms": {"two_call_prefill": round(t_prefill, 4), "two_call_decide": round(t_decide, 4),
                                       "fused": round(t_fused, 4)},
                       "class_ms_per_step": phase_split},
            "roofline": roofline, "decide_roofline": decide_roofline, "clocks": clk.summary(),
            "gpu_launches": int(launches), "e2e": e2e}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = time_oracle(cfg, W, req, budget_s=float(os.environ.get("S1_CPU_BUDGET", "25")))
    if rank == 0:
        print(json.dumps(line), flush=True)
    st.close()
    model.close()
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
