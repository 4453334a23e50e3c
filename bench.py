#!/usr/bin/env python3
"""Benchmark: one Medusa draft-and-verify step on one B300 (per rank).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload vicuna7b-b1]

A step = medusa_heads -> tree_attention -> lm_verify -> verify_accept ->
compact_kv on the seeded synthetic workload (default: the Vicuna-7B-shaped
batch-1 workload, d=4096, V=32000, 32 heads x 128, K=4, tree (4,3,2,2),
prefix 2048, typical acceptance).  Inputs are resident in HBM; each step's
bytes (about 0.8 GB) exceed the 126 MB L2, so no L2 flush is inserted.  The
prefix length is restored before every step (one 4-byte device copy), so
every timed step verifies against the same prefix length.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle on this host instead (a bounded sample of the same workload).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import medusa_synth as ms  # noqa: E402

METRIC = "Medusa draft+verify steps/s"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return dict(hbm=float(j["hbm_gbs"]), bf16=float(j["bf16_tflops"]),
                    bf16_sustained=float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                    src="measured")
    return dict(hbm=6400.0, bf16=1800.0, bf16_sustained=1400.0, src="fallback")


def step_bytes(w, N):
    """Algorithmic HBM bytes of one step (bf16): each weight and the prefix
    KV read once, small activations and outputs added."""
    e = 2 if w.dtype == "bf16" else 4
    d, V, K, B = w.d, w.V, w.K, w.B
    qkv = (w.Hq + 2 * w.Hkv) * w.dh * d * e
    wo = d * w.Hq * w.dh * e
    return dict(heads=K * d * d * e, lm=V * d * e, qkv=qkv, wo=wo)


PROFILE_VERIFY = os.path.join(ROOT, "profiles", "gemm_verify_vicuna7b-b1.md")
GEMM_SOURCE = os.path.join(ROOT, "speculative_decoding_08_b300", "csrc", "gemm_tc.cu")


def profiled_traffic():
    """DRAM bytes (read + write) per launch of the verify-pass GEMM from the
    committed ncu summary, or None when the summary is missing or was taken
    on another version of the kernel source (its sha256 is recorded there)."""
    import hashlib
    import re
    try:
        text = open(PROFILE_VERIFY).read()
        src = hashlib.sha256(open(GEMM_SOURCE, "rb").read()).hexdigest()
    except OSError:
        return None
    m_hash = re.search(r"gemm_tc\.cu sha256:\s*([0-9a-f]{64})", text)
    m_bytes = re.search(r"DRAM bytes per launch \(read \+ write\):\s*([0-9]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != src:
        return None
    return int(m_bytes.group(1))


def lm_verify_bytes(w, N):
    e = 2 if w.dtype == "bf16" else 4
    rows = w.B * N
    return w.V * w.d * e + rows * w.d * e + rows * (4 * 4 + 4 + 4) + rows * 4


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        # raw samples go to MDS_CLOCKS_CSV when set (kept as evidence), else
        # to a temporary file
        self.path = os.environ.get("MDS_CLOCKS_CSV") or os.path.join(
            tempfile.gettempdir(), f"mds_clocks_gpu{index}_{os.getpid()}.csv")

    def start(self):
        try:
            d = os.path.dirname(self.path)
            if d:
                os.makedirs(d, exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for ln in f:
                c = [v.strip() for v in ln.split(",")]
                if len(c) < 9:
                    continue
                try:
                    sm.append(float(c[1]))
                    smax = float(c[2])
                except ValueError:
                    continue
                for nm, v in zip(names, c[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def oracle_sample(w, x, budget_s=15.0, steps=50, warmup=0, warmup_budget_s=30.0):
    """Time the fp64 oracle's step on this host: up to `warmup` untimed steps
    (at most ~warmup_budget_s), then up to `steps` timed steps (at most
    ~budget_s, at least one).  Returns (cpu_baseline dict, timed steps,
    seconds, warm-up steps run)."""
    import oracle
    try:
        from threadpoolctl import threadpool_info
        cores = max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except Exception:
        cores = os.cpu_count() or 1
    f = {k: ms.as_f64(x[k], w.dtype) for k in ("h", "W", "lm", "emb", "wq", "wk", "wv", "wo")}
    f["kc"] = ms.as_f64(x["kc"][:1], w.dtype)
    f["vc"] = ms.as_f64(x["vc"][:1], w.dtype)
    f["h"] = f["h"][:1]
    mode = "greedy" if w.accept == "greedy" else "typical"
    nw = 0
    t0 = time.perf_counter()
    while nw < warmup and time.perf_counter() - t0 < warmup_budget_s:
        oracle.step(w, f, x["P"][:1], mode, batch=[0])
        nw += 1
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle.step(w, f, x["P"][:1], mode, batch=[0])
        n += 1
        if time.perf_counter() - t0 >= budget_s or n >= steps:
            break
    dt = time.perf_counter() - t0
    # one oracle step processes one sequence; a GPU step processes B
    return dict(value=n / dt / w.B, unit="steps/s", cores=cores, kind="oracle",
                sample=f"{n} oracle step(s) of one sequence of {w.name} "
                       f"(scaled by 1/B={w.B} to whole-batch steps/s)"), n, dt, nw


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    x = ms.make_inputs(w)
    # W untimed warm-up steps, then K timed ones, each one oracle step of one
    # sequence; both legs are capped in time so that the run ends within a
    # few minutes (the line reports the counts actually run)
    cb, n, dt, nw = oracle_sample(w, x, budget_s=180.0, steps=max(1, args.steps),
                                  warmup=args.warmup, warmup_budget_s=30.0)
    line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "steps/s",
            "n_gpus": args.gpus, "steps": n, "warmup": nw, "ms_per_step": 1e3 * dt / n,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "B": w.B, "d": w.d, "V": w.V,
                                            "K": w.K, "shortlist": list(w.shortlist),
                                            "prefix": list(w.P)},
            "cpu_baseline": cb, "e2e": {"value": cb["value"], "unit": "steps/s",
                                        "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def rank_max(values, dev):
    """Element-wise maximum over the ranks of a list of times: the slowest
    rank sets each whole-job time (a no-op without a process group)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=dev)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_rate(world, units_per_rank, seconds):
    """Units all ranks processed per second of the slowest rank."""
    return world * units_per_rank / seconds


def run_ours(args, w):
    import torch
    import torch.distributed as dist
    import speculative_decoding_08_b300 as mds
    from speculative_decoding_08_b300 import build as mbuild

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    if rank == 0 or world == 1:
        mbuild.build()
    if world > 1:
        dist.barrier()
    mds.load()
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    x = ms.make_inputs(w)

    def t(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    wt = {k: t(x[k]) for k in ("W", "lm", "emb", "wqkv", "wo", "kc", "vc")}
    P0 = torch.from_numpy(x["P"]).to(dev)
    P = P0.clone()
    h = t(x["h"])
    mode = 0 if w.accept == "greedy" else 1
    step = mds.MedusaStep(W=wt["W"], lm=wt["lm"], emb=wt["emb"], wqkv=wt["wqkv"], wo=wt["wo"],
                          Kc=wt["kc"], Vc=wt["vc"], P=P, shortlist=w.shortlist,
                          max_rank_sum=w.max_rank_sum, Hq=w.Hq, Hkv=w.Hkv, B=w.B)
    N = step.N

    def one():
        P.copy_(P0)
        step.run(h, mode=mode, eps=w.eps, delta=w.delta)

    s = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(s):
        for _ in range(max(args.warmup, 3)):
            one()
    s.synchronize()
    # capture the step in a CUDA graph
    g = torch.cuda.CUDAGraph()
    n0 = mds.launch_count()
    with torch.cuda.graph(g, stream=s):
        one()
    per_step_kernels = mds.launch_count() - n0
    for _ in range(max(args.warmup, 3)):
        g.replay()
    torch.cuda.synchronize()
    assert mds.status_check(step.ws) == 0, "device latched a data error"

    clocks = Clocks(dev.index)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(args.steps):
            g.replay()
        e1.record(s)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms_total = e0.elapsed_time(e1)

    # per-call device time: each C-ABI call alone, captured 10 times back to
    # back in a CUDA graph and replayed; CUDA events on the launching stream
    calls = ["medusa_heads", "tree_attention", "lm_verify", "verify_accept", "compact_kv"]
    fns = {
        "medusa_heads": lambda: mds.medusa_heads(h, step.W, step.lm, step.shortlist, step.smax,
                                                 step.U, step.root, step.topk_id,
                                                 step.topk_val, step.ws),
        "tree_attention": lambda: mds.tree_attention(
            step.P, step.tok, step.mask, step.emb, step.wqkv, step.wo, step.Kc, step.Vc,
            step.y, step.ws, Hq=step.Hq, Hkv=step.Hkv, K=step.K, smax=step.smax,
            root=step.root, topk_id=step.topk_id, depth=step.depth, rank=step.rank),
        "lm_verify": lambda: mds.lm_verify(step.y, step.lm, step.tok, step.parent, step.argmax,
                                           step.stats, step.childlogit, step.ws),
        "verify_accept": lambda: mds.verify_accept(mode, w.eps, w.delta, step.parent,
                                                   step.depth, step.tok, step.argmax,
                                                   step.stats, step.childlogit, step.L,
                                                   step.path, step.next_root, step.ws,
                                                   ok=step.ok),
        "compact_kv": lambda: (P.copy_(P0), mds.compact_kv(step.L, step.path, step.Kc,
                                                           step.Vc, step.P, step.ws)),
    }
    per = {}
    reps = 10
    with torch.cuda.stream(s):
        P.copy_(P0)
        for c in calls:
            gc = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gc, stream=s):
                for _ in range(reps):
                    fns[c]()
            gc.replay()
            s.synchronize()
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(s)
            for _ in range(3):
                gc.replay()
            ev1.record(s)
            s.synchronize()
            per[c] = ev0.elapsed_time(ev1) / (3 * reps)
            P.copy_(P0)
    clk = clocks.stop()

    # end to end through the public API with host buffers: every step copies
    # h in from pinned host memory, runs the step and copies the emitted
    # tokens (L, path, tree tokens, next_root) back to pinned host memory,
    # all inside the captured step (MedusaStep.capture with h_host and
    # outputs_to_host); the host waits for the step every time.  The prefix
    # length is restored before each step (one 4-byte device copy) so that
    # every step verifies against the same prefix.
    h_host = torch.empty_like(h, device="cpu").pin_memory()
    h_host.copy_(h.cpu())
    h_dev = torch.empty_like(h)
    with torch.cuda.stream(s):
        P.copy_(P0)
        step.capture(h_dev, mode=mode, eps=w.eps, delta=w.delta, h_host=h_host,
                     outputs_to_host=True)
    s.synchronize()
    outs = list(step.host_out.values())
    e2e_steps = max(args.steps, 10)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        with torch.cuda.stream(s):
            P.copy_(P0)
            step.replay()
        s.synchronize()
    e2e_dt = time.perf_counter() - t0
    h2d = h.numel() * h.element_size()
    d2h = sum(o.numel() * o.element_size() for o in outs)
    L_host = step.host_out["L"].numpy().copy()

    # max over ranks (device-timed steps and the end-to-end loop)
    ms_total, e2e_dt = rank_max([ms_total, e2e_dt], dev)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    ms_step = ms_total / args.steps
    steps_per_s = whole_job_rate(world, args.steps, ms_total / 1e3)
    mean_emit = float(np.mean(L_host + 1))
    pk = peaks()
    lmv_bytes = lm_verify_bytes(w, N)
    lmv_s = per["lm_verify"] / 1e3
    achieved = lmv_bytes / lmv_s / 1e9
    sb = step_bytes(w, N)
    prefix_bytes = int(np.sum(x["P"])) * w.Hkv * w.dh * 2 * (2 if w.dtype == "bf16" else 4)
    total_bytes = sb["heads"] + 2 * sb["lm"] + sb["qkv"] + sb["wo"] + prefix_bytes
    line = {
        "metric": METRIC, "value": steps_per_s, "unit": "steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic (seeded; value laws of the workload description)",
        "config": {"workload": w.name, "B": w.B, "d": w.d, "V": w.V, "Hq": w.Hq, "Hkv": w.Hkv,
                   "dh": w.dh, "K": w.K, "shortlist": list(w.shortlist),
                   "max_rank_sum": w.max_rank_sum, "prefix": list(w.P), "accept": w.accept,
                   "parallelism": f"replicas x{world}", "cuda_graph": True,
                   "l2": "per-step bytes (~%.0f MB) exceed the 126 MB L2; no flush" % (total_bytes / 1e6)},
        "accepted_tok_per_s": steps_per_s * w.B * mean_emit,
        "mean_tokens_per_step": mean_emit,
        "step_hbm_gbs": total_bytes / (ms_step / 1e3) / 1e9,
        "step_hbm_frac": total_bytes / (ms_step / 1e3) / 1e9 / pk["hbm"],
        "per_call_us": {c: 1e3 * v for c, v in per.items()},
        "roofline": {"kernel": "lm_verify call: k_gemm_tc<VERIFY> LM-projection stream over the "
                               "verify rows + its statistics merge and child-logit gather",
                     "bound": "hbm",
                     "achieved": achieved, "peak": pk["hbm"], "unit": "GB/s",
                     "frac": achieved / pk["hbm"], "traffic": profiled_traffic(),
                     "peak_src": pk["src"], "algorithmic_bytes_per_launch": lmv_bytes},
        "gpu_launches": per_step_kernels * args.steps,
        "clocks": clk,
        "e2e": {"value": whole_job_rate(world, e2e_steps, e2e_dt), "unit": "steps/s",
                "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
    }
    if not args.no_cpu_baseline:
        cb, _, _, _ = oracle_sample(w, x, budget_s=args.cpu_budget)
        line["cpu_baseline"] = cb
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="vicuna7b-b1")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    w = ms.workload(args.workload)
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
