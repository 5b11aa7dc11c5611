#!/usr/bin/env python
"""Benchmark of the MTP decode step of the DSA layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one pass of the whole hot path over the verify workload (32
requests x 8192 cached tokens, 6 verify rows each, 128 query heads, bf16
576-wide latent, FP8 64 x 128 indexer, top-2048): ragged merge, FP8 query
quantization, indexer scores + top-k, sparse MLA, greedy acceptance,
accepted-segment write-back into the draft-layer caches, and the 4-step
shared-index draft loop (indexer + top-k at step 0, sparse MLA at every step).
The metric is verify rows per second.  Inputs are resident in HBM; L2 is
flushed (a 512 MB write) before every timed step and each step is timed with
CUDA events on its stream.  `e2e` is the same metric with every step's inputs
copied from pinned host memory and its outputs copied back inside the timed
region.  With --gpus N > 1 (torchrun) each rank runs its own replica of the
workload (weak scaling, no collective on the data path) and the slowest
rank's time counts.

--impl reference times the CPU oracle (the reference arm of this
benchmark) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MTP verify rows/s (DSA indexer+top-k+sparse MLA); % HBM roofline on 1 GB300"
WORKLOAD = "verify"
WORKLOAD_DESC = ("verify step, 1 layer: 32 requests x 8192 cached tokens, 6 verify rows each (1 + 5 drafts), "
                 "128 query heads, bf16 576-d latent, FP8 e4m3 64x128 indexer with block-128 scales, top-k 2048; "
                 "plus merge, greedy acceptance, draft-layer write-back and a 4-step shared-index draft loop "
                 "over the same requests")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-sample", type=float, default=0.0, help=argparse.SUPPRESS)
    return ap.parse_args()


# ----------------------------------------------------------------------------- distributed

def dist_setup(n):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = tempfile.mktemp(suffix=".csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- peaks

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm": d["hbm_gbs"], "bf16": d["bf16_tflops"], "bf16_sus": d["bf16_tflops_sustained"],
                "src": "measured"}
    return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sus": 1700.0, "src": "fallback"}


# ----------------------------------------------------------------------------- CPU oracle

def oracle_rows(seconds: float, max_rows: int):
    """Run the oracle over the first verify rows of the workload until
    `seconds` of CPU time pass; returns (rows, elapsed)."""
    from mtp_speculative_decode_gb300 import workloads as W
    from oracle.pipeline import OracleStep
    w = W.build(WORKLOAD)
    o = OracleStep(w)
    t0 = time.perf_counter()
    n = 0
    for r in range(min(max_rows, w.R)):
        sc = o.verify_scores([r])
        tk = o.verify_topk(sc)
        o.verify_mla(tk)
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    return n, time.perf_counter() - t0


def cpu_baseline_subprocess(seconds: float):
    """The oracle timed in a fresh process on all host cores."""
    cores = os.cpu_count() or 1
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = str(cores)
    env["CUDA_VISIBLE_DEVICES"] = ""
    res = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-sample", str(seconds)],
                         capture_output=True, text=True, env=env, timeout=600)
    line = [x for x in res.stdout.splitlines() if x.startswith("{")]
    if res.returncode != 0 or not line:
        return {"error": (res.stderr or res.stdout)[-300:]}
    d = json.loads(line[-1])
    return {"value": d["rows"] / d["seconds"], "unit": "rows/s", "cores": cores, "kind": "oracle",
            "sample": f"first {d['rows']} verify rows of the workload (indexer scores + top-k + sparse MLA "
                      f"per row, float64 numpy), {d['seconds']:.1f} s"}


# ----------------------------------------------------------------------------- our arm

def run_ours(a, world, rank, local):
    import numpy as np
    import torch

    from mtp_speculative_decode_gb300 import pipeline, roofline
    from mtp_speculative_decode_gb300 import workloads as W

    dev = f"cuda:{local}"
    stream = torch.cuda.current_stream()
    w = W.build(WORKLOAD)
    d = W.draft_tensors(w)
    g = pipeline.DecodeStep(w, dev, d)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)

    for _ in range(max(a.warmup, 3)):
        g.step()
    torch.cuda.synchronize()
    if g.status.item() != 0:
        raise RuntimeError(f"device status {g.status.item()} after warm-up")

    # algorithmic work of the verify sparse-MLA launch (from this workload's own selection)
    sel = g.topk_idx.cpu().numpy()
    union = []
    for b in range(w.B):
        rows = sel[b * w.r:(b + 1) * w.r]
        union.append(len(np.unique(rows[rows >= 0])))
    n_sel = (sel >= 0).sum(axis=1)
    mla_flops = roofline.mla_flops(n_sel, w.spec.H_Q)
    mla_bytes = roofline.mla_bytes(union, w.R, w.spec.H_Q, w.spec.topk)
    vis_req = w.L + w.r
    idx_bytes = roofline.indexer_bytes(vis_req, w.R, w.spec.H_I, w.spec.D_I)

    ev = lambda: torch.cuda.Event(enable_timing=True)
    phases = ["verify_indexer_topk", "verify_mla", "accept_writeback", "draft_indexer_topk", "draft_mla"]
    t_phase = {p: [] for p in phases}
    t_step = []
    clocks = ClockSampler(torch.cuda.current_device())
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    for _ in range(a.steps):
        flush.zero_()
        e = [ev() for _ in range(7)]
        e[0].record(stream)
        g.merge()
        g.verify_indexer()
        e[1].record(stream)
        g.verify_mla()
        e[2].record(stream)
        g.accept()
        g.writeback()
        e[3].record(stream)
        g.draft_indexer()
        e[4].record(stream)
        for j in range(w.spec.draft_steps):
            g.draft_mla(j)
        e[5].record(stream)
        torch.cuda.synchronize()
        t_step.append(e[0].elapsed_time(e[5]))
        for i, p in enumerate(phases):
            t_phase[p].append(e[i].elapsed_time(e[i + 1]))
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms_step = max_over_ranks(statistics.mean(t_step), world)
    value = world * w.R / (ms_step / 1e3)

    # end to end: inputs from pinned host memory, outputs back, inside the timed region
    e2e = None
    if not a.no_e2e:
        ins = [g.prompt_tokens, g.draft_tokens, g.target_argmax, g.q_idx_raw, g.w_idx, g.q_mla,
               g.src_latent, g.src_idxk, g.src_idxs, g.d_q_idx_raw, g.d_w_idx] + list(g.d_q_mla)
        outs = [g.out, g.lse, g.num_accepted, g.next_tokens] + list(g.d_out) + list(g.d_lse)
        h_in = [t.cpu().pin_memory() for t in ins]
        h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
        bi = sum(t.numel() * t.element_size() for t in h_in)
        bo = sum(t.numel() * t.element_size() for t in h_out)
        t_e2e = []
        for it in range(a.warmup + a.steps):
            flush.zero_()
            s, f = ev(), ev()
            s.record(stream)
            for dt, ht in zip(ins, h_in):
                dt.copy_(ht, non_blocking=True)
            g.step()
            for ht, dt in zip(h_out, outs):
                ht.copy_(dt, non_blocking=True)
            f.record(stream)
            torch.cuda.synchronize()
            if it >= a.warmup:
                t_e2e.append(s.elapsed_time(f))
        ms_e2e = max_over_ranks(statistics.mean(t_e2e), world)
        e2e = {"value": world * w.R / (ms_e2e / 1e3), "unit": "rows/s", "ms_per_step": ms_e2e,
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo}

    pk = peaks()
    ms_mla = statistics.mean(t_phase["verify_mla"])
    achieved = mla_flops / (ms_mla / 1e3) / 1e12
    t_hbm = mla_bytes / (pk["hbm"] * 1e9)
    traffic = _traffic_from_profile()
    roof = {"kernel": "sparse_mla (verify)", "bound": "tensor", "achieved": achieved, "peak": pk["bf16_sus"],
            "unit": "TFLOP/s", "frac": achieved / pk["bf16_sus"], "peak_source": pk["src"] + " sustained bf16",
            "traffic": traffic, "algorithmic_flops": mla_flops, "algorithmic_bytes": mla_bytes,
            "hbm_frac": (mla_bytes / (ms_mla / 1e3) / 1e9) / pk["hbm"], "ms": ms_mla,
            "t_hbm_ms": t_hbm * 1e3, "t_tensor_ms": mla_flops / (pk["bf16_sus"] * 1e12) * 1e3}
    out = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8e4m3+bf16 (fp32 accumulate)", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC, "B": w.B, "context": int(w.L[0]), "verify_rows": w.R,
                   "topk": w.spec.topk, "l2": "flushed (512 MB write) before every timed step",
                   "parallelism": f"replicas x{world}"},
        "clocks": clk, "e2e": e2e, "gpu_launches": a.steps * g.launches_per_step(),
        "roofline": roof,
        "phases_ms": {p: statistics.mean(v) for p, v in t_phase.items()},
        "indexer_algorithmic_bytes": idx_bytes,
    }
    return out


def _traffic_from_profile():
    """DRAM bytes per launch of the profiled kernel (profiles/traffic.json),
    or None when there is no capture or the kernel source changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        src = os.path.join(ROOT, d["source"])
        with open(src, "rb") as f:
            if hashlib.sha1(f.read()).hexdigest() != d["source_sha1"]:
                return None
        return d.get("sparse_mla_verify_dram_bytes")
    except Exception:
        return None


# ----------------------------------------------------------------------------- reference arm

def run_reference(a, world, rank):
    if rank != 0:
        return None
    from mtp_speculative_decode_gb300 import workloads as W
    from oracle.pipeline import OracleStep
    w = W.build(WORKLOAD)
    o = OracleStep(w)
    rows_per_step = w.r      # one request's verify rows per step: a bounded sample
    times = []
    for it in range(a.warmup + a.steps):
        rows = [((it * rows_per_step) + i) % w.R for i in range(rows_per_step)]
        t0 = time.perf_counter()
        sc = o.verify_scores(rows)
        tk = o.verify_topk(sc)
        o.verify_mla(tk)
        dt = time.perf_counter() - t0
        if it >= a.warmup:
            times.append(dt)
    ms = statistics.mean(times) * 1e3
    value = rows_per_step / (ms / 1e3)
    cores = os.cpu_count() or 1
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC, "sample": f"{rows_per_step} verify rows (one request) per step"},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows_per_step} verify rows per step: indexer + top-k + sparse MLA"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    a = parse()
    if a.cpu_sample > 0:
        n, s = oracle_rows(a.cpu_sample, 10 ** 9)
        print(json.dumps({"rows": n, "seconds": s}))
        return
    world, rank, local = dist_setup(a.gpus)
    if a.impl == "reference":
        out = run_reference(a, world, rank)
        if rank == 0:
            print(json.dumps(out))
        return
    cpu = None
    if rank == 0 and not a.no_cpu:
        cpu = cpu_baseline_subprocess(15.0)     # before the first GPU call of this process
    out = run_ours(a, world, rank, local)
    if rank == 0:
        out["cpu_baseline"] = cpu
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
