#!/usr/bin/env python
"""Benchmark of the MTP decode step of the DSA layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config decode|verify|draft|long|tiny] [--no-sub]

A step is one pass of the whole hot path over one batch of the chosen
workload (default ``decode``: 128 ragged requests, contexts log-uniform in
[1024, 131072]): ragged merge of 1 + 5 tokens per request, FP8 query
quantization, indexer scores, top-2048, sparse MLA over the 6 verify rows,
greedy acceptance, write-back of the accepted segment into the draft-layer
caches, and the 4-step shared-index draft loop (indexer + top-k at step 0,
sparse MLA at every step).  ``value`` is verify rows per second of whole
steps.  The same line carries, under ``configs``, the verify (32 x 8192),
draft-loop (64 x 32768, draft rows/s) and long-context (8 requests up to 1M)
workloads, the draft loop over the FP8 latent cache and with draft_extend
seeding, a 4-layer verify with the cross-layer indexer schedule, and
rejection-sampling acceptance over a 154880-token vocabulary, each with its
own timing and roofline.

Inputs are resident in HBM; L2 is flushed (a 512 MB write) before every timed
step; every step is timed with CUDA events on its stream: a first pass times
whole steps (the headline), a second pass puts events between the phases
(merge | scores | top-k | MLA | ...) for the breakdown and the rooflines.
`e2e` is the headline metric with every step's inputs copied from pinned host
memory and its outputs copied back inside the timed region.  With --gpus N > 1
(torchrun) each rank runs its own replica (weak scaling, no collective on the
data path) and the slowest rank's time counts.

--impl reference times the CPU oracle (the reference arm of this benchmark) on
a bounded sample of the same workload.
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
DEFAULT = "decode"
BASE = ("tiny", "verify", "draft", "long", "decode")      # workloads of workloads.build (headline candidates)
SUBS = ("verify", "draft", "long", "draft_fp8", "draft_seeded", "verify_layered", "verify_paged", "accept_stochastic")
DESC = {
    "tiny": "2 requests (contexts 100, 300), 4 verify rows each, 8 query heads, float32 latent, float32 4x64 "
            "indexer, top-k 32, 4 shared-index draft steps",
    "verify": "verify step, 1 layer: 32 requests x 8192 cached tokens, 6 verify rows each (1 + 5 drafts), "
              "128 query heads, bf16 576-d latent, FP8 e4m3 64x128 indexer with block-128 scales, top-k 2048; "
              "plus merge, greedy acceptance, draft-layer write-back and a 4-step shared-index draft loop",
    "draft": "draft loop with index_share_for_mtp_iteration, 1 sparse NextN layer: 64 requests x 32768 context; "
             "write-back of the accepted rows, then 4 one-row draft forwards (indexer + top-2048 at step 0, "
             "steps 1-3 on the shared indices plus the appended positions)",
    "long": "long-context ragged verify, 1 layer: 8 requests with contexts log-uniform in [4096, 1048576], "
            "6 verify rows each, full FP8 indexer scan, top-2048, sparse MLA over 128 heads",
    "decode": "full decode-step ledger, 1 target layer + 1 draft layer: 128 ragged requests with contexts "
              "log-uniform in [1024, 131072]; merge of 1 + 5 tokens, 6-row verify (FP8 64x128 indexer, top-2048, "
              "sparse MLA over 128 heads of the 576-d bf16 latent), greedy acceptance (mean accept length about "
              "2.76), draft-layer write-back, 4 shared-index draft steps",
    "draft_fp8": "the draft loop (64 requests x 32768 context) over the FP8 latent cache: 656-byte rows "
                 "(512 E4M3 + 4 float32 scales + 64 bf16 rope) instead of 1152-byte bf16 rows",
    "draft_seeded": "the draft loop (64 requests x 32768) with seed_dsa_topk_from_draft_extend: draft_extend's "
                    "attention over the 6 window rows (indexer, top-2048, sparse MLA), its selection at the last "
                    "accepted row seeds all 4 draft steps (no step-0 indexer)",
    "verify_layered": "verify (32 requests x 8192, 6 rows) over 4 DSA layers with the cross-layer indexer "
                      "schedule full, shared, shared, shared: one indexer + top-k, four sparse MLA",
    "verify_paged": "the verify workload (32 requests x 8192, 6 rows, write-back, 4-step shared-index draft loop) "
                    "over paged caches: pages of 64 tokens in shuffled order, one block table shared by the target "
                    "and draft layers; adds the window's slot plan and the accepted-KV move, and writes back by slot",
    "accept_stochastic": "rejection-sampling acceptance: 128 requests x 5 drafts over the 154880-token "
                         "vocabulary (synthetic softmax rows), draw from the residual of the first rejected row",
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=[c for c in DESC if c not in SUBS or c in BASE], default=DEFAULT)
    ap.add_argument("--no-sub", action="store_true", help="only the chosen workload")
    ap.add_argument("--subs", default="", help="comma-separated sub-workloads to run (default: all)")
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


# ----------------------------------------------------------------------------- peaks and profiles

def peaks():
    """Measured peaks of the GB300s: HBM copy bandwidth and cuBLAS bf16 (burst for kernels timed
    on their own, sustained for seconds-long loops).  FP8 dense is taken as 2x the bf16 figure (the
    nominal ratio of the two tensor rates)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm": d["hbm_gbs"], "bf16": d["bf16_tflops"], "bf16_sus": d["bf16_tflops_sustained"],
                "src": "measured"}
    return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sus": 1700.0, "src": "fallback"}


def _sources_sha1(paths):
    h = hashlib.sha1()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profile_record(key):
    """A kernel's ncu figures from profiles/ncu_metrics.json, or None when the entry is missing or
    any source that compiles into the kernel changed since the capture."""
    p = os.path.join(ROOT, "profiles", "ncu_metrics.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p)).get(key)
        if not d or _sources_sha1(d["sources"]) != d["sources_sha1"]:
            return None
        return d
    except Exception:
        return None


# ----------------------------------------------------------------------------- CPU oracle

def oracle_rows(config: str, seconds: float, max_rows: int):
    """Run the oracle over the first verify rows (draft rows for the draft loop) of the workload until
    `seconds` pass; returns (rows, elapsed)."""
    from mtp_speculative_decode_gb300 import workloads as W
    from oracle.pipeline import OracleStep
    w = W.build(config)
    o = OracleStep(w, W.draft_tensors(w))
    t0 = time.perf_counter()
    n = 0
    if w.spec.verify:
        for r in range(min(max_rows, w.R)):
            sc = o.verify_scores([r])
            tk = o.verify_topk(sc)
            o.verify_mla(tk)
            n += 1
            if time.perf_counter() - t0 >= seconds:
                break
    else:
        n_acc, _ = o.accept()
        for b in range(min(max_rows, w.B)):
            _, s0 = o.draft_step0(n_acc, [b])
            for j in range(w.spec.draft_steps):
                o.draft_mla(n_acc, s0, j, [b])
                n += 1
            if time.perf_counter() - t0 >= seconds:
                break
    return n, time.perf_counter() - t0


def cpu_baseline_subprocess(config: str, seconds: float):
    """The oracle timed in a fresh process on all host cores."""
    cores = os.cpu_count() or 1
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = str(cores)
    env["CUDA_VISIBLE_DEVICES"] = ""
    res = subprocess.run([sys.executable, os.path.abspath(__file__), "--config", config,
                          "--cpu-sample", str(seconds)], capture_output=True, text=True, env=env, timeout=900)
    line = [x for x in res.stdout.splitlines() if x.startswith("{")]
    if res.returncode != 0 or not line:
        return {"error": (res.stderr or res.stdout)[-300:]}
    d = json.loads(line[-1])
    what = "verify rows (indexer scores + top-k + sparse MLA per row)" if config != "draft" else \
        "draft rows (step-0 indexer + top-k per request, then sparse MLA per draft step)"
    return {"value": d["rows"] / d["seconds"], "unit": "rows/s", "cores": cores, "kind": "oracle",
            "sample": f"first {d['rows']} {what} of the {config} workload, float64 numpy, {d['seconds']:.1f} s"}


# ----------------------------------------------------------------------------- our arm

def work_model(g, w):
    """Algorithmic bytes and flops of the step's kernels, from this workload's own selections."""
    import numpy as np

    from mtp_speculative_decode_gb300 import roofline
    if w is None:   # rejection-sampling acceptance
        n_acc = g.num_accepted.cpu().numpy()
        return {"accept_stochastic": {"rows": g.B, "flops": 0.0,
                                      "bytes": roofline.accept_stochastic_bytes(g.B, g.K, g.V, n_acc)}}
    spec = w.spec
    m = {}
    if hasattr(g, "layers"):   # layered verify: per full layer the indexer, per layer the MLA
        vis_row = w.row_pos + 1
        vis_req = w.L + w.r
        for l, L in enumerate(g.layers):
            if L["type"] == "full":
                m[f"L{l}_scores"] = {"rows": w.R, "bytes": roofline.indexer_bytes(vis_req, w.R, spec.H_I, spec.D_I),
                                     "flops": roofline.indexer_flops(vis_row, spec.H_I, spec.D_I), "dtype": "fp8"}
                m[f"L{l}_topk"] = {"bytes": int(np.sum(vis_row)) * 8, "flops": 0.0}
            sel = g.layers[L["src"]]["topk"].cpu().numpy()
            union = [len(np.unique(sel[b * w.r:(b + 1) * w.r][sel[b * w.r:(b + 1) * w.r] >= 0])) for b in range(w.B)]
            m[f"L{l}_mla"] = {"rows": w.R, "bytes": roofline.mla_bytes(union, w.R, spec.H_Q, spec.topk),
                              "flops": roofline.mla_flops((sel >= 0).sum(axis=1), spec.H_Q), "dtype": "bf16"}
        return m
    row_bytes = roofline.FP8_LATENT_ROW_BYTES if getattr(g, "latent_fp8", False) else roofline.LATENT_ROW_BYTES
    if spec.verify:
        vis_row = w.row_pos + 1
        vis_req = w.L + w.r
        m["verify_scores"] = {"rows": w.R, "bytes": roofline.indexer_bytes(vis_req, w.R, spec.H_I, spec.D_I),
                              "flops": roofline.indexer_flops(vis_row, spec.H_I, spec.D_I), "dtype": "fp8"}
        m["verify_topk"] = {"bytes": int(np.sum(vis_row)) * 8, "flops": 0.0}
        sel = g.topk_idx.cpu().numpy()
        union = [len(np.unique(sel[b * w.r:(b + 1) * w.r][sel[b * w.r:(b + 1) * w.r] >= 0])) for b in range(w.B)]
        m["verify_mla"] = {"rows": w.R, "bytes": roofline.mla_bytes(union, w.R, spec.H_Q, spec.topk, row_bytes),
                           "flops": roofline.mla_flops((sel >= 0).sum(axis=1), spec.H_Q), "dtype": "bf16"}
    if spec.draft_steps and getattr(g, "seeded", False):
        Wn = spec.K + 1
        vis = (np.repeat(w.L, Wn) + np.tile(np.arange(Wn), w.B) + 1)
        m["extend_scores"] = {"rows": w.B * Wn, "bytes": roofline.indexer_bytes(w.L + Wn, w.B * Wn, spec.H_I, spec.D_I),
                              "flops": roofline.indexer_flops(vis, spec.H_I, spec.D_I), "dtype": "fp8"}
        m["extend_topk"] = {"bytes": int(np.sum(vis)) * 8, "flops": 0.0}
        xs = g.x_topk.cpu().numpy()
        union = [len(np.unique(xs[b * Wn:(b + 1) * Wn][xs[b * Wn:(b + 1) * Wn] >= 0])) for b in range(w.B)]
        m["extend_mla"] = {"rows": w.B * Wn, "bytes": roofline.mla_bytes(union, w.B * Wn, spec.H_Q, spec.topk, row_bytes),
                           "flops": roofline.mla_flops((xs >= 0).sum(axis=1), spec.H_Q), "dtype": "bf16"}
        n_sel = (g.shared_idx.cpu().numpy() >= 0).sum(axis=1)
        for j in range(spec.draft_steps):
            m[f"draft_mla{j}"] = {"rows": w.B, "bytes": roofline.mla_bytes(n_sel + j + 1, w.B, spec.H_Q, spec.topk, row_bytes),
                                  "flops": roofline.mla_flops(n_sel + j + 1, spec.H_Q), "dtype": "bf16"}
    elif spec.draft_steps:
        P = g.next_pos.cpu().numpy()
        m["draft_scores"] = {"rows": w.B, "bytes": roofline.indexer_bytes(P + 1, w.B, spec.H_I, spec.D_I),
                             "flops": roofline.indexer_flops(P + 1, spec.H_I, spec.D_I), "dtype": "fp8"}
        m["draft_topk"] = {"bytes": int(np.sum(P + 1)) * 8, "flops": 0.0}
        n_sel = (g.shared_idx.cpu().numpy() >= 0).sum(axis=1)
        for j in range(spec.draft_steps):
            m[f"draft_mla{j}"] = {"rows": w.B, "bytes": roofline.mla_bytes(n_sel + j, w.B, spec.H_Q, spec.topk, row_bytes),
                                  "flops": roofline.mla_flops(n_sel + j, spec.H_Q), "dtype": "bf16"}
    return m


def kernel_roofline(model, ms, pk, burst=True):
    """Where one launch sits: HBM fraction of its algorithmic bytes and tensor fraction of its
    algorithmic flops (FP8 against 2x the bf16 peak)."""
    bf16 = pk["bf16"] if burst else pk["bf16_sus"]
    tpeak = bf16 * (2.0 if model.get("dtype") == "fp8" else 1.0)
    gbs = model["bytes"] / (ms / 1e3) / 1e9
    tfs = model["flops"] / (ms / 1e3) / 1e12
    out = {"ms": ms, "algorithmic_bytes": model["bytes"], "hbm_gbs": gbs, "hbm_frac": gbs / pk["hbm"]}
    if model["flops"]:
        out.update({"algorithmic_flops": model["flops"], "tflops": tfs, "tensor_peak": tpeak,
                    "tensor_frac": tfs / tpeak, "tensor_peak_source": f"{pk['src']} "
                    f"{'burst' if burst else 'sustained'} bf16" + (" x2 (fp8)" if model.get("dtype") == "fp8" else "")})
    return out


def path_roofline(model, phase_ms, names, pk, what):
    b = sum(model[n]["bytes"] for n in names if n in model and not n.endswith("topk"))
    t = sum(phase_ms[n] for n in names)
    gbs = b / (t / 1e3) / 1e9
    return {"what": what, "algorithmic_bytes": b, "ms": t, "hbm_gbs": gbs, "hbm_frac": gbs / pk["hbm"],
            "peak_gbs": pk["hbm"], "peak_source": pk["src"] + " copy bandwidth"}


def measure(config, a, world, local, e2e: bool, clocks_on: bool):
    import torch

    from mtp_speculative_decode_gb300 import pipeline
    from mtp_speculative_decode_gb300 import workloads as W

    dev = f"cuda:{local}"
    stream = torch.cuda.current_stream()
    t_build = time.perf_counter()
    if config == "draft_fp8":
        w = W.build("draft")
        g = pipeline.DecodeStep(w, dev, W.draft_tensors(w), latent_fp8=True)
    elif config == "draft_seeded":
        w = W.add_draft_extend(W.build("draft"))
        g = pipeline.DecodeStep(w, dev, W.draft_tensors(w), seeded=True)
    elif config == "verify_layered":
        w = W.add_layers(W.build("verify"), 4)
        g = pipeline.LayeredVerify(w, ["full", "shared", "shared", "shared"], dev)
    elif config == "verify_paged":
        w = W.build("verify")
        g = pipeline.DecodeStep(w, dev, W.draft_tensors(w), page_size=64)
    elif config == "accept_stochastic":
        w = None
        g = pipeline.StochasticAccept(128, 5, 154880, dev)
    else:
        w = W.build(config)
        g = pipeline.DecodeStep(w, dev, W.draft_tensors(w))
    torch.cuda.synchronize()
    t_build = time.perf_counter() - t_build
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    phases = g.phases()

    for _ in range(max(a.warmup, 3)):
        g.step()
    torch.cuda.synchronize()
    if g.status.item() != 0:
        raise RuntimeError(f"{config}: device status {g.status.item()} after warm-up")

    ev = lambda: torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch.cuda.current_device()) if clocks_on else None
    barrier(world)
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
    # pass 1: whole steps
    t_step = []
    for _ in range(a.steps):
        flush.zero_()
        s, f = ev(), ev()
        s.record(stream)
        g.step()
        f.record(stream)
        torch.cuda.synchronize()
        t_step.append(s.elapsed_time(f))
    # pass 2: events between the phases
    t_ph = {n: [] for n, _ in phases}
    for _ in range(a.steps):
        flush.zero_()
        e = [ev() for _ in range(len(phases) + 1)]
        e[0].record(stream)
        for i, (_, fn) in enumerate(phases):
            fn()
            e[i + 1].record(stream)
        torch.cuda.synchronize()
        for i, (n, _) in enumerate(phases):
            t_ph[n].append(e[i].elapsed_time(e[i + 1]))
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop() if clocks else None
    if g.status.item() != 0:
        raise RuntimeError(f"{config}: device status {g.status.item()} after the timed steps")
    ms_step = max_over_ranks(statistics.mean(t_step), world)
    phase_ms = {n: statistics.mean(v) for n, v in t_ph.items()}

    pk = peaks()
    model = work_model(g, w)
    res = {"workload": DESC[config], "name": config, "ms_per_step": ms_step, "phases_ms": phase_ms,
           "build_s": t_build, "launches_per_step": g.launches_per_step(), "clocks": clk}
    if w is None:
        res["metric"] = "requests/s (acceptance of 5 drafts per request)"
        res["value"] = world * g.B / (ms_step / 1e3)
        res["unit"] = "requests/s"
        res["mean_accept_length"] = float(g.num_accepted.float().mean().item()) + 1.0
        res["roofline"] = {n: kernel_roofline(m, phase_ms[n], pk) for n, m in model.items()}
        res["_g"], res["_w"], res["_model"], res["_flush"] = g, w, model, flush
        return res
    spec = w.spec
    if config == "verify_layered":
        res["metric"] = "verify rows/s (whole steps, 4 layers)"
        res["value"] = world * w.R / (ms_step / 1e3)
        res["unit"] = "rows/s"
        res["roofline"] = {n: kernel_roofline(m, phase_ms[n], pk) for n, m in model.items() if n in phase_ms}
        res["_g"], res["_w"], res["_model"], res["_flush"] = g, w, model, flush
        return res
    if spec.verify:
        res["metric"] = "verify rows/s (whole steps)"
        res["value"] = world * w.R / (ms_step / 1e3)
        vnames = ["verify_scores", "verify_topk", "verify_mla"]
        res["verify_path_rows_per_s"] = world * w.R / (sum(phase_ms[n] for n in vnames) / 1e3)
    else:
        res["metric"] = "draft rows/s (whole steps)"
        res["value"] = world * w.B * spec.draft_steps / (ms_step / 1e3)
    res["unit"] = "rows/s"
    roof = {}
    for n, mdl in model.items():
        if n in phase_ms:
            roof[n] = kernel_roofline(mdl, phase_ms[n], pk)
    if spec.verify:
        roof["verify_path"] = path_roofline(model, phase_ms, ["verify_scores", "verify_topk", "verify_mla"], pk,
                                            "verify indexer + top-k + sparse MLA: (indexer + MLA algorithmic "
                                            "bytes) / (scores + top-k + MLA time)")
    if spec.draft_steps:
        dn = (["extend_scores", "extend_topk", "extend_mla"] if getattr(g, "seeded", False) else
              ["draft_scores", "draft_topk"]) + [f"draft_mla{j}" for j in range(spec.draft_steps)]
        roof["draft_path"] = path_roofline(model, phase_ms, dn, pk,
                                           "draft loop: (indexer + MLA algorithmic bytes) / (its scores + "
                                           "top-k + MLA time)")
    rec = profile_record("indexer_tc_kernel")
    roof["indexer_tensor_pipe_ncu"] = None if rec is None else {
        k: rec[k] for k in ("tensor_pipe_active_pct", "workload", "capture") if k in rec}
    res["roofline"] = roof
    res["_g"] = g
    res["_w"] = w
    res["_model"] = model
    res["_flush"] = flush
    return res


def headline_roofline(res, pk):
    """The contract's roofline object for the kernel with the largest share of the step."""
    phase_ms = res["phases_ms"]
    model = res["_model"]
    cand = [n for n in model if n in phase_ms and (n.endswith("mla0") or n.endswith("mla") or n.endswith("scores"))]
    # draft MLA steps are separate launches of one kernel: compare the kernels' largest single launch
    top = max(cand or [n for n in model if n in phase_ms], key=lambda n: phase_ms[n])
    mdl, ms = model[top], phase_ms[top]
    tpeak = pk["bf16"] * (2.0 if mdl.get("dtype") == "fp8" else 1.0)
    t_hbm = mdl["bytes"] / (pk["hbm"] * 1e9)
    t_tc = mdl["flops"] / (tpeak * 1e12)
    kern = ("sparse_mla_tc_kernel" if "mla" in top else "indexer_tc_kernel" if "scores" in top
            else "accept_stochastic_kernel")
    rec = profile_record(kern)
    traffic = None
    if rec and rec.get("dram_bytes") and rec.get("algorithmic_bytes"):
        # the captured launch's DRAM bytes per algorithmic byte, applied to this launch's algorithmic bytes
        traffic = rec["dram_bytes"] / rec["algorithmic_bytes"] * mdl["bytes"]
    if t_tc >= t_hbm:
        achieved = mdl["flops"] / (ms / 1e3) / 1e12
        out = {"bound": "tensor", "achieved": achieved, "peak": tpeak, "unit": "TFLOP/s", "frac": achieved / tpeak,
               "peak_source": f"{pk['src']} burst bf16" + (" x2 (fp8)" if mdl.get("dtype") == "fp8" else "")}
    else:
        achieved = mdl["bytes"] / (ms / 1e3) / 1e9
        out = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm"], "unit": "GB/s", "frac": achieved / pk["hbm"],
               "peak_source": f"{pk['src']} copy bandwidth"}
    out.update({"traffic": traffic, "kernel": f"{kern} ({top} launch of the {res['name']} workload)",
                "algorithmic_bytes": mdl["bytes"], "algorithmic_flops": mdl["flops"], "ms": ms,
                "hbm_frac": mdl["bytes"] / (ms / 1e3) / 1e9 / pk["hbm"],
                "traffic_source": None if traffic is None else rec.get("capture")})
    return out


def run_e2e(res, a, world):
    """The headline metric end to end: every step's inputs from pinned host memory and its outputs back
    to pinned host memory inside the timed region."""
    import torch
    g, w, flush = res["_g"], res["_w"], res["_flush"]
    stream = torch.cuda.current_stream()
    ins = [g.q_idx_raw, g.w_idx, g.q_mla, g.target_argmax]
    outs = [g.num_accepted, g.next_tokens]
    if w.spec.verify:
        ins += [g.prompt_tokens, g.draft_tokens]
        outs += [g.out, g.lse]
    if g.has_draft:
        ins += [g.src_latent, g.src_idxk, g.d_q_idx_raw, g.d_w_idx] + list(g.d_q_mla)
        if g.src_idxs is not None:
            ins.append(g.src_idxs)
        outs += list(g.d_out) + list(g.d_lse)
    h_in = [t.cpu().pin_memory() for t in ins]
    h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    bi = sum(t.numel() * t.element_size() for t in h_in)
    bo = sum(t.numel() * t.element_size() for t in h_out)
    ev = lambda: torch.cuda.Event(enable_timing=True)
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
    ms = max_over_ranks(statistics.mean(t_e2e), world)
    units = w.R if w.spec.verify else w.B * w.spec.draft_steps
    return {"value": world * units / (ms / 1e3), "unit": "rows/s", "ms_per_step": ms,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo}


def _public(res):
    return {k: v for k, v in res.items() if not k.startswith("_")}


def run_ours(a, world, rank, local):
    import torch
    pk = peaks()
    head = measure(a.config, a, world, local, e2e=True, clocks_on=True)
    roof = headline_roofline(head, pk)
    e2e = None if a.no_e2e else run_e2e(head, a, world)
    launches = a.steps * head["launches_per_step"]
    w = head["_w"]
    out = {
        "metric": METRIC, "value": head["value"], "unit": "rows/s", "n_gpus": world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8e4m3+bf16 (fp32 accumulate)", "data": "synthetic",
        "config": {"workload": head["workload"], "name": a.config, "B": w.B, "context_total": int(w.L.sum()),
                   "context_max": int(w.L.max()), "verify_rows": w.R if w.spec.verify else 0,
                   "topk": w.spec.topk, "l2": "flushed (512 MB write) before every timed step",
                   "parallelism": f"replicas x{world}"},
        "value_is": head["metric"],
        "clocks": head["clocks"], "e2e": e2e, "gpu_launches": launches,
        "roofline": roof,
        "phases_ms": head["phases_ms"],
        "rooflines": head["roofline"],
    }
    if "verify_path_rows_per_s" in head:
        out["verify_path_rows_per_s"] = head["verify_path_rows_per_s"]
    for k in ("_g", "_w", "_model", "_flush"):
        head.pop(k)
    del head
    torch.cuda.empty_cache()
    subs = {}
    if not a.no_sub and a.config == DEFAULT:
        names = [n for n in a.subs.split(",") if n] or list(SUBS)
        for name in names:
            if name not in SUBS:
                raise SystemExit(f"unknown sub-workload {name}")
            r = measure(name, a, world, local, e2e=False, clocks_on=True)
            r["roofline_headline"] = headline_roofline(r, pk)
            for k in ("_g", "_w", "_model", "_flush"):
                r.pop(k)
            subs[name] = _public(r)
            del r
            torch.cuda.empty_cache()
    out["configs"] = subs
    return out


# ----------------------------------------------------------------------------- reference arm

def run_reference(a, world, rank):
    if rank != 0:
        return None
    from mtp_speculative_decode_gb300 import workloads as W
    from oracle.pipeline import OracleStep
    w = W.build(a.config)
    o = OracleStep(w, W.draft_tensors(w))
    times, units = [], 0
    n_acc = None if w.spec.verify else o.accept()[0]
    for it in range(a.warmup + a.steps):
        t0 = time.perf_counter()
        if w.spec.verify:
            # one request's verify rows per step: a bounded sample
            b = it % w.B
            rows = list(range(b * w.r, (b + 1) * w.r))
            sc = o.verify_scores(rows)
            tk = o.verify_topk(sc)
            o.verify_mla(tk)
            units = len(rows)
        else:
            b = it % w.B
            _, s0 = o.draft_step0(n_acc, [b])
            for j in range(w.spec.draft_steps):
                o.draft_mla(n_acc, s0, j, [b])
            units = w.spec.draft_steps
        dt = time.perf_counter() - t0
        if it >= a.warmup:
            times.append(dt)
    ms = statistics.mean(times) * 1e3
    value = units / (ms / 1e3)
    cores = os.cpu_count() or 1
    what = "verify rows (one request's) per step: indexer + top-k + sparse MLA" if w.spec.verify else \
        "one request's 4 draft rows per step: step-0 indexer + top-k, sparse MLA per step"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": DESC[a.config], "name": a.config, "sample": what},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle", "sample": what},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    a = parse()
    if a.cpu_sample > 0:
        n, s = oracle_rows(a.config, a.cpu_sample, 10 ** 9)
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
        cpu = cpu_baseline_subprocess(a.config, 15.0)     # before the first GPU call of this process
    out = run_ours(a, world, rank, local)
    if rank == 0:
        out["cpu_baseline"] = cpu
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
