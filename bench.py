#!/usr/bin/env python
"""Throughput of the GPT-2 124M training step (bf16, B=16, T=1024) on B300s.

One step = zero_grad, forward (with the fused classifier and the loss read
back), backward, and the fused global-norm clip + AdamW update: every kernel
of the hot path, over one batch of synthetic Zipf(1.1) tokens.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) each rank trains an independent replica on its own
batches (the step shards as data parallelism; this single-GPU build has no
gradient exchange), so per-GPU work is fixed: weak scaling.  Rank 0 prints one
JSON line.  ``--impl reference`` times the CPU oracle on the host cores on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthetic  # noqa: E402

METRIC = "GPT-2 124M train tokens/s and MFU on 1 B300 (bf16, B=16, T=1024)"
NOMINAL_BF16_TFLOPS = 2250.0  # B300 dense bf16 tensor peak (no sparsity)
FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def flops_per_token(w):
    """Algorithmic training FLOPs per token: 3x forward; LM head over V; causal attention."""
    L, C, V, T = w["L"], w["C"], w["V"], w["T"]
    fwd = 24.0 * L * C * C + 2.0 * C * V + 2.0 * C * (T + 1) * L
    return 3.0 * fwd


def flops_per_token_6n(w):
    """The 6N + 12 L C T convention (N = parameters without the position table, full T x T attention),
    reported beside the algorithmic count for comparison with published MFU figures."""
    L, C, V, T = w["L"], w["C"], w["V"], w["T"]
    n = V * C + L * (12 * C * C + 13 * C) + 2 * C
    return 6.0 * n + 12.0 * L * C * T


# AdamW learning rate of optimizer step `it` (0-based): linear warmup over 700
# steps to 6e-4, then cosine decay to 6e-5 at step 19073 (10B tokens / 524,288
# tokens a step), "Let's reproduce GPT-2 (124M)", §Video özeti.
LR_MAX, LR_MIN, LR_WARMUP, LR_HORIZON = 6e-4, 6e-5, 700, 19073


def lr_at(it):
    if it < LR_WARMUP:
        return LR_MAX * (it + 1) / LR_WARMUP
    if it > LR_HORIZON:
        return LR_MIN
    r = (it - LR_WARMUP) / (LR_HORIZON - LR_WARMUP)
    return LR_MIN + 0.5 * (1.0 + math.cos(math.pi * r)) * (LR_MAX - LR_MIN)


def workload_label(name, w, accum):
    return "%s: L=%d C=%d H=%d V=%d (Vp=%d) B=%d T=%d%s, %d micro-step(s) (fwd+bwd) + clip + AdamW per step" % (
        name, w["L"], w["C"], w["H"], w["V"], w["Vp"], w["B"], w["T"],
        ", GELU recompute" if w.get("recompute_gelu") else "", accum)


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK if k in d}, "measured"
    return dict(FALLBACK), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# DRAM traffic per GEMM launch of the step (dram__bytes_read.sum +
# dram__bytes_write.sum from ncu, one launch of each of the step's GEMM shapes,
# weighted by how often the step launches that shape).  It is a stored
# capture, not a measurement of this run, and is reported only while the GEMM
# sources hash to the ones that were captured.
GEMM_TRAFFIC = {
    "sources": ["gpt_decoder_only_train_b300/csrc/tc_gemm.cu", "gpt_decoder_only_train_b300/csrc/tc_gemm.cuh",
                "gpt_decoder_only_train_b300/csrc/common.cuh"],
    "workload": "gpt2_124m",
    "sha256": "ffb2b0d940636f3b58d2a5886e13260ecca3761adc6cee2861fd3ac139c9a4c7",
    "bytes_per_launch": 21.786e9 / 123,
}


def gemm_traffic():
    import hashlib

    h = hashlib.sha256()
    try:
        for f in GEMM_TRAFFIC["sources"]:
            with open(os.path.join(ROOT, f), "rb") as fh:
                h.update(fh.read())
    except OSError:
        return None
    return GEMM_TRAFFIC["bytes_per_launch"] if h.hexdigest() == GEMM_TRAFFIC["sha256"] else None


def _oracle_sample_steps(w, max_steps, min_s, budget_s, warmup=0):
    """Run the oracle step (fwd + bwd + clip + AdamW) on one full-length sequence of the
    workload (B=1, the workload's T, so attention keeps its share of the work) until
    max_steps steps or min_s seconds have passed, never starting a step that would end past
    budget_s.  Returns (timed steps, seconds, tokens per step, threads)."""
    import torch

    from oracle import gpt2 as og

    torch.set_num_threads(os.cpu_count() or 1)
    cfg = og.Config.from_dict(dict(w, B=1))
    T = w["T"]
    x, y = synthetic.zipf_window(w["seed"], 1, T, w["V"])
    m = og.OracleGPT2(cfg, w["seed"])

    def one(i):
        m.zero_grad()
        m.forward(x, y)
        m.backward(1.0)
        m.clip_and_adamw(lr_at(i))

    for i in range(warmup):
        one(i)
    t0 = time.perf_counter()
    steps = 0
    while steps < max_steps:
        one(warmup + steps)
        steps += 1
        el = time.perf_counter() - t0
        if el >= min_s or el + el / steps > budget_s:
            break
    return steps, time.perf_counter() - t0, T, torch.get_num_threads()


def rank_micro_steps(rank, nsteps, accum):
    """Stream-window indices of every micro-step a replica runs: [step][micro-step].  Replica r
    reads the windows after those of replicas 0..r-1, so no two replicas see the same tokens."""
    return [[(rank * nsteps + i) * accum + j for j in range(accum)] for i in range(nsteps)]


def max_over_ranks(ms, dist, device):
    """The slowest replica's time (the job's time), or ms itself on one process."""
    if dist is None:
        return ms
    import torch

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, steps, tokens_per_step, ms):
    """Whole-job tokens/s: the tokens of all replicas over the slowest replica's time."""
    return world * steps * tokens_per_step / (ms / 1e3)


def cpu_baseline(w, min_s=12.0, budget_s=30.0):
    """The oracle, as it stands, on a bounded sample of the workload (see _oracle_sample_steps)."""
    steps, el, tok, cores = _oracle_sample_steps(w, 10 ** 9, min_s, budget_s)
    return {"value": steps * tok / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": "GPT-2 fp64 oracle step (fwd+bwd+clip+AdamW) on 1 x %d Zipf tokens of the workload, "
                      "%d step(s) in %.1f s" % (tok, steps, el)}


def run_reference(args, w, rank, world):
    """The CPU oracle timed as the reference arm (rank 0 only): W untimed and up to K timed
    steps, each one full-length sequence of the workload, within a few minutes in all."""
    if rank != 0:
        return
    accum = int(w.get("grad_accum", 1))
    steps, el, tok, cores = _oracle_sample_steps(w, args.steps, float("inf"), 240.0, warmup=min(args.warmup, 1))
    value = steps * tok / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": steps, "warmup": min(args.warmup, 1),
        "ms_per_step": 1e3 * el / steps,
        "ms_per_step_note": "one sample step: the oracle step on 1 x %d tokens; the workload's own step "
                            "(%d tokens) would take about %.0f ms at this rate (extrapolated, not run)"
                            % (tok, w["B"] * w["T"] * accum, 1e3 * w["B"] * w["T"] * accum / value),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_label(args.workload, w, accum), "global_batch": w["B"] * accum,
                   "seq_len": w["T"], "parallelism": "host cores, rank 0 only"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": "%d step(s) of 1 x %d tokens of the workload in %.1f s" % (steps, tok, el)},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def attention_sweep(args):
    """The isolated causal attention workload: H=12, hd=64, B*T = 65,536 at T in {256, 1024, 2048,
    4096}; Q, K, V, dO ~ N(0,1) rounded to bf16 (seed 4).  Forward and backward are timed apart with
    CUDA events after warm-up (every operand is 100 MB, together above L2); FLOPs count the causal
    pairs: 4 hd T(T+1)/2 per head forward, twice that backward.  "bwd" is the backward the model
    runs (dS kept in a workspace, dQ formed from it); "bwd_recompute" the entry without that
    workspace (a second kernel recomputes S and dP per query block).  The oracle's naive attention
    (full T x T scores, float64) is timed at T=256 on the host cores as the CPU baseline."""
    import torch

    import gpt_decoder_only_train_b300 as g
    from gpt_decoder_only_train_b300 import build

    if args.warmup < 3:
        raise SystemExit("at least 3 warm-up steps are required")
    build.build()
    H, hd = 12, 64
    stream = torch.cuda.current_stream()
    rows = []
    launches0 = g.launch_count()
    for cfg in synthetic.ATTN_SWEEP:
        T, B = cfg["T"], cfg["B"]
        dev = [torch.from_numpy(a).to(torch.bfloat16).cuda() for a in synthetic.attention_operands(4, B, H, T, hd)]
        q, k, v, do = dev
        o = torch.empty_like(q)
        lse = torch.empty(B, H, T, dtype=torch.float32, device="cuda")
        dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
        scratch = torch.empty(B * H * T, dtype=torch.float32, device="cuda")
        ds = torch.empty(g.attention_backward_ds_bytes(B, T, H), dtype=torch.uint8, device="cuda")
        fwd = lambda: g.attention_forward(q, k, v, o, lse, B, T, H)
        bwd = lambda: g.attention_backward_ds(q, k, v, o, do, lse, dq, dk, dv, scratch, ds, B, T, H)
        bwd_rc = lambda: g.attention_backward(q, k, v, o, do, lse, dq, dk, dv, scratch, B, T, H)
        out = {"T": T, "B": B}
        for name, fn, mult in (("fwd", fwd, 1.0), ("bwd", bwd, 2.0), ("bwd_recompute", bwd_rc, 2.0)):
            for _ in range(args.warmup):
                fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            # at least --steps calls and at least 0.6 s, so that the clock sampler (every 200 ms)
            # records the timed region
            calls = max(args.steps, int(600.0 / max(e0.elapsed_time(e1), 1e-3)) + 1)
            with ClockSampler(0) as clk:
                e0.record(stream)
                for _ in range(calls):
                    fn()
                e1.record(stream)
                torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / calls
            flops = mult * 4.0 * hd * (T * (T + 1) / 2.0) * B * H
            out[name] = {"ms": ms, "tflops": flops / ms / 1e9, "calls": calls, "clocks": clk.summary()}
        rows.append(out)
        del dev, q, k, v, do, o, lse, dq, dk, dv, scratch, ds
        torch.cuda.empty_cache()
    launches = g.launch_count() - launches0
    line = {
        "metric": "causal attention fwd+bwd TFLOP/s (H=12, hd=64, B*T=65536, bf16, fp32 softmax statistics)",
        "unit": "TFLOP/s", "higher_is_better": True, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "dtype": "bf16", "data": "synthetic N(0,1) Q, K, V, dO (seed 4)",
        "value": min(r["fwd"]["tflops"] for r in rows), "value_note": "slowest forward of the sweep",
        "sweep": rows, "gpu_launches": launches,
        "config": {"workload": "isolated causal attention sweep, T in {256, 1024, 2048, 4096}, B*T = 65536",
                   "l2": "every operand is 100 MB (inputs larger than L2)"},
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = attention_cpu_baseline()
    print(json.dumps(line), flush=True)


def attention_cpu_baseline(min_s=5.0, budget_s=30.0):
    """The oracle's naive causal attention (forward + backward, float64, full T x T scores) at T=256
    on the host cores, on a sample of heads of the sweep's T=256 inputs."""
    import torch

    from oracle import gpt2 as og

    torch.set_num_threads(os.cpu_count() or 1)
    B, H, T, hd = 4, 12, 256, 64
    q, k, v, do = (torch.from_numpy(a).double().permute(0, 2, 1, 3).contiguous()
                   for a in synthetic.attention_operands(4, B, H, T, hd))
    t0 = time.perf_counter()
    n = 0
    while True:
        b = n % B
        og.causal_attention_forward(q[b], k[b], v[b])
        og.causal_attention_backward(q[b], k[b], v[b], do[b])
        n += 1
        el = time.perf_counter() - t0
        if el >= min_s or el + el / n > budget_s:
            break
    flops = 3.0 * 4.0 * hd * (T * (T + 1) / 2.0) * H * n
    return {"value": flops / el / 1e12, "unit": "TFLOP/s", "cores": torch.get_num_threads(), "kind": "oracle",
            "sample": "naive fp64 causal attention fwd+bwd, T=256, %d sequence(s) x 12 heads in %.1f s" % (n, el)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gpt2_124m", choices=sorted(synthetic.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fp8", action="store_true",
                    help="E4M3 block projections in the forward (fp8_forward); a separate line, not the headline")
    ap.add_argument("--fused-lm-head", action="store_true",
                    help="LM head fused with the cross-entropy, no logits buffer; a separate line, not the headline")
    ap.add_argument("--attention-sweep", action="store_true",
                    help="time the isolated causal attention workload instead of the training step")
    args = ap.parse_args()
    if args.attention_sweep:
        attention_sweep(args)
        return
    w = dict(synthetic.WORKLOADS[args.workload])
    if args.fp8:
        w["fp8_forward"] = 1
    if args.fused_lm_head:
        w["fused_lm_head"] = 1
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return

    import torch

    import gpt_decoder_only_train_b300 as g
    from gpt_decoder_only_train_b300 import build

    if args.warmup < 3:
        raise SystemExit("at least 3 warm-up steps are required")
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build.build()
    B, T = w["B"], w["T"]
    accum = int(w.get("grad_accum", 1))  # micro-steps (consecutive stream windows) per optimizer step
    BT = B * T * accum  # tokens per step
    nsteps = args.warmup + args.steps
    # independent batches per rank: the replica r reads stream windows offset by r
    xs, ys = [], []
    for row in rank_micro_steps(rank, nsteps, accum):
        for ms_ in row:
            x, y = synthetic.zipf_window(w["seed"], B, T, w["V"], micro_step=ms_)
            xs.append(x)
            ys.append(y)
    X = torch.from_numpy(np.stack(xs).reshape(nsteps, accum, B, T)).cuda()
    Y = torch.from_numpy(np.stack(ys).reshape(nsteps, accum, B, T)).cuda()
    stream = torch.cuda.current_stream()
    model = g.GPT2(w, seed=w["seed"], stream=stream)

    def step(i, x, y):
        """One optimizer step over x, y [accum, B, T]: the loss is the mean over its micro-steps."""
        model.zero_grad()
        loss = 0.0
        for j in range(accum):
            loss += model.forward(x[j], y[j]) / accum
            model.backward(1.0 / accum)
        norm = model.clip_and_adamw(lr_at(i), 0.9, 0.95, 1e-8, 0.1, 1.0)
        return loss, norm

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    losses = []
    for i in range(args.warmup):
        losses.append(step(i, X[i], Y[i])[0])
    # ---- timed region (device time, CUDA events on the model's stream)
    barrier()
    launches0 = g.launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        ev0.record(stream)
        for i in range(args.warmup, nsteps):
            losses.append(step(i, X[i], Y[i])[0])
        ev1.record(stream)
        barrier()
    launches = g.launch_count() - launches0
    ms = max_over_ranks(ev0.elapsed_time(ev1), dist, "cuda")
    ms_per_step = ms / args.steps
    value = job_throughput(world, args.steps, BT, ms)

    # ---- per-step and per-phase pass (same steps, events at the step and phase boundaries on the
    # model's stream): the median step and the forward / backward / optimizer split
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    barrier()
    for n, i in enumerate(range(args.warmup, nsteps)):
        model.zero_grad()
        ev[n][0].record(stream)
        model.forward(X[i][0], Y[i][0])
        ev[n][1].record(stream)
        model.backward(1.0 / accum)
        for j in range(1, accum):  # accumulation: the remaining pairs, timed as backward
            model.forward(X[i][j], Y[i][j])
            model.backward(1.0 / accum)
        ev[n][2].record(stream)
        model.clip_and_adamw(lr_at(i), 0.9, 0.95, 1e-8, 0.1, 1.0)
        ev[n][3].record(stream)
    barrier()
    step_ms = sorted(e[0].elapsed_time(e[3]) for e in ev)
    phases = {"forward": sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps,
              "backward": sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps,
              "clip_adamw": sum(e[2].elapsed_time(e[3]) for e in ev) / args.steps}

    # ---- per-launch timing pass (same steps, events around every launch) for the roofline
    model.profile(True)
    for i in range(args.warmup, nsteps):
        step(i, X[i], Y[i])
    prof = model.profile_read()
    model.profile(False)

    # ---- end to end through the public API: host buffers, copies inside the timed region
    Xh = torch.from_numpy(np.stack(xs).reshape(nsteps, accum, B, T)).pin_memory()
    Yh = torch.from_numpy(np.stack(ys).reshape(nsteps, accum, B, T)).pin_memory()
    xd = torch.empty(accum, B, T, dtype=torch.int32, device="cuda")
    yd = torch.empty_like(xd)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.warmup, nsteps):
        xd.copy_(Xh[i], non_blocking=True)
        yd.copy_(Yh[i], non_blocking=True)
        step(i, xd, yd)
    e1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist, "cuda")
    e2e_value = job_throughput(world, args.steps, BT, e2e_ms)

    if rank == 0:
        peaks, peak_src = read_peaks()
        fpt = flops_per_token(w)
        per_gpu = value / world
        mm_ms, mm_flops, mm_n = prof["matmul"]
        achieved = mm_flops / (mm_ms / 1e3) / 1e12 if mm_ms > 0 else None
        # The burst peak was measured over a short run at high clocks, the sustained one over
        # seconds under the power cap: a short timed region near the maximum SM clock is held
        # to the burst figure, a long or power-capped one to the sustained figure.
        clocks = clk.summary()
        near_max = (clocks["sm_mhz"] is not None and clocks["sm_max_mhz"]
                    and clocks["sm_mhz"] >= 0.9 * clocks["sm_max_mhz"])
        burst = ms / 1e3 < 2.0 and (near_max or clocks["sm_mhz"] is None)
        peak_key = "bf16_tflops" if burst else "bf16_tflops_sustained"
        peak = peaks[peak_key]
        kernels = {}
        for cat, (cms, work, n) in prof.items():
            if n == 0:
                continue
            unit = "TFLOP/s" if cat in ("matmul", "attention", "matmul_e4m3") else "GB/s"
            rate = (work / (cms / 1e3) / (1e12 if unit == "TFLOP/s" else 1e9)) if cms > 0 else None
            kernels[cat] = {"ms_per_step": cms / args.steps, "launches_per_step": n / args.steps,
                            "achieved": rate, "unit": unit}
        line = {
            "metric": METRIC,
            "value": value,
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms_per_step,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16+e4m3" if args.fp8 else "bf16",
            "data": "synthetic Zipf(1.1) tokens over V=50257, random-init weights (seeded)",
            "config": {"workload": workload_label(args.workload, w, accum), "global_batch": B * accum * world,
                       "seq_len": T,
                       "parallelism": "replicas x%d (no gradient exchange)" % world,
                       "l2": "inputs larger than L2 (9 GB arena per step)"},
            "mfu": {"flops_per_token": fpt, "vs_nominal_dense_bf16_2250": per_gpu * fpt / (NOMINAL_BF16_TFLOPS * 1e12),
                    "vs_measured_bf16_burst": per_gpu * fpt / (peaks["bf16_tflops"] * 1e12),
                    "flops_per_token_6n_12lct": flops_per_token_6n(w),
                    "vs_nominal_dense_bf16_2250_6n_12lct":
                        per_gpu * flops_per_token_6n(w) / (NOMINAL_BF16_TFLOPS * 1e12)},
            "roofline": {"kernel": "tcgen05 bf16 GEMM (all matmuls of the step)", "bound": "tensor",
                         "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": (achieved / peak) if achieved else None,
                         "frac_vs_burst": (achieved / peaks["bf16_tflops"]) if achieved else None,
                         "frac_vs_sustained": (achieved / peaks["bf16_tflops_sustained"]) if achieved else None,
                         "traffic": gemm_traffic() if args.workload == GEMM_TRAFFIC["workload"] else None,
                         "traffic_unit": "bytes per launch (DRAM read + write, ncu)",
                         "traffic_source": "stored ncu capture of the same GEMM sources (not measured in this run)",
                         "peak_source": "%s %s (timed region %.2f s, median SM clock %s MHz)"
                                        % (peak_src, peak_key, ms / 1e3, clocks["sm_mhz"]),
                         "launches_per_step": mm_n / args.steps,
                         "timing": "CUDA events around each launch, second pass over the same steps"},
            "kernels": kernels,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": 2 * BT * 4,
                    "d2h_bytes_per_step": 8},
            "gpu_launches": launches,
            "step_ms": {"median": step_ms[len(step_ms) // 2], "min": step_ms[0], "max": step_ms[-1],
                        "note": "a separate pass over the same steps, events at the step boundaries"},
            "phases_ms_per_step": dict(phases, note=(
                "forward = the first micro-step's forward (with the loss read back), backward = its backward "
                "plus the remaining micro-steps, clip_adamw = norm, clip and AdamW; a separate pass")),
            "clocks": clocks,
            "loss_first_last": [losses[0], losses[-1]],
        }
        if args.fp8:
            # E4M3 operands run at twice the bf16 tensor rate (nominal 4.5 vs 2.25 PFLOP/s dense)
            f8_ms, f8_flops, f8_n = prof["matmul_e4m3"]
            f8_ach = f8_flops / (f8_ms / 1e3) / 1e12 if f8_ms > 0 else None
            f8_peak = 2.0 * peak
            line["config"]["precision"] = ("E4M3 QKV / attention-output / FC / FC-output products in the forward "
                                           "(activations per row, weights per tensor); LM head, backward and "
                                           "optimizer bf16/fp32")
            line["roofline_e4m3"] = {
                "kernel": "tcgen05 kind::f8f6f4 GEMM (the forward's block projections)", "bound": "tensor",
                "achieved": f8_ach, "peak": f8_peak, "unit": "TFLOP/s",
                "frac": (f8_ach / f8_peak) if f8_ach else None,
                "peak_source": "%s %s x 2 (nominal E4M3 / bf16 dense ratio)" % (peak_src, peak_key),
                "launches_per_step": f8_n / args.steps}
        if args.fused_lm_head:
            line["config"]["lm_head"] = ("fused with the cross-entropy: row partials in the forward, logits "
                                         "recomputed in 8,192-position chunks in the backward (no full logits buffer)")
        if not (args.no_cpu_baseline or args.fp8 or args.fused_lm_head):  # the bf16 headline's baseline
            line["cpu_baseline"] = cpu_baseline(w)
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
