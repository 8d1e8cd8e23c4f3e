"""Write ``gpt2_124m_accum32_curve.json``: the oracle's loss curve over the
first two optimizer steps of the GPT-2 124M gradient-accumulation workload.

The workload ("Let's reproduce GPT-2 (124M)", §Video özeti: gradient
accumulation, AdamW, warmup + cosine learning rate): 32 micro-steps of
B=16, T=1024 per optimizer step (524,288 tokens), the loss of a step is the
mean of its micro-steps' losses, the gradient is the mean of theirs, then
global-norm clipping at 1.0 and AdamW (betas 0.9 / 0.95, eps 1e-8, weight
decay 0.1 on 2-D weights) at the schedule's learning rate for that step.
Tokens are the Zipf(1.1) stream of seed 2, micro-step i reading window i.

Only ``oracle/`` computes anything here (``synthetic`` draws the tokens).
Each micro-step is split into its 16 sequences: the micro-step loss is the
mean of the 16 per-sequence losses and the gradient of one sequence is taken
with weight 1/(16*32), which is the same quantity as the batched form in
exact arithmetic (sequences do not interact in the forward).  Sequences run
in a pool of single-threaded worker processes (started with ``spawn``).

The file records, per step, the learning rate, the mean loss, the 32
micro-step losses and (step 1) the pre-clip gradient norm, together with a
SHA-256 of the code it was computed with: the source text of every oracle
and input-generator function the curve depends on, the oracle's constants
and its C initialiser.  A test that reads the file recomputes that hash and
fails if any of it changed.

Usage: ``python tests/golden/make_accum32_curve.py [--workers N] [--scratch DIR]``
(about two hours on five cores).  ``--scratch`` keeps the step-1 result so
that an interrupted run resumes at step 2.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import multiprocessing as mp
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

OUT = os.path.join(HERE, "gpt2_124m_accum32_curve.json")
HASHED_FILES = ["oracle/init_rng.c"]
HASHED_ORACLE = ["Config", "param_specs", "init_params", "layernorm_forward", "layernorm_backward", "gelu_forward",
                 "gelu_derivative", "_causal_scores", "causal_attention_forward", "causal_attention_backward",
                 "cross_entropy_forward", "cross_entropy_backward", "embedding_backward", "_split_heads",
                 "_merge_heads", "_attention_per_sequence", "model_forward", "model_backward", "global_norm",
                 "lr_schedule", "OracleGPT2"]
HASHED_CONSTANTS = ["F64", "LN_EPS", "GELU_K", "GELU_C"]
HASHED_SYNTHETIC = ["sm64", "draws", "unit_open0", "zipf_cdf", "zipf_tokens", "zipf_window"]
ADAMW = dict(beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1, clip=1.0)
MICRO = 32
STEPS = 2


def source_hash() -> str:
    """SHA-256 of the code and constants the curve depends on."""
    import inspect

    import synthetic
    from oracle import gpt2 as og

    h = hashlib.sha256()

    def put(tag, text):
        h.update(tag.encode() + b"\0" + text.encode() + b"\0")

    for rel in HASHED_FILES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            put(rel, f.read().decode())
    for name in HASHED_ORACLE:
        put("oracle." + name, inspect.getsource(getattr(og, name)))
    for name in HASHED_CONSTANTS:
        put("oracle." + name, repr(getattr(og, name)))
    for name in HASHED_SYNTHETIC:
        put("synthetic." + name, inspect.getsource(getattr(synthetic, name)))
    for name in ("_GAMMA", "_M1", "_M2", "STREAM_ZIPF"):
        put("synthetic." + name, repr(getattr(synthetic, name)))
    put("workload", repr(sorted(synthetic.WORKLOADS["gpt2_124m_accum32"].items())))
    return h.hexdigest()


def _workload():
    import synthetic

    return dict(synthetic.WORKLOADS["gpt2_124m_accum32"])


_P = None  # per-worker parameters


def _init_worker(params_path):
    global _P
    import torch

    torch.set_num_threads(1)
    from oracle import gpt2 as og

    w = _workload()
    if params_path is None:
        _P = og.init_params(og.Config.from_dict(dict(w, B=1)), w["seed"])
    else:
        _P = torch.load(params_path)


def _run_chunk(args):
    """Losses (and summed weighted gradients) of a list of (micro_step, b)."""
    items, want_grad = args
    import torch

    import synthetic
    from oracle import gpt2 as og

    w = _workload()
    cfg = og.Config.from_dict(dict(w, B=1))
    losses = {}
    G = None
    for i, b in items:
        x, y = synthetic.zipf_window(w["seed"], w["B"], w["T"], w["V"], micro_step=i)
        loss, _, cache = og.model_forward(cfg, _P, x[b:b + 1], y[b:b + 1])
        losses[(i, b)] = float(loss)
        if want_grad:
            g = og.model_backward(cfg, _P, cache, 1.0 / (w["B"] * MICRO))
            if G is None:
                G = g
            else:
                for k in G:
                    G[k] += g[k]
        del cache
    return losses, G


def _pass(step, params_path, want_grad, workers):
    """One optimizer step's micro-steps over the pool: (per-micro-step losses, gradient)."""
    w = _workload()
    items = [(step * MICRO + i, b) for i in range(MICRO) for b in range(w["B"])]
    nchunk = workers * 4
    chunks = [(items[c::nchunk], want_grad) for c in range(nchunk)]
    losses, G = {}, None
    ctx = mp.get_context("spawn")
    with ctx.Pool(workers, initializer=_init_worker, initargs=(params_path,)) as pool:
        for n, (ls, g) in enumerate(pool.imap_unordered(_run_chunk, chunks)):
            losses.update(ls)
            if g is not None:
                if G is None:
                    G = g
                else:
                    for k in G:
                        G[k] += g[k]
            print("  step %d: chunk %d/%d done (%s)" % (step + 1, n + 1, nchunk, time.strftime("%H:%M:%S")),
                  flush=True)
    micro = [sum(losses[(step * MICRO + i, b)] for b in range(w["B"])) / w["B"] for i in range(MICRO)]
    return micro, G


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workers", type=int, default=5)
    ap.add_argument("--scratch", default=None, help="directory for the resumable step-1 result")
    a = ap.parse_args()
    import torch

    from oracle import gpt2 as og

    w = _workload()
    cfg = og.Config.from_dict(dict(w, B=1))
    digest = source_hash()
    steps = []
    ref = og.OracleGPT2(cfg, w["seed"])
    ck = os.path.join(a.scratch, "accum32_step1_%s.pt" % digest[:16]) if a.scratch else None
    if ck and os.path.exists(ck):
        saved = torch.load(ck)
        steps.append(saved["step"])
        ref.params = saved["params"]
        print("resumed step 1 from", ck, flush=True)
    else:
        t0 = time.time()
        micro, G = _pass(0, None, True, a.workers)
        for k in ref.grads:
            ref.grads[k] = G[k]
        lr = og.lr_schedule(0)
        norm = ref.clip_and_adamw(lr, ADAMW["beta1"], ADAMW["beta2"], ADAMW["eps"], ADAMW["wd"], ADAMW["clip"])
        steps.append(dict(step=1, lr=lr, loss=sum(micro) / MICRO, micro_losses=micro, grad_norm=norm))
        print("step 1: loss %.6f norm %.6f (%.0f s)" % (steps[0]["loss"], norm, time.time() - t0), flush=True)
        if ck:
            os.makedirs(a.scratch, exist_ok=True)
            torch.save(dict(step=steps[0], params=ref.params), ck)
    # step 2: the loss at the updated parameters (forward only)
    if ck:
        params_path = ck + ".params"
    else:
        import tempfile

        params_path = os.path.join(tempfile.mkdtemp(), "params.pt")
    torch.save(ref.params, params_path)
    t0 = time.time()
    micro, _ = _pass(1, params_path, False, a.workers)
    steps.append(dict(step=2, lr=og.lr_schedule(1), loss=sum(micro) / MICRO, micro_losses=micro, grad_norm=None))
    print("step 2: loss %.6f (%.0f s)" % (steps[1]["loss"], time.time() - t0), flush=True)
    doc = dict(workload="gpt2_124m_accum32", seed=w["seed"], B=w["B"], T=w["T"], micro_steps=MICRO,
               adamw=ADAMW, lr_schedule="oracle.gpt2.lr_schedule(it), it = step - 1",
               sources_sha256=digest, steps=steps)
    assert all(math.isfinite(s["loss"]) for s in steps)
    with open(OUT, "w") as f:
        json.dump(doc, f, indent=1)
    print("wrote", OUT)


if __name__ == "__main__":
    main()
