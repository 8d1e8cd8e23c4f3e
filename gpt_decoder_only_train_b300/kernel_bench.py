"""Time single kernels of the library through the op-level C ABI.

    python -m gpt_decoder_only_train_b300.kernel_bench matmul --M 16384 --N 50304 --K 768
    python -m gpt_decoder_only_train_b300.kernel_bench matmul --M 768 --N 768 --K 16384 --a-mn --b-mn --epi accum
    python -m gpt_decoder_only_train_b300.kernel_bench matmul-accum2 --M 768 --N 3072 --M2 3072 --N2 768 --K 16384
    python -m gpt_decoder_only_train_b300.kernel_bench attention --B 16 --T 1024 --H 12 [--bwd [--recompute]]
    python -m gpt_decoder_only_train_b300.kernel_bench classifier --N 16384 --V 50257 --Vp 50304
    python -m gpt_decoder_only_train_b300.kernel_bench layernorm --N 16384 --C 768
    python -m gpt_decoder_only_train_b300.kernel_bench attention-sweep
    python -m gpt_decoder_only_train_b300.kernel_bench generate --B 16 --prompt 32 --new 64 --top-k 50
    python -m gpt_decoder_only_train_b300.kernel_bench attention-fb --B 64 --T 1024 --H 12
    python -m gpt_decoder_only_train_b300.kernel_bench adamw
    python -m gpt_decoder_only_train_b300.kernel_bench matmul --M 16384 --N 3072 --K 768 --epi gelu --fp8

Inputs are seeded random bf16 on the device; each line reports the mean time
per launch (CUDA events, after warm-up) and the algorithmic FLOP/s or bytes/s.
`matmul-accum2` times two weight-gradient products in one grouped launch;
`attention --bwd` times the backward with the dS workspace (the model's),
`--recompute` the one without it.
Repeated launches reuse the same inputs, so operands smaller than L2 (126 MB)
may be served from L2.
"""
from __future__ import annotations

import argparse
import json
import sys

import torch

import gpt_decoder_only_train_b300 as g

EPIS = {"store": g.EPI_STORE, "residual": g.EPI_RESIDUAL, "gelu": g.EPI_GELU, "gelu_bwd": g.EPI_GELU_BWD,
        "accum": g.EPI_ACCUM_F32}


def _time(fn, iters, warmup):
    for _ in range(warmup):
        fn(0)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(iters):
        fn(i)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters


def bench_matmul_fp8(a):
    """E4M3 operands (row-scaled A, tensor-scaled B, both K-major), bf16 epilogue."""
    M, N, K = a.M, a.N, a.K
    gen = torch.Generator(device="cuda").manual_seed(0)
    A = torch.randn(M, K, device="cuda", generator=gen).to(torch.bfloat16)
    B = torch.randn(N, K, device="cuda", generator=gen).to(torch.bfloat16)
    qa = torch.empty(M, K, dtype=torch.uint8, device="cuda")
    qb = torch.empty(N, K, dtype=torch.uint8, device="cuda")
    ainv = torch.empty(M, device="cuda")
    binv = torch.empty(1, device="cuda")
    work = torch.empty(1, dtype=torch.int32, device="cuda")
    g.quantize_e4m3_rows(A, qa, ainv, M, K)
    g.quantize_e4m3_tensor(B, qb, binv, work)
    epi = EPIS[a.epi]
    D = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
    D2 = torch.empty_like(D) if epi == g.EPI_GELU else None
    R = torch.randn(M, N, device="cuda", generator=gen).to(torch.bfloat16) if epi == g.EPI_RESIDUAL else None
    bias = torch.randn(N, device="cuda", generator=gen)
    ms = _time(lambda i: g.matmul_e4m3(qa, ainv, qb, binv, D, M, N, K, epilogue=epi, D2=D2, R=R, bias=bias),
               a.iters, a.warmup)
    qms = _time(lambda i: g.quantize_e4m3_rows(A, qa, ainv, M, K), a.iters, a.warmup)
    return {"op": "matmul_e4m3", "M": M, "N": N, "K": K, "epi": a.epi, "ms": ms,
            "TFLOP/s": 2.0 * M * N * K / ms / 1e9, "quantize_rows_ms": qms,
            "quantize_rows_GB/s": (3.0 * M * K + 4 * M) / qms / 1e6}


def bench_matmul(a):
    if getattr(a, "fp8", False):
        return bench_matmul_fp8(a)
    M, N, K = a.M, a.N, a.K
    gen = torch.Generator(device="cuda").manual_seed(0)
    A = torch.randn(K if a.a_mn else M, M if a.a_mn else K, device="cuda", generator=gen).to(torch.bfloat16)
    B = torch.randn(K if a.b_mn else N, N if a.b_mn else K, device="cuda", generator=gen).to(torch.bfloat16)
    epi = EPIS[a.epi]
    D = torch.zeros(M, N, device="cuda", dtype=torch.float32 if epi == g.EPI_ACCUM_F32 else torch.bfloat16)
    D2 = torch.empty(M, N, device="cuda", dtype=torch.bfloat16) if epi == g.EPI_GELU else None
    R = torch.randn(M, N, device="cuda", generator=gen).to(torch.bfloat16) if epi in (g.EPI_RESIDUAL,
                                                                                        g.EPI_GELU_BWD) else None
    bias = torch.randn(N, device="cuda", generator=gen) if epi in (g.EPI_STORE, g.EPI_RESIDUAL, g.EPI_GELU) else None
    lda = M if a.a_mn else K
    ldb = N if a.b_mn else K

    def run(i):
        g.matmul(A, lda, not a.a_mn, B, ldb, not a.b_mn, D, N, M, N, K, epi, D2=D2, R=R, bias=bias)

    ms = _time(run, a.iters, a.warmup)
    flops = 2.0 * M * N * K
    return {"op": "matmul", "M": M, "N": N, "K": K, "a_major": "mn" if a.a_mn else "k",
            "b_major": "mn" if a.b_mn else "k", "epi": a.epi, "ms": ms, "TFLOP/s": flops / ms / 1e9}


def bench_matmul_accum2(a):
    """Two weight-gradient products (M0 x N0 and M1 x N1, both K) in one grouped launch."""
    K = a.K
    gen = torch.Generator(device="cuda").manual_seed(0)
    A0 = torch.randn(K, a.M, device="cuda", generator=gen).to(torch.bfloat16)
    B0 = torch.randn(K, a.N, device="cuda", generator=gen).to(torch.bfloat16)
    A1 = torch.randn(K, a.M2, device="cuda", generator=gen).to(torch.bfloat16)
    B1 = torch.randn(K, a.N2, device="cuda", generator=gen).to(torch.bfloat16)
    D0 = torch.zeros(a.M, a.N, device="cuda")
    D1 = torch.zeros(a.M2, a.N2, device="cuda")
    ms = _time(lambda i: g.matmul_accum2(A0, a.M, B0, a.N, D0, a.M, a.N, A1, a.M2, B1, a.N2, D1, a.M2, a.N2, K),
               a.iters, a.warmup)
    flops = 2.0 * K * (a.M * a.N + a.M2 * a.N2)
    return {"op": "matmul_accum2", "M0": a.M, "N0": a.N, "M1": a.M2, "N1": a.N2, "K": K, "ms": ms,
            "TFLOP/s": flops / ms / 1e9}


def attn_flops(B, T, H, hd=64):
    return 4.0 * hd * (T * (T + 1) / 2) * B * H


def bench_attention(B, T, H, bwd, iters, warmup, recompute=False):
    hd = 64
    gen = torch.Generator(device="cuda").manual_seed(0)
    mk = lambda: torch.randn(B, T, H, hd, device="cuda", generator=gen).to(torch.bfloat16)
    q, k, v, do = mk(), mk(), mk(), mk()
    o = torch.empty_like(q)
    lse = torch.empty(B, H, T, device="cuda")
    g.attention_forward(q, k, v, o, lse, B, T, H)
    if not bwd:
        ms = _time(lambda i: g.attention_forward(q, k, v, o, lse, B, T, H), iters, warmup)
        fl = attn_flops(B, T, H)
    else:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
        sc = torch.empty(B * H * T, device="cuda")
        if recompute:
            ms = _time(lambda i: g.attention_backward(q, k, v, o, do, lse, dq, dk, dv, sc, B, T, H), iters, warmup)
        else:  # the model's backward: dS kept in a workspace, dQ formed from it
            ds = torch.empty(g.attention_backward_ds_bytes(B, T, H), dtype=torch.uint8, device="cuda")
            ms = _time(lambda i: g.attention_backward_ds(q, k, v, o, do, lse, dq, dk, dv, sc, ds, B, T, H), iters,
                       warmup)
        fl = 2.0 * attn_flops(B, T, H)
    op = "attention_" + ("fwd" if not bwd else "bwd_recompute" if recompute else "bwd")
    return {"op": op, "B": B, "T": T, "H": H, "ms": ms, "TFLOP/s": fl / ms / 1e9}


def bench_attention_fb(B, T, H, iters, warmup):
    """Forward then backward per iteration (one launch of each attention kernel)."""
    hd = 64
    gen = torch.Generator(device="cuda").manual_seed(0)
    mk = lambda: torch.randn(B, T, H, hd, device="cuda", generator=gen).to(torch.bfloat16)
    q, k, v, do = mk(), mk(), mk(), mk()
    o = torch.empty_like(q)
    lse = torch.empty(B, H, T, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    sc = torch.empty(B * H * T, device="cuda")
    ds = torch.empty(g.attention_backward_ds_bytes(B, T, H), dtype=torch.uint8, device="cuda")

    def run(i):
        g.attention_forward(q, k, v, o, lse, B, T, H)
        g.attention_backward_ds(q, k, v, o, do, lse, dq, dk, dv, sc, ds, B, T, H)

    ms = _time(run, iters, warmup)
    return {"op": "attention_fwd_bwd", "B": B, "T": T, "H": H, "ms": ms, "TFLOP/s": 3.0 * attn_flops(B, T, H) / ms / 1e9}


def bench_adamw(a):
    """The fused clip + AdamW over the 124M parameters (a model with a one-row batch, so the
    arena is the parameter state plus little else)."""
    import synthetic

    w = dict(synthetic.WORKLOADS["gpt2_124m"], B=1, T=64)
    m = g.GPT2(w, seed=1)
    rng = torch.Generator().manual_seed(0)
    for i in range(len(m.names)):
        gr = torch.randn(m.shapes[i], generator=rng) * 1e-3
        m.set_grads(i, gr.numpy())
    n_params = sum(int(torch.tensor(s).prod()) for s in m.shapes)
    ms = _time(lambda i: m.clip_and_adamw(6e-4), a.iters, a.warmup)
    m.close()
    # norm pass reads g (4 B); the update reads p, g, m, v (16 B), writes p, m, v (12 B) and the bf16 copy (2 B)
    return {"op": "clip_adamw", "params": n_params, "ms": ms, "GB/s": 34.0 * n_params / ms / 1e6,
            "note": "ms includes the host read-back of the norm"}


def bench_classifier(a):
    gen = torch.Generator(device="cuda").manual_seed(0)
    z0 = torch.randn(a.N, a.Vp, device="cuda", generator=gen).to(torch.bfloat16)
    z = z0.clone()
    t = torch.randint(0, a.V, (a.N,), device="cuda", dtype=torch.int32, generator=gen)
    rows = torch.empty(a.N, device="cuda")
    ms = _time(lambda i: g.classifier(z, t, rows, a.N, a.V, a.Vp, 1.0 / a.N), a.iters, a.warmup)
    nbytes = 2.0 * a.N * a.Vp * 2
    return {"op": "classifier", "N": a.N, "Vp": a.Vp, "ms": ms, "GB/s": nbytes / ms / 1e6}


def bench_generate(a):
    """KV-cached sampling with the 124M model: B rows, a T0-token prompt, n_new new tokens."""
    import numpy as np

    import synthetic

    w = dict(synthetic.WORKLOADS["gpt2_124m"])
    m = g.GPT2(w, seed=w["seed"])
    B, T0, n_new = a.B, a.prompt, a.new
    x, _ = synthetic.zipf_window(w["seed"], B, T0, w["V"])
    seq0 = torch.zeros(B, T0 + n_new, dtype=torch.int32)
    seq0[:, :T0] = torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32))
    seq = seq0.cuda()
    u = torch.rand(n_new, B, device="cuda")
    ms = _time(lambda i: m.generate(seq, T0, u, 1.0, a.top_k), a.iters, a.warmup)
    m.close()
    return {"op": "generate", "model": "gpt2_124m", "B": B, "prompt": T0, "new": n_new, "top_k": a.top_k, "ms": ms,
            "tokens/s": B * n_new / ms * 1e3, "ms_per_position": ms / (T0 + n_new - 1)}


def bench_layernorm(a):
    gen = torch.Generator(device="cuda").manual_seed(0)
    N, C = a.N, a.C
    x = torch.randn(N, C, device="cuda", generator=gen).to(torch.bfloat16)
    dy = torch.randn(N, C, device="cuda", generator=gen).to(torch.bfloat16)
    g_ = torch.randn(C, device="cuda", generator=gen)
    b_ = torch.randn(C, device="cuda", generator=gen)
    y = torch.empty_like(x)
    mean = torch.empty(N, device="cuda")
    rstd = torch.empty(N, device="cuda")
    g.layernorm_forward(x, g_, b_, y, mean, rstd, N, C)
    out = []
    ms = _time(lambda i: g.layernorm_forward(x, g_, b_, y, mean, rstd, N, C), a.iters, a.warmup)
    out.append({"op": "layernorm_fwd", "N": N, "C": C, "ms": ms, "GB/s": (2.0 * N * C * 2 + 8 * N) / ms / 1e6})
    dres = torch.randn(N, C, device="cuda", generator=gen).to(torch.bfloat16)
    dg = torch.zeros(C, device="cuda")
    db = torch.zeros(C, device="cuda")
    ms = _time(lambda i: g.layernorm_backward(dy, x, mean, rstd, g_, dres, dres, dg, db, N, C), a.iters, a.warmup)
    out.append({"op": "layernorm_bwd", "N": N, "C": C, "ms": ms, "GB/s": (4.0 * N * C * 2 + 8 * N) / ms / 1e6})
    return out


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("op", choices=["matmul", "matmul-accum2", "attention", "classifier", "layernorm", "attention-sweep", "generate",
                                   "attention-fb", "adamw"])
    ap.add_argument("--C", type=int, default=768)
    ap.add_argument("--M", type=int, default=16384)
    ap.add_argument("--N", type=int, default=2304)
    ap.add_argument("--K", type=int, default=768)
    ap.add_argument("--M2", type=int, default=3072, help="matmul-accum2: the second product's M")
    ap.add_argument("--N2", type=int, default=768, help="matmul-accum2: the second product's N")
    ap.add_argument("--a-mn", action="store_true")
    ap.add_argument("--b-mn", action="store_true")
    ap.add_argument("--epi", default="store", choices=sorted(EPIS))
    ap.add_argument("--fp8", action="store_true", help="matmul: E4M3 operands (K-major) instead of bf16")
    ap.add_argument("--B", type=int, default=16)
    ap.add_argument("--T", type=int, default=1024)
    ap.add_argument("--H", type=int, default=12)
    ap.add_argument("--bwd", action="store_true")
    ap.add_argument("--V", type=int, default=50257)
    ap.add_argument("--Vp", type=int, default=50304)
    ap.add_argument("--prompt", type=int, default=32)
    ap.add_argument("--new", type=int, default=64)
    ap.add_argument("--top-k", type=int, default=50)
    ap.add_argument("--recompute", action="store_true",
                    help="attention: time the backward without the dS workspace (S and dP recomputed for dQ)")
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    a = ap.parse_args(argv)
    from gpt_decoder_only_train_b300 import build

    build.build()
    if a.op == "matmul":
        out = [bench_matmul(a)]
    elif a.op == "matmul-accum2":
        out = [bench_matmul_accum2(a)]
    elif a.op == "attention":
        out = [bench_attention(a.B, a.T, a.H, a.bwd, a.iters, a.warmup, a.recompute)]
    elif a.op == "classifier":
        out = [bench_classifier(a)]
    elif a.op == "layernorm":
        out = bench_layernorm(a)
    elif a.op == "generate":
        out = [bench_generate(a)]
    elif a.op == "attention-fb":
        out = [bench_attention_fb(a.B, a.T, a.H, a.iters, a.warmup)]
    elif a.op == "adamw":
        out = [bench_adamw(a)]
    else:
        out = []
        for T, B in ((256, 256), (1024, 64), (2048, 32), (4096, 16)):
            for bwd, rc in ((False, False), (True, False), (True, True)):
                out.append(bench_attention(B, T, 12, bwd, a.iters, a.warmup, rc))
    for r in out:
        print(json.dumps(r), flush=True)


if __name__ == "__main__":
    main()
