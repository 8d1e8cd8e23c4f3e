"""Seeded synthetic inputs shared by the CUDA path's harness and by the oracle.

This module draws the INPUTS of a training step (token windows, attention
operands). It holds none of the method's arithmetic: no model, no loss, no
optimizer. Both the oracle tests and ``bench.py`` call it so that the two sides
see bit-identical inputs.

Generators
----------
* Counter-based SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
  number generators", OOPSLA 2014): ``sm64(x)`` is the output the generator
  gives when its state is ``x``.  A draw is addressed by ``(seed, stream, ctr)``
  as ``sm64(sm64(sm64(seed) + stream) + ctr)`` (all arithmetic mod 2^64).
* Uniform tokens in ``[0, V)``: ``floor(((x >> 11) * 2^-53) * V)``.
* Zipf(s) tokens over ranks ``k = 1..V`` with ``P(k) ~ k^-s``: inverse CDF in
  double, ``k`` = smallest rank whose CDF is ``>= u`` with ``u`` in ``(0, 1]``;
  token id = ``k - 1``.  Zipf(1.1) stands in for the BPE token frequencies of
  the FineWeb text the pages train on ("llm.c kullanarak GPT-2 modelini düşük
  maliyetle yeniden uygulamak", §Eğitim süreci); the dataset itself is not used.
* A micro-step window is ``B*T + 1`` consecutive stream tokens; inputs are the
  first ``B*T`` and targets the last ``B*T`` (shifted by one), per the
  batch-chunk data loader of "Let's build GPT: from scratch", chapter
  00:14:27.  Consecutive micro-steps advance the window by ``B*T``.
* Attention operands: N(0,1) by Box-Muller on the same counter stream, rounded
  to bf16 (round-to-nearest-even) for the bf16 attention workload.
"""
from __future__ import annotations

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# stream ids of the token generators
STREAM_TOKENS = 0
STREAM_TARGETS = 1
STREAM_ZIPF = 2
STREAM_ATTN = 16  # + 0..3 for q, k, v, dO


def sm64(x: np.ndarray) -> np.ndarray:
    """SplitMix64 output for state(s) ``x`` (uint64, wraps mod 2^64)."""
    x = np.asarray(x, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = x + _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def draws(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """``n`` raw 64-bit draws ``(seed, stream, offset + i)``."""
    with np.errstate(over="ignore"):
        key = sm64(sm64(np.uint64(seed)) + np.uint64(stream))
        ctr = np.arange(offset, offset + n, dtype=np.uint64)
        return sm64(key + ctr)


def unit_open0(x: np.ndarray) -> np.ndarray:
    """Map raw draws to doubles in (0, 1]."""
    return ((x >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def unit_closed0(x: np.ndarray) -> np.ndarray:
    """Map raw draws to doubles in [0, 1)."""
    return (x >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def uniform_tokens(seed: int, stream: int, n: int, V: int) -> np.ndarray:
    u = unit_closed0(draws(seed, stream, n))
    return np.minimum(np.floor(u * V), V - 1).astype(np.int32)


def zipf_cdf(V: int, s: float = 1.1) -> np.ndarray:
    k = np.arange(1, V + 1, dtype=np.float64)
    w = k ** (-s)
    cdf = np.cumsum(w) / w.sum()
    cdf[-1] = 1.0
    return cdf


def zipf_tokens(seed: int, n: int, V: int, s: float = 1.1, offset: int = 0) -> np.ndarray:
    cdf = zipf_cdf(V, s)
    u = unit_open0(draws(seed, STREAM_ZIPF, n, offset))
    k = np.searchsorted(cdf, u, side="left") + 1  # smallest k with cdf[k-1] >= u
    return (np.minimum(k, V) - 1).astype(np.int32)


def zipf_window(seed: int, B: int, T: int, V: int, micro_step: int = 0, s: float = 1.1):
    """Tokens and targets ``[B, T]`` int32 for one micro-step of the Zipf stream."""
    BT = B * T
    w = zipf_tokens(seed, BT + 1, V, s, offset=micro_step * BT)
    return w[:BT].reshape(B, T).copy(), w[1:].reshape(B, T).copy()


def uniform_batch(seed: int, B: int, T: int, V: int):
    """Independent uniform tokens and targets ``[B, T]`` int32 (tiny fp32 workload)."""
    x = uniform_tokens(seed, STREAM_TOKENS, B * T, V).reshape(B, T)
    y = uniform_tokens(seed, STREAM_TARGETS, B * T, V).reshape(B, T)
    return x, y


def normal(seed: int, stream: int, n: int) -> np.ndarray:
    """N(0,1) doubles by Box-Muller (cosine branch) on draw pairs (2i, 2i+1)."""
    d = draws(seed, stream, 2 * n)
    u1 = unit_open0(d[0::2])
    u2 = unit_closed0(d[1::2])
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def attention_operands(seed: int, B: int, H: int, T: int, hd: int):
    """q, k, v, dO as float32 arrays [B, T, H, hd] holding bf16-representable values."""
    import torch

    out = []
    for i in range(4):
        a = normal(seed, STREAM_ATTN + i, B * T * H * hd).astype(np.float32)
        t = torch.from_numpy(a).to(torch.bfloat16).to(torch.float32)
        out.append(t.numpy().reshape(B, T, H, hd))
    return tuple(out)


# --- workload descriptions (sizes of the five configurations) -----------------

WORKLOADS = {
    "tiny_fp32": dict(L=2, C=64, H=4, V=256, Vp=256, T=32, B=2, dtype="fp32", recompute_gelu=0, seed=0,
                      tokens="uniform"),
    "gpt2_124m": dict(L=12, C=768, H=12, V=50257, Vp=50304, T=1024, B=16, dtype="bf16", recompute_gelu=0, seed=1),
    "gpt2_124m_accum32": dict(L=12, C=768, H=12, V=50257, Vp=50304, T=1024, B=16, dtype="bf16", recompute_gelu=0,
                              seed=2, grad_accum=32, steps=20),
    "gpt2_350m_recompute": dict(L=24, C=1024, H=16, V=50257, Vp=50304, T=1024, B=8, dtype="bf16", recompute_gelu=1,
                                seed=3),
}

ATTN_SWEEP = [dict(T=256, B=256), dict(T=1024, B=64), dict(T=2048, B=32), dict(T=4096, B=16)]


def step_batch(workload: dict, micro_step: int = 0):
    """Tokens/targets for one micro-step of a named workload."""
    if workload.get("tokens", "zipf") == "uniform":
        return uniform_batch(workload["seed"], workload["B"], workload["T"], workload["V"])
    return zipf_window(workload["seed"], workload["B"], workload["T"], workload["V"], micro_step)
