"""Plain float64 CPU oracle of one GPT-2 training step.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, the smoke check and the
CPU-baseline leg of ``bench.py``; never by the product path.

The step, and the passage each part follows
-------------------------------------------
Page titles are those of the source web pages; sections are their headings or
chapter timestamps.

* Token + position embedding -- "Let's build GPT: from scratch" (从头开始用代码构建GPT),
  chapter 01:00:18 (position encoding), and the batch-chunk loader, 00:14:27.
* Pre-LN decoder block ``x += attn(ln1(x)); x += mlp(ln2(x))`` with a final
  LayerNorm -- same page, chapters 01:21:59 (multi-head self-attention),
  01:24:25 (feed-forward layer), 01:26:48 (residual connections), 01:32:51
  (LayerNorm).  The pages name the parts but not the order; the pre-LN order of
  GPT-2 is taken (reading).
* Causal attention, scale ``1/sqrt(head_size)`` -- same page, chapters 01:02:00
  (self-attention), 01:16:56 ("scaled" attention) and the two errata at its
  end: future tokens cannot communicate (00:57:00) and normalise by head_size,
  not C (01:20:05).  A position attends to itself and to the past.
* Cross-entropy loss -- "Let's reproduce GPT-2 (124M)", §Bölümler 4 (Cross-entropy
  loss ve overfit testleri): the mean over all B*T positions of
  ``logsumexp(z) - z[target]``; padded vocabulary columns (v >= V) are left out.
* AdamW, warmup + cosine decay, gradient accumulation -- same page, §Video özeti.
* Global grad-norm clipping against the early gradient explosion --
  "llm.c kullanarak GPT-2 modelini düşük maliyetle yeniden uygulamak",
  §Eğitim süreci.
* GELU recompute (``-r``) only changes what is stored, not what is computed:
  same page, §Eğitimi çalıştırma.  The oracle has no recompute switch.

Readings where the pages are silent (also listed in the design notes):
GELU is GPT-2's tanh form; LayerNorm eps = 1e-5 with biased variance; Q|K|V
column blocks with head h at columns h*hd..(h+1)*hd; LM head tied to wte, no
bias; dropout 0; clip coefficient ``clip/(norm + 1e-6)`` applied when < 1,
pre-clip norm returned; AdamW decoupled (PyTorch form), bias correction from
t = 1, eps outside the sqrt, weight decay only on the 2-D weights.

Pins (tests that tie each function to something other than itself)
-----------------------------------------------------------------
* backward of every op and of the whole step: central finite differences in
  float64 (``tests/test_oracle_gradcheck.py``), plus an independent autograd
  cross-check;
* attention: brute-force per-(b,h,i,j) Python loops on T <= 8 and the
  softmax/causality invariants (``tests/test_oracle_ops.py``);
* LayerNorm: zero mean / unit variance rows, dx orthogonal to 1 and x_hat;
* cross-entropy: uniform logits give ln V exactly, dz rows sum to 0;
* step: initial loss ~= ln V + 0.02^2 C / 2, one fixed batch overfits to loss
  < 0.1, AdamW step 1 closed form, clipped norm equals ``clip``, LR schedule
  values, causality of the logits, embedding backward vs a counting brute force;
* init: SplitMix64 published outputs, Box-Muller moments (KS test);
* sampling: the set of u in [0, 1) that draws token i has measure
  softmax(z/temperature)_i over the candidates (exact interval lengths);
  top_k = 1 is the argmax with the lower index on ties; a small temperature
  tends to the argmax; generation agrees with teacher forcing.
"""
from __future__ import annotations

import math
from collections import OrderedDict
from dataclasses import dataclass

import numpy as np
import torch

from . import init_lib

F64 = torch.float64
LN_EPS = 1e-5
GELU_K = math.sqrt(2.0 / math.pi)
GELU_C = 0.044715


@dataclass
class Config:
    L: int
    C: int
    H: int
    V: int
    Vp: int
    T: int
    B: int
    dtype: str = "fp32"
    recompute_gelu: int = 0

    @property
    def hd(self) -> int:
        return self.C // self.H

    @staticmethod
    def from_dict(d: dict) -> "Config":
        return Config(**{k: d[k] for k in ("L", "C", "H", "V", "Vp", "T", "B", "dtype", "recompute_gelu") if k in d})


# --------------------------------------------------------------------------- #
# parameters
# --------------------------------------------------------------------------- #

def param_specs(cfg: Config):
    """(name, shape, init, std, weight_decay) in tensor-id order.

    Tensor ids (the RNG stream of each tensor) are the list positions: wte, wpe,
    then per layer ln1.g, ln1.b, qkv.w, qkv.b, proj.w, proj.b, ln2.g, ln2.b,
    fc.w, fc.b, fcproj.w, fcproj.b, and finally lnf.g, lnf.b.
    """
    L, C, V, Vp, T = cfg.L, cfg.C, cfg.V, cfg.Vp, cfg.T
    std = 0.02
    resid_std = 0.02 / math.sqrt(2.0 * L)
    s = [("wte", (Vp, C), "normal_rows", std, True), ("wpe", (T, C), "normal", std, True)]
    for l in range(L):
        p = "h%d." % l
        s += [
            (p + "ln1.g", (C,), "ones", 0.0, False),
            (p + "ln1.b", (C,), "zeros", 0.0, False),
            (p + "qkv.w", (3 * C, C), "normal", std, True),
            (p + "qkv.b", (3 * C,), "zeros", 0.0, False),
            (p + "proj.w", (C, C), "normal", resid_std, True),
            (p + "proj.b", (C,), "zeros", 0.0, False),
            (p + "ln2.g", (C,), "ones", 0.0, False),
            (p + "ln2.b", (C,), "zeros", 0.0, False),
            (p + "fc.w", (4 * C, C), "normal", std, True),
            (p + "fc.b", (4 * C,), "zeros", 0.0, False),
            (p + "fcproj.w", (C, 4 * C), "normal", resid_std, True),
            (p + "fcproj.b", (C,), "zeros", 0.0, False),
        ]
    s += [("lnf.g", (C,), "ones", 0.0, False), ("lnf.b", (C,), "zeros", 0.0, False)]
    return s


def init_params(cfg: Config, seed: int) -> "OrderedDict[str, torch.Tensor]":
    """fp32-valued initial parameters (held as float64 tensors).

    wte rows v >= V (vocabulary padding) are zero: only the V real rows are
    drawn.  Normal draws come from the oracle's own C initialiser.
    """
    lib = init_lib()
    out = OrderedDict()
    for tid, (name, shape, kind, std, _) in enumerate(param_specs(cfg)):
        n = int(np.prod(shape))
        buf = np.zeros(n, dtype=np.float32)
        if kind == "ones":
            buf[:] = 1.0
        elif kind in ("normal", "normal_rows"):
            ndraw = cfg.V * cfg.C if kind == "normal_rows" else n
            lib.oracle_normal_fill(seed, tid, ndraw, std, buf.ctypes.data)
        out[name] = torch.from_numpy(buf.astype(np.float64)).reshape(shape)
    return out


# --------------------------------------------------------------------------- #
# ops (forward and hand-derived backward)
# --------------------------------------------------------------------------- #

def layernorm_forward(x, g, b, eps=LN_EPS):
    """Row LayerNorm: ``(x - mean)/sqrt(var + eps) * g + b``, biased variance."""
    mean = x.mean(-1, keepdim=True)
    var = ((x - mean) ** 2).mean(-1, keepdim=True)
    rstd = 1.0 / torch.sqrt(var + eps)
    xhat = (x - mean) * rstd
    return xhat * g + b, mean, rstd


def layernorm_backward(dy, x, mean, rstd, g):
    """dx, dg, db of :func:`layernorm_forward` (rows over all leading dims)."""
    xhat = (x - mean) * rstd
    dxhat = dy * g
    dx = rstd * (dxhat - dxhat.mean(-1, keepdim=True) - xhat * (dxhat * xhat).mean(-1, keepdim=True))
    C = x.shape[-1]
    dg = (dy * xhat).reshape(-1, C).sum(0)
    db = dy.reshape(-1, C).sum(0)
    return dx, dg, db


def gelu_forward(h):
    """GPT-2's tanh GELU: ``0.5 h (1 + tanh(sqrt(2/pi) (h + 0.044715 h^3)))``."""
    return 0.5 * h * (1.0 + torch.tanh(GELU_K * (h + GELU_C * h ** 3)))


def gelu_derivative(h):
    u = GELU_K * (h + GELU_C * h ** 3)
    t = torch.tanh(u)
    return 0.5 * (1.0 + t) + 0.5 * h * (1.0 - t * t) * GELU_K * (1.0 + 3.0 * GELU_C * h * h)


def _causal_scores(q, k):
    hd = q.shape[-1]
    s = (q @ k.transpose(-1, -2)) * (1.0 / math.sqrt(hd))
    T = q.shape[-2]
    future = torch.ones(T, T, dtype=torch.bool).triu(1)
    return s.masked_fill(future, float("-inf"))


def causal_attention_forward(q, k, v):
    """Naive causal attention on ``[..., T, hd]``: full T x T scores, mask j > i
    with -inf, max-subtracted softmax, then x V.  Returns (O, lse)."""
    s = _causal_scores(q, k)
    m = s.max(-1, keepdim=True).values
    e = torch.exp(s - m)
    l = e.sum(-1, keepdim=True)
    o = (e / l) @ v
    return o, (m + torch.log(l)).squeeze(-1)


def causal_attention_backward(q, k, v, do):
    """dq, dk, dv of :func:`causal_attention_forward` (probabilities recomputed)."""
    hd = q.shape[-1]
    scale = 1.0 / math.sqrt(hd)
    p = torch.softmax(_causal_scores(q, k), dim=-1)
    dv = p.transpose(-1, -2) @ do
    dp = do @ v.transpose(-1, -2)
    ds = p * (dp - (p * dp).sum(-1, keepdim=True))
    dq = (ds @ k) * scale
    dk = (ds.transpose(-1, -2) @ q) * scale
    return dq, dk, dv


def cross_entropy_forward(z, targets):
    """Mean over rows of ``logsumexp(z) - z[target]``; z is ``[N, V]`` (real columns only)."""
    m = z.max(-1, keepdim=True).values
    lse = m + torch.log(torch.exp(z - m).sum(-1, keepdim=True))
    rows = lse.squeeze(-1) - z.gather(-1, targets.reshape(-1, 1)).squeeze(-1)
    return rows.mean(), lse, rows


def cross_entropy_backward(z, lse, targets, dloss):
    """dz of the mean loss times ``dloss``: ``(softmax(z) - onehot) * dloss / N``."""
    p = torch.exp(z - lse)
    n = z.shape[0]
    p[torch.arange(n), targets.reshape(-1)] -= 1.0
    return p * (dloss / n)


def embedding_backward(dx, tokens, Vp, Tmax):
    """Scatter-add of dx rows into dwte[token] and (summed over the batch) dwpe[t]."""
    B, T, C = dx.shape
    dwte = torch.zeros(Vp, C, dtype=dx.dtype)
    dwte.index_add_(0, tokens.reshape(-1).long(), dx.reshape(-1, C))
    dwpe = torch.zeros(Tmax, C, dtype=dx.dtype)
    dwpe[:T] = dx.sum(0)
    return dwte, dwpe


# --------------------------------------------------------------------------- #
# the model step
# --------------------------------------------------------------------------- #

def _split_heads(t, B, T, H, hd):
    return t.reshape(B, T, H, hd).permute(0, 2, 1, 3)


def _merge_heads(t, B, T, C):
    return t.permute(0, 2, 1, 3).reshape(B, T, C)


def _attention_per_sequence(fn, *args):
    """Apply an attention function one batch element at a time (bounds the T x T memory)."""
    outs = [fn(*(a[b] for a in args)) for b in range(args[0].shape[0])]
    return tuple(torch.stack(o) for o in zip(*outs))


def model_forward(cfg: Config, P, tokens, targets=None):
    """Forward pass.  tokens/targets ``[B, T]`` int tensors.

    Returns (loss or None, logits ``[B*T, V]``, cache for :func:`model_backward`).
    """
    tokens = torch.as_tensor(tokens).long()
    B, T = tokens.shape
    C, H, V = cfg.C, cfg.H, cfg.V
    hd = C // H
    x = P["wte"][tokens] + P["wpe"][:T]
    layers = []
    for l in range(cfg.L):
        p = "h%d." % l
        c = {"x": x}
        y, c["m1"], c["r1"] = layernorm_forward(x, P[p + "ln1.g"], P[p + "ln1.b"])
        c["y"] = y
        qkv = y @ P[p + "qkv.w"].T + P[p + "qkv.b"]
        q = _split_heads(qkv[..., 0:C], B, T, H, hd)
        k = _split_heads(qkv[..., C:2 * C], B, T, H, hd)
        v = _split_heads(qkv[..., 2 * C:3 * C], B, T, H, hd)
        o, lse = _attention_per_sequence(causal_attention_forward, q, k, v)
        c["q"], c["k"], c["v"], c["lse"] = q, k, v, lse
        of = _merge_heads(o, B, T, C)
        c["o"] = of
        x1 = x + of @ P[p + "proj.w"].T + P[p + "proj.b"]
        c["x1"] = x1
        y2, c["m2"], c["r2"] = layernorm_forward(x1, P[p + "ln2.g"], P[p + "ln2.b"])
        c["y2"] = y2
        h = y2 @ P[p + "fc.w"].T + P[p + "fc.b"]
        c["h"] = h
        g = gelu_forward(h)
        x = x1 + g @ P[p + "fcproj.w"].T + P[p + "fcproj.b"]
        layers.append(c)
    yf, mf, rf = layernorm_forward(x, P["lnf.g"], P["lnf.b"])
    z = yf.reshape(B * T, C) @ P["wte"][:V].T
    cache = {"tokens": tokens, "targets": targets, "layers": layers, "xL": x, "yf": yf, "mf": mf, "rf": rf,
             "z": z, "B": B, "T": T}
    loss = None
    if targets is not None:
        tg = torch.as_tensor(targets).long().reshape(-1)
        loss, lse, rows = cross_entropy_forward(z, tg)
        cache["lse"], cache["tg"], cache["rows"] = lse, tg, rows
    return loss, z, cache


def model_backward(cfg: Config, P, cache, grad_scale=1.0):
    """Gradients of ``grad_scale * loss`` for every parameter (fresh dict)."""
    B, T = cache["B"], cache["T"]
    C, H, V = cfg.C, cfg.H, cfg.V
    hd = C // H
    G = OrderedDict((k, torch.zeros_like(v)) for k, v in P.items())
    dz = cross_entropy_backward(cache["z"], cache["lse"], cache["tg"], grad_scale)  # [BT, V]
    yf = cache["yf"].reshape(B * T, C)
    G["wte"][:V] += dz.T @ yf
    dyf = (dz @ P["wte"][:V]).reshape(B, T, C)
    dx, G["lnf.g"], G["lnf.b"] = layernorm_backward(dyf, cache["xL"], cache["mf"], cache["rf"], P["lnf.g"])
    for l in reversed(range(cfg.L)):
        p = "h%d." % l
        c = cache["layers"][l]
        # x_out = x1 + gelu(h) Wfcproj^T + b
        g = gelu_forward(c["h"])
        G[p + "fcproj.w"] = dx.reshape(-1, C).T @ g.reshape(-1, 4 * C)
        G[p + "fcproj.b"] = dx.reshape(-1, C).sum(0)
        dg = dx @ P[p + "fcproj.w"]
        dh = dg * gelu_derivative(c["h"])
        G[p + "fc.w"] = dh.reshape(-1, 4 * C).T @ c["y2"].reshape(-1, C)
        G[p + "fc.b"] = dh.reshape(-1, 4 * C).sum(0)
        dy2 = dh @ P[p + "fc.w"]
        dln2, G[p + "ln2.g"], G[p + "ln2.b"] = layernorm_backward(dy2, c["x1"], c["m2"], c["r2"], P[p + "ln2.g"])
        dx1 = dx + dln2
        # x1 = x + O Wproj^T + b
        G[p + "proj.w"] = dx1.reshape(-1, C).T @ c["o"].reshape(-1, C)
        G[p + "proj.b"] = dx1.reshape(-1, C).sum(0)
        do = _split_heads(dx1 @ P[p + "proj.w"], B, T, H, hd)
        dq, dk, dv = _attention_per_sequence(causal_attention_backward, c["q"], c["k"], c["v"], do)
        dqkv = torch.cat([_merge_heads(dq, B, T, C), _merge_heads(dk, B, T, C), _merge_heads(dv, B, T, C)], -1)
        G[p + "qkv.w"] = dqkv.reshape(-1, 3 * C).T @ c["y"].reshape(-1, C)
        G[p + "qkv.b"] = dqkv.reshape(-1, 3 * C).sum(0)
        dy = dqkv @ P[p + "qkv.w"]
        dln1, G[p + "ln1.g"], G[p + "ln1.b"] = layernorm_backward(dy, c["x"], c["m1"], c["r1"], P[p + "ln1.g"])
        dx = dx1 + dln1
    dwte_e, dwpe = embedding_backward(dx, cache["tokens"], cfg.Vp, cfg.T)
    G["wte"] += dwte_e
    G["wpe"] = dwpe
    return G


def global_norm(grads) -> float:
    return math.sqrt(sum(float((g * g).sum()) for g in grads.values()))


def lr_schedule(it: int, max_lr=6e-4, min_lr=6e-5, warmup=700, max_steps=19073) -> float:
    """Linear warmup ``max_lr*(it+1)/warmup`` then cosine decay to ``min_lr`` at ``max_steps``.

    ``max_steps`` = 10e9 tokens / 524288 tokens per step ("~20K steps" of
    "llm.c kullanarak ...", §Eğitim süreci).
    """
    if it < warmup:
        return max_lr * (it + 1) / warmup
    if it > max_steps:
        return min_lr
    ratio = (it - warmup) / (max_steps - warmup)
    coeff = 0.5 * (1.0 + math.cos(math.pi * ratio))
    return min_lr + coeff * (max_lr - min_lr)


# --------------------------------------------------------------------------- #
# sampling ("llm.c kullanarak GPT-2 modelini düşük maliyetle yeniden
# uygulamak", §Sampling and §SSS: a trained model can be sampled, with or
# without a prompt; "Let's reproduce GPT-2 (124M)", §Bölümler 3: the sampling
# loop).  The pages give no sampling rule; the reading used on both sides:
# temperature-scaled softmax restricted to the top_k logits, the token drawn
# by inverse CDF with a caller-supplied uniform.
# --------------------------------------------------------------------------- #

def sample_next(z, temperature: float, top_k: int, u: float) -> int:
    """One draw from logits ``z`` [V] (any real dtype; compared as given).

    Candidates: the top_k entries in the order (larger value first, equal
    values lower index first).  Weights ``exp((z_i - z_max) / temperature)``;
    when ``z_max`` is not finite (+inf, or every candidate -inf) the weights
    are the limit of that rule: 1 for the candidates equal to ``z_max``, 0 for
    the others.  The token is the first candidate whose cumulative weight
    exceeds ``u * sum(weights)``; if rounding leaves none, the last candidate.
    """
    z = np.asarray(z, dtype=np.float64)
    order = [int(i) for i in np.lexsort((np.arange(z.shape[0]), -z))[:top_k]]  # by -z, then by index
    zmax = z[order[0]]
    if math.isfinite(zmax):
        w = [math.exp((z[i] - zmax) / temperature) for i in order]
    else:
        w = [1.0 if z[i] == zmax else 0.0 for i in order]
    target = u * sum(w)
    cum = 0.0
    for i, wi in zip(order, w):
        cum += wi
        if cum > target:
            return int(i)
    return int(order[-1])


def generate(cfg: Config, P, prompt, n_new: int, temperature: float, top_k: int, uniforms):
    """Autoregressive sampling by recomputing the whole forward for every new
    token (no cache): prompt int [B, T0] -> [B, T0 + n_new]; uniforms [n_new, B].
    Returns the sequences and the logits each token was drawn from
    ([n_new, B, V], float64)."""
    seq = torch.as_tensor(prompt).long().clone()
    B = seq.shape[0]
    drawn = []
    for s in range(n_new):
        _, z, _ = model_forward(cfg, P, seq, None)
        last = z.reshape(B, seq.shape[1], -1)[:, -1, :]
        drawn.append(last)
        nxt = [sample_next(last[b].numpy(), temperature, top_k, float(uniforms[s][b])) for b in range(B)]
        seq = torch.cat([seq, torch.tensor(nxt, dtype=torch.long).reshape(B, 1)], dim=1)
    return seq, torch.stack(drawn)


class OracleGPT2:
    """Stateful wrapper with the same call shapes as the C ABI."""

    def __init__(self, cfg: Config, seed: int):
        self.cfg = cfg
        self.params = init_params(cfg, seed)
        self.decay = {name: dec for name, _, _, _, dec in param_specs(cfg)}
        self.grads = OrderedDict((k, torch.zeros_like(v)) for k, v in self.params.items())
        self.m = OrderedDict((k, torch.zeros_like(v)) for k, v in self.params.items())
        self.v = OrderedDict((k, torch.zeros_like(v)) for k, v in self.params.items())
        self.t = 0
        self._cache = None

    def forward(self, tokens, targets=None):
        loss, z, self._cache = model_forward(self.cfg, self.params, tokens, targets)
        return None if loss is None else float(loss)

    def logits(self, tokens):
        _, z, _ = model_forward(self.cfg, self.params, tokens, None)
        return z

    def backward(self, grad_scale=1.0):
        g = model_backward(self.cfg, self.params, self._cache, grad_scale)
        for k in self.grads:
            self.grads[k] += g[k]
        self._cache = None

    def zero_grad(self):
        for g in self.grads.values():
            g.zero_()

    def clip_and_adamw(self, lr, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1, clip=1.0) -> float:
        norm = global_norm(self.grads)
        coef = min(1.0, clip / (norm + 1e-6))
        self.t += 1
        bc1 = 1.0 - beta1 ** self.t
        bc2 = 1.0 - beta2 ** self.t
        for k, p in self.params.items():
            g = self.grads[k] * coef
            self.m[k] = beta1 * self.m[k] + (1.0 - beta1) * g
            self.v[k] = beta2 * self.v[k] + (1.0 - beta2) * g * g
            mhat = self.m[k] / bc1
            vhat = self.v[k] / bc2
            if self.decay[k]:
                p.mul_(1.0 - lr * wd)
            p.sub_(lr * mhat / (torch.sqrt(vhat) + eps))
        return norm
