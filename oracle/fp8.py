"""FP8 (E4M3) quantisation and the FP8 matmul it feeds, in plain float64 / numpy.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): imported by ``tests/``
and never by the product path.

What it follows
---------------
* The pages name FP8 as the next precision step for this training code
  ("llm.c kullanarak GPT-2 modelini düşük maliyetle yeniden uygulamak", §SSS:
  FP8 support is planned; the "PyTorch Howsam" post on llm.c: what remains
  is FP8 testing).  They give no format or scaling rule.
* Readings (also listed in the design notes): the E4M3 format of the OCP 8-bit
  floating point specification -- 1 sign bit, 4 exponent bits with bias 7, 3
  mantissa bits, no infinities, the all-ones exponent with all-ones mantissa
  is NaN, largest finite value 448, smallest normal 2^-6, subnormals k 2^-9;
  conversion rounds to nearest, ties to even, and saturates finite values
  beyond 448 to +-448.  Scaling is per row of the activation operand and per
  tensor of the weight operand: a row (or tensor) with largest magnitude
  ``amax`` is multiplied by ``s = 448 / amax`` before rounding and its
  dequantisation factor is ``amax / 448``; a row of zeros keeps factor 1 and
  codes 0.  The scale and the scaled values are computed in fp32 (IEEE
  round to nearest): the quantised code is an integer decided by floating
  point, so both sides take that decision in the same precision.
* The matmul: ``D[m, n] = a_f[m] b_f sum_k qa[m, k] qb[n, k] (+ bias[n])``
  with the codes' exact values; everything after decoding is float64.
* The E4M3 forward of the model (:func:`model_forward_e4m3`): the four
  projections of every block (QKV, attention output, FC, FC output) multiply
  E4M3 codes -- the activation operand quantised per row, the weight operand
  per tensor from the bf16 weight copy the bf16 forward multiplies -- and
  everything else (embeddings, LayerNorm, attention, GELU, residual adds,
  the tied LM head, the loss) is the float64 forward of :mod:`oracle.gpt2`.
  The backward is that module's ``model_backward`` applied to this forward's
  cache with the unquantised weights (straight-through: the quantiser counts
  as the identity in the backward).  Readings: which products are quantised,
  the scaling granularity and the straight-through backward are not on the
  pages; they are the usual choices of FP8 training recipes and are listed
  in the design notes.

Pins (``tests/test_oracle_fp8.py``): every one of the 254 finite codes
decodes to the value the format defines and re-encodes to itself; the
printed limits (448, 2^-6, 2^-9); ties go to the even mantissa; values past
448 saturate; rounding error at most half a quantum; a brute-force nearest
search over all finite codes agrees with the rounding everywhere; row
quantisation reproduces the row to within its quantisation bound; the E4M3
forward with its quantiser switched off is bit-identical to the float64
forward (same block structure), and with it on stays within the loss change
that 3-bit mantissas allow.
"""
from __future__ import annotations

import numpy as np
import torch

from . import gpt2 as og

E4M3_MAX = 448.0


def e4m3_decode(code) -> np.ndarray:
    """float64 value of E4M3 codes (uint8); NaN for 0x7F / 0xFF."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


def e4m3_round(x) -> np.ndarray:
    """Nearest E4M3 value (ties to even mantissa), finite values past 448 saturated."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    # spacing of representable values around a: 2^-9 below 2^-6, else 2^(e - 3)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    q = np.where(a < 2.0 ** -6, 2.0 ** -9, np.exp2(e - 3.0))
    r = np.round(a / q) * q  # numpy rounds halves to even: the even multiple has the even mantissa
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, x)


def e4m3_encode(x) -> np.ndarray:
    """E4M3 codes (uint8) of the rounded values of x."""
    r = e4m3_round(x)
    a = np.abs(r)
    sign = np.where(np.signbit(r), 0x80, 0)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    sub = a < 2.0 ** -6
    exp_field = np.where(sub, 0, e + 7).astype(np.int64)
    mant = np.where(sub, a / 2.0 ** -9, (a / np.exp2(e) - 1.0) * 8.0)
    code = sign | (exp_field << 3) | np.rint(mant).astype(np.int64)
    return code.astype(np.uint8)


def quantize_rows(x):
    """Per-row E4M3 quantisation of a 2-D array (values exactly representable in fp32).

    Returns (codes uint8 [M, K], dequantisation factor fp32 [M]): row m is
    multiplied by ``s = float32(448) / float32(amax_m)`` in fp32, rounded to
    E4M3, and represents ``codes * amax_m / 448``.
    """
    x = np.asarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=1)
    s = np.where(amax > 0, np.float32(E4M3_MAX) / np.where(amax > 0, amax, np.float32(1)), np.float32(1))
    s = s.astype(np.float32)
    scaled = (x * s[:, None]).astype(np.float32)  # one fp32 multiply per element
    codes = e4m3_encode(scaled.astype(np.float64))
    inv = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1)).astype(np.float32)
    return codes, inv


def quantize_tensor(x):
    """Per-tensor E4M3 quantisation: (codes uint8, dequantisation factor fp32) with one amax."""
    x = np.asarray(x, dtype=np.float32)
    codes, inv = quantize_rows(x.reshape(1, -1))
    return codes.reshape(x.shape), np.float32(inv[0])


def matmul_e4m3(qa, a_inv, qb, b_inv, bias=None):
    """``D[m, n] = a_inv[m] b_inv sum_k decode(qa[m, k]) decode(qb[n, k]) (+ bias[n])`` in float64."""
    a = e4m3_decode(qa)
    b = e4m3_decode(qb)
    d = (a @ b.T) * np.asarray(a_inv, dtype=np.float64)[:, None] * float(b_inv)
    if bias is not None:
        d = d + np.asarray(bias, dtype=np.float64)[None, :]
    return d


def _product(x, w, quantise: bool):
    """``x @ w^T`` over the last axis; with ``quantise`` both operands go through E4M3 first."""
    if not quantise:
        return x @ w.T
    lead = x.shape[:-1]
    qa, ai = quantize_rows(x.reshape(-1, x.shape[-1]).numpy())
    wb = w.to(torch.bfloat16).to(og.F64).numpy()  # the bf16 weight copy of the forward
    qb, bi = quantize_tensor(wb)
    return torch.from_numpy(matmul_e4m3(qa, ai, qb, bi)).reshape(*lead, w.shape[0])


def model_forward_e4m3(cfg, P, tokens, targets=None, quantise: bool = True):
    """The model's forward with E4M3 block projections; returns what ``og.model_forward`` returns.

    The cache feeds ``og.model_backward`` unchanged (straight-through backward).
    With ``quantise=False`` the result is bit-identical to ``og.model_forward``.
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
        y, c["m1"], c["r1"] = og.layernorm_forward(x, P[p + "ln1.g"], P[p + "ln1.b"])
        c["y"] = y
        qkv = _product(y, P[p + "qkv.w"], quantise) + P[p + "qkv.b"]
        q = og._split_heads(qkv[..., 0:C], B, T, H, hd)
        k = og._split_heads(qkv[..., C:2 * C], B, T, H, hd)
        v = og._split_heads(qkv[..., 2 * C:3 * C], B, T, H, hd)
        o, lse = og._attention_per_sequence(og.causal_attention_forward, q, k, v)
        c["q"], c["k"], c["v"], c["lse"] = q, k, v, lse
        of = og._merge_heads(o, B, T, C)
        c["o"] = of
        x1 = x + _product(of, P[p + "proj.w"], quantise) + P[p + "proj.b"]
        c["x1"] = x1
        y2, c["m2"], c["r2"] = og.layernorm_forward(x1, P[p + "ln2.g"], P[p + "ln2.b"])
        c["y2"] = y2
        h = _product(y2, P[p + "fc.w"], quantise) + P[p + "fc.b"]
        c["h"] = h
        g = og.gelu_forward(h)
        x = x1 + _product(g, P[p + "fcproj.w"], quantise) + P[p + "fcproj.b"]
        layers.append(c)
    yf, mf, rf = og.layernorm_forward(x, P["lnf.g"], P["lnf.b"])
    z = yf.reshape(B * T, C) @ P["wte"][:V].T
    cache = {"tokens": tokens, "targets": targets, "layers": layers, "xL": x, "yf": yf, "mf": mf, "rf": rf,
             "z": z, "B": B, "T": T}
    loss = None
    if targets is not None:
        tg = torch.as_tensor(targets).long().reshape(-1)
        loss, lse, rows = og.cross_entropy_forward(z, tg)
        cache["lse"], cache["tg"], cache["rows"] = lse, tg, rows
    return loss, z, cache
