"""Pins of the oracle's E4M3 quantisation (no GPU).

What pins it (the format as the OCP 8-bit floating point specification
defines it: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
infinities, NaN at exponent and mantissa all ones, round to nearest even,
saturating conversion):
* decoding: each of the 256 codes by the format's formula written out
  separately here per field, and the printed limits 448, 2^-6, 2^-9;
* every finite code re-encodes to itself;
* rounding equals a brute-force nearest search over all finite values, with
  ties to the code whose mantissa is even, on random and on exactly-halfway
  inputs; values beyond 448 saturate;
* row quantisation: each row's largest magnitude maps to 448 and every
  element is within half a quantum of the scaled value.
"""
import numpy as np

from oracle import fp8


def _finite_table():
    codes = np.arange(256, dtype=np.uint8)
    vals = fp8.e4m3_decode(codes)
    ok = ~np.isnan(vals)
    return codes[ok], vals[ok]


def test_decode_matches_the_format_fields():
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        v = fp8.e4m3_decode(np.uint8(c))
        if e == 15 and m == 7:
            assert np.isnan(v)
            continue
        mag = m / 8.0 * 2.0 ** (1 - 7) if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        assert v == (-mag if s else mag), c
    assert fp8.e4m3_decode(np.uint8(0x7E)) == 448.0
    assert fp8.e4m3_decode(np.uint8(0x08)) == 2.0 ** -6
    assert fp8.e4m3_decode(np.uint8(0x01)) == 2.0 ** -9
    assert fp8.e4m3_decode(np.uint8(0x38)) == 1.0


def test_every_finite_code_round_trips():
    codes, vals = _finite_table()
    back = fp8.e4m3_encode(vals)
    zero = vals == 0
    assert np.array_equal(back[~zero], codes[~zero])
    assert set(back[zero].tolist()) <= {0x00, 0x80}


def _nearest_brute(x, vals, codes):
    """Nearest finite value; on a tie, the one whose code (mantissa) is even."""
    out = np.empty_like(x)
    for i, xi in enumerate(x):
        if abs(xi) > 448.0:
            out[i] = np.sign(xi) * 448.0
            continue
        d = np.abs(vals - xi)
        best = np.flatnonzero(d == d.min())
        if len(best) > 1:
            best = [b for b in best if codes[b] % 2 == 0] or best
        out[i] = vals[best[0]]
    return out


def test_rounding_is_the_nearest_value_ties_to_even():
    codes, vals = _finite_table()
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(scale=s, size=400) for s in (1e-3, 0.05, 1.0, 30.0, 300.0)])
    # exactly halfway between neighbours (positive values, sorted)
    pos = np.unique(vals[vals >= 0])
    mids = (pos[:-1] + pos[1:]) / 2.0
    x = np.concatenate([x, mids, -mids, [500.0, -1e6, 448.0, 464.0, 479.0]])
    got = fp8.e4m3_round(x)
    want = _nearest_brute(x, vals, codes)
    assert np.array_equal(np.abs(got), np.abs(want))
    assert np.array_equal(np.signbit(got) | (got == 0), np.signbit(want) | (want == 0))


def test_rounding_error_is_at_most_half_a_quantum():
    rng = np.random.default_rng(1)
    x = rng.uniform(-448, 448, size=20000) * rng.choice([1e-4, 1e-2, 1.0], size=20000)
    r = fp8.e4m3_round(x)
    a = np.abs(x)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    q = np.where(a < 2.0 ** -6, 2.0 ** -9, 2.0 ** (e - 3))
    assert (np.abs(r - x) <= q / 2 + 1e-300).all()


def test_row_quantisation_maps_amax_to_448_and_stays_within_bounds():
    rng = np.random.default_rng(2)
    x = (rng.normal(size=(16, 96)) * rng.uniform(0.01, 10, size=(16, 1))).astype(np.float32)
    x[3] = 0.0
    codes, inv = fp8.quantize_rows(x)
    deq = fp8.e4m3_decode(codes) * inv[:, None].astype(np.float64)
    assert (codes[3] == 0).all() and inv[3] == 1.0
    for m in range(16):
        if m == 3:
            continue
        amax = np.abs(x[m]).max()
        assert np.abs(fp8.e4m3_decode(codes[m])).max() == 448.0
        # half a quantum of the scaled value (relative 2^-4 for normals), plus the fp32 steps
        assert (np.abs(deq[m] - x[m]) <= np.abs(x[m]) * 2.0 ** -4 + amax * 2.0 ** -9 / 448 * 8 + 1e-12).all()


def test_matmul_is_the_decoded_product():
    rng = np.random.default_rng(3)
    a = rng.normal(size=(8, 64)).astype(np.float32)
    b = rng.normal(size=(5, 64)).astype(np.float32)
    qa, ai = fp8.quantize_rows(a)
    qb, bi = fp8.quantize_tensor(b)
    d = fp8.matmul_e4m3(qa, ai, qb, bi, bias=np.arange(5.0))
    ref = (fp8.e4m3_decode(qa) * ai[:, None]) @ (fp8.e4m3_decode(qb) * bi).T + np.arange(5.0)
    assert np.allclose(d, ref, rtol=1e-12, atol=1e-12)
    # and close to the unquantised product (E4M3 keeps 3 mantissa bits)
    assert np.abs(d - (a @ b.T + np.arange(5.0))).max() <= 0.2 * np.abs(a @ b.T).max()


# ---- the E4M3 forward of the model ------------------------------------------------

TINY = dict(L=2, C=32, H=2, V=61, Vp=64, T=8, B=2)


def _tiny_model(seed=7):
    from oracle import gpt2 as og

    cfg = og.Config.from_dict(TINY)
    P = og.init_params(cfg, seed)
    # larger weights than the initial 0.02 so that the blocks move the logits
    rng = np.random.default_rng(seed)
    for k, v in P.items():
        if v.dim() == 2:
            P[k] = v * 10.0
        elif not k.endswith(".g"):
            P[k] = torch.from_numpy(rng.normal(scale=0.1, size=v.shape))
    tok = torch.from_numpy(rng.integers(0, TINY["V"], size=(TINY["B"], TINY["T"])))
    tg = torch.from_numpy(rng.integers(0, TINY["V"], size=(TINY["B"], TINY["T"])))
    return og, cfg, P, tok, tg


import torch  # noqa: E402


def test_e4m3_forward_without_quantiser_is_the_float64_forward():
    og, cfg, P, tok, tg = _tiny_model()
    l0, z0, _ = og.model_forward(cfg, P, tok, tg)
    l1, z1, _ = fp8.model_forward_e4m3(cfg, P, tok, tg, quantise=False)
    assert float(l0) == float(l1)
    assert torch.equal(z0, z1)


def _brute_dequantised(x2d, per_row: bool):
    """E4M3 quantise-dequantise by nearest-value search over the finite codes (ties to the
    even code): scale 448 / amax and factor amax / 448 in fp32, per row or per tensor."""
    codes, vals = _finite_table()
    x32 = np.asarray(x2d, dtype=np.float32)
    amax = np.abs(x32).max(axis=1, keepdims=True) if per_row else np.abs(x32).max(keepdims=True)
    safe = np.where(amax > 0, amax, np.float32(1))
    s = np.where(amax > 0, np.float32(448) / safe, np.float32(1)).astype(np.float32)
    inv = np.where(amax > 0, safe / np.float32(448), np.float32(1)).astype(np.float32)
    scaled = (x32 * s).astype(np.float64)
    d = np.abs(scaled[..., None] - vals)
    best = d == d.min(-1, keepdims=True)
    pick = np.where(best & (codes % 2 == 0), 0, 1) + np.where(best, 0, 2)  # even ties first, then any
    v = vals[np.argmin(pick, axis=-1)]
    return v * inv.astype(np.float64)


def test_e4m3_forward_products_are_the_quantised_products():
    og, cfg, P, tok, tg = _tiny_model()
    _, _, cache = fp8.model_forward_e4m3(cfg, P, tok, tg)
    C = cfg.C
    for l, c in enumerate(cache["layers"]):
        p = "h%d." % l
        # the cache keeps every projection's input and output
        checks = [
            (c["y"], P[p + "qkv.w"], P[p + "qkv.b"],
             torch.cat([og._merge_heads(t, cfg.B, cfg.T, C) for t in (c["q"], c["k"], c["v"])], -1)),
            (c["o"], P[p + "proj.w"], P[p + "proj.b"], c["x1"] - c["x"]),
            (c["y2"], P[p + "fc.w"], P[p + "fc.b"], c["h"]),
        ]
        nxt = cache["layers"][l + 1]["x"] if l + 1 < cfg.L else cache["xL"]
        checks.append((og.gelu_forward(c["h"]), P[p + "fcproj.w"], P[p + "fcproj.b"], nxt - c["x1"]))
        for x, w, b, got in checks:
            xq = _brute_dequantised(x.reshape(-1, x.shape[-1]).numpy(), per_row=True)
            wq = _brute_dequantised(w.to(torch.bfloat16).double().numpy(), per_row=False)
            want = torch.from_numpy(xq @ wq.T).reshape(got.shape) + b
            scale = (x.abs() @ w.abs().T).reshape(got.shape) + b.abs() + 1
            assert ((got - want).abs() <= 1e-12 * scale).all(), l
            # and it is not the unquantised product
            assert not torch.allclose(got, x @ w.T + b, rtol=1e-6, atol=0)


def test_e4m3_forward_backward_is_straight_through():
    og, cfg, P, tok, tg = _tiny_model()
    loss, _, cache = fp8.model_forward_e4m3(cfg, P, tok, tg)
    l0, _, cache0 = og.model_forward(cfg, P, tok, tg)
    # the loss differs from the float64 forward's by quantisation noise only
    assert float(loss) != float(l0)
    assert abs(float(loss) - float(l0)) < 0.05 * float(l0)
    # the backward of the quantised forward's cache is the float64 backward evaluated at
    # that forward's activations: close to the unquantised gradients, tensor by tensor
    G = og.model_backward(cfg, P, cache)
    G0 = og.model_backward(cfg, P, cache0)
    for k in G:
        a, b = G[k].flatten(), G0[k].flatten()
        if float(b.norm()) == 0.0:
            continue
        cos = float(a @ b / (a.norm() * b.norm()))
        assert cos > 0.98, (k, cos)
