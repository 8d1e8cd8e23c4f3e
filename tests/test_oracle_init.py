"""Pins of the oracle's initialiser and of the shared input generators."""
import math
import os

import numpy as np
import pytest
import scipy.stats

import synthetic
from oracle import init_lib
from oracle.gpt2 import Config, init_params, param_specs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_ints(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [int(l, 16) for l in f if l.strip() and not l.startswith("#")]


def test_splitmix64_published_outputs():
    """Both SplitMix64 implementations reproduce the generator's published outputs for seed 0."""
    expected = _golden_ints("splitmix64_seed0.txt")
    lib = init_lib()
    gamma = 0x9E3779B97F4A7C15
    state = 0
    for want in expected:
        assert lib.oracle_sm64(state) == want
        assert int(synthetic.sm64(np.uint64(state))) == want
        state = (state + gamma) % (1 << 64)


def test_draw_addressing_matches_between_oracle_and_inputs():
    lib = init_lib()
    d = synthetic.draws(7, 3, 16, offset=5)
    for i in range(16):
        assert lib.oracle_draw(7, 3, 5 + i) == int(d[i])


def test_normal_fill_moments_and_ks():
    """Box-Muller draws are N(0,1): moments and a Kolmogorov-Smirnov test."""
    lib = init_lib()
    n = 200_000
    buf = np.zeros(n, dtype=np.float32)
    lib.oracle_normal_fill(123, 9, n, 1.0, buf.ctypes.data)
    x = buf.astype(np.float64)
    assert abs(x.mean()) < 0.01
    assert abs(x.std() - 1.0) < 0.01
    assert abs(scipy.stats.skew(x)) < 0.03
    assert abs(scipy.stats.kurtosis(x)) < 0.06
    assert scipy.stats.kstest(x, "norm").pvalue > 1e-3


def test_normal_fill_matches_its_written_definition():
    """The C fill equals the documented formula evaluated with Python's libm."""
    lib = init_lib()
    n = 64
    buf = np.zeros(n, dtype=np.float32)
    lib.oracle_normal_fill(5, 2, n, 0.02, buf.ctypes.data)
    for i in range(n):
        a = lib.oracle_draw(5, 2, 2 * i)
        b = lib.oracle_draw(5, 2, 2 * i + 1)
        u1 = ((a >> 11) + 1) * 2.0 ** -53
        u2 = (b >> 11) * 2.0 ** -53
        z = math.sqrt(-2.0 * math.log(u1)) * math.cos(6.283185307179586 * u2)
        assert np.float32(0.02 * z) == buf[i]


def test_init_params_structure():
    cfg = Config(L=2, C=32, H=2, V=100, Vp=112, T=16, B=1)
    P = init_params(cfg, seed=11)
    specs = param_specs(cfg)
    assert list(P.keys()) == [s[0] for s in specs]
    assert len(specs) == 2 + 12 * cfg.L + 2
    wte = P["wte"]
    assert wte.shape == (cfg.Vp, cfg.C)
    assert (wte[cfg.V:] == 0).all()           # padded rows are zero
    assert (wte[: cfg.V].abs() > 0).float().mean() > 0.99
    for name, shape, kind, std, decay in specs:
        t = P[name]
        assert tuple(t.shape) == shape
        assert decay == (len(shape) == 2)
        if kind == "ones":
            assert (t == 1).all()
        if kind == "zeros":
            assert (t == 0).all()
        # values are exactly representable in fp32
        assert (t.float().double() == t).all()


def test_init_std_and_residual_scaling():
    cfg = Config(L=4, C=128, H=4, V=512, Vp=512, T=64, B=1)
    P = init_params(cfg, seed=3)
    assert abs(P["h0.qkv.w"].std().item() - 0.02) < 0.001
    assert abs(P["h1.fc.w"].std().item() - 0.02) < 0.001
    want = 0.02 / math.sqrt(2 * cfg.L)
    assert abs(P["h2.proj.w"].std().item() - want) < 0.1 * want
    assert abs(P["h3.fcproj.w"].std().item() - want) < 0.05 * want


def test_uniform_tokens_range_and_independence():
    x, y = synthetic.uniform_batch(0, 2, 32, 256)
    assert x.shape == (2, 32) and x.dtype == np.int32
    assert x.min() >= 0 and x.max() < 256 and y.min() >= 0 and y.max() < 256
    assert (x != y).mean() > 0.9
    big = synthetic.uniform_tokens(0, 0, 256_000, 256)
    counts = np.bincount(big, minlength=256)
    assert scipy.stats.chisquare(counts).pvalue > 1e-4


def test_zipf_frequencies_match_cdf():
    """Empirical rank frequencies of the Zipf(1.1) stream match its CDF (chi-square)."""
    V = 1000
    n = 400_000
    tok = synthetic.zipf_tokens(1, n, V)
    assert tok.min() >= 0 and tok.max() < V
    counts = np.bincount(tok, minlength=V)
    k = np.arange(1, V + 1, dtype=np.float64)
    p = k ** -1.1
    p /= p.sum()
    # pool the tail so every expected count is >= 20
    exp = p * n
    small = np.nonzero(exp < 20)[0]
    cut = int(small[0]) if len(small) else V
    obs, ex = counts[:cut].astype(np.float64), exp[:cut]
    if cut < V:
        obs, ex = np.append(obs, counts[cut:].sum()), np.append(ex, exp[cut:].sum())
    assert scipy.stats.chisquare(obs, ex).pvalue > 1e-4
    # rank 1 is the most common token and the stream covers many ranks
    assert counts.argmax() == 0


def test_zipf_window_shift_and_advance():
    x0, y0 = synthetic.zipf_window(2, 2, 8, 50257, micro_step=0)
    x1, _ = synthetic.zipf_window(2, 2, 8, 50257, micro_step=1)
    flat_x0, flat_y0 = x0.reshape(-1), y0.reshape(-1)
    assert (flat_y0[:-1] == flat_x0[1:]).all()   # targets are inputs shifted by one
    assert flat_y0[-1] == x1.reshape(-1)[0]      # the next window starts where this one ended
    assert x0.max() < 50257


def test_attention_operands_are_bf16_values():
    import torch
    q, k, v, do = synthetic.attention_operands(4, 1, 2, 16, 8)
    for a in (q, k, v, do):
        t = torch.from_numpy(a)
        assert (t.to(torch.bfloat16).float() == t).all()
        assert a.shape == (1, 16, 2, 8)
