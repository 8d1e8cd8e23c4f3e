"""Pins of the oracle's individual ops against brute force, closed forms and invariants."""
import math

import numpy as np
import pytest
import torch

from oracle import gpt2 as og

F64 = torch.float64


def _rand(*shape, seed=0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=F64)


# ---------------------------------------------------------------- attention

def _brute_attention(q, k, v):
    """Per (i, j) loops with math.exp: causal softmax(q.k / sqrt(hd)) v."""
    T, hd = q.shape
    out = np.zeros((T, hd))
    lse = np.zeros(T)
    for i in range(T):
        s = [sum(q[i, d] * k[j, d] for d in range(hd)) / math.sqrt(hd) for j in range(i + 1)]
        m = max(s)
        w = [math.exp(x - m) for x in s]
        tot = sum(w)
        lse[i] = m + math.log(tot)
        for j in range(i + 1):
            for d in range(hd):
                out[i, d] += w[j] / tot * v[j, d]
    return out, lse


@pytest.mark.parametrize("T,hd", [(1, 4), (5, 3), (8, 8)])
def test_attention_forward_brute_force(T, hd):
    q, k, v = _rand(T, hd, seed=1), _rand(T, hd, seed=2), _rand(T, hd, seed=3)
    o, lse = og.causal_attention_forward(q, k, v)
    ob, lb = _brute_attention(q.numpy(), k.numpy(), v.numpy())
    np.testing.assert_allclose(o.numpy(), ob, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse.numpy(), lb, rtol=1e-12, atol=1e-12)


def test_attention_first_row_copies_v0_and_is_causal():
    q, k, v = _rand(2, 6, 4, seed=4), _rand(2, 6, 4, seed=5), _rand(2, 6, 4, seed=6)
    o, _ = og.causal_attention_forward(q, k, v)
    assert torch.allclose(o[:, 0], v[:, 0])
    k2, v2 = k.clone(), v.clone()
    k2[:, 4:] += 10.0
    v2[:, 4:] -= 3.0
    o2, _ = og.causal_attention_forward(q, k2, v2)
    assert torch.equal(o[:, :4], o2[:, :4])     # future keys/values do not reach the past
    assert not torch.allclose(o[:, 4:], o2[:, 4:])


def test_attention_scale_is_head_size():
    """With identical keys the weights are uniform; with q = k scaled, the logit is |q|^2/sqrt(hd)."""
    hd = 16
    q = _rand(1, hd, seed=7)
    k = q.clone()
    s = og._causal_scores(q, k)
    assert torch.allclose(s[0, 0], (q * q).sum() / math.sqrt(hd))


def _numgrad(f, x, h=1e-6):
    g = torch.zeros_like(x)
    flat = x.view(-1)
    for i in range(flat.numel()):
        old = flat[i].item()
        flat[i] = old + h
        fp = f()
        flat[i] = old - h
        fm = f()
        flat[i] = old
        g.view(-1)[i] = (fp - fm) / (2 * h)
    return g


def test_attention_backward_finite_differences():
    T, hd = 6, 4
    q, k, v = _rand(T, hd, seed=8), _rand(T, hd, seed=9), _rand(T, hd, seed=10)
    w = _rand(T, hd, seed=11)  # loss = sum(w * O)
    f = lambda: float((og.causal_attention_forward(q, k, v)[0] * w).sum())
    dq, dk, dv = og.causal_attention_backward(q, k, v, w)
    for x, g in ((q, dq), (k, dk), (v, dv)):
        torch.testing.assert_close(g, _numgrad(f, x), rtol=1e-6, atol=1e-8)


# ---------------------------------------------------------------- layernorm

def test_attention_bias_gradient_identities():
    """Two identities of the attention backward that the CUDA path uses for the bias of the
    fused Q|K|V projection: a bias added to every key moves all scores of a query by the same
    amount, so the keys' gradients sum to zero over the sequence; a bias added to every value
    adds itself to every output row (each softmax row sums to one), so the values' gradients
    sum to the output gradients' sum.  Checked on the oracle's hand-derived backward, and on
    the gradient of the forward by finite differences in the bias direction."""
    g = torch.Generator().manual_seed(11)
    T, hd = 9, 8
    q, k, v, do = (torch.randn(T, hd, generator=g, dtype=torch.float64) for _ in range(4))
    dq, dk, dv = og.causal_attention_backward(q, k, v, do)
    assert torch.allclose(dk.sum(0), torch.zeros(hd, dtype=torch.float64), atol=1e-12)
    assert torch.allclose(dv.sum(0), do.sum(0), rtol=1e-12, atol=1e-12)
    assert float(dq.sum(0).abs().max()) > 1e-3  # the query part is not degenerate
    bk = torch.randn(hd, generator=g, dtype=torch.float64)
    bv = torch.randn(hd, generator=g, dtype=torch.float64)
    f = lambda kk, vv: float((og.causal_attention_forward(q, kk, vv)[0] * do).sum())
    h = 1e-6
    assert abs((f(k + h * bk, v) - f(k - h * bk, v)) / (2 * h)) < 1e-8
    fd_v = (f(k, v + h * bv) - f(k, v - h * bv)) / (2 * h)
    assert abs(fd_v - float(do.sum(0) @ bv)) < 1e-7


def test_layernorm_invariants():
    x = _rand(5, 64, seed=12) * 3 + 1.5
    g, b = torch.ones(64, dtype=F64), torch.zeros(64, dtype=F64)
    y, mean, rstd = og.layernorm_forward(x, g, b)
    assert torch.allclose(y.mean(-1), torch.zeros(5, dtype=F64), atol=1e-12)
    var = (y * y).mean(-1)
    assert torch.allclose(var, x.var(-1, unbiased=False) / (x.var(-1, unbiased=False) + og.LN_EPS))
    dy = _rand(5, 64, seed=13)
    # dx is orthogonal to 1 for any eps, and to x_hat exactly when eps = 0
    _, mean, rstd = og.layernorm_forward(x, g, b, eps=0.0)
    dx, dg, db = og.layernorm_backward(dy, x, mean, rstd, g)
    xhat = (x - mean) * rstd
    assert torch.allclose(dx.sum(-1), torch.zeros(5, dtype=F64), atol=1e-10)        # orthogonal to 1
    assert torch.allclose((dx * xhat).sum(-1), torch.zeros(5, dtype=F64), atol=1e-9)  # orthogonal to x_hat
    assert torch.allclose(db, dy.sum(0))


def test_layernorm_backward_finite_differences():
    x, g, b = _rand(3, 8, seed=14), _rand(8, seed=15), _rand(8, seed=16)
    w = _rand(3, 8, seed=17)
    f = lambda: float((og.layernorm_forward(x, g, b)[0] * w).sum())
    _, mean, rstd = og.layernorm_forward(x, g, b)
    dx, dg, db = og.layernorm_backward(w, x, mean, rstd, g)
    torch.testing.assert_close(dx, _numgrad(f, x), rtol=1e-6, atol=1e-8)
    torch.testing.assert_close(dg, _numgrad(f, g), rtol=1e-6, atol=1e-8)
    torch.testing.assert_close(db, _numgrad(f, b), rtol=1e-6, atol=1e-8)


# ---------------------------------------------------------------- gelu

def test_gelu_tanh_form_against_exact_gelu():
    """The tanh form approximates x*Phi(x) to ~1e-3 everywhere; limits and slope at 0."""
    h = torch.linspace(-8, 8, 2001, dtype=F64)
    exact = h * 0.5 * (1 + torch.erf(h / math.sqrt(2)))
    assert (og.gelu_forward(h) - exact).abs().max() < 1e-3
    assert og.gelu_forward(torch.tensor([0.0], dtype=F64)).item() == 0.0
    assert abs(og.gelu_derivative(torch.tensor([0.0], dtype=F64)).item() - 0.5) < 1e-15
    assert abs(og.gelu_forward(torch.tensor([10.0], dtype=F64)).item() - 10.0) < 1e-12
    hd = h.clone()
    num = (og.gelu_forward(hd + 1e-6) - og.gelu_forward(hd - 1e-6)) / 2e-6
    assert (num - og.gelu_derivative(h)).abs().max() < 1e-7


# ---------------------------------------------------------------- cross-entropy

def test_cross_entropy_uniform_logits_is_ln_v():
    for V in (2, 256, 50257):
        z = torch.full((3, V), 0.37, dtype=F64)
        loss, _, _ = og.cross_entropy_forward(z, torch.tensor([0, 1, V - 1]))
        assert abs(loss.item() - math.log(V)) < 1e-12


def test_cross_entropy_gradient_rows_sum_to_zero_and_fd():
    z = _rand(4, 10, seed=18)
    t = torch.tensor([3, 0, 9, 3])
    loss, lse, _ = og.cross_entropy_forward(z, t)
    dz = og.cross_entropy_backward(z, lse, t, 2.5)
    assert torch.allclose(dz.sum(-1), torch.zeros(4, dtype=F64), atol=1e-15)
    f = lambda: 2.5 * float(og.cross_entropy_forward(z, t)[0])
    torch.testing.assert_close(dz, _numgrad(f, z), rtol=1e-6, atol=1e-9)


def test_cross_entropy_one_hot_limit():
    z = torch.zeros(1, 5, dtype=F64)
    z[0, 2] = 60.0
    loss, _, _ = og.cross_entropy_forward(z, torch.tensor([2]))
    assert loss.item() < 1e-20 + 4 * math.exp(-60)


# ---------------------------------------------------------------- embedding

def test_embedding_backward_counting_brute_force():
    rng = np.random.default_rng(0)
    B, T, C, Vp = 3, 7, 5, 11
    tokens = torch.from_numpy(rng.integers(0, 6, size=(B, T)))
    dx = _rand(B, T, C, seed=19)
    dwte, dwpe = og.embedding_backward(dx, tokens, Vp, 9)
    for v in range(Vp):
        want = torch.zeros(C, dtype=F64)
        cnt = 0
        for b in range(B):
            for t in range(T):
                if tokens[b, t] == v:
                    want += dx[b, t]
                    cnt += 1
        assert torch.allclose(dwte[v], want)
        if cnt == 0:
            assert (dwte[v] == 0).all()
    assert torch.allclose(dwpe[:T], dx.sum(0))
    assert (dwpe[T:] == 0).all()


# ---------------------------------------------------------------- optimizer

def test_lr_schedule_values():
    assert abs(og.lr_schedule(0) - 6e-4 / 700) < 1e-18
    assert abs(og.lr_schedule(0) - 8.571428571e-7) < 1e-15
    assert abs(og.lr_schedule(19) - 1.7142857142857142e-05) < 1e-15
    assert og.lr_schedule(699) == pytest.approx(6e-4, rel=1e-15)
    assert og.lr_schedule(700) == pytest.approx(6e-4, rel=1e-15)
    mid = 700 + (19073 - 700) / 2
    assert og.lr_schedule(mid) == pytest.approx((6e-4 + 6e-5) / 2, rel=1e-12)
    assert og.lr_schedule(19073) == pytest.approx(6e-5, rel=1e-12)
    assert og.lr_schedule(10 ** 6) == 6e-5
    # monotone decreasing after warmup
    vals = [og.lr_schedule(i) for i in range(700, 19074, 500)]
    assert all(a >= b for a, b in zip(vals, vals[1:]))


def test_adamw_first_step_closed_form_and_clip():
    cfg = og.Config(L=1, C=8, H=2, V=16, Vp=16, T=4, B=1)
    m = og.OracleGPT2(cfg, seed=1)
    p0 = {k: v.clone() for k, v in m.params.items()}
    g = {k: _rand(*v.shape, seed=100 + i) * 1e-3 for i, (k, v) in enumerate(m.params.items())}
    for k in m.grads:
        m.grads[k].copy_(g[k])
    norm0 = og.global_norm(m.grads)
    assert norm0 < 1.0  # no clipping in this case
    lr, wd, eps = 1e-2, 0.1, 1e-8
    ret = m.clip_and_adamw(lr, 0.9, 0.95, eps, wd, 1.0)
    assert ret == pytest.approx(norm0, rel=1e-14)
    for k, p in m.params.items():
        decay = wd if p.dim() == 2 else 0.0
        want = p0[k] * (1 - lr * decay) - lr * g[k] / (g[k].abs() + eps)
        torch.testing.assert_close(p, want, rtol=1e-12, atol=1e-14)


def test_clipping_scales_norm_to_clip():
    cfg = og.Config(L=1, C=8, H=2, V=16, Vp=16, T=4, B=1)
    m = og.OracleGPT2(cfg, seed=1)
    for i, (k, v) in enumerate(m.grads.items()):
        v.copy_(_rand(*v.shape, seed=200 + i))
    norm = og.global_norm(m.grads)
    assert norm > 1.0
    coef = min(1.0, 1.0 / (norm + 1e-6))
    clipped = math.sqrt(sum(float(((g * coef) ** 2).sum()) for g in m.grads.values()))
    assert clipped == pytest.approx(1.0, rel=1e-5)
    # with beta1 = 0 the first step's m equals the clipped gradient
    ret = m.clip_and_adamw(1e-3, 0.0, 0.95, 1e-8, 0.0, 1.0)
    assert ret == pytest.approx(norm)
    mnorm = math.sqrt(sum(float((x ** 2).sum()) for x in m.m.values()))
    assert mnorm == pytest.approx(1.0, rel=1e-5)
