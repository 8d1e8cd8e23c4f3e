"""Whole-step pins of the oracle: finite differences and an autograd cross-check."""
import numpy as np
import pytest
import torch

from oracle import gpt2 as og

TINY = og.Config(L=2, C=16, H=2, V=32, Vp=40, T=8, B=2)


def _batch(cfg, seed=0):
    rng = np.random.default_rng(seed)
    x = torch.from_numpy(rng.integers(0, cfg.V, size=(cfg.B, cfg.T)))
    y = torch.from_numpy(rng.integers(0, cfg.V, size=(cfg.B, cfg.T)))
    return x, y


def _perturbed(P, seed=5):
    """Init params with zero biases and unit gains moved off their special values."""
    g = torch.Generator().manual_seed(seed)
    Q = {k: v.clone() for k, v in P.items()}
    for k, v in Q.items():
        v += 0.05 * torch.randn(v.shape, generator=g, dtype=v.dtype)
    Q["wte"][TINY.V:] = 0.0
    return Q


def _loss(cfg, P, x, y):
    return float(og.model_forward(cfg, P, x, y)[0])


@pytest.mark.parametrize("grad_scale", [1.0, 0.25])
def test_step_gradients_central_differences(grad_scale):
    """Every parameter element vs central differences (h=1e-5): relative error <= 1e-3."""
    cfg = TINY
    P = _perturbed(og.init_params(cfg, seed=3))
    x, y = _batch(cfg)
    _, _, cache = og.model_forward(cfg, P, x, y)
    G = og.model_backward(cfg, P, cache, grad_scale)
    h = 1e-5
    for name, p in P.items():
        flat = p.view(-1)
        n = flat.numel()
        idx = range(n) if n <= 4096 else np.random.default_rng(1).choice(n, 64, replace=False)
        fd = torch.zeros(len(idx), dtype=torch.float64)
        an = G[name].reshape(-1)[list(idx)]
        for j, i in enumerate(idx):
            old = flat[i].item()
            flat[i] = old + h
            lp = _loss(cfg, P, x, y)
            flat[i] = old - h
            lm = _loss(cfg, P, x, y)
            flat[i] = old
            fd[j] = grad_scale * (lp - lm) / (2 * h)
        scale = max(fd.abs().max().item(), 1e-12)
        err = (fd - an).abs().max().item() / scale
        assert err <= 1e-3, (name, err)
    # padded vocabulary rows get no gradient
    assert (G["wte"][cfg.V:] == 0).all()


def test_step_gradients_match_autograd():
    """Hand-derived backward equals torch autograd through the same forward."""
    cfg = og.Config(L=2, C=32, H=4, V=50, Vp=64, T=12, B=3)
    P = _perturbed(og.init_params(cfg, seed=4))
    P["wte"][cfg.V:] = 0.0
    x, y = _batch(cfg, seed=2)
    _, _, cache = og.model_forward(cfg, P, x, y)
    G = og.model_backward(cfg, P, cache, 1.0)
    Pa = {k: v.clone().requires_grad_(True) for k, v in P.items()}
    loss, _, _ = og.model_forward(cfg, Pa, x, y)
    loss.backward()
    for k in P:
        torch.testing.assert_close(G[k], Pa[k].grad, rtol=1e-9, atol=1e-12)
