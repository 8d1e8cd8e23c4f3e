"""Training-level pins of the oracle: initial loss, overfitting one batch, causality."""
import math

import numpy as np
import pytest
import torch

import synthetic
from oracle import gpt2 as og


def test_initial_loss_tiny_is_ln_v():
    w = synthetic.WORKLOADS["tiny_fp32"]
    cfg = og.Config.from_dict(w)
    x, y = synthetic.step_batch(w)
    m = og.OracleGPT2(cfg, w["seed"])
    loss = m.forward(x, y)
    assert abs(loss - math.log(cfg.V)) <= 0.05


@pytest.mark.slow
def test_initial_loss_124m_shapes():
    """At the 124M shapes the init loss is ln V + sigma^2/2 with sigma^2 = 0.02^2 * C.

    The final LayerNorm output has squared norm C and the tied wte rows are
    N(0, 0.02^2), so the logits are ~N(0, 0.02^2 C) and E[logsumexp] ~= ln V +
    sigma^2/2 (0.154 above ln 50257 at C = 768).
    """
    w = dict(synthetic.WORKLOADS["gpt2_124m"])
    cfg = og.Config.from_dict(w)
    B, T = 8, 256
    x, y = synthetic.zipf_window(w["seed"], B, T, cfg.V)
    m = og.OracleGPT2(cfg, w["seed"])
    loss = m.forward(x, y)
    want = math.log(cfg.V) + 0.02 ** 2 * cfg.C / 2
    assert abs(loss - want) <= 0.05, (loss, want)


def test_overfit_one_batch():
    """One fixed batch of the tiny workload is driven to loss < 0.1 ("overfit test")."""
    w = synthetic.WORKLOADS["tiny_fp32"]
    cfg = og.Config.from_dict(w)
    x, y = synthetic.step_batch(w)
    m = og.OracleGPT2(cfg, w["seed"])
    loss = None
    for it in range(400):
        loss = m.forward(x, y)
        if loss < 0.1:
            break
        m.backward(1.0)
        m.clip_and_adamw(3e-3, 0.9, 0.95, 1e-8, 0.0, 1.0)
        m.zero_grad()
    assert loss < 0.1, loss


def test_logits_are_causal():
    cfg = og.Config(L=2, C=32, H=4, V=64, Vp=64, T=16, B=1)
    m = og.OracleGPT2(cfg, seed=9)
    rng = np.random.default_rng(3)
    x = rng.integers(0, cfg.V, size=(1, cfg.T))
    z0 = m.logits(x)
    x2 = x.copy()
    x2[0, 9] = (x2[0, 9] + 1) % cfg.V
    z1 = m.logits(x2)
    assert torch.equal(z0[:9], z1[:9])
    assert not torch.allclose(z0[9:], z1[9:])


def test_gradient_accumulation_equals_big_batch():
    """Two micro-steps with grad_scale 1/2 equal one step over both halves of the batch."""
    cfg = og.Config(L=1, C=16, H=2, V=32, Vp=32, T=8, B=4)
    rng = np.random.default_rng(4)
    x = rng.integers(0, cfg.V, size=(4, 8))
    y = rng.integers(0, cfg.V, size=(4, 8))
    a = og.OracleGPT2(cfg, seed=1)
    a.forward(x, y)
    a.backward(1.0)
    b = og.OracleGPT2(cfg, seed=1)
    for s in (slice(0, 2), slice(2, 4)):
        b.forward(x[s], y[s])
        b.backward(0.5)
    for k in a.grads:
        torch.testing.assert_close(a.grads[k], b.grads[k], rtol=1e-10, atol=1e-14)
