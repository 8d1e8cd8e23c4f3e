"""Pins of the oracle's sampling rule and generation loop (no GPU).

The rule: candidates are the top_k logits (larger first, equal values lower
index first); token = first candidate whose cumulative weight
exp((z_i - z_max) / temperature) exceeds u * sum.  What pins it:
* an inverse-CDF draw is correct when the set of u in [0, 1) that selects
  candidate i has measure softmax(z / temperature)_i over the candidates, and
  the intervals come in candidate order;
* top_k = 1 is the argmax with the lower index winning ties, for every u;
* a vanishing temperature turns any top_k into the argmax;
* generation equals teacher forcing: every drawn token is the draw from the
  forward pass over the sequence before it;
* non-finite maxima (+inf, or every candidate -inf) draw exactly as the limit
  of large finite logits: as if the infinite entries were equal finite values
  far from the rest.
"""
import math

import numpy as np
import torch

from oracle import gpt2 as og


def _draws(z, temperature, top_k, n=100001):
    us = (np.arange(n) + 0.5) / n
    return np.array([og.sample_next(z, temperature, top_k, u) for u in us])


def test_preimage_measures_are_the_softmax_over_the_candidates():
    z = np.array([0.3, -1.2, 2.0, 0.3, 0.0])
    temperature, top_k, n = 0.7, 3, 100001
    d = _draws(z, temperature, top_k, n)
    cand = [2, 0, 3]  # 2.0 first, then the two 0.3 in index order
    w = np.exp((z[cand] - z.max()) / temperature)
    p = w / w.sum()
    for i, pi in zip(cand, p):
        assert abs((d == i).mean() - pi) <= 2.0 / n
    assert not np.isin(d, [1, 4]).any()  # outside the top 3
    # the intervals follow the candidate order: u below p0 draws 2, then 0, then 3
    first = [int(np.argmax(d == i)) for i in cand]
    assert first == sorted(first)


def test_full_candidate_set_matches_softmax_of_all_logits():
    rng = np.random.default_rng(3)
    z = rng.normal(size=7)
    n = 70001
    d = _draws(z, 1.3, 7, n)
    p = np.exp(z / 1.3) / np.exp(z / 1.3).sum()
    for i in range(7):
        assert abs((d == i).mean() - p[i]) <= 2.0 / n


def test_top1_is_argmax_with_lower_index_on_ties():
    z = np.array([1.0, 5.0, 5.0, 2.0])
    for u in (0.0, 0.3, 0.999999):
        assert og.sample_next(z, 1.0, 1, u) == 1
        assert og.sample_next(z, 0.01, 4, u * 0.5) == 1  # tiny temperature: argmax side of the tie


def test_small_temperature_tends_to_argmax():
    z = np.array([0.1, 0.4, -0.2, 0.39])
    for u in np.linspace(0.0, 0.99, 11):
        assert og.sample_next(z, 1e-4, 4, float(u)) == 1


def _tiny():
    cfg = og.Config.from_dict(dict(L=1, C=16, H=2, V=20, Vp=20, T=12, B=2, dtype="fp32"))
    P = og.init_params(cfg, 5)
    gen = torch.Generator().manual_seed(0)
    for k in P:  # larger weights than the init so the logits spread out
        if P[k].dim() == 2:
            P[k] = torch.randn(P[k].shape, generator=gen, dtype=torch.float64) * 0.5
    return cfg, P


def test_generation_equals_teacher_forcing():
    cfg, P = _tiny()
    prompt = torch.tensor([[3, 7, 1], [0, 19, 4]])
    n_new = 6
    uniforms = np.random.default_rng(1).random((n_new, 2))
    for temperature, top_k in ((1.0, 1), (0.8, 5), (1.5, 20)):
        seq, drawn = og.generate(cfg, P, prompt, n_new, temperature, top_k, uniforms)
        assert seq.shape == (2, 3 + n_new)
        assert torch.equal(seq[:, :3], prompt)
        for s in range(n_new):
            t = 3 + s
            _, z, _ = og.model_forward(cfg, P, seq[:, :t], None)
            last = z.reshape(2, t, -1)[:, -1, :]
            assert torch.allclose(last, drawn[s], rtol=0, atol=1e-12)
            for b in range(2):
                assert int(seq[b, t]) == og.sample_next(last[b].numpy(), temperature, top_k, float(uniforms[s][b]))
                if top_k == 1:
                    assert int(seq[b, t]) == int(torch.argmax(last[b]))


def test_nonfinite_maximum_draws_as_the_finite_limit():
    n = 20001
    inf = float("inf")
    cases = [
        # one +inf: always that entry
        (np.array([0.3, -1.2, inf, 0.3, 0.0]), np.array([0.3, -1.2, 1e300, 0.3, 0.0])),
        # two +inf: the two, half each, lower index first
        (np.array([inf, -1.2, inf, 0.3]), np.array([1e300, -1.2, 1e300, 0.3])),
        # every candidate -inf: uniform over the top_k lowest indices
        (np.array([-inf, -inf, -inf, -inf]), np.array([-1e300, -1e300, -1e300, -1e300])),
    ]
    for z_inf, z_big in cases:
        for top_k in (1, 3, 4):
            a = _draws(z_inf, 0.7, top_k, n)
            b = _draws(z_big, 0.7, top_k, n)
            assert np.array_equal(a, b), (z_inf, top_k)
    d = _draws(cases[1][0], 1.0, 4, n)
    assert set(np.unique(d)) == {0, 2} and abs((d == 0).mean() - 0.5) <= 2.0 / n
