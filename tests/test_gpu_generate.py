"""KV-cached generation and top-k sampling on the GPU against the oracle.

* The sampler alone (gpt2_op_sample) on bf16 logits: the drawn token equals the
  oracle's draw from the same values wherever u * sum(w) is not within 1e-5
  (relative) of a cumulative boundary, and is a neighbour candidate otherwise.
* fp32 mode: the generated sequence equals the oracle's generation (full
  recompute per token) with the same uniforms, up to the first draw whose
  boundary margin is below 1e-5.
* bf16 mode: greedy tokens are the oracle's argmax of the teacher-forced
  logits within the bf16 tolerance; the logits of the last draw match the
  oracle's and the GPU's own full forward.
* Argument and token errors return their codes and leave the model usable.
"""
import math

import numpy as np
import pytest
import torch

import synthetic
from oracle import gpt2 as og

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gpt_decoder_only_train_b300 import build

    build.build()
    import gpt_decoder_only_train_b300 as mod

    mod.lib()
    return mod


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def _margin(z, temperature, top_k, u):
    """Distance (relative to the weight sum) from u * sum(w) to the nearest cumulative boundary."""
    z = np.asarray(z, dtype=np.float64)
    order = np.lexsort((np.arange(z.shape[0]), -z))[:top_k]
    w = np.exp((z[order] - z[order[0]]) / temperature)
    cum = np.cumsum(w)
    return float(np.min(np.abs(cum[:-1] - u * cum[-1])) / cum[-1]) if len(w) > 1 else 1.0


@pytest.mark.parametrize("V,ldl", [(50257, 50304), (1000, 1024), (70, 72)])
def test_sampler_matches_the_oracle_rule(g, V, ldl):
    rng = np.random.default_rng(V)
    B = 16
    z = torch.from_numpy(rng.normal(scale=3.0, size=(B, ldl)).astype(np.float32)).to(torch.bfloat16)
    z[:, V:] = 100.0  # padding columns are never candidates
    u = rng.random(B).astype(np.float32)
    zd, ud = z.cuda(), torch.from_numpy(u).cuda()
    out = torch.empty(B, dtype=torch.int32, device="cuda")
    for temperature, top_k in ((1.0, 1), (0.7, 5), (1.0, 50), (1.5, 128)):
        g.sample(zd, ldl, B, V, ud, temperature, top_k, out)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        for b in range(B):
            zb = z[b, :V].double().numpy()
            ref = og.sample_next(zb, temperature, top_k, float(u[b]))
            if _margin(zb, temperature, top_k, float(u[b])) > 1e-5:
                assert got[b] == ref, (b, temperature, top_k)
            else:
                order = list(np.lexsort((np.arange(V), -zb))[:top_k])
                assert abs(order.index(int(got[b])) - order.index(ref)) <= 1


def test_sampler_nonfinite_maximum_matches_the_oracle(g):
    """+inf logits, and rows whose candidates are all -inf, follow the oracle's limit rule."""
    V, ldl, B = 300, 304, 6
    rng = np.random.default_rng(11)
    z = torch.from_numpy(rng.normal(size=(B, ldl)).astype(np.float32)).to(torch.bfloat16)
    inf = float("inf")
    z[0, 17] = inf                      # one +inf
    z[1, 5] = inf
    z[1, 250] = inf                     # two +inf
    z[2, :V] = -inf                     # every logit -inf
    z[3, :V] = -inf
    z[3, 40] = 2.0                      # one finite logit among -inf
    z[4, 3] = -inf                      # finite maximum, a -inf candidate excluded by its weight
    z[5, 299] = inf                     # +inf in the last real column
    zd = z.cuda()
    out = torch.empty(B, dtype=torch.int32, device="cuda")
    for top_k in (1, 2, 7):
        for u0 in (0.05, 0.45, 0.55, 0.95):
            u = np.full(B, u0, dtype=np.float32)
            g.sample(zd, ldl, B, V, torch.from_numpy(u).cuda(), 0.8, top_k, out)
            torch.cuda.synchronize()
            got = out.cpu().numpy()
            for b in range(B):
                ref = og.sample_next(z[b, :V].double().numpy(), 0.8, top_k, float(u[b]))
                assert got[b] == ref, (b, top_k, u0, int(got[b]), ref)


def _peaked(g, cfg, seed, scale):
    """GPU model and oracle parameters with the 2-D weights scaled (spread-out logits)."""
    m = g.GPT2(cfg, seed=seed)
    P = og.init_params(og.Config.from_dict(cfg), seed)
    for i, name in enumerate(m.names):
        if P[name].dim() == 2 and name != "wpe":
            P[name] = (P[name] * scale).float().double()
            m.set_params(i, P[name].numpy().astype(np.float32))
    return m, P


def test_fp32_generation_equals_the_oracle(g):
    cfg = dict(L=2, C=64, H=4, V=256, Vp=256, T=32, B=2, dtype="fp32", recompute_gelu=0)
    ocfg = og.Config.from_dict(cfg)
    m, P = _peaked(g, cfg, 11, 8.0)
    rng = np.random.default_rng(2)
    T0, T_total = 4, 20
    prompt = rng.integers(0, cfg["V"], size=(2, T0))
    uniforms = rng.random((T_total - T0, 2)).astype(np.float32)
    for temperature, top_k in ((1.0, 1), (0.9, 20), (1.3, 128)):
        seq = np.zeros((2, T_total), dtype=np.int32)
        seq[:, :T0] = prompt
        sd = _dev(seq)
        m.generate(sd, T0, torch.from_numpy(uniforms).cuda(), temperature, top_k)
        got = sd.cpu().numpy()
        ref, drawn = og.generate(ocfg, P, prompt, T_total - T0, temperature, top_k, uniforms.astype(np.float64))
        ref = ref.numpy()
        assert np.array_equal(got[:, :T0], prompt)
        for b in range(2):
            for t in range(T0, T_total):
                if got[b, t] != ref[b, t]:
                    # only a draw on a boundary may differ; the sequences diverge after it
                    assert _margin(drawn[t - T0, b].numpy(), temperature, top_k, float(uniforms[t - T0, b])) < 1e-5
                    break
    m.close()


SMALL_BF16 = dict(L=2, C=128, H=2, V=500, Vp=512, T=64, B=3, dtype="bf16", recompute_gelu=0)


def test_bf16_greedy_generation_follows_the_oracle(g):
    cfg = SMALL_BF16
    ocfg = og.Config.from_dict(cfg)
    m, P = _peaked(g, cfg, 4, 6.0)
    rng = np.random.default_rng(5)
    B, T0, T_total = 3, 5, 40
    seq = np.zeros((B, T_total), dtype=np.int32)
    seq[:, :T0] = rng.integers(0, cfg["V"], size=(B, T0))
    sd = _dev(seq)
    u = torch.zeros(T_total - T0, B, device="cuda")
    m.generate(sd, T0, u, 1.0, 1)
    got = sd.cpu().numpy()
    last_gpu = m.debug_tensor("logits", torch.bfloat16, (B, cfg["Vp"]))[:, :cfg["V"]].double().cpu().clone()
    assert np.array_equal(got[:, :T0], seq[:, :T0])
    assert ((got >= 0) & (got < cfg["V"])).all()
    # teacher forcing on the GPU's own sequence
    _, z, _ = og.model_forward(ocfg, P, got.astype(np.int64), None)
    z = z.reshape(B, T_total, -1)
    for t in range(T0, T_total):
        zt = z[:, t - 1, :]
        for b in range(B):
            top = float(zt[b].max())
            assert float(zt[b, got[b, t]]) >= top - 2e-2 * max(1.0, abs(top)), (b, t)
    # the logits of the last draw (position T_total - 2)
    ref = z[:, T_total - 2, :]
    err = (last_gpu - ref).abs().max().item()
    assert err <= 2e-2 * ref.abs().max().item()
    # the same position through the GPU's full forward
    m.forward(_dev(got[:, :T_total - 1]), None)
    torch.cuda.synchronize()
    full = m.debug_tensor("logits", torch.bfloat16, (B * (T_total - 1), cfg["Vp"]))
    full = full.reshape(B, T_total - 1, cfg["Vp"])[:, T_total - 2, :cfg["V"]].double().cpu()
    assert (full - last_gpu).abs().max().item() <= 2e-2 * ref.abs().max().item()
    m.close()


def test_124m_greedy_generation_follows_the_oracle(g):
    w = dict(synthetic.WORKLOADS["gpt2_124m"])
    m = g.GPT2(w, seed=w["seed"])
    ocfg = og.Config.from_dict(w)
    P = og.init_params(ocfg, w["seed"])
    B, T0, T_total = 2, 8, 16
    x, _ = synthetic.zipf_window(w["seed"], B, T0, w["V"])
    seq = np.zeros((B, T_total), dtype=np.int32)
    seq[:, :T0] = x
    sd = _dev(seq)
    m.generate(sd, T0, torch.zeros(T_total - T0, B, device="cuda"), 1.0, 1)
    got = sd.cpu().numpy()
    _, z, _ = og.model_forward(ocfg, P, got.astype(np.int64), None)
    z = z.reshape(B, T_total, -1)
    for t in range(T0, T_total):
        for b in range(B):
            zt = z[b, t - 1]
            top = float(zt.max())
            assert float(zt[got[b, t]]) >= top - 2e-2 * max(1.0, abs(top)), (b, t)
    m.close()


def test_generation_errors_leave_the_model_usable(g):
    cfg = SMALL_BF16
    m = g.GPT2(cfg, seed=2)
    B, T_total, T0 = 2, 10, 3
    seq = _dev(np.ones((B, T_total)))
    u = torch.zeros(T_total - T0, B, device="cuda")
    for kwargs, code in ((dict(top_k=0), -8), (dict(top_k=129), -8), (dict(temperature=0.0), -8)):
        args = dict(temperature=1.0, top_k=1)
        args.update(kwargs)
        with pytest.raises(g.Gpt2Error) as e:
            m.generate(seq, T0, u, **args)
        assert e.value.status == code
    with pytest.raises(g.Gpt2Error) as e:
        m.generate(_dev(np.ones((B, cfg["T"] + 1))), T0, u)
    assert e.value.status == -2
    with pytest.raises(g.Gpt2Error) as e:
        m.generate(seq, 0, u)
    assert e.value.status == -2
    bad = np.ones((B, T_total))
    bad[1, 1] = cfg["V"]
    with pytest.raises(g.Gpt2Error) as e:
        m.generate(_dev(bad), T0, u)
    assert e.value.status == -3
    m.generate(seq, T0, u)  # the next valid call succeeds
    with pytest.raises(g.Gpt2Error) as e:
        m.backward(1.0)  # generation leaves no forward to differentiate
    assert e.value.status == -10
    x, y = synthetic.zipf_window(1, cfg["B"], cfg["T"], cfg["V"])
    loss = m.forward(_dev(x), _dev(y))
    m.backward(1.0)
    assert math.isfinite(loss)
    m.close()


def test_generation_is_the_bf16_path_in_every_mode(g):
    """Sampling decodes with the bf16 weights whatever the training forward's precision or LM-head
    mode: an E4M3-forward model and a fused-LM-head model draw the same tokens as the plain one."""
    cfg = SMALL_BF16
    rng = np.random.default_rng(9)
    B, T0, T_total = 3, 6, 30
    prompt = rng.integers(0, cfg["V"], size=(B, T0))
    uniforms = torch.from_numpy(rng.random((T_total - T0, B)).astype(np.float32)).cuda()
    out = []
    for mode in ({}, {"fp8_forward": 1}, {"fused_lm_head": 1}):
        m, _ = _peaked(g, dict(cfg, **mode), 12, 6.0)
        seq = np.zeros((B, T_total), dtype=np.int32)
        seq[:, :T0] = prompt
        sd = _dev(seq)
        m.generate(sd, T0, uniforms, 0.9, 20)
        out.append(sd.cpu().numpy())
        m.close()
    assert np.array_equal(out[0], out[1]) and np.array_equal(out[0], out[2])
