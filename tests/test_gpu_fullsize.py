"""Parity at the full workload sizes, in the launch configuration the benchmark times.

* GPT-2 124M, B=16, T=1024 (bf16): the whole step against the fp64 oracle on
  the same seeded batch -- loss within 2e-2, every gradient tensor cosine
  >= 0.995, clipped-norm / AdamW update consistent.
* GPT-2 350M (L=24, C=1024, H=16) with GELU recompute: the whole step on one
  T=1024 sequence against the oracle -- loss within 2e-2, every gradient tensor
  cosine >= 0.995, norm within 2%; at B=8, per-position losses of a sampled
  sequence against the oracle (each sequence's forward is independent) and the
  recompute property at full size (loss bit-identical, grads equal to fp32
  summation noise with and without recompute).
* 32-micro-step accumulation (124M): the first two optimizer steps of the
  recipe (warmup learning rate, clip 1.0, AdamW) against the oracle's loss
  curve, computed once by tests/golden/make_accum32_curve.py and stored with a
  hash of the oracle code it came from -- every micro-step loss and both step
  losses within 2e-2, the step-1 gradient norm within 2%; and accumulated
  gradients equal the mean of the per-micro-step gradients (linearity).
* Causal attention sweep (H=12, hd=64, B*T = 65536): every head at T=256 and
  sampled heads at T=1024/2048/4096 against the naive fp64 oracle.
"""
import importlib.util
import json
import math
import os

import numpy as np
import pytest
import torch

import synthetic
from oracle import fp8 as of
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


def _cos(a, b):
    a = np.asarray(a, dtype=np.float64).reshape(-1)
    b = np.asarray(b, dtype=np.float64).reshape(-1)
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    return 1.0 if na == nb == 0 else float(a @ b / (na * nb))


def test_124m_full_step_parity(g):
    torch.set_num_threads(max(1, torch.get_num_threads()))
    w = synthetic.WORKLOADS["gpt2_124m"]
    x, y = synthetic.step_batch(w)
    m = g.GPT2(w, seed=w["seed"])
    loss = m.forward(_dev(x), _dev(y))
    m.backward(1.0)
    gpu_grads = [m.grads(i) for i in range(len(m.names))]
    norm = m.clip_and_adamw(6e-4)
    ref = og.OracleGPT2(og.Config.from_dict(w), w["seed"])
    ref_loss = ref.forward(x, y)
    assert abs(loss - ref_loss) <= 2e-2, (loss, ref_loss)
    ref.backward(1.0)
    worst = (1.0, None)
    for i, name in enumerate(m.names):
        c = _cos(gpu_grads[i], ref.grads[name].numpy())
        worst = min(worst, (c, name))
    assert worst[0] >= 0.995, worst
    # magnitudes too (a product counted twice or missed keeps the cosine): the projection
    # weight gradients, two of which share a launch per block, within 3% in norm
    for i, name in enumerate(m.names):
        if name.endswith(".w") and any(k in name for k in ("qkv", "proj", "fc")):
            r = np.linalg.norm(gpu_grads[i]) / np.linalg.norm(ref.grads[name].numpy())
            assert 0.97 <= r <= 1.03, (name, r)
    ref_norm = og.global_norm(ref.grads)
    assert abs(norm - ref_norm) <= 0.02 * ref_norm, (norm, ref_norm)
    assert (gpu_grads[0][w["V"]:] == 0).all()


def test_124m_e4m3_forward_sampled_sequence_and_gradients(g):
    """E4M3 block projections at 124M: the full batch in the bench's launch configuration,
    one sampled sequence's per-position losses against the oracle's E4M3 forward, and the
    gradients of that sequence (a B=1 call) against its straight-through backward."""
    w = dict(synthetic.WORKLOADS["gpt2_124m"], fp8_forward=1)
    x, y = synthetic.step_batch(w)
    m = g.GPT2(w, seed=w["seed"])
    loss = m.forward(_dev(x), _dev(y))
    assert math.isfinite(loss)
    rows = m.debug_tensor("loss_rows", torch.float32, (w["B"] * w["T"],)).cpu().numpy().reshape(w["B"], w["T"])
    b = 5
    ref = og.OracleGPT2(og.Config.from_dict(dict(w, B=1)), w["seed"])
    ref_loss, _, cache = of.model_forward_e4m3(ref.cfg, ref.params, x[b:b + 1], y[b:b + 1])
    ref_rows = cache["rows"].numpy().reshape(-1)
    assert abs(rows[b].mean() - float(ref_loss)) <= 2e-2
    assert np.corrcoef(rows[b], ref_rows)[0, 1] >= 0.99
    m.zero_grad()
    m.forward(_dev(x[b:b + 1]), _dev(y[b:b + 1]))
    m.backward(1.0)
    G = og.model_backward(ref.cfg, ref.params, cache)
    worst = (1.0, None)
    for i, name in enumerate(m.names):
        worst = min(worst, (_cos(m.grads(i), G[name].numpy()), name))
    assert worst[0] >= 0.99, worst
    m.close()


def test_124m_fused_lm_head_matches_stored_logits(g):
    """The LM head fused with the cross-entropy at 124M (two backward chunks of 8,192 positions):
    per-position losses within 2e-2 of the step with stored logits, every gradient's cosine
    >= 0.999, the same norm within 0.5%, and the padded vocabulary rows untouched."""
    w = synthetic.WORKLOADS["gpt2_124m"]
    x, y = synthetic.step_batch(w)
    BT = w["B"] * w["T"]
    out = []
    for fused in (1, 0):
        m = g.GPT2(dict(w, fused_lm_head=fused), seed=w["seed"])
        loss = m.forward(_dev(x), _dev(y))
        rows = m.debug_tensor("loss_rows", torch.float32, (BT,)).cpu().numpy().copy()
        m.backward(1.0)
        grads = [m.grads(i) for i in range(len(m.names))]
        norm = m.clip_and_adamw(6e-4)
        out.append((loss, rows, grads, norm))
        m.close()
        del m
        torch.cuda.empty_cache()
    (l1, r1, g1, n1), (l0, r0, g0, n0) = out
    assert abs(l1 - l0) <= 1e-2
    assert np.abs(r1 - r0).max() <= 2e-2
    for a, b in zip(g1, g0):
        assert _cos(a, b) >= 0.999
    assert abs(n1 - n0) <= 0.005 * n0
    assert (g1[0][w["V"]:] == 0).all()


def test_350m_recompute_sampled_rows_and_property(g):
    w = synthetic.WORKLOADS["gpt2_350m_recompute"]
    x, y = synthetic.step_batch(w)
    m = g.GPT2(w, seed=w["seed"])
    loss = m.forward(_dev(x), _dev(y))
    rows = m.debug_tensor("loss_rows", torch.float32, (w["B"] * w["T"],)).cpu().numpy().reshape(w["B"], w["T"])
    m.backward(1.0)
    grads_r = {i: m.grads(i) for i in (2, 10, 24 * 12 + 1)}
    norm_r = m.clip_and_adamw(6e-4)
    m.close()
    del m
    torch.cuda.empty_cache()
    # the sampled sequence b = 3 against the oracle (sequences do not interact)
    b = 3
    ref = og.OracleGPT2(og.Config.from_dict(dict(w, B=1)), w["seed"])
    _, _, cache = og.model_forward(ref.cfg, ref.params, x[b:b + 1], y[b:b + 1])
    ref_rows = cache["rows"].numpy()
    assert abs(rows[b].mean() - ref_rows.mean()) <= 2e-2
    assert np.abs(rows[b] - ref_rows).max() <= 0.15
    assert np.corrcoef(rows[b], ref_rows)[0, 1] >= 0.99
    # recompute changes nothing but memory
    m2 = g.GPT2(dict(w, recompute_gelu=0), seed=w["seed"])
    loss2 = m2.forward(_dev(x), _dev(y))
    m2.backward(1.0)
    assert loss2 == loss
    for i, a in grads_r.items():
        bb = m2.grads(i)
        assert np.abs(a - bb).max() <= 1e-5 * max(np.abs(bb).max(), 1e-30), i
    assert abs(m2.clip_and_adamw(6e-4) - norm_r) <= 1e-5 * norm_r
    m2.close()


def test_124m_embedding_gradients_bitwise_reproducible(g):
    """At 124M, B=16, T=1024: two backward passes of the same batch give bit-identical wte
    and wpe gradients."""
    w = synthetic.WORKLOADS["gpt2_124m"]
    x, y = synthetic.step_batch(w)
    m = g.GPT2(w, seed=w["seed"])
    res = []
    for _ in range(2):
        m.zero_grad()
        m.forward(_dev(x), _dev(y))
        m.backward(1.0)
        res.append((m.grads(0), m.grads(1)))
    m.close()
    assert res[0][0].tobytes() == res[1][0].tobytes()
    assert res[0][1].tobytes() == res[1][1].tobytes()
    assert np.abs(res[0][0]).max() > 0


def test_350m_recompute_one_sequence_gradient_parity(g):
    """The 350M step with GELU recompute on one full-length sequence: loss, every gradient
    tensor and the global norm against the fp64 oracle."""
    w = synthetic.WORKLOADS["gpt2_350m_recompute"]
    x, y = synthetic.step_batch(w)
    b = 3
    x1, y1 = x[b:b + 1].copy(), y[b:b + 1].copy()
    cfg = dict(w, B=1)
    m = g.GPT2(cfg, seed=w["seed"])
    loss = m.forward(_dev(x1), _dev(y1))
    m.backward(1.0)
    gpu_grads = [m.grads(i) for i in range(len(m.names))]
    norm = m.clip_and_adamw(6e-4)
    names = list(m.names)
    m.close()
    del m
    torch.cuda.empty_cache()
    ref = og.OracleGPT2(og.Config.from_dict(cfg), w["seed"])
    ref_loss = ref.forward(x1, y1)
    assert abs(loss - ref_loss) <= 2e-2, (loss, ref_loss)
    ref.backward(1.0)
    worst = (1.0, None)
    for i, name in enumerate(names):
        worst = min(worst, (_cos(gpu_grads[i], ref.grads[name].numpy()), name))
    assert worst[0] >= 0.995, worst
    ref_norm = og.global_norm(ref.grads)
    assert abs(norm - ref_norm) <= 0.02 * ref_norm, (norm, ref_norm)
    assert (gpu_grads[0][w["V"]:] == 0).all()


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden_maker():
    spec = importlib.util.spec_from_file_location("make_accum32_curve", os.path.join(GOLDEN, "make_accum32_curve.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_accum32_two_step_loss_curve_vs_oracle(g):
    """Two optimizer steps of 32 micro-steps (B=16, T=1024) at the warmup learning rate,
    against the oracle's stored curve (tests/golden/gpt2_124m_accum32_curve.json)."""
    mk = _golden_maker()
    with open(mk.OUT) as f:
        gold = json.load(f)
    assert gold["sources_sha256"] == mk.source_hash(), "oracle code changed: regenerate the golden curve"
    w = synthetic.WORKLOADS["gpt2_124m_accum32"]
    assert (gold["seed"], gold["B"], gold["T"], gold["micro_steps"]) == (w["seed"], w["B"], w["T"], 32)
    a = gold["adamw"]
    m = g.GPT2(w, seed=w["seed"])
    for it, st in enumerate(gold["steps"]):
        m.zero_grad()
        losses = []
        for i in range(32):
            x, y = synthetic.zipf_window(w["seed"], w["B"], w["T"], w["V"], micro_step=it * 32 + i)
            losses.append(m.forward(_dev(x), _dev(y)))
            m.backward(1.0 / 32)
        diffs = np.abs(np.array(losses) - np.array(st["micro_losses"]))
        assert diffs.max() <= 2e-2, (it, diffs.max())
        assert abs(np.mean(losses) - st["loss"]) <= 2e-2, (it, np.mean(losses), st["loss"])
        assert st["lr"] == og.lr_schedule(it)
        norm = m.clip_and_adamw(st["lr"], a["beta1"], a["beta2"], a["eps"], a["wd"], a["clip"])
        if st["grad_norm"] is not None:
            assert abs(norm - st["grad_norm"]) <= 0.02 * st["grad_norm"], (it, norm, st["grad_norm"])
    m.close()


def test_accumulation_is_linear_124m(g):
    w = synthetic.WORKLOADS["gpt2_124m_accum32"]
    n = 4
    batches = [synthetic.zipf_window(w["seed"], w["B"], w["T"], w["V"], micro_step=i) for i in range(n)]
    m = g.GPT2(w, seed=w["seed"])
    ids = (2, 4 + 12, len(m.names) - 2)
    losses = []
    for x, y in batches:
        losses.append(m.forward(_dev(x), _dev(y)))
        m.backward(1.0 / n)
    acc = {i: m.grads(i).astype(np.float64) for i in ids}
    mean = {i: np.zeros_like(acc[i]) for i in ids}
    for x, y in batches:
        m.zero_grad()
        m.forward(_dev(x), _dev(y))
        m.backward(1.0)
        for i in ids:
            mean[i] += m.grads(i) / n
    for i in ids:
        assert np.abs(acc[i] - mean[i]).max() <= 1e-4 * np.abs(mean[i]).max(), i
    # the first micro-step's loss against the oracle (loss only: forward of all 16 sequences)
    ref = og.OracleGPT2(og.Config.from_dict(w), w["seed"])
    assert abs(losses[0] - ref.forward(*batches[0])) <= 2e-2


@pytest.mark.parametrize("T,B", [(256, 256), (1024, 64), (2048, 32), (4096, 16)])
def test_attention_sweep(g, T, B):
    H, hd = 12, 64
    q, k, v, do = [torch.from_numpy(a) for a in synthetic.attention_operands(4, B, H, T, hd)]
    dev = lambda a: a.to(torch.bfloat16).cuda().contiguous()
    qd, kd, vd, dod = dev(q), dev(k), dev(v), dev(do)
    o = torch.empty_like(qd)
    lse = torch.empty(B, H, T, dtype=torch.float32, device="cuda")
    g.attention_forward(qd, kd, vd, o, lse, B, T, H)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(qd), torch.empty_like(qd)
    scratch = torch.empty(B * H * T, dtype=torch.float32, device="cuda")
    g.attention_backward(qd, kd, vd, o, dod, lse, dq, dk, dv, scratch, B, T, H)
    # and the backward the model and the sweep's "bwd" run: dS kept in a workspace
    dq2, dk2, dv2 = torch.empty_like(qd), torch.empty_like(qd), torch.empty_like(qd)
    ds = torch.empty(g.attention_backward_ds_bytes(B, T, H), dtype=torch.uint8, device="cuda")
    g.attention_backward_ds(qd, kd, vd, o, dod, lse, dq2, dk2, dv2, scratch, ds, B, T, H)
    torch.cuda.synchronize()
    del ds
    if T == 256:
        heads = [(b, h) for b in range(B) for h in range(H)]
    else:
        rng = np.random.default_rng(T)
        heads = [(int(rng.integers(B)), int(rng.integers(H))) for _ in range(3)] + [(B - 1, H - 1)]
    o_c, lse_c = o.cpu().double(), lse.cpu().double()
    outs = [t.cpu().double() for t in (dq, dk, dv)]
    outs2 = [t.cpu().double() for t in (dq2, dk2, dv2)]
    bs = sorted({b for b, _ in heads})
    for b in bs:
        hs = [h for bb, h in heads if bb == b]
        sel = lambda a: a[b, :, hs].permute(1, 0, 2).double()
        Q, K, Vv, dO = sel(q), sel(k), sel(v), sel(do)
        ro, rl = og.causal_attention_forward(Q, K, Vv)
        rq, rk, rv = og.causal_attention_backward(Q, K, Vv, dO)
        for hi, h in enumerate(hs):
            def chk(out, ref, tol_e, tol_f):
                err = (out - ref).abs().max().item()
                fro = ((out - ref).norm() / ref.norm()).item()
                assert err <= tol_e * ref.abs().max().item() and fro <= tol_f, (T, b, h, err, fro)
            chk(o_c[b, :, h], ro[hi], 2e-2, 1e-2)
            assert (lse_c[b, h] - rl[hi]).abs().max().item() < 2e-3
            for out, ref in zip(outs + outs2, (rq, rk, rv) * 2):
                chk(out[b, :, h], ref[hi], 4e-2, 2e-2)
