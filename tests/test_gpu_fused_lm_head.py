"""The LM head fused with the cross-entropy (fused_lm_head) against the oracle and
against the step with stored logits, through the C ABI.

The fused mode computes the same loss and gradients as the plain definition
("Let's reproduce GPT-2 (124M)", §Bölümler 4: the mean over all positions of
logsumexp(z) - z[target] over the real vocabulary), so it carries the bf16
step's tolerances against the oracle: |loss - ref| <= 2e-2, per-tensor
gradient cosine >= 0.995, norm within 2%.  Against the stored-logits step on
the same weights the two differ only in where the logits are rounded (the
fused path takes lse and dlogits from fp32 logits, the classifier from bf16
ones): per-position losses within 2e-2 and every gradient's cosine >= 0.999.
Configurations cover one and several backward chunks (8,192 positions each,
with a ragged last chunk) and a vocabulary that is not a multiple of the tile.
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


def _cos(a, b):
    a = np.asarray(a, dtype=np.float64).reshape(-1)
    b = np.asarray(b, dtype=np.float64).reshape(-1)
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if na == 0 and nb == 0:
        return 1.0
    return float(a @ b / (na * nb))


SMALL = dict(L=2, C=128, H=2, V=500, Vp=512, T=192, B=3, dtype="bf16", recompute_gelu=0, fused_lm_head=1)
RAGGED = dict(L=1, C=192, H=3, V=1000, Vp=1024, T=77, B=2, dtype="bf16", recompute_gelu=0, fused_lm_head=1)
CHUNKED = dict(L=1, C=128, H=2, V=700, Vp=768, T=1024, B=9, dtype="bf16", recompute_gelu=0, fused_lm_head=1)


@pytest.mark.parametrize("cfg", [SMALL, RAGGED, CHUNKED], ids=["small", "ragged", "two_chunks"])
def test_fused_step_parity(g, cfg):
    seed = 31
    m = g.GPT2(cfg, seed=seed)
    ref = og.OracleGPT2(og.Config.from_dict(cfg), seed)
    x, y = synthetic.zipf_window(seed, cfg["B"], cfg["T"], cfg["V"])
    loss = m.forward(_dev(x), _dev(y))
    ref_loss = ref.forward(x, y)
    assert abs(loss - ref_loss) <= 2e-2, (loss, ref_loss)
    m.backward(1.0)
    ref.backward(1.0)
    for i, name in enumerate(m.names):
        c = _cos(m.grads(i), ref.grads[name].numpy())
        assert c >= 0.995, (name, c)
    norm = m.clip_and_adamw(6e-4)
    ref_norm = ref.clip_and_adamw(6e-4)
    assert abs(norm - ref_norm) <= 0.02 * ref_norm
    assert (m.grads(0)[cfg["V"]:] == 0).all() and (m.params(0)[cfg["V"]:] == 0).all()
    m.close()


@pytest.mark.parametrize("cfg", [SMALL, CHUNKED], ids=["small", "two_chunks"])
def test_fused_matches_stored_logits_step(g, cfg):
    seed = 32
    x, y = synthetic.zipf_window(seed, cfg["B"], cfg["T"], cfg["V"])
    out = []
    for fused in (1, 0):
        m = g.GPT2(dict(cfg, fused_lm_head=fused), seed=seed)
        loss = m.forward(_dev(x), _dev(y))
        BT = cfg["B"] * cfg["T"]
        rows = m.debug_tensor("loss_rows", torch.float32, (BT,)).cpu().numpy().copy()
        m.backward(0.5)
        out.append((loss, rows, [m.grads(i) for i in range(len(m.names))]))
        m.close()
    (l1, r1, g1), (l0, r0, g0) = out
    assert abs(l1 - l0) <= 1e-2
    assert np.abs(r1 - r0).max() <= 2e-2
    for a, b in zip(g1, g0):
        assert _cos(a, b) >= 0.999


def test_fused_accumulation_and_optimizer_steps(g):
    """Two optimizer steps of two micro-steps each against the oracle (grad_scale = 1/2)."""
    cfg = dict(SMALL, B=2, T=128)
    seed, lr = 33, 2e-3
    m = g.GPT2(cfg, seed=seed)
    ref = og.OracleGPT2(og.Config.from_dict(cfg), seed)
    for step in range(2):
        m.zero_grad()
        ref.zero_grad()
        for j in range(2):
            x, y = synthetic.zipf_window(seed, cfg["B"], cfg["T"], cfg["V"], micro_step=2 * step + j)
            loss = m.forward(_dev(x), _dev(y))
            ref_loss = ref.forward(x, y)
            assert abs(loss - ref_loss) <= 2e-2, (step, j, loss, ref_loss)
            m.backward(0.5)
            ref.backward(0.5)
        norm = m.clip_and_adamw(lr)
        ref_norm = ref.clip_and_adamw(lr)
        assert abs(norm - ref_norm) <= 0.02 * ref_norm, (step, norm, ref_norm)
    m.close()


def test_fused_errors_and_logits_only(g):
    cfg = CHUNKED
    m = g.GPT2(cfg, seed=34)
    x, y = synthetic.zipf_window(34, cfg["B"], cfg["T"], cfg["V"])
    # logits without targets: at most one chunk of positions
    with pytest.raises(g.Gpt2Error) as e:
        m.forward(_dev(x), None)
    assert e.value.status == -9  # GPT2_ERR_UNSUPPORTED
    xs = x[:2]
    m.forward(_dev(xs), None)
    ref = g.GPT2(dict(cfg, fused_lm_head=0), seed=34)
    ref.forward(_dev(xs), None)
    n = 2 * cfg["T"] * cfg["Vp"]
    a = m.debug_tensor("logits", torch.bfloat16, (n,)).float().cpu()
    b = ref.debug_tensor("logits", torch.bfloat16, (n,)).float().cpu()
    assert torch.equal(a, b)
    ref.close()
    # an out-of-range target is reported; the model stays usable
    yb = y.copy()
    yb[1, 5] = cfg["V"] + 3
    with pytest.raises(g.Gpt2Error) as e:
        m.forward(_dev(x), _dev(yb))
    assert e.value.status == -3  # GPT2_ERR_BAD_TOKEN
    loss = m.forward(_dev(x), _dev(y))
    assert math.isfinite(loss)
    m.backward(1.0)
    m.close()
