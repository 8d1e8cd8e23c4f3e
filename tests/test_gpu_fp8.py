"""E4M3 (FP8) quantisation and matmul on the GPU against the oracle (oracle/fp8.py).

* Quantisation is integer work decided by fp32 arithmetic on both sides: the
  codes and the dequantisation factors equal the oracle's bit for bit, per row
  and per tensor, including a row of zeros.
* The matmul: D = a_inv[m] b_inv sum_k A(m,k) B(n,k) on E4M3 codes with the
  bf16 epilogues (bias, residual, GELU).  The oracle quantises the same bf16
  inputs itself and multiplies the decoded codes in float64; the products of
  two E4M3 values are exact in fp32, so the GPU's error is the fp32
  accumulation and one bf16 rounding: |D - ref| <= 2^-8 |ref| + 1e-3 max|ref|.
  Shapes are ragged in M and N and cover single-CTA and CTA-pair tiles.
* The model with E4M3 block projections (fp8_forward) against the oracle's
  E4M3 forward (model_forward_e4m3) and its straight-through backward: the
  GPU quantises the bf16 activations it stores, the oracle its float64 ones,
  so a few codes per row sit one quantum apart and the comparison carries
  the bf16 step's tolerances, |loss - ref| <= 2e-2 and per-tensor gradient
  cosine >= 0.99, also over optimizer steps at a learning rate that moves
  the weights by several E4M3 quanta per step (stale weight codes would show).
"""
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


def _bf16(rng, shape, scale=1.0, row_scales=False):
    x = rng.normal(size=shape) * scale
    if row_scales:
        x *= rng.uniform(1e-3, 30.0, size=(shape[0], 1))
    t = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    return t, t.float().numpy()


def test_row_quantisation_is_bit_exact(g):
    rng = np.random.default_rng(0)
    M, K = 300, 768
    x, xf = _bf16(rng, (M, K), row_scales=True)
    x[7] = 0
    xf[7] = 0
    q = torch.empty(M, K, dtype=torch.uint8, device="cuda")
    inv = torch.empty(M, dtype=torch.float32, device="cuda")
    g.quantize_e4m3_rows(x.cuda(), q, inv, M, K)
    torch.cuda.synchronize()
    rq, rinv = of.quantize_rows(xf)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert inv.cpu().numpy().tobytes() == rinv.astype(np.float32).tobytes()


def test_tensor_quantisation_is_bit_exact(g):
    rng = np.random.default_rng(1)
    w, wf = _bf16(rng, (384, 768), scale=0.02)
    q = torch.empty(384, 768, dtype=torch.uint8, device="cuda")
    inv = torch.empty(1, dtype=torch.float32, device="cuda")
    work = torch.empty(1, dtype=torch.int32, device="cuda")
    g.quantize_e4m3_tensor(w.cuda(), q, inv, work)
    torch.cuda.synchronize()
    rq, rinv = of.quantize_tensor(wf)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert inv.cpu().numpy()[0] == rinv


def _check(out, ref, what):
    err = np.abs(out - ref)
    tol = 2.0 ** -8 * np.abs(ref) + 1e-3 * np.abs(ref).max()
    assert (err <= tol).all(), (what, float(err.max()), float((err - tol).max()))


@pytest.mark.parametrize("M,N,K,epi", [
    (300, 384, 768, "store"),      # ragged M and N, single-CTA tiles
    (257, 256, 512, "residual"),
    (200, 640, 768, "gelu"),
    (2048, 2304, 768, "store"),    # CTA-pair tiles (N >= 2048)
    (1024, 768, 3072, "residual"),  # long K: CTA pairs
])
def test_e4m3_matmul_matches_the_oracle(g, M, N, K, epi):
    rng = np.random.default_rng(M + N + K)
    a, af = _bf16(rng, (M, K), row_scales=True)
    b, bf = _bf16(rng, (N, K), scale=0.02)
    bias = torch.from_numpy(rng.normal(size=N).astype(np.float32))
    qa = torch.empty(M, K, dtype=torch.uint8, device="cuda")
    ainv = torch.empty(M, dtype=torch.float32, device="cuda")
    qb = torch.empty(N, K, dtype=torch.uint8, device="cuda")
    binv = torch.empty(1, dtype=torch.float32, device="cuda")
    work = torch.empty(1, dtype=torch.int32, device="cuda")
    g.quantize_e4m3_rows(a.cuda(), qa, ainv, M, K)
    g.quantize_e4m3_tensor(b.cuda(), qb, binv, work)
    D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    D2 = torch.empty_like(D) if epi == "gelu" else None
    R = None
    rf = None
    if epi == "residual":
        rt, rf = _bf16(rng, (M, N))
        R = rt.cuda()
    e = {"store": g.EPI_STORE, "residual": g.EPI_RESIDUAL, "gelu": g.EPI_GELU}[epi]
    g.matmul_e4m3(qa, ainv, qb, binv, D, M, N, K, epilogue=e, D2=D2, R=R, bias=bias.cuda())
    torch.cuda.synchronize()
    # the oracle quantises the same inputs itself
    rqa, rainv = of.quantize_rows(af)
    rqb, rbinv = of.quantize_tensor(bf)
    ref = of.matmul_e4m3(rqa, rainv, rqb, rbinv, bias=bias.numpy())
    if epi == "residual":
        ref = ref + rf
    out = D.float().cpu().numpy()
    _check(out, ref, epi)
    if epi == "gelu":
        # GELU of the stored (bf16) pre-activation against the oracle's GELU of its own h
        g2 = D2.float().cpu().numpy()
        rg = og.gelu_forward(torch.from_numpy(ref)).numpy()
        err = np.abs(g2 - rg)
        assert (err <= 2.0 ** -7 * np.abs(ref) * 1.2 + 2e-3 * np.abs(rg).max()).all(), float(err.max())


def test_e4m3_matmul_full_size_sampled_rows(g):
    """The MLP up-projection shape (16384 x 3072 x 768), rows sampled against the oracle."""
    M, N, K = 16384, 3072, 768
    rng = np.random.default_rng(5)
    a, af = _bf16(rng, (M, K))
    b, bf = _bf16(rng, (N, K), scale=0.02)
    qa = torch.empty(M, K, dtype=torch.uint8, device="cuda")
    ainv = torch.empty(M, dtype=torch.float32, device="cuda")
    qb = torch.empty(N, K, dtype=torch.uint8, device="cuda")
    binv = torch.empty(1, dtype=torch.float32, device="cuda")
    work = torch.empty(1, dtype=torch.int32, device="cuda")
    g.quantize_e4m3_rows(a.cuda(), qa, ainv, M, K)
    g.quantize_e4m3_tensor(b.cuda(), qb, binv, work)
    D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    g.matmul_e4m3(qa, ainv, qb, binv, D, M, N, K)
    torch.cuda.synchronize()
    rows = np.sort(rng.choice(M, 24, replace=False))
    rqa, rainv = of.quantize_rows(af[rows])
    rqb, rbinv = of.quantize_tensor(bf)
    ref = of.matmul_e4m3(rqa, rainv, rqb, rbinv)
    _check(D.float().cpu().numpy()[rows], ref, "full size")


# ---- the model's E4M3 forward -------------------------------------------------------

SMALL_F8 = dict(L=2, C=128, H=2, V=500, Vp=512, T=192, B=3, dtype="bf16", recompute_gelu=0, fp8_forward=1)
RAGGED_F8 = dict(L=1, C=192, H=3, V=1000, Vp=1024, T=77, B=2, dtype="bf16", recompute_gelu=0, fp8_forward=1)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def _cos(a, b):
    a = np.asarray(a, dtype=np.float64).reshape(-1)
    b = np.asarray(b, dtype=np.float64).reshape(-1)
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if na == 0 and nb == 0:
        return 1.0
    return float(a @ b / (na * nb))


def _oracle_e4m3_micro_step(ref, x, y, grad_scale=1.0):
    loss, _, cache = of.model_forward_e4m3(ref.cfg, ref.params, x, y)
    ref._cache = cache
    ref.backward(grad_scale)
    return float(loss)


@pytest.mark.parametrize("cfg", [SMALL_F8, RAGGED_F8, dict(SMALL_F8, recompute_gelu=1)],
                         ids=["small", "ragged", "gelu_recompute"])
def test_e4m3_forward_step_parity(g, cfg):
    seed = 21
    m = g.GPT2(cfg, seed=seed)
    ref = og.OracleGPT2(og.Config.from_dict(cfg), seed)
    x, y = synthetic.zipf_window(seed, cfg["B"], cfg["T"], cfg["V"])
    loss = m.forward(_dev(x), _dev(y))
    m.backward(1.0)
    ref_loss = _oracle_e4m3_micro_step(ref, x, y)
    assert abs(loss - ref_loss) <= 2e-2, (loss, ref_loss)
    for i, name in enumerate(m.names):
        c = _cos(m.grads(i), ref.grads[name].numpy())
        assert c >= 0.99, (name, c)
    norm = m.clip_and_adamw(6e-4)
    ref_norm = ref.clip_and_adamw(6e-4)
    assert abs(norm - ref_norm) <= 0.02 * ref_norm
    # the quantiser is active: the bf16 forward of the same weights gives another loss
    m16 = g.GPT2(dict(cfg, fp8_forward=0), seed=seed)
    assert m16.forward(_dev(x), _dev(y)) != loss
    m16.close()
    m.close()


def test_e4m3_forward_follows_the_oracle_over_optimizer_steps(g):
    cfg = dict(SMALL_F8, B=2, T=128)
    seed, lr = 5, 3e-3
    m = g.GPT2(cfg, seed=seed)
    ref = og.OracleGPT2(og.Config.from_dict(cfg), seed)
    for step in range(3):
        x, y = synthetic.zipf_window(seed, cfg["B"], cfg["T"], cfg["V"], micro_step=step)
        m.zero_grad()
        ref.zero_grad()
        loss = m.forward(_dev(x), _dev(y))
        m.backward(1.0)
        ref_loss = _oracle_e4m3_micro_step(ref, x, y)
        assert abs(loss - ref_loss) <= 2e-2, (step, loss, ref_loss)
        norm = m.clip_and_adamw(lr)
        ref_norm = ref.clip_and_adamw(lr)
        assert abs(norm - ref_norm) <= 0.02 * ref_norm, (step, norm, ref_norm)
    m.close()


def test_e4m3_weight_codes_follow_set_params(g):
    """Weights written through the ABI are re-quantised before the next forward."""
    cfg = SMALL_F8
    m = g.GPT2(cfg, seed=3)
    ref = og.OracleGPT2(og.Config.from_dict(cfg), 3)
    rng = np.random.default_rng(0)
    for i, name in enumerate(m.names):
        if len(m.shapes[i]) == 2 and name != "wte" and name != "wpe":
            w = (rng.normal(size=m.shapes[i]) * 0.08).astype(np.float32)
            m.set_params(i, w)
            ref.params[name] = torch.from_numpy(w.astype(np.float64))
    x, y = synthetic.zipf_window(3, cfg["B"], cfg["T"], cfg["V"])
    loss = m.forward(_dev(x), _dev(y))
    ref_loss, _, _ = of.model_forward_e4m3(ref.cfg, ref.params, x, y)
    assert abs(loss - float(ref_loss)) <= 2e-2, (loss, float(ref_loss))
    m.close()


def test_e4m3_model_codes_and_first_product(g):
    """The model's weight codes and factors equal the oracle's quantisation of its bf16
    weights bit for bit; layer 0's QKV product, from the model's own LayerNorm output (the
    same bf16 input on both sides, hence the same activation codes), matches the oracle's
    E4M3 product within the matmul tolerance."""
    cfg = SMALL_F8
    m = g.GPT2(cfg, seed=21)
    L, C, BT = cfg["L"], cfg["C"], cfg["B"] * cfg["T"]
    inv = m.debug_tensor("w8_inv", torch.float32, (4 * L,)).cpu().numpy()
    for l in range(L):
        for j, nm in enumerate(("qkv.w", "proj.w", "fc.w", "fcproj.w")):
            i = m.names.index("h%d.%s" % (l, nm))
            codes = m.debug_tensor("w8.%d" % i, torch.uint8, tuple(m.shapes[i])).cpu().numpy()
            wb = torch.from_numpy(m.params(i)).to(torch.bfloat16).double().numpy()
            rq, rinv = of.quantize_tensor(wb)
            assert np.array_equal(codes, rq), (l, nm)
            assert inv[4 * l + j] == np.float32(rinv), (l, nm)
    x, _ = synthetic.zipf_window(21, cfg["B"], cfg["T"], cfg["V"])
    m.forward(_dev(x), None)
    torch.cuda.synchronize()
    y = m.debug_tensor("ln1.0", torch.bfloat16, (BT, C)).float().cpu().numpy().astype(np.float64)
    qkv = m.debug_tensor("qkv.0", torch.bfloat16, (BT, 3 * C)).float().cpu().numpy()
    i = m.names.index("h0.qkv.w")
    qa, ai = of.quantize_rows(y)
    qb, bi = of.quantize_tensor(torch.from_numpy(m.params(i)).to(torch.bfloat16).double().numpy())
    ref = of.matmul_e4m3(qa, ai, qb, bi, bias=m.params(m.names.index("h0.qkv.b")).astype(np.float64))
    _check(qkv, ref, "qkv.0")
    m.close()
