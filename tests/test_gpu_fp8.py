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
"""
import numpy as np
import pytest
import torch

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
