"""Per-kernel parity on the GPU, through the C ABI, against the fp64 oracle.

Tolerances (bf16 path): inputs are exact bf16 values; products accumulate in
fp32 and bf16 outputs carry one rounding (relative 2^-9), so outputs are
compared with |d| <= 1e-2 * max|ref| elementwise and a Frobenius relative error
<= 4e-3; fp32 outputs (ACCUM_F32) with relative error <= 1e-5 of the norm.
"""
import math

import numpy as np
import pytest
import torch

import synthetic
from oracle import gpt2 as og

pytestmark = pytest.mark.gpu

F64 = torch.float64


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gpt_decoder_only_train_b300 import build

    build.build()
    import gpt_decoder_only_train_b300 as mod

    mod.lib()
    return mod


def _bf16(shape, seed, scale=1.0):
    gen = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=gen) * scale).to(torch.bfloat16)


def _close(out, ref, rel_elem=1e-2, rel_fro=4e-3):
    out = out.double().cpu()
    ref = ref.double().cpu()
    mx = ref.abs().max().item()
    err = (out - ref).abs().max().item()
    fro = ((out - ref).norm() / max(ref.norm().item(), 1e-30)).item()
    assert err <= rel_elem * mx + 1e-6, (err, mx)
    assert fro <= rel_fro, fro


# ------------------------------------------------------------------ matmul

def _operand(M, K, kmajor, seed):
    """Logical [M, K] matrix and its storage (K-major: [M, ld]; MN-major: [K, ld]).

    The leading dimension is rounded up to a multiple of 8 (the 16-byte row
    pitch rule of the tensor maps); the padding columns hold garbage that the
    kernel must not read."""
    a = _bf16((M, K), seed)
    inner = K if kmajor else M
    ld = (inner + 7) // 8 * 8
    rows = M if kmajor else K
    store = torch.full((rows, ld), float("nan"), dtype=torch.bfloat16)
    store[:, :inner] = a if kmajor else a.t()
    return a, store, ld


@pytest.mark.parametrize("a_km,b_km", [(1, 1), (1, 0), (0, 1), (0, 0)])
@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (128, 64, 64), (77, 136, 1000)])
def test_matmul_store_all_majorness(g, a_km, b_km, M, N, K):
    A, As, lda = _operand(M, K, a_km, 1)
    B, Bs, ldb = _operand(N, K, b_km, 2)
    D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    bias = torch.randn(N, dtype=torch.float32)
    g.matmul(As.cuda(), lda, a_km, Bs.cuda(), ldb, b_km, D, N, M, N, K, g.EPI_STORE, bias=bias.cuda())
    torch.cuda.synchronize()
    ref = A.double() @ B.double().T + bias.double()
    _close(D, ref)


def test_matmul_residual_gelu_and_gelu_bwd(g):
    M, N, K = 260, 384, 192
    A, As, lda = _operand(M, K, 1, 3)
    B, Bs, ldb = _operand(N, K, 1, 4)
    bias = (torch.randn(N) * 0.1).float()
    R = _bf16((M, N), 5)
    acc = A.double() @ B.double().T
    D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    g.matmul(As.cuda(), lda, 1, Bs.cuda(), ldb, 1, D, N, M, N, K, g.EPI_RESIDUAL, R=R.cuda(), bias=bias.cuda())
    torch.cuda.synchronize()
    _close(D, acc + bias.double() + R.double())
    H = torch.empty_like(D)
    G2 = torch.empty_like(D)
    g.matmul(As.cuda(), lda, 1, Bs.cuda(), ldb, 1, H, N, M, N, K, g.EPI_GELU, D2=G2, bias=bias.cuda())
    torch.cuda.synchronize()
    h = acc + bias.double()
    _close(H, h)
    _close(G2, og.gelu_forward(h), rel_fro=6e-3)
    # GELU of the stored (bf16) pre-activation reproduces the stored output exactly
    assert torch.equal(G2.cpu(), og.gelu_forward(H.cpu().double()).to(torch.bfloat16)) or \
        (G2.cpu().double() - og.gelu_forward(H.cpu().double())).abs().max() < 2e-2
    DB = torch.empty_like(D)
    g.matmul(As.cuda(), lda, 1, Bs.cuda(), ldb, 1, DB, N, M, N, K, g.EPI_GELU_BWD, R=R.cuda())
    torch.cuda.synchronize()
    _close(DB, acc * og.gelu_derivative(R.double()))


@pytest.mark.parametrize("M,N,K", [(256, 512, 4096), (200, 72, 3000), (768, 768, 1024)])
def test_matmul_accumulate_fp32_split_k(g, M, N, K):
    """dW-style product (both operands MN-major, long K) accumulated into fp32."""
    A, As, lda = _operand(M, K, 0, 6)
    B, Bs, ldb = _operand(N, K, 0, 7)
    base = torch.randn(M, N, dtype=torch.float32)
    D = base.clone().cuda()
    g.matmul(As.cuda(), lda, 0, Bs.cuda(), ldb, 0, D, N, M, N, K, g.EPI_ACCUM_F32)
    torch.cuda.synchronize()
    ref = base.double() + A.double() @ B.double().T
    out = D.double().cpu()
    assert ((out - ref).norm() / ref.norm()).item() < 1e-5
    assert (out - ref).abs().max().item() < 1e-4 * ref.abs().max().item() + 1e-5


@pytest.mark.parametrize("M,N,ldd,K", [(300, 136, 144, 128), (1024, 1024, 1032, 256), (130, 264, 272, 2048)])
def test_matmul_accumulate_fp32_touches_only_its_block(g, M, N, ldd, K):
    """fp32 accumulation with a row pitch wider than N, one split and several: the
    product is added to every element of the [M, N] block and the pitch padding
    keeps its value."""
    A, As, lda = _operand(M, K, 0, 8)
    B, Bs, ldb = _operand(N, K, 0, 9)
    base = torch.randn(M, ldd, dtype=torch.float32)
    base[:, N:] = 12345.0
    D = base.clone().cuda()
    g.matmul(As.cuda(), lda, 0, Bs.cuda(), ldb, 0, D, ldd, M, N, K, g.EPI_ACCUM_F32)
    torch.cuda.synchronize()
    out = D.double().cpu()
    assert torch.equal(out[:, N:], base[:, N:].double())
    ref = base[:, :N].double() + A.double() @ B.double().T
    assert ((out[:, :N] - ref).norm() / ref.norm()).item() < 1e-5
    assert (out[:, :N] - ref).abs().max().item() < 1e-4 * ref.abs().max().item() + 1e-5


@pytest.mark.parametrize("p0,p1,K", [((768, 3072), (3072, 768), 2048), ((300, 520), (130, 264), 1000),
                                      ((768, 768), (2304, 768), 4096), ((200, 136), (256, 512), 512)])
def test_matmul_accum2_is_two_products(g, p0, p1, K):
    """Two weight-gradient products in one launch (the last case has N < 256 on one side
    and runs as two launches): each output gets its own product added, fp32 bounds."""
    outs = []
    for (M, N), seed in ((p0, 20), (p1, 30)):
        A, As, lda = _operand(M, K, 0, seed)
        B, Bs, ldb = _operand(N, K, 0, seed + 1)
        base = torch.randn(M, N, dtype=torch.float32)
        outs.append((A, As, lda, B, Bs, ldb, base, base.clone().cuda(), M, N))
    (A0, As0, lda0, B0, Bs0, ldb0, base0, D0, M0, N0), (A1, As1, lda1, B1, Bs1, ldb1, base1, D1, M1, N1) = outs
    g.matmul_accum2(As0.cuda(), lda0, Bs0.cuda(), ldb0, D0, M0, N0, As1.cuda(), lda1, Bs1.cuda(), ldb1, D1, M1, N1, K)
    torch.cuda.synchronize()
    for A, B, base, D in ((A0, B0, base0, D0), (A1, B1, base1, D1)):
        ref = base.double() + A.double() @ B.double().T
        out = D.double().cpu()
        assert ((out - ref).norm() / ref.norm()).item() < 1e-5
        assert (out - ref).abs().max().item() < 1e-4 * ref.abs().max().item() + 1e-5


def test_matmul_rejects_bad_shapes(g):
    a = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    d = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(g.Gpt2Error):
        g.matmul(a, 63, 1, a, 64, 1, d, 64, 64, 64, 64)  # lda not a multiple of 8
    with pytest.raises(g.Gpt2Error):
        g.matmul(a, 64, 1, a, 64, 1, d, 64, 64, 60, 64)  # N not a multiple of 8
    with pytest.raises(g.Gpt2Error):
        g.matmul(a, 64, 1, a, 64, 1, d, 64, 64, 64, 0)   # K = 0


# ------------------------------------------------------------------ attention

def _attn_inputs(B, T, H, seed, hd=64):
    q, k, v, do = synthetic.attention_operands(seed, B, H, T, hd)
    return [torch.from_numpy(a) for a in (q, k, v, do)]


def _attn_oracle(q, k, v, do):
    """fp64 oracle on [B, T, H, hd] -> (o, lse [B,H,T], dq, dk, dv) in [B, T, H, hd]."""
    t = lambda a: a.double().permute(0, 2, 1, 3)
    Q, K, V, dO = t(q), t(k), t(v), t(do)
    o, lse = og._attention_per_sequence(og.causal_attention_forward, Q, K, V)
    dq, dk, dv = og._attention_per_sequence(og.causal_attention_backward, Q, K, V, dO)
    back = lambda a: a.permute(0, 2, 1, 3)
    return back(o), lse, back(dq), back(dk), back(dv)


# the last two put several single-block items on each CTA of the persistent backward kernels
@pytest.mark.parametrize("B,T,H", [(2, 200, 3), (1, 64, 2), (1, 1, 1), (3, 129, 2), (48, 64, 8), (40, 129, 8)])
def test_attention_forward_backward_parity(g, B, T, H):
    q, k, v, do = _attn_inputs(B, T, H, seed=T)
    dev = lambda a: a.to(torch.bfloat16).cuda().contiguous()
    qd, kd, vd, dod = dev(q), dev(k), dev(v), dev(do)
    o = torch.empty_like(qd)
    lse = torch.empty(B, H, T, dtype=torch.float32, device="cuda")
    g.attention_forward(qd, kd, vd, o, lse, B, T, H)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(qd), torch.empty_like(qd)
    scratch = torch.empty(B * H * T, dtype=torch.float32, device="cuda")
    g.attention_backward(qd, kd, vd, o, dod, lse, dq, dk, dv, scratch, B, T, H)
    torch.cuda.synchronize()
    ro, rlse, rdq, rdk, rdv = _attn_oracle(q, k, v, do)
    _close(o, ro, rel_elem=2e-2, rel_fro=1e-2)
    assert (lse.double().cpu() - rlse).abs().max().item() < 2e-3
    for out, ref in ((dq, rdq), (dk, rdk), (dv, rdv)):
        _close(out, ref, rel_elem=3e-2, rel_fro=2e-2)


@pytest.mark.parametrize("B,T,H", [(2, 200, 3), (1, 1, 1), (3, 129, 2), (40, 129, 8), (2, 1000, 2), (1, 384, 3)])
def test_attention_backward_with_stored_ds_parity(g, B, T, H):
    """The backward that keeps dS^T in a workspace (dQ = dS K from it): same oracle and
    tolerances as the recomputing backward.  The workspace starts filled with NaN, so a
    block that dQ read without the dK/dV kernel having written it would show."""
    q, k, v, do = _attn_inputs(B, T, H, seed=T + 7)
    dev = lambda a: a.to(torch.bfloat16).cuda().contiguous()
    qd, kd, vd, dod = dev(q), dev(k), dev(v), dev(do)
    o = torch.empty_like(qd)
    lse = torch.empty(B, H, T, dtype=torch.float32, device="cuda")
    g.attention_forward(qd, kd, vd, o, lse, B, T, H)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(qd), torch.empty_like(qd)
    scratch = torch.empty(B * H * T, dtype=torch.float32, device="cuda")
    nbytes = g.attention_backward_ds_bytes(B, T, H)
    Tp = (T + 127) // 128 * 128
    assert nbytes == B * H * Tp * Tp * 2
    ds = torch.full((nbytes // 2,), float("nan"), dtype=torch.bfloat16, device="cuda")
    g.attention_backward_ds(qd, kd, vd, o, dod, lse, dq, dk, dv, scratch, ds, B, T, H)
    torch.cuda.synchronize()
    _, _, rdq, rdk, rdv = _attn_oracle(q, k, v, do)
    for out, ref in ((dq, rdq), (dk, rdk), (dv, rdv)):
        assert torch.isfinite(out.float()).all()
        if ref.abs().max().item() == 0.0:
            # T = 1: P = 1, so dS = dP - D = 0 exactly; D and dP are summed in different
            # orders here, which leaves fp32 rounding noise only
            assert out.double().abs().max().item() <= 1e-6
        else:
            _close(out, ref, rel_elem=3e-2, rel_fro=2e-2)
    # the stored blocks are dS^T (row = key, column = query) in 64 x 64 blocks, ordered
    # (b*h, key block, query block): finite on the causal side; in the blocks written
    # (queries from the start of the key's 128-block on) zero above the diagonal; blocks
    # further above the diagonal are never written nor read
    nb = Tp // 64
    dsm = ds.view(B * H, nb, nb, 64, 64).permute(0, 1, 3, 2, 4).reshape(B * H, Tp, Tp)[:, :T, :T].float().cpu()
    key, qry = torch.arange(T)[:, None], torch.arange(T)[None, :]
    assert torch.isfinite(dsm[:, key <= qry]).all()
    assert (dsm[:, (key > qry) & (qry >= key // 128 * 128)] == 0).all()
    # against the recomputing backward: dK and dV from the same kernel, dQ from another route
    dq2, dk2, dv2 = torch.empty_like(qd), torch.empty_like(qd), torch.empty_like(qd)
    g.attention_backward(qd, kd, vd, o, dod, lse, dq2, dk2, dv2, scratch, B, T, H)
    torch.cuda.synchronize()
    for a, b in ((dq, dq2), (dk, dk2), (dv, dv2)):
        if b.abs().max().item() > 1e-6:
            _close(a, b.double(), rel_elem=2e-2, rel_fro=1e-2)


def test_attention_fused_qkv_layout(g):
    """q/k/v read with row stride 3C out of one [B*T, 3C] buffer, as the model does."""
    B, T, H = 2, 96, 2
    C = 64 * H
    q, k, v, do = _attn_inputs(B, T, H, seed=11)
    qkv = torch.cat([a.reshape(B * T, C) for a in (q, k, v)], dim=1).to(torch.bfloat16).cuda().contiguous()
    o = torch.empty(B * T, C, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, H, T, dtype=torch.float32, device="cuda")
    g.attention_forward(qkv, qkv[:, C:], qkv[:, 2 * C:], o, lse, B, T, H, qkv_row_stride=3 * C, o_row_stride=C)
    torch.cuda.synchronize()
    ro, rlse, *_ = _attn_oracle(q, k, v, do)
    _close(o.reshape(B, T, H, 64), ro, rel_elem=2e-2, rel_fro=1e-2)


def test_attention_is_causal_bitwise(g):
    B, T, H = 1, 150, 1
    q, k, v, _ = _attn_inputs(B, T, H, seed=3)
    dev = lambda a: a.to(torch.bfloat16).cuda().contiguous()
    qd, kd, vd = dev(q), dev(k), dev(v)
    o1 = torch.empty_like(qd)
    lse = torch.empty(B, H, T, dtype=torch.float32, device="cuda")
    g.attention_forward(qd, kd, vd, o1, lse, B, T, H)
    kd2, vd2 = kd.clone(), vd.clone()
    kd2[:, 100:] = 3.0
    vd2[:, 100:] = -2.0
    o2 = torch.empty_like(qd)
    g.attention_forward(qd, kd2, vd2, o2, lse, B, T, H)
    torch.cuda.synchronize()
    assert torch.equal(o1[:, :100], o2[:, :100])


# ------------------------------------------------------------------ classifier

@pytest.mark.parametrize("N,V,Vp", [(37, 1000, 1024), (5, 50257, 50304), (64, 256, 256)])
def test_classifier_parity(g, N, V, Vp):
    z = _bf16((N, Vp), seed=N, scale=2.0)
    gen = torch.Generator().manual_seed(1)
    t = torch.randint(0, V, (N,), generator=gen, dtype=torch.int32)
    zd = z.cuda()
    rows = torch.empty(N, dtype=torch.float32, device="cuda")
    dscale = 1.0 / N
    g.classifier(zd, t.cuda(), rows, N, V, Vp, dscale)
    torch.cuda.synchronize()
    zr = z.double()[:, :V]
    loss, lse, ref_rows = og.cross_entropy_forward(zr, t.long())
    dz = og.cross_entropy_backward(zr, lse, t.long(), 1.0)  # = (softmax - onehot) / N
    assert (rows.double().cpu() - ref_rows).abs().max().item() < 2e-4 * max(1.0, ref_rows.abs().max().item())
    out = zd.double().cpu()
    assert torch.all(out[:, V:] == 0)
    _close(out[:, :V], dz * (dscale * N), rel_elem=1e-2, rel_fro=6e-3)


# ------------------------------------------------------------------ layernorm

@pytest.mark.parametrize("N,C", [(37, 768), (300, 64), (16, 1024), (5, 2048)])
def test_layernorm_forward_backward_parity(g, N, C):
    gen = torch.Generator().manual_seed(C)
    x = (torch.randn(N, C, generator=gen) * 2 + 0.5).to(torch.bfloat16)
    dy = torch.randn(N, C, generator=gen).to(torch.bfloat16)
    dres = torch.randn(N, C, generator=gen).to(torch.bfloat16)
    gg = (1 + 0.1 * torch.randn(C, generator=gen)).float()
    bb = (0.1 * torch.randn(C, generator=gen)).float()
    y = torch.empty(N, C, dtype=torch.bfloat16, device="cuda")
    mean = torch.empty(N, device="cuda")
    rstd = torch.empty(N, device="cuda")
    xd = x.cuda()
    g.layernorm_forward(xd, gg.cuda(), bb.cuda(), y, mean, rstd, N, C)
    out = dres.clone().cuda()
    dg = torch.full((C,), 0.25, device="cuda")
    db = torch.full((C,), -0.5, device="cuda")
    g.layernorm_backward(dy.cuda(), xd, mean, rstd, gg.cuda(), out, out, dg, db, N, C)  # in place
    torch.cuda.synchronize()
    ry, rm, rr = og.layernorm_forward(x.double(), gg.double(), bb.double())
    _close(y, ry)
    assert (mean.cpu().double() - rm.squeeze(-1)).abs().max() < 1e-5 * max(1.0, rm.abs().max().item())
    assert ((rstd.cpu().double() - rr.squeeze(-1)) / rr.squeeze(-1)).abs().max() < 1e-5
    dx, rdg, rdb = og.layernorm_backward(dy.double(), x.double(), rm, rr, gg.double())
    _close(out, dres.double() + dx)
    assert ((dg.cpu().double() - 0.25 - rdg).norm() / rdg.norm()).item() < 1e-5
    assert ((db.cpu().double() + 0.5 - rdb).norm() / rdb.norm()).item() < 1e-5
