"""The C-ABI library builds, loads without a GPU and exports every declared symbol."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gpt2b300.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(gpt2_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def libh():
    from gpt_decoder_only_train_b300 import build

    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_step_calls():
    names = _declared()
    for want in ("gpt2_build", "gpt2_forward", "gpt2_backward", "gpt2_clip_and_adamw", "gpt2_get_grads",
                 "gpt2_get_params", "gpt2_arena_bytes", "gpt2_free"):
        assert want in names


def test_library_exports_every_declared_symbol(libh):
    missing = [n for n in _declared() if not hasattr(libh, n)]
    assert not missing, missing


def test_binding_signatures_cover_header():
    import gpt_decoder_only_train_b300 as g

    assert set(_declared()) <= set(g._SIGS)


def test_arena_bytes_and_config_validation(libh):
    import gpt_decoder_only_train_b300 as g

    L = g.lib()
    ok = g.make_config(dict(L=12, C=768, H=12, V=50257, Vp=50304, T=1024, B=16, dtype="bf16"))
    n = L.gpt2_arena_bytes(ctypes.byref(ok))
    # fp32 params + grads + m + v + bf16 copy alone are ~2.2 GB at 124M
    assert 2.2e9 < n < 20e9
    bad = [
        dict(L=12, C=768, H=11, V=50257, Vp=50304, T=1024, B=16, dtype="bf16"),  # C % H
        dict(L=12, C=768, H=12, V=50257, Vp=50000, T=1024, B=16, dtype="bf16"),  # Vp < V
        dict(L=2, C=96, H=3, V=256, Vp=256, T=32, B=2, dtype="bf16"),            # head dim 32 in bf16
        dict(L=0, C=64, H=4, V=256, Vp=256, T=32, B=2, dtype="fp32"),
    ]
    for d in bad:
        c = g.make_config(d)
        assert L.gpt2_arena_bytes(ctypes.byref(c)) == 0, d


def test_precision_and_lm_head_modes_are_validated_and_sized(libh):
    """fp8_forward and fused_lm_head: bf16 only, 0 or 1; the E4M3 mode adds its code buffers
    (one byte a parameter, the [B*T, 4C] activation codes and their factors), the fused LM head
    replaces the [B*T, Vp] logits by one chunk of 8,192 rows plus its row partials."""
    import gpt_decoder_only_train_b300 as g

    L = g.lib()
    base = dict(L=12, C=768, H=12, V=50257, Vp=50304, T=1024, B=16, dtype="bf16")
    size = lambda **kw: L.gpt2_arena_bytes(ctypes.byref(g.make_config(dict(base, **kw))))
    n0 = size()
    n8 = size(fp8_forward=1)
    nf = size(fused_lm_head=1)
    assert n0 > 0 and n8 > 0 and nf > 0
    BT, C, Vp = 16 * 1024, 768, 50304
    # E4M3: at least one byte per parameter (124.5M) and the activation codes, at most a few MB more
    extra8 = n8 - n0
    assert 124.4e6 + BT * 4 * C <= extra8 <= 124.5e6 + BT * 4 * C + 8e6, extra8
    # fused LM head: the logits shrink from B*T to 8,192 rows; partials (2 x 197 float2 a row) and
    # two floats a row are added
    saved = n0 - nf
    want = (BT - 8192) * Vp * 2 - BT * 2 * 197 * 8 - 2 * BT * 4
    assert abs(saved - want) <= 4096, (saved, want)
    for bad in (dict(fp8_forward=1, dtype="fp32"), dict(fused_lm_head=1, dtype="fp32"), dict(fp8_forward=2),
                dict(fused_lm_head=-1), dict(fp8_forward=1, C=64, H=1)):
        assert size(**bad) == 0, bad


def test_build_rejects_bad_arguments_without_touching_a_gpu(libh):
    import gpt_decoder_only_train_b300 as g

    L = g.lib()
    c = g.make_config(dict(L=2, C=64, H=4, V=256, Vp=256, T=32, B=2, dtype="fp32"))
    h = ctypes.c_void_p()
    assert L.gpt2_build(ctypes.byref(c), 0, None, 0, None, ctypes.byref(h)) == -8  # NULL arena
    c.C = 65
    assert L.gpt2_build(ctypes.byref(c), 0, ctypes.c_void_p(256), 1 << 30, None, ctypes.byref(h)) == -1
    assert L.gpt2_strerror(-3) == b"token or target out of range"
    assert L.gpt2_forward(None, None, None, 1, 1, None) == -8


def test_attention_entries_check_shapes_before_any_device_work(libh):
    """The op-level attention calls return an error code for shapes their
    kernels cannot launch; the checks run before any pointer is touched."""
    import gpt_decoder_only_train_b300 as g

    L = g.lib()
    p = ctypes.c_void_p(1 << 20)  # never dereferenced: every call below fails its checks first
    f = ctypes.cast(p, ctypes.POINTER(ctypes.c_float))
    fwd = lambda B, T, H, hd, rs=192: L.gpt2_op_attention_forward(p, p, p, rs, p, 64, f, B, T, H, hd, None)
    bwd = lambda B, T, H, hd, rs=192: L.gpt2_op_attention_backward(p, p, p, rs, p, p, 64, f, p, p, p, f, B, T, H,
                                                                   hd, None)
    bad_shape = -2  # GPT2_ERR_BAD_SHAPE
    for call in (fwd, bwd):
        assert call(2, 65535 * 64 + 1, 1, 64) == bad_shape  # more than 65535 blocks of 64 rows
        assert call(2, 128, 1, 32) == bad_shape  # head dim other than 64
        assert call(2, 128, 1, 64, rs=100) == bad_shape  # row stride not a multiple of 8
        assert call(0, 128, 1, 64) == bad_shape
    assert L.gpt2_op_attention_forward(None, p, p, 192, p, 64, f, 2, 128, 1, 64, None) == -8  # NULL pointer


def test_attention_ds_entry_sizes_and_checks_its_workspace(libh):
    """The workspace of the stored-dS backward is B H Tp^2 bf16 (Tp = T rounded up to
    128); the entry refuses a missing, misaligned or short workspace, and shapes its
    kernels cannot take, before any pointer is touched."""
    import gpt_decoder_only_train_b300 as g

    L = g.lib()
    assert L.gpt2_attention_backward_ds_bytes(16, 1024, 12) == 16 * 12 * 1024 * 1024 * 2
    assert L.gpt2_attention_backward_ds_bytes(1, 129, 1) == 256 * 256 * 2
    assert L.gpt2_attention_backward_ds_bytes(3, 128, 2) == 3 * 2 * 128 * 128 * 2
    assert L.gpt2_attention_backward_ds_bytes(0, 8, 1) == 0
    p = ctypes.c_void_p(1 << 20)  # never dereferenced: every call below fails its checks first
    f = ctypes.cast(p, ctypes.POINTER(ctypes.c_float))

    def bwd(B, T, H, hd, ds, nbytes, rs=192):
        return L.gpt2_op_attention_backward_ds(p, p, p, rs, p, p, 64, f, p, p, p, f, ds, nbytes, B, T, H, hd, None)

    n = L.gpt2_attention_backward_ds_bytes(2, 128, 1)
    bad_arg, bad_shape, unsupported = -8, -2, -9
    assert bwd(2, 128, 1, 64, p, n - 1) == bad_arg  # short workspace
    assert bwd(2, 128, 1, 64, None, n) == bad_arg  # no workspace
    assert bwd(2, 128, 1, 64, ctypes.c_void_p((1 << 20) + 8), n) == bad_arg  # not 16-byte aligned
    assert bwd(2, 128, 1, 32, p, n) == bad_shape  # head dim other than 64
    assert bwd(2, 128, 1, 64, p, n, rs=100) == bad_shape  # row stride not a multiple of 8
    assert bwd(0, 128, 1, 64, p, n) == bad_shape
    assert bwd(1, 128, 33, 64, p, 1 << 40, rs=33 * 64 * 3) == unsupported  # H * 64 above 2048


def test_grouped_matmul_checks_both_products_before_any_device_work(libh):
    """gpt2_op_matmul_accum2 rejects a bad first or second product with the same codes as
    gpt2_op_matmul, before any tensor map is built or kernel launched (so a bad second
    product never leaves the first one applied)."""
    import gpt_decoder_only_train_b300 as g

    L = g.lib()
    p = ctypes.c_void_p(1 << 20)  # never dereferenced: every call below fails its checks first
    f = ctypes.cast(p, ctypes.POINTER(ctypes.c_float))

    def call(M0=768, N0=3072, M1=3072, N1=768, K=1024, lda0=768, ldb0=3072, lda1=3072, ldb1=768, a1=p):
        return L.gpt2_op_matmul_accum2(p, lda0, p, ldb0, f, M0, N0, a1, lda1, p, ldb1, f, M1, N1, K, None)

    bad_shape, bad_arg = -2, -8
    assert call(K=0) == bad_shape
    assert call(M0=0) == bad_shape
    assert call(lda0=770) == bad_shape  # leading dimension not a multiple of 8
    assert call(N1=100) == bad_shape  # the second product: N not a multiple of 8
    assert call(ldb1=772) == bad_shape
    assert call(a1=None) == bad_arg  # the second product's A missing
    assert call(a1=ctypes.c_void_p((1 << 20) + 8)) == bad_arg  # not 16-byte aligned


def test_arena_keeps_the_stored_ds_only_below_its_cap(libh):
    """The model keeps the attention backward's dS workspace (B H Tp^2 bf16) up to 16 GiB:
    one position block past that size the arena shrinks by the workspace it no longer holds
    (the backward then recomputes S and dP for dQ)."""
    import gpt_decoder_only_train_b300 as g

    L = g.lib()

    def arena(T):
        c = g.make_config(dict(L=1, C=768, H=12, V=256, Vp=256, T=T, B=1, dtype="bf16"))
        return L.gpt2_arena_bytes(ctypes.byref(c))

    ds = lambda T: L.gpt2_attention_backward_ds_bytes(1, T, 12)
    assert ds(26752) <= 16 << 30 < ds(26880)
    assert arena(26880) < arena(26752) - ds(26752) + (1 << 30)
    assert arena(1024) > ds(1024)  # small T: kept
