"""Python binding of ``libgpt2b300.so``: one GPT-2 training step on a B300.

Argument marshalling only: every step of the computation runs in the CUDA
library.  PyTorch provides device memory (the arena, token tensors) and the
CUDA stream.  The raw C functions are available under their C names
(``gpt2_build``, ``gpt2_forward``, ...) via :func:`lib`; :class:`GPT2` wraps
them for torch tensors.

If the library has not been built, or the machine has no sm_103 GPU, calls fail
with an exception: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgpt2b300.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "gpt2b300.h")

GPT2_DTYPE_FP32 = 0
GPT2_DTYPE_BF16 = 1
EPI_STORE, EPI_RESIDUAL, EPI_GELU, EPI_GELU_BWD, EPI_ACCUM_F32 = range(5)

STATUS = {
    0: "OK", -1: "BAD_CONFIG", -2: "BAD_SHAPE", -3: "BAD_TOKEN", -4: "ARENA_TOO_SMALL", -5: "CUDA",
    -6: "NONFINITE", -7: "TIMEOUT", -8: "BAD_ARG", -9: "UNSUPPORTED", -10: "STATE",
}


class Gpt2Error(RuntimeError):
    def __init__(self, fn, status, detail=""):
        self.status = status
        msg = "%s failed: %s (%d)" % (fn, STATUS.get(status, "?"), status)
        if detail:
            msg += ": " + detail
        super().__init__(msg)


class gpt2_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int)
                for n in ("L", "C", "H", "V", "Vp", "T", "B", "dtype", "recompute_gelu", "fp8_forward",
                          "fused_lm_head")]


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_F = ctypes.c_float
_SIGS = {
    "gpt2_arena_bytes": (ctypes.c_size_t, [ctypes.POINTER(gpt2_config)]),
    "gpt2_build": (_I, [ctypes.POINTER(gpt2_config), ctypes.c_uint64, _P, ctypes.c_size_t, _P, ctypes.POINTER(_P)]),
    "gpt2_forward": (_I, [_P, _P, _P, _I, _I, ctypes.POINTER(_F)]),
    "gpt2_backward": (_I, [_P, _F]),
    "gpt2_zero_grad": (_I, [_P]),
    "gpt2_clip_and_adamw": (_I, [_P, _F, _F, _F, _F, _F, _F, ctypes.POINTER(_F)]),
    "gpt2_num_tensors": (_I, [_P]),
    "gpt2_tensor_info": (_I, [_P, _I, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(_I), ctypes.POINTER(_I64)]),
    "gpt2_get_params": (_I, [_P, _I, _P, ctypes.c_size_t]),
    "gpt2_get_grads": (_I, [_P, _I, _P, ctypes.c_size_t]),
    "gpt2_get_adam_state": (_I, [_P, _I, _P, _P, ctypes.c_size_t]),
    "gpt2_set_params": (_I, [_P, _I, _P, ctypes.c_size_t]),
    "gpt2_set_grads": (_I, [_P, _I, _P, ctypes.c_size_t]),
    "gpt2_debug_buffer": (_I, [_P, ctypes.c_char_p, ctypes.POINTER(_P), ctypes.POINTER(ctypes.c_size_t)]),
    "gpt2_adam_step": (_I, [_P, ctypes.POINTER(_I)]),
    "gpt2_free": (None, [_P]),
    "gpt2_strerror": (ctypes.c_char_p, [_I]),
    "gpt2_last_error_detail": (ctypes.c_char_p, []),
    "gpt2_launch_count": (ctypes.c_longlong, []),
    "gpt2_profile": (_I, [_P, _I]),
    "gpt2_profile_read": (_I, [_P, _I, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
                               ctypes.POINTER(ctypes.c_longlong)]),
    "gpt2_op_attention_forward": (_I, [_P, _P, _P, _I64, _P, _I64, _P, _I, _I, _I, _I, _P]),
    "gpt2_op_attention_backward": (_I, [_P, _P, _P, _I64, _P, _P, _I64, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "gpt2_op_attention_backward_noalloc": (_I, [_P, _P, _P, _I64, _P, _P, _I64, _P, _P, _P, _P, _I, _I, _I, _I,
                                                _P]),
    "gpt2_op_attention_backward_ds": (_I, [_P, _P, _P, _I64, _P, _P, _I64, _P, _P, _P, _P, _P, _P, ctypes.c_size_t,
                                           _I, _I, _I, _I, _P]),
    "gpt2_attention_backward_ds_bytes": (ctypes.c_size_t, [_I, _I, _I]),
    "gpt2_op_matmul": (_I, [_P, _I64, _I, _P, _I64, _I, _P, _P, _P, _I64, _P, _I, _I, _I, _I, _P]),
    "gpt2_op_matmul_accum2": (_I, [_P, _I64, _P, _I64, _P, _I, _I, _P, _I64, _P, _I64, _P, _I, _I, _I, _P]),
    "gpt2_op_classifier": (_I, [_P, _P, _P, _I, _I, _I, _F, _P]),
    "gpt2_op_sample": (_I, [_P, _I64, _I, _I, _P, _F, _I, _P, _P]),
    "gpt2_generate": (_I, [_P, _P, _I, _I, _I, _P, _F, _I]),
    "gpt2_op_layernorm_forward": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _P]),
    "gpt2_op_layernorm_backward": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _P]),
    "gpt2_op_embedding_backward": (_I, [_P, _I, _P, _I, _I, _I, _I, _P, _P, _P, _P]),
    "gpt2_embedding_backward_workspace": (ctypes.c_size_t, [_I, _I, _I]),
    "gpt2_debug_set_barrier_wait": (_I, [ctypes.c_ulonglong, _I]),
    "gpt2_set_graphs": (_I, [_P, _I]),
    "gpt2_op_quantize_e4m3_rows": (_I, [_P, _I64, _I, _I, _P, _I64, _P, _P]),
    "gpt2_op_quantize_e4m3_tensor": (_I, [_P, _I64, _P, _P, _P, _P]),
    "gpt2_op_matmul_e4m3": (_I, [_P, _I64, _P, _P, _I64, _P, _P, _P, _P, _I64, _P, _I, _I, _I, _I, _P]),
}


def lib():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libgpt2b300.so is not built: run python -m gpt_decoder_only_train_b300.build")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib = h
    return _lib


def check(fn_name, status):
    if status != 0:
        detail = lib().gpt2_last_error_detail().decode() if status == -5 else ""
        raise Gpt2Error(fn_name, status, detail)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_config(d: dict) -> gpt2_config:
    dt = d.get("dtype", "bf16")
    dtype = GPT2_DTYPE_BF16 if dt in ("bf16", GPT2_DTYPE_BF16) else GPT2_DTYPE_FP32
    return gpt2_config(d["L"], d["C"], d["H"], d["V"], d["Vp"], d["T"], d["B"], dtype, int(d.get("recompute_gelu", 0)),
                       int(d.get("fp8_forward", 0)), int(d.get("fused_lm_head", 0)))


def launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(lib().gpt2_launch_count())


def arena_bytes(cfg: dict) -> int:
    c = make_config(cfg)
    return int(lib().gpt2_arena_bytes(ctypes.byref(c)))


class GPT2:
    """A model in a torch-allocated device arena; methods map 1:1 to the C calls."""

    def __init__(self, cfg: dict, seed: int, device="cuda", stream=None):
        import torch

        self.cfg_dict = dict(cfg)
        self.cfg = make_config(cfg)
        L = lib()
        nbytes = int(L.gpt2_arena_bytes(ctypes.byref(self.cfg)))
        if nbytes == 0:
            raise Gpt2Error("gpt2_arena_bytes", -1)
        self.arena = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.arena.device)
        h = ctypes.c_void_p()
        check("gpt2_build", L.gpt2_build(ctypes.byref(self.cfg), ctypes.c_uint64(seed), _ptr(self.arena), nbytes,
                                         _stream(self.stream), ctypes.byref(h)))
        self.handle = h
        self.names, self.shapes = [], []
        for i in range(L.gpt2_num_tensors(h)):
            nm, nd, shp = ctypes.c_char_p(), ctypes.c_int(), (ctypes.c_int64 * 2)()
            check("gpt2_tensor_info", L.gpt2_tensor_info(h, i, ctypes.byref(nm), ctypes.byref(nd), shp))
            self.names.append(nm.value.decode())
            self.shapes.append(tuple(shp[: nd.value]))

    def close(self):
        if getattr(self, "handle", None):
            lib().gpt2_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # --- step -----------------------------------------------------------
    def forward(self, tokens, targets=None):
        """tokens/targets: device int32 tensors [B, T].  Returns the mean loss (float) or None."""
        B, T = tokens.shape
        loss = ctypes.c_float(0.0)
        check("gpt2_forward", lib().gpt2_forward(self.handle, _ptr(tokens), _ptr(targets), B, T, ctypes.byref(loss)))
        return loss.value if targets is not None else None

    def backward(self, grad_scale=1.0):
        check("gpt2_backward", lib().gpt2_backward(self.handle, grad_scale))

    def generate(self, seq, T0, uniforms, temperature=1.0, top_k=1):
        """KV-cached sampling in place: seq device int32 [B, T_total] holds the prompt in
        columns [0, T0) and receives the sampled tokens; uniforms device float32
        [T_total - T0, B] in [0, 1) (see gpt2_generate)."""
        B, T_total = seq.shape
        check("gpt2_generate", lib().gpt2_generate(self.handle, _ptr(seq), B, T_total, T0, _ptr(uniforms),
                                                   temperature, top_k))

    def zero_grad(self):
        check("gpt2_zero_grad", lib().gpt2_zero_grad(self.handle))

    def set_graphs(self, enable: bool):
        """CUDA-graph replay of forward / backward (on by default; see gpt2_set_graphs)."""
        check("gpt2_set_graphs", lib().gpt2_set_graphs(self.handle, int(bool(enable))))

    def clip_and_adamw(self, lr, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1, clip=1.0):
        norm = ctypes.c_float(0.0)
        check("gpt2_clip_and_adamw", lib().gpt2_clip_and_adamw(self.handle, lr, beta1, beta2, eps, wd, clip,
                                                               ctypes.byref(norm)))
        return norm.value

    # --- inspection -----------------------------------------------------
    def _get(self, fn, i):
        out = np.empty(int(np.prod(self.shapes[i])), dtype=np.float32)
        check(fn, getattr(lib(), fn)(self.handle, i, out.ctypes.data, out.size))
        return out.reshape(self.shapes[i])

    def params(self, i):
        return self._get("gpt2_get_params", i)

    def grads(self, i):
        return self._get("gpt2_get_grads", i)

    def adam_state(self, i):
        m = np.empty(int(np.prod(self.shapes[i])), dtype=np.float32)
        v = np.empty_like(m)
        check("gpt2_get_adam_state", lib().gpt2_get_adam_state(self.handle, i, m.ctypes.data, v.ctypes.data, m.size))
        return m.reshape(self.shapes[i]), v.reshape(self.shapes[i])

    def set_params(self, i, arr):
        a = np.ascontiguousarray(arr, dtype=np.float32)
        check("gpt2_set_params", lib().gpt2_set_params(self.handle, i, a.ctypes.data, a.size))

    def set_grads(self, i, arr):
        a = np.ascontiguousarray(arr, dtype=np.float32)
        check("gpt2_set_grads", lib().gpt2_set_grads(self.handle, i, a.ctypes.data, a.size))

    def adam_step(self):
        t = ctypes.c_int()
        check("gpt2_adam_step", lib().gpt2_adam_step(self.handle, ctypes.byref(t)))
        return t.value

    PROF_CATEGORIES = ("matmul", "attention", "classifier", "adamw", "layernorm", "other", "matmul_e4m3")

    def profile(self, enable: bool):
        """Start (clearing totals) or stop per-launch CUDA-event timing of model calls."""
        check("gpt2_profile", lib().gpt2_profile(self.handle, int(bool(enable))))

    def profile_read(self):
        """{category: (total_ms, total_work, launches)}; synchronises the stream."""
        out = {}
        for i, name in enumerate(self.PROF_CATEGORIES):
            ms, work, n = ctypes.c_double(), ctypes.c_double(), ctypes.c_longlong()
            check("gpt2_profile_read", lib().gpt2_profile_read(self.handle, i, ctypes.byref(ms), ctypes.byref(work),
                                                               ctypes.byref(n)))
            out[name] = (ms.value, work.value, n.value)
        return out

    def debug_buffer(self, name):
        """(device pointer, bytes) of an internal activation buffer."""
        p, n = ctypes.c_void_p(), ctypes.c_size_t()
        check("gpt2_debug_buffer", lib().gpt2_debug_buffer(self.handle, name.encode(), ctypes.byref(p),
                                                           ctypes.byref(n)))
        return p.value, n.value

    def debug_tensor(self, name, dtype, shape):
        """A torch view (no copy) of an internal buffer inside the arena."""
        import torch

        ptr, nbytes = self.debug_buffer(name)
        off = ptr - self.arena.data_ptr()
        count = int(np.prod(shape)) * torch.empty(0, dtype=dtype).element_size()
        assert 0 <= off and count <= nbytes
        return self.arena[off: off + count].view(dtype).view(*shape)


# --- op-level wrappers (torch tensors in, results written in place) ------------

def attention_forward(q, k, v, o, lse, B, T, H, hd=64, qkv_row_stride=None, o_row_stride=None, stream=None):
    rs = qkv_row_stride if qkv_row_stride is not None else H * hd
    ors = o_row_stride if o_row_stride is not None else H * hd
    check("gpt2_op_attention_forward", lib().gpt2_op_attention_forward(
        _ptr(q), _ptr(k), _ptr(v), rs, _ptr(o), ors, _ptr(lse), B, T, H, hd, _stream(stream)))


def attention_backward(q, k, v, o, do, lse, dq, dk, dv, scratch, B, T, H, hd=64, qkv_row_stride=None,
                       o_row_stride=None, stream=None):
    rs = qkv_row_stride if qkv_row_stride is not None else H * hd
    ors = o_row_stride if o_row_stride is not None else H * hd
    check("gpt2_op_attention_backward", lib().gpt2_op_attention_backward(
        _ptr(q), _ptr(k), _ptr(v), rs, _ptr(o), _ptr(do), ors, _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
        _ptr(scratch), B, T, H, hd, _stream(stream)))


def attention_backward_ds_bytes(B, T, H) -> int:
    return int(lib().gpt2_attention_backward_ds_bytes(B, T, H))


def attention_backward_ds(q, k, v, o, do, lse, dq, dk, dv, scratch, ds, B, T, H, hd=64, qkv_row_stride=None,
                          o_row_stride=None, stream=None):
    """attention_backward that keeps dS^T in `ds` (a device tensor of at least
    attention_backward_ds_bytes(B, T, H) bytes) and forms dQ from it."""
    rs = qkv_row_stride if qkv_row_stride is not None else H * hd
    ors = o_row_stride if o_row_stride is not None else H * hd
    nbytes = ds.numel() * ds.element_size()
    check("gpt2_op_attention_backward_ds", lib().gpt2_op_attention_backward_ds(
        _ptr(q), _ptr(k), _ptr(v), rs, _ptr(o), _ptr(do), ors, _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
        _ptr(scratch), _ptr(ds), nbytes, B, T, H, hd, _stream(stream)))


NOALLOC_ATTN_MAX_ROWS = 1 << 20


def attention_backward_noalloc(q, k, v, o, do, lse, dq, dk, dv, B, T, H, hd=64, qkv_row_stride=None,
                               o_row_stride=None, stream=None):
    """Attention backward without a caller workspace (the library's fixed array holds it)."""
    rs = qkv_row_stride if qkv_row_stride is not None else H * hd
    ors = o_row_stride if o_row_stride is not None else H * hd
    check("gpt2_op_attention_backward_noalloc", lib().gpt2_op_attention_backward_noalloc(
        _ptr(q), _ptr(k), _ptr(v), rs, _ptr(o), _ptr(do), ors, _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
        B, T, H, hd, _stream(stream)))


def matmul(A, lda, a_kmajor, B, ldb, b_kmajor, D, ldd, M, N, K, epilogue=EPI_STORE, D2=None, R=None, bias=None,
           stream=None):
    check("gpt2_op_matmul", lib().gpt2_op_matmul(
        _ptr(A), lda, int(a_kmajor), _ptr(B), ldb, int(b_kmajor), _ptr(D), _ptr(D2), _ptr(R), ldd, _ptr(bias),
        M, N, K, epilogue, _stream(stream)))


def matmul_accum2(A0, lda0, B0, ldb0, D0, M0, N0, A1, lda1, B1, ldb1, D1, M1, N1, K, stream=None):
    """D_i += A_i^T B_i for two weight-gradient products in one launch (A_i [K, M_i], B_i [K, N_i]
    bf16, D_i fp32 [M_i, N_i])."""
    check("gpt2_op_matmul_accum2", lib().gpt2_op_matmul_accum2(
        _ptr(A0), lda0, _ptr(B0), ldb0, _ptr(D0), M0, N0, _ptr(A1), lda1, _ptr(B1), ldb1, _ptr(D1), M1, N1, K,
        _stream(stream)))


def layernorm_forward(x, g, b, y, mean, rstd, N, C, stream=None):
    check("gpt2_op_layernorm_forward", lib().gpt2_op_layernorm_forward(
        _ptr(x), _ptr(g), _ptr(b), _ptr(y), _ptr(mean), _ptr(rstd), N, C, _stream(stream)))


def layernorm_backward(dy, x, mean, rstd, g, dres_in, dres_out, dg, db, N, C, stream=None):
    check("gpt2_op_layernorm_backward", lib().gpt2_op_layernorm_backward(
        _ptr(dy), _ptr(x), _ptr(mean), _ptr(rstd), _ptr(g), _ptr(dres_in), _ptr(dres_out), _ptr(dg), _ptr(db),
        N, C, _stream(stream)))


def sample(logits, ldl, B, V, uniforms, temperature, top_k, out, stream=None):
    """out[b] = the token drawn from bf16 logits row b with uniforms[b] (the rule of gpt2_generate)."""
    check("gpt2_op_sample", lib().gpt2_op_sample(
        _ptr(logits), ldl, B, V, _ptr(uniforms), temperature, top_k, _ptr(out), _stream(stream)))


def classifier(logits, targets, loss_rows, N, V, Vp, dscale, stream=None):
    check("gpt2_op_classifier", lib().gpt2_op_classifier(
        _ptr(logits), _ptr(targets), _ptr(loss_rows), N, V, Vp, dscale, _stream(stream)))


def embedding_backward_workspace(B, T, C) -> int:
    return int(lib().gpt2_embedding_backward_workspace(B, T, C))


def embedding_backward(dx, tokens, dwte, dwpe, B, T, C, V, workspace=None, stream=None):
    """dwte[tokens] += dx rows; dwpe[t] += sum over the batch (device tensors).  With a
    workspace (uint8 device tensor of embedding_backward_workspace bytes) the rows are summed
    in a fixed order; without, with atomics."""
    import torch

    dtype = GPT2_DTYPE_FP32 if dx.dtype == torch.float32 else GPT2_DTYPE_BF16
    check("gpt2_op_embedding_backward",
          lib().gpt2_op_embedding_backward(_ptr(dx), dtype, _ptr(tokens), B, T, C, V, _ptr(dwte), _ptr(dwpe),
                                           _ptr(workspace), _stream(stream)))


def set_barrier_wait(wait_ns: int = 0, never_arrive: bool = False):
    """Test hook: time limit of the clip + AdamW grid barrier (0: default) and an unreachable barrier."""
    check("gpt2_debug_set_barrier_wait", lib().gpt2_debug_set_barrier_wait(int(wait_ns), int(bool(never_arrive))))


def quantize_e4m3_rows(x, q, row_inv, M, K, stream=None):
    """Per-row E4M3 codes of bf16 x [M, K] into uint8 q [M, K] and fp32 row_inv [M]."""
    check("gpt2_op_quantize_e4m3_rows", lib().gpt2_op_quantize_e4m3_rows(
        _ptr(x), x.stride(0), M, K, _ptr(q), q.stride(0), _ptr(row_inv), _stream(stream)))


def quantize_e4m3_tensor(x, q, inv, work, stream=None):
    """Per-tensor E4M3 codes of bf16 x into uint8 q and fp32 inv [1]; work: one int32 of scratch."""
    check("gpt2_op_quantize_e4m3_tensor", lib().gpt2_op_quantize_e4m3_tensor(
        _ptr(x), x.numel(), _ptr(q), _ptr(inv), _ptr(work), _stream(stream)))


def matmul_e4m3(A, a_inv, B, b_inv, D, M, N, K, epilogue=EPI_STORE, D2=None, R=None, bias=None, stream=None):
    """D = a_inv[m] b_inv sum_k A(m,k) B(n,k) (E4M3 codes, K-major) with a bf16 epilogue."""
    check("gpt2_op_matmul_e4m3", lib().gpt2_op_matmul_e4m3(
        _ptr(A), A.stride(0), _ptr(a_inv), _ptr(B), B.stride(0), _ptr(b_inv), _ptr(D), _ptr(D2), _ptr(R),
        D.stride(0), _ptr(bias), M, N, K, epilogue, _stream(stream)))
