"""The attention backward that allocates nothing agrees with the regular one.

Callers that cannot allocate device memory when they run the backward (their
memory is owned by a pool, or allocation is frozen) use
gpt2_op_attention_backward_noalloc, whose workspace is a fixed array in the
library.  Its results must match gpt2_op_attention_backward, which takes a
caller workspace, within the attention tests' tolerance; two calls in a row
(different sizes, reusing the shared array) must both match.  This file is
collected last so that, if it fails, a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

import synthetic

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


def _case(g, B, T, H, seed):
    q, k, v, do = [torch.from_numpy(a).to(torch.bfloat16).cuda().contiguous()
                   for a in synthetic.attention_operands(seed, B, H, T, 64)]
    o = torch.empty_like(q)
    lse = torch.empty(B, H, T, dtype=torch.float32, device="cuda")
    g.attention_forward(q, k, v, o, lse, B, T, H)
    return q, k, v, do, o, lse


def _close(a, b):
    a, b = a.double().cpu(), b.double().cpu()
    err = (a - b).abs().max().item()
    assert err <= 3e-2 * b.abs().max().item(), err
    assert ((a - b).norm() / b.norm()).item() <= 2e-2


def test_noalloc_backward_matches_regular_two_calls(g):
    for B, T, H, seed in ((2, 200, 3, 1), (4, 1024, 12, 2)):
        q, k, v, do, o, lse = _case(g, B, T, H, seed)
        ref = [torch.empty_like(q) for _ in range(3)]
        scratch = torch.empty(B * H * T, dtype=torch.float32, device="cuda")
        g.attention_backward(q, k, v, o, do, lse, *ref, scratch, B, T, H)
        out = [torch.full_like(q, float("nan")) for _ in range(3)]
        g.attention_backward_noalloc(q, k, v, o, do, lse, *out, B, T, H)
        torch.cuda.synchronize()
        for a, b in zip(out, ref):
            assert torch.isfinite(a.float()).all()
            _close(a, b)


def test_noalloc_rejects_sizes_over_the_limit(g):
    B, T, H = 1, 64, 1
    q, k, v, do, o, lse = _case(g, B, T, H, 3)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    big_B = g.NOALLOC_ATTN_MAX_ROWS // (H * T) + 1  # B*H*T just above the limit; no kernel runs
    with pytest.raises(g.Gpt2Error) as e:
        g.attention_backward_noalloc(q, k, v, o, do, lse, dq, dk, dv, big_B, T, H)
    assert e.value.status == -2
