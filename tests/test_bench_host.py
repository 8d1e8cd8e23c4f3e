"""Host-side checks of the benchmark's accounting (no GPU).

The FLOP counts that MFU divides by are pinned against an independent count:
the sum of 2*M*N*K over the matmuls the step performs (listed here shape by
shape, forward and both backward products) plus the causal attention pairs,
and the 6N + 12 L C T convention against the parameter count of the oracle's
own parameter list.
"""
import bench
import synthetic
from oracle import gpt2 as og


def _matmul_flops_per_token(w):
    """Sum of 2*M*N*K over the step's matmuls, per token (M = tokens)."""
    L, C, V = w["L"], w["C"], w["V"]
    fwd_shapes = []
    for _ in range(L):
        fwd_shapes += [(C, 3 * C), (C, C), (C, 4 * C), (4 * C, C)]  # (in, out) of qkv, proj, fc, fcproj
    fwd_shapes.append((C, V))  # tied LM head over the real vocabulary
    fwd = sum(2 * k * n for k, n in fwd_shapes)
    return 3 * fwd  # forward, dX and dW products have the same size


def _attention_flops_per_token(w):
    """QK^T and PV over the causal pairs (j <= i): 2 * 2 * hd per pair and head, 3x for training."""
    L, C, T = w["L"], w["C"], w["T"]
    pairs_per_token = (T + 1) / 2.0  # T(T+1)/2 pairs over T tokens
    return 3 * L * 4 * C * pairs_per_token


def test_flops_per_token_matches_the_shape_sum():
    for name in ("gpt2_124m", "gpt2_350m_recompute"):
        w = synthetic.WORKLOADS[name]
        expect = _matmul_flops_per_token(w) + _attention_flops_per_token(w)
        assert abs(bench.flops_per_token(w) - expect) <= 1e-9 * expect, name
    # the figures the step is quoted with: 0.798 and 2.272 GFLOP per token
    assert round(bench.flops_per_token(synthetic.WORKLOADS["gpt2_124m"]) / 1e9, 3) == 0.798
    assert round(bench.flops_per_token(synthetic.WORKLOADS["gpt2_350m_recompute"]) / 1e9, 3) == 2.272


def test_6n_convention_counts_the_oracle_parameters():
    w = synthetic.WORKLOADS["gpt2_124m"]
    cfg = og.Config.from_dict(w)
    n = 0
    for name, shape, _kind, _std, _decay in og.param_specs(cfg):
        numel = 1
        for s in shape:
            numel *= s
        if name == "wpe":
            continue  # the convention leaves the position table out
        if name == "wte":
            numel = cfg.V * cfg.C  # padded rows are not parameters of the model
        n += numel
    expect = 6 * n + 12 * w["L"] * w["C"] * w["T"]
    assert bench.flops_per_token_6n(w) == expect


def test_workload_label_names_the_shape():
    w = synthetic.WORKLOADS["gpt2_124m_accum32"]
    label = bench.workload_label("gpt2_124m_accum32", w, 32)
    for part in ("L=12", "C=768", "B=16", "T=1024", "32 micro-step"):
        assert part in label


def test_bench_learning_rate_is_the_oracle_schedule():
    """bench.py restates the warmup + cosine schedule; it must give the oracle's values."""
    for it in (0, 1, 19, 20, 698, 699, 700, 701, 5000, 9886, 19072, 19073, 19074, 25000):
        assert bench.lr_at(it) == og.lr_schedule(it), it


def test_stored_gemm_traffic_is_gated_on_the_gemm_sources(monkeypatch):
    """The stored per-launch GEMM DRAM traffic is reported only while the GEMM sources hash to
    the version it was captured from, and then it is plausible against the algorithmic bytes
    (every operand read once, every output written once, fp32 weight gradients read and
    written: 24.0 GB a step): below them (L2 keeps some re-reads off DRAM) but not by more than
    half."""
    w = synthetic.WORKLOADS["gpt2_124m"]
    BT, C, V = w["B"] * w["T"], w["C"], w["Vp"]
    algo = 0.0
    for k, n in [(C, 3 * C), (C, C), (C, 4 * C), (4 * C, C)]:  # per block: in, out
        act_in, act_out, weight = BT * k * 2, BT * n * 2, k * n
        algo += w["L"] * (act_in + act_out + weight * 2)  # forward: x, W read, y written
        algo += w["L"] * (act_out + weight * 2 + act_in)  # dX: dy, W read, dx written
        algo += w["L"] * (act_out + act_in + weight * 8)  # dW: dy, x read, fp32 dW read + written
    # epilogue operands: the FC product's second output (GELU), the GELU backward reading h,
    # the residual read by the two output projections
    algo += w["L"] * (BT * 4 * C * 2 + BT * 4 * C * 2 + 2 * BT * C * 2)
    algo += BT * C * 2 + V * C * 2 + BT * V * 2  # LM head forward
    algo += BT * V * 2 + V * C * 2 + BT * C * 2  # dX
    algo += BT * V * 2 + BT * C * 2 + V * C * 8  # dW
    traffic = bench.gemm_traffic()
    if traffic is not None:
        per_step = traffic * 123
        assert abs(algo / 1e9 - 24.0) < 0.05
        assert 0.5 * algo <= per_step <= 1.05 * algo, (per_step / 1e9, algo / 1e9)
    monkeypatch.setitem(bench.GEMM_TRAFFIC, "sha256", "0" * 64)
    assert bench.gemm_traffic() is None
