"""The stored oracle loss curve of the 32-micro-step workload (no GPU): it was
made by the oracle code that is in the tree now (the hash its maker computes
over the oracle and input functions it calls), and it has the shape and the
values that the definitions fix: 32 finite micro-step losses per optimizer
step whose mean is the step's loss, a first loss near ln V plus the small
initial logit variance ("Let's reproduce GPT-2 (124M)", §Bölümler 4: the
initial loss of a random model), the warmup learning rates of the schedule,
and a loss that falls from step 1 to step 2."""
import importlib.util
import json
import math
import os

from oracle import gpt2 as og

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _maker():
    spec = importlib.util.spec_from_file_location("make_accum32_curve", os.path.join(GOLDEN, "make_accum32_curve.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_golden_curve_matches_the_oracle_in_the_tree():
    mk = _maker()
    with open(mk.OUT) as f:
        gold = json.load(f)
    assert gold["sources_sha256"] == mk.source_hash(), "oracle code changed: regenerate the golden curve"
    assert (gold["B"], gold["T"], gold["micro_steps"]) == (16, 1024, 32)
    steps = gold["steps"]
    assert [s["step"] for s in steps] == [1, 2]
    V, C = 50257, 768
    for s in steps:
        ml = s["micro_losses"]
        assert len(ml) == 32 and all(math.isfinite(x) for x in ml)
        assert abs(sum(ml) / 32 - s["loss"]) <= 1e-12 * s["loss"]
        assert s["lr"] == og.lr_schedule(s["step"] - 1)
    # the maker records the pre-clip norm of step 1 (the GPU test compares it)
    assert math.isfinite(steps[0]["grad_norm"]) and steps[0]["grad_norm"] > 0
    # initial loss: ln V plus half the logit variance (0.02^2 C of the tied head), within a few 1e-2
    assert abs(steps[0]["micro_losses"][0] - (math.log(V) + 0.5 * 0.02 ** 2 * C)) < 5e-2
    assert steps[1]["loss"] < steps[0]["loss"]
