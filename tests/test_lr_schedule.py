"""The learning-rate schedule the pages' runs use (linear warmup, then cosine
decay to a final fraction), through the C ABI, pinned to the warmup values the
run logs print and to closed forms of the cosine part.  Host only."""
import json
import math
import os

from pretraining_step_train_b300 import binding

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.json")))


def _lr(t, max_lr, warmup, total, frac):
    return binding.lib().gpt2_lr_schedule(t, max_lr, warmup, total, frac)


def test_warmup_matches_the_printed_run_logs():
    g = GOLDEN["d48_warmup_lr"]
    for step, printed in g["steps"].items():
        got = _lr(int(step), g["max_lr"], g["warmup_steps"], g["total_steps"], g["final_frac"])
        # the logs print three significant digits: within half a unit of the third
        half_unit = 0.5 * 10 ** (math.floor(math.log10(printed)) - 2)
        assert abs(got - printed) <= half_unit * 1.0001, (step, got, printed)
    one = GOLDEN["d48_step1_lr"]
    assert abs(_lr(1, one["max_lr"], one["warmup_steps"], 32000, 0.1) - one["value"]) <= 0.5e-9


def test_cosine_part_closed_forms():
    max_lr, warmup, total, f = 6e-4, 700, 32000, 0.1
    assert math.isclose(_lr(warmup, max_lr, warmup, total, f), max_lr, rel_tol=1e-6)
    assert math.isclose(_lr(warmup + 1, max_lr, warmup, total, f), max_lr, rel_tol=1e-6)  # r = 0
    # r = 1/2: halfway between max_lr and f * max_lr
    t_half = warmup + 1 + (total - warmup) // 2
    assert math.isclose(_lr(t_half, max_lr, warmup, total, f), max_lr * (1 + f) / 2, rel_tol=1e-6)
    # r = 1 and beyond: the final fraction
    assert math.isclose(_lr(total + 1, max_lr, warmup, total, f), f * max_lr, rel_tol=1e-6)
    assert math.isclose(_lr(10 * total, max_lr, warmup, total, f), f * max_lr, rel_tol=1e-6)
    # non-increasing after the warmup, increasing during it
    prev = _lr(1, max_lr, warmup, total, f)
    for t in range(2, warmup + 1):
        cur = _lr(t, max_lr, warmup, total, f)
        assert cur > prev
        prev = cur
    for t in range(warmup + 1, total + 2, 97):
        cur = _lr(t, max_lr, warmup, total, f)
        assert cur <= prev * (1 + 1e-7)
        prev = cur


def test_invalid_arguments_are_refused():
    assert _lr(0, 6e-4, 700, 32000, 0.1) < 0
    assert _lr(5, 6e-4, -1, 32000, 0.1) < 0
    assert _lr(5, 6e-4, 700, 700, 0.1) < 0
    assert _lr(5, -1.0, 700, 32000, 0.1) < 0
