"""The bounded oracle timings that bench.py reports beside its decode, layer and
backward sections, run on CPU on small shapes: each returns a positive rate with
its unit, core count and sample description, and a failure is reported in the
line rather than raised."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from linear_attention_recurrence_14_b300.inputs import make_backward_grads, make_prefill_inputs  # noqa: E402


def _check(res, unit):
    assert res["kind"] == "oracle" and "error" not in res, res
    assert res["unit"] == unit and res["value"] > 0 and res["cores"] >= 1 and res["sample"]


def test_decode_layer_and_backward_oracle_timings():
    w = dict(kind="decode", B=8, steps=4, Hqk=1, Hv=2, d=64, dtype="bf16", decay_scale=0.05, s0_std=0.02)
    _check(bench.time_oracle_decode(w, 0, 0.05, sample_b=4), "steps/s")
    _check(bench.time_oracle_layer(1, 1, 2, 64, 4, 256, 0, 0.05), "tokens/s")
    x = make_prefill_inputs(2, 100, 1, 2, 64, "bf16", seed=1)
    g = make_backward_grads(2, 100, 2, 64, "bf16", seed=1)
    _check(bench.time_oracle_backward(x, g, 0, 0.05), "tokens/s")


def test_oracle_timing_failure_is_reported():
    res = bench._oracle_timed(lambda: 1 / 0, "probe")
    assert res["kind"] == "oracle" and res["error"].startswith("probe: ZeroDivisionError")
