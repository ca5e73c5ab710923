"""The benchmark's host logic on CPU: workload construction from the command line, the rule
that reports the scorer's measured DRAM traffic only for the source it was measured on, and the
reference arm (the float64 oracle timed on the host cores), which needs no GPU."""
import sys

import pytest

import bench
from workload import LLAMA_128K, TINY


def _args(*argv):
    old = sys.argv
    sys.argv = ["bench.py", *argv]
    try:
        return bench.parse()
    finally:
        sys.argv = old


def test_default_workload_is_the_128k_headline():
    w = bench.workload_from(_args())
    assert w == LLAMA_128K
    assert (w.seq_len, w.batch, w.layers, w.v_place, w.dtype, w.new_keys) == (131072, 8, 32, "host", "bf16", "exact")


@pytest.mark.parametrize("argv,field,value", [
    (["--v-place", "hbm"], "v_place", "hbm"),
    (["--dtype", "fp8"], "dtype", "fp8"),
    (["--new-keys", "lowrank"], "new_keys", "lowrank"),
    (["--batch", "4"], "batch", 4),
    (["--layers", "2"], "layers", 2),
    (["--drift", "0.5"], "drift", 0.5),
])
def test_flags_change_one_field(argv, field, value):
    w = bench.workload_from(_args(*argv))
    assert getattr(w, field) == value
    for f in ("seq_len", "head_dim", "rank", "n_select", "n_outlier"):
        assert getattr(w, f) == getattr(LLAMA_128K, f)


def test_variant_names_say_what_changed():
    assert bench.workload_from(_args("--dtype", "fp8")).name.endswith("-fp8")
    assert bench.workload_from(_args("--new-keys", "lowrank")).name.endswith("-plus")


def test_scorer_traffic_only_for_the_measured_source(monkeypatch):
    real = bench.score_traffic_per_launch(LLAMA_128K)
    monkeypatch.setattr(bench, "SCORE_TRAFFIC_SHA256", "0" * 64)
    assert bench.score_traffic_per_launch(LLAMA_128K) is None          # another source
    monkeypatch.undo()
    if real is None:
        pytest.skip("the scorer source differs from the profiled one")
    assert real == pytest.approx(bench.SCORE_TRAFFIC["bf16"]["bytes_per_unit"] * LLAMA_128K.units)
    assert bench.score_traffic_per_launch(LLAMA_128K.with_(batch=4)) == pytest.approx(real / 2)   # per unit
    f8 = bench.score_traffic_per_launch(LLAMA_128K.with_(dtype="fp8"))                           # its own capture
    assert f8 == pytest.approx(bench.SCORE_TRAFFIC["fp8"]["bytes_per_unit"] * LLAMA_128K.units)
    assert bench.score_traffic_per_launch(LLAMA_128K.with_(dtype="f32")) is None                 # not captured
    assert bench.score_traffic_per_launch(LLAMA_128K.with_(seq_len=65536)) is None               # other length


def test_reference_arm_prints_the_same_metric_and_workload():
    args = _args("--impl", "reference", "--config", TINY.name, "--steps", "2", "--warmup", "1", "--ref-budget", "0.05")
    w = bench.workload_from(args)
    line = bench.run_reference(args, w, 1, 0)
    assert line["impl"] == "reference"
    assert (line["metric"], line["unit"], line["higher_is_better"]) == (bench.METRIC, bench.UNIT, True)
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert (line["steps"], line["warmup"]) == (2, 1)
    # the workload keys are those the GPU arm reports for the same run
    assert {k: line["config"][k] for k in bench.workload_config(w, w.layers)} == bench.workload_config(w, w.layers)
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": bench.UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert bench.run_reference(args, w, 2, 1) is None          # other ranks print nothing
