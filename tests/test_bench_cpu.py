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
    args = _args()
    w = bench.workload_from(args)
    assert w == LLAMA_128K
    assert args.host_mem == "pinned" and args.microbatches == 1
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
    args = _args("--impl", "reference", "--config", TINY.name, "--steps", "2", "--warmup", "1",
                 "--ref-budget", "0.05", "--ref-workers", "2")
    w = bench.workload_from(args)
    line = bench.run_reference(args, w, 1, 0)
    assert line["impl"] == "reference"
    assert (line["metric"], line["unit"], line["higher_is_better"]) == (bench.METRIC, bench.UNIT, True)
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert (line["steps"], line["warmup"]) == (2, 1)
    # the whole config dict is the one the GPU arm prints for the same command line
    assert line["config"] == bench.line_config(args, w, w.layers, 1)
    # the step time is the measured sample step; the whole workload's step is labelled as scaled
    assert line["extrapolated_ms_per_full_step"] > 0 and "measured" in line["ms_per_step_kind"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["cores"] == 2
    assert line["e2e"] == {"value": line["value"], "unit": bench.UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert bench.run_reference(args, w, 2, 1) is None          # other ranks print nothing


def test_cpu_baseline_single_and_all_core():
    cb = bench.cpu_baseline(TINY, workers=2, budget_s=0.05)
    assert cb["kind"] == "oracle" and cb["cores"] == 2 and cb["median_of"] == 3
    assert cb["value"] > 0 and cb["single_thread_value"] > 0
    assert cb["blas_threads_per_process"] == 1 and cb["nproc"] >= 1


def test_kernel_rooflines_use_the_byte_model():
    w = LLAMA_128K
    st2 = [{"misses": 100 * w.units}]           # 100 missed chunks per unit, one launch
    ph = {"score": 0.05, "select": 0.02, "rebuild": 0.025, "fetch": 0.1, "attn": 0.03}   # ms
    n = {k: 1 for k in ph}
    rows = {r["phase"]: r for r in bench.kernel_rooflines(w, 1, st2, ph, n, 40, 6800.0, 200.0)}
    U, d = w.units, w.head_dim
    assert rows["score"]["bytes_per_launch"] == U * (w.n_selectable * 2 + w.group * 2) * d
    assert rows["fetch"]["bound"] == "link" and rows["fetch"]["bytes_per_launch"] == 100 * U * w.chunk * d * 2
    assert rows["fetch"]["peak_gbs"] == 200.0 and rows["score"]["peak_gbs"] == 6800.0
    assert abs(rows["fetch"]["achieved_gbs"] - 100 * U * 8 * 128 * 2 / 1e-4 / 1e9) < 1e-6
    hbm = {r["phase"]: r for r in bench.kernel_rooflines(w.with_(v_place="hbm"), 1, st2, ph, n, 40, 6800.0, None)}
    assert hbm["fetch"]["bound"] == "hbm" and hbm["fetch"]["bytes_per_launch"] == 2 * rows["fetch"]["bytes_per_launch"]


def test_huge_page_storm_threshold():
    # 128 huge pages of a 64 GiB arena: a handful of splits is repaired in place, dozens mean a
    # storm and the bench falls back to page-locked values
    assert not bench.huge_storm(0, 128) and not bench.huge_storm(14, 128)
    assert not bench.huge_storm(32, 128) and bench.huge_storm(33, 128) and bench.huge_storm(86, 128)
