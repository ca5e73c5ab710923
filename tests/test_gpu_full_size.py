"""Parity at the full per-layer sizes of the benchmark workloads, in the same
launch configuration the benchmark times (one layer; every layer of a step is
launched identically).  The oracle checks sampled units one by one."""
import pytest

from tests.gpu_harness import run_and_check
from workload import LLAMA_128K, LLAMA_1M, LLAMA_32K, SWEEP_64K

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def test_llama_32k_b4():
    run_and_check(LLAMA_32K, 4, units=[0, 13, 31], gen_device="cuda", check_cache=True)


def test_llama_128k_b8_host_values():
    rep = run_and_check(LLAMA_128K, 4, units=[0, 37, 63], gen_device="cuda", check_cache=False,
                        host_alloc="arena")
    assert rep.steps == 4


def test_llama_1m_b1_host_values():
    run_and_check(LLAMA_1M, 2, units=[5], gen_device="cuda", check_cache=False)


def test_sweep_64k_b48_host_values():
    w = SWEEP_64K.with_(batch=48, v_place="host", drift=0.5)
    run_and_check(w, 2, units=[0, 200, 383], gen_device="cuda", check_cache=False)


# The 64K sweep: every batch size, both value placements and every query drift appear in at
# least one full-size case (drift 0 draws an independent query each step, drift 0.99 nearly
# repeats it: the two ends of the hit-rate range).
@pytest.mark.parametrize("batch,place,drift,steps", [
    (1, "hbm", 0.0, 4),
    (8, "host", 0.99, 4),
    (16, "hbm", 0.5, 3),
    (32, "host", 0.9, 3),
    (48, "hbm", 0.99, 2),
])
def test_sweep_64k_points(batch, place, drift, steps):
    w = SWEEP_64K.with_(batch=batch, v_place=place, drift=drift)
    U = w.units
    units = sorted({0, U // 2, U - 1})
    run_and_check(w, steps, units=units, gen_device="cuda", check_cache=True, cache_units=units[:1],
                  host_alloc="huge")


def test_llama_128k_b8_host_values_64_steps():
    """The headline workload over all 64 decode steps of its configuration, huge-page host
    values as the bench allocates them; cache slots checked on one sampled unit every step."""
    rep = run_and_check(LLAMA_128K, 64, units=[5, 42], gen_device="cuda", check_cache=True, cache_units=[42],
                        host_alloc="huge")
    assert rep.steps == 64


def test_llama_128k_b8_fp8_host_values():
    """The e5m2 configuration at the benchmark's 128K size (bench.py --dtype fp8)."""
    rep = run_and_check(LLAMA_128K.with_(dtype="fp8"), 3, units=[1, 38, 62], gen_device="cuda",
                        check_cache=False, host_alloc="arena")
    assert rep.steps == 3


def test_llama_128k_b8_lowrank_new_keys():
    """ShadowKV+ at the benchmark's 128K size (bench.py --new-keys lowrank), values in HBM."""
    run_and_check(LLAMA_128K.with_(new_keys="lowrank", v_place="hbm"), 10, units=[2, 40, 63],
                  gen_device="cuda", check_cache=False)


def test_llama_32k_b4_exact_keys():
    """Pre-filling from exact keys at the 32K b4 size."""
    run_and_check(LLAMA_32K, 3, units=[0, 17, 31], gen_device="cuda", check_cache=True, exact_keys=True)


def test_llama_1m_b1_hbm_values():
    """1M context with values in HBM: the attention reads its 2048 cache slots' values in V
    through the selection's slot -> chunk table, and the selection runs on a cluster."""
    run_and_check(LLAMA_1M.with_(v_place="hbm"), 2, units=[3], gen_device="cuda", check_cache=True)


def test_llama_128k_b8_fp8_hbm_values():
    """The e5m2 configuration at 128K b8 with values in HBM, read in place (one 1 KB bulk copy
    per chunk)."""
    run_and_check(LLAMA_128K.with_(dtype="fp8", v_place="hbm"), 3, units=[4, 41], gen_device="cuda",
                  check_cache=True, cache_units=[41])
