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
