"""GPU parity of ShadowKV+ (generated keys kept at rank r) against the float64
oracle, through the C ABI.

The generated tokens' rank-r states a = k'.Psi must match the oracle's
projection within one storage ulp; outputs must match the oracle's attention
over the GPU's index set, with every generated key rebuilt as RoPE(a.B_h) at
its position, within 2e-2 (bf16, fp8) or 1e-4 relative (fp32).  The other bars
are those of the bf16 / fp32 / fp8 parity tests.  Step counts cross whole and
partial chunks of generated tokens.
"""
import pytest

from tests.gpu_harness import run_and_check
from workload import TINY, Workload

pytestmark = pytest.mark.gpu

SMALL_PLUS = Workload(
    name="bf16-8k-plus", layers=1, batch=2, seq_len=8192, n_kv_heads=8, n_q_heads=32, head_dim=128,
    rank=160, chunk=8, n_select=64, n_outlier=16, local_window=32, steps=19, dtype="bf16",
    v_place="hbm", drift=0.9, seed=41, new_keys="lowrank")


def test_plus_bf16_hbm_values_19_steps():
    rep = run_and_check(SMALL_PLUS, 19)
    assert rep.steps == 19


def test_plus_fp32_tiny():
    run_and_check(TINY.with_(new_keys="lowrank", seed=42, steps=10), 10)


def test_plus_fp8():
    run_and_check(SMALL_PLUS.with_(dtype="fp8", seed=43, steps=9), 9)


def test_plus_host_values_arena():
    run_and_check(SMALL_PLUS.with_(v_place="host", seed=44, steps=5), 5, host_alloc="arena")


def test_plus_no_local_window():
    run_and_check(TINY.with_(new_keys="lowrank", local_window=0, n_outlier=0, spike_chunks=0, seed=45,
                             steps=9), 9)
