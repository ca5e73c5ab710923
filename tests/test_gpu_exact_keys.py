"""GPU parity of pre-filling from exact keys (the digest's Algorithm 1 with K and
K_RoPE as inputs) against the float64 oracle, through the C ABI.

The exact keys are the factors' keys plus N(0, 0.01) noise, so landmarks,
min-cosines and outliers differ from the factor-built ones.  Bars as in the
other parity tests: landmarks within one storage step of the rounded oracle,
min-cos within 1e-4, outliers identical outside the near-tie band, outlier and
local keys equal to RoPE(K) within one storage ulp, and every decode step's
selection and output against the oracle on the GPU's state.
"""
import pytest

from tests.gpu_harness import run_and_check
from workload import TINY, Workload

pytestmark = pytest.mark.gpu

SMALL_X = Workload(
    name="bf16-8k-exact-keys", layers=1, batch=2, seq_len=8192, n_kv_heads=8, n_q_heads=32, head_dim=128,
    rank=160, chunk=8, n_select=64, n_outlier=16, local_window=32, steps=5, dtype="bf16",
    v_place="hbm", drift=0.9, seed=61)


def test_exact_keys_bf16():
    run_and_check(SMALL_X, 5, exact_keys=True)


def test_exact_keys_fp32_tiny():
    run_and_check(TINY.with_(seed=62), 6, exact_keys=True)


def test_exact_keys_fp8_host_values():
    run_and_check(SMALL_X.with_(dtype="fp8", v_place="host", seed=63), 4, exact_keys=True, host_alloc="arena")


def test_exact_keys_with_lowrank_new_keys():
    run_and_check(SMALL_X.with_(new_keys="lowrank", seed=64, steps=9), 9, exact_keys=True)
