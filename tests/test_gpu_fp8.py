"""GPU parity of the fp8 configuration (e5m2 landmarks and values, bf16 keys and factors)
against the float64 oracle, through the C ABI.

Bars as for bf16 storage: selections identical except inside the near-tie band, outputs within
2e-2 absolute of the oracle's attention over the GPU's index set (keys rounded to bf16, the
appended values to e5m2), landmarks within one e5m2 step of the rounded oracle landmark, value
rows (outliers, local window, cache slots) bit-exact copies of the e5m2 inputs.
"""
import pytest

from tests.gpu_harness import run_and_check
from workload import Workload

pytestmark = pytest.mark.gpu

SMALL_FP8 = Workload(
    name="fp8-8k", layers=1, batch=2, seq_len=8192, n_kv_heads=8, n_q_heads=32, head_dim=128,
    rank=160, chunk=8, n_select=64, n_outlier=16, local_window=32, steps=6, dtype="fp8",
    v_place="hbm", drift=0.9, seed=21)


def test_fp8_hbm_values():
    run_and_check(SMALL_FP8, 6)


def test_fp8_host_values():
    run_and_check(SMALL_FP8.with_(v_place="host", seed=22), 4, host_alloc="arena")


@pytest.mark.parametrize("G", [1, 8])
def test_fp8_group_sizes(G):
    # G = 8 needs 24 query-term rows: the scorer's N = 32 form
    run_and_check(SMALL_FP8.with_(n_q_heads=8 * G, seed=23 + G, n_select=32), 3)
