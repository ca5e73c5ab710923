"""GPU parity: every stage of the decode path (through the C ABI) against the
float64 oracle on the same seeded inputs.

Bars: selected chunk ids identical except inside the near-tie band (1e-4
relative of the K-th score), outputs within 1e-4 relative (fp32 storage) or
2e-2 absolute (bf16 storage) of the oracle's attention over the GPU's index
set, outliers identical except near-ties, landmarks within one bf16 ulp of the
rounded oracle landmark (bf16) or 2e-5 (fp32), value rows bit-exact.
"""
import pytest
import torch

from tests.gpu_harness import run_and_check
from workload import LLAMA_32K, TINY, Workload

pytestmark = pytest.mark.gpu

SMALL_BF16 = Workload(
    name="bf16-8k", layers=1, batch=2, seq_len=8192, n_kv_heads=8, n_q_heads=32, head_dim=128,
    rank=160, chunk=8, n_select=64, n_outlier=16, local_window=32, steps=6, dtype="bf16",
    v_place="hbm", drift=0.9, seed=11)


def test_tiny_fp32_all_units_16_steps():
    rep = run_and_check(TINY, 16)
    assert rep.steps == 16
    assert rep.max_out_rel <= 1e-4


def test_tiny_fp32_single_stream():
    run_and_check(TINY.with_(seed=5), 4, side_stream=False)


def test_bf16_hbm_values():
    run_and_check(SMALL_BF16, 6)


def test_bf16_host_pinned_values():
    run_and_check(SMALL_BF16.with_(v_place="host", seed=12), 5)


def test_bf16_host_arena_values():
    # page-locked memory from shadowkv_host_alloc, passed as an interior slice
    run_and_check(SMALL_BF16.with_(v_place="host", seed=14), 4, host_alloc="arena")


def test_bf16_host_huge_page_values():
    # huge-page pageable memory from shadowkv_host_alloc_kind(SKV_HOST_HUGE), read through the
    # host page tables, passed as an interior slice
    run_and_check(SMALL_BF16.with_(v_place="host", seed=15), 4, host_alloc="huge")


def test_full_budget_selects_every_chunk():
    w = SMALL_BF16.with_(seq_len=1024, n_outlier=4, batch=1, seed=13)
    w = w.with_(n_select=w.n_selectable)
    rep = run_and_check(w, 3)
    assert rep.alphas[0] == 1.0          # every chunk selected: all hits after step 0


def test_repeated_query_hits_everything():
    rep = run_and_check(TINY.with_(drift=1.0, seed=7), 5)
    assert rep.alphas[0] == 1.0


def test_no_outliers_no_local_window():
    run_and_check(TINY.with_(n_outlier=0, local_window=0, spike_chunks=0, seed=8), 4)


def test_ragged_sizes():
    # n_c and K not multiples of any tile, 3 batch elements, odd rank
    w = Workload(name="ragged", layers=1, batch=3, seq_len=4096 + 8 * 13, n_kv_heads=2, n_q_heads=8,
                 head_dim=128, rank=40, chunk=8, n_select=33, n_outlier=5, local_window=24, steps=4,
                 dtype="bf16", v_place="hbm", drift=0.7, seed=9, spike_chunks=3)
    run_and_check(w, 4)


@pytest.mark.parametrize("G", [1, 2, 8])
def test_group_sizes(G):
    run_and_check(TINY.with_(n_q_heads=2 * G, seed=20 + G), 3)


def test_merge_of_many_contributors():
    # one unit whose attention spans ~67 CTAs: more partial records than the merge stages in
    # shared memory (96 KB, 46 contributors at G = 4), so they are loaded directly
    w = Workload(name="merge-many", layers=1, batch=1, seq_len=32768, n_kv_heads=1, n_q_heads=4,
                 head_dim=128, rank=160, chunk=8, n_select=1024, n_outlier=16, local_window=32, steps=2,
                 dtype="bf16", v_place="hbm", drift=0.9, seed=51)
    run_and_check(w, 2)


@pytest.mark.parametrize("G,dtype", [(1, "f32"), (2, "bf16")])
def test_selection_reads_unstaged_scores(G, dtype):
    # n_c = 505 selectable chunks: a unit's scores are not whole 16-byte words for G < 4, so the
    # selection reads them straight from global memory instead of staging them in shared memory
    run_and_check(TINY.with_(seq_len=4096 + 8, n_q_heads=2 * G, dtype=dtype, seed=40 + G), 3)


@pytest.mark.parametrize("rank", [8, 256])
def test_rank_extremes_bf16(rank):
    run_and_check(SMALL_BF16.with_(rank=rank, batch=1, seed=30 + rank), 3)


def test_fp32_rank_256_full_width():
    run_and_check(TINY.with_(rank=256, seed=31), 3)
