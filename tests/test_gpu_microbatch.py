"""Two handles of one layer decoding side by side, as bench.py --microbatches 2 [--pipeline]
runs a batch split in two: each half-batch is its own handle on its own (main, side) stream
pair, and with the pipeline each one's step waits for the other's selection
(shadowkv_set_select_event), so one's value fetch overlaps the other's scoring.  Each handle
is checked against the oracle after every step, as in the single-handle parity tests."""
import pytest
import torch

from tests.gpu_harness import REPORTS, LayerRun, Report, check_prefill, check_step, summary
from workload import LLAMA_32K, Workload

pytestmark = pytest.mark.gpu

HALF = Workload(name="microbatch-bf16", layers=1, batch=2, seq_len=8192, n_kv_heads=8, n_q_heads=32,
                head_dim=128, rank=160, chunk=8, n_select=64, n_outlier=16, local_window=32, steps=6,
                dtype="bf16", v_place="host", drift=0.9, seed=81)


def _side_by_side(wa: Workload, wb: Workload, steps: int, units, pipelined: bool, host_alloc="huge",
                  gen_device="cpu", check_cache=True):
    ra = LayerRun(wa, steps, gen_device=gen_device, host_alloc=host_alloc)
    rb = LayerRun(wb, steps, gen_device=gen_device, host_alloc=host_alloc)
    ea, eb = torch.cuda.Event(), torch.cuda.Event()
    if pipelined:
        ra.layer.set_select_event(ea)
        rb.layer.set_select_event(eb)
    check_prefill(ra, units)
    check_prefill(rb, units)
    reps, prevs = [Report(), Report()], [{}, {}]
    torch.cuda.synchronize()
    for _ in range(steps):
        if pipelined:
            ra.main.wait_event(eb)         # a scores after b's previous selection
        ra.enqueue()
        if pipelined:
            rb.main.wait_event(ea)         # b scores after a's selection of this step
        rb.enqueue()
        torch.cuda.synchronize()
        for r, rep, prev in zip((ra, rb), reps, prevs):
            check_step(r, units, rep, prev, check_cache=check_cache)
    for r, rep in zip((ra, rb), reps):
        st = r.layer.stats()
        assert st["status"] == 0 and st["device_error"] == 0 and st["steps"] == steps
        rep.alphas = [st["alpha_mean"], st["alpha_last"]]
        REPORTS.append(summary(r.w, steps, units, rep, f"{host_alloc} {'pipelined' if pipelined else 'side-by-side'}"))
        r.layer.close()


@pytest.mark.parametrize("pipelined", [False, True])
def test_two_half_batches_side_by_side(pipelined):
    _side_by_side(HALF, HALF.with_(seed=82), 6, units=list(range(HALF.units)), pipelined=pipelined)


def test_two_half_batches_hbm_values_pipelined():
    w = HALF.with_(v_place="hbm", seed=83)
    _side_by_side(w, w.with_(seed=84), 5, units=list(range(w.units)), pipelined=True)


@pytest.mark.slow
def test_llama_32k_two_half_batches_pipelined():
    """The 32K b4 workload split in two b2 handles, at its full per-layer size, host values."""
    w = LLAMA_32K.with_(batch=2, v_place="host")
    _side_by_side(w, w.with_(seed=LLAMA_32K.seed + 1), 4, units=[0, 9, 15], pipelined=True,
                  gen_device="cuda", check_cache=True)
