"""Exact ties at the top-K boundary of a long unit.

ShadowKV (section 3.3, sparse budget selection) keeps the K chunks of highest
max-over-group probability; this build breaks equal scores towards the lower
chunk position.  Here every chunk after the first 1024 has zero keys, so its
landmark is zero and its score equals that of every other such chunk bit for
bit, on the GPU and in the oracle alike.  With 32768 selectable chunks and
K = 4096 the boundary falls inside that tie group, and the tie members taken
reach past the first 4096 positions: the selection has to rank ties across
the whole unit, not within a part of it.  A second step with a zero query makes
every score equal, the degenerate case where the K lowest positions win.
"""
import numpy as np
import pytest
import torch

from tests.gpu_harness import LayerRun, Report, check_prefill, check_step, np64
from workload import LLAMA_1M

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TIES_256K = LLAMA_1M.with_(name="ties-256k-b1", seq_len=262560, n_select=4096, n_outlier=48,
                           v_place="hbm", spike_chunks=0, dense_chunks=1024, steps=2, seed=5)


def test_tie_group_at_the_boundary_and_zero_query():
    w = TIES_256K
    assert w.n_selectable == 32768
    units = [0, 3, 7]
    run = LayerRun(w, 2, gen_device="cuda")
    run.q_d[1].zero_()
    run.q_src[1].zero_()
    check_prefill(run, units)
    rep, prev = Report(), {}
    U, K, d = w.units, w.n_select, w.head_dim
    for t in range(2):
        run.step()
        check_step(run, units, rep, prev, check_cache=True)
        L = run.export("landmarks", run.vdtype(), (U, w.n_selectable, d))
        ids = run.export("chunk_ids", torch.int32, (U, w.n_selectable)).cpu().numpy()
        sel = run.sel.view(U, K).cpu().numpy()
        for u in range(U):
            zero = np.all(np64(L[u]) == 0.0, axis=1)
            # the outliers are zero chunks too (min-cos 0), so every dense chunk stays selectable
            assert zero.sum() == w.n_selectable - w.dense_chunks
            if t == 1:
                # all scores equal: the K lowest positions
                assert np.array_equal(sel[u], ids[u][:K]), f"zero query (unit {u})"
                continue
            zid = ids[u][zero]
            taken = np.isin(zid, sel[u])
            m = int(taken.sum())
            assert m > 0 and np.all(taken[:m]) and not np.any(taken[m:]), \
                f"tied chunks taken are not the lowest positions (unit {u})"
            last = int(np.nonzero(zero)[0][m - 1])
            assert last >= 4096, f"tie boundary at position {last} (unit {u})"
    st = run.layer.stats()
    assert st["status"] == 0 and st["device_error"] == 0
    run.layer.close()

