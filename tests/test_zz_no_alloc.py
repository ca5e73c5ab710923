"""The attention entry point that allocates nothing.

Callers that cannot allocate device memory on their hot path (a server that
owns all of HBM through one pool, code under an allocator lock) use
shadowkv_sparse_attention_noalloc, whose scratch is a fixed array inside the
library.  These tests call it through the C ABI:

* against the float64 oracle's attention (softmax(q.K^T/sqrt(d)).V over the
  exact bf16 rows the call reads), for every group size, with and without
  outlier and cache regions (NULL pointers for empty ones), on shapes of one
  and of several 128-token splits, two calls in a row on the shared array;
* against the decode step's own attention output on a layer's regions, on two
  consecutive steps;
* the refusals: too many units, a unit whose merge state exceeds shared
  memory, a host pointer -- all decided on the host before anything runs.

This file sorts last so that a run stopping at the first failure has run every
other test first.  It passes alone in a fresh process too: the first call on
the device does the per-device set-up itself.
"""
import numpy as np
import pytest
import torch

import sparse_kv_cache_gb300 as skv
from oracle import shadowkv_ref as ref
from tests.gpu_harness import LayerRun
from workload import Workload, make_normal

pytestmark = pytest.mark.gpu

TOL = 2e-2   # bf16 output bar of the parity tests (max abs error)
d = 128

W = Workload(name="noalloc-bf16", layers=1, batch=2, seq_len=8192, n_kv_heads=8, n_q_heads=32,
             head_dim=128, rank=160, chunk=8, n_select=64, n_outlier=16, local_window=32, steps=2,
             dtype="bf16", v_place="hbm", drift=0.9, seed=21)


def _regions(units, group, n_out, n_cache, cap, seed):
    dev = "cuda"
    q = make_normal((units * group, d), seed, device=dev)
    ko = make_normal((units, n_out, d), seed + 1, device=dev) if n_out else None
    vo = make_normal((units, n_out, d), seed + 2, device=dev) if n_out else None
    kc = make_normal((units, n_cache, d), seed + 3, device=dev) if n_cache else None
    vc = make_normal((units, n_cache, d), seed + 4, device=dev) if n_cache else None
    kl = make_normal((units, cap, d), seed + 5, device=dev)
    vl = make_normal((units, cap, d), seed + 6, device=dev)
    return q, ko, vo, kc, vc, kl, vl


def _oracle(q, ko, vo, kc, vc, kl, vl, units, group, n_loc):
    """Per unit: the oracle's exact attention over [outlier rows; cache rows; first n_loc local rows]."""
    f = lambda t: t.float().cpu().double().numpy()  # noqa: E731 (bf16 values are exact in float64)
    out = np.empty((units * group, d))
    for u in range(units):
        ks = [f(kl[u, :n_loc])]
        vs = [f(vl[u, :n_loc])]
        if kc is not None:
            ks.insert(0, f(kc[u]))
            vs.insert(0, f(vc[u]))
        if ko is not None:
            ks.insert(0, f(ko[u]))
            vs.insert(0, f(vo[u]))
        out[u * group:(u + 1) * group] = ref.attend(f(q[u * group:(u + 1) * group]), np.concatenate(ks),
                                                    np.concatenate(vs))
    return out


@pytest.mark.parametrize("group,units,n_out,n_cache,cap,n_loc", [
    (1, 3, 0, 0, 40, 33),          # local rows only, one split, NULL outlier and cache pointers
    (2, 5, 24, 0, 64, 50),         # no cache region (NULL), one split
    (4, 4, 384, 2048, 100, 90),    # the decode step's regions at 32K: 20 splits, ragged tail
    (8, 2, 0, 700, 16, 16),        # no outliers (NULL), 6 splits with a ragged last one
    (8, 1, 128, 5000, 300, 257),   # one long unit: 43 splits merged by the last CTA
])
def test_noalloc_matches_oracle_twice(group, units, n_out, n_cache, cap, n_loc):
    q, ko, vo, kc, vc, kl, vl = _regions(units, group, n_out, n_cache, cap, seed=100 + group)
    expect = _oracle(q, ko, vo, kc, vc, kl, vl, units, group, n_loc)
    s = torch.cuda.current_stream()
    for call in range(2):   # the second call reuses the array the first one left behind
        out = torch.full((units * group, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = skv.sparse_attention_noalloc(q, ko, vo, kc, vc, kl, vl, out, units=units, group=group,
                                          n_outlier_tokens=n_out, n_cache_tokens=n_cache,
                                          n_local_tokens=n_loc, local_capacity=cap, stream=s)
        assert rc == 0, skv.strerror(rc)
        assert skv.sparse_attention_noalloc_status(s) == 0
        err = np.abs(out.float().cpu().double().numpy() - expect).max()
        assert err <= TOL, f"call {call}: max abs error {err} against the oracle"


def test_noalloc_matches_decode_step_twice():
    run = LayerRun(W, 2)
    U, G, C, K, O = W.units, W.group, W.chunk, W.n_select, W.n_outlier
    cap = W.local_window + 2
    for t in range(2):
        run.step()
        ko = run.export("k_outlier", torch.bfloat16, (U, O * C, d))
        vo = run.export("v_outlier", torch.bfloat16, (U, O * C, d))
        kc = run.export("k_cache", torch.bfloat16, (U, K * C, d))
        vc = run.export("v_cache", torch.bfloat16, (U, K * C, d))
        kl = run.export("k_local", torch.bfloat16, (U, cap, d))
        vl = run.export("v_local", torch.bfloat16, (U, cap, d))
        out = torch.full_like(run.out, float("nan"))
        rc = skv.sparse_attention_noalloc(run.q_d[t], ko, vo, kc, vc, kl, vl, out, units=U, group=G,
                                          n_outlier_tokens=O * C, n_cache_tokens=K * C,
                                          n_local_tokens=W.local_window + t + 1, local_capacity=cap,
                                          stream=run.main)
        assert rc == 0, skv.strerror(rc)
        run.main.synchronize()
        err = (out.float() - run.out.float()).abs().max().item()
        assert err <= TOL, f"call {t}: max abs difference {err} against the decode step"
    assert skv.sparse_attention_noalloc_status(run.main) == 0
    run.layer.close()


def test_noalloc_setup_call_launches_nothing():
    assert skv.sparse_attention_noalloc_setup() == 0
    assert skv.sparse_attention_noalloc_status() == 0


def test_noalloc_refuses_shapes_beyond_its_scratch():
    q = torch.zeros((1, d), dtype=torch.bfloat16, device="cuda")
    # more units than merge tickets
    rc = skv.sparse_attention_noalloc(q, None, None, None, None, q, q, q, units=20000, group=1,
                                      n_outlier_tokens=0, n_cache_tokens=0, n_local_tokens=1,
                                      local_capacity=1)
    assert rc == -1
    # one unit of 340K rows at group 8: the partials fit in the array (11 MB) but the merge
    # state of 2657 splits x 8 heads does not fit in one CTA's shared memory.  The buffers are
    # real, so the shape would be in bounds even if it were launched.
    rows = 340_000
    kl = torch.zeros((1, rows, d), dtype=torch.bfloat16, device="cuda")
    q8 = torch.zeros((8, d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q8)
    rc = skv.sparse_attention_noalloc(q8, None, None, None, None, kl, kl, out, units=1, group=8,
                                      n_outlier_tokens=0, n_cache_tokens=0, n_local_tokens=rows,
                                      local_capacity=rows)
    assert rc == -1
    torch.cuda.synchronize()
    assert skv.sparse_attention_noalloc_status() == 0


def test_noalloc_refuses_host_pointers():
    q = torch.zeros((4, d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    host = torch.zeros((1, 8, d), dtype=torch.bfloat16)   # pageable CPU memory
    dev = torch.zeros((1, 8, d), dtype=torch.bfloat16, device="cuda")
    rc = skv.sparse_attention_noalloc(q, None, None, None, None, host, dev, out, units=1, group=4,
                                      n_outlier_tokens=0, n_cache_tokens=0, n_local_tokens=8,
                                      local_capacity=8)
    assert rc == -1
    rc = skv.sparse_attention_noalloc(q, None, None, host, dev, dev, dev, out, units=1, group=4,
                                      n_outlier_tokens=0, n_cache_tokens=8, n_local_tokens=8,
                                      local_capacity=8)
    assert rc == -1
