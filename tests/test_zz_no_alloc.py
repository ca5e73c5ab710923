"""The attention entry point that allocates nothing, against the decode step.

Callers that cannot allocate device memory on their hot path (a server that
owns all of HBM through one pool, code under an allocator lock) use
shadowkv_sparse_attention_noalloc, whose scratch is a fixed array inside the
library.  Here a layer runs two decode steps; after each, the no-allocation
call is made through the C ABI on the layer's own key/value regions and the
same queries, and its output must match the decode step's output within the
bf16 output tolerance of the parity tests.  This file sorts last so that a run
stopping at the first failure has run every other test first.
"""
import pytest
import torch

import sparse_kv_cache_gb300 as skv
from tests.gpu_harness import LayerRun
from workload import Workload

pytestmark = pytest.mark.gpu

W = Workload(name="noalloc-bf16", layers=1, batch=2, seq_len=8192, n_kv_heads=8, n_q_heads=32,
             head_dim=128, rank=160, chunk=8, n_select=64, n_outlier=16, local_window=32, steps=2,
             dtype="bf16", v_place="hbm", drift=0.9, seed=21)


def test_noalloc_attention_matches_decode_step_twice():
    run = LayerRun(W, 2)
    U, G, d, C, K, O = W.units, W.group, W.head_dim, W.chunk, W.n_select, W.n_outlier
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
        assert err <= 2e-2, f"call {t}: max abs difference {err}"
    run.layer.close()


def test_noalloc_rejects_shapes_beyond_its_scratch():
    q = torch.zeros((1, 128), dtype=torch.bfloat16, device="cuda")
    rc = skv.sparse_attention_noalloc(q, None, None, None, None, q, q, q, units=20000, group=1,
                                      n_outlier_tokens=0, n_cache_tokens=0, n_local_tokens=1,
                                      local_capacity=1)
    assert rc == -1
