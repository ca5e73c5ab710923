"""The five synthetic decode workloads (Llama-3.1-8B attention shape unless noted).

Shapes follow the ShadowKV summary page ("ShadowKV: KV Cache in Shadows for
High-Throughput Long-Context LLM Inference", section 3.4: rank 160, chunk 8,
outlier budget 48, sparse budget 1.56 %, 8 KV heads of head dim 128).  The
suites the pages evaluate on (RULER, LongBench, NIAH) and the model weights are
not available; these seeded synthetic workloads stand in for them.

This module holds no arithmetic of the method itself: it only names sizes.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    batch: int
    seq_len: int          # S, context tokens after prefill
    n_kv_heads: int       # H
    n_q_heads: int        # H * G
    head_dim: int         # d
    rank: int             # r (shared across the H heads of one batch element)
    chunk: int            # C
    n_select: int         # K chunks per KV head and step
    n_outlier: int        # O outlier chunks per KV head
    local_window: int     # W tokens kept exact (multiple of C)
    steps: int            # decode steps
    dtype: str            # "f32", "bf16" or "fp8" (storage; fp8: e5m2 landmarks and values, bf16
                          # keys and factors); accumulation is fp32 on the GPU
    v_place: str          # "hbm" or "host"
    drift: float = 0.9    # AR(1) coefficient of the query between steps
    seed: int = 0
    rope_base: float = 500000.0
    ar_rho: float = 0.95  # AR(1) coefficient of A rows along tokens
    spike_chunks: int = -1     # planted outlier chunks per batch element (-1: 0.3 % of chunks, capped at O)
    spike_scale: float = 6.0
    new_keys: str = "exact"    # "exact": generated keys kept whole; "lowrank": ShadowKV+ (kept at rank r)
    dense_chunks: int = -1     # >= 0: only the first dense_chunks chunks have nonzero A rows; every
                               # later chunk has zero keys, so all of them score exactly alike

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def n_chunks(self) -> int:
        return self.seq_len // self.chunk

    @property
    def n_selectable(self) -> int:
        """n_c: chunks that remain selectable after outliers and the local window."""
        return self.n_chunks - self.n_outlier - self.local_window // self.chunk

    @property
    def units(self) -> int:
        """Independent (batch, KV head) units per layer."""
        return self.batch * self.n_kv_heads

    @property
    def n_spikes(self) -> int:
        if self.spike_chunks >= 0:
            return self.spike_chunks
        cand = self.n_chunks - self.local_window // self.chunk
        return min(self.n_outlier, int(0.003 * self.n_chunks), cand)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


TINY = Workload(
    name="tiny-f32-4k", layers=1, batch=1, seq_len=4096, n_kv_heads=2, n_q_heads=8,
    head_dim=128, rank=32, chunk=8, n_select=16, n_outlier=4, local_window=32,
    steps=16, dtype="f32", v_place="hbm", drift=0.9, seed=0, spike_chunks=4, spike_scale=8.0)

LLAMA_32K = Workload(
    name="llama3.1-8b-attn-32k-b4", layers=32, batch=4, seq_len=32768, n_kv_heads=8,
    n_q_heads=32, head_dim=128, rank=160, chunk=8, n_select=64, n_outlier=16,
    local_window=32, steps=64, dtype="bf16", v_place="hbm", drift=0.9, seed=0)

LLAMA_128K = Workload(
    name="llama3.1-8b-attn-128k-b8", layers=32, batch=8, seq_len=131072, n_kv_heads=8,
    n_q_heads=32, head_dim=128, rank=160, chunk=8, n_select=256, n_outlier=48,
    local_window=32, steps=64, dtype="bf16", v_place="host", drift=0.9, seed=0)

LLAMA_1M = Workload(
    name="llama3-8b-attn-1m-b1", layers=32, batch=1, seq_len=1048576, n_kv_heads=8,
    n_q_heads=32, head_dim=128, rank=160, chunk=8, n_select=2048, n_outlier=384,
    local_window=32, steps=32, dtype="bf16", v_place="host", drift=0.9, seed=3)

SWEEP_64K = Workload(
    name="llama3.1-8b-attn-64k-sweep", layers=32, batch=1, seq_len=65536, n_kv_heads=8,
    n_q_heads=32, head_dim=128, rank=160, chunk=8, n_select=128, n_outlier=24,
    local_window=32, steps=32, dtype="bf16", v_place="hbm", drift=0.9, seed=0)

SWEEP_BATCHES = (1, 8, 16, 32, 48)
SWEEP_DRIFTS = (0.0, 0.5, 0.9, 0.99)

ALL = {w.name: w for w in (TINY, LLAMA_32K, LLAMA_128K, LLAMA_1M, SWEEP_64K)}


def sweep_points():
    """Every (batch, placement, drift) point of the 64K sweep."""
    for b in SWEEP_BATCHES:
        for place in ("hbm", "host"):
            for drift in SWEEP_DRIFTS:
                yield SWEEP_64K.with_(batch=b, v_place=place, drift=drift,
                                      name=f"{SWEEP_64K.name}-b{b}-{place}-drift{drift}")
