"""Seeded synthetic inputs shared by the CUDA path and the oracle.

Both sides receive the same bytes from here; neither side's arithmetic lives
here.  The recipe (one seeded torch generator per layer and purpose):

* A rows [b][S][r]: AR(1) along tokens per coordinate, A[0] ~ N(0,1),
  A[i] = rho*A[i-1] + sqrt(1-rho^2)*eps, so every row is N(0,1) marginally.
* planted outlier chunks: per batch element, ``n_spikes`` chunks drawn uniformly
  without replacement outside the local window; the A rows of their odd token
  offsets are replaced by ``spike_scale * N(0,1)``.
* B [b][H][r][d] ~ N(0, 1/r), so every pre-RoPE key coordinate has variance 1.
  For ShadowKV+ workloads (``new_keys == "lowrank"``) B is the right singular
  basis an SVD would give: B_b read as [r][H*d] has orthonormal rows (QR of a
  Gaussian matrix), and A is scaled by sqrt(H*d/r) so that the keys keep unit
  per-coordinate variance.
* V [b][H][S][d] ~ N(0,1).
* exact pre-RoPE keys (pre-filling from exact keys only): A.B_h + N(0, 0.01).
* queries q [T][b][H*G][d]: q_0 ~ N(0,1), q_t = drift*q_{t-1} + sqrt(1-drift^2)*eps
  (already post-RoPE, as a model hands them to the attention).
* new tokens k_new, v_new [T][b][H][d] ~ N(0,1): the key of a generated token
  arrives post-RoPE from the model's own projection, outside this path, so it is
  drawn with the per-coordinate variance of the rebuilt keys.  For ShadowKV+
  workloads k_new is the pre-RoPE key, drawn inside the context's subspace plus
  a small residue: k'_t = c_t.B_b + 0.1*eps with c_t ~ N(0, H*d/r).

The generator on a CUDA device uses torch's Philox stream and the one on the CPU
uses torch's CPU stream, so the same seed gives different numbers on the two;
a test generates once and hands the same tensors to both sides.
"""
from __future__ import annotations

import math

import torch

from .configs import Workload

_PURPOSE = {"A": 1, "spike": 2, "B": 3, "V": 4, "q": 5, "k_new": 6, "v_new": 7, "k_exact": 8}


def _gen(w: Workload, layer: int, purpose: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((w.seed * 1_000_003 + layer * 7919 + _PURPOSE[purpose] * 104_729) % (2**63 - 1))
    return g


def storage_dtype(w: Workload) -> torch.dtype:
    """Storage of A, B, the queries and the new keys and values as handed in."""
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


def value_dtype(w: Workload) -> torch.dtype:
    """Storage of the context values: float8 e5m2 in the "fp8" configuration."""
    return torch.float8_e5m2 if w.dtype == "fp8" else storage_dtype(w)


def ar1_scan(e: torch.Tensor, rho: float, dim: int) -> torch.Tensor:
    """x_i = rho*x_{i-1} + e_i along ``dim`` (x_0 = e_0), by log-depth doubling."""
    x = e.movedim(dim, 0).clone()
    n = x.shape[0]
    step, coef = 1, rho
    while step < n and coef != 0.0:
        x[step:] += coef * x[:-step]
        step *= 2
        coef = coef * coef
    return x.movedim(0, dim)


def spike_chunks(w: Workload, layer: int) -> torch.Tensor:
    """[b][n_spikes] planted chunk ids (int64, sorted), drawn on the CPU."""
    g = _gen(w, layer, "spike", "cpu")
    cand = w.n_chunks - w.local_window // w.chunk
    out = torch.empty((w.batch, w.n_spikes), dtype=torch.int64)
    for b in range(w.batch):
        out[b] = torch.randperm(cand, generator=g)[: w.n_spikes].sort().values
    return out


def _lowrank_scale(w: Workload) -> float:
    return math.sqrt(w.n_kv_heads * w.head_dim / w.rank)


def make_A(w: Workload, layer: int, device="cpu") -> torch.Tensor:
    g = _gen(w, layer, "A", device)
    e = torch.randn((w.batch, w.seq_len, w.rank), generator=g, device=device, dtype=torch.float32)
    e[:, 1:] *= math.sqrt(1.0 - w.ar_rho ** 2)
    A = ar1_scan(e, w.ar_rho, dim=1)
    del e
    if w.dense_chunks >= 0:
        A[:, w.dense_chunks * w.chunk:] = 0
    sp = spike_chunks(w, layer)
    if sp.numel():
        gs = _gen(w, layer, "spike", device)
        odd = torch.arange(1, w.chunk, 2)
        for b in range(w.batch):
            rows = (sp[b][:, None] * w.chunk + odd[None, :]).reshape(-1).to(device)
            A[b, rows] = w.spike_scale * torch.randn((rows.numel(), w.rank), generator=gs,
                                                     device=device, dtype=torch.float32)
    if w.new_keys == "lowrank":
        A *= _lowrank_scale(w)
    return A.to(storage_dtype(w))


def make_B(w: Workload, layer: int, device="cpu") -> torch.Tensor:
    g = _gen(w, layer, "B", device)
    if w.new_keys == "lowrank":
        H, d, r = w.n_kv_heads, w.head_dim, w.rank
        if r > H * d:
            raise ValueError("a rank-r orthonormal basis needs r <= H*d")
        G = torch.randn((w.batch, H * d, r), generator=g, device=device, dtype=torch.float64)
        Q = torch.linalg.qr(G).Q                                  # [b][H*d][r], orthonormal columns
        B = Q.transpose(1, 2).reshape(w.batch, r, H, d).permute(0, 2, 1, 3).contiguous()
        return B.to(torch.float32).to(storage_dtype(w))
    B = torch.randn((w.batch, w.n_kv_heads, w.rank, w.head_dim), generator=g, device=device,
                    dtype=torch.float32) / math.sqrt(w.rank)
    return B.to(storage_dtype(w))


def make_K_exact(w: Workload, layer: int, device="cpu", A=None, B=None) -> torch.Tensor:
    """Exact pre-RoPE keys [b][H][S][d] for pre-filling from exact keys: the
    factors' keys A.B_h plus N(0, 0.01) noise (the configs' noisy keys), so the
    factors are a close but not exact low-rank fit of them."""
    A = make_A(w, layer, device) if A is None else A
    B = make_B(w, layer, device) if B is None else B
    g = _gen(w, layer, "k_exact", device)
    K = torch.empty((w.batch, w.n_kv_heads, w.seq_len, w.head_dim), dtype=storage_dtype(w), device=device)
    for b in range(w.batch):
        Af = A[b].float()
        for h in range(w.n_kv_heads):
            noise = torch.randn((w.seq_len, w.head_dim), generator=g, device=device, dtype=torch.float32)
            K[b, h] = (Af @ B[b, h].float() + 0.1 * noise).to(K.dtype)
    return K


def make_V(w: Workload, layer: int, device="cpu") -> torch.Tensor:
    g = _gen(w, layer, "V", device)
    dt = value_dtype(w)
    V = torch.empty((w.batch, w.n_kv_heads, w.seq_len, w.head_dim), dtype=dt, device=device)
    # fill one (b, h) slab at a time to bound the fp32 temporary
    for b in range(w.batch):
        for h in range(w.n_kv_heads):
            V[b, h] = torch.randn((w.seq_len, w.head_dim), generator=g, device=device,
                                  dtype=torch.float32).to(dt)
    return V


def make_decode_inputs(w: Workload, layer: int, steps: int | None = None, device="cpu"):
    """q [T][b][H*G][d], k_new [T][b][H][d], v_new [T][b][H][d] in storage dtype."""
    T = w.steps if steps is None else steps
    dt = storage_dtype(w)
    gq = _gen(w, layer, "q", device)
    e = torch.randn((T, w.batch, w.n_q_heads, w.head_dim), generator=gq, device=device,
                    dtype=torch.float32)
    e[1:] *= math.sqrt(max(0.0, 1.0 - w.drift ** 2))
    q = ar1_scan(e, w.drift, dim=0) if w.drift != 0.0 else e
    gk = _gen(w, layer, "k_new", device)
    k_new = torch.randn((T, w.batch, w.n_kv_heads, w.head_dim), generator=gk, device=device,
                        dtype=torch.float32)
    if w.new_keys == "lowrank":
        Bf = make_B(w, layer, device).float()                     # [b][H][r][d]
        c = torch.randn((T, w.batch, w.rank), generator=gk, device=device,
                        dtype=torch.float32) * _lowrank_scale(w)
        k_new = 0.1 * k_new + torch.einsum("tbj,bhjd->tbhd", c, Bf)
    gv = _gen(w, layer, "v_new", device)
    v_new = torch.randn((T, w.batch, w.n_kv_heads, w.head_dim), generator=gv, device=device,
                        dtype=torch.float32)
    return q.to(dt), k_new.to(dt), v_new.to(dt)


def make_layer(w: Workload, layer: int, device="cpu"):
    """All prefill inputs of one layer: dict(A, B, V) in storage dtype on ``device``."""
    return {"A": make_A(w, layer, device), "B": make_B(w, layer, device),
            "V": make_V(w, layer, device)}


def make_normal(shape, seed: int, dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    """N(0,1) draws of a given shape from a generator seeded with ``seed`` (CPU stream),
    rounded to ``dtype``: plain attention regions for tests of the attention call alone."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return torch.randn(tuple(shape), generator=g, dtype=torch.float32).to(dtype).to(device)
