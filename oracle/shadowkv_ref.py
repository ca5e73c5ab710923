"""ShadowKV decode-step sparse attention: a plain, slow float64 CPU oracle.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module.  The product path
(the CUDA library and its Python binding) never calls it and shares no code
with it; both sides take their inputs from ``workload``.

Everything here is numpy in float64 and follows the two algorithms of the
pages in their order and notation:

* "ShadowKV: KV Cache in Shadows for High-Throughput Long-Context LLM
  Inference" (Chinese digest, section A2, Algorithm 1 "pre-filling" and
  Algorithm 2 "decoding"),
* the English summary of the same paper, section 3.4 ("Landmark Construction
  and Outlier Detection", "Decoding-Time KV Selection", "Sparse KV
  Reconstruction", "Theoretical Equivalent Bandwidth Model") and its
  appendix A.2 memory-savings formula.

Readings where the pages are silent (each is also listed in the design notes):

* RoPE is the Llama/NeoX half-split rotation, theta_i = base^(-2i/d), positions
  0-based, no frequency scaling.
* q-head j belongs to KV head j // G (contiguous grouped-query mapping).
* A is shared by the KV heads of one batch element: A [S][r], B_h [r][d].
* Outliers are chosen per (batch, KV head) among the chunks outside the local
  window, by the lowest minimum cosine between each token and its chunk mean;
  equal values rank the lower chunk id first.
* The local window (the last W prefill tokens) and every decode token are kept
  exact and are neither landmarks nor selectable.
* The softmax of the selection runs over the n_c selectable chunks only.
* The query and the new key arrive post-RoPE at position S+t.
* ShadowKV+ (generated keys at rank r): the new key arrives pre-RoPE, over all
  H heads of its batch element, and is kept as k' Psi with Psi = B^T; attention
  uses each generated token's key rebuilt from that state, RoPE(a.B_h) at S+t.
* FP8 storage (the summary's precision study runs ShadowKV in e5m2): landmarks
  and values are held in e5m2 (nearest, ties to the even mantissa, saturating);
  the query enters the score exactly, every kept key stays in bf16.
* Pre-filling from exact keys (Algorithm 1 takes K and K_RoPE): when the keys
  are given, landmarks, the min-cosine test and the outlier keys come from
  RoPE(K); A and B serve the decode-time rebuild only.

Parity pins: see ``tests/test_oracle_pins.py`` and ``tests/test_golden.py``.
The selection scores' near-tie band is not pinned by the pages (no page prints
per-element outputs); nothing here is "parity unpinned" beyond that.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

# ----------------------------------------------------------------------------
# RoPE (pages silent on the convention; reading: Llama half-split)
# ----------------------------------------------------------------------------


def rope_theta(d: int, base: float) -> np.ndarray:
    """theta_i = base^(-2i/d) for i < d/2, in float64."""
    i = np.arange(d // 2, dtype=np.float64)
    return np.power(float(base), -2.0 * i / d)


def apply_rope(x: np.ndarray, pos: np.ndarray, base: float) -> np.ndarray:
    """Rotate rows x [n][d] at integer positions pos [n] (half-split pairs i, i+d/2)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    h = d // 2
    ang = np.asarray(pos, dtype=np.float64)[:, None] * rope_theta(d, base)[None, :]
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[:, :h], x[:, h:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=1)


def rebuild_keys(A_rows: np.ndarray, B_h: np.ndarray, pos: np.ndarray, base: float) -> np.ndarray:
    """Post-RoPE keys of the given tokens from the low-rank factors.

    Summary page, section 3.4 "Sparse KV Reconstruction": K_sparse =
    MatMul(Gather(A, I), B), then RoPE at the tokens' own positions.
    """
    return apply_rope(np.asarray(A_rows, np.float64) @ np.asarray(B_h, np.float64), pos, base)


def chunk_tokens(chunk_ids, C: int) -> np.ndarray:
    """Token positions of the given chunks, chunk by chunk."""
    ids = np.asarray(chunk_ids, dtype=np.int64)
    return (ids[:, None] * C + np.arange(C, dtype=np.int64)[None, :]).reshape(-1)


# ----------------------------------------------------------------------------
# Algorithm 1 (pre-filling)
# ----------------------------------------------------------------------------


def reduce_chunks(K_rope: np.ndarray, C: int) -> np.ndarray:
    """Landmark of chunk j: the mean of its C post-RoPE keys (summary page,
    "Landmark Construction": k_bar_j = (1/c) sum_i k_RoPE)."""
    n = K_rope.shape[0] // C
    return K_rope[: n * C].reshape(n, C, -1).mean(axis=1)


def cosine(x: np.ndarray, y: np.ndarray) -> np.ndarray:
    """cos(x, y) = x.y / max(|x||y|, 1e-12), row-wise."""
    num = np.sum(x * y, axis=-1)
    den = np.linalg.norm(x, axis=-1) * np.linalg.norm(y, axis=-1)
    return num / np.maximum(den, 1e-12)


def chunk_min_cos(K_rope: np.ndarray, L: np.ndarray, C: int) -> np.ndarray:
    """Min over the chunk's tokens of cos(token key, chunk landmark)
    (Algorithm 1: S = CosineSimilarity(C, K_RoPE), then Min(S, dim=-1))."""
    n = L.shape[0]
    Kc = K_rope[: n * C].reshape(n, C, -1)
    return cosine(Kc, L[:, None, :]).min(axis=1)


def arg_topk(scores: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest scores in rank order; equal scores rank the
    lower index first (ArgTopK of Algorithms 1 and 2 with a fixed tie rule)."""
    scores = np.asarray(scores, dtype=np.float64)
    order = np.lexsort((np.arange(scores.shape[0]), -scores))
    return order[:k]


@dataclass
class UnitPrefill:
    """Per (batch, KV head) state that Algorithm 1 leaves on the GPU."""
    landmarks: np.ndarray      # [n_c][d]   L = C \ Gather(C, I), selectable chunks only
    ids: np.ndarray            # [n_c]      original chunk id of each landmark (ascending)
    outlier_ids: np.ndarray    # [O]        ascending
    min_cos: np.ndarray        # [S/C - W/C] per candidate chunk
    all_landmarks: np.ndarray  # [S/C - W/C][d]
    k_outlier: np.ndarray      # [O*C][d]
    v_outlier: np.ndarray      # [O*C][d]
    k_local: list = field(default_factory=list)   # rows, W prefill tokens then decode tokens
    v_local: list = field(default_factory=list)


def prefill_unit(A_b, B_bh, V_bh, C: int, O: int, W: int, base: float, K_exact=None) -> UnitPrefill:
    """Algorithm 1 for one (batch, KV head), with the factors A, B given.

    The SVD step is out of scope: A [S][r] and B_h [r][d] are inputs.  K_RoPE
    is the rotation at positions 0..S-1 of the pre-RoPE keys: the exact keys
    K_exact [S][d] when the caller has them (Algorithm 1 takes K and K_RoPE as
    inputs and builds landmarks, outliers and the outlier keys from K_RoPE),
    else A.B_h.
    """
    A_b = np.asarray(A_b, np.float64)
    V_bh = np.asarray(V_bh, np.float64)
    S = A_b.shape[0]
    n_chunk = S // C
    n_cand = n_chunk - W // C
    if K_exact is not None:
        K_rope = apply_rope(np.asarray(K_exact, np.float64), np.arange(S), base)   # K_RoPE
    else:
        K_rope = rebuild_keys(A_b, B_bh, np.arange(S), base)      # K_RoPE of the factors
    Cm = reduce_chunks(K_rope[: n_cand * C], C)                    # C = Reduce(K_RoPE)
    mcos = chunk_min_cos(K_rope, Cm, C)                            # Min(CosineSimilarity)
    out_ids = np.sort(arg_topk(-mcos, O))                          # ArgTopK(-Min(S), o)
    keep = np.ones(n_cand, dtype=bool)
    keep[out_ids] = False
    ids = np.nonzero(keep)[0]
    tok_o = chunk_tokens(out_ids, C)
    st = UnitPrefill(landmarks=Cm[ids], ids=ids, outlier_ids=out_ids, min_cos=mcos,
                     all_landmarks=Cm, k_outlier=K_rope[tok_o], v_outlier=V_bh[tok_o])
    for p in range(S - W, S):
        st.k_local.append(K_rope[p])
        st.v_local.append(V_bh[p])
    return st


# ----------------------------------------------------------------------------
# Algorithm 2 (decoding)
# ----------------------------------------------------------------------------


def softmax_rows(x: np.ndarray) -> np.ndarray:
    m = x.max(axis=-1, keepdims=True)
    e = np.exp(x - m)
    return e / e.sum(axis=-1, keepdims=True)


def select_chunks(q_group: np.ndarray, landmarks: np.ndarray, ids: np.ndarray, k: int) -> dict:
    """Landmark-guided selection for one KV head.

    q_group [G][d] are the post-RoPE queries of the G query heads that share
    this KV head (s_q = 1).  P = MatMul(Q, L^T); S = Softmax(P / sqrt(d));
    S1 = sum over query tokens (a no-op for one token); S2 = max over the group;
    I = ArgTopK(S2, k).  Returns the selected original chunk ids ascending.
    """
    q = np.asarray(q_group, np.float64)
    L = np.asarray(landmarks, np.float64)
    d = q.shape[-1]
    P = q @ L.T                              # [G][n_c]
    S = softmax_rows(P / math.sqrt(d))       # per query head over the n_c chunks
    S1 = S                                   # sum over s_q = 1 query tokens
    S2 = S1.max(axis=0)                      # max_kv_group
    ranked = arg_topk(S2, k)
    return {"P": P, "S": S, "S2": S2, "ranked": ranked,
            "sel": np.sort(np.asarray(ids)[ranked])}


def hit_miss(prev_sel, cur_sel):
    """Index scan against the previous step's selection: (hits, misses), each ascending."""
    cur = np.asarray(cur_sel, dtype=np.int64)
    if prev_sel is None:
        return np.zeros(0, np.int64), np.sort(cur)
    inprev = np.isin(cur, np.asarray(prev_sel, dtype=np.int64))
    return np.sort(cur[inprev]), np.sort(cur[~inprev])


def attend(q_group: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """Exact softmax(q K^T / sqrt(d)) V for each of the G query rows."""
    q = np.asarray(q_group, np.float64)
    d = q.shape[-1]
    s = q @ np.asarray(K, np.float64).T / math.sqrt(d)
    return softmax_rows(s) @ np.asarray(V, np.float64)


def round_to_storage(x: np.ndarray, storage: str | None) -> np.ndarray:
    """Value of x once stored in the configured storage dtype: "bf16" rounds
    to bfloat16 (nearest even), "f32" to float32, "e5m2" to the 8-bit float
    with 5 exponent and 2 mantissa bits, None keeps float64."""
    if storage is None:
        return np.asarray(x, np.float64)
    if storage == "bf16":
        return bf16_round(x)
    if storage == "f32":
        return np.asarray(x, np.float32).astype(np.float64)
    if storage == "e5m2":
        return e5m2_round(x)
    raise ValueError(storage)


def key_storage(dtype: str | None) -> str | None:
    """Storage of the keys the method keeps for a configuration dtype.  In the
    "fp8" configuration (summary page, section 5, "Precision sensitivity":
    ShadowKV run with float8 e5m2) landmarks and values are stored in e5m2
    while the keys, A and B stay bf16 (reading: the pages keep the factors at
    higher precision; the rebuilt keys are formed like the bf16 ones)."""
    return "bf16" if dtype == "fp8" else dtype


def value_storage(dtype: str | None) -> str | None:
    """Storage of the values (and of the landmarks) for a configuration dtype."""
    return "e5m2" if dtype == "fp8" else dtype


def attend_on_index_set(q_group, A_b, B_bh, V_bh, outlier_ids, sel_ids, k_local, v_local,
                        C: int, base: float, storage: str | None = None,
                        v_storage: str | None = None, k_outlier=None) -> np.ndarray:
    """Attention over [K_outlier; RoPE(K_sparse); K_local] for given index sets
    (summary page, "Assembly of the final sparse KV cache").  Keys of outlier
    and selected chunks are rebuilt here in float64 from A and B; with
    ``storage`` set, the keys the method keeps (outlier keys, rebuilt keys,
    local-window keys) take the value they have once stored in that dtype, and
    with ``v_storage`` set the local-window values likewise (context values
    arrive already stored).  ``k_outlier`` [O*C][d] gives the outlier keys when
    pre-filling took them from exact keys instead of the factors."""
    A_b = np.asarray(A_b, np.float64)
    V_bh = np.asarray(V_bh, np.float64)
    to = chunk_tokens(outlier_ids, C)
    ts = chunk_tokens(sel_ids, C)
    d = np.asarray(B_bh).shape[1]
    Ko = rebuild_keys(A_b[to], B_bh, to, base) if k_outlier is None else np.asarray(k_outlier, np.float64)
    K = np.concatenate([round_to_storage(Ko.reshape(-1, d), storage),
                        round_to_storage(rebuild_keys(A_b[ts], B_bh, ts, base), storage),
                        round_to_storage(np.asarray(k_local, np.float64).reshape(-1, d), storage)])
    V = np.concatenate([V_bh[to], V_bh[ts],
                        round_to_storage(np.asarray(v_local, np.float64).reshape(-1, d), v_storage)])
    return attend(q_group, K, V)


# ----------------------------------------------------------------------------
# ShadowKV+: generated tokens' keys kept at rank r (summary page, "The ShadowKV+
# extension for generated tokens"; digest, section A7 "handling of newly
# generated tokens")
# ----------------------------------------------------------------------------


def project_new_key(k_pre_b: np.ndarray, B_b: np.ndarray, storage: str | None = None) -> np.ndarray:
    """Rank-r state of one generated token of one batch element: k' Psi.

    k_pre_b [H][d] is the token's pre-RoPE key over the H KV heads, read as one
    row k' of width H*d; Psi is the context's right singular basis, which is B_b
    [H][r][d] read as the [r][H*d] matrix B = Psi^T.  The result a = k' Psi [r]
    is held in the storage dtype, as the context rows of A are.
    """
    B = np.asarray(B_b, np.float64)
    H, r, d = B.shape
    Psi_T = B.transpose(1, 0, 2).reshape(r, H * d)          # row j: (B[0][j], ..., B[H-1][j])
    k = np.asarray(k_pre_b, np.float64).reshape(H * d)
    return round_to_storage(Psi_T @ k, storage)


def new_token_key(a: np.ndarray, B_bh: np.ndarray, pos: int, base: float) -> np.ndarray:
    """Key of a generated token when attention needs it: head h's slice of the
    reconstruction (k' Psi) Psi^T is a.B_h, rotated at the token's position like
    a rebuilt context key."""
    return rebuild_keys(np.asarray(a, np.float64)[None, :], B_bh, np.array([pos]), base)[0]


@dataclass
class UnitDecodeState:
    pre: UnitPrefill
    prev_sel: np.ndarray | None = None
    steps: int = 0


def decode_step_unit(st: UnitDecodeState, q_group, k_new, v_new, A_b, B_bh, V_bh,
                     k: int, C: int, base: float) -> dict:
    """One step of Algorithm 2 for one (batch, KV head).

    Appends the new token to the exact local set, selects k chunks, rebuilds
    their keys, takes their values and attends over outliers + selected
    chunks + local tokens.  Returns the output [G][d], the selection and the
    hit/miss split against the previous step.
    """
    st.pre.k_local.append(np.asarray(k_new, np.float64))
    st.pre.v_local.append(np.asarray(v_new, np.float64))
    sel = select_chunks(q_group, st.pre.landmarks, st.pre.ids, k)
    hits, misses = hit_miss(st.prev_sel, sel["sel"])
    A_b = np.asarray(A_b, np.float64)
    V_bh = np.asarray(V_bh, np.float64)
    ts = chunk_tokens(sel["sel"], C)
    K = np.concatenate([st.pre.k_outlier, rebuild_keys(A_b[ts], B_bh, ts, base),
                        np.stack(st.pre.k_local)])
    V = np.concatenate([st.pre.v_outlier, V_bh[ts], np.stack(st.pre.v_local)])
    out = attend(q_group, K, V)
    st.prev_sel = sel["sel"]
    st.steps += 1
    return {"out": out, "sel": sel["sel"], "S2": sel["S2"], "ranked": sel["ranked"],
            "hits": hits, "misses": misses}


# ----------------------------------------------------------------------------
# Analytical models (summary page section 3.4 and appendix A.2; digest A2)
# ----------------------------------------------------------------------------


def equivalent_bandwidth(S, C, K, O, alpha, B_gpu, B_pcie):
    """B~ = 2 S B_GPU / (S/C + 2(K+O)C + (1-alpha) K C B_GPU / B_PCIe)."""
    return 2.0 * S * B_gpu / (S / C + 2.0 * (K + O) * C + (1.0 - alpha) * K * C * B_gpu / B_pcie)


def equivalent_bandwidth_terms(S, C, K, O, alpha, B_gpu, B_pcie):
    """The three denominator terms of the equivalent-bandwidth formula."""
    return (S / C, 2.0 * (K + O) * C, (1.0 - alpha) * K * C * B_gpu / B_pcie)


def memory_savings(S, M, C, K, O, r):
    """2SM / (SM/C + 2(K+O)C + Sr + rM), taken literally as printed."""
    return 2.0 * S * M / (S * M / C + 2.0 * (K + O) * C + S * r + r * M)


def compression_ratio(s, d, r):
    """sd / (r(s + d)): storage of A and B against the full key cache."""
    return s * d / (r * (s + d))


def sparse_budget_tokens(K, O, C):
    """Tokens attended from the context per KV head: (K + O) C."""
    return (K + O) * C


# ----------------------------------------------------------------------------
# Helpers for comparing with stored low-precision state
# ----------------------------------------------------------------------------


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bfloat16 (nearest even, via float32) and return float64."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = (u + 0x7FFF + lsb) >> 16 << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


E5M2_MAX = 57344.0          # 1.75 * 2^15, the largest finite e5m2 value
E5M2_MIN_NORMAL = 2.0 ** -14
E5M2_MIN_SUB = 2.0 ** -16   # subnormal spacing


def e5m2_round(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest e5m2 value (1 sign, 5 exponent bits
    with bias 15, 2 mantissa bits; ties to the even mantissa), saturating at
    the largest finite magnitude; returned as float64.  Between 2^e and
    2^(e+1) (normal range) the spacing is 2^(e-2); below 2^-14 it is 2^-16."""
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    # guard log2 rounding at exact powers of two
    e = np.where(2.0 ** e > a, e - 1, e)
    e = np.where(2.0 ** (e + 1) <= a, e + 1, e)
    q = np.where(a >= E5M2_MIN_NORMAL, 2.0 ** (e - 2), E5M2_MIN_SUB)
    m = a / q                                  # exact: q is a power of two
    r = np.floor(m)
    frac = m - r
    up = (frac > 0.5) | ((frac == 0.5) & (np.mod(r, 2) == 1))
    r = np.where(up, r + 1, r)
    y = np.minimum(r * q, E5M2_MAX)
    return np.where(np.isfinite(x), np.copysign(y, x), x)


def near_tie_band(scores: np.ndarray, k: int, rel: float = 1e-4):
    """Indices whose score lies within ``rel`` (relative) of the k-th largest
    score: membership of these may legitimately differ between two correct
    implementations that round differently."""
    scores = np.asarray(scores, np.float64)
    kth = scores[arg_topk(scores, k)[-1]]
    return np.nonzero(np.abs(scores - kth) <= rel * abs(kth))[0], kth
