"""Plant plausible mistakes in the oracle (CPU only) and check that the pins catch each."""
import math

import numpy as np
import pytest

from oracle import shadowkv_ref as ref
from tests import test_oracle_pins as pins


def _rope_wrong_sign(x, pos, base):
    x = np.asarray(x, np.float64)
    h = x.shape[-1] // 2
    ang = np.asarray(pos, np.float64)[:, None] * ref.rope_theta(x.shape[-1], base)[None, :]
    c, s = np.cos(ang), np.sin(ang)
    return np.concatenate([x[:, :h] * c + x[:, h:] * s, -x[:, :h] * s + x[:, h:] * c], axis=1)


def _rope_interleaved(x, pos, base):
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    ang = np.asarray(pos, np.float64)[:, None] * ref.rope_theta(d, base)[None, :]
    c, s = np.cos(ang), np.sin(ang)
    out = np.empty_like(x)
    out[:, 0::2] = x[:, 0::2] * c - x[:, 1::2] * s
    out[:, 1::2] = x[:, 0::2] * s + x[:, 1::2] * c
    return out


def _attend_scale_1_over_d(q_group, K, V):
    q = np.asarray(q_group, np.float64)
    s = q @ np.asarray(K, np.float64).T / q.shape[-1]
    return ref.softmax_rows(s) @ np.asarray(V, np.float64)


def _e5m2_ties_away(x):
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    q = np.where(a >= 2.0 ** -14, 2.0 ** (e - 2), 2.0 ** -16)
    y = np.minimum(np.floor(a / q + 0.5) * q, 57344.0)
    return np.copysign(y, x)


def _select_raw_logit_max(q_group, landmarks, ids, k):
    P = np.asarray(q_group) @ np.asarray(landmarks).T
    S2 = P.max(axis=0)
    ranked = ref.arg_topk(S2, k)
    return {"P": P, "S": ref.softmax_rows(P), "S2": S2, "ranked": ranked,
            "sel": np.sort(np.asarray(ids)[ranked])}


def _select_group_sum(q_group, landmarks, ids, k):
    P = np.asarray(q_group) @ np.asarray(landmarks).T
    S = ref.softmax_rows(P / math.sqrt(np.asarray(q_group).shape[-1]))
    S2 = S.sum(axis=0)
    ranked = ref.arg_topk(S2, k)
    return {"P": P, "S": S, "S2": S2, "ranked": ranked, "sel": np.sort(np.asarray(ids)[ranked])}


def _reduce_sum(K, C):
    n = K.shape[0] // C
    return K[: n * C].reshape(n, C, -1).sum(axis=1) * 1.0001


def _min_cos_max(K, L, C):
    n = L.shape[0]
    return ref.cosine(K[: n * C].reshape(n, C, -1), L[:, None, :]).max(axis=1)


def _topk_upper_ties(scores, k):
    s = np.asarray(scores, np.float64)
    return np.lexsort((-np.arange(s.shape[0]), -s))[:k]


def _prefill_no_outlier_kv(*a, **kw):
    st = _orig_prefill(*a, **kw)
    st.k_outlier = st.k_outlier[:0]
    st.v_outlier = st.v_outlier[:0]
    return st


_orig_prefill = ref.prefill_unit


def _hit_miss_swapped(prev, cur):
    h, m = _orig_hit_miss(prev, cur)
    return m, h


_orig_hit_miss = ref.hit_miss


def _prefill_ignores_exact_keys(A_b, B_bh, V_bh, C, O, W, base, K_exact=None):
    return _orig_prefill_unit(A_b, B_bh, V_bh, C, O, W, base)


_orig_prefill_unit = ref.prefill_unit


def _project_no_transpose(k_pre_b, B_b, storage=None):
    B = np.asarray(B_b, np.float64)
    H, r, d = B.shape
    return ref.round_to_storage(B.reshape(r, H * d) @ np.asarray(k_pre_b, np.float64).reshape(H * d), storage)


def _project_first_head_only(k_pre_b, B_b, storage=None):
    B = np.asarray(B_b, np.float64)
    return ref.round_to_storage(B[0] @ np.asarray(k_pre_b, np.float64)[0], storage)


def _new_key_without_rope(a, B_bh, pos, base):
    return np.asarray(a, np.float64) @ np.asarray(B_bh, np.float64)

MUTANTS = [
    ("e5m2_round", _e5m2_ties_away, [pins.test_e5m2_round_hand_values]),
    ("apply_rope", _rope_wrong_sign, [pins.test_rope_closed_form_basis_vectors]),
    ("apply_rope", _rope_interleaved, [pins.test_rope_closed_form_basis_vectors,
                                       pins.test_full_rank_full_budget_equals_dense_causal_attention]),
    ("attend", _attend_scale_1_over_d, [pins.test_full_rank_full_budget_equals_dense_causal_attention]),
    ("select_chunks", _select_raw_logit_max, [pins.test_selection_closed_form_softmax_before_group_max]),
    ("select_chunks", _select_group_sum, [pins.test_selection_closed_form_softmax_before_group_max]),
    ("reduce_chunks", _reduce_sum, [pins.test_landmarks_and_min_cos_brute_force]),
    ("chunk_min_cos", _min_cos_max, [pins.test_landmarks_and_min_cos_brute_force]),
    ("arg_topk", _topk_upper_ties, [pins.test_arg_topk_matches_brute_force_with_ties]),
    ("prefill_unit", _prefill_no_outlier_kv, [pins.test_full_rank_full_budget_equals_dense_causal_attention]),
    ("hit_miss", _hit_miss_swapped, [pins.test_hit_miss_matches_python_sets]),
    ("project_new_key", _project_no_transpose, [pins.test_plus_projection_closed_form_in_span,
                                                pins.test_plus_projection_brute_force]),
    ("project_new_key", _project_first_head_only, [pins.test_plus_projection_closed_form_in_span,
                                                   pins.test_plus_projection_brute_force]),
    ("new_token_key", _new_key_without_rope, [pins.test_plus_full_rank_equals_exact_new_keys]),
    ("prefill_unit", _prefill_ignores_exact_keys, [pins.test_exact_key_prefill_brute_force]),
]


@pytest.mark.parametrize("name,fn,tests", MUTANTS, ids=[f"{m[0]}:{m[1].__name__}" for m in MUTANTS])
def test_pins_catch_planted_mistake(monkeypatch, name, fn, tests):
    monkeypatch.setattr(ref, name, fn)
    caught = False
    for t in tests:
        try:
            if t is pins.test_arg_topk_matches_brute_force_with_ties:
                t(17, 5, 2)
            else:
                t()
        except AssertionError:
            caught = True
    assert caught, f"no pin caught the planted mistake in {name}"
