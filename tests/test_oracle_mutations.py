"""Plant plausible mistakes in the oracle (CPU only) and check that the pins catch each."""
import math

import numpy as np
import pytest

from oracle import shadowkv_ref as ref
from tests import test_golden as golden
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


def _rebuild_rope_one_late(A_rows, B_h, pos, base):
    return ref.apply_rope(np.asarray(A_rows, np.float64) @ np.asarray(B_h, np.float64), np.asarray(pos) + 1, base)


def _softmax_over_columns(x):
    m = x.max(axis=0, keepdims=True)
    e = np.exp(x - m)
    return e / e.sum(axis=0, keepdims=True)


def _bf16_truncate(x):
    f = np.asarray(x, np.float64).astype(np.float32)
    return (f.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)


def _decode_without_append(st, q_group, k_new, v_new, A_b, B_bh, V_bh, k, C, base):
    sel = ref.select_chunks(q_group, st.pre.landmarks, st.pre.ids, k)
    hits, misses = ref.hit_miss(st.prev_sel, sel["sel"])
    A_b = np.asarray(A_b, np.float64)
    V_bh = np.asarray(V_bh, np.float64)
    ts = ref.chunk_tokens(sel["sel"], C)
    K = np.concatenate([st.pre.k_outlier, ref.rebuild_keys(A_b[ts], B_bh, ts, base), np.stack(st.pre.k_local)])
    V = np.concatenate([st.pre.v_outlier, V_bh[ts], np.stack(st.pre.v_local)])
    out = ref.attend(q_group, K, V)
    st.prev_sel = sel["sel"]
    st.steps += 1
    return {"out": out, "sel": sel["sel"], "S2": sel["S2"], "ranked": sel["ranked"], "hits": hits, "misses": misses}


def _attend_index_set_without_local(q_group, A_b, B_bh, V_bh, outlier_ids, sel_ids, k_local, v_local, C, base,
                                    **kw):
    return _orig_attend_on_index_set(q_group, A_b, B_bh, V_bh, outlier_ids, sel_ids, [], [], C, base, **kw)


_orig_attend_on_index_set = ref.attend_on_index_set


def _eqbw_all_misses(S, C, K, O, alpha, B_gpu, B_pcie):
    return 2.0 * S * B_gpu / (S / C + 2.0 * (K + O) * C + K * C * B_gpu / B_pcie)


def _eqbw_terms_single_kv(S, C, K, O, alpha, B_gpu, B_pcie):
    return (S / C, (K + O) * C, (1.0 - alpha) * K * C * B_gpu / B_pcie)


def _memory_savings_one_cache(S, M, C, K, O, r):
    return S * M / (S * M / C + 2.0 * (K + O) * C + S * r + r * M)


def _theta_without_two(d, base):
    i = np.arange(d // 2, dtype=np.float64)
    return np.power(float(base), -i / d)


def _cosine_one_norm(x, y):
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    return (x * y).sum(axis=-1) / np.maximum((x * x).sum(axis=-1), 1e-12)


def _values_like_keys(dtype):
    return "bf16" if dtype == "fp8" else dtype


def _compression_without_d(s, d, r):
    return s * d / (r * s)


def _budget_without_outliers(K, O, C):
    return K * C


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
    ("rebuild_keys", _rebuild_rope_one_late, [pins.test_rebuild_is_rank_exact]),
    ("softmax_rows", _softmax_over_columns, [pins.test_group_max_and_softmax_rows]),
    ("bf16_round", _bf16_truncate, [pins.test_bf16_round_matches_torch]),
    ("decode_step_unit", _decode_without_append, [pins.test_full_rank_full_budget_equals_dense_causal_attention]),
    ("attend_on_index_set", _attend_index_set_without_local, [pins.test_attend_on_index_set_matches_decode_step]),
    ("equivalent_bandwidth", _eqbw_all_misses, [golden.test_equivalent_bandwidth_worked_example]),
    ("equivalent_bandwidth_terms", _eqbw_terms_single_kv, [golden.test_equivalent_bandwidth_terms]),
    ("memory_savings", _memory_savings_one_cache, [golden.test_memory_savings_worked_example]),
    ("sparse_budget_tokens", _budget_without_outliers, [golden.test_sparse_budget_tokens]),
    ("rope_theta", _theta_without_two, [pins.test_rope_closed_form_basis_vectors]),
    ("cosine", _cosine_one_norm, [pins.test_min_cos_closed_forms]),
    ("value_storage", _values_like_keys, [pins.test_fp8_storage_readings]),
    ("compression_ratio", _compression_without_d, [golden.test_compression_ratio_worked_example,
                                                   golden.test_compression_ratio_counts_stored_elements]),
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
