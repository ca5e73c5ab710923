"""Pins of the float64 oracle to things other than itself.

Each test checks the oracle against a closed form, a brute-force routine, a
library routine for a special case, an invariant, or a number the pages print
(see test_golden.py).  They are chosen so that a dropped term, a wrong sign or
index, or a transposed operand fails at least one of them.
"""
import cmath
import itertools
import math

import numpy as np
import pytest
import torch

from oracle import shadowkv_ref as ref


# --------------------------------------------------------------------- RoPE


def _rope_complex(x, pos, base):
    """Independent RoPE: pair (x_i, x_{i+d/2}) as one complex number times e^{i pos theta_i}."""
    x = np.asarray(x, np.float64)
    n, d = x.shape
    h = d // 2
    out = np.empty_like(x)
    for a in range(n):
        for i in range(h):
            th = float(base) ** (-(2.0 * i) / d)
            z = complex(x[a, i], x[a, i + h]) * cmath.exp(1j * float(pos[a]) * th)
            out[a, i], out[a, i + h] = z.real, z.imag
    return out


def test_rope_closed_form_basis_vectors():
    # d = 4, base 10000: theta = (1, 1/100).
    e = np.eye(4)
    r = ref.apply_rope(e, np.array([1, 2, 1, 3]), 10000.0)
    np.testing.assert_allclose(r[0], [math.cos(1), 0, math.sin(1), 0], atol=1e-15)
    np.testing.assert_allclose(r[1], [0, math.cos(0.02), 0, math.sin(0.02)], atol=1e-15)
    np.testing.assert_allclose(r[2], [-math.sin(1), 0, math.cos(1), 0], atol=1e-15)
    np.testing.assert_allclose(r[3], [0, -math.sin(0.03), 0, math.cos(0.03)], atol=1e-15)


def test_rope_matches_complex_form_and_invariants():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((6, 16))
    pos = np.array([0, 1, 7, 4095, 131071, 1048575])
    r = ref.apply_rope(x, pos, 500000.0)
    np.testing.assert_allclose(r, _rope_complex(x, pos, 500000.0), rtol=0, atol=1e-9)
    np.testing.assert_allclose(np.linalg.norm(r, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    np.testing.assert_array_equal(r[0], x[0])          # position 0 is the identity
    # relative-position property: <R(q,m), R(k,n)> depends on m - n only
    q, k = rng.standard_normal((1, 16)), rng.standard_normal((1, 16))
    a = (ref.apply_rope(q, np.array([900]), 1e4) @ ref.apply_rope(k, np.array([300]), 1e4).T).item()
    b = (ref.apply_rope(q, np.array([600]), 1e4) @ k.T).item()
    assert abs(a - b) < 1e-11


def test_rebuild_is_rank_exact():
    rng = np.random.default_rng(2)
    S, r, d = 24, 5, 8
    A = rng.standard_normal((S, r))
    B = rng.standard_normal((r, d))
    pos = np.arange(100, 100 + S)
    Kt = ref.rebuild_keys(A, B, pos, 500000.0)
    # undo the rotation independently, compare with a brute-force product A.B
    back = _rope_complex(Kt, -pos, 500000.0)
    brute = np.array([[sum(A[i, k] * B[k, j] for k in range(r)) for j in range(d)] for i in range(S)])
    np.testing.assert_allclose(back, brute, rtol=0, atol=1e-12)


# --------------------------------------------------------------- selection


def _brute_topk(s, k):
    return sorted(range(len(s)), key=lambda j: (-s[j], j))[:k]


@pytest.mark.parametrize("n,k,levels", [(1, 1, 3), (17, 5, 2), (64, 64, 4), (300, 16, 5),
                                        (512, 200, 50), (512, 1, 1)])
def test_arg_topk_matches_brute_force_with_ties(n, k, levels):
    rng = np.random.default_rng(n * 31 + k)
    s = rng.integers(0, levels, n).astype(np.float64) * 0.25   # many exact ties
    assert list(ref.arg_topk(s, k)) == _brute_topk(list(s), k)
    s2 = rng.standard_normal(n)
    assert list(ref.arg_topk(s2, k)) == _brute_topk(list(s2), k)


def test_selection_closed_form_softmax_before_group_max():
    # d = 16 so the scale is 1/4.  Landmarks are unit basis vectors so P is exact.
    d = 16
    L = np.eye(d)[:3]
    ids = np.array([10, 11, 12])
    q = np.zeros((2, d))
    q[0, 0] = 8.0                  # head 0 logits (8, 0, 0)
    q[1, 1], q[1, 2] = 12.0, 11.6  # head 1 logits (0, 12, 11.6)
    res = ref.select_chunks(q, L, ids, 1)
    e = math.exp
    s00 = e(2.0) / (e(2.0) + 2.0)
    s11 = e(3.0) / (1.0 + e(3.0) + e(2.9))
    s12 = e(2.9) / (1.0 + e(3.0) + e(2.9))
    np.testing.assert_allclose(res["S2"], [s00, s11, s12], rtol=1e-14)
    # the largest raw logit (chunk 11) is not the top chunk once each head is normalised
    assert list(res["sel"]) == [10]
    assert list(ref.select_chunks(q, L, ids, 2)["sel"]) == [10, 11]
    np.testing.assert_allclose(res["S"].sum(axis=1), 1.0, rtol=1e-15)


def test_group_max_and_softmax_rows():
    rng = np.random.default_rng(3)
    G, n, d = 4, 257, 32
    q = rng.standard_normal((G, d))
    L = rng.standard_normal((n, d))
    res = ref.select_chunks(q, L, np.arange(n) * 3 + 1, 9)
    np.testing.assert_allclose(res["S"].sum(axis=1), 1.0, rtol=1e-13)
    brute = [max(res["S"][g][j] for g in range(G)) for j in range(n)]
    np.testing.assert_array_equal(res["S2"], brute)
    assert list(res["sel"]) == sorted(3 * j + 1 for j in _brute_topk(brute, 9))


# --------------------------------------------------------------- prefill


def test_landmarks_and_min_cos_brute_force():
    rng = np.random.default_rng(4)
    C, n, d = 4, 5, 6
    K = rng.standard_normal((n * C, d))
    L = ref.reduce_chunks(K, C)
    m = ref.chunk_min_cos(K, L, C)
    for j in range(n):
        mean = [sum(K[j * C + i][t] for i in range(C)) / C for t in range(d)]
        np.testing.assert_allclose(L[j], mean, rtol=1e-14)
        cs = []
        for i in range(C):
            x = K[j * C + i]
            cs.append(sum(x[t] * mean[t] for t in range(d)) /
                      (math.sqrt(sum(v * v for v in x)) * math.sqrt(sum(v * v for v in mean))))
        assert abs(m[j] - min(cs)) < 1e-13


def test_min_cos_closed_forms():
    v = np.array([3.0, 4.0, 0.0])
    K = np.stack([v, v, v, v, v, v, v, -v])        # mean = 0.75 v
    L = ref.reduce_chunks(K, 8)
    np.testing.assert_allclose(L[0], 0.75 * v)
    assert abs(ref.chunk_min_cos(K, L, 8)[0] - (-1.0)) < 1e-15
    K2 = np.stack([v] * 8)
    assert abs(ref.chunk_min_cos(K2, ref.reduce_chunks(K2, 8), 8)[0] - 1.0) < 1e-15


def test_prefill_counts_and_planted_outliers():
    from workload import TINY, make_A, make_B, make_V, spike_chunks
    w = TINY
    A, B, V = make_A(w, 0), make_B(w, 0), make_V(w, 0)
    pre = ref.prefill_unit(A[0].double().numpy(), B[0, 1].double().numpy(),
                           V[0, 1].double().numpy(), w.chunk, w.n_outlier, w.local_window,
                           w.rope_base)
    # chunk-count invariant O + n_c + W/C = S/C
    assert len(pre.outlier_ids) + len(pre.ids) + w.local_window // w.chunk == w.n_chunks
    assert len(pre.ids) == w.n_selectable
    assert np.all(np.diff(pre.ids) > 0) and np.all(np.diff(pre.outlier_ids) > 0)
    assert not set(pre.ids) & set(pre.outlier_ids)
    assert max(pre.ids) < w.n_chunks - w.local_window // w.chunk
    # planted spike chunks (scale 8, odd offsets replaced) are the outliers
    assert set(spike_chunks(w, 0)[0].tolist()) == set(pre.outlier_ids.tolist())
    # outliers are exactly the lowest min-cos candidates
    brute = _brute_topk(list(-pre.min_cos), w.n_outlier)
    assert sorted(brute) == list(pre.outlier_ids)


# --------------------------------------------------------------- decode


def test_hit_miss_matches_python_sets():
    rng = np.random.default_rng(5)
    prev = None
    for _ in range(6):
        cur = np.sort(rng.choice(40, 12, replace=False))
        hits, misses = ref.hit_miss(prev, cur)
        if prev is None:
            assert hits.size == 0 and list(misses) == list(cur)
        else:
            assert list(hits) == sorted(set(prev.tolist()) & set(cur.tolist()))
            assert list(misses) == sorted(set(cur.tolist()) - set(prev.tolist()))
        prev = cur


def _dense_case(seed=6, S=256, C=8, W=16, O=3, H=2, G=4, d=16, steps=4):
    """Full rank r = H*d (A holds the raw keys, B_h selects head h) and K = n_c:
    the step must equal dense causal attention over all tokens."""
    rng = np.random.default_rng(seed)
    r = H * d
    keys = rng.standard_normal((H, S, d))
    A = np.concatenate([keys[h] for h in range(H)], axis=1)          # [S][H*d]
    Bs = [np.eye(r)[:, h * d:(h + 1) * d] for h in range(H)]          # [r][d] selectors
    V = rng.standard_normal((H, S, d))
    n_c = S // C - O - W // C
    qs = rng.standard_normal((steps, H * G, d))
    kn = rng.standard_normal((steps, H, d))
    vn = rng.standard_normal((steps, H, d))
    return dict(rng=rng, S=S, C=C, W=W, O=O, H=H, G=G, d=d, r=r, keys=keys, A=A, Bs=Bs, V=V,
                n_c=n_c, qs=qs, kn=kn, vn=vn, steps=steps)


def test_full_rank_full_budget_equals_dense_causal_attention():
    c = _dense_case()
    base = 500000.0
    for h in range(c["H"]):
        st = ref.UnitDecodeState(ref.prefill_unit(c["A"], c["Bs"][h], c["V"][h], c["C"], c["O"],
                                                  c["W"], base))
        krot = _rope_complex(c["keys"][h], np.arange(c["S"]), base)   # independent RoPE
        Kall, Vall = list(krot), list(c["V"][h])
        for t in range(c["steps"]):
            qg = c["qs"][t, h * c["G"]:(h + 1) * c["G"]]                # q-head j -> KV head j // G
            res = ref.decode_step_unit(st, qg, c["kn"][t, h], c["vn"][t, h], c["A"], c["Bs"][h],
                                       c["V"][h], c["n_c"], c["C"], base)
            Kall.append(c["kn"][t, h])
            Vall.append(c["vn"][t, h])
            Kt = torch.tensor(np.stack(Kall))[None, None]
            Vt = torch.tensor(np.stack(Vall))[None, None]
            qt = torch.tensor(qg)[None, :, None, :]
            dense = torch.nn.functional.scaled_dot_product_attention(
                qt, Kt.expand(1, c["G"], -1, -1), Vt.expand(1, c["G"], -1, -1))[0, :, 0, :].numpy()
            np.testing.assert_allclose(res["out"], dense, rtol=0, atol=1e-12)
            assert len(res["sel"]) == c["n_c"]
            if t >= 1:
                assert len(res["misses"]) == 0          # everything selected: all hits


def test_attend_on_index_set_matches_decode_step():
    c = _dense_case(seed=7, steps=2)
    base, h = 500000.0, 1
    K = 5
    st = ref.UnitDecodeState(ref.prefill_unit(c["A"], c["Bs"][h], c["V"][h], c["C"], c["O"],
                                              c["W"], base))
    for t in range(2):
        qg = c["qs"][t, h * c["G"]:(h + 1) * c["G"]]
        res = ref.decode_step_unit(st, qg, c["kn"][t, h], c["vn"][t, h], c["A"], c["Bs"][h],
                                   c["V"][h], K, c["C"], base)
        again = ref.attend_on_index_set(qg, c["A"], c["Bs"][h], c["V"][h], st.pre.outlier_ids,
                                        res["sel"], st.pre.k_local, st.pre.v_local, c["C"], base)
        np.testing.assert_allclose(again, res["out"], rtol=0, atol=1e-13)


def test_repeated_query_hits_everything_after_first_step():
    c = _dense_case(seed=8, steps=3)
    base, h = 500000.0, 0
    st = ref.UnitDecodeState(ref.prefill_unit(c["A"], c["Bs"][h], c["V"][h], c["C"], c["O"],
                                              c["W"], base))
    qg = c["qs"][0, :c["G"]]
    for t in range(3):
        res = ref.decode_step_unit(st, qg, c["kn"][t, h], c["vn"][t, h], c["A"], c["Bs"][h],
                                   c["V"][h], 6, c["C"], base)
        if t == 0:
            assert len(res["misses"]) == 6
        else:
            assert len(res["hits"]) == 6 and len(res["misses"]) == 0


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(9)
    x = np.concatenate([rng.standard_normal(5000) * 10.0 ** rng.integers(-8, 8, 5000),
                        [0.0, -0.0, 1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9]])
    want = torch.tensor(x.astype(np.float32)).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(ref.bf16_round(x), want)


def test_near_tie_band():
    s = np.array([1.0, 0.5, 0.50004, 0.2, 0.49999])
    band, kth = ref.near_tie_band(s, 2, 1e-4)
    assert kth == 0.50004 and set(band.tolist()) == {1, 2, 4}


def test_storage_rounding_of_kept_keys():
    c = _dense_case(seed=10, steps=1)
    h, base = 0, 500000.0
    st = ref.UnitDecodeState(ref.prefill_unit(c["A"], c["Bs"][h], c["V"][h], c["C"], c["O"], c["W"], base))
    qg = c["qs"][0, :c["G"]]
    kl = list(st.pre.k_local) + [c["kn"][0, h]]
    vl = list(st.pre.v_local) + [c["vn"][0, h]]
    sel = np.arange(5)
    a = ref.attend_on_index_set(qg, c["A"], c["Bs"][h], c["V"][h], st.pre.outlier_ids, sel, kl, vl, c["C"], base)
    b = ref.attend_on_index_set(qg, c["A"], c["Bs"][h], c["V"][h], st.pre.outlier_ids, sel, kl, vl, c["C"], base,
                                storage="f32")
    d = ref.attend_on_index_set(qg, c["A"], c["Bs"][h], c["V"][h], st.pre.outlier_ids, sel, kl, vl, c["C"], base,
                                storage="bf16")
    assert 0 < np.max(np.abs(a - b)) < 1e-5 < np.max(np.abs(a - d)) < 0.1
    x = np.array([1.0 + 2 ** -9, 3.0, -2.0 ** -130])
    np.testing.assert_array_equal(ref.round_to_storage(x, "bf16"), ref.bf16_round(x))


# e5m2: 1 sign bit, 5 exponent bits (bias 15), 2 mantissa bits.  Values worked out by hand from
# that definition: spacing 2^(e-2) in [2^e, 2^(e+1)), 2^-16 below 2^-14, ties to the even
# mantissa, the largest finite value 1.75 * 2^15 = 57344.
E5M2_CASES = [
    (1.0, 1.0), (1.1, 1.0), (1.125, 1.0),        # tie between mantissas 00 and 01 -> 00
    (1.375, 1.5),                                # tie between 01 and 10 -> 10
    (1.4, 1.5), (1.74, 1.75), (1.9, 2.0),
    (3.3, 3.5), (-0.3, -0.3125),                 # [0.25, 0.5) spacing 1/16
    (57344.0, 57344.0), (60000.0, 57344.0),      # saturation at the largest finite value
    (2.0 ** -14, 2.0 ** -14),                    # smallest normal
    (2.0 ** -16, 2.0 ** -16),                    # smallest subnormal
    (2.0 ** -17, 0.0),                           # tie between 0 and 2^-16 -> 0 (even)
    (3 * 2.0 ** -17, 2.0 ** -15),                # tie between 1 and 2 subnormal steps -> 2
    (0.0, 0.0),
]


def test_e5m2_round_hand_values():
    got = ref.e5m2_round(np.array([x for x, _ in E5M2_CASES]))
    for (x, want), g in zip(E5M2_CASES, got):
        assert g == want, (x, want, g)


def test_e5m2_grid_is_closed_and_monotone():
    # every value of the grid between 2^-16 and 57344 rounds to itself, and rounding is monotone
    grid = [0.0] + [k * 2.0 ** -16 for k in range(1, 4)]
    for e in range(-14, 16):
        grid += [(1 + m / 4) * 2.0 ** e for m in range(4)]
    grid = np.array(sorted(set(grid)))
    np.testing.assert_array_equal(ref.e5m2_round(grid), grid)
    np.testing.assert_array_equal(ref.e5m2_round(-grid), -grid)
    x = np.sort(np.random.default_rng(3).uniform(-60000, 60000, 20000))
    assert np.all(np.diff(ref.e5m2_round(x)) >= 0)
    assert len(grid) == 1 + 3 + 30 * 4   # zero, 3 subnormals, 30 binades of 4: all finite e5m2 >= 0


def test_e5m2_round_agrees_with_torch_in_range():
    rng = np.random.default_rng(4)
    x = rng.standard_normal(20000) * 10.0 ** rng.integers(-4, 4, 20000)
    x = x[np.abs(x) < 57000]
    want = torch.tensor(x.astype(np.float32)).to(torch.float8_e5m2).double().numpy()
    np.testing.assert_array_equal(ref.e5m2_round(x.astype(np.float32).astype(np.float64)), want)


def test_bf16_is_three_e5m2_terms():
    # The fp8 scorer feeds the bf16 query to an e5m2 tensor-core product as three e5m2 terms
    # t1 = e5m2(q), t2 = e5m2(q - t1), t3 = e5m2(q - t1 - t2): each term holds the next three
    # significant bits, so the sum is q exactly when the last residual is still a multiple of
    # e5m2's smallest step, i.e. for 2^-9 <= |q| <= 57344.
    rng = np.random.default_rng(5)
    q = ref.bf16_round(rng.standard_normal(50000) * 2.0 ** rng.integers(-6, 8, 50000))
    q = q[(np.abs(q) >= 2.0 ** -9) & (np.abs(q) <= 57344)]
    t1 = ref.e5m2_round(q)
    t2 = ref.e5m2_round(q - t1)
    t3 = ref.e5m2_round(q - t1 - t2)
    np.testing.assert_array_equal(t1 + t2 + t3, q)
    # Hence the scorer scales each head's query by 2^s, the largest power of two with
    # max|q| * 2^s <= 2^14, before splitting: every component down to max|q| * 2^-22 is exact,
    # and a smaller one is off by less than 2^-16 * 2^-s.
    for _ in range(200):
        v = ref.bf16_round(rng.standard_normal(128) * 2.0 ** rng.integers(-20, 10))
        sc = 2.0 ** np.floor(np.log2(2.0 ** 14 / np.max(np.abs(v))))
        x = v * sc
        t1 = ref.e5m2_round(x)
        t2 = ref.e5m2_round(x - t1)
        t3 = ref.e5m2_round(x - t1 - t2)
        err = np.abs((t1 + t2 + t3) - x)
        big = np.abs(v) >= np.max(np.abs(v)) * 2.0 ** -22
        assert np.all(err[big] == 0) and np.all(err < 2.0 ** -16)


def test_fp8_storage_readings():
    assert ref.key_storage("fp8") == "bf16" and ref.value_storage("fp8") == "e5m2"
    assert ref.key_storage("bf16") == "bf16" and ref.value_storage("bf16") == "bf16"
    x = np.array([1.1, -0.3, 2.0 ** -17])
    np.testing.assert_array_equal(ref.round_to_storage(x, "e5m2"), [1.0, -0.3125, 0.0])


# --------------------------------------------------------------------- ShadowKV+ (generated keys at rank r)


def _orthonormal_basis(rng, n, r):
    """[n][r] with orthonormal columns."""
    q, _ = np.linalg.qr(rng.standard_normal((n, r)))
    return q


def _B_from_basis(Q, H, d):
    """B_b [H][r][d] whose [r][H*d] reading is Q^T (Psi = Q)."""
    return np.stack([Q[h * d:(h + 1) * d, :].T for h in range(H)])


def test_plus_projection_closed_form_in_span():
    rng = np.random.default_rng(31)
    H, d, r = 3, 8, 5
    Q = _orthonormal_basis(rng, H * d, r)
    B = _B_from_basis(Q, H, d)
    c = rng.standard_normal(r)
    k = (Q @ c).reshape(H, d)                       # a key inside the context's subspace
    a = ref.project_new_key(k, B)
    np.testing.assert_allclose(a, c, rtol=0, atol=1e-12)
    for h in range(H):                              # position 0: RoPE is the identity
        np.testing.assert_allclose(ref.new_token_key(a, B[h], 0, 10000.0), k[h], rtol=0, atol=1e-12)


def test_plus_projection_drops_the_orthogonal_part():
    rng = np.random.default_rng(32)
    H, d, r = 2, 8, 3
    Q = _orthonormal_basis(rng, H * d, r)
    B = _B_from_basis(Q, H, d)
    c = rng.standard_normal(r)
    g = rng.standard_normal(H * d)
    z = g - Q @ (Q.T @ g)                           # orthogonal to the subspace
    a = ref.project_new_key((Q @ c + z).reshape(H, d), B)
    np.testing.assert_allclose(a, c, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ref.project_new_key(z.reshape(H, d), B), 0.0, rtol=0, atol=1e-12)


def test_plus_projection_brute_force():
    rng = np.random.default_rng(33)
    H, r, d = 3, 5, 4
    B = rng.standard_normal((H, r, d))              # any basis: the definition is the plain sum
    k = rng.standard_normal((H, d))
    want = np.zeros(r)
    for j in range(r):
        for h in range(H):
            for i in range(d):
                want[j] += k[h, i] * B[h, j, i]
    np.testing.assert_allclose(ref.project_new_key(k, B), want, rtol=0, atol=1e-12)
    # stored in bf16 like the context rows of A
    np.testing.assert_array_equal(ref.project_new_key(k, B, "bf16"), ref.bf16_round(want))


def test_plus_full_rank_equals_exact_new_keys():
    """With r = H*d and an orthogonal basis the projection loses nothing, so
    ShadowKV+ must give the same outputs as ShadowKV fed the exact post-RoPE
    new keys."""
    c = _dense_case(seed=34, steps=3)
    H, d, r, S, base = c["H"], c["d"], c["r"], c["S"], 500000.0
    rng = np.random.default_rng(35)
    Q = _orthonormal_basis(rng, r, r)               # square: orthogonal
    B = _B_from_basis(Q, H, d)                      # [H][r][d]
    A = np.concatenate([c["keys"][h] for h in range(H)], axis=1) @ Q   # A.B_h = keys_h
    kpre = c["kn"]                                  # [T][H][d], pre-RoPE in this case
    for h in range(H):
        st_exact = ref.UnitDecodeState(ref.prefill_unit(A, B[h], c["V"][h], c["C"], c["O"], c["W"], base))
        st_plus = ref.UnitDecodeState(ref.prefill_unit(A, B[h], c["V"][h], c["C"], c["O"], c["W"], base))
        for t in range(c["steps"]):
            qg = c["qs"][t, h * c["G"]:(h + 1) * c["G"]]
            k_exact = _rope_complex(kpre[t, h][None, :], np.array([S + t]), base)[0]
            k_plus = ref.new_token_key(ref.project_new_key(kpre[t], B), B[h], S + t, base)
            r1 = ref.decode_step_unit(st_exact, qg, k_exact, c["vn"][t, h], A, B[h], c["V"][h], 6, c["C"], base)
            r2 = ref.decode_step_unit(st_plus, qg, k_plus, c["vn"][t, h], A, B[h], c["V"][h], 6, c["C"], base)
            assert np.array_equal(r1["sel"], r2["sel"])
            np.testing.assert_allclose(r2["out"], r1["out"], rtol=0, atol=1e-11)


# --------------------------------------------------------------------- exact-key pre-filling


def test_exact_key_prefill_brute_force():
    """Landmarks, min-cos, outliers and kept keys come from RoPE(K_exact), not A.B:
    checked against loops with an independent RoPE on keys unrelated to the factors."""
    rng = np.random.default_rng(51)
    S, C, W, O, d, r, base = 64, 8, 8, 2, 8, 4, 10000.0
    K = rng.standard_normal((S, d))
    K[3 * C + 1] *= 9.0                                  # one token far from its chunk mean
    A = rng.standard_normal((S, r))
    B = rng.standard_normal((r, d))
    V = rng.standard_normal((S, d))
    pre = ref.prefill_unit(A, B, V, C, O, W, base, K_exact=K)
    Kr = _rope_complex(K, np.arange(S), base)
    n_cand = S // C - W // C
    mc = np.empty(n_cand)
    for c in range(n_cand):
        mean = Kr[c * C:(c + 1) * C].mean(axis=0)
        np.testing.assert_allclose(pre.all_landmarks[c], mean, rtol=0, atol=1e-12)
        mc[c] = min(float(Kr[i] @ mean) / max(np.linalg.norm(Kr[i]) * np.linalg.norm(mean), 1e-12)
                    for i in range(c * C, (c + 1) * C))
    np.testing.assert_allclose(pre.min_cos, mc, rtol=0, atol=1e-12)
    want_out = sorted(sorted(range(n_cand), key=lambda c: (mc[c], c))[:O])
    assert list(pre.outlier_ids) == want_out and 3 in want_out
    tok = ref.chunk_tokens(pre.outlier_ids, C)
    np.testing.assert_allclose(pre.k_outlier, Kr[tok], rtol=0, atol=1e-12)
    np.testing.assert_allclose(np.stack(pre.k_local), Kr[S - W:], rtol=0, atol=1e-12)


def test_exact_keys_equal_to_the_factors_change_nothing():
    c = _dense_case(seed=52, steps=1)
    base, h = 500000.0, 1
    a = ref.prefill_unit(c["A"], c["Bs"][h], c["V"][h], c["C"], c["O"], c["W"], base)
    b = ref.prefill_unit(c["A"], c["Bs"][h], c["V"][h], c["C"], c["O"], c["W"], base,
                         K_exact=c["A"] @ c["Bs"][h])
    np.testing.assert_allclose(b.all_landmarks, a.all_landmarks, rtol=0, atol=1e-12)
    assert np.array_equal(a.outlier_ids, b.outlier_ids)


def test_attend_with_exact_outlier_keys_matches_decode_step():
    rng = np.random.default_rng(53)
    c = _dense_case(seed=53, steps=2)
    base, h, K = 500000.0, 0, 5
    Kx = c["A"] @ c["Bs"][h] + 0.3 * rng.standard_normal((c["S"], c["d"]))
    st = ref.UnitDecodeState(ref.prefill_unit(c["A"], c["Bs"][h], c["V"][h], c["C"], c["O"], c["W"], base,
                                              K_exact=Kx))
    for t in range(2):
        qg = c["qs"][t, h * c["G"]:(h + 1) * c["G"]]
        res = ref.decode_step_unit(st, qg, c["kn"][t, h], c["vn"][t, h], c["A"], c["Bs"][h],
                                   c["V"][h], K, c["C"], base)
        again = ref.attend_on_index_set(qg, c["A"], c["Bs"][h], c["V"][h], st.pre.outlier_ids,
                                        res["sel"], st.pre.k_local, st.pre.v_local, c["C"], base,
                                        k_outlier=st.pre.k_outlier)
        np.testing.assert_allclose(again, res["out"], rtol=0, atol=1e-13)
