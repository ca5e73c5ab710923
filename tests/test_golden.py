"""The oracle's analytical models against the numbers the pages print
(fixtures in tests/golden/model_formulas.json, each with its citation)."""
import json
import os

import pytest

from oracle import shadowkv_ref as ref

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "model_formulas.json")))


def test_equivalent_bandwidth_worked_example():
    g = GOLD["equivalent_bandwidth"]
    i = g["inputs"]
    b = ref.equivalent_bandwidth(i["S"], i["C"], i["K"], i["O"], i["alpha"], i["B_gpu_gbs"],
                                 i["B_pcie_gbs"]) / 1000.0
    assert abs(b - g["expected_tbs"]) <= g["abs_tol"]


def test_equivalent_bandwidth_terms():
    g = GOLD["equivalent_bandwidth_terms"]
    i = g["inputs"]
    terms = ref.equivalent_bandwidth_terms(i["S"], i["C"], i["K"], i["O"], i["alpha"], i["B_ratio"], 1.0)
    for t, e in zip(terms, g["expected_terms"]):
        assert abs(t - e) <= g["abs_tol"]


def test_memory_savings_worked_example():
    g = GOLD["memory_savings"]
    i = g["inputs"]
    assert abs(ref.memory_savings(i["S"], i["M"], i["C"], i["K"], i["O"], i["r"]) - g["expected"]) <= g["abs_tol"]


def test_compression_ratio_worked_example():
    g = GOLD["compression_ratio"]
    i = g["inputs"]
    assert abs(ref.compression_ratio(i["s"], i["d"], i["r"]) - g["expected"]) <= g["abs_tol"]


def test_compression_ratio_counts_stored_elements():
    # the full key cache [s][d] against the factors A [s][r] and B [r][d], counted on real arrays
    import numpy as np
    for s, d, r in [(64, 16, 4), (100, 128, 8), (37, 5, 3)]:
        K, A, B = np.zeros((s, d)), np.zeros((s, r)), np.zeros((r, d))
        assert ref.compression_ratio(s, d, r) == pytest.approx(K.size / (A.size + B.size), rel=1e-15)


def test_sparse_budget_tokens():
    g = GOLD["sparse_budget_tokens"]
    i = g["inputs"]
    assert ref.sparse_budget_tokens(i["K"], i["O"], i["C"]) == g["expected"]


@pytest.mark.parametrize("alpha", [0.0, 0.6, 1.0])
def test_equivalent_bandwidth_limits(alpha):
    # with the link as fast as HBM and no misses the formula reduces to 2S / (S/C + 2(K+O)C)
    S, C, K, O = 131072, 8, 256, 48
    b = ref.equivalent_bandwidth(S, C, K, O, 1.0, 1.0, 1.0)
    assert abs(b - 2 * S / (S / C + 2 * (K + O) * C)) < 1e-12
    assert ref.equivalent_bandwidth(S, C, K, O, alpha, 2000.0, 31.5) <= b * 2000.0
