"""Pins of the oracle's batched sampler ("Engine 与采样器" 采样器 and 测试;
"Mini-SGLang 源码解析（四）" 14; "Mini-SGLang 完整剖析" 4.8.5).

The printed worked values (tests/golden/sampler_pages.json), the library
softmax, a pairwise brute-force statement of the filter that shares no step
with the oracle's sort-and-cumsum, and closed forms fix every step: the
temperature, the sort direction and tie order, the top-k cut, the
renormalisation before top-p, the top-p rule and the direction of the
inverse-CDF draw."""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sampler_pages.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


# ----------------------------------------------------------- Sampler.prepare
def test_prepare_all_greedy_gives_no_temperatures():
    g = _golden()["engine_test"]
    assert g["all_greedy_gives_no_temperatures"]
    assert oracle.sampling_args([0.0, 0.0], [-1, -1], [1.0, 1.0], 6) == (None, None, None)


def test_prepare_clamps_and_sparse_arguments():
    c = _golden()["clamps"]
    assert oracle.SAMPLE_MIN_T == c["min_temperature"] and oracle.SAMPLE_MIN_P == c["min_top_p"]
    t, k, p = oracle.sampling_args([0.7, 0.0, 2.0], [-1, 0, -5], [1.0, 3.0, 1.0], 100)
    assert np.allclose(t, [0.7, 1e-6, 2.0]) and t.dtype == np.float32
    assert k is None and p is None                    # nobody restricts: no tensors
    t, k, p = oracle.sampling_args([1.0, 1.0], [50, -1], [0.0, 0.95], 100)
    assert k.tolist() == [50, 100] and k.dtype == np.int32
    assert p.dtype == np.float32 and np.allclose(p, [1e-6, 0.95])


def test_is_greedy_follows_the_pages_rule():
    # the printed property: (temperature <= 0 or top_k == 1) and top_p == 1
    for c in _golden()["greedy_rule"]["cases"]:
        assert oracle.is_greedy(c["temperature"], c["top_k"], c["top_p"]) is c["greedy"], c


def test_prepare_temperature_zero_with_top_p_is_sampled():
    # every temperature is 0, but one request has top_p < 1: it is not greedy,
    # so the batch takes the sampled branch (temperatures present), that
    # request at MIN_T, and the top-p tensor exists
    t, k, p = oracle.sampling_args([0.0, 0.0], [-1, -1], [1.0, 0.9], 100)
    assert t is not None and np.allclose(t, [1e-6, 1e-6])
    assert k is None and np.allclose(p, [1.0, 0.9])


def test_prepare_top_k_one_is_greedy():
    # temperature > 0 with top_k == 1 and top_p == 1 is greedy: a batch of such
    # requests takes the argmax, and in a mixed batch it gets MIN_T
    assert oracle.sampling_args([0.8, 1.5], [1, 1], [1.0, 1.0], 100) == (None, None, None)
    t, k, p = oracle.sampling_args([0.8, 1.5], [1, 3], [1.0, 1.0], 100)
    assert np.allclose(t, [1e-6, 1.5]) and k.tolist() == [1, 3] and p is None


# --------------------------------------------------------- printed examples
def test_engine_test_case_support_and_frequency():
    g = _golden()["engine_test"]
    V = g["vocab_size"]
    L = np.array([g["logits"]] * 3)
    reqs = g["requests"]
    t, k, p = oracle.sampling_args([r["temperature"] for r in reqs], [r["top_k"] for r in reqs],
                                   [r["top_p"] for r in reqs], V)
    u = np.random.default_rng(0).random((g["draws"], 3)).astype(np.float32)
    draws = np.stack([oracle.sample(L, t, k, p, u[i]) for i in range(g["draws"])])
    for row, support in enumerate(g["support"]):
        assert set(draws[:, row].tolist()) == set(support)
    freq = float((draws[:, 0] == 0).mean())
    assert abs(freq - g["first_token_frequency_row0"]) < g["frequency_tolerance"]
    # the exact kept distribution of row 0: e^5 / (e^5 + e^4) = 1 / (1 + e^-1)
    q, _ = oracle.sample_filter(L[0], 1.0, 2, None)
    assert abs(q[0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-12
    assert abs(q[0] - g["first_token_frequency_row0"]) < 5e-4
    assert q[2:].sum() == 0.0


def test_top_k_printed_example():
    g = _golden()["top_k_example"]
    q, _ = oracle.sample_filter(np.log(g["probs"]), 1.0, g["top_k"], None)
    assert np.round(q, g["decimals"]).tolist() == g["normalized"]


def test_top_p_printed_example():
    g = _golden()["top_p_example"]
    q, _ = oracle.sample_filter(np.log(g["probs"]), 1.0, None, g["top_p"])
    assert np.nonzero(q)[0].tolist() == g["kept"]


def test_top_p_sees_the_top_k_renormalised_mass():
    # logits of the engine test: after top-k = 2 the first token holds 0.731 of
    # the mass, so top-p = 0.7 keeps it alone; on the unrenormalised softmax it
    # holds 0.656 and the second token would survive
    L = np.array([5.0, 4.0, 3.0, 0.0, 0.0, 0.0])
    q, _ = oracle.sample_filter(L, 1.0, 2, 0.7)
    assert np.nonzero(q)[0].tolist() == [0]
    q, _ = oracle.sample_filter(L, 1.0, None, 0.7)
    assert np.nonzero(q)[0].tolist() == [0, 1]


# ------------------------------------------------------------- closed forms
def test_no_cut_is_the_library_softmax():
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(1)
    for T in (0.3, 1.0, 2.5):
        L = rng.normal(0, 3, 40).astype(np.float32)
        q, _ = oracle.sample_filter(L, T, None, None)
        ref = scipy_special.softmax(L.astype(np.float64) / float(np.float32(T)))
        assert np.allclose(q, ref, rtol=1e-12, atol=1e-15)
        q2, _ = oracle.sample_filter(L, T, len(L), 1.0)   # k = V and p = 1 cut nothing
        assert np.array_equal(q, q2)


def test_inverse_cdf_covers_each_token_with_its_mass():
    # a fine grid of uniforms lands on token i for a fraction q_i of the grid
    q = np.array([0.1, 0.0, 0.25, 0.4, 0.0, 0.25])
    n = 200000
    grid = (np.arange(n) + 0.5) / n
    toks = np.array([oracle.inverse_cdf(q, u) for u in grid[::10]])
    freq = np.bincount(toks, minlength=len(q)) / len(toks)
    assert np.allclose(freq, q, atol=1e-4)
    # direction: small uniforms take the low indices
    assert oracle.inverse_cdf(q, 0.0) == 0 and oracle.inverse_cdf(q, 0.0999) == 0
    assert oracle.inverse_cdf(q, 0.1001) == 2 and oracle.inverse_cdf(q, 0.9999) == 5


def test_cut_to_one_token_is_the_argmax():
    rng = np.random.default_rng(2)
    for _ in range(20):
        L = rng.normal(0, 2, 64)
        L[rng.integers(0, 64, 3)] = L.max()               # tied maxima
        first = int(np.argmax(L))
        for k, p in ((1, None), (None, 1e-6), (1, 0.5)):
            q, _ = oracle.sample_filter(L, 0.8, k, p)
            assert np.nonzero(q)[0].tolist() == [first]
        assert oracle.sample(L[None], None, None, None, None)[0] == first


def test_temperature_scale_identity():
    # logits * 2 at temperature T * 2 is the same distribution (exact in binary)
    rng = np.random.default_rng(3)
    L = rng.normal(0, 2, 300).astype(np.float32)
    for k, p in ((None, None), (17, None), (None, 0.8), (40, 0.9)):
        a, _ = oracle.sample_filter(L, 0.75, k, p)
        b, _ = oracle.sample_filter(L * np.float32(2), 1.5, k, p)
        assert np.array_equal(a, b)


def test_tiny_temperature_is_greedy_for_separated_maxima():
    # the mixed-batch greedy request (temperature MIN_T): a one-hot distribution
    rng = np.random.default_rng(4)
    L = rng.normal(0, 1, 1000)
    q, _ = oracle.sample_filter(L, 0.0, None, None)
    assert q[int(np.argmax(L))] == 1.0


# --------------------------------------------------- pairwise brute force
def _brute_kept(p, k, P):
    """Kept set by pairwise comparisons: j beats i if p_j > p_i, or p_j == p_i
    and j < i; i survives top-k if fewer than k tokens beat it, and top-p if
    the top-k survivors that beat it hold less than P of the top-k mass."""
    V = len(p)
    beats = [[(p[j] > p[i]) or (p[j] == p[i] and j < i) for j in range(V)] for i in range(V)]
    kk = V if k is None or k < 1 or k >= V else k
    in_k = [sum(beats[i]) < kk for i in range(V)]
    mass_k = sum(p[i] for i in range(V) if in_k[i])
    kept = []
    for i in range(V):
        if not in_k[i]:
            continue
        if P is not None:
            ahead = sum(p[j] for j in range(V) if in_k[j] and beats[i][j])
            if not ahead < P * mass_k:
                continue
        kept.append(i)
    return kept


def test_filter_matches_pairwise_brute_force():
    rng = np.random.default_rng(5)
    checked = 0
    for trial in range(400):
        V = int(rng.integers(2, 13))
        L = rng.normal(0, 1.5, V)
        if trial % 4 == 0:                                  # exact ties
            L[rng.integers(0, V, V // 2)] = L[0]
        T = float(np.float32(rng.choice([0.5, 1.0, 1.7])))
        k = [None, int(rng.integers(0, V + 2))][int(rng.integers(0, 2))]
        P = [None, float(np.float32(rng.uniform(0.05, 1.0)))][int(rng.integers(0, 2))]
        x = L / T
        p = np.exp(x - x.max())
        p = p / p.sum()
        q, _ = oracle.sample_filter(L, T, k, P)
        # skip draws whose top-p decision sits within rounding of the threshold
        if P is not None:
            kk = _brute_kept(p, k, None)
            mk = sum(p[i] for i in kk)
            s = sorted(kk, key=lambda i: (-p[i], i))
            ahead = np.cumsum([0.0] + [p[i] for i in s])[:-1] / mk
            if np.min(np.abs(ahead - P)) < 1e-9:
                continue
        assert np.nonzero(q)[0].tolist() == _brute_kept(list(p), k, P)
        kept = np.nonzero(q)[0]
        assert np.allclose(q[kept], p[kept] / p[kept].sum(), rtol=1e-12)
        checked += 1
    assert checked > 300


def test_equal_probabilities_keep_the_lowest_indices():
    L = np.array([0.0, 1.0, 1.0, 1.0, 0.5, 1.0])
    q, order = oracle.sample_filter(L, 1.0, 2, None)
    assert np.nonzero(q)[0].tolist() == [1, 2]
    assert order.tolist()[:4] == [1, 2, 3, 5]


def test_filter_is_permutation_equivariant_without_ties():
    rng = np.random.default_rng(6)
    L = rng.normal(0, 2, 200)
    perm = rng.permutation(200)
    for k, p in ((None, 0.9), (30, None), (30, 0.6)):
        a, _ = oracle.sample_filter(L, 1.0, k, p)
        b, _ = oracle.sample_filter(L[perm], 1.0, k, p)
        assert np.allclose(a[perm], b, rtol=1e-12, atol=0)
