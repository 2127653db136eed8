"""Pins for the fp64 CPU oracle: values and facts fixed by the pages and by
mathematics, independent of the oracle's own code.

* worked request-length examples printed on the pages (tests/golden/req_lengths.json);
* brute-force contiguous (unpaged) attention on tiny inputs, written as the
  matrix form of the "第 0 步" attention operator (repeat K/V heads, full score
  matrix, explicit causal mask);
* torch's scaled_dot_product_attention in float64 for cached_len = 0, where the
  method is textbook causal self-attention;
* closed forms: constant V, a single visible key, constant K;
* invariants: page permutation, page_size, chunked prefill vs one extend;
* store_kv round trip and untouched rows.

Each case is chosen so a plausible slip in the oracle (dropped scale, wrong GQA
mapping, off-by-one mask, wrong causal offset, wrong page gather, transposed
operand) breaks at least one of them.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_store_gb300 import workload as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "req_lengths.json")


# ------------------------------------------------------------ worked examples
def _lengths(cached, device, max_device):
    return [cached, device, device - cached, max_device - device]


def test_req_lengths_worked_examples():
    g = json.load(open(GOLDEN))
    for case in g["cases"]:
        cached, device = case["cached_len"], case["prompt_len"]
        max_device = case["prompt_len"] + case["max_tokens"]
        states = [_lengths(cached, device, max_device)]
        n_steps = max(len(case.get("states", [])), 1 + max(
            int(k) for k in case.get("checkpoints", {"0": 0})))
        for _ in range(n_steps - 1):
            cached, device = oracle.complete_one(cached, device)
            states.append(_lengths(cached, device, max_device))
        if "states" in case:
            assert states == case["states"], case["cite"]
        for k, v in case.get("checkpoints", {}).items():
            assert states[int(k)] == v, case["cite"]


def test_metadata_worked_example_prompt6_cached2():
    # prompt 6 with 2 cached tokens: this step feeds 4 tokens at positions 2..5
    # whose K/V go to page_table[row, 2:6]; after the step device_len is 7.
    rng = np.random.default_rng(0)
    pt = rng.permutation(4096)[:32].astype(np.int32).reshape(1, 32)
    m = oracle.metadata(pt, cached_len=[2], extend_len=[4])
    assert m["qo_indptr"].tolist() == [0, 4]
    assert m["kv_len"].tolist() == [6]
    assert m["positions"].tolist() == [2, 3, 4, 5]
    assert m["out_loc"].tolist() == pt[0, 2:6].tolist()
    c, d = oracle.complete_one(2, 6)
    m2 = oracle.metadata(pt, cached_len=[c], extend_len=[d - c])
    assert (c, d) == (6, 7)
    assert m2["positions"].tolist() == [6] and m2["out_loc"].tolist() == [pt[0, 6]]


def test_metadata_two_prompt_batch_token_counts():
    g = json.load(open(GOLDEN))["batch"]
    lens = g["prompt_lens"]
    pt = np.arange(2 * 256, dtype=np.int32).reshape(2, 256)   # rows as in the driver
    m = oracle.metadata(pt, cached_len=[0, 0], extend_len=lens)
    assert int(m["qo_indptr"][-1]) == g["prefill_tokens"]
    assert m["out_loc"].tolist() == list(range(0, lens[0])) + list(range(256, 256 + lens[1]))
    cached = [lens[0], lens[1]]
    m = oracle.metadata(pt, cached_len=cached, extend_len=[1, 1])
    assert int(m["qo_indptr"][-1]) == g["decode_tokens_per_step"]
    assert m["positions"].tolist() == cached


def test_metadata_req_rows_and_ragged():
    rng = np.random.default_rng(1)
    pt = rng.integers(0, 1 << 20, size=(7, 64)).astype(np.int32)
    rows = np.array([5, 0, 3], np.int32)
    cached = np.array([0, 10, 33], np.int32)
    ext = np.array([7, 1, 30], np.int32)
    m = oracle.metadata(pt, cached, ext, req_rows=rows)
    assert m["qo_indptr"].tolist() == [0, 7, 8, 38]
    exp_loc = np.concatenate([pt[5, 0:7], pt[0, 10:11], pt[3, 33:63]])
    assert m["out_loc"].tolist() == exp_loc.tolist()
    assert m["positions"].tolist() == list(range(7)) + [10] + list(range(33, 63))


# ------------------------------------------------------------ helpers
def _paged_setup(seed, cached, ext, Hq, Hkv, D, page_size=1, num_pages=None):
    rng = np.random.default_rng(seed)
    cached = np.asarray(cached, np.int32)
    ext = np.asarray(ext, np.int32)
    dev = cached.astype(np.int64) + ext
    if num_pages is None:
        num_pages = int(((dev + page_size - 1) // page_size).sum()) + 7
    pt = wl.assign_pages(rng, dev, page_size, num_pages)
    T = int(ext.sum())
    q = wl.random_bf16(rng, (T, Hq, D))
    # Full contiguous K/V per request (prefix + new), then scattered into pools.
    kv = [(wl.random_bf16(rng, (int(L), Hkv, D)), wl.random_bf16(rng, (int(L), Hkv, D)))
          for L in dev]
    return rng, cached, ext, dev, pt, q, kv, num_pages * page_size


def _pools_from(kv, pt, dev, num_slots, Hkv, D):
    kp = np.full((num_slots, Hkv, D), wl.CANARY_BF16, np.uint16)
    vp = np.full((num_slots, Hkv, D), wl.CANARY_BF16, np.uint16)
    for r, (k, v) in enumerate(kv):
        slots = pt[r, :dev[r]]
        kp[slots] = k
        vp[slots] = v
    return kp, vp


def _brute(q_req, k_req, v_req, scale):
    """Contiguous attention for one request: q [T,Hq,D], k/v [S,Hkv,D] in fp64;
    query t sits at absolute position S-T+t and sees keys at positions <= it."""
    T, Hq, D = q_req.shape
    S, Hkv, _ = k_req.shape
    kk = np.repeat(k_req, Hq // Hkv, axis=1)          # repeat_interleave on heads
    vv = np.repeat(v_req, Hq // Hkv, axis=1)
    scores = np.einsum("thd,shd->hts", q_req, kk) * scale
    mask = np.arange(S)[None, :] <= np.arange(S - T, S)[:, None]
    scores = np.where(mask[None], scores, -np.inf)
    w = np.exp(scores - scores.max(-1, keepdims=True))
    w /= w.sum(-1, keepdims=True)
    return np.einsum("hts,shd->thd", w, vv)


def _oracle_out(q, kp, vp, pt, cached, ext, Hq, Hkv, D, scale=None):
    qo = np.concatenate([[0], np.cumsum(ext)]).astype(np.int32)
    return oracle.paged_attention(q, kp, vp, pt, cached, qo, Hq, Hkv, D, scale=scale)


# ------------------------------------------------------------ brute force
@pytest.mark.parametrize("Hq,Hkv,D", [(4, 2, 8), (16, 8, 128), (6, 2, 16), (4, 4, 8)])
def test_oracle_matches_brute_force(Hq, Hkv, D):
    cached, ext = [0, 3, 5, 1, 0], [1, 4, 1, 7, 3]
    _, cached, ext, dev, pt, q, kv, ns = _paged_setup(11 + Hq + D, cached, ext, Hq, Hkv, D)
    kp, vp = _pools_from(kv, pt, dev, ns, Hkv, D)
    got = _oracle_out(q, kp, vp, pt, cached, ext, Hq, Hkv, D)
    qf = wl.bf16_bits_to_f64(q)
    off = 0
    for r in range(len(cached)):
        e = int(ext[r])
        ref = _brute(qf[off:off + e], wl.bf16_bits_to_f64(kv[r][0]),
                     wl.bf16_bits_to_f64(kv[r][1]), 1.0 / np.sqrt(D))
        np.testing.assert_allclose(got[off:off + e], ref, rtol=1e-12, atol=1e-12)
        off += e


def test_brute_force_is_sensitive_to_gqa_mapping():
    # Guard on the pin itself: h -> h % Hkv differs from h -> h // G on this input.
    rng = np.random.default_rng(3)
    q = wl.bf16_bits_to_f64(wl.random_bf16(rng, (3, 4, 8)))
    k = wl.bf16_bits_to_f64(wl.random_bf16(rng, (5, 2, 8)))
    v = wl.bf16_bits_to_f64(wl.random_bf16(rng, (5, 2, 8)))
    a = _brute(q, k, v, 1 / np.sqrt(8))
    kt = np.tile(k, (1, 2, 1))
    vt = np.tile(v, (1, 2, 1))
    b = np.einsum("hts,shd->thd", torch.softmax(torch.from_numpy(np.where(
        (np.arange(5)[None, :] <= np.arange(2, 5)[:, None])[None],
        np.einsum("thd,shd->hts", q, kt) / np.sqrt(8), -np.inf)), -1).numpy(), vt)
    assert np.abs(a - b).max() > 1e-3


# ------------------------------------------------------------ library routine
@pytest.mark.parametrize("T", [1, 5, 33])
def test_oracle_matches_sdpa_when_nothing_cached(T):
    Hq, Hkv, D = 16, 8, 128
    _, cached, ext, dev, pt, q, kv, ns = _paged_setup(100 + T, [0, 0], [T, T + 3], Hq, Hkv, D)
    kp, vp = _pools_from(kv, pt, dev, ns, Hkv, D)
    got = _oracle_out(q, kp, vp, pt, cached, ext, Hq, Hkv, D)
    qf = torch.from_numpy(wl.bf16_bits_to_f64(q))
    off = 0
    for r in range(2):
        e = int(ext[r])
        k = torch.from_numpy(wl.bf16_bits_to_f64(kv[r][0])).repeat_interleave(Hq // Hkv, dim=1)
        v = torch.from_numpy(wl.bf16_bits_to_f64(kv[r][1])).repeat_interleave(Hq // Hkv, dim=1)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qf[off:off + e].transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1),
            is_causal=True).transpose(0, 1).numpy()
        np.testing.assert_allclose(got[off:off + e], ref, rtol=1e-10, atol=1e-12)
        off += e


def test_oracle_decode_matches_sdpa_full_visibility():
    # A decode row (cached c, extend 1) sees every key: unmasked SDPA over c+1 keys.
    Hq, Hkv, D = 16, 8, 128
    _, cached, ext, dev, pt, q, kv, ns = _paged_setup(7, [40], [1], Hq, Hkv, D)
    kp, vp = _pools_from(kv, pt, dev, ns, Hkv, D)
    got = _oracle_out(q, kp, vp, pt, cached, ext, Hq, Hkv, D)
    qf = torch.from_numpy(wl.bf16_bits_to_f64(q))
    k = torch.from_numpy(wl.bf16_bits_to_f64(kv[0][0])).repeat_interleave(2, dim=1)
    v = torch.from_numpy(wl.bf16_bits_to_f64(kv[0][1])).repeat_interleave(2, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        qf.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1)).transpose(0, 1).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


# ------------------------------------------------------------ closed forms
def test_constant_v_gives_v():
    Hq, Hkv, D = 16, 8, 128
    _, cached, ext, dev, pt, q, kv, ns = _paged_setup(5, [0, 9, 30], [6, 1, 12], Hq, Hkv, D)
    rng = np.random.default_rng(9)
    vconst = wl.random_bf16(rng, (Hkv, D))
    kv = [(k, np.broadcast_to(vconst, v.shape).copy()) for k, v in kv]
    kp, vp = _pools_from(kv, pt, dev, ns, Hkv, D)
    got = _oracle_out(q, kp, vp, pt, cached, ext, Hq, Hkv, D)
    expect = np.repeat(wl.bf16_bits_to_f64(vconst), Hq // Hkv, axis=0)
    np.testing.assert_allclose(got, np.broadcast_to(expect, got.shape), rtol=0, atol=1e-12)


def test_single_visible_key_gives_v0():
    # kv_len 1 (cached 0, extend 1): the only key is the new one -> output = V_0,
    # whatever the scores; the first query of any prefill likewise sees key 0 only.
    Hq, Hkv, D = 16, 8, 128
    _, cached, ext, dev, pt, q, kv, ns = _paged_setup(6, [0, 0], [1, 5], Hq, Hkv, D)
    kp, vp = _pools_from(kv, pt, dev, ns, Hkv, D)
    got = _oracle_out(q, kp, vp, pt, cached, ext, Hq, Hkv, D)
    for row, r in [(0, 0), (1, 1)]:
        v0 = np.repeat(wl.bf16_bits_to_f64(kv[r][1][0]), Hq // Hkv, axis=0)
        np.testing.assert_allclose(got[row], v0, rtol=0, atol=1e-15)


def test_constant_k_gives_mean_of_visible_v():
    Hq, Hkv, D = 16, 8, 128
    _, cached, ext, dev, pt, q, kv, ns = _paged_setup(8, [3, 20], [5, 1], Hq, Hkv, D)
    rng = np.random.default_rng(10)
    kconst = wl.random_bf16(rng, (Hkv, D))
    kv = [(np.broadcast_to(kconst, k.shape).copy(), v) for k, v in kv]
    kp, vp = _pools_from(kv, pt, dev, ns, Hkv, D)
    got = _oracle_out(q, kp, vp, pt, cached, ext, Hq, Hkv, D)
    off = 0
    for r in range(2):
        vf = np.repeat(wl.bf16_bits_to_f64(kv[r][1]), Hq // Hkv, axis=1)
        for i in range(int(ext[r])):
            p = int(cached[r]) + i
            np.testing.assert_allclose(got[off + i], vf[:p + 1].mean(0), rtol=1e-12, atol=1e-13)
        off += int(ext[r])


def test_scale_enters_as_one_over_sqrt_d():
    # Doubling q with scale halved gives the same result; dropping the scale does not.
    Hq, Hkv, D = 4, 2, 8
    _, cached, ext, dev, pt, q, kv, ns = _paged_setup(12, [4], [3], Hq, Hkv, D)
    kp, vp = _pools_from(kv, pt, dev, ns, Hkv, D)
    a = _oracle_out(q, kp, vp, pt, cached, ext, Hq, Hkv, D)
    b = _oracle_out(q, kp, vp, pt, cached, ext, Hq, Hkv, D, scale=1.0)
    assert np.abs(a - b).max() > 1e-3
    ref = _brute(wl.bf16_bits_to_f64(q), wl.bf16_bits_to_f64(kv[0][0]),
                 wl.bf16_bits_to_f64(kv[0][1]), 1 / np.sqrt(D))
    np.testing.assert_allclose(a, ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ invariants
def test_page_permutation_invariance_exact():
    Hq, Hkv, D = 16, 8, 128
    _, cached, ext, dev, pt, q, kv, ns = _paged_setup(21, [7, 0, 50], [5, 9, 1], Hq, Hkv, D)
    kp, vp = _pools_from(kv, pt, dev, ns, Hkv, D)
    a = _oracle_out(q, kp, vp, pt, cached, ext, Hq, Hkv, D)
    perm = np.random.default_rng(22).permutation(ns).astype(np.int32)
    pt2 = perm[pt]
    kp2, vp2 = _pools_from(kv, pt2, dev, ns, Hkv, D)
    b = _oracle_out(q, kp2, vp2, pt2, cached, ext, Hq, Hkv, D)
    assert np.array_equal(a, b)


def test_page_size_invariance_exact():
    Hq, Hkv, D = 16, 8, 128
    cached, ext = [70, 0, 130], [3, 65, 1]
    outs = []
    for P in (1, 16, 64):
        rng_seed = 31
        _, c, e, dev, pt, q, kv, ns = _paged_setup(rng_seed, cached, ext, Hq, Hkv, D,
                                                   page_size=1)
        # same values, different page geometry
        rng = np.random.default_rng(100 + P)
        pt_p = wl.assign_pages(rng, dev, P, int(((dev + P - 1) // P).sum()) + 3)
        ns_p = (int(((dev + P - 1) // P).sum()) + 3) * P
        kp, vp = _pools_from(kv, pt_p, dev, ns_p, Hkv, D)
        outs.append(_oracle_out(q, kp, vp, pt_p, c, e, Hq, Hkv, D))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_chunked_prefill_equals_single_extend():
    # One extend of 11 tokens over 4 cached == chunks 3+5+3 == 11 single steps.
    Hq, Hkv, D = 16, 8, 128
    rng = np.random.default_rng(41)
    L = 15
    pt = wl.assign_pages(rng, [L], 1, 64)
    q = wl.random_bf16(rng, (11, Hq, D))
    k_all = wl.random_bf16(rng, (L, Hkv, D))
    v_all = wl.random_bf16(rng, (L, Hkv, D))
    kp = np.full((64, Hkv, D), wl.CANARY_BF16, np.uint16)
    vp = kp.copy()
    kp[pt[0, :4]] = k_all[:4]
    vp[pt[0, :4]] = v_all[:4]

    def run(chunks):
        kpc, vpc = kp.copy(), vp.copy()
        cached, outs, qi = 4, [], 0
        for e in chunks:
            m = oracle.metadata(pt, [cached], [e])
            oracle.store_kv(k_all[cached:cached + e], v_all[cached:cached + e],
                            m["out_loc"], kpc, vpc)
            outs.append(oracle.paged_attention(q[qi:qi + e], kpc, vpc, pt, [cached],
                                               m["qo_indptr"], Hq, Hkv, D))
            cached += e
            qi += e
        return np.concatenate(outs)

    one = run([11])
    assert np.array_equal(one, run([3, 5, 3]))
    assert np.array_equal(one, run([1] * 11))


# ------------------------------------------------------------ store_kv
def test_store_kv_round_trip_and_untouched_rows():
    rng = np.random.default_rng(51)
    Hkv, D, T, ns = 8, 128, 37, 512
    k = wl.random_bf16(rng, (T, Hkv, D))
    v = wl.random_bf16(rng, (T, Hkv, D))
    loc = rng.permutation(ns)[:T]
    kp = np.full((ns, Hkv, D), wl.CANARY_BF16, np.uint16)
    vp = kp.copy()
    oracle.store_kv(k, v, loc, kp, vp)
    assert np.array_equal(kp[loc], k) and np.array_equal(vp[loc], v)
    untouched = np.setdiff1d(np.arange(ns), loc)
    assert (kp[untouched] == wl.CANARY_BF16).all() and (vp[untouched] == wl.CANARY_BF16).all()


def test_store_kv_later_duplicate_wins_in_oracle():
    # Only padding may repeat a slot; the oracle writes in order, so the last wins.
    Hkv, D = 2, 8
    k = np.arange(3 * Hkv * D, dtype=np.uint16).reshape(3, Hkv, D)
    kp = np.zeros((4, Hkv, D), np.uint16)
    vp = kp.copy()
    oracle.store_kv(k, k, np.array([1, 3, 1]), kp, vp)
    assert np.array_equal(kp[1], k[2]) and np.array_equal(kp[3], k[1])


def test_bf16_input_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.140625], np.float32)
    b = wl.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(b, ref)
    big = np.random.default_rng(0).standard_normal(10000, dtype=np.float32)
    ref = torch.from_numpy(big).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(wl.f32_to_bf16_bits(big), ref)


def test_thread_count_does_not_change_results():
    # the CPU baseline times the oracle on one core and on all of them: every
    # output element is computed by one thread in one order, so the results
    # are bit-identical whatever the thread count
    Hq, Hkv, D = 16, 8, 128
    _, cached, ext, dev, pt, q, kv, ns = _paged_setup(41, [40, 0, 300, 7], [1, 33, 1, 12],
                                                      Hq, Hkv, D)
    kp, vp = _pools_from(kv, pt, dev, ns, Hkv, D)
    n = oracle.num_threads()
    try:
        oracle.set_num_threads(1)
        a = _oracle_out(q, kp, vp, pt, cached, ext, Hq, Hkv, D)
        oracle.set_num_threads(max(n, 3))
        b = _oracle_out(q, kp, vp, pt, cached, ext, Hq, Hkv, D)
    finally:
        oracle.set_num_threads(n)
    assert np.array_equal(a, b)
