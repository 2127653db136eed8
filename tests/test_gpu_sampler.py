"""GPU parity of the batched sampler (msg_sample) against the fp64 oracle
("Engine 与采样器" 采样器 and 测试; "Mini-SGLang 源码解析（四）" 14).

Bars: greedy rows (no temperatures) bit-exact against the first argmax;
sampled rows either the oracle's own draw, or valid within the kernel's
fp32 error bound (tests/_sampler_check.py derives it: the uniform within
4 delta of the token's interval, delta ~ 1e-6 of the kept mass); rows built
with every decision far from a boundary bit-exact; the printed engine test
reproduced; bad logits and parameters reported, not faulted."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_store_gb300 as msg
from paged_kv_gqa_store_gb300 import workload as wl

from _sampler_check import check_batch, check_draw

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    msg.load_library()


def _dev_logits(spec):
    if spec.is_bf16:
        return wl.bits_to_torch(spec.logits, "cuda")
    return torch.from_numpy(spec.logits).cuda()


def _run(spec, greedy=False, status=None):
    V = spec.vocab
    t, k, p = oracle.sampling_args(spec.temperature, spec.top_k, spec.top_p, V)
    dt, dk, dp = msg.sampling_args(spec.temperature, spec.top_k, spec.top_p, V)
    u = torch.from_numpy(spec.uniforms).cuda()
    out = msg.msg_sample(_dev_logits(spec), dt, dk, dp, u, dev_status=status)
    torch.cuda.synchronize()
    return out.cpu().numpy(), (t, k, p)


def _status():
    return torch.zeros(4, dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("vocab", [1000, 5003, 24577, 60000])
def test_mixed_batch_valid(vocab, bf16):
    spec = wl.sampler_batch("mixed", 7000 + vocab, 64, vocab, bf16=bf16)
    st = _status()
    got, (t, k, p) = _run(spec, status=st)
    assert msg.msg_read_device_status(st)[0] == msg.MSG_OK
    exact, boundary = check_batch(spec.logits_f64(), t, k, p, spec.uniforms, got)
    assert exact + boundary == spec.batch
    assert exact >= spec.batch * 0.75, (exact, boundary)


@pytest.mark.parametrize("bf16", [True, False])
def test_full_vocab_batch(bf16):
    # the benchmark's launch: 256 rows of Qwen3's 151,936-token vocabulary
    spec = wl.sampler_batch("full", 8100 + bf16, 256, wl.QWEN3_VOCAB, bf16=bf16)
    st = _status()
    got, (t, k, p) = _run(spec, status=st)
    assert msg.msg_read_device_status(st)[0] == msg.MSG_OK
    exact, boundary = check_batch(spec.logits_f64(), t, k, p, spec.uniforms, got)
    assert exact + boundary == spec.batch
    # deterministic: the same inputs give the same tokens
    again, _ = _run(spec)
    assert np.array_equal(got, again)


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("vocab", [1, 7, 1000, 24577, wl.QWEN3_VOCAB])
def test_greedy_is_first_argmax(vocab, bf16):
    spec = wl.sampler_batch("greedy", 9000 + vocab, 96, vocab, bf16=bf16, greedy_only=True)
    if vocab > 3:                                    # tied maxima across chunks
        L = spec.logits_f64()
        for r in range(0, spec.batch, 3):
            m = int(np.argmax(L[r]))
            spec.logits[r, [0, vocab // 2, vocab - 1]] = spec.logits[r, m]
    L = spec.logits_f64()
    got, (t, _, _) = _run(spec)
    assert t is None
    assert np.array_equal(got, oracle.sample(L, None, None, None, None))


def test_separated_rows_are_exact():
    # every probability far from every other and every uniform mid-interval:
    # no rounding can move a decision, so the draw must be the oracle's
    rng = np.random.default_rng(11)
    B, V = 96, 64
    L = np.empty((B, V), np.float32)
    for r in range(B):
        L[r] = rng.permutation(np.arange(V, dtype=np.float32) * 0.37)
    mix = [(1.0, -1, 1.0), (0.8, 5, 1.0), (1.2, -1, 0.6), (0.9, 12, 0.8), (0.0, -1, 1.0),
           (1.0, 1, 1.0), (2.0, 40, 0.97), (0.5, -1, 0.999)]
    T = np.array([mix[r % 8][0] for r in range(B)], np.float32)
    K = np.array([mix[r % 8][1] for r in range(B)], np.int32)
    P = np.array([mix[r % 8][2] for r in range(B)], np.float32)
    t, k, p = oracle.sampling_args(T, K, P, V)
    u = np.empty(B, np.float32)
    for r in range(B):
        q, _ = oracle.sample_filter(L[r], t[r], k[r], p[r])
        c = np.cumsum(q)
        kept = np.nonzero(q > 1e-3)[0]                # intervals far wider than rounding
        i = kept[rng.integers(0, len(kept))]
        u[r] = np.float32(((c[i - 1] if i else 0.0) + c[i]) / 2)
    spec = wl.SamplerSpec("separated", L, False, T, K, P, u)
    got, _ = _run(spec)
    assert np.array_equal(got, oracle.sample(L.astype(np.float64), t, k, p, u))


def test_ties_keep_lowest_indices():
    # bf16 logits with a block of exactly equal maxima: top-k cuts inside the
    # tie, so only the lowest indices may be drawn, each with equal mass
    B, V = 64, 3000
    rng = np.random.default_rng(12)
    L = rng.normal(0, 1, (B, V)).astype(np.float32)
    tied = np.sort(rng.choice(V, 10, replace=False))
    L[:, tied] = 6.0
    bits = wl.f32_to_bf16_bits(L)
    T = np.full(B, 1.0, np.float32)
    K = np.full(B, 4, np.int32)
    P = np.ones(B, np.float32)
    u = ((np.arange(B) % 8) / 8 + 1 / 16).astype(np.float32)
    spec = wl.SamplerSpec("ties", bits, True, T, K, P, u)
    got, _ = _run(spec)
    want = tied[:4][np.minimum((u * 4).astype(int), 3)]
    assert np.array_equal(got, want)


def test_engine_test_case_on_the_gpu():
    # the printed sampler test: logits [5, 4, 3, 0, 0, 0]; top-k 2, top-p 0.5,
    # and a greedy request in the same batch
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                    "sampler_pages.json")))["engine_test"]
    n = g["draws"]
    reqs = g["requests"] * n
    L = np.array([g["logits"]] * len(reqs), np.float32)
    T = np.array([r["temperature"] for r in reqs], np.float32)
    K = np.array([r["top_k"] for r in reqs], np.int32)
    P = np.array([r["top_p"] for r in reqs], np.float32)
    u = np.random.default_rng(0).random(len(reqs)).astype(np.float32)
    spec = wl.SamplerSpec("engine_test", L, False, T, K, P, u)
    got, _ = _run(spec)
    draws = got.reshape(n, 3)
    for row, support in enumerate(g["support"]):
        assert set(draws[:, row].tolist()) == set(support)
    assert abs((draws[:, 0] == 0).mean() - g["first_token_frequency_row0"]) < g["frequency_tolerance"]


def test_edge_parameters():
    V = 5003
    rng = np.random.default_rng(13)
    L = rng.normal(0, 2, (8, V)).astype(np.float32)
    L[:, 17] += 30.0                                  # one dominant token
    # k > V, k = V, top_p = 1 exactly, u = 0, u just below 1, T = 0 (greedy row)
    T = np.array([1.0, 1.0, 1.0, 0.0, 1.0, 1.0, 3.0, 1.0], np.float32)
    K = np.array([V + 5, V, -1, -1, 1, -1, 2, 3], np.int32)
    P = np.array([1.0, 1.0, 1.0, 1.0, 1.0, 1e-9, 0.999, 0.9], np.float32)
    u = np.array([0.0, 0.99999994, 0.5, 0.3, 0.9, 0.7, 0.0, 0.99999994], np.float32)
    spec = wl.SamplerSpec("edges", L, False, T, K, P, u)
    got, (t, k, p) = _run(spec)
    exact, boundary = check_batch(L.astype(np.float64), t, k, p, u, got)
    assert exact + boundary == 8
    assert got[3] == 17 and got[4] == 17 and got[5] == 17


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("col0", [0, 1, 3, 5])
def test_row_stride_and_unaligned_rows(col0, bf16):
    # rows 3013 elements apart, the first logit at column col0 of the buffer:
    # rows start at every alignment and nothing outside them is used
    V, W, B = 3001, 3013, 32
    spec = wl.sampler_batch("stride", 14, B, V, bf16=bf16)
    wide = np.zeros((B, W), spec.logits.dtype)
    wide[:, :] = wl.f32_to_bf16_bits(np.float32(1e30)) if bf16 else np.float32(1e30)
    wide[:, col0:col0 + V] = spec.logits
    t, k, p = oracle.sampling_args(spec.temperature, spec.top_k, spec.top_p, V)
    dt, dk, dp = msg.sampling_args(spec.temperature, spec.top_k, spec.top_p, V)
    full = wl.bits_to_torch(wide, "cuda") if bf16 else torch.from_numpy(wide).cuda()
    out = msg.msg_sample(full[:, col0:col0 + V], dt, dk, dp, torch.from_numpy(spec.uniforms).cuda())
    got = out.cpu().numpy()
    exact, boundary = check_batch(spec.logits_f64(), t, k, p, spec.uniforms, got)
    assert exact + boundary == B
    g = msg.msg_sample(full[:, col0:col0 + V], None, None, None, None).cpu().numpy()
    assert np.array_equal(g, np.argmax(spec.logits_f64(), axis=1))


def test_bad_inputs_are_reported():
    spec = wl.sampler_batch("bad", 15, 6, 2000)
    spec.logits[1, 7] = np.nan
    spec.uniforms[3] = 1.0
    st = _status()
    got, (t, k, p) = _run(spec, status=st)
    code, info = msg.msg_read_device_status(st)
    assert code == msg.MSG_ERR_DEVICE_CHECK
    assert info[0] in (msg.MSG_DEV_BAD_LOGIT, msg.MSG_DEV_BAD_SAMPLING)
    assert got[1] == -1 and got[3] == -1
    for r in (0, 2, 4, 5):
        check_draw(spec.logits_f64()[r], t[r], None if k is None else k[r],
                   None if p is None else p[r], spec.uniforms[r], int(got[r]))
    # +inf has no softmax; greedy rows take it as their maximum but report a NaN
    st = _status()
    spec = wl.sampler_batch("badinf", 17, 3, 2000)
    spec.logits[0, 5] = np.inf
    got, _ = _run(spec, status=st)
    assert msg.msg_read_device_status(st)[1][0] == msg.MSG_DEV_BAD_LOGIT and got[0] == -1
    st = _status()
    g = wl.sampler_batch("badg", 16, 4, 2000, greedy_only=True)
    g.logits[2, 1999] = np.nan
    g.logits[3, 7] = np.inf
    got, _ = _run(g, status=st)
    assert msg.msg_read_device_status(st)[1][0] == msg.MSG_DEV_BAD_LOGIT
    assert got[2] == -1 and got[3] == 7


@pytest.mark.parametrize("bf16", [False, True])
def test_minus_infinity_masks_tokens(bf16):
    # -inf logits are tokens of probability zero: never drawn, and a row
    # whose every logit is -inf is reported
    V, B = 5003, 48
    spec = wl.sampler_batch("masked", 18, B, V)
    rng = np.random.default_rng(19)
    mask = rng.random((B, V)) < 0.7
    spec.logits[mask] = -np.inf
    spec.logits[:, 11] = -np.inf
    spec.logits[B - 1, :] = -np.inf
    if bf16:
        spec = wl.SamplerSpec("masked", wl.f32_to_bf16_bits(spec.logits), True, spec.temperature,
                              spec.top_k, spec.top_p, spec.uniforms)
    st = _status()
    got, (t, k, p) = _run(spec, status=st)
    assert msg.msg_read_device_status(st)[1][0] == msg.MSG_DEV_BAD_LOGIT
    assert got[B - 1] == -1
    L = spec.logits_f64()
    for r in range(B - 1):
        assert np.isfinite(L[r, got[r]]) and got[r] != 11
        check_draw(L[r], t[r], None if k is None else k[r], None if p is None else p[r],
                   spec.uniforms[r], int(got[r]))
