"""Pins of the oracle's attention prologue: RMSNorm and the rotary embedding
("第 0 步：一个能跑的最小推理引擎", 四个算子; "Mini-SGLang 完整剖析" 4.5.6 and
4.6.7).  Closed forms, invariants and an independent complex-number
formulation of the rotation fix every step."""
import math

import numpy as np
import pytest

import oracle


def _bits(x):
    """float -> bf16 bits (round to nearest even), for building inputs."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) & 0xFFFF).astype(np.uint16)


# ------------------------------------------------------------ rotary cache
def test_cache_row_zero_is_identity():
    cs = oracle.rope_cos_sin_cache(1e6, 128, 4)
    assert (cs[0, :64] == 1.0).all() and (cs[0, 64:] == 0.0).all()


def test_cache_first_frequency_is_one_radian_per_position():
    # inv_freq_0 = theta^0 = 1, so the angle of column 0 is the position itself
    cs = oracle.rope_cos_sin_cache(1e6, 128, 3000)
    p = np.arange(3000)
    assert np.array_equal(cs[:, 0], np.cos(p.astype(np.float64)).astype(np.float32))
    assert np.array_equal(cs[:, 64], np.sin(p.astype(np.float64)).astype(np.float32))


def test_cache_frequencies_closed_form():
    # theta = 10000, D = 128: inv_freq_1 = exp(-ln(10000) / 64); angle at p = 1
    cs = oracle.rope_cos_sin_cache(10000.0, 128, 2)
    f1 = math.exp(-math.log(10000.0) / 64)
    assert abs(float(cs[1, 1]) - math.cos(f1)) < 2e-7
    assert abs(float(cs[1, 65]) - math.sin(f1)) < 2e-7
    # theta = 1e6: inv_freq_32 = theta^(-1/2) = 1e-3
    cs = oracle.rope_cos_sin_cache(1e6, 128, 1001)
    assert abs(float(cs[1000, 32]) - math.cos(1.0)) < 1e-6


def test_cache_is_on_the_unit_circle():
    cs = oracle.rope_cos_sin_cache(1e6, 128, 5000).astype(np.float64)
    r = cs[:, :64] ** 2 + cs[:, 64:] ** 2
    assert np.abs(r - 1).max() < 4e-7


# ------------------------------------------------------------ RMSNorm
def test_rmsnorm_constant_vector():
    x = np.full(128, -3.0)
    w = np.linspace(0.5, 2.0, 128)
    eps = 1e-6
    out = oracle.rmsnorm(x, w, eps)
    assert np.allclose(out, w * -3.0 / math.sqrt(9.0 + eps), rtol=0, atol=1e-15)


def test_rmsnorm_scale_invariant_and_unit_rms_without_eps():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 128))
    out = oracle.rmsnorm(x, np.ones(128), 0.0)
    assert np.allclose(oracle.rmsnorm(7.5 * x, np.ones(128), 0.0), out, rtol=1e-13, atol=0)
    assert np.allclose((out ** 2).mean(-1), 1.0, rtol=1e-13)


def test_rmsnorm_eps_shrinks_toward_zero():
    x = np.full(128, 1e-3)
    out = oracle.rmsnorm(x, np.ones(128), 1e-6)      # mean x^2 = 1e-6 = eps
    assert np.allclose(out, 1e-3 / math.sqrt(2e-6), rtol=1e-13)


# ------------------------------------------------------------ rope
def test_rope_position_zero_is_identity():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((3, 4, 128))
    cs = oracle.rope_cos_sin_cache(1e6, 128, 1)
    assert np.array_equal(oracle.rope(x, np.repeat(cs[:1], 3, 0)), x)


def test_rope_matches_complex_rotation():
    # pair (x1_i, x2_i) as x1_i + j x2_i, multiplied by e^{j angle_i}
    rng = np.random.default_rng(3)
    x = rng.standard_normal((6, 2, 128))
    cs = oracle.rope_cos_sin_cache(1e6, 128, 4000)
    pos = np.array([0, 1, 17, 999, 2048, 3999])
    rows = cs[pos].astype(np.float64)
    z = (x[..., :64] + 1j * x[..., 64:]) * (rows[:, None, :64] + 1j * rows[:, None, 64:])
    want = np.concatenate([z.real, z.imag], axis=-1)
    assert np.allclose(oracle.rope(x, cs[pos]), want, rtol=0, atol=1e-12)


def test_rope_preserves_pair_norms():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((50, 128))
    cs = oracle.rope_cos_sin_cache(1e6, 128, 50000)
    y = oracle.rope(x, cs[rng.integers(0, 50000, size=50)])
    n0 = x[:, :64] ** 2 + x[:, 64:] ** 2
    n1 = y[:, :64] ** 2 + y[:, 64:] ** 2
    assert np.allclose(n0, n1, rtol=1e-6)


def test_rope_scores_depend_on_relative_position_only():
    # exact angles (float64), so the identity holds to rounding
    D, theta = 128, 1e6
    inv = theta ** (-2.0 * np.arange(64) / D)

    def row(p):
        a = p * inv
        return np.concatenate([np.cos(a), np.sin(a)])

    rng = np.random.default_rng(5)
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    for m, n, s in ((10, 3, 100), (500, 499, 7), (0, 40, 1234)):
        d0 = oracle.rope(q, row(m)) @ oracle.rope(k, row(n))
        d1 = oracle.rope(q, row(m + s)) @ oracle.rope(k, row(n + s))
        assert abs(d0 - d1) < 1e-9 * (1 + abs(d0))


# ------------------------------------------------------------ the fused front
def test_qk_norm_rope_splits_qkv_and_copies_v():
    Hq, Hk, D, T = 4, 2, 128, 3
    rng = np.random.default_rng(6)
    qkv = _bits(rng.standard_normal((T, (Hq + 2 * Hk) * D)))
    qw, kw = _bits(np.full(D, 1.0)), _bits(np.full(D, 2.0))
    cs = oracle.rope_cos_sin_cache(1e6, D, 10)
    q, k, v = oracle.qk_norm_rope(qkv, [0, 0, 0], qw, kw, 0.0, cs, Hq, Hk, D)
    x = oracle.bf16_bits_to_f64(qkv)
    # position 0: no rotation, so q and k are just the normed inputs (k twice as large)
    assert np.allclose(q, oracle.rmsnorm(x[:, :Hq * D].reshape(T, Hq, D), 1.0, 0.0), atol=1e-14)
    assert np.allclose(k, oracle.rmsnorm(x[:, Hq * D:(Hq + Hk) * D].reshape(T, Hk, D), 2.0, 0.0),
                       atol=1e-14)
    assert np.array_equal(v, qkv[:, (Hq + Hk) * D:].reshape(T, Hk, D))
