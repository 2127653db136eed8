"""The sampler's validity check must not be vacuous: planted mistakes on the
CPU (a token off by one, a token from outside the kept set, the draw taken
from the wrong end) fail it; perturbations within the derived error bound
pass it."""
import numpy as np
import pytest

import oracle
from _sampler_check import check_draw, row_delta


def _rows(seed, n, V):
    rng = np.random.default_rng(seed)
    L = rng.normal(0, 2, (n, V)).astype(np.float32)
    for r in range(n):
        L[r, rng.choice(V, 3, replace=False)] += rng.uniform(2, 8, 3).astype(np.float32)
    return L.astype(np.float64), rng.random(n).astype(np.float32)


def test_oracle_draws_pass():
    L, u = _rows(1, 30, 500)
    for r in range(30):
        q, _ = oracle.sample_filter(L[r], 1.0, 50, 0.9)
        assert check_draw(L[r], 1.0, 50, 0.9, u[r], oracle.inverse_cdf(q, u[r])) == "exact"


def test_planted_mistakes_fail():
    L, u = _rows(2, 40, 300)
    caught = 0
    for r in range(40):
        q, _ = oracle.sample_filter(L[r], 1.0, 20, 0.95)
        tok = oracle.inverse_cdf(q, u[r])
        c = np.cumsum(q)
        if min(abs(u[r] - (c[tok - 1] if tok else 0.0)), abs(u[r] - c[tok])) < 1e-4:
            continue                                  # the uniform sits on a boundary
        kept = np.nonzero(q)[0]
        wrong = [kept[(list(kept).index(tok) + 1) % len(kept)],      # the next kept token
                 int(np.argmin(L[r])),                                # a cut token
                 oracle.inverse_cdf(q[::-1], u[r])]                   # draw from the wrong end
        for w in wrong:
            if w == tok:
                continue
            with pytest.raises(AssertionError):
                check_draw(L[r], 1.0, 20, 0.95, u[r], int(w))
            caught += 1
    assert caught > 80


def test_perturbation_within_bound_passes():
    # a CDF moved by less than the bound may shift the draw to a neighbour
    L, _ = _rows(3, 20, 2000)
    for r in range(20):
        q, _ = oracle.sample_filter(L[r], 1.3, None, None)
        c = np.cumsum(q)
        d = row_delta(L[r], 1.3)
        i = int(np.argmax(q))
        u = np.float32(c[i] + 0.5 * d)                # just past token i's interval
        tok_near = i                                  # a kernel 0.5 delta off draws i
        assert check_draw(L[r], 1.3, None, None, u, tok_near) in ("exact", "boundary")


def test_bound_is_small():
    L, _ = _rows(4, 10, 151936 // 10)
    for r in range(10):
        for T in (0.5, 1.0, 1.3):
            assert row_delta(L[r], T) < 1e-5
