"""Validity of a sampled token against the fp64 oracle (test helper).

The kernel computes each weight e_i = 2^y_i, y_i = (l_i - max) * log2(e) / T,
in fp32: the subtraction, log2(e), the division by T and the product each
round once (|dy| <= 4 * 2^-24 |y|) and ex2.approx adds at most 2^-22
relative, so e_i is off by at most rho_i = ln2 * |y_i| * 2^-22 + 2^-22
relative.  Its fp32 sums run through at most 48 roundings (a lane's eight
terms, warp trees, a chunk rescale, block sums and scans).  A cumulative
share of the kept mass is then off by at most
    delta = 2 * sum_i p_i rho_i + 48 * 2^-24.
A token is accepted when it is the oracle's own draw, or when the uniform
lies within 4 delta of its interval under the oracle's kept set with any of
the decisions that sit within that error of a cut flipped (a top-k boundary
token whose probability is within 8 rho of the k-th one, a token whose top-p
mass ahead is within 4 delta of top_p)."""
from __future__ import annotations

import itertools
import math

import numpy as np

import oracle

LN2 = math.log(2.0)


def _weights(L, T):
    T = float(np.float32(max(float(T), oracle.SAMPLE_MIN_T)))
    y = (np.asarray(L, np.float64) - np.max(L)) / T / LN2
    e = np.exp2(y)
    return y, e


def row_delta(L, T) -> float:
    y, e = _weights(L, T)
    p = e / e.sum()
    rho = LN2 * np.abs(np.where(p > 0, y, 0.0)) * 2.0 ** -22 + 2.0 ** -22
    return float(2.0 * (p * rho).sum() + 48.0 * 2.0 ** -24)


def check_draw(L, T, k, P, u, tok) -> str:
    """'exact' if tok is the oracle's draw, 'boundary' if it is valid within
    the kernel's error bound; AssertionError otherwise."""
    q, order = oracle.sample_filter(L, T, k, P)
    if tok == oracle.inverse_cdf(q, u):
        return "exact"
    V = len(L)
    assert 0 <= tok < V, f"token {tok} outside [0, {V})"
    y, e = _weights(L, T)
    p = e / e.sum()
    tol = 4.0 * row_delta(L, T)
    sp = p[order]
    amb = set()
    kk = V
    if k is not None and 1 <= int(k) < V:
        kk = int(k)
        yk = y[order[kk - 1]]
        rho_k = LN2 * (abs(yk) if np.isfinite(yk) else 0.0) * 2.0 ** -22 + 2.0 ** -22
        pk = sp[kk - 1]
        amb |= set(order[np.nonzero(np.abs(sp - pk) <= 8.0 * rho_k * pk)[0]].tolist())
    Pc = 1.0 if P is None else float(np.float32(min(max(float(P), oracle.SAMPLE_MIN_P), 1.0)))
    if Pc < 1.0:
        m = sp.copy()
        m[kk:] = 0.0
        m /= m.sum()
        before = np.concatenate([[0.0], np.cumsum(m)[:-1]])
        near = np.nonzero((np.abs(before - Pc) <= tol) & (np.arange(V) < kk))[0]
        amb |= set(order[near].tolist())
    amb = sorted(amb)[:8]
    base = q > 0
    for r in range(len(amb) + 1):
        for flip in itertools.combinations(amb, r):
            kept = base.copy()
            for i in flip:
                kept[i] = not kept[i]
            if not kept[tok]:
                continue
            qa = np.where(kept, p, 0.0)
            c = np.cumsum(qa / qa.sum())
            lo = c[tok - 1] if tok else 0.0
            if lo - tol <= float(u) <= c[tok] + tol:
                return "boundary"
    want = oracle.inverse_cdf(q, u)
    raise AssertionError(
        f"token {tok} (oracle {want}): u={float(u):.9f}, kept={bool(q[tok] > 0)}, "
        f"tol={tol:.2e}, ambiguous={amb}")


def check_batch(logits_f64, temperatures, top_k, top_p, uniforms, tokens):
    """check_draw for every row (arguments as sampling_args returns them);
    returns (exact, boundary) counts."""
    exact = boundary = 0
    for r in range(len(tokens)):
        kind = check_draw(logits_f64[r], temperatures[r],
                          None if top_k is None else top_k[r],
                          None if top_p is None else top_p[r], uniforms[r], int(tokens[r]))
        exact += kind == "exact"
        boundary += kind == "boundary"
    return exact, boundary
