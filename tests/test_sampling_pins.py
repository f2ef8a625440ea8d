"""Pins of the temperature-sampled verification oracle (oracle/sampling.py).

The key pin is the exactness of speculative sampling: when the draft token is
itself drawn from p and the uniforms are uniform, the token emitted at a position
is distributed exactly as q.  The test integrates the oracle's own accept rule and
inverse-CDF draw over fine grids of the uniforms (no formula is retyped), so a
wrong acceptance test, a wrong residual or an off-by-one in the draw fails it.
"""

import numpy as np
import pytest

from oracle.sampling import inverse_cdf, residual, sampled_accept, softmax_t, verify_sampled
from synth.workloads import custom
from synth import materialize

RNG = np.random.default_rng(7)


def test_inverse_cdf_matches_searchsorted():
    for _ in range(500):
        n = int(RNG.integers(1, 12))
        wts = RNG.random(n) * (RNG.random(n) < 0.7)
        if wts.sum() == 0:
            wts[RNG.integers(n)] = 1.0
        w = float(RNG.random())
        ref = int(np.searchsorted(np.cumsum(wts), w * wts.sum(), side="right"))
        assert inverse_cdf(wts, w) == min(ref, int(np.flatnonzero(wts > 0)[-1]))
    assert inverse_cdf(np.array([0.0, 2.0, 0.0, 1.0]), 0.0) == 1
    assert inverse_cdf(np.array([0.0, 2.0, 0.0, 1.0]), 0.999999) == 3


def _emitted_distribution(z0, t0, t1, T, grid=20001):
    """Distribution of the token emitted at position 0, with x ~ p and the uniforms
    integrated over a midpoint grid, using only the oracle's functions."""
    V = len(z0)
    p = softmax_t(z0, T)
    us = (np.arange(grid) + 0.5) / grid
    out = np.zeros(V)
    for x in range(V):
        # measure of the accepting uniforms
        acc = np.mean([sampled_accept([z0], [t0, t1], [x], T, [u], 0.5)[0] == 1 for u in us[::20]])
        # residual draw distribution over w
        _, _, wts = sampled_accept([z0], [t0, t1], [x], T, [1.0], 0.5)
        draws = np.bincount([inverse_cdf(wts, w) for w in us[::4]], minlength=V) / len(us[::4])
        out[x] += p[x] * acc
        out += p[x] * (1.0 - acc) * draws
    return out


@pytest.mark.parametrize("T", [0.7, 1.0, 1.8])
def test_speculative_sampling_emits_the_target_distribution(T):
    for _ in range(3):
        V = 5
        z0 = RNG.normal(0, 1.5, size=V)
        t0 = RNG.normal(0, 1.5, size=V)
        t1 = RNG.normal(0, 1.5, size=V)
        got = _emitted_distribution(z0, t0, t1, T)
        q = softmax_t(t0, T)
        assert np.allclose(got, q, atol=2e-3), (got, q)


def test_accept_rule_boundaries():
    z = np.array([0.0, 1.0, -1.0])
    t = np.array([0.5, 0.2, 0.1])
    p, q = softmax_t(z, 1.0), softmax_t(t, 1.0)
    for x in range(3):
        assert sampled_accept([z], [t, t], [x], 1.0, [0.0], 0.3)[0] == 1      # u = 0 always accepts
        L = sampled_accept([z], [t, t], [x], 1.0, [np.nextafter(1.0, 0.0)], 0.3)[0]
        assert L == (1 if p[x] < q[x] else 0)                                 # u -> 1: accept iff p < q


def test_equal_rows_always_accept_and_draw_from_q():
    z = RNG.normal(0, 2, size=50)
    for x in (0, 17, 49):
        L, tok, wts = sampled_accept([z, z], [z, z, z + 1.0], [x, x], 1.3, [0.999, 0.999], 0.42)
        assert L == 2
        assert tok == inverse_cdf(softmax_t(z + 1.0, 1.3), 0.42)
    # residual of identical distributions is all zero: fall back to q
    pq = softmax_t(z, 0.9)
    assert np.array_equal(residual(pq, pq), pq)


def test_residual_is_target_minus_draft_clipped():
    z, t = RNG.normal(size=30), RNG.normal(size=30)
    p, q = softmax_t(z, 1.0), softmax_t(t, 1.0)
    r = residual(p, q)
    assert np.all(r >= 0) and np.all((q > p) == (r > 0))
    assert abs(float(np.sum(r)) - 0.5 * float(np.sum(np.abs(q - p)))) < 1e-12  # total variation identity


def test_packed_batch_walks_requests():
    w = custom(vocab=64, k=[3, 1, 5], d_dtype="fp32", t_dtype="fp32")
    b = materialize(w)
    u = RNG.random(w.num_draft_rows)
    ws = RNG.random(w.num_requests)
    res = verify_sampled(b.draft_f64, b.target_f64, b.tokens, b.doff, 1.0, u, ws)
    for i in range(w.num_requests):
        d0, k = int(b.doff[i]), int(w.k[i])
        L, tok, _ = sampled_accept([b.draft_f64(d0 + j) for j in range(k)],
                                   [b.target_f64(d0 + i + j) for j in range(k + 1)],
                                   b.tokens[d0:d0 + k], 1.0, u[d0:d0 + k], ws[i])
        assert res[i]["accept_len"] == L and res[i]["next_token"] == tok
        assert 0 <= L <= k
