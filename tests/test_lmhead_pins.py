"""Pins of the logit-free oracle (oracle/lmhead.py) and of the LM-head generator.

* head_logits against a pure-Python integer brute force on non-square integer
  inputs (catches a transposed operand or a wrong index);
* the composed row forward against the logits oracle on those exact logits;
* the generator's planted structure: the spike token is the target's argmax in most
  rows, and where it is in all of a request's rows greedy verification finds the
  planted prefix.
"""

import numpy as np

from oracle import opd
from oracle.lmhead import head_logits, row_forward, verify_packed
from synth.lmhead import make_lmhead_workload, materialize_lmhead

RNG = np.random.default_rng(5)


def _brute(h, w):
    return [[sum(int(h[r][k]) * int(w[v][k]) for k in range(len(h[r]))) for v in range(len(w))] for r in range(len(h))]


def test_head_logits_integer_brute_force():
    for n, H, V in ((1, 3, 5), (3, 7, 2), (2, 16, 11)):
        h = RNG.integers(-8, 9, size=(n, H))
        w = RNG.integers(-8, 9, size=(V, H))
        got = head_logits(h.astype(np.float64), w.astype(np.float32))
        assert got.shape == (n, V)
        assert np.array_equal(got, np.array(_brute(h.tolist(), w.tolist()), dtype=np.float64))


def test_row_forward_is_the_logits_oracle_on_head_logits():
    H, V = 6, 9
    hd = RNG.integers(-3, 4, size=H).astype(np.float64) / 4
    ht = RNG.integers(-3, 4, size=H).astype(np.float64) / 4
    wd = RNG.integers(-3, 4, size=(V, H)).astype(np.float32)
    wt = RNG.integers(-3, 4, size=(V, H)).astype(np.float32)
    z = np.array(_brute([list((hd * 4).astype(int))], wd.astype(int).tolist())[0], dtype=np.float64) / 4
    t = np.array(_brute([list((ht * 4).astype(int))], wt.astype(int).tolist())[0], dtype=np.float64) / 4
    for c in (0.05, 1.0, np.inf):
        a = row_forward(hd, ht, wd, wt, c, 0.7)
        b = opd.row_forward(z, t, c, 0.7)
        for key in ("kl", "ce", "lse_z", "lse_t", "S"):
            assert abs(a[key] - b[key]) <= 1e-12 * (1 + abs(b[key])), key
        assert a["argmax"] == b["argmax"] and a["n_clipped"] == b["n_clipped"]


def test_generator_plants_the_target_argmax_and_the_prefix():
    # The spike lifts one logit per target row well above the bulk; it is the argmax
    # of most rows (its own noise can sink it in a few), and where every target row of
    # a request peaks at its spike, greedy verification finds the planted prefix.
    w = make_lmhead_workload("lm_tiny")
    b = materialize_lmhead(w)
    ht = b.f32("ht")
    wt = b.f32("wt")
    t = head_logits(ht, wt)
    hits = [opd.first_argmax(t[s]) == b.spike_token[s] for s in range(w.num_target_rows)]
    assert np.mean(hits) >= 0.8
    res = verify_packed(lambda s: ht[s], wt, b.tokens, b.doff)
    checked = 0
    for i in range(w.num_requests):
        d0, k = int(b.doff[i]), int(w.k[i])
        if all(hits[d0 + i + j] for j in range(k + 1)):
            assert res[i]["accept_len"] == w.planted_accept[i]
            checked += 1
    assert checked >= 1
