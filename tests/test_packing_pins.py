"""Pins of the packing oracle (oracle/packing.py) against what the arithmetic fixes.

* the EMA against its closed form after n equal observations;
* the admitted count against a brute-force search over queue prefixes;
* a hand-worked round;
* serving-stream invariants: never over budget, FIFO order, nothing lost or repeated;
* the steady state under a constant length.
"""

import math

import numpy as np
import pytest

from oracle.packing import MAX_K, Packer, capacity, ema_update, plan, rows_of, simulate

RNG = np.random.default_rng(11)


@pytest.mark.parametrize("alpha", [0.05, 0.2, 0.5, 1.0])
def test_ema_closed_form(alpha):
    e0, x = 40.0, 13.0
    e = e0
    for n in range(1, 60):
        e = ema_update(e, x, alpha)
        assert abs(e - (x + (1 - alpha) ** n * (e0 - x))) <= 1e-12 * max(1.0, abs(e0))


def test_hand_worked_round():
    # budget 100, estimate 20 rows per request: capacity 5; rows 33+33+33+3+3 = 105 > 100,
    # give back the two k = 1 requests: 99 rows, 3 requests, offsets 0, 16, 32, 48
    admitted, offsets, cap, rows = plan(100, 20.0, [16, 16, 16, 1, 1, 4])
    assert (admitted, offsets, cap, rows) == (3, [0, 16, 32, 48], 5, 99)
    assert capacity(100, 20.0, 6) == 5 and capacity(100, 1000.0, 6) == 1 and capacity(100, 0.5, 6) == 6
    assert rows_of(16) == 33 and rows_of(1) == 3


def test_admitted_is_the_longest_prefix_within_capacity_and_budget():
    for _ in range(400):
        n = int(RNG.integers(0, 12))
        q = list(RNG.integers(1, MAX_K + 1, size=n))
        budget = int(RNG.integers(33, 200))
        e = float(RNG.uniform(3.0, 40.0))
        admitted, offsets, cap, rows = plan(budget, e, q)
        # brute force over prefixes
        best = 0
        for a in range(0, min(n, cap) + 1):
            if sum(2 * k + 1 for k in q[:a]) <= budget:
                best = a
        assert admitted == best
        assert rows == sum(2 * k + 1 for k in q[:admitted]) <= budget
        assert offsets == list(np.concatenate([[0], np.cumsum(q[:admitted])]).astype(int))
        assert cap == (0 if n == 0 else max(1, min(n, math.floor(budget / e))))


def test_stream_invariants():
    arrivals = [list(RNG.integers(1, MAX_K + 1, size=int(RNG.integers(0, 40)))) for _ in range(30)]
    out = simulate(300, 0.3, 17.0, arrivals, 60)
    served = []
    for admitted, offsets, cap, rows, e in out:
        assert rows <= 300 and admitted <= cap
        served.extend(int(b - a) for a, b in zip(offsets[:-1], offsets[1:]))
    flat = [int(k) for a in arrivals for k in a]
    assert served == flat[:len(served)]          # FIFO, nothing lost or repeated
    assert len(served) == len(flat)              # the queue drains within 60 rounds


def test_steady_state_constant_length():
    p = Packer(500, 0.5, 3.0)
    for _ in range(80):
        admitted, offsets, cap, rows = p.plan([7] * 1000)
        p.observe(rows, admitted)
    assert abs(p.e - rows_of(7)) < 1e-9
    assert cap == 500 // 15 and admitted == cap and rows == cap * 15
