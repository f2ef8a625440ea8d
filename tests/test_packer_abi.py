"""The library's host packer (adaflash_packer_*) against the packing oracle, on CPU.

The packer touches no GPU, so it is compared here on synthetic request streams:
every round's admitted count, offsets, capacity and rows must equal the oracle's,
and the float64 estimate must match bit for bit (same operations, same order).
"""

import ctypes

import numpy as np
import pytest

from oracle.packing import Packer as OraclePacker
from serving_packed_var_gb300 import _native
from serving_packed_var_gb300.build import build


@pytest.fixture(scope="module")
def af():
    build()
    import serving_packed_var_gb300 as m
    return m


def _stream(seed, rounds, max_arrivals, dist):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(rounds):
        n = int(rng.integers(0, max_arrivals + 1))
        if dist == "uniform":
            k = rng.integers(1, 17, size=n)
        elif dist == "short":
            k = np.minimum(16, 1 + rng.geometric(0.4, size=n))
        else:  # bursts of full-length drafts
            k = np.where(rng.random(n) < 0.7, 16, rng.integers(1, 5, size=n))
        out.append([int(x) for x in k])
    return out


@pytest.mark.parametrize("budget,alpha,e0,dist", [
    (33, 1.0, 33.0, "uniform"), (300, 0.2, 17.0, "uniform"), (1042 + 914, 0.1, 10.0, "short"),
    (4000, 0.5, 40.0, "burst"), (777, 0.05, 5.0, "burst"),
])
def test_matches_oracle_over_a_stream(af, budget, alpha, e0, dist):
    arrivals = _stream(budget * 7 + len(dist), 50, 80, dist)
    lib = af.Packer(budget, alpha, e0)
    ref = OraclePacker(budget, alpha, e0)
    q = []
    for r in range(80):
        if r < len(arrivals):
            q.extend(arrivals[r])
        got = lib.plan(q)
        admitted, offsets, cap, rows = ref.plan(q)
        assert got["admitted"] == admitted and got["capacity"] == cap and got["rows"] == rows, r
        assert list(got["draft_offsets"]) == offsets, r
        lib.observe(got["rows"], got["admitted"])
        ref.observe(rows, admitted)
        assert np.float64(lib.estimate).view(np.uint64) == np.float64(ref.e).view(np.uint64), r
        q = q[admitted:]
    lib.close()


def test_empty_queue_and_zero_requests(af):
    p = af.Packer(100, 0.3, 12.0)
    got = p.plan([])
    assert got["admitted"] == 0 and got["capacity"] == 0 and got["rows"] == 0 and list(got["draft_offsets"]) == [0]
    p.observe(0, 0)
    assert p.estimate == 12.0


def test_rejects_bad_arguments(af):
    lib = _native.lib()
    h = ctypes.c_void_p()
    INVALID = _native.ADAFLASH_ERR_INVALID_ARG
    assert lib.adaflash_packer_create(32, 0.2, 10.0, ctypes.byref(h)) == INVALID   # a k = 16 request must fit
    assert lib.adaflash_packer_create(100, 0.0, 10.0, ctypes.byref(h)) == INVALID
    assert lib.adaflash_packer_create(100, 1.5, 10.0, ctypes.byref(h)) == INVALID
    assert lib.adaflash_packer_create(100, 0.5, 0.0, ctypes.byref(h)) == INVALID
    assert lib.adaflash_packer_create(100, 0.5, float("nan"), ctypes.byref(h)) == INVALID
    assert lib.adaflash_packer_create(100, 0.5, 10.0, None) == INVALID
    p = af.Packer(100, 0.5, 10.0)
    for bad in ([0], [17], [3, -1]):
        with pytest.raises(af.AdaflashError):
            p.plan(bad)
    assert lib.adaflash_packer_observe(p._h, -1, 3) == INVALID
