"""The plain C++ float64 oracle (``oracle/opd_ref.cpp``): its own pins, and
element-by-element agreement with the Python oracle on the generated workloads.

Its pins do not go through the Python oracle: brute force at 40 digits (sympy) on
V = 4 integer logits, the uniform-draft closed forms, central differences of its own
row loss, and the packed walk against an objective built from request blocks.  The
cross-check then compares every output of both oracles on the same stored inputs
(float64 on both sides; only the summation order differs).
"""

import math

import numpy as np
import pytest

import oracle
from oracle import cpp
from synth import make_workload, materialize
from synth.workloads import custom, draft_row, target_row

RNG = np.random.default_rng(4321)


def test_builds_and_loads():
    assert cpp.build()
    lib = cpp.lib()
    for name in ("oracle_row_forward", "oracle_row_grad", "oracle_verify_packed", "oracle_opd_rows"):
        assert hasattr(lib, name)


# ---------------------------------------------------------------------------
# pins of the C++ oracle on its own
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("c", [0.02, 0.3, 1.0, math.inf])
def test_kl_brute_force_v4(c):
    sympy = pytest.importorskip("sympy")
    for _ in range(40):
        z = RNG.integers(-2, 3, size=4)
        t = RNG.integers(-2, 3, size=4)
        Zp = sum(sympy.exp(sympy.Integer(int(v))) for v in z)
        Zq = sum(sympy.exp(sympy.Integer(int(v))) for v in t)
        terms = []
        for zv, tv in zip(z, t):
            p = sympy.exp(sympy.Integer(int(zv))) / Zp
            q = sympy.exp(sympy.Integer(int(tv))) / Zq
            terms.append(float((p * sympy.log(p / q)).evalf(40)))
        got = cpp.row_forward(z.astype(np.float64), t.astype(np.float64), c)
        assert abs(got["kl"] - sum(min(x, c) for x in terms)) < 1e-13
        assert got["n_clipped"] == sum(1 for x in terms if x > c)
        a = int(np.flatnonzero(t == t.max())[0])
        assert got["argmax"] == a
        want_ce = float((-sympy.log(sympy.exp(sympy.Integer(int(z[a]))) / Zp)).evalf(40))
        assert abs(got["ce"] - want_ce) < 1e-13


def test_closed_forms():
    for V in (1, 5, 1024):
        z = np.full(V, -0.5)
        t = RNG.normal(0, 3, size=V)
        r = cpp.row_forward(z, t, math.inf)
        assert abs(r["ce"] - math.log(V)) < 1e-12  # uniform draft: CE = log V
        want = float(np.log(np.sum(np.exp(t - t.max()))) + t.max() - np.mean(t) - math.log(V))
        assert abs(r["kl"] - want) < 1e-11  # uniform draft: KL = LSE(t) - mean(t) - log V
    z = RNG.normal(0, 3, size=300)
    eq = cpp.row_forward(z, z.copy(), 1.0)
    assert eq["kl"] == 0.0 and eq["n_clipped"] == 0
    p = np.exp(z - eq["lse_z"])
    a = int(np.argmax(z))
    want = p.copy()
    want[a] -= 1.0
    assert np.allclose(cpp.row_grad(z, z.copy(), 1.0, 1.0), want, atol=1e-15, rtol=0)  # equal rows: CE only


@pytest.mark.parametrize("c,beta", [(0.03, 1.0), (1.0, 0.4), (math.inf, 0.0)])
def test_grad_central_differences(c, beta):
    checked = 0
    for _ in range(6):
        V = 40
        z = RNG.normal(0, 2, size=V)
        t = RNG.normal(0, 2, size=V)
        z[:4] += 4.0
        t[:4] -= 4.0
        p = np.exp(z - np.log(np.sum(np.exp(z))))
        q = np.exp(t - np.log(np.sum(np.exp(t))))
        if np.any(np.abs(p * np.log(p / q) - c) < 1e-3):
            continue
        grad = cpp.row_grad(z, t, c, beta, 0.8)
        h = 1e-6
        for u in range(V):
            zp, zm = z.copy(), z.copy()
            zp[u] += h
            zm[u] -= h
            fd = 0.8 * (cpp.row_forward(zp, t, c, beta)["loss_row"] - cpp.row_forward(zm, t, c, beta)["loss_row"]) / (2 * h)
            assert abs(fd - grad[u]) <= 1e-6 + 1e-4 * abs(fd), (u, fd, grad[u])
        checked += 1
    assert checked >= 3


def test_packed_walk_against_block_objective():
    """The batch gradient with per-row weights (k = {4, 1, 3}) against central differences of
    J = sum over request blocks of g * loss_row, and the batch loss against J / N_d."""
    V, ks, c, beta = 16, [4, 1, 3], 0.35, 0.7
    blocks = []
    for k in ks:
        D = RNG.normal(0, 2, size=(k, V)).astype(np.float32)
        T = RNG.normal(0, 2, size=(k + 1, V)).astype(np.float32)
        D[:, :3] += 3.0
        T[:, :3] -= 3.0
        blocks.append((D, T))
    draft = np.concatenate([D for D, _ in blocks])
    target = np.concatenate([T for _, T in blocks])
    doff = np.array([0, 4, 5, 8], dtype=np.int32)
    g = RNG.uniform(0.5, 2.0, size=8)

    def J(bl, w):
        tot, d = 0.0, 0
        for D, T in bl:
            for j in range(len(D)):
                tot += w[d] * cpp.row_forward(D[j].astype(np.float64), T[j].astype(np.float64), c, beta)["loss_row"]
                d += 1
        return tot

    _, grads, loss = cpp.opd_rows(draft, "fp32", target, "fp32", doff, V, c, beta, grad=True, grad_row=g)
    assert abs(loss - J(blocks, np.ones(8)) / 8) < 1e-13
    h = 1e-4  # the rows are float32 storage; differences are taken in float64 on the widened values
    d = 0
    checked = 0
    for i, (D, T) in enumerate(blocks):
        for j in range(len(D)):
            row = D[j].astype(np.float64)
            tr = T[j].astype(np.float64)
            f0 = cpp.row_forward(row, tr, c, beta)
            p = np.exp(row - f0["lse_z"])
            r = (row - f0["lse_z"]) - (tr - f0["lse_t"])
            if np.all(np.abs(p * r - c) > 1e-2):
                for u in range(V):
                    zp, zm = row.copy(), row.copy()
                    zp[u] += h
                    zm[u] -= h
                    fd = g[d] * (cpp.row_forward(zp, tr, c, beta)["loss_row"] -
                                 cpp.row_forward(zm, tr, c, beta)["loss_row"]) / (2 * h)
                    assert abs(fd - grads[d][u]) <= 1e-6 + 1e-4 * abs(fd), (i, j, u)
                checked += 1
            d += 1
    assert checked >= 5


# ---------------------------------------------------------------------------
# agreement with the Python oracle
# ---------------------------------------------------------------------------

REL, ABS = 1e-11, 1e-13
GREL, GABS = 1e-9, 1e-15


def _same_row(a, b):
    for key in ("kl", "ce", "loss_row", "lse_z", "lse_t", "S", "S_l1"):
        assert abs(a[key] - b[key]) <= REL * abs(b[key]) + ABS * (1 + b.get("S_l1", 0.0)), (key, a[key], b[key])
    assert a["argmax"] == b["argmax"]
    assert a["n_clipped"] == b["n_clipped"]


def _check_batch(b, threads=4, grad=True):
    w = b.w
    per, grads, loss = cpp.opd_rows(b.draft, w.d_dtype, b.target, w.t_dtype, b.doff, w.vocab, w.clip_c,
                                    w.ce_weight, grad=grad, threads=threads)
    ref_per, ref_loss = oracle.opd_loss_fwd(b.draft_f64, b.target_f64, b.doff, w.clip_c, w.ce_weight)
    for d in range(w.num_draft_rows):
        _same_row(per[d], ref_per[d])
    assert abs(loss - ref_loss) <= REL * abs(ref_loss)
    if grad:
        ref_g = oracle.opd_loss_bwd(b.draft_f64, b.target_f64, b.doff, w.clip_c, w.ce_weight)
        for d in range(w.num_draft_rows):
            assert np.all(np.abs(grads[d] - ref_g[d]) <= GABS + GREL * np.abs(ref_g[d])), d
    am, L, bonus, rate = cpp.verify_packed(b.target, w.t_dtype, b.tokens, b.doff, w.vocab, threads=threads)
    ver = oracle.verify_packed(b.target_f64, b.tokens, b.doff)
    for i in range(w.num_requests):
        v = ver[i]
        assert L[i] == v["accept_len"] and bonus[i] == v["bonus_token"]
        assert rate[i].view(np.uint32) == np.float32(v["accept_rate"]).view(np.uint32)
        assert np.array_equal(am[v["target_rows"]], v["target_argmax"])


def test_agrees_on_tiny():
    _check_batch(materialize(make_workload("tiny")))


@pytest.mark.parametrize("dd,td", [("bf16", "bf16"), ("fp32", "bf16"), ("bf16", "fp32")])
def test_agrees_on_mixed_dtypes_and_padded_rows(dd, td):
    w = custom(vocab=777, k=[3, 16, 1, 7], d_dtype=dd, t_dtype=td, clip_c=0.3, ce_weight=0.6, ld_d=800, ld_t=781)
    _check_batch(materialize(w))


def test_agrees_on_first_requests_of_the_stress_batch():
    """V = 151937, float32 draft / bfloat16 target: the first three requests of the stress batch."""
    w = make_workload("stress")
    sub = make_workload("stress", k=w.k[:3], planted_accept=w.planted_accept[:3],
                        tie_rows=np.zeros(0, np.int64), equal_rows=np.zeros(0, np.int64))
    _check_batch(materialize(sub), threads=8, grad=False)


def test_agrees_on_stress_tie_and_equal_rows_and_binding_clip():
    w = make_workload("stress")
    for s in list(w.tie_rows[:3]):
        t = target_row(w, int(s)).astype(np.float64)
        d = w.draft_of_target(int(s))
        z = draft_row(w, d).astype(np.float64) if d >= 0 else RNG.normal(0, 3, size=w.vocab)
        _same_row(cpp.row_forward(z, t, w.clip_c), oracle.row_forward(z, t, w.clip_c))
    for d in list(w.equal_rows[:3]):
        t = target_row(w, w.pair_target_row(int(d))).astype(np.float64)
        z = draft_row(w, int(d)).astype(np.float64)
        got = cpp.row_forward(z, t, w.clip_c)
        assert got["kl"] == 0.0
        _same_row(got, oracle.row_forward(z, t, w.clip_c))
    wc = make_workload("c128_clip")
    for d in list(wc.clip_rows[:2]):
        t = target_row(wc, wc.pair_target_row(int(d))).astype(np.float64)
        z = draft_row(wc, int(d)).astype(np.float64)
        got = cpp.row_forward(z, t, wc.clip_c)
        assert got["n_clipped"] == 64
        _same_row(got, oracle.row_forward(z, t, wc.clip_c))
        gg = cpp.row_grad(z, t, wc.clip_c, 1.0)
        gr = oracle.row_grad(z, t, wc.clip_c, 1.0)
        assert np.all(np.abs(gg - gr) <= GABS + GREL * np.abs(gr))
