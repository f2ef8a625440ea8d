"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle against a fact the mathematics or the construction
of the inputs fixes: brute force on tiny inputs (high-precision sympy or
unshifted exact sums), closed forms of special cases, invariants, central finite
differences, and the accept prefixes the generator plants.  A plausible slip in
the oracle (a dropped term, a sign, a swapped operand, a wrong index) fails at
least one of them.
"""

import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle.opd import clipped_reverse_kl_terms
from synth import materialize, make_workload
from synth.workloads import custom

sympy = pytest.importorskip("sympy")

RNG = np.random.default_rng(12345)


# ---------------------------------------------------------------------------
# argmax: brute force and planted ties
# ---------------------------------------------------------------------------

def test_first_argmax_brute_force():
    for _ in range(2000):
        n = int(RNG.integers(1, 12))
        x = RNG.integers(-3, 4, size=n).astype(np.float64)  # many ties
        best = 0
        for v in range(1, n):
            if x[v] > x[best]:
                best = v
        assert oracle.first_argmax(x) == best


def test_first_argmax_signed_zero_and_all_equal():
    assert oracle.first_argmax(np.array([-0.0, 0.0, -1.0])) == 0
    assert oracle.first_argmax(np.array([0.0, -0.0])) == 0
    assert oracle.first_argmax(np.full(17, 2.5)) == 0


def test_first_argmax_planted_ties():
    w = make_workload("stress")
    # only the tie rows matter here: build them one by one
    from synth.workloads import target_row
    for s in list(w.tie_rows[:6]):
        x = target_row(w, int(s)).astype(np.float64)
        top = np.flatnonzero(x == x.max())
        assert len(top) >= 2, "a tie row carries two equal maxima"
        assert oracle.first_argmax(x) == top[0]


# ---------------------------------------------------------------------------
# log-sum-exp and cross-entropy
# ---------------------------------------------------------------------------

def _lse_sympy(x):
    return float(sympy.log(sum(sympy.exp(sympy.Integer(int(v))) for v in x)).evalf(40))


def test_lse_brute_force_small_integers():
    for _ in range(200):
        n = int(RNG.integers(1, 9))
        x = RNG.integers(-6, 7, size=n)
        assert abs(oracle.log_sum_exp(x.astype(np.float64)) - _lse_sympy(x)) < 1e-13


def test_lse_shift_invariance_large_offsets():
    x = RNG.normal(0, 3, size=300)
    base = oracle.log_sum_exp(x)
    for s in (-1000.0, 1000.0, 1e5):
        assert abs(oracle.log_sum_exp(x + s) - (base + s)) < 1e-9 * max(1.0, abs(s))


def test_ce_uniform_draft_is_log_v():
    for V in (1, 2, 7, 1024, 151936):
        z = np.full(V, 0.375)
        for a in (0, V - 1):
            assert abs(oracle.hard_label_ce(z, a) - math.log(V)) < 1e-12


def test_ce_brute_force():
    for _ in range(100):
        n = int(RNG.integers(2, 7))
        z = RNG.integers(-4, 5, size=n)
        a = int(RNG.integers(n))
        Z = sum(sympy.exp(sympy.Integer(int(v))) for v in z)
        want = float((-sympy.log(sympy.exp(sympy.Integer(int(z[a]))) / Z)).evalf(40))
        assert abs(oracle.hard_label_ce(z.astype(np.float64), a) - want) < 1e-13


# ---------------------------------------------------------------------------
# clipped reverse KL
# ---------------------------------------------------------------------------

def _rkl_terms_sympy(z, t):
    Zp = sum(sympy.exp(sympy.Integer(int(v))) for v in z)
    Zq = sum(sympy.exp(sympy.Integer(int(v))) for v in t)
    out = []
    for zv, tv in zip(z, t):
        p = sympy.exp(sympy.Integer(int(zv))) / Zp
        q = sympy.exp(sympy.Integer(int(tv))) / Zq
        out.append(float((p * sympy.log(p / q)).evalf(40)))
    return out


@pytest.mark.parametrize("c", [0.02, 0.1, 0.3, 1.0, math.inf])
def test_clipped_kl_brute_force_v4_grid(c):
    """V = 4, logits drawn from {-2..2}: KL = sum_v min(p_v log(p_v/q_v), c) at 40 digits."""
    for _ in range(60):
        z = RNG.integers(-2, 3, size=4)
        t = RNG.integers(-2, 3, size=4)
        terms = _rkl_terms_sympy(z, t)
        want = sum(min(x, c) for x in terms)
        got = oracle.row_forward(z.astype(np.float64), t.astype(np.float64), c)
        assert abs(got["kl"] - want) < 1e-13
        assert got["n_clipped"] == sum(1 for x in terms if x > c)


def test_unclipped_kl_nonnegative_and_zero_on_equal_rows():
    for _ in range(50):
        V = int(RNG.integers(2, 400))
        z = RNG.normal(0, 3, size=V)
        t = RNG.normal(0, 3, size=V)
        assert oracle.row_forward(z, t, math.inf)["kl"] >= -1e-15
        res = oracle.row_forward(z, z.copy(), 1.0)
        assert res["kl"] == 0.0
        assert res["n_clipped"] == 0


def test_kl_uniform_draft_closed_form():
    """p uniform: KL(p||q) = LSE(t) - mean(t) - log V."""
    for V in (3, 64, 1024):
        t = RNG.normal(0, 3, size=V)
        z = np.full(V, -1.25)
        want = oracle.log_sum_exp(t) - float(np.mean(t)) - math.log(V)
        assert abs(oracle.row_forward(z, t, math.inf)["kl"] - want) < 1e-11


def test_clip_monotone_in_c_and_limits():
    z = RNG.normal(0, 3, size=256)
    t = RNG.normal(0, 3, size=256)
    z[:5] += 9.0
    t[:5] -= 9.0
    vals = [oracle.row_forward(z, t, c)["kl"] for c in (1e-4, 1e-2, 0.1, 0.5, 2.0, 1e9)]
    assert all(a <= b + 1e-15 for a, b in zip(vals, vals[1:]))
    assert abs(vals[-1] - oracle.row_forward(z, t, math.inf)["kl"]) < 1e-15
    # c -> 0+: every positive term is replaced by (almost) 0, negative terms stay
    p, r, term = clipped_reverse_kl_terms(z, t)
    assert abs(oracle.row_forward(z, t, 1e-12)["kl"] - float(np.sum(np.minimum(term, 0.0)))) < 1e-9


def test_clip_binds_on_exactly_the_planted_entries():
    """Draft +16 / target -30 on 64 entries at c = 0.5: those 64 terms (about 0.65) clip."""
    from synth.workloads import draft_row, target_row
    w = make_workload("c128_clip")
    for d in list(w.clip_rows[:3]):
        s = w.pair_target_row(int(d))
        t = target_row(w, s).astype(np.float64)
        z = draft_row(w, int(d)).astype(np.float64)
        res = oracle.row_forward(z, t, w.clip_c)
        assert res["n_clipped"] == 64
        p, r, term = clipped_reverse_kl_terms(z, t)
        planted = np.flatnonzero(t == -30.0)
        assert set(np.flatnonzero(term > w.clip_c)) == set(planted)
    # the +6 variant does not reach c = 0.5 on these rows
    w6 = make_workload("c128")
    d = int(w6.clip_rows[0])
    res = oracle.row_forward(draft_row(w6, d).astype(np.float64),
                             target_row(w6, w6.pair_target_row(d)).astype(np.float64), w6.clip_c)
    assert res["n_clipped"] == 0


# ---------------------------------------------------------------------------
# gradient
# ---------------------------------------------------------------------------

def _row_loss(z, t, c, beta):
    return oracle.row_forward(z, t, c, beta)["loss_row"]


def _fd_check(z, t, c, beta, g=1.0, h=1e-5, idx=None):
    _, _, term = clipped_reverse_kl_terms(z, t)
    if np.any(np.abs(term - c) < 1e-3):
        return False  # the kink of the clip is too close for a central difference
    grad = oracle.row_grad(z, t, c, beta, g)
    idx = range(len(z)) if idx is None else idx
    for u in idx:
        zp = z.copy(); zp[u] += h
        zm = z.copy(); zm[u] -= h
        fd = g * (_row_loss(zp, t, c, beta) - _row_loss(zm, t, c, beta)) / (2 * h)
        assert abs(fd - grad[u]) <= 1e-6 + 1e-4 * abs(fd), (u, fd, grad[u])
    return True


def test_grad_finite_differences_tiny_workload():
    b = materialize(make_workload("tiny"))
    w = b.w
    checked = 0
    for d in range(w.num_draft_rows):
        z = b.draft_f64(d)
        t = b.target_f64(w.pair_target_row(d))
        idx = list(RNG.choice(w.vocab, size=24, replace=False)) + [oracle.first_argmax(t)]
        if _fd_check(z, t, w.clip_c, 1.0, g=0.7, idx=idx):
            checked += 1
    assert checked >= 20


@pytest.mark.parametrize("c,beta", [(0.02, 1.0), (0.05, 0.0), (math.inf, 0.3)])
def test_grad_finite_differences_clip_binding(c, beta):
    hit = 0
    for _ in range(8):
        V = 48
        z = RNG.normal(0, 2, size=V)
        t = RNG.normal(0, 2, size=V)
        z[:4] += 4.0
        t[:4] -= 4.0
        if _fd_check(z, t, c, beta):
            hit += 1
            if c < 1:
                assert oracle.row_forward(z, t, c)["n_clipped"] > 0
    assert hit >= 4


def test_grad_rows_sum_to_zero():
    for c in (0.05, 1.0, math.inf):
        z = RNG.normal(0, 3, size=500)
        t = RNG.normal(0, 3, size=500)
        assert abs(float(np.sum(oracle.row_grad(z, t, c, 1.0)))) < 1e-12


def test_grad_closed_form_unclipped_kl_only():
    """c = inf, beta = 0: d KL(p||q) / dz = p (r - KL)."""
    z = RNG.normal(0, 3, size=300)
    t = RNG.normal(0, 3, size=300)
    p, r, _ = clipped_reverse_kl_terms(z, t)
    kl = oracle.row_forward(z, t, math.inf)["kl"]
    assert np.allclose(oracle.row_grad(z, t, math.inf, 0.0), p * (r - kl), atol=1e-14, rtol=0)


def test_grad_equal_rows_is_ce_only():
    z = RNG.normal(0, 3, size=300)
    p = np.exp(z - oracle.log_sum_exp(z))
    a = oracle.first_argmax(z)
    want = p.copy(); want[a] -= 1.0
    assert np.allclose(oracle.row_grad(z, z.copy(), 1.0, 1.0), want, atol=1e-15, rtol=0)


# ---------------------------------------------------------------------------
# verification: planted answers and the acceptance rate
# ---------------------------------------------------------------------------

def _nearest_f32(fr: Fraction) -> np.float32:
    f = np.float32(float(fr))
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    return min(cands, key=lambda x: (abs(Fraction(float(x)) - fr), int(np.float32(x).view(np.uint32)) & 1))


def test_acceptance_rate_is_correctly_rounded():
    for k in range(1, 17):
        for L in range(0, k + 1):
            assert oracle.acceptance_rate(L, k) == _nearest_f32(Fraction(L, k))


@pytest.mark.parametrize("name", ["tiny", "single", "c32"])
def test_verify_reproduces_planted_prefix(name):
    b = materialize(make_workload(name))
    w = b.w
    res = oracle.verify_packed(b.target_f64, b.tokens, b.doff)
    for i in range(w.num_requests):
        assert res[i]["accept_len"] == int(w.planted_accept[i])
        assert res[i]["bonus_token"] == int(b.gen_argmax[w.doff[i] + i + w.planted_accept[i]])
        assert 0 <= res[i]["accept_len"] <= int(w.k[i])


def test_verify_edge_prefixes():
    for accept in ("full", "none"):
        w = custom(vocab=40, k=[1, 16, 5], accept=accept, d_dtype="fp32", t_dtype="fp32")
        b = materialize(w)
        res = oracle.verify_packed(b.target_f64, b.tokens, b.doff)
        for i in range(w.num_requests):
            assert res[i]["accept_len"] == int(w.planted_accept[i])


def test_loss_is_mean_over_draft_rows():
    """Two copies of the same request: the batch loss equals one copy's mean."""
    w = custom(vocab=64, k=[5], d_dtype="fp32", t_dtype="fp32")
    b = materialize(w)
    per, loss1 = oracle.opd_loss_fwd(b.draft_f64, b.target_f64, b.doff, 1.0)
    doff2 = np.array([0, 5, 10])
    dr = lambda d: b.draft_f64(d % 5)
    tr = lambda s: b.target_f64(s % 6)
    per2, loss2 = oracle.opd_loss_fwd(dr, tr, doff2, 1.0)
    assert abs(loss1 - loss2) < 1e-14
    assert abs(loss1 * 5 - sum(per[d]["kl"] + per[d]["ce"] for d in range(5))) < 1e-12


# ---------------------------------------------------------------------------
# the packed batch walk of the forward and the gradient
# ---------------------------------------------------------------------------

def _packed_blocks(ks, V, rng):
    """Per-request blocks (k_i draft rows, k_i + 1 target rows) with some clipped terms."""
    blocks = []
    for k in ks:
        D = rng.normal(0, 2, size=(k, V))
        T = rng.normal(0, 2, size=(k + 1, V))
        D[:, :3] += 3.0
        T[:, :3] -= 3.0
        blocks.append((D, T))
    return blocks


def _blocks_objective(blocks, g, c, beta):
    """J = sum over requests i and positions j < k_i of g * loss_row(D_i[j], T_i[j]).

    Written from the blocks themselves (position j of a request pairs its j-th draft row
    with its j-th target row), not through the packed offsets the oracle walks."""
    total, d = 0.0, 0
    for D, T in blocks:
        for j in range(len(D)):
            total += g[d] * oracle.row_forward(D[j], T[j], c, beta)["loss_row"]
            d += 1
    return total


def test_packed_walk_forward_and_gradient_against_the_block_objective():
    """opd_loss_fwd's batch loss and opd_loss_bwd's packed gradient on three requests of
    k = {4, 1, 3} with per-row upstream weights, against the objective built from the
    request blocks and its central differences.  Pairing draft row d with target row d
    (instead of d + i), or weighting by request instead of by row, fails here."""
    rng = np.random.default_rng(2024)
    V, ks, c, beta = 20, [4, 1, 3], 0.35, 0.7
    blocks = _packed_blocks(ks, V, rng)
    draft = np.concatenate([D for D, _ in blocks])
    target = np.concatenate([T for _, T in blocks])
    doff = np.array([0, 4, 5, 8])
    Nd = 8
    g = rng.uniform(0.5, 2.0, size=Nd)

    # the forward's batch loss is the unweighted objective over N_d
    _, loss = oracle.opd_loss_fwd(lambda d: draft[d], lambda s: target[s], doff, c, beta)
    assert abs(loss - _blocks_objective(blocks, np.ones(Nd), c, beta) / Nd) < 1e-13

    grad = oracle.opd_loss_bwd(lambda d: draft[d], lambda s: target[s], doff, c, beta, grad_row=g)
    assert sorted(grad) == list(range(Nd))
    h, checked, clipped = 1e-6, 0, 0
    d = 0
    for i, (D, T) in enumerate(blocks):
        for j in range(len(D)):
            _, _, term = clipped_reverse_kl_terms(D[j], T[j])
            clipped += int(np.count_nonzero(term > c))
            if np.any(np.abs(term - c) < 1e-3):
                d += 1
                continue  # the clip's kink is too close for a central difference
            for u in range(V):
                Dp = [(Dk.copy(), Tk) for Dk, Tk in blocks]
                Dm = [(Dk.copy(), Tk) for Dk, Tk in blocks]
                Dp[i][0][j, u] += h
                Dm[i][0][j, u] -= h
                fd = (_blocks_objective(Dp, g, c, beta) - _blocks_objective(Dm, g, c, beta)) / (2 * h)
                assert abs(fd - grad[d][u]) <= 1e-6 + 1e-4 * abs(fd), (i, j, u, fd, grad[d][u])
            checked += 1
            d += 1
    assert checked >= 6 and clipped > 0


def test_packed_gradient_scalar_weight_is_the_mean_loss_gradient():
    """grad_scale = 1 / N_d gives the gradient of opd_loss_fwd's mean loss (central differences
    through the packed forward itself, on a request of k = 1 between two longer ones)."""
    rng = np.random.default_rng(99)
    V, ks, c, beta = 12, [3, 1, 2], 0.5, 1.0
    blocks = _packed_blocks(ks, V, rng)
    draft = np.concatenate([D for D, _ in blocks])
    target = np.concatenate([T for _, T in blocks])
    doff = np.array([0, 3, 4, 6])
    Nd = 6
    grad = oracle.opd_loss_bwd(lambda d: draft[d], lambda s: target[s], doff, c, beta, grad_scale=1.0 / Nd)
    h = 1e-6
    for d in (0, 3, 5):
        for u in range(V):
            zp, zm = draft.copy(), draft.copy()
            zp[d, u] += h
            zm[d, u] -= h
            lp = oracle.opd_loss_fwd(lambda r: zp[r], lambda s: target[s], doff, c, beta)[1]
            lm = oracle.opd_loss_fwd(lambda r: zm[r], lambda s: target[s], doff, c, beta)[1]
            fd = (lp - lm) / (2 * h)
            assert abs(fd - grad[d][u]) <= 1e-7 + 1e-4 * abs(fd), (d, u, fd, grad[d][u])
