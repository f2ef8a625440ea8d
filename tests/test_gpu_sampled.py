"""Temperature-sampled verification: CUDA path vs the float64 oracle (oracle/sampling.py).

Both sides decide from the same float32 uniforms.  A decision is compared exactly
unless the float64 margin that decides it is within float32 rounding of zero:

  accept at position j   -- |u_j p(x_j) - q(x_j)| <= 1e-5 max(q, u p), else exact;
  inverse-CDF draw       -- the GPU's token must have weight >= -1e-5 (p + q) and lie
                            within 1e-4 * total of the threshold w * total (its CDF
                            interval, widened by that much), else it must be exact.

Such near-ties are rare with random uniforms; each test also bounds how many
requests may take the tolerant branch.  row_lse is compared with float64
log-sum-exp(x / T) to 1e-6 relative + 2e-5 absolute.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from concurrent.futures import ThreadPoolExecutor  # noqa: E402

from oracle.opd import log_sum_exp  # noqa: E402
from oracle.sampling import inverse_cdf, residual, sampled_accept, softmax_t  # noqa: E402
from parity_lib import THREADS, to_device  # noqa: E402
from synth import make_workload, materialize  # noqa: E402
from synth.workloads import bf16_bits_to_f32, custom, f32_to_bf16_bits  # noqa: E402

ACCEPT_REL = 1e-5
DRAW_REL = 1e-4
LSE_REL, LSE_ABS = 1e-6, 2e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def uniforms(w, seed):
    rng = np.random.default_rng(seed)
    u = rng.random(w.num_draft_rows, dtype=np.float32)
    ws = rng.random(w.num_requests, dtype=np.float32)
    return u, ws


class SampledRun:
    def __init__(self, b, T, u, ws, misalign=0, canary=16):
        import serving_packed_var_gb300 as af
        w = b.w
        dev = torch.device("cuda:0")
        self.z = to_device(b.draft, w.d_dtype, dev, misalign)
        self.t = to_device(b.target, w.t_dtype, dev, misalign)
        tok = torch.from_numpy(b.tokens).to(dev)
        doff = torch.from_numpy(b.doff).to(dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        R, Nd = w.num_requests, w.num_draft_rows
        self._bufs = {}

        def buf(name, n, dtype, fill):
            full = torch.full((n + canary,), fill, dtype=dtype, device=dev)
            self._bufs[name] = (full, n, fill)
            return full[:n]

        out = dict(row_lse=buf("row_lse", 2 * Nd + R, torch.float32, -7.0),
                   accept_len=buf("accept_len", R, torch.int32, -7),
                   next_token=buf("next_token", R, torch.int32, -7),
                   accept_rate=buf("accept_rate", R, torch.float32, -7.0))
        ua = torch.from_numpy(np.ascontiguousarray(u, dtype=np.float32)).to(dev)
        us = torch.from_numpy(np.ascontiguousarray(ws, dtype=np.float32)).to(dev)
        self.out = af.adaflash_verify_sampled(self.z, self.t, tok, doff, T, ua, us, vocab=w.vocab, out=out,
                                              status=self.status)
        torch.cuda.synchronize()
        self.h = {k: v.cpu().numpy() for k, v in self.out.items()}
        self.status_word = int(self.status.item())

    def canaries_intact(self):
        for name, (full, n, fill) in self._bufs.items():
            if not bool((full[n:].cpu() == fill).all()):
                return name
        return None


def _draw_ok(weights, w, g, ref_tok, pq_scale):
    """The GPU's draw g is the oracle's, or lies on the oracle's CDF within rounding of w * total."""
    if g == ref_tok:
        return True, False
    if not (0 <= g < len(weights)):
        return False, True
    total = float(np.sum(weights))
    target = min(max(float(w), 0.0), 1.0) * total
    c = np.cumsum(weights)
    tol = DRAW_REL * total
    if weights[g] < -1e-5 * pq_scale[g]:
        return False, True
    if g > ref_tok:
        ok = c[g - 1] - target <= tol
    else:
        ok = target - c[g] <= tol
    return bool(ok), True


def check_request(b, T, u, ws, h, i):
    """Returns (ok, tolerant_branch_taken, message) for request i."""
    w = b.w
    d0, k = int(b.doff[i]), int(w.k[i])
    zr = [b.draft_f64(d0 + j) for j in range(k)]
    tr = [b.target_f64(d0 + i + j) for j in range(k + 1)]
    uu = u[d0:d0 + k].astype(np.float64)
    L_ref, tok_ref, wts_ref = sampled_accept(zr, tr, b.tokens[d0:d0 + k], T, uu, float(ws[i]))
    gL, gtok = int(h["accept_len"][i]), int(h["next_token"][i])
    rate = np.float32(gL) / np.float32(k)
    if h["accept_rate"][i].view(np.uint32) != rate.view(np.uint32):
        return False, False, f"rate {h['accept_rate'][i]} for L={gL}"
    tolerant = False
    if gL != L_ref:
        if not (0 <= gL <= k):
            return False, True, f"accept_len {gL} out of range"
        j = min(gL, L_ref)
        p = softmax_t(zr[j], T)
        q = softmax_t(tr[j], T)
        x = int(b.tokens[d0 + j])
        margin = abs(uu[j] * p[x] - q[x])
        if margin > ACCEPT_REL * max(q[x], uu[j] * p[x]):
            return False, True, f"accept_len {gL} vs {L_ref}: margin {margin:.3e} at j={j}"
        tolerant = True
    if gL < k:
        p = softmax_t(zr[gL], T)
        q = softmax_t(tr[gL], T)
        wts = residual(p, q)
        scale = p + q
    else:
        wts = softmax_t(tr[k], T)
        scale = wts
    ref_tok = tok_ref if gL == L_ref else inverse_cdf(wts, float(ws[i]))
    ok, tol2 = _draw_ok(wts, ws[i], gtok, ref_tok, scale)
    if not ok:
        return False, True, f"next_token {gtok} vs {ref_tok} (L={gL})"
    return True, tolerant or tol2, ""


def check_all(b, T, u, ws, run, requests=None, max_tolerant_frac=0.02):
    w = b.w
    reqs = list(range(w.num_requests)) if requests is None else list(requests)
    with ThreadPoolExecutor(THREADS) as ex:
        res = list(ex.map(lambda i: (i,) + check_request(b, T, u, ws, run.h, i), reqs))
    bad = [(i, m) for i, ok, _, m in res if not ok]
    assert not bad, bad[:5]
    n_tol = sum(1 for _, _, t, _ in res if t)
    assert n_tol <= max(1, int(max_tolerant_frac * len(reqs))), n_tol


def check_lse(b, T, run, draft_rows, target_rows):
    w = b.w
    Nd = w.num_draft_rows
    lse = run.h["row_lse"]
    for d in draft_rows:
        ref = log_sum_exp(b.draft_f64(d) / T)
        assert abs(lse[d] - ref) <= LSE_REL * abs(ref) + LSE_ABS, ("draft", d, lse[d], ref)
    for s in target_rows:
        ref = log_sum_exp(b.target_f64(s) / T)
        assert abs(lse[Nd + s] - ref) <= LSE_REL * abs(ref) + LSE_ABS, ("target", s, lse[Nd + s], ref)


def _run_and_check(b, T, seed=0, misalign=0, lse_rows=None, requests=None):
    w = b.w
    u, ws = uniforms(w, seed)
    run = SampledRun(b, T, u, ws, misalign=misalign)
    assert run.status_word == 0, run.status_word
    assert run.canaries_intact() is None, run.canaries_intact()
    if lse_rows is None:
        check_lse(b, T, run, range(w.num_draft_rows), range(w.num_target_rows))
    else:
        check_lse(b, T, run, lse_rows[0], lse_rows[1])
    check_all(b, T, u, ws, run, requests=requests)
    return run, u, ws


@pytest.mark.parametrize("T", [0.5, 1.0, 2.0])
def test_tiny_fp32_every_request(T):
    run, _, _ = _run_and_check(materialize(make_workload("tiny")), T, seed=int(T * 10))
    assert (run.h["accept_len"] >= 0).all()


def test_concurrency_32_qwen3_vocab():
    b = materialize(make_workload("c32"))
    rng = np.random.default_rng(5)
    w = b.w
    dr = sorted(set(rng.choice(w.num_draft_rows, 24, replace=False)) | {0, w.num_draft_rows - 1})
    tr = sorted(set(rng.choice(w.num_target_rows, 24, replace=False)) | {w.num_target_rows - 1})
    _run_and_check(b, 1.0, seed=11, lse_rows=(dr, tr))


def test_concurrency_128_bench_workload():
    b = materialize(make_workload("c128"))
    w = b.w
    rng = np.random.default_rng(6)
    dr = sorted(rng.choice(w.num_draft_rows, 16, replace=False))
    tr = sorted(rng.choice(w.num_target_rows, 16, replace=False))
    run, _, _ = _run_and_check(b, 0.8, seed=12, lse_rows=(dr, tr))
    L = run.h["accept_len"]
    # both branches of the draw occur on this workload
    assert (L < w.k).any() and (L == w.k).any()


def test_stress_odd_vocab_mixed_dtypes_unaligned():
    b = materialize(make_workload("stress"))
    w = b.w
    rng = np.random.default_rng(7)
    reqs = sorted(rng.choice(w.num_requests, 96, replace=False))
    dr = sorted(rng.choice(w.num_draft_rows, 12, replace=False))
    tr = sorted(rng.choice(w.num_target_rows, 12, replace=False))
    _run_and_check(b, 1.3, seed=13, lse_rows=(dr, tr), requests=reqs)
    _run_and_check(b, 0.7, seed=14, misalign=1, lse_rows=(dr, tr), requests=reqs[:32])


EDGE = [
    dict(vocab=1, k=[1, 2]),
    dict(vocab=7, k=[3, 1, 16]),
    dict(vocab=9, k=[5, 5], d_dtype="fp32", t_dtype="fp32"),
    dict(vocab=1023, k=[16, 1], d_dtype="fp32", t_dtype="bf16"),
    dict(vocab=4097, k=[2, 7, 1], d_dtype="bf16", t_dtype="fp32"),
    dict(vocab=2048, k=[6, 2], ld_d=2048 + 5, ld_t=2048 + 3),
    dict(vocab=96, k=list(np.random.default_rng(9).integers(1, 17, size=300)), d_dtype="fp32", t_dtype="fp32"),
    dict(vocab=524288, k=[16, 1], d_dtype="bf16", t_dtype="bf16"),
    dict(vocab=524287, k=[4, 9], d_dtype="fp32", t_dtype="bf16"),
]


@pytest.mark.parametrize("case", EDGE, ids=lambda c: f"V{c['vocab']}_k{len(c['k'])}")
def test_edge_shapes(case):
    _run_and_check(materialize(custom(**case)), 0.9, seed=len(case["k"]))


def _equal_pair_batch(vocab, k, d_dtype="fp32", t_dtype="fp32"):
    """A batch whose paired target rows hold the draft rows' values (exactly, in either storage type)."""
    b = materialize(custom(vocab=vocab, k=k, d_dtype=d_dtype, t_dtype=t_dtype))
    w = b.w
    for d in range(w.num_draft_rows):
        s = w.pair_target_row(d)
        if d_dtype == t_dtype:
            b.target[s] = b.draft[d]
        elif d_dtype == "fp32":  # bf16 target: round once, store the rounded values in both
            bits = f32_to_bf16_bits(b.draft[d, :vocab])
            b.target[s, :vocab] = bits
            b.draft[d, :vocab] = bf16_bits_to_f32(bits)
        else:
            b.target[s, :vocab] = bf16_bits_to_f32(b.draft[d, :vocab])
    return b


@pytest.mark.parametrize("dtypes", [("fp32", "fp32"), ("fp32", "bf16"), ("bf16", "fp32"), ("bf16", "bf16")])
def test_equal_rows_accept_everything_and_draw_from_bonus_row(dtypes):
    # V = 3001: consecutive rows start at different 16-byte alignments
    b = _equal_pair_batch(3001, [4, 16, 1, 7], *dtypes)
    w = b.w
    u = np.full(w.num_draft_rows, np.float32(np.nextafter(np.float32(1), np.float32(0))))
    ws = np.random.default_rng(3).random(w.num_requests, dtype=np.float32)
    run = SampledRun(b, 1.1, u, ws)
    assert run.status_word == 0
    assert np.array_equal(run.h["accept_len"], w.k)
    assert (run.h["accept_rate"] == 1.0).all()
    Nd = w.num_draft_rows
    for d in range(Nd):
        assert run.h["row_lse"][d] == run.h["row_lse"][Nd + w.pair_target_row(d)], d
    check_all(b, 1.1, u, ws, run)


def test_zero_residual_falls_back_to_target():
    # u = 1 rejects even when p = q; the residual max(0, q - p) is then all zero
    b = _equal_pair_batch(5000, [3, 5, 2])
    w = b.w
    u = np.ones(w.num_draft_rows, dtype=np.float32)
    ws = np.array([0.0, 0.37, 0.999], dtype=np.float32)
    run = SampledRun(b, 0.6, u, ws)
    assert run.status_word == 0
    assert (run.h["accept_len"] == 0).all()
    check_all(b, 0.6, u, ws, run, max_tolerant_frac=0.0)
    for i in range(w.num_requests):
        q = softmax_t(b.target_f64(int(b.doff[i]) + i), 0.6)
        g = int(run.h["next_token"][i])
        assert q[g] > 0


def test_uniform_edges():
    b = materialize(custom(vocab=6000, k=[5, 5, 5, 5, 5, 5], d_dtype="fp32", t_dtype="fp32"))
    w = b.w
    u = np.zeros(w.num_draft_rows, dtype=np.float32)  # u = 0 accepts every token with q > 0
    ws = np.array([0.0, np.nextafter(np.float32(1), np.float32(0)), 1.0, 0.5, np.nan, -0.25], dtype=np.float32)
    run = SampledRun(b, 1.0, u, ws)
    assert run.status_word == 0
    assert np.array_equal(run.h["accept_len"], w.k)
    # the kernel clamps w to [0, 1] and reads NaN as 0
    wsc = np.clip(np.nan_to_num(ws, nan=0.0), 0.0, 1.0).astype(np.float32)
    check_all(b, 1.0, u, wsc, run)
    # w = 0 draws the first entry with positive weight
    for i in (0, 4, 5):
        q = softmax_t(b.target_f64(int(b.doff[i + 1]) + i), 1.0)
        assert run.h["next_token"][i] == int(np.flatnonzero(q > 0)[0])


def test_deterministic_bitwise():
    b = materialize(make_workload("c32"))
    u, ws = uniforms(b.w, 21)
    r1 = SampledRun(b, 0.9, u, ws)
    r2 = SampledRun(b, 0.9, u, ws)
    for key in r1.h:
        assert np.array_equal(r1.h[key].view(np.uint8), r2.h[key].view(np.uint8)), key


def test_bad_offsets_and_tokens_set_status():
    import serving_packed_var_gb300 as af
    w = custom(vocab=300, k=[4, 4, 4])
    b = materialize(w)
    dev = torch.device("cuda:0")
    z = to_device(b.draft, w.d_dtype, dev)
    t = to_device(b.target, w.t_dtype, dev)
    tok = torch.from_numpy(b.tokens).to(dev)
    ua = torch.full((12,), 0.5, dtype=torch.float32, device=dev)
    us = torch.full((3,), 0.5, dtype=torch.float32, device=dev)
    bad_doff = torch.tensor([0, 4, 4, 12], dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    out = af.adaflash_verify_sampled(z, t, tok, bad_doff, 1.0, ua, us, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & (1 << af.ADAFLASH_ERR_BAD_OFFSETS)
    assert out["accept_len"][1].item() == -1 and out["next_token"][1].item() == -1
    tok2 = tok.clone()
    tok2[1] = 300
    tok2[8] = -5
    st.zero_()
    out = af.adaflash_verify_sampled(z, t, tok2, torch.from_numpy(b.doff).to(dev), 1.0, ua, us, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == (1 << af.ADAFLASH_ERR_BAD_TOKEN)
    assert out["accept_len"][0].item() <= 1 and out["accept_len"][2].item() == 0
    assert 0 <= out["next_token"][0].item() < 300 and 0 <= out["next_token"][2].item() < 300
