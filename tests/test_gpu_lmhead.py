"""The logit-free path on the GPU: the tensor-core head GEMM (adaflash_lmhead_logits)
against a float64 product, then adaflash_lmhead_opd_fwd against the oracle
(oracle/lmhead.py), through the C ABI.

Bars.  Logits: |d| <= 1e-5 (1 + sum_k |h_k w_k|) (float32 accumulation over H terms).
Loss outputs: the bf16 bars of the logits path (2e-3 relative + 1e-5), S against its
summands' size as there.  The target argmax is exact unless the oracle's two largest
logits of a row lie within the GEMM's rounding (1e-4 (1 + max |t|)), where either is
valid; the acceptance outputs are exact given the argmax.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from oracle import opd  # noqa: E402
from oracle.lmhead import head_logits  # noqa: E402
from synth.lmhead import custom_lmhead, make_lmhead_workload, materialize_lmhead  # noqa: E402
from synth.workloads import bf16_bits_to_f32, f32_to_bf16_bits  # noqa: E402

REL, ABS = 2e-3, 1e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


@pytest.mark.parametrize("rows,V,H", [(1, 256, 64), (200, 1000, 256), (128, 4096, 512), (37, 2049, 1024)])
def test_head_gemm_matches_float64(rows, V, H):
    import serving_packed_var_gb300 as af
    rng = np.random.default_rng(rows + V + H)
    hb = f32_to_bf16_bits(rng.standard_normal((rows, H), dtype=np.float32))
    wb = f32_to_bf16_bits(rng.standard_normal((V, H), dtype=np.float32) * np.float32(0.05))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = af.adaflash_lmhead_logits(_dev_bf16(hb), _dev_bf16(wb), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    h, w = bf16_bits_to_f32(hb).astype(np.float64), bf16_bits_to_f32(wb).astype(np.float64)
    ref = head_logits(h, w)
    mag = np.abs(h) @ np.abs(w).T
    err = np.abs(out.cpu().numpy().astype(np.float64) - ref)
    assert (err <= 1e-5 * (1 + mag)).all(), float((err / (1 + mag)).max())


def _run(b, clip_c=None):
    import serving_packed_var_gb300 as af
    w = b.w
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    wd = _dev_bf16(b.wd)
    wt = wd if b.wd is b.wt else _dev_bf16(b.wt)
    out = af.adaflash_lmhead_opd_fwd(_dev_bf16(b.hd), _dev_bf16(b.ht), wd, wt, torch.from_numpy(b.tokens).cuda(),
                                     torch.from_numpy(b.doff).cuda(), w.clip_c if clip_c is None else clip_c,
                                     w.ce_weight, status=st)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}, int(st.item())


def _check(b, h, rows, clip_c=None):
    w = b.w
    c = w.clip_c if clip_c is None else clip_c
    hd, ht = b.f32("hd"), b.f32("ht")
    wd, wt = b.f32("wd"), b.f32("wt")
    for d in rows:
        s = w.pair_target_row(d)
        z = head_logits(hd[d], wd)[0]
        t = head_logits(ht[s], wt)[0]
        f = opd.row_forward(z, t, c, w.ce_weight)
        for key, got in (("kl", h["kl_row"][d]), ("ce", h["ce_row"][d]), ("lse_z", h["row_stats"][d][0]),
                         ("lse_t", h["row_stats"][d][1])):
            assert abs(got - f[key]) <= REL * abs(f[key]) + ABS, (key, d, got, f[key])
        assert abs(h["row_stats"][d][2] - f["S"]) <= REL * (abs(f["S"]) + f["S_l1"]) + ABS, ("S", d)
        assert int(h["row_stats"][d][3]) == f["n_clipped"], ("n_clipped", d)
        assert h["target_argmax"][s] == f["argmax"], ("argmax", d)


def _oracle_target_argmax(b):
    """First maximiser of every target row's float64 logits, and the runner-up gap."""
    ht, wt = b.f32("ht"), b.f32("wt")
    am, tops = [], []
    for r0 in range(0, ht.shape[0], 256):
        t = head_logits(ht[r0:r0 + 256], wt)
        for row in t:
            a = opd.first_argmax(row)
            am.append(a)
            tops.append(row)
    return am, tops


def _check_verify(b, h):
    w = b.w
    am, tops = _oracle_target_argmax(b)
    got = h["target_argmax"]
    for s in range(w.num_target_rows):
        if got[s] != am[s]:
            row = tops[s]
            assert row[got[s]] >= row[am[s]] - 1e-4 * (1 + abs(row[am[s]])), ("argmax", s, got[s], am[s])
    # acceptance from the GPU's own argmax (exact given it)
    for i in range(w.num_requests):
        d0, k = int(b.doff[i]), int(w.k[i])
        L, bonus = opd.greedy_accept(b.tokens[d0:d0 + k], [int(x) for x in got[d0 + i:d0 + i + k + 1]])
        assert h["accept_len"][i] == L, i
        assert h["bonus_token"][i] == bonus, i
        assert h["accept_rate"][i].view(np.uint32) == opd.acceptance_rate(L, k).view(np.uint32), i
    assert np.mean(np.asarray(got) == np.asarray(am)) > 0.99


@pytest.mark.parametrize("clip_c", [1.0, 0.05, float("inf")])
def test_tiny_every_row(clip_c):
    b = materialize_lmhead(make_lmhead_workload("lm_tiny"))
    h, st = _run(b, clip_c)
    assert st == 0
    _check_verify(b, h)
    assert float(np.mean(h["kl_row"])) > 0.05 and float(np.mean(h["ce_row"])) > 0.05  # not a degenerate batch
    _check(b, h, range(b.w.num_draft_rows), clip_c)
    w = b.w
    rows = range(w.num_draft_rows)
    fs = [opd.row_forward(head_logits(b.f32("hd")[d], b.f32("wd"))[0],
                          head_logits(b.f32("ht")[w.pair_target_row(d)], b.f32("wt"))[0], clip_c, w.ce_weight)
          for d in rows]
    ref = sum(f["loss_row"] for f in fs) / len(fs)
    assert abs(float(h["loss"][0]) - ref) <= REL * abs(ref) + ABS


def test_small_shared_head():
    b = materialize_lmhead(make_lmhead_workload("lm_small"))
    h, st = _run(b)
    assert st == 0
    _check_verify(b, h)
    _check(b, h, range(b.w.num_draft_rows))


@pytest.mark.parametrize("case", [dict(vocab=300, hidden=64, k=[2, 1]), dict(vocab=5000, hidden=192, k=[16] * 9),
                                  dict(vocab=257, hidden=128, k=[3, 16, 1, 7])])
def test_edge_shapes(case):
    b = materialize_lmhead(custom_lmhead(**case, shared_head=False))
    h, st = _run(b)
    assert st == 0
    _check_verify(b, h)
    _check(b, h, range(b.w.num_draft_rows))


def test_padded_rows_and_strided_views():
    # every matrix a view with ld > H (rows still 16-byte aligned), separate heads
    import serving_packed_var_gb300 as af
    b = materialize_lmhead(custom_lmhead(vocab=1500, hidden=256, k=[5, 16, 2], shared_head=False))
    w = b.w

    def padded(bits, extra):
        n, H = bits.shape
        full = np.zeros((n, H + extra), dtype=np.uint16)
        full[:, :H] = bits
        return _dev_bf16(full)[:, :H]

    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    hd, ht, wd, wt = padded(b.hd, 8), padded(b.ht, 64), padded(b.wd, 24), padded(b.wt, 8)
    assert hd.stride(0) == 264 and ht.stride(0) == 320
    out = af.adaflash_lmhead_opd_fwd(hd, ht, wd, wt, torch.from_numpy(b.tokens).cuda(), torch.from_numpy(b.doff).cuda(),
                                     w.clip_c, w.ce_weight, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    h = {k: v.cpu().numpy() for k, v in out.items()}
    _check_verify(b, h)
    _check(b, h, range(w.num_draft_rows))


def test_single_request_qwen3_8b_shapes():
    b = materialize_lmhead(custom_lmhead(vocab=151936, hidden=4096, k=[16], spike=18.0))
    h, st = _run(b)
    assert st == 0
    _check_verify(b, h)
    _check(b, h, [0, 9, 15])


def test_qwen3_8b_shapes_c32_sampled_rows():
    b = materialize_lmhead(make_lmhead_workload("lm_c32"))
    h, st = _run(b)
    assert st == 0
    _check_verify(b, h)
    nd = b.w.num_draft_rows
    _check(b, h, sorted({0, 7, nd // 2, nd - 1}))
