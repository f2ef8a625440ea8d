"""CUDA path vs the float64 oracle, through the C ABI, on the seeded workloads.

Small cases are compared in full (every row, every gradient entry); the
full-size workloads are compared in full for the verification outputs, the
per-row losses and the batch loss, and on sampled rows for the gradient.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from parity_lib import (GpuRun, check_loss, check_rows, check_verify, oracle_argmax_all,  # noqa: E402
                        oracle_rows)
from synth import make_workload, materialize  # noqa: E402
from synth.workloads import custom  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _full_check(b, bwd=True, grad_rows=None, loss=True, run_kw=None):
    run = GpuRun(b, bwd=bwd, **(run_kw or {}))
    assert run.status_word == 0, run.status_word
    assert run.canaries_intact() is None, run.canaries_intact()
    check_verify(run, oracle_argmax_all(b))
    w = b.w
    rows = list(range(w.num_draft_rows))
    per, _ = oracle_rows(b, rows, bwd=False)
    gsel = rows if grad_rows is None else grad_rows
    grads = None
    if bwd:
        _, grads = oracle_rows(b, gsel, bwd=True, **{k: v for k, v in (run_kw or {}).items()
                                                       if k in ("grad_row", "grad_scale")})
    check_rows(run, per, grads)
    if loss:
        ref = sum(per[d]["loss_row"] for d in rows) / len(rows)
        check_loss(run, ref)
    return run, per


def test_tiny_fp32_full():
    _full_check(materialize(make_workload("tiny")))


def test_single_request_qwen3_vocab():
    _full_check(materialize(make_workload("single")))


def test_concurrency_32():
    b = materialize(make_workload("c32"))
    rng = np.random.default_rng(1)
    _full_check(b, grad_rows=sorted(rng.choice(b.w.num_draft_rows, 48, replace=False)))


def test_concurrency_128():
    b = materialize(make_workload("c128"))
    w = b.w
    rng = np.random.default_rng(2)
    rows = sorted(set(rng.choice(w.num_draft_rows, 40, replace=False)) | set(int(r) for r in w.clip_rows[:8]))
    run, per = _full_check(b, grad_rows=rows)
    # the -30/+6 plant stays below c = 0.5 on these rows
    assert all(per[int(d)]["n_clipped"] == 0 for d in w.clip_rows)


def test_concurrency_128_clip_binds():
    b = materialize(make_workload("c128_clip"))
    w = b.w
    rows = [int(r) for r in w.clip_rows[:12]] + [0, w.num_draft_rows - 1]
    run, per = _full_check(b, grad_rows=rows)
    for d in w.clip_rows:
        assert int(run.h["row_stats"][int(d)][3]) == 64


def test_stress_odd_vocab_mixed_dtypes():
    b = materialize(make_workload("stress"))
    w = b.w
    run = GpuRun(b, bwd=True)
    assert run.status_word == 0
    assert run.canaries_intact() is None
    check_verify(run, oracle_argmax_all(b))
    rng = np.random.default_rng(3)
    tie_drafts = [w.draft_of_target(int(s)) for s in w.tie_rows if w.draft_of_target(int(s)) >= 0][:8]
    rows = sorted(set(rng.choice(w.num_draft_rows, 40, replace=False)) | set(int(r) for r in w.equal_rows[:8])
                  | set(tie_drafts) | {0, w.num_draft_rows - 1})
    per, grads = oracle_rows(b, rows)
    check_rows(run, per, grads)
    for d in w.equal_rows:
        assert run.h["kl_row"][int(d)] == 0.0, ("draft == target must give KL = 0", int(d))
    # every row's loss, for the batch mean
    per_all, _ = oracle_rows(b, list(range(w.num_draft_rows)), bwd=False)
    check_loss(run, sum(f["loss_row"] for f in per_all.values()) / w.num_draft_rows)
    rel = 2e-3
    for d, f in per_all.items():
        assert abs(run.h["kl_row"][d] - f["kl"]) <= rel * abs(f["kl"]) + 1e-5, d
        assert abs(run.h["ce_row"][d] - f["ce"]) <= rel * abs(f["ce"]) + 1e-5, d


def test_verify_only_entry_point():
    import serving_packed_var_gb300 as af
    from parity_lib import to_device
    for name in ("tiny", "c32", "stress"):
        b = materialize(make_workload(name))
        w = b.w
        dev = torch.device("cuda:0")
        t = to_device(b.target, w.t_dtype, dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        out = af.adaflash_verify_packed(t, torch.from_numpy(b.tokens).to(dev), torch.from_numpy(b.doff).to(dev),
                                        vocab=w.vocab, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        ref = oracle_argmax_all(b)
        assert np.array_equal(out["target_argmax"].cpu().numpy(), ref)
        res = oracle.verify_packed(b.target_f64, b.tokens, b.doff)
        acc = out["accept_len"].cpu().numpy()
        bon = out["bonus_token"].cpu().numpy()
        rate = out["accept_rate"].cpu().numpy()
        for i in range(w.num_requests):
            assert acc[i] == res[i]["accept_len"] == w.planted_accept[i]
            assert bon[i] == res[i]["bonus_token"]
            assert rate[i].view(np.uint32) == res[i]["accept_rate"].view(np.uint32)


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------

EDGE = [
    dict(vocab=1, k=[1, 2], accept="full"),
    dict(vocab=7, k=[3, 1, 16]),
    dict(vocab=8, k=[16]),
    dict(vocab=9, k=[5, 5], d_dtype="fp32", t_dtype="fp32"),
    dict(vocab=1023, k=[16, 1], d_dtype="fp32", t_dtype="bf16"),
    dict(vocab=4097, k=[2, 7, 1], d_dtype="bf16", t_dtype="fp32"),
    dict(vocab=40001, k=[4, 4], accept="none"),
    dict(vocab=80003, k=[3, 16, 1], d_dtype="fp32", t_dtype="fp32"),
    dict(vocab=151936, k=[1], accept="full"),
    dict(vocab=4096, k=[16] * 40, accept="uniform"),
    dict(vocab=2048, k=[6, 2], ld_d=2048 + 5, ld_t=2048 + 3),
    dict(vocab=3000, k=[9], clip_c=0.01),
    # the largest vocabulary the library takes, on and off the 16-byte grid
    dict(vocab=524288, k=[16, 1], d_dtype="fp32", t_dtype="fp32"),
    dict(vocab=524287, k=[5, 2], d_dtype="fp32", t_dtype="bf16"),
]


@pytest.mark.parametrize("case", EDGE, ids=lambda c: f"V{c['vocab']}_k{len(c['k'])}")
def test_edge_shapes(case):
    w = custom(**case)
    _full_check(materialize(w))


@pytest.mark.parametrize("misalign", [1, 3])
def test_unaligned_base_pointers(misalign):
    w = custom(vocab=5000, k=[3, 8], d_dtype="bf16", t_dtype="bf16")
    _full_check(materialize(w), run_kw=dict(misalign=misalign))


def test_constant_and_equal_rows():
    w = custom(vocab=777, k=[4, 3], constant_target_rows=np.array([0, 5]), equal_rows=np.array([1, 4]))
    b = materialize(w)
    run, per = _full_check(b)
    assert run.h["target_argmax"][0] == 0 and run.h["target_argmax"][5] == 0
    assert run.h["kl_row"][1] == 0.0 and run.h["kl_row"][4] == 0.0


@pytest.mark.parametrize("requests", [3, 4, 6, 8, 16])
def test_mid_batches_at_qwen3_vocab(requests):
    # k = 16 per request at V = 151936: the forward and verification take every row in one round of
    # resident clusters with the largest cluster size that allows it (8 down to 1 as the batch grows)
    b = materialize(custom(vocab=151936, k=[16] * requests, d_dtype="bf16", t_dtype="bf16", seed=requests))
    rng = np.random.default_rng(requests)
    _full_check(b, grad_rows=sorted(set(rng.choice(b.w.num_draft_rows, 6, replace=False)) | {0, b.w.num_draft_rows - 1}))


def test_many_requests_small_vocab():
    rng = np.random.default_rng(9)
    k = rng.integers(1, 17, size=700)
    _full_check(materialize(custom(vocab=96, k=k, d_dtype="fp32", t_dtype="fp32")), grad_rows=list(range(64)))


def test_per_row_upstream_weights():
    w = custom(vocab=3001, k=[5, 2, 9])
    b = materialize(w)
    gr = np.linspace(-1.5, 2.0, w.num_draft_rows)
    _full_check(b, run_kw=dict(grad_row=gr))


def test_grad_scale_mean():
    w = custom(vocab=2500, k=[6, 6])
    b = materialize(w)
    _full_check(b, run_kw=dict(grad_scale=1.0 / w.num_draft_rows))


def test_deterministic_bitwise():
    b = materialize(make_workload("c32"))
    r1 = GpuRun(b)
    r2 = GpuRun(b)
    for k in r1.h:
        assert np.array_equal(r1.h[k].view(np.uint8), r2.h[k].view(np.uint8)), k
    assert torch.equal(r1.grad, r2.grad)


# ---------------------------------------------------------------------------
# device-detected errors: status bits, no fault
# ---------------------------------------------------------------------------

def test_bad_offsets_and_tokens_set_status():
    import serving_packed_var_gb300 as af
    w = custom(vocab=300, k=[4, 4, 4])
    b = materialize(w)
    dev = torch.device("cuda:0")
    z = torch.from_numpy(b.draft.view(np.int16)).to(dev).view(torch.bfloat16)
    t = torch.from_numpy(b.target.view(np.int16)).to(dev).view(torch.bfloat16)
    tok = torch.from_numpy(b.tokens).to(dev)
    # k_1 = 0 and a final offset that does not match N_d
    bad_doff = torch.tensor([0, 4, 4, 12], dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    af.adaflash_opd_loss_fwd(z, t, tok, bad_doff, 1.0, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & (1 << af.ADAFLASH_ERR_BAD_OFFSETS)
    # a token outside the vocabulary
    tok2 = tok.clone()
    tok2[1] = 300
    st.zero_()
    out = af.adaflash_opd_loss_fwd(z, t, tok2, torch.from_numpy(b.doff).to(dev), 1.0, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == (1 << af.ADAFLASH_ERR_BAD_TOKEN)
    assert out["accept_len"][0].item() <= 1


def test_bounded_wait_gives_up_with_status():
    import serving_packed_var_gb300 as af
    st = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    af.adaflash_selftest_bounded_wait(st, limit_us=2000)
    torch.cuda.synchronize()
    assert int(st.item()) == (1 << af.ADAFLASH_ERR_TIMEOUT)
    # the context is still usable afterwards
    x = torch.ones(4, device="cuda:0")
    assert float(x.sum().item()) == 4.0
