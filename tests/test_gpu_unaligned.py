"""Rows off the 16-byte grid, through the C ABI: every byte shift of the draft row
against the target row's grid, on every dtype pair, for the forward, the backward,
the single-call forward + backward and greedy verification.

With ld = V odd, consecutive rows start at every shift a dtype allows, so one batch
walks all the loop instances the kernels pick per row; separate base offsets of the
draft, target and gradient tensors move the classes against each other.  Outputs
are checked against the float64 oracle with the usual bars, and the single call
against the separate calls.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from oracle import cpp  # noqa: E402
from parity_lib import GpuRun, check_loss, check_rows, check_verify, oracle_argmax_all, oracle_rows, to_device  # noqa: E402
from synth import make_workload, materialize  # noqa: E402
from synth.workloads import custom  # noqa: E402
from test_gpu_fused import INT_KEYS, FusedRun, _close_to_separate  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


PAIRS = [("bf16", "bf16"), ("fp32", "bf16"), ("bf16", "fp32"), ("fp32", "fp32")]
# (draft, target, gradient) base offsets in elements
SHIFTS = [(0, 1, 0), (1, 0, 3), (3, 5, 1), (2, 7, 2)]


@pytest.mark.parametrize("dd,td", PAIRS)
@pytest.mark.parametrize("mz,mt,mg", SHIFTS)
def test_every_shift_class(dd, td, mz, mt, mg):
    # V = 1001: each row starts 2 (bf16) or 4 (fp32) bytes further along the grid than
    # the one before; c = 0.05 makes some terms clip, so the clip screen re-reads rows
    # at every shift too
    w = custom(vocab=1001, k=[16, 9, 16, 3, 7], d_dtype=dd, t_dtype=td, clip_c=0.05, ce_weight=0.8)
    b = materialize(w)
    f, s = _close_to_separate(b, grad_scale=0.7, misalign_z=mz, misalign_t=mt, misalign_g=mg)
    assert s.canaries_intact() is None, s.canaries_intact()
    assert int(np.sum(f.h["row_stats"][:, 3])) > 0, "the clip binds somewhere"


@pytest.mark.parametrize("V", [1, 5, 9, 17, 4099])
def test_heads_longer_than_the_row_and_short_rows(V):
    # rows shorter than a target head, or a head and one ragged group
    w = custom(vocab=V, k=[2, 16, 1], d_dtype="bf16", t_dtype="bf16", accept="full" if V == 1 else "uniform")
    _close_to_separate(materialize(w), misalign_z=3, misalign_t=5, misalign_g=1)


def test_stress_shape_small_batch():
    """V = 151937, float32 draft / bfloat16 target, natural packed layout (ld = V): few
    rows, so the call splits each row over a cluster and each CTA's slice starts at a
    different shift."""
    w = custom(vocab=151937, k=[16, 16, 5], d_dtype="fp32", t_dtype="bf16")
    b = materialize(w)
    nd = w.num_draft_rows
    _close_to_separate(b, grad_scale=0.5, oracle_grad_rows=[0, 1, 2, 3, 17, nd - 1])


def test_verify_only_at_every_shift():
    import serving_packed_var_gb300 as af
    for td in ("bf16", "fp32"):
        w = custom(vocab=1001, k=[16, 9, 16, 3, 7], t_dtype=td)
        b = materialize(w)
        dev = torch.device("cuda:0")
        ref = oracle_argmax_all(b)
        for mt in range(0, 8):
            t = to_device(b.target, td, dev, mt)
            st = torch.zeros(1, dtype=torch.int32, device=dev)
            out = af.adaflash_verify_packed(t, torch.from_numpy(b.tokens).to(dev), torch.from_numpy(b.doff).to(dev),
                                            vocab=w.vocab, status=st)
            torch.cuda.synchronize()
            assert int(st.item()) == 0
            assert np.array_equal(out["target_argmax"].cpu().numpy(), ref), (td, mt)


def test_stress_workload_single_call():
    """The stress workload (512 requests of 16, V = 151937, float32 draft / bfloat16 target,
    tie rows and draft == target rows) through adaflash_opd_loss_fwd_bwd: the row pass
    with the gradient on rows off the grid.  Every row's verification outputs and loss
    terms against the oracle, sampled gradient rows, and the separate calls."""
    b = materialize(make_workload("stress"))
    w = b.w
    f = FusedRun(b, grad_scale=1.0)
    assert f.status_word == 0, f.status_word
    assert f.canaries_intact() is None, f.canaries_intact()
    check_verify(f, oracle_argmax_all(b))
    per_all, _, loss = cpp.opd_rows(b.draft, w.d_dtype, b.target, w.t_dtype, b.doff, w.vocab, w.clip_c, w.ce_weight,
                                    threads=16)
    rel, ab = 2e-3, 1e-5
    for d, ref in per_all.items():
        assert abs(f.h["kl_row"][d] - ref["kl"]) <= rel * abs(ref["kl"]) + ab, d
        assert abs(f.h["ce_row"][d] - ref["ce"]) <= rel * abs(ref["ce"]) + ab, d
    check_loss(f, loss)
    for d in w.equal_rows:
        assert f.h["kl_row"][int(d)] == 0.0, int(d)
    rng = np.random.default_rng(13)
    tie_drafts = [w.draft_of_target(int(s)) for s in w.tie_rows if w.draft_of_target(int(s)) >= 0][:6]
    rows = sorted(set(rng.choice(w.num_draft_rows, 24, replace=False)) | set(int(r) for r in w.equal_rows[:4])
                  | set(tie_drafts) | {0, 1, 2, 3, w.num_draft_rows - 1})
    per, grads = oracle_rows(b, rows)
    check_rows(f, per, grads)
    s = GpuRun(b, bwd=True)
    assert s.status_word == 0
    for k in INT_KEYS:
        assert np.array_equal(f.h[k].view(np.uint8), s.h[k].view(np.uint8)), k
    for k in ("kl_row", "ce_row", "loss"):
        assert np.allclose(f.h[k], s.h[k], rtol=1e-5, atol=1e-6), k
    gd = (f.grad - s.grad).abs()
    assert float(gd.max()) <= 1e-6 + 1e-4 * float(s.grad.abs().max()), float(gd.max())
