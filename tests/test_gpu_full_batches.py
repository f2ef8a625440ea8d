"""Full-size batches through the benchmark's call, every row checked against the C++ oracle.

The step the benchmark times is one adaflash_opd_loss_fwd_bwd call (on these batches the row pass with the
gradient, then the acceptance scan / loss kernel).  The float64 C++ oracle, on every host core, is fast
enough to check all of it: every request's verification outputs, every row's loss terms and row statistics,
the batch loss, and every entry of every gradient row (in blocks of rows, so host memory stays small).  The
bars are those of the parity tests (parity_lib).
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from oracle import cpp  # noqa: E402
from parity_lib import GRAD_ABS, GRAD_REL, check_loss, check_rows, check_verify, oracle_argmax_all  # noqa: E402
from synth import make_workload, materialize  # noqa: E402
from test_gpu_fused import FusedRun  # noqa: E402

THREADS = 16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _check_every_row(name, every=1, block=64):
    b = materialize(make_workload(name))
    w = b.w
    f = FusedRun(b, grad_scale=1.0)
    assert f.status_word == 0, f.status_word
    assert f.canaries_intact() is None, f.canaries_intact()
    check_verify(f, oracle_argmax_all(b))
    rows = list(range(0, w.num_draft_rows, every))
    checked = 0
    for lo in range(0, len(rows), block):
        sel = rows[lo:lo + block]
        per, grads, _ = cpp.opd_rows(b.draft, w.d_dtype, b.target, w.t_dtype, b.doff, w.vocab, w.clip_c, w.ce_weight,
                                     rows=sel, grad=True, grad_scale=1.0, threads=THREADS)
        check_rows(f, per)
        got = f.grad[sel].cpu().numpy().astype(np.float64)
        for k, d in enumerate(sel):
            ref = grads[d]
            bad = np.abs(got[k] - ref) > GRAD_ABS + GRAD_REL * np.abs(ref)
            assert not bad.any(), ("grad", d, int(np.argmax(bad)))
        checked += len(sel)
    if every == 1:
        _, _, loss = cpp.opd_rows(b.draft, w.d_dtype, b.target, w.t_dtype, b.doff, w.vocab, w.clip_c, w.ce_weight,
                                  threads=THREADS)
        check_loss(f, loss)
    return f, checked


def test_concurrency_128_every_row():
    f, n = _check_every_row("c128")
    assert n == 914


def test_concurrency_128_binding_clip_every_row():
    f, n = _check_every_row("c128_clip")
    w = f.w
    for d in w.clip_rows:
        assert int(f.h["row_stats"][int(d)][3]) == 64


def test_concurrency_32_every_row():
    _check_every_row("c32")


def test_stress_every_row():
    # the 8192 rows off the 16-byte grid, every gradient entry of each
    f, n = _check_every_row("stress", block=128)
    assert n == 8192
