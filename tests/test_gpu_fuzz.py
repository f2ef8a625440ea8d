"""Seeded random batches through every logits entry point, all outputs against the oracle.

Each case draws its own vocabulary size (small, medium and large, on and off the 16-byte grid),
request count and draft lengths, dtype pair, padded leading dimensions, base-pointer offsets,
clip threshold and hard-label weight.  It runs the separate forward and backward calls, the
single-call step and the sampled verification, and checks every request, every row and every
gradient entry against the float64 C++ oracle (the sampled path against its numpy oracle), with
the parity tests' bars.  The draws are fixed by the case number, so a failure replays exactly.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from oracle import cpp  # noqa: E402
from parity_lib import GRAD_ABS, GRAD_REL, GpuRun, check_loss, check_rows, check_verify, oracle_argmax_all  # noqa: E402
from synth import materialize  # noqa: E402
from synth.workloads import custom  # noqa: E402
from test_gpu_fused import FusedRun  # noqa: E402
from test_gpu_sampled import _run_and_check  # noqa: E402

CASES = 64
THREADS = 16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _case(i):
    rng = np.random.default_rng(7000 + i)
    size = i % 3
    V = int(rng.integers(1, 64) if size == 0 else rng.integers(64, 5000) if size == 1 else rng.integers(5000, 40000))
    R = int(rng.integers(1, 17))
    k = [int(x) for x in rng.integers(1, 17, size=R)]
    d_dtype, t_dtype = (str(x) for x in rng.choice(["fp32", "bf16"], 2))
    case = dict(vocab=V, k=k, d_dtype=d_dtype, t_dtype=t_dtype, seed=i,
                clip_c=float(rng.choice([0.05, 0.3, 1.0, 5.0])), ce_weight=float(rng.choice([0.0, 0.5, 1.0, 2.0])),
                ld_d=V + int(rng.integers(0, 9)), ld_t=V + int(rng.integers(0, 9)))
    offsets = dict(misalign_z=int(rng.integers(0, 4)), misalign_t=int(rng.integers(0, 4)))
    return case, offsets


def _check_grads(grad, ref):
    got = grad.cpu().numpy().astype(np.float64)
    for d, r in ref.items():
        bad = np.abs(got[d] - r) > GRAD_ABS + GRAD_REL * np.abs(r)
        assert not bad.any(), ("grad", d, int(np.argmax(bad)))


@pytest.mark.parametrize("i", range(CASES))
def test_random_batch(i):
    case, offsets = _case(i)
    b = materialize(custom(**case))
    w = b.w
    per, grads, loss = cpp.opd_rows(b.draft, w.d_dtype, b.target, w.t_dtype, b.doff, w.vocab, w.clip_c, w.ce_weight,
                                    grad=True, grad_scale=1.0, threads=THREADS)
    amax = oracle_argmax_all(b)
    # the separate forward and backward calls
    run = GpuRun(b, bwd=True, **offsets)
    assert run.status_word == 0, (case, run.status_word)
    assert run.canaries_intact() is None, (case, run.canaries_intact())
    check_verify(run, amax)
    check_rows(run, per)
    check_loss(run, loss)
    _check_grads(run.grad, grads)
    # the single-call step (on-chip kernel or the row pass with the gradient)
    f = FusedRun(b, grad_scale=1.0, **offsets)
    assert f.status_word == 0, (case, f.status_word)
    assert f.canaries_intact() is None, (case, f.canaries_intact())
    check_verify(f, amax)
    check_rows(f, per)
    check_loss(f, loss)
    _check_grads(f.grad, grads)
    # sampled verification at a temperature drawn with the case
    _run_and_check(b, float(np.random.default_rng(i).choice([0.5, 1.0, 1.7])), seed=i, misalign=offsets["misalign_z"])
