"""Packer -> kernels, end to end: each round's offsets from the host packer drive
adaflash_opd_loss_fwd_bwd on a batch of exactly the admitted requests, and the
outputs meet the oracle's bars (parity_lib)."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from parity_lib import check_loss, check_rows, check_verify, oracle_argmax_all, oracle_rows, to_device  # noqa: E402
from synth import materialize  # noqa: E402
from synth.workloads import custom  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


class _Run:
    pass


def test_packed_rounds_run_through_the_fused_step():
    import serving_packed_var_gb300 as af
    rng = np.random.default_rng(21)
    packer = af.Packer(row_budget=400, alpha=0.3, initial_rows_per_request=20.0)
    queue = []
    dev = torch.device("cuda:0")
    served = 0
    for rnd in range(5):
        queue.extend(int(k) for k in rng.integers(1, 17, size=int(rng.integers(5, 30))))
        plan = packer.plan(queue)
        n = plan["admitted"]
        assert n >= 1 and plan["rows"] <= 400
        ks = queue[:n]
        w = custom(vocab=4096, k=ks, d_dtype="bf16", t_dtype="bf16", seed=rnd)
        b = materialize(w)
        assert np.array_equal(plan["draft_offsets"], b.doff)
        z = to_device(b.draft, w.d_dtype, dev)
        t = to_device(b.target, w.t_dtype, dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        doff = torch.from_numpy(plan["draft_offsets"]).to(dev)
        out = af.adaflash_opd_loss_fwd_bwd(z, t, torch.from_numpy(b.tokens).to(dev), doff, w.clip_c, w.ce_weight,
                                           grad_scale=1.0 / w.num_draft_rows, vocab=w.vocab, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        r = _Run()
        r.w, r.b = w, b
        r.h = {k: v.cpu().numpy() for k, v in out.items() if k != "grad"}
        r.grad_rows = lambda rows, g=out["grad"]: {d: g[d].cpu().numpy().astype(np.float64) for d in rows}
        check_verify(r, oracle_argmax_all(b))
        rows = list(range(w.num_draft_rows))
        per, grads = oracle_rows(b, rows, bwd=True, grad_scale=1.0 / w.num_draft_rows)
        check_rows(r, per, grads)
        check_loss(r, sum(per[d]["loss_row"] for d in rows) / len(rows))
        packer.observe(plan["rows"], n)
        queue = queue[n:]
        served += n
    assert served > 0
    packer.close()
