"""prepare(): a call marshalled once and replayed gives the entry point's own results.

Every GPU entry point is prepared on a small batch and a mid-size one; each prepared call is
replayed several times into outputs first overwritten with a marker, and must reproduce, bit for
bit, what the entry point itself wrote, with the same number of kernel launches per call.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from parity_lib import to_device  # noqa: E402
from synth import materialize, make_workload  # noqa: E402
from synth.workloads import custom  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _calls(af, b, z, t, tok, doff, st, u_acc, u_smp):
    w = b.w
    return {
        "verify": (af.adaflash_verify_packed, (t, tok, doff), dict(status=st)),
        "fwd": (af.adaflash_opd_loss_fwd, (z, t, tok, doff, w.clip_c, w.ce_weight), dict(status=st)),
        "step": (af.adaflash_opd_loss_fwd_bwd, (z, t, tok, doff, w.clip_c, w.ce_weight),
                 dict(grad_scale=0.5, status=st)),
        "sampled": (af.adaflash_verify_sampled, (z, t, tok, doff, 0.8, u_acc, u_smp), dict(status=st)),
    }


def _tensors(out):
    return out if isinstance(out, dict) else {"out": out}


@pytest.mark.parametrize("name", ["single", "c32"])
def test_prepared_calls_match_the_entry_points(name):
    import serving_packed_var_gb300 as af
    b = materialize(make_workload(name))
    w = b.w
    dev = torch.device("cuda:0")
    z, t = to_device(b.draft, w.d_dtype, dev), to_device(b.target, w.t_dtype, dev)
    tok, doff = torch.from_numpy(b.tokens).to(dev), torch.from_numpy(b.doff).to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    rng = np.random.default_rng(3)
    u_acc = torch.from_numpy(rng.random(w.num_draft_rows, dtype=np.float32)).to(dev)
    u_smp = torch.from_numpy(rng.random(w.num_requests, dtype=np.float32)).to(dev)
    for key, (fn, args, kw) in _calls(af, b, z, t, tok, doff, st, u_acc, u_smp).items():
        ref = {k: v.clone() for k, v in _tensors(fn(*args, **kw)).items()}
        torch.cuda.synchronize()
        n0 = af.adaflash_kernel_launches()
        fn(*args, **kw)
        torch.cuda.synchronize()
        per_call = af.adaflash_kernel_launches() - n0
        call, out = af.prepare(fn, *args, **kw)
        outs = _tensors(out)
        for _ in range(3):
            for v in outs.values():
                v.fill_(-3)
            n0 = af.adaflash_kernel_launches()
            call()
            torch.cuda.synchronize()
            assert af.adaflash_kernel_launches() - n0 == per_call, key
            for k in ref:
                assert torch.equal(outs[k], ref[k]), (key, k)
    # the backward, prepared on the forward's outputs
    f = af.adaflash_opd_loss_fwd(z, t, tok, doff, w.clip_c, w.ce_weight, status=st)
    g_ref = af.adaflash_opd_loss_bwd(z, t, doff, f["target_argmax"], f["row_stats"], w.clip_c, w.ce_weight,
                                     grad_scale=0.25, status=st).clone()
    call, g = af.prepare(af.adaflash_opd_loss_bwd, z, t, doff, f["target_argmax"], f["row_stats"], w.clip_c,
                         w.ce_weight, grad_scale=0.25, status=st)
    g.fill_(-3)
    call()
    torch.cuda.synchronize()
    assert torch.equal(g, g_ref)
    assert int(st.item()) == 0


def test_prepared_call_raises_like_the_entry_point():
    import serving_packed_var_gb300 as af
    b = materialize(custom(vocab=1024, k=[3, 2]))
    w = b.w
    dev = torch.device("cuda:0")
    t = to_device(b.target, w.t_dtype, dev)
    tok, doff = torch.from_numpy(b.tokens).to(dev), torch.from_numpy(b.doff).to(dev)
    with pytest.raises(af.AdaflashError):  # clip_c must be > 0: refused on the host, also when prepared
        af.prepare(af.adaflash_opd_loss_fwd, t, t, tok, doff, 0.0)[0]()
