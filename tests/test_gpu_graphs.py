"""The entry points enqueue only kernels (no allocation, no synchronisation), so a step
can be captured once into a CUDA graph and replayed: replays must give the eager
results bit for bit.  The first eager call of each entry point comes before the
capture (it caches per-device launch geometry)."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from parity_lib import to_device  # noqa: E402
from synth import make_workload, materialize  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("name", ["single", "c32"])
def test_step_replays_in_a_cuda_graph(name):
    import serving_packed_var_gb300 as af
    b = materialize(make_workload(name))
    w = b.w
    dev = torch.device("cuda:0")
    z, t = to_device(b.draft, w.d_dtype, dev), to_device(b.target, w.t_dtype, dev)
    tok, doff = torch.from_numpy(b.tokens).to(dev), torch.from_numpy(b.doff).to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        # eager, on the capture stream (also fills every cache before the capture)
        out = af.adaflash_opd_loss_fwd(z, t, tok, doff, w.clip_c, w.ce_weight, status=st)
        g = af.adaflash_opd_loss_bwd(z, t, doff, out["target_argmax"], out["row_stats"], w.clip_c, w.ce_weight,
                                     grad_scale=1.0 / w.num_draft_rows, status=st)
        fb = af.adaflash_opd_loss_fwd_bwd(z, t, tok, doff, w.clip_c, w.ce_weight, grad_scale=1.0 / w.num_draft_rows,
                                          status=st)
    s.synchronize()
    ref = {k: v.clone() for k, v in out.items()}
    ref_g, ref_fb = g.clone(), {k: v.clone() for k, v in fb.items()}
    for v in list(out.values()) + [g] + list(fb.values()):
        v.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        af.adaflash_opd_loss_fwd(z, t, tok, doff, w.clip_c, w.ce_weight, out=out, status=st)
        af.adaflash_opd_loss_bwd(z, t, doff, out["target_argmax"], out["row_stats"], w.clip_c, w.ce_weight,
                                 grad_scale=1.0 / w.num_draft_rows, out=g, status=st)
        af.adaflash_opd_loss_fwd_bwd(z, t, tok, doff, w.clip_c, w.ce_weight, grad_scale=1.0 / w.num_draft_rows,
                                     out=fb, status=st)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for k in ref:
        assert torch.equal(out[k], ref[k]), k
    assert torch.equal(g, ref_g)
    for k in ref_fb:
        assert torch.equal(fb[k], ref_fb[k]), ("fwd_bwd", k)
