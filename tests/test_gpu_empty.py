"""An empty batch (no requests, no rows) through every entry point.

Nothing is read: the row, token and offset pointers of empty tensors are NULL and are accepted.
Nothing is launched: the library's kernel count does not move.  The only write is the loss,
set to 0, where the entry point has one.
"""

import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def test_empty_batch_every_entry_point():
    import serving_packed_var_gb300 as af
    dev = torch.device("cuda:0")
    V, H = 1024, 64
    z = torch.empty((0, V), dtype=torch.bfloat16, device=dev)
    t = torch.empty((0, V), dtype=torch.float32, device=dev)
    tok = torch.empty(0, dtype=torch.int32, device=dev)
    doff = torch.zeros(1, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    nan = float("nan")
    torch.cuda.synchronize()
    n0 = af.adaflash_kernel_launches()

    v = af.adaflash_verify_packed(t, tok, doff, status=st)
    assert all(x.numel() == 0 for x in v.values())
    f = af.adaflash_opd_loss_fwd(z, t, tok, doff, 0.5, out={"loss": torch.full((1,), nan, device=dev)}, status=st)
    g = af.adaflash_opd_loss_bwd(z, t, doff, f["target_argmax"], f["row_stats"], 0.5, status=st)
    assert g.numel() == 0
    fb = af.adaflash_opd_loss_fwd_bwd(z, t, tok, doff, 0.5, out={"loss": torch.full((1,), nan, device=dev)},
                                      status=st)
    u = torch.empty(0, dtype=torch.float32, device=dev)
    s = af.adaflash_verify_sampled(z, t, tok, doff, 0.8, u, u, status=st)
    assert all(x.numel() == 0 for x in s.values())
    hidden = torch.empty((0, H), dtype=torch.bfloat16, device=dev)
    head = torch.randn((V, H), device=dev).to(torch.bfloat16)
    lm = af.adaflash_lmhead_opd_fwd(hidden, hidden, head, head, tok, doff, 0.5,
                                    out={"loss": torch.full((1,), nan, device=dev)}, status=st)
    torch.cuda.synchronize()
    assert af.adaflash_kernel_launches() == n0
    assert int(st.item()) == 0
    for o in (f, fb, lm):
        assert float(o["loss"].item()) == 0.0
