"""adaflash_lmhead_opd_fwd_static: the logit-free forward for callers that cannot allocate.

A plugin that runs inside a framework owning all device memory may be unable (or not
allowed) to call cudaMalloc, so it cannot provide the workspace that
adaflash_lmhead_opd_fwd takes.  This entry point keeps that scratch in a static
device array inside the library instead.  The test calls it through the C ABI twice in
a row and checks each call against adaflash_lmhead_opd_fwd with a caller-provided
workspace, with the bars of the LM-head tests (integer outputs equal; float outputs
within 2e-3 relative + 1e-5), and checks that a batch larger than the array is refused.
"""

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from synth.lmhead import make_lmhead_workload, materialize_lmhead  # noqa: E402

REL, ABS = 2e-3, 1e-5
INT_KEYS = ("target_argmax", "accept_len", "bonus_token", "accept_rate")
FLOAT_KEYS = ("kl_row", "ce_row", "row_stats", "loss")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _call_static(lib, hd, ht, wd, wt, tok, doff, w, status):
    R, Nd = w.num_requests, w.num_draft_rows
    o = dict(target_argmax=torch.full((Nd + R,), -7, dtype=torch.int32, device="cuda"),
             accept_len=torch.full((R,), -7, dtype=torch.int32, device="cuda"),
             bonus_token=torch.full((R,), -7, dtype=torch.int32, device="cuda"),
             accept_rate=torch.full((R,), -7.0, device="cuda"),
             kl_row=torch.full((Nd,), -7.0, device="cuda"),
             ce_row=torch.full((Nd,), -7.0, device="cuda"),
             row_stats=torch.full((Nd, 4), -7.0, device="cuda"),
             loss=torch.full((1,), -7.0, device="cuda"))
    H = w.hidden
    code = lib.adaflash_lmhead_opd_fwd_static(
        hd.data_ptr(), hd.stride(0), ht.data_ptr(), ht.stride(0), wd.data_ptr(), wd.stride(0), wt.data_ptr(),
        wt.stride(0), H, tok.data_ptr(), doff.data_ptr(), R, Nd, w.vocab, w.clip_c, w.ce_weight,
        o["target_argmax"].data_ptr(), o["accept_len"].data_ptr(), o["bonus_token"].data_ptr(),
        o["accept_rate"].data_ptr(), o["kl_row"].data_ptr(), o["ce_row"].data_ptr(), o["row_stats"].data_ptr(),
        o["loss"].data_ptr(), status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return code, o


@pytest.mark.parametrize("name", ["lm_tiny", "lm_small"])
def test_static_scratch_matches_workspace_path_twice(name):
    import serving_packed_var_gb300 as af
    from serving_packed_var_gb300 import _native
    lib = _native.lib()
    b = materialize_lmhead(make_lmhead_workload(name))
    w = b.w
    hd, ht = _dev_bf16(b.hd), _dev_bf16(b.ht)
    wd = _dev_bf16(b.wd)
    wt = wd if b.wd is b.wt else _dev_bf16(b.wt)
    tok, doff = torch.from_numpy(b.tokens).cuda(), torch.from_numpy(b.doff).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = af.adaflash_lmhead_opd_fwd(hd, ht, wd, wt, tok, doff, w.clip_c, w.ce_weight, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = {k: v.cpu().numpy() for k, v in ref.items()}
    for call in range(2):
        st.zero_()
        code, out = _call_static(lib, hd, ht, wd, wt, tok, doff, w, st)
        torch.cuda.synchronize()
        assert code == _native.ADAFLASH_OK, (call, _native.status_string(code))
        assert int(st.item()) == 0, call
        got = {k: v.cpu().numpy() for k, v in out.items()}
        for k in INT_KEYS:
            assert np.array_equal(got[k].view(np.uint8), ref[k].view(np.uint8)), (call, k)
        for k in FLOAT_KEYS:
            assert np.allclose(got[k], ref[k], rtol=REL, atol=ABS), (call, k)


def test_batch_beyond_the_array_is_refused():
    from serving_packed_var_gb300 import _native
    lib = _native.lib()
    fake = ctypes.c_void_p(0x10000)
    R, Nd, V, H = 128, 2000, 524288, 4096
    assert lib.adaflash_lmhead_workspace_bytes(R, Nd, V, H) > (48 << 20)
    code = lib.adaflash_lmhead_opd_fwd_static(fake, H, fake, H, fake, H, fake, H, H, fake, fake, R, Nd, V, 1.0, 1.0,
                                              fake, fake, fake, fake, fake, fake, fake, fake, None, None)
    assert code == _native.ADAFLASH_ERR_UNSUPPORTED
