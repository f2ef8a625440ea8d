"""The C-ABI library builds, loads, exports every declared entry point, and
rejects malformed arguments on the host before touching CUDA (no GPU needed)."""

import ctypes
import math

import pytest

from serving_packed_var_gb300 import _native
from serving_packed_var_gb300.build import build

INVALID = _native.ADAFLASH_ERR_INVALID_ARG
UNSUPPORTED = _native.ADAFLASH_ERR_UNSUPPORTED
FAKE = 0x10000  # a non-NULL, well-aligned address; never dereferenced by host validation


@pytest.fixture(scope="module")
def lib():
    build()
    return _native.lib()


def test_exports_every_declared_function(lib):
    names = _native.declared_functions()
    assert set(names) == set(_native.SIGNATURES), names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(7):
        s = _native.status_string(code)
        assert s.startswith("ADAFLASH_") and "UNKNOWN" not in s
    assert "UNKNOWN" in _native.status_string(99)


def _verify(lib, **kw):
    a = dict(t=FAKE, t_dtype=1, ld_t=1024, tok=FAKE, doff=FAKE, R=4, Nd=29, V=1024, amax=FAKE, acc=FAKE,
             bonus=FAKE, rate=FAKE, status=None, stream=None)
    a.update(kw)
    return lib.adaflash_verify_packed(a["t"], a["t_dtype"], a["ld_t"], a["tok"], a["doff"], a["R"], a["Nd"],
                                      a["V"], a["amax"], a["acc"], a["bonus"], a["rate"], a["status"], a["stream"])


def _fwd(lib, **kw):
    a = dict(z=FAKE, zd=1, ldz=1024, t=FAKE, td=1, ldt=1024, tok=FAKE, doff=FAKE, R=4, Nd=29, V=1024, c=1.0,
             beta=1.0)
    a.update(kw)
    return lib.adaflash_opd_loss_fwd(a["z"], a["zd"], a["ldz"], a["t"], a["td"], a["ldt"], a["tok"], a["doff"],
                                     a["R"], a["Nd"], a["V"], a["c"], a["beta"], FAKE, FAKE, FAKE, FAKE, FAKE,
                                     FAKE, FAKE, a.get("loss", FAKE), None, None)


def _bwd(lib, **kw):
    a = dict(z=FAKE, zd=1, ldz=1024, t=FAKE, td=1, ldt=1024, doff=FAKE, R=4, Nd=29, V=1024, c=1.0, beta=1.0,
             amax=FAKE, stats=FAKE, grow=None, gs=1.0, g=FAKE, ldg=1024)
    a.update(kw)
    return lib.adaflash_opd_loss_bwd(a["z"], a["zd"], a["ldz"], a["t"], a["td"], a["ldt"], a["doff"], a["R"],
                                     a["Nd"], a["V"], a["c"], a["beta"], a["amax"], a["stats"], a["grow"], a["gs"],
                                     a["g"], a["ldg"], None, None)


@pytest.mark.parametrize("kw", [
    dict(t=None), dict(tok=None), dict(doff=None), dict(amax=None), dict(acc=None), dict(bonus=None),
    dict(rate=None), dict(V=0), dict(V=-3), dict(ld_t=1000), dict(t_dtype=2), dict(t_dtype=-1), dict(R=-1),
    dict(Nd=3), dict(Nd=4 * 16 + 1), dict(R=0, Nd=5), dict(t=FAKE + 1), dict(tok=FAKE + 2),
    dict(status=FAKE + 1),
])
def test_verify_rejects(lib, kw):
    assert _verify(lib, **kw) == INVALID


def test_empty_batch_reads_no_row_pointers(lib):
    # An empty batch passes the argument checks with NULL row, token, offset and output
    # pointers: the status is the device check's (OK on a GB300), never INVALID_ARG.  No
    # case here reaches a write (the loss write of an empty forward is not exercised).
    empty = dict(R=0, Nd=0)
    assert _verify(lib, t=None, tok=None, doff=None, amax=None, acc=None, bonus=None, rate=None, **empty) != INVALID
    assert _bwd(lib, z=None, t=None, doff=None, amax=None, stats=None, g=None, **empty) != INVALID
    # what is still checked: the loss pointer, the scalars, the counts
    assert _fwd(lib, z=None, t=None, tok=None, doff=None, loss=None, **empty) == INVALID
    assert _fwd(lib, c=0.0, loss=None, **empty) == INVALID
    assert _bwd(lib, gs=float("nan"), **empty) == INVALID
    assert _verify(lib, R=0, Nd=3) == INVALID


def test_verify_vocab_too_large(lib):
    V = _native.ADAFLASH_MAX_VOCAB + 1
    assert _verify(lib, V=V, ld_t=V) == UNSUPPORTED


@pytest.mark.parametrize("kw", [
    dict(z=None), dict(t=None), dict(zd=3), dict(ldz=10), dict(ldt=10), dict(c=0.0), dict(c=-1.0),
    dict(c=float("nan")), dict(beta=float("inf")), dict(beta=float("nan")), dict(loss=None), dict(z=FAKE + 2, zd=0),
    dict(Nd=2),
])
def test_fwd_rejects(lib, kw):
    assert _fwd(lib, **kw) == INVALID


@pytest.mark.parametrize("kw", [
    dict(g=None), dict(stats=None), dict(amax=None), dict(ldg=100), dict(gs=float("nan")), dict(grow=FAKE + 1),
    dict(c=0.0), dict(g=FAKE + 2),
])
def test_bwd_rejects(lib, kw):
    assert _bwd(lib, **kw) == INVALID


def _fwdbwd(lib, **kw):
    a = dict(z=FAKE, zd=1, ldz=1024, t=FAKE, td=1, ldt=1024, tok=FAKE, doff=FAKE, R=4, Nd=29, V=1024, c=1.0,
             beta=1.0, grow=None, gs=1.0, loss=FAKE, g=FAKE, ldg=1024)
    a.update(kw)
    return lib.adaflash_opd_loss_fwd_bwd(a["z"], a["zd"], a["ldz"], a["t"], a["td"], a["ldt"], a["tok"], a["doff"],
                                         a["R"], a["Nd"], a["V"], a["c"], a["beta"], a["grow"], a["gs"], FAKE, FAKE,
                                         FAKE, FAKE, FAKE, FAKE, FAKE, a["loss"], a["g"], a["ldg"], None, None)


@pytest.mark.parametrize("kw", [
    dict(z=None), dict(t=None), dict(tok=None), dict(doff=None), dict(loss=None), dict(g=None), dict(ldg=1000),
    dict(g=FAKE + 2), dict(grow=FAKE + 1), dict(c=0.0), dict(c=float("nan")), dict(beta=float("inf")),
    dict(gs=float("nan")), dict(zd=7), dict(ldz=5), dict(Nd=3), dict(R=-2),
])
def test_fwd_bwd_rejects(lib, kw):
    assert _fwdbwd(lib, **kw) == INVALID


def _sampled(lib, **kw):
    a = dict(z=FAKE, zd=1, ldz=1024, t=FAKE, td=1, ldt=1024, tok=FAKE, doff=FAKE, R=4, Nd=29, V=1024, T=1.0,
             ua=FAKE, us=FAKE, lse=FAKE, acc=FAKE, nxt=FAKE, rate=FAKE, status=None)
    a.update(kw)
    return lib.adaflash_verify_sampled(a["z"], a["zd"], a["ldz"], a["t"], a["td"], a["ldt"], a["tok"], a["doff"],
                                       a["R"], a["Nd"], a["V"], a["T"], a["ua"], a["us"], a["lse"], a["acc"],
                                       a["nxt"], a["rate"], a["status"], None)


@pytest.mark.parametrize("kw", [
    dict(z=None), dict(t=None), dict(tok=None), dict(doff=None), dict(ua=None), dict(us=None), dict(lse=None),
    dict(acc=None), dict(nxt=None), dict(rate=None), dict(ua=FAKE + 2), dict(lse=FAKE + 1), dict(T=0.0),
    dict(T=-1.0), dict(T=float("nan")), dict(T=float("inf")), dict(T=1e-45), dict(ldz=100), dict(td=5),
    dict(Nd=3), dict(status=FAKE + 3),
])
def test_sampled_rejects(lib, kw):
    assert _sampled(lib, **kw) == INVALID


def test_sampled_vocab_too_large(lib):
    V = _native.ADAFLASH_MAX_VOCAB + 1
    assert _sampled(lib, V=V, ldz=V, ldt=V) == UNSUPPORTED


def test_selftest_rejects_bad_limit(lib):
    assert lib.adaflash_selftest_bounded_wait(FAKE, 0, None) == INVALID
    assert lib.adaflash_selftest_bounded_wait(None, 10, None) == INVALID
    assert lib.adaflash_selftest_bounded_wait(FAKE, 2000000, None) == INVALID


def test_valid_call_without_gpu_reports_cuda_or_unsupported(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; the device path is covered by the gpu tests")
    # arguments pass host validation, the device check then fails cleanly
    assert _fwd(lib, c=math.inf) in (_native.ADAFLASH_ERR_CUDA, UNSUPPORTED)


def test_python_binding_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    import serving_packed_var_gb300 as af
    t = torch.zeros(2, 8)
    with pytest.raises(ValueError):
        af.adaflash_verify_packed(t, torch.zeros(1, dtype=torch.int32), torch.zeros(2, dtype=torch.int32))


def _lmhead(lib, static, **kw):
    a = dict(hd=FAKE, ldhd=256, ht=FAKE, ldht=256, wd=FAKE, ldwd=256, wt=FAKE, ldwt=256, H=256, tok=FAKE, doff=FAKE,
             R=4, Nd=29, V=2048, c=1.0, beta=1.0, loss=FAKE, kl=FAKE, status=None)
    a.update(kw)
    head = (a["hd"], a["ldhd"], a["ht"], a["ldht"], a["wd"], a["ldwd"], a["wt"], a["ldwt"], a["H"], a["tok"],
            a["doff"], a["R"], a["Nd"], a["V"], a["c"], a["beta"])
    outs = (FAKE, FAKE, FAKE, FAKE, a["kl"], FAKE, FAKE, a["loss"], a["status"], None)
    if static:
        return lib.adaflash_lmhead_opd_fwd_static(*head, *outs)
    return lib.adaflash_lmhead_opd_fwd(*head, FAKE, 1 << 40, *outs)


@pytest.mark.parametrize("kw", [
    dict(hd=None), dict(wt=None), dict(hd=FAKE + 8), dict(ldhd=100), dict(ldwd=260), dict(H=100), dict(H=32),
    dict(tok=None), dict(doff=FAKE + 2), dict(loss=None), dict(kl=FAKE + 1), dict(c=0.0), dict(c=float("nan")),
    dict(beta=float("inf")), dict(Nd=3), dict(R=-1), dict(status=FAKE + 2),
    # oversized for the static array as well as invalid: the argument error wins
    dict(R=128, Nd=2000, V=524288, H=4096, ldhd=4096, ldht=4096, ldwd=4096, ldwt=4096, tok=None),
])
def test_lmhead_entry_points_reject_alike(lib, kw):
    """The static-scratch entry point reports the same status as the workspace one for bad arguments."""
    assert _lmhead(lib, False, **kw) == INVALID
    assert _lmhead(lib, True, **kw) == INVALID
