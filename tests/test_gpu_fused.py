"""adaflash_opd_loss_fwd_bwd (the forward and the backward in one call) through the C ABI.

The call takes the on-chip fused kernel when rows are on the 16-byte grid and a row
pair fits a cluster's shared memory, the separate kernels otherwise.  Either way its
outputs are checked against the float64 oracle with the bars of the separate path
(parity_lib), and against adaflash_opd_loss_fwd + adaflash_opd_loss_bwd on the same
inputs: the integer outputs equal, the float outputs within float32 rounding of each
other (the two paths may split a row over different numbers of CTAs, which changes
the order of the partial sums).
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from parity_lib import GpuRun, check_loss, check_rows, check_verify, oracle_argmax_all, oracle_rows, to_device  # noqa: E402
from synth import make_workload, materialize  # noqa: E402
from synth.workloads import custom  # noqa: E402

KEYS = ("target_argmax", "accept_len", "bonus_token", "accept_rate", "kl_row", "ce_row", "row_stats", "loss")
INT_KEYS = ("target_argmax", "accept_len", "bonus_token", "accept_rate")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


class FusedRun:
    def __init__(self, b, grad_row=None, grad_scale=1.0, misalign=0, canary=16, ld_g=None, misalign_z=None,
                 misalign_t=None, misalign_g=0):
        import serving_packed_var_gb300 as af
        w = b.w
        dev = torch.device("cuda:0")
        z = to_device(b.draft, w.d_dtype, dev, misalign if misalign_z is None else misalign_z)
        t = to_device(b.target, w.t_dtype, dev, misalign if misalign_t is None else misalign_t)
        tok = torch.from_numpy(b.tokens).to(dev)
        doff = torch.from_numpy(b.doff).to(dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        R, Nd = w.num_requests, w.num_draft_rows
        Nt = Nd + R
        self._bufs = {}

        def buf(name, n, dtype, fill):
            full = torch.full((n + canary,), fill, dtype=dtype, device=dev)
            self._bufs[name] = (full, n, fill)
            return full[:n]

        ldg = w.vocab if ld_g is None else ld_g
        mg = misalign_g
        gfull = torch.full((mg + Nd * ldg + canary,), -7.0, dtype=torch.float32, device=dev)
        self._bufs["grad"] = (gfull, mg + Nd * ldg, -7.0)
        self._head = (gfull, mg, -7.0)
        out = dict(target_argmax=buf("target_argmax", Nt, torch.int32, -7),
                   accept_len=buf("accept_len", R, torch.int32, -7),
                   bonus_token=buf("bonus_token", R, torch.int32, -7),
                   accept_rate=buf("accept_rate", R, torch.float32, -7.0),
                   kl_row=buf("kl_row", Nd, torch.float32, -7.0),
                   ce_row=buf("ce_row", Nd, torch.float32, -7.0),
                   loss=buf("loss", 1, torch.float32, -7.0),
                   row_stats=buf("row_stats", 4 * Nd, torch.float32, -7.0).view(Nd, 4),
                   grad=gfull[mg:mg + Nd * ldg].view(Nd, ldg)[:, :w.vocab])
        gr = None if grad_row is None else torch.from_numpy(np.asarray(grad_row, dtype=np.float32)).to(dev)
        self.out = af.adaflash_opd_loss_fwd_bwd(z, t, tok, doff, w.clip_c, w.ce_weight, grad_row=gr,
                                                grad_scale=grad_scale, vocab=w.vocab, out=out, status=self.status)
        torch.cuda.synchronize()
        self.h = {k: v.cpu().numpy() for k, v in self.out.items() if k != "grad"}
        self.grad = self.out["grad"]
        self.status_word = int(self.status.item())
        self.w, self.b = w, b

    def grad_rows(self, rows):
        return {d: self.grad[d].cpu().numpy().astype(np.float64) for d in rows}

    def canaries_intact(self):
        for name, (full, n, fill) in self._bufs.items():
            if not bool((full[n:].cpu() == fill).all()):
                return name
        full, n, fill = self._head
        if n and not bool((full[:n].cpu() == fill).all()):
            return "grad head"
        return None


def _close_to_separate(b, grad_row=None, grad_scale=1.0, misalign=0, oracle_grad_rows=None, **shifts):
    f = FusedRun(b, grad_row=grad_row, grad_scale=grad_scale, misalign=misalign, **shifts)
    s = GpuRun(b, bwd=True, grad_row=grad_row, grad_scale=grad_scale, misalign=misalign, **shifts)
    assert f.status_word == s.status_word == 0, (f.status_word, s.status_word)
    assert f.canaries_intact() is None, f.canaries_intact()
    for k in INT_KEYS:
        assert np.array_equal(f.h[k].view(np.uint8), s.h[k].view(np.uint8)), k
    for k in ("kl_row", "ce_row", "loss"):
        assert np.allclose(f.h[k], s.h[k], rtol=1e-5, atol=1e-6), k
    fs, ss = f.h["row_stats"], s.h["row_stats"]
    assert np.allclose(fs[:, :2], ss[:, :2], rtol=1e-6, atol=1e-5), "lse"
    # S and the clipped count: equal unless a term lies within rounding of the clip
    assert np.mean(fs[:, 3] == ss[:, 3]) > 0.99, "n_clipped"
    gd = (f.grad - s.grad).abs()
    assert float(gd.max()) <= 1e-6 + 1e-4 * float(s.grad.abs().max()), float(gd.max())
    # and the oracle, with the separate path's bars
    w = b.w
    check_verify(f, oracle_argmax_all(b))
    rows = list(range(w.num_draft_rows))
    per, _ = oracle_rows(b, rows, bwd=False)
    gsel = rows if oracle_grad_rows is None else oracle_grad_rows
    _, grads = oracle_rows(b, gsel, bwd=True, grad_row=grad_row, grad_scale=grad_scale)
    check_rows(f, per, grads)
    if grad_row is None:
        check_loss(f, sum(per[d]["loss_row"] for d in rows) / len(rows))
    return f, s


@pytest.mark.parametrize("name", ["tiny", "single", "c32", "c128", "c128_clip"])
def test_workloads_against_oracle_and_separate(name):
    b = materialize(make_workload(name))
    nd = b.w.num_draft_rows
    gsel = None if nd <= 64 else sorted(set(np.random.default_rng(4).choice(nd, 24, replace=False)) | {0, nd - 1})
    _close_to_separate(b, grad_scale=0.37, oracle_grad_rows=gsel)


EDGE = [
    dict(vocab=1, k=[1, 2], accept="full"),
    dict(vocab=7, k=[3, 1, 16]),
    dict(vocab=9, k=[5, 5], d_dtype="fp32", t_dtype="fp32"),
    dict(vocab=1023, k=[16, 1], d_dtype="fp32", t_dtype="bf16"),
    dict(vocab=4096, k=[2, 7, 1], d_dtype="bf16", t_dtype="fp32"),
    dict(vocab=80000, k=[3, 16, 1], d_dtype="fp32", t_dtype="fp32"),
    dict(vocab=151936, k=[4, 9], d_dtype="fp32", t_dtype="bf16"),
    dict(vocab=262144, k=[2, 3], d_dtype="bf16", t_dtype="bf16"),
    dict(vocab=2048, k=[6, 2], ld_d=2048 + 8, ld_t=2048 + 16),
    dict(vocab=3000, k=[9], clip_c=0.01),
    dict(vocab=96, k=list(np.random.default_rng(9).integers(1, 17, size=700)), d_dtype="fp32", t_dtype="fp32"),
    # the largest vocabulary: no on-chip cluster holds a row, so the row pass with the gradient
    dict(vocab=524288, k=[16, 1], d_dtype="bf16", t_dtype="bf16"),
    dict(vocab=524287, k=[3, 16], d_dtype="fp32", t_dtype="bf16"),
]


@pytest.mark.parametrize("case", EDGE, ids=lambda c: f"V{c['vocab']}_k{len(c['k'])}")
def test_edge_shapes(case):
    b = materialize(custom(**case))
    nd = b.w.num_draft_rows
    gsel = None if nd * b.w.vocab <= 2_000_000 else sorted({0, nd // 2, nd - 1})
    _close_to_separate(b, oracle_grad_rows=gsel)


# More row units than the on-chip kernel takes: the single-pass row pass with the gradient (each
# slice read from HBM once; the second pass over it, for dz, is served by L2).
STREAM = [
    dict(vocab=151936, k=[16] * 8),
    # paired rows that all fit the L2 at once: one round of clusters (C = 8, 8, 6 here)
    dict(vocab=151936, k=[16] * 3),
    dict(vocab=151936, k=[16] * 4, d_dtype="fp32", t_dtype="bf16"),
    dict(vocab=151937, k=[16, 9, 16, 12, 16, 1], d_dtype="fp32", t_dtype="bf16"),
    dict(vocab=151936, k=[16, 3, 9, 1] * 6, d_dtype="fp32", t_dtype="bf16"),
    dict(vocab=40000, k=list(np.random.default_rng(11).integers(1, 17, size=200)), clip_c=0.05),
    dict(vocab=1000, k=[16] * 300, d_dtype="fp32", t_dtype="fp32"),
    dict(vocab=151936, k=[16, 5, 11] * 4, d_dtype="fp32", t_dtype="fp32", clip_c=0.2),
    # one float32 input and one bf16: a four-stage ring, so slices of three to six chunks take
    # the second pass's first chunks from the ring and the rest from memory
    dict(vocab=24577, k=[16] * 40, d_dtype="fp32", t_dtype="bf16"),
    dict(vocab=12291, k=[16, 7] * 30, d_dtype="bf16", t_dtype="fp32"),
    dict(vocab=49153, k=[16, 2] * 24, d_dtype="fp32", t_dtype="bf16"),
]


@pytest.mark.parametrize("case", STREAM, ids=lambda c: f"V{c['vocab']}_k{len(c['k'])}_{c.get('d_dtype', 'bf16')}")
def test_streaming_fwd_bwd_shapes(case):
    b = materialize(custom(**case))
    nd = b.w.num_draft_rows
    gsel = sorted(set(np.random.default_rng(5).choice(nd, 6, replace=False)) | {0, nd - 1})
    _close_to_separate(b, grad_scale=0.5, oracle_grad_rows=gsel)


def test_streaming_per_row_weights():
    # more row units than the on-chip kernel takes: the streaming pass with
    # an upstream weight per draft row
    w = custom(vocab=20000, k=[16, 7, 12, 3] * 12, clip_c=0.3)
    nd = w.num_draft_rows
    gsel = sorted(set(np.random.default_rng(6).choice(nd, 6, replace=False)) | {0, nd - 1})
    _close_to_separate(materialize(w), grad_row=np.linspace(-1.5, 2.0, nd), oracle_grad_rows=gsel)


def test_streaming_ragged_vocab_padded_rows():
    # V = 151937 (not a multiple of 8) with padded leading dimensions, so every row
    # still starts on the 16-byte grid: the last slice ends in a ragged group
    w = custom(vocab=151937, k=[5, 12] * 6, ld_d=151944, ld_t=151952)
    b = materialize(w)
    f = FusedRun(b, grad_scale=0.25, ld_g=151940)
    assert f.status_word == 0
    assert f.canaries_intact() is None, f.canaries_intact()
    check_verify(f, oracle_argmax_all(b))
    nd = w.num_draft_rows
    rows = [0, 7, nd - 1]
    per, grads = oracle_rows(b, rows, bwd=True, grad_scale=0.25)
    check_rows(f, per, grads)


@pytest.mark.parametrize("misalign", [1, 3])
def test_unaligned_rows_take_the_row_pass_with_the_gradient(misalign):
    _close_to_separate(materialize(custom(vocab=5000, k=[3, 8])), misalign=misalign)


def test_per_row_weights():
    w = custom(vocab=3000, k=[5, 2, 9], d_dtype="fp32", t_dtype="fp32")
    _close_to_separate(materialize(w), grad_row=np.linspace(-1.5, 2.0, w.num_draft_rows))


def test_clip_binds_against_oracle():
    b = materialize(make_workload("c128_clip"))
    w = b.w
    f = FusedRun(b, grad_scale=1.0)
    assert f.status_word == 0
    rows = sorted(set(int(r) for r in w.clip_rows[:6]) | {0, w.num_draft_rows - 1})
    per, grads = oracle_rows(b, rows, bwd=True)
    check_rows(f, per, grads)
    for d in w.clip_rows[:6]:
        assert int(f.h["row_stats"][int(d)][3]) == 64


def test_deterministic_bitwise():
    b = materialize(make_workload("c32"))
    r1, r2 = FusedRun(b), FusedRun(b)
    for k in KEYS:
        assert np.array_equal(r1.h[k].view(np.uint8), r2.h[k].view(np.uint8)), k
    assert torch.equal(r1.grad, r2.grad)


def test_bad_offsets_set_status():
    import serving_packed_var_gb300 as af
    w = custom(vocab=300, k=[4, 4, 4])
    b = materialize(w)
    dev = torch.device("cuda:0")
    z = to_device(b.draft, w.d_dtype, dev)
    t = to_device(b.target, w.t_dtype, dev)
    tok = torch.from_numpy(b.tokens).to(dev)
    bad_doff = torch.tensor([0, 4, 4, 12], dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    af.adaflash_opd_loss_fwd_bwd(z, t, tok, bad_doff, 1.0, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & (1 << af.ADAFLASH_ERR_BAD_OFFSETS)
