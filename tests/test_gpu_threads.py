"""Host threads calling the library at once, each on its own stream.

The entry points keep small host-side tables (occupancy per kernel and cluster size, each
kernel's shared-memory limit, device attributes) that several host threads may fill at the same
time.  Four threads run the step, the forward, the verification and the sampled verification on
batches of different vocabularies (so different cluster sizes and shared-memory sizes of the same
kernels), each many times; every result must equal, bit for bit, the one the same call gave from
a single thread before.
"""

import threading

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

from parity_lib import to_device  # noqa: E402
from synth import materialize  # noqa: E402
from synth.workloads import custom  # noqa: E402

CASES = [dict(vocab=151936, k=[16, 3, 7]), dict(vocab=40001, k=[5] * 12, d_dtype="fp32", t_dtype="bf16"),
         dict(vocab=9000, k=[16] * 9, d_dtype="fp32", t_dtype="fp32"), dict(vocab=151937, k=[2, 16, 9, 1],
                                                                            d_dtype="fp32", t_dtype="bf16")]
ITERS = 12


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


class Batch:
    def __init__(self, case, dev):
        import serving_packed_var_gb300 as af
        self.af = af
        b = materialize(custom(**case))
        w = self.w = b.w
        self.z, self.t = to_device(b.draft, w.d_dtype, dev), to_device(b.target, w.t_dtype, dev)
        self.tok, self.doff = torch.from_numpy(b.tokens).to(dev), torch.from_numpy(b.doff).to(dev)
        g = torch.Generator().manual_seed(3)
        self.ua = torch.rand(w.num_draft_rows, generator=g).to(dev)
        self.us = torch.rand(w.num_requests, generator=g).to(dev)

    def run(self, st, stream):
        af, w = self.af, self.w
        return {
            "step": af.adaflash_opd_loss_fwd_bwd(self.z, self.t, self.tok, self.doff, w.clip_c, w.ce_weight,
                                                 grad_scale=1.0, status=st, stream=stream),
            "fwd": af.adaflash_opd_loss_fwd(self.z, self.t, self.tok, self.doff, w.clip_c, w.ce_weight, status=st,
                                            stream=stream),
            "verify": af.adaflash_verify_packed(self.t, self.tok, self.doff, status=st, stream=stream),
            "sampled": af.adaflash_verify_sampled(self.z, self.t, self.tok, self.doff, 0.9, self.ua, self.us,
                                                  status=st, stream=stream),
        }


def _same(a, b):
    for call in a:
        for k in a[call]:
            if not torch.equal(a[call][k], b[call][k]):
                return (call, k)
    return None


def test_four_host_threads_on_their_own_streams():
    dev = torch.device("cuda:0")
    batches = [Batch(c, dev) for c in CASES]
    st0 = torch.zeros(1, dtype=torch.int32, device=dev)
    refs = [b.run(st0, None) for b in batches]
    torch.cuda.synchronize()
    assert int(st0.item()) == 0
    errors = []

    def worker(j):
        try:
            stream = torch.cuda.Stream(device=dev)
            st = torch.zeros(1, dtype=torch.int32, device=dev)
            for it in range(ITERS):
                b = batches[(j + it) % len(batches)]
                out = b.run(st, stream)
                stream.synchronize()
                bad = _same(out, refs[(j + it) % len(batches)])
                if bad is not None:
                    errors.append((j, it, bad))
            if int(st.item()) != 0:
                errors.append((j, "status", int(st.item())))
        except Exception as e:  # reported below, with the thread's number
            errors.append((j, repr(e)))

    threads = [threading.Thread(target=worker, args=(j,)) for j in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors[:5]
