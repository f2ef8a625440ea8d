"""Helpers shared by the GPU parity tests: upload a generated batch, run the CUDA
path through the C ABI, and compare with the oracle on the same inputs.

Tolerances (GPU vs float64 oracle):
  argmax, accept_len, bonus_token, accept_rate, n_clipped  -- bit-exact
  kl_row, ce_row, loss  -- |d| <= 1e-4 |ref| + 1e-6 for float32 inputs,
                           |d| <= 2e-3 |ref| + 1e-5 when an input is bfloat16
  row_stats S           -- the same, with |ref| replaced by |S| + sum_v m_v p_v |r_v + 1|
  grad                  -- |d| <= 1e-5 + 1e-3 |ref|   (upstream weight 1)
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle
import serving_packed_var_gb300 as af

THREADS = min(32, os.cpu_count() or 1)


def loss_tol(w):
    if w.d_dtype == "fp32" and w.t_dtype == "fp32":
        return 1e-4, 1e-6
    return 2e-3, 1e-5


GRAD_ABS, GRAD_REL = 1e-5, 1e-3


def to_device(arr: np.ndarray, dtype: str, dev, misalign: int = 0) -> torch.Tensor:
    """Host array (float32, or uint16 bf16 bits) -> 2-D CUDA tensor, optionally at an odd offset."""
    if dtype == "bf16":
        host = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16))
        tdt = torch.bfloat16
    else:
        host = torch.from_numpy(np.ascontiguousarray(arr))
        tdt = torch.float32
    if misalign == 0:
        return host.to(dev).view(tdt)
    n = host.numel()
    flat = torch.empty(n + misalign + 8, dtype=host.dtype, device=dev)
    flat[misalign:misalign + n].copy_(host.reshape(-1))
    return flat[misalign:misalign + n].view(tdt).view(arr.shape)


class GpuRun:
    """The forward, then (bwd) the backward, as separate calls.  misalign shifts the base
    pointers of both logit tensors by that many elements; misalign_z / misalign_t set
    them apart and misalign_g shifts the gradient's base."""

    def __init__(self, batch, dev="cuda:0", bwd=True, grad_row=None, grad_scale=1.0, misalign=0, canary=16,
                 misalign_z=None, misalign_t=None, misalign_g=0):
        w = batch.w
        self.b = batch
        self.w = w
        dev = torch.device(dev)
        self.z = to_device(batch.draft, w.d_dtype, dev, misalign if misalign_z is None else misalign_z)
        self.t = to_device(batch.target, w.t_dtype, dev, misalign if misalign_t is None else misalign_t)
        self.tok = torch.from_numpy(batch.tokens).to(dev)
        self.doff = torch.from_numpy(batch.doff).to(dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        R, Nd = w.num_requests, w.num_draft_rows
        Nt = Nd + R
        self.canary = canary
        self._bufs = {}

        def buf(name, n, dtype, fill):
            full = torch.full((n + canary,), fill, dtype=dtype, device=dev)
            self._bufs[name] = (full, n, fill)
            return full[:n]

        out = dict(
            target_argmax=buf("target_argmax", Nt, torch.int32, -7),
            accept_len=buf("accept_len", R, torch.int32, -7),
            bonus_token=buf("bonus_token", R, torch.int32, -7),
            accept_rate=buf("accept_rate", R, torch.float32, -7.0),
            kl_row=buf("kl_row", Nd, torch.float32, -7.0),
            ce_row=buf("ce_row", Nd, torch.float32, -7.0),
            loss=buf("loss", 1, torch.float32, -7.0),
        )
        rs = buf("row_stats", 4 * Nd, torch.float32, -7.0)
        out["row_stats"] = rs.view(Nd, 4)
        self.out = af.adaflash_opd_loss_fwd(self.z, self.t, self.tok, self.doff, w.clip_c, w.ce_weight,
                                            vocab=w.vocab, out=out, status=self.status)
        self.grad = None
        if bwd:
            self.grad_row = None if grad_row is None else torch.from_numpy(
                np.asarray(grad_row, dtype=np.float32)).to(dev)
            mg = misalign_g
            gfull = torch.full((mg + Nd * w.vocab + canary,), -7.0, dtype=torch.float32, device=dev)
            self._bufs["grad"] = (gfull, mg + Nd * w.vocab, -7.0)
            self._heads = [(gfull, mg, -7.0)]
            g = gfull[mg:mg + Nd * w.vocab].view(Nd, w.vocab)
            self.grad = af.adaflash_opd_loss_bwd(self.z, self.t, self.doff, self.out["target_argmax"],
                                                 self.out["row_stats"], w.clip_c, w.ce_weight,
                                                 grad_row=self.grad_row, grad_scale=grad_scale, vocab=w.vocab,
                                                 out=g, status=self.status)
        torch.cuda.synchronize()
        self.h = {k: v.cpu().numpy() for k, v in self.out.items()}
        self.status_word = int(self.status.item())

    def canaries_intact(self):
        for name, (full, n, fill) in self._bufs.items():
            tail = full[n:].cpu()
            if not bool((tail == fill).all()):
                return name
        for full, n, fill in getattr(self, "_heads", []):
            if n and not bool((full[:n].cpu() == fill).all()):
                return "grad head"
        return None

    def grad_rows(self, rows):
        return {d: self.grad[d].cpu().numpy().astype(np.float64) for d in rows}


def oracle_rows(batch, rows, bwd=True, grad_row=None, grad_scale=1.0):
    """Oracle forward (and gradient) of the listed draft rows, thread-parallel."""
    w = batch.w

    def one(d):
        s = w.pair_target_row(d)
        z = batch.draft_f64(d)
        t = batch.target_f64(s)
        f = oracle.row_forward(z, t, w.clip_c, w.ce_weight)
        g = None
        if bwd:
            gw = float(grad_row[d]) if grad_row is not None else grad_scale
            g = oracle.row_grad(z, t, w.clip_c, w.ce_weight, gw)
        return d, f, g

    with ThreadPoolExecutor(THREADS) as ex:
        res = list(ex.map(one, rows))
    return {d: f for d, f, _ in res}, {d: g for d, _, g in res}


def oracle_argmax_all(batch):
    w = batch.w
    with ThreadPoolExecutor(THREADS) as ex:
        return np.array(list(ex.map(lambda s: oracle.first_argmax(batch.target_f64(s)),
                                    range(w.num_target_rows))), dtype=np.int64)


def check_verify(run: GpuRun, argmax_ref: np.ndarray):
    """Bit-exact verification outputs for every request."""
    w, b, h = run.w, run.b, run.h
    assert np.array_equal(h["target_argmax"].astype(np.int64), argmax_ref), "target_argmax differs"
    for i in range(w.num_requests):
        d0 = int(b.doff[i])
        k = int(w.k[i])
        L, bonus = oracle.greedy_accept(b.tokens[d0:d0 + k], argmax_ref[d0 + i:d0 + i + k + 1])
        assert h["accept_len"][i] == L, (i, h["accept_len"][i], L)
        assert h["bonus_token"][i] == bonus, (i, h["bonus_token"][i], bonus)
        assert h["accept_rate"][i].view(np.uint32) == oracle.acceptance_rate(L, k).view(np.uint32), i


def check_rows(run: GpuRun, per: dict, grads: dict | None = None):
    w, h = run.w, run.h
    rel, ab = loss_tol(w)
    for d, f in per.items():
        for key in ("kl", "ce"):
            got = float(h[key + "_row"][d])
            assert abs(got - f[key]) <= rel * abs(f[key]) + ab, (key, d, got, f[key])
        st = h["row_stats"][d]
        assert abs(st[0] - f["lse_z"]) <= 1e-5 * abs(f["lse_z"]) + 1e-5, ("lse_z", d, st[0], f["lse_z"])
        assert abs(st[1] - f["lse_t"]) <= 1e-5 * abs(f["lse_t"]) + 1e-5, ("lse_t", d, st[1], f["lse_t"])
        # S = sum m p (r+1) can be a small difference of large sums: judged against its summands' size
        assert abs(st[2] - f["S"]) <= rel * (abs(f["S"]) + f["S_l1"]) + ab, ("S", d, st[2], f["S"])
        assert int(st[3]) == f["n_clipped"], ("n_clipped", d, st[3], f["n_clipped"])
        assert h["target_argmax"][w.pair_target_row(d)] == f["argmax"], ("argmax", d)
    if grads:
        g = run.grad_rows(list(grads))
        for d, ref in grads.items():
            err = np.abs(g[d] - ref)
            bad = err > GRAD_ABS + GRAD_REL * np.abs(ref)
            assert not bad.any(), ("grad", d, int(np.argmax(err)), float(err.max()))


def check_loss(run: GpuRun, loss_ref: float):
    rel, ab = loss_tol(run.w)
    got = float(run.h["loss"][0])
    assert abs(got - loss_ref) <= rel * abs(loss_ref) + ab, (got, loss_ref)
