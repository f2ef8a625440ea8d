"""Seeded hidden states and LM-head weights for the logit-free verify + loss pass.

Shapes follow the Qwen3-8B setting of the AdaFlash article ("AdaFlash: Adaptive
Speculative Decoding with Online Self-Improvement for High-Concurrency LLM
Inference", "Experimental Results": Qwen3-8B target, hidden size 4096, vocabulary
151936) with the packed draft-block layout of the logits workloads.  No logits
are computed here: the module only draws random numbers, rounds them to bfloat16
and plants structure.

Recipe (all bfloat16, round to nearest even):
* target head W_t [V, H] ~ N(0, (sigma / sqrt(H))^2), so a unit-variance hidden row
  gives logits of standard deviation about sigma;
* draft head W_d = W_t (shared) or W_t + N(0, (head_noise * sigma / sqrt(H))^2);
* target hidden row s: h_s ~ N(0, 1) plus (spike / sigma^2) * W_t[a_s] for a seeded
  token a_s, which lifts logit a_s by about ``spike`` (chosen per vocabulary size so
  that a_s stays the argmax by several standard deviations while the target still
  puts visible mass elsewhere, and the draft much more);
* draft hidden row d (paired with target row s): draft_scale * Ht[s] + N(0, draft_noise^2);
* draft tokens: a_s for the planted accepted prefix j < L_i (a_s is the target's
  argmax by a wide margin), another token at j = L_i, uniform tokens after it.
"""

from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .workloads import Workload, _rng, bf16_bits_to_f32, f32_to_bf16_bits

_S_W = 11
_S_WD = 12
_S_HT = 13
_S_HD = 14
_S_SPIKE = 15
_S_TOK = 16


@dataclasses.dataclass
class LMHeadWorkload:
    name: str
    vocab: int
    hidden: int
    k: np.ndarray
    planted_accept: np.ndarray
    clip_c: float = 1.0
    ce_weight: float = 1.0
    seed: int = 0
    shared_head: bool = True
    sigma: float = 2.5
    spike: float = 18.0
    head_noise: float = 0.05
    draft_scale: float = 0.8
    draft_noise: float = 0.35

    def __post_init__(self):
        self.k = np.asarray(self.k, dtype=np.int32)
        self.planted_accept = np.asarray(self.planted_accept, dtype=np.int32)
        # the packed layout (row maps) of the logits workloads
        self.layout = Workload(name=self.name, vocab=self.vocab, k=self.k, planted_accept=self.planted_accept,
                               d_dtype="bf16", t_dtype="bf16", clip_c=self.clip_c, ce_weight=self.ce_weight,
                               seed=self.seed)

    @property
    def num_requests(self):
        return self.layout.num_requests

    @property
    def num_draft_rows(self):
        return self.layout.num_draft_rows

    @property
    def num_target_rows(self):
        return self.layout.num_target_rows

    @property
    def doff(self):
        return self.layout.doff

    def pair_target_row(self, d):
        return self.layout.pair_target_row(d)


@dataclasses.dataclass
class LMHeadBatch:
    w: LMHeadWorkload
    hd: np.ndarray      # uint16 bf16 bits [N_d, H]
    ht: np.ndarray      # uint16 bf16 bits [N_t, H]
    wd: np.ndarray      # uint16 bf16 bits [V, H] (the same array as wt when the head is shared)
    wt: np.ndarray      # uint16 bf16 bits [V, H]
    tokens: np.ndarray  # int32 [N_d]
    doff: np.ndarray    # int32 [R + 1]
    spike_token: np.ndarray  # int64 [N_t]

    def f32(self, name):
        return bf16_bits_to_f32(getattr(self, name))


def _normal_bf16(seed, stream, index, n, scale):
    rng = _rng(seed, stream, index)
    return f32_to_bf16_bits(rng.standard_normal(n, dtype=np.float32) * np.float32(scale))


def materialize_lmhead(w: LMHeadWorkload, threads: int | None = None) -> LMHeadBatch:
    V, H = w.vocab, w.hidden
    threads = threads or min(32, os.cpu_count() or 1)
    ws = w.sigma / np.sqrt(H)
    wt = np.empty((V, H), dtype=np.uint16)
    blk = 2048

    def head_block(b0):
        b1 = min(V, b0 + blk)
        wt[b0:b1] = _normal_bf16(w.seed, _S_W, b0, (b1 - b0) * H, ws).reshape(b1 - b0, H)

    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(head_block, range(0, V, blk)))
    if w.shared_head:
        wd = wt
    else:
        wd = np.empty_like(wt)

        def dhead_block(b0):
            b1 = min(V, b0 + blk)
            base = bf16_bits_to_f32(wt[b0:b1])
            noise = _rng(w.seed, _S_WD, b0).standard_normal((b1 - b0, H), dtype=np.float32) * np.float32(
                w.head_noise * ws)
            wd[b0:b1] = f32_to_bf16_bits(base + noise)

        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(dhead_block, range(0, V, blk)))

    Nd, Nt = w.num_draft_rows, w.num_target_rows
    ht = np.empty((Nt, H), dtype=np.uint16)
    spike = np.empty(Nt, dtype=np.int64)
    beta = np.float32(w.spike / (w.sigma ** 2))
    for s in range(Nt):
        rng = _rng(w.seed, _S_HT, s)
        a = int(_rng(w.seed, _S_SPIKE, s).integers(V))
        spike[s] = a
        h = rng.standard_normal(H, dtype=np.float32) + beta * bf16_bits_to_f32(wt[a])
        ht[s] = f32_to_bf16_bits(h)
    hd = np.empty((Nd, H), dtype=np.uint16)
    for d in range(Nd):
        s = w.pair_target_row(d)
        rng = _rng(w.seed, _S_HD, d)
        h = np.float32(w.draft_scale) * bf16_bits_to_f32(ht[s]) + np.float32(w.draft_noise) * rng.standard_normal(
            H, dtype=np.float32)
        hd[d] = f32_to_bf16_bits(h)

    toks = np.zeros(Nd, dtype=np.int32)
    doff = w.doff
    for i in range(w.num_requests):
        rng = _rng(w.seed, _S_TOK, i)
        L = int(w.planted_accept[i])
        for j in range(int(w.k[i])):
            d = int(doff[i]) + j
            a = int(spike[d + i])
            if j < L:
                toks[d] = a
            elif j == L:
                e = int(rng.integers(V - 1)) if V > 1 else 0
                toks[d] = e if e < a else e + 1
            else:
                toks[d] = int(rng.integers(V))
    return LMHeadBatch(w=w, hd=hd, ht=ht, wd=wd, wt=wt, tokens=toks, doff=np.asarray(doff, dtype=np.int32),
                       spike_token=spike)


def make_lmhead_workload(name: str, seed: int = 0, **over) -> LMHeadWorkload:
    """Named workloads.

    lm_tiny   V = 2048, H = 256, k = {16, 9, 3, 1}, separate heads
    lm_small  V = 8192, H = 512, 8 requests, k ~ U{1..16}, shared head
    lm_c32    V = 151936, H = 4096, 32 requests, k ~ U{1..16}, L ~ Bin(k, 0.6), shared head
    lm_c128   V = 151936, H = 4096, 128 requests, k ~ truncated geometric (p = 0.07), L ~ Bin(k, 0.6), shared head
    """
    meta = _rng(seed, 1, 99)
    if name == "lm_tiny":
        k = np.array([16, 9, 3, 1], dtype=np.int32)
        kw = dict(vocab=2048, hidden=256, shared_head=False, spike=12.0)
    elif name == "lm_small":
        k = meta.integers(1, 17, size=8).astype(np.int32)
        kw = dict(vocab=8192, hidden=512, spike=14.0)
    elif name == "lm_c32":
        k = meta.integers(1, 17, size=32).astype(np.int32)
        kw = dict(vocab=151936, hidden=4096)
    elif name == "lm_c128":
        ks = np.arange(1, 17)
        pr = 0.93 ** (ks - 1)
        k = meta.choice(ks, size=128, p=pr / pr.sum()).astype(np.int32)
        kw = dict(vocab=151936, hidden=4096, clip_c=0.5)
    else:
        raise KeyError(name)
    L = meta.binomial(k, 0.6).astype(np.int32)
    kw.update(name=name, k=k, planted_accept=L, seed=seed)
    kw.update(over)
    return LMHeadWorkload(**kw)


def custom_lmhead(vocab: int, hidden: int, k, seed: int = 0, **over) -> LMHeadWorkload:
    meta = _rng(seed, 1, 98)
    over.setdefault("spike", 12.0 if vocab <= 4096 else 14.0)
    k = np.asarray(k, dtype=np.int32)
    L = np.array([meta.integers(0, ki + 1) for ki in k], dtype=np.int32)
    return LMHeadWorkload(name=over.pop("name", "lm_custom"), vocab=vocab, hidden=hidden, k=k, planted_accept=L,
                          seed=seed, **over)
