"""Workload definitions and seeded generators.

Every random draw comes from its own counter-keyed Philox stream
``(seed, stream, index)``, so any row can be rebuilt on its own and rows can be
generated on many threads in any order with the same result.

The workloads mirror the shapes of the AdaFlash serving setting (page
"AdaFlash: Adaptive Speculative Decoding with Online Self-Improvement for
High-Concurrency LLM Inference", sections "Adaptive Length Head", "Variable-length
request packing" and "Experimental Results"):

* a draft block holds k_i <= 16 tokens (the fixed verification length k = 16
  that the length head shortens);
* requests of different k_i are packed back to back, described by an int32
  exclusive prefix sum ``doff`` of the k_i;
* serving concurrency 1, 32 and 128;
* the Qwen3 vocabulary of 151936 entries.

Packed layout (shared by every consumer):

* draft logits: ``N_d = doff[R]`` rows, request i owns rows ``doff[i] .. doff[i+1]-1``;
* target logits: ``N_t = N_d + R`` rows, request i owns rows
  ``doff[i]+i .. doff[i+1]+i``; draft row ``doff[i]+j`` pairs with target row
  ``doff[i]+i+j`` and target row ``doff[i+1]+i`` is the request's bonus row.

Value recipe (all workloads): target ~ N(0, 3^2) in float32 plus +8 at one
seeded entry per row; draft = 0.8 * (rounded target) + N(0, 1); each tensor is
then rounded to its storage dtype (float32, or bfloat16 round-to-nearest-even).
Draft tokens equal the target row's first maximising index for the planted
prefix j < L_i, a different uniformly drawn token at j = L_i, and uniform
tokens after it.
"""

from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

# Stream identifiers of the counter-keyed generators.
_S_META = 1
_S_TARGET = 2
_S_DRAFT = 3
_S_TOKEN = 4
_S_PLANT = 5
_S_TIE = 6

# Value written to row padding (ld > V): a huge finite number, so a kernel that
# reads past the vocabulary gets visibly wrong maxima instead of NaN noise.
PAD_F32 = np.float32(3.0e38)
PAD_BF16_BITS = np.uint16(0x7F7F)  # largest finite bfloat16 (~3.39e38)

MAX_K = 16


def _rng(seed: int, stream: int, index: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, stream, index])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to the float32 values they encode (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to the storage dtype; returns float32 holding exact stored values."""
    if dtype == "fp32":
        return np.asarray(x, dtype=np.float32)
    if dtype == "bf16":
        return bf16_bits_to_f32(f32_to_bf16_bits(x))
    raise ValueError(dtype)


@dataclasses.dataclass
class Workload:
    """One packed batch description.  Row contents come from :func:`target_row` / :func:`draft_row`."""

    name: str
    vocab: int
    k: np.ndarray                 # int32 [R], 1 <= k_i <= 16
    planted_accept: np.ndarray    # int32 [R], 0 <= L_i <= k_i
    d_dtype: str                  # "fp32" | "bf16"
    t_dtype: str
    clip_c: float
    ce_weight: float = 1.0
    seed: int = 0
    ld_d: int = 0                 # row stride in elements (0 -> vocab)
    ld_t: int = 0
    sigma: float = 3.0
    spike: float = 8.0
    draft_scale: float = 0.8
    draft_noise: float = 1.0
    clip_rows: np.ndarray = dataclasses.field(default_factory=lambda: np.zeros(0, np.int64))
    clip_entries: int = 64
    clip_target_value: float = -30.0
    clip_draft_value: float = 6.0
    tie_rows: np.ndarray = dataclasses.field(default_factory=lambda: np.zeros(0, np.int64))
    equal_rows: np.ndarray = dataclasses.field(default_factory=lambda: np.zeros(0, np.int64))
    constant_target_rows: np.ndarray = dataclasses.field(default_factory=lambda: np.zeros(0, np.int64))
    description: str = ""

    def __post_init__(self):
        self.k = np.asarray(self.k, dtype=np.int32)
        self.planted_accept = np.asarray(self.planted_accept, dtype=np.int32)
        if self.ld_d == 0:
            self.ld_d = self.vocab
        if self.ld_t == 0:
            self.ld_t = self.vocab
        self._clip_set = set(int(r) for r in self.clip_rows)
        self._tie_set = set(int(r) for r in self.tie_rows)
        self._equal_set = set(int(r) for r in self.equal_rows)
        self._const_set = set(int(r) for r in self.constant_target_rows)
        doff = np.zeros(len(self.k) + 1, dtype=np.int64)
        np.cumsum(self.k, out=doff[1:])
        self._doff = doff
        # draft row -> request, draft row -> paired target row
        self._req_of_draft = np.repeat(np.arange(len(self.k)), self.k)
        self._pair_of_draft = np.arange(self.num_draft_rows) + self._req_of_draft
        self._draft_of_target = np.full(self.num_target_rows, -1, dtype=np.int64)
        self._draft_of_target[self._pair_of_draft] = np.arange(self.num_draft_rows)

    # -- packed layout ---------------------------------------------------
    @property
    def num_requests(self) -> int:
        return int(len(self.k))

    @property
    def doff(self) -> np.ndarray:
        return self._doff.astype(np.int32)

    @property
    def num_draft_rows(self) -> int:
        return int(self._doff[-1])

    @property
    def num_target_rows(self) -> int:
        return self.num_draft_rows + self.num_requests

    def pair_target_row(self, d: int) -> int:
        return int(self._pair_of_draft[d])

    def request_of_draft(self, d: int) -> int:
        return int(self._req_of_draft[d])

    def bonus_target_row(self, i: int) -> int:
        return int(self._doff[i + 1] + i)

    def draft_of_target(self, s: int) -> int:
        """Draft row paired with target row s, or -1 for a bonus row."""
        return int(self._draft_of_target[s])

    @property
    def bytes_per_draft_elem(self) -> int:
        return 4 if self.d_dtype == "fp32" else 2

    @property
    def bytes_per_target_elem(self) -> int:
        return 4 if self.t_dtype == "fp32" else 2


# ---------------------------------------------------------------------------
# row generators
# ---------------------------------------------------------------------------

def _clip_plant_index(w: Workload, d: int, argmax_t: int) -> np.ndarray:
    """Entries of draft row d (and its paired target row) that carry the clip plant."""
    rng = _rng(w.seed, _S_PLANT, d)
    e = rng.choice(w.vocab - 1, size=w.clip_entries, replace=False)
    return np.where(e < argmax_t, e, e + 1)  # skip the target row's maximiser


def target_row(w: Workload, s: int) -> np.ndarray:
    """Stored values of target row s (float32 array of exactly representable values)."""
    V = w.vocab
    if s in w._const_set:
        return np.full(V, _round_to(np.float32([1.5]), w.t_dtype)[0], dtype=np.float32)
    rng = _rng(w.seed, _S_TARGET, s)
    x = rng.standard_normal(V, dtype=np.float32) * np.float32(w.sigma)
    spike_at = int(rng.integers(V))
    x[spike_at] += np.float32(w.spike)
    x = _round_to(x, w.t_dtype)
    d = w.draft_of_target(s)
    if d >= 0 and d in w._clip_set:
        a = int(np.argmax(x))
        x[_clip_plant_index(w, d, a)] = np.float32(w.clip_target_value)
    if s in w._tie_set:
        trng = _rng(w.seed, _S_TIE, s)
        i1, i2 = np.sort(trng.choice(V, size=2, replace=False))
        v = _round_to(np.float32([x.max() + np.float32(1.0)]), w.t_dtype)[0]
        x[i1] = v
        x[i2] = v
    return x


def draft_row(w: Workload, d: int, t_row: np.ndarray | None = None) -> np.ndarray:
    """Stored values of draft row d, built from its paired target row."""
    s = w.pair_target_row(d)
    if t_row is None:
        t_row = target_row(w, s)
    if d in w._equal_set:
        return _round_to(t_row.copy(), w.d_dtype)
    rng = _rng(w.seed, _S_DRAFT, d)
    x = np.float32(w.draft_scale) * t_row + np.float32(w.draft_noise) * rng.standard_normal(
        w.vocab, dtype=np.float32)
    x = _round_to(x, w.d_dtype)
    if d in w._clip_set:
        a = int(np.argmax(t_row))
        x[_clip_plant_index(w, d, a)] = _round_to(np.float32([w.clip_draft_value]), w.d_dtype)[0]
    return x


def draft_tokens(w: Workload, target_first_max) -> np.ndarray:
    """Draft tokens with the planted accept prefix.

    ``target_first_max(s)`` gives the first maximising index of stored target
    row s (the generator's own ``np.argmax``).
    """
    toks = np.zeros(w.num_draft_rows, dtype=np.int32)
    V = w.vocab
    for i in range(w.num_requests):
        rng = _rng(w.seed, _S_TOKEN, i)
        L = int(w.planted_accept[i])
        for j in range(int(w.k[i])):
            d = int(w._doff[i]) + j
            if j < L:
                toks[d] = target_first_max(d + i)
            elif j == L:
                if V == 1:  # a one-entry vocabulary cannot hold a mismatch
                    toks[d] = 0
                    continue
                a = target_first_max(d + i)
                e = int(rng.integers(V - 1))
                toks[d] = e if e < a else e + 1
            else:
                toks[d] = int(rng.integers(V))
    return toks


# ---------------------------------------------------------------------------
# whole-batch materialisation
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class Batch:
    w: Workload
    draft: np.ndarray        # [N_d, ld_d] float32 or uint16 (bf16 bits)
    target: np.ndarray       # [N_t, ld_t] float32 or uint16 (bf16 bits)
    tokens: np.ndarray       # int32 [N_d]
    doff: np.ndarray         # int32 [R+1]
    gen_argmax: np.ndarray   # int64 [N_t], the generator's np.argmax of each target row

    def target_f64(self, s: int) -> np.ndarray:
        row = self.target[s, : self.w.vocab]
        return (bf16_bits_to_f32(row) if self.w.t_dtype == "bf16" else row).astype(np.float64)

    def draft_f64(self, d: int) -> np.ndarray:
        row = self.draft[d, : self.w.vocab]
        return (bf16_bits_to_f32(row) if self.w.d_dtype == "bf16" else row).astype(np.float64)


def _store_dtype(dtype: str):
    return np.float32 if dtype == "fp32" else np.uint16


def _pad_value(dtype: str):
    return PAD_F32 if dtype == "fp32" else PAD_BF16_BITS


def _encode(x: np.ndarray, dtype: str) -> np.ndarray:
    return x if dtype == "fp32" else f32_to_bf16_bits(x)


def materialize(w: Workload, threads: int | None = None) -> Batch:
    """Generate every row of the batch (thread-parallel, deterministic)."""
    V = w.vocab
    Nd, Nt = w.num_draft_rows, w.num_target_rows
    threads = threads or min(32, os.cpu_count() or 1)
    target = np.empty((Nt, w.ld_t), dtype=_store_dtype(w.t_dtype))
    draft = np.empty((Nd, w.ld_d), dtype=_store_dtype(w.d_dtype))
    if w.ld_t > V:
        target[:, V:] = _pad_value(w.t_dtype)
    if w.ld_d > V:
        draft[:, V:] = _pad_value(w.d_dtype)
    gen_argmax = np.zeros(Nt, dtype=np.int64)

    def do_target(rows):
        for s in rows:
            x = target_row(w, s)
            target[s, :V] = _encode(x, w.t_dtype)
            gen_argmax[s] = int(np.argmax(x))

    def do_draft(rows):
        for d in rows:
            s = w.pair_target_row(d)
            t = target[s, :V]
            t32 = bf16_bits_to_f32(t) if w.t_dtype == "bf16" else t.copy()
            draft[d, :V] = _encode(draft_row(w, d, t32), w.d_dtype)

    def blocks(n):
        step = max(1, (n + threads * 4 - 1) // (threads * 4))
        return [range(a, min(n, a + step)) for a in range(0, n, step)]

    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(do_target, blocks(Nt)))
        list(ex.map(do_draft, blocks(Nd)))
    toks = draft_tokens(w, lambda s: int(gen_argmax[s]))
    return Batch(w=w, draft=draft, target=target, tokens=toks, doff=w.doff, gen_argmax=gen_argmax)


# ---------------------------------------------------------------------------
# named workloads
# ---------------------------------------------------------------------------

def _trunc_geom_k(rng, n, p=0.07):
    ks = np.arange(1, MAX_K + 1)
    probs = (1.0 - p) ** (ks - 1)
    probs /= probs.sum()
    return rng.choice(ks, size=n, p=probs).astype(np.int32)


def _pick_rows(rng, n_total, frac):
    n = int(round(frac * n_total))
    return np.sort(rng.choice(n_total, size=n, replace=False)).astype(np.int64)


def make_workload(name: str, seed: int = 0, **over) -> Workload:
    """Build a named workload.

    tiny       V=1024, fp32/fp32, k = {16, 9, 3, 1}, L_i ~ U{0..k_i}, c = 1.0
    single     V=151936, bf16, one request of k = 16, L ~ U{0..16}, c = 1.0
    c32        V=151936, bf16, 32 requests, k_i ~ U{1..16}, L_i ~ Bin(k_i, 0.6), c = 1.0
    c128       V=151936, bf16, 128 requests, k_i ~ truncated geometric (p = 0.07) on 1..16,
               L_i ~ Bin(k_i, 0.6); 5% of draft rows carry 64 entries with target -30 and
               draft +6; c = 0.5
    c128_clip  as c128 with the planted draft value +16, so the clip binds on all 64 entries
    stress     V=151937 (odd, rows unaligned), fp32 draft / bf16 target, 512 requests of
               k = 16, L ~ U{0..16}, 1% exact-tie target rows, 1% draft == target rows, c = 1.0
    """
    meta = _rng(seed, _S_META, 0)
    kw = dict(seed=seed)
    if name == "tiny":
        k = np.array([16, 9, 3, 1], dtype=np.int32)
        L = np.array([meta.integers(0, ki + 1) for ki in k], dtype=np.int32)
        kw.update(name=name, vocab=1024, k=k, planted_accept=L, d_dtype="fp32", t_dtype="fp32",
                  clip_c=1.0)
    elif name == "single":
        k = np.array([16], dtype=np.int32)
        L = np.array([meta.integers(0, 17)], dtype=np.int32)
        kw.update(name=name, vocab=151936, k=k, planted_accept=L, d_dtype="bf16", t_dtype="bf16",
                  clip_c=1.0)
    elif name == "c32":
        k = meta.integers(1, 17, size=32).astype(np.int32)
        L = meta.binomial(k, 0.6).astype(np.int32)
        kw.update(name=name, vocab=151936, k=k, planted_accept=L, d_dtype="bf16", t_dtype="bf16",
                  clip_c=1.0)
    elif name in ("c128", "c128_clip"):
        k = _trunc_geom_k(meta, 128)
        L = meta.binomial(k, 0.6).astype(np.int32)
        nd = int(k.sum())
        clip_rows = _pick_rows(meta, nd, 0.05)
        kw.update(name=name, vocab=151936, k=k, planted_accept=L, d_dtype="bf16", t_dtype="bf16",
                  clip_c=0.5, clip_rows=clip_rows,
                  clip_draft_value=16.0 if name == "c128_clip" else 6.0)
    elif name == "stress":
        k = np.full(512, 16, dtype=np.int32)
        L = meta.integers(0, 17, size=512).astype(np.int32)
        nd = int(k.sum())
        nt = nd + 512
        tie_rows = _pick_rows(meta, nt, 0.01)
        equal_rows = _pick_rows(meta, nd, 0.01)
        kw.update(name=name, vocab=151937, k=k, planted_accept=L, d_dtype="fp32", t_dtype="bf16",
                  clip_c=1.0, tie_rows=tie_rows, equal_rows=equal_rows)
    else:
        raise KeyError(name)
    kw.update(over)
    return Workload(**kw)


def custom(vocab: int, k, d_dtype="bf16", t_dtype="bf16", clip_c=1.0, ce_weight=1.0, seed=0,
           accept="uniform", **over) -> Workload:
    """A small workload for edge-case tests (same value recipe, chosen shapes)."""
    meta = _rng(seed, _S_META, 7)
    k = np.asarray(k, dtype=np.int32)
    if accept == "uniform":
        L = np.array([meta.integers(0, ki + 1) for ki in k], dtype=np.int32)
    elif accept == "full":
        L = k.copy()
    elif accept == "none":
        L = np.zeros_like(k)
    else:
        L = np.asarray(accept, dtype=np.int32)
    return Workload(name=over.pop("name", "custom"), vocab=vocab, k=k, planted_accept=L,
                    d_dtype=d_dtype, t_dtype=t_dtype, clip_c=clip_c, ce_weight=ce_weight,
                    seed=seed, **over)


WORKLOADS = ("tiny", "single", "c32", "c128", "c128_clip", "stress")
