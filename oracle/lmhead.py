"""Plain float64 CPU oracle for the logit-free verify + OPD-loss forward.

TEST INFRASTRUCTURE ONLY -- imported by ``tests/`` and never by the product path.

The logits of a row are the LM head applied to the row's final hidden state,
z = W_d h_d and t = W_t h_t (the draft model's and the target's heads); the
verification and the loss are then exactly those of ``oracle/opd.py`` (AdaFlash
article, "AdaFlash: Adaptive Speculative Decoding with Online Self-Improvement for
High-Concurrency LLM Inference": the opening section for verification, "On-Policy
Distillation (OPD) for Domain Adaptation" for the loss).  The product by the head
is a library matrix product in float64 of the bfloat16-valued inputs (every
product of two bfloat16 values is exact in float64, and the sums round far below
the float32 accumulation of any GPU path); it is taken in vocabulary chunks so
that a full 151936 x 4096 head is never widened at once.

Pinned by ``tests/test_lmhead_pins.py`` (integer brute force through the
composition, and the agreement with the logits oracle on explicit logits).
"""

from __future__ import annotations

import numpy as np

from . import opd

CHUNK = 8192


def head_logits(h: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Logits of hidden rows h [n, H] (float values) under head w [V, H]: h @ w.T in float64."""
    h = np.asarray(h, dtype=np.float64)
    if h.ndim == 1:
        h = h[None, :]
    V = w.shape[0]
    out = np.empty((h.shape[0], V), dtype=np.float64)
    for c0 in range(0, V, CHUNK):
        c1 = min(V, c0 + CHUNK)
        out[:, c0:c1] = h @ np.asarray(w[c0:c1], dtype=np.float64).T
    return out


def row_forward(hd_row, ht_row, wd, wt, clip_c, ce_weight=1.0):
    """Forward of one (draft row, paired target row): the logits oracle on the head's logits."""
    z = head_logits(hd_row, wd)[0]
    t = head_logits(ht_row, wt)[0]
    return opd.row_forward(z, t, clip_c, ce_weight)


def target_argmax(ht_row, wt):
    return opd.first_argmax(head_logits(ht_row, wt)[0])


def verify_packed(ht_rows, wt, tokens, doff, requests=None):
    """Greedy verification of the listed (or all) requests from target hidden rows."""
    doff = np.asarray(doff, dtype=np.int64)
    out = {}
    for i in range(len(doff) - 1):
        if requests is not None and i not in requests:
            continue
        d0, d1 = int(doff[i]), int(doff[i + 1])
        k = d1 - d0
        rows = [ht_rows(d0 + i + j) for j in range(k + 1)]
        t = head_logits(np.stack(rows), wt)
        am = [opd.first_argmax(t[j]) for j in range(k + 1)]
        L, bonus = opd.greedy_accept(tokens[d0:d1], am)
        out[i] = dict(accept_len=L, bonus_token=bonus, accept_rate=opd.acceptance_rate(L, k), argmax=am)
    return out
