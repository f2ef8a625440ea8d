"""Plain float64 CPU oracle for temperature-sampled verification of packed draft blocks.

TEST INFRASTRUCTURE ONLY -- imported by ``tests/`` and never by the product path.

The AdaFlash article ("AdaFlash: Adaptive Speculative Decoding with Online
Self-Improvement for High-Concurrency LLM Inference", opening section) describes
the target verifying drafted tokens in parallel; the skill card "Adaflash
Adaptive Speculative Decoding", section "Implementation Steps", lists the
temperature as a tunable.  With a temperature the verification is the standard
speculative-sampling rule, taken here as the plainest reading:

* p = softmax(z / T) (draft), q = softmax(t / T) (target) at each position;
* draft token x_j is accepted when u_j * p(x_j) < q(x_j), u_j uniform in [0, 1)
  (accept with probability min(1, q/p));
* at the first rejected position j, the emitted token is drawn from the residual
  max(0, q - p) (normalised); when that residual is all zero the draw is from q;
* when all k tokens are accepted, the emitted token is drawn from q at the bonus
  position;
* a draw from weights pi with uniform w is the smallest v whose prefix sum
  sum_{u<=v} pi_u exceeds w * sum_u pi_u (inverse CDF in vocabulary order).

Uniforms are inputs (one per draft row, one per request), so the CUDA path and
this oracle decide from the same random numbers.

Pinned by ``tests/test_sampling_pins.py`` (brute force, and the exactness of
speculative sampling: integrated over the draft token and the uniforms, the
emitted token is distributed as q).
"""

from __future__ import annotations

import numpy as np

from .opd import log_sum_exp


def softmax_t(x: np.ndarray, temperature: float) -> np.ndarray:
    """softmax(x / T) in float64."""
    y = np.asarray(x, dtype=np.float64) / float(temperature)
    return np.exp(y - log_sum_exp(y))


def inverse_cdf(weights: np.ndarray, w: float) -> int:
    """Smallest v with sum_{u<=v} weights_u > w * sum(weights); weights >= 0, sum > 0."""
    weights = np.asarray(weights, dtype=np.float64)
    total = float(np.sum(weights))
    target = w * total
    acc = 0.0
    for v in range(len(weights)):
        acc += float(weights[v])
        if acc > target:
            return v
    # w * total rounded up to the full sum: the last entry with positive weight
    return int(np.flatnonzero(weights > 0)[-1])


def residual(p: np.ndarray, q: np.ndarray) -> np.ndarray:
    """max(0, q - p), or q itself when that is all zero."""
    r = np.maximum(q - p, 0.0)
    return r if float(np.sum(r)) > 0.0 else q


def sampled_accept(z_rows, t_rows, tokens, temperature: float, u, w):
    """One request: k draft rows z_rows[j], k + 1 target rows t_rows[j], draft tokens,
    accept uniforms u[0..k), and the draw uniform w.  Returns (L, next_token, detail)."""
    k = len(tokens)
    L = k
    for j in range(k):
        p = softmax_t(z_rows[j], temperature)
        q = softmax_t(t_rows[j], temperature)
        x = int(tokens[j])
        if not (u[j] * p[x] < q[x]):
            L = j
            break
    if L < k:
        p = softmax_t(z_rows[L], temperature)
        q = softmax_t(t_rows[L], temperature)
        weights = residual(p, q)
    else:
        weights = softmax_t(t_rows[k], temperature)
    return L, inverse_cdf(weights, w), weights


def verify_sampled(draft_row, target_row, tokens, doff, temperature, u_accept, w_sample, requests=None):
    """Every (or the listed) request of a packed batch: dict i -> (accept_len, next_token, rate)."""
    doff = np.asarray(doff, dtype=np.int64)
    out = {}
    for i in range(len(doff) - 1):
        if requests is not None and i not in requests:
            continue
        d0, k = int(doff[i]), int(doff[i + 1] - doff[i])
        zr = [draft_row(d0 + j) for j in range(k)]
        tr = [target_row(d0 + i + j) for j in range(k + 1)]
        L, tok, _ = sampled_accept(zr, tr, tokens[d0:d0 + k], temperature, u_accept[d0:d0 + k], float(w_sample[i]))
        out[i] = dict(accept_len=L, next_token=tok, accept_rate=np.float32(L) / np.float32(k))
    return out
