"""Plain CPU oracle for variable-length request packing with an EMA capacity estimate.

TEST INFRASTRUCTURE ONLY -- imported by ``tests/`` and never by the product path.

The AdaFlash article ("AdaFlash: Adaptive Speculative Decoding with Online
Self-Improvement for High-Concurrency LLM Inference", section "Infrastructure:
Async Training & Variable-Length Batching", "Variable-length request packing")
packs requests of different predicted verification lengths into compact batches
and sizes the next round with an exponential moving average, so that the GPU is
well used without running out of memory; its closing section has the scheduler
repack batches as concurrency and lengths change.  The pages give no formula; the
plainest reading, taken here:

* a request with predicted draft length k (1 <= k <= 16) occupies 2k + 1 logit
  rows in a round (k draft rows, k + 1 target rows: the packed layout);
* a round may hold at most ``row_budget`` rows (the memory budget);
* the estimate e of rows per request is an EMA over rounds,
  e <- alpha * x + (1 - alpha) * e, x = a round's rows / its requests;
* plan: capacity = floor(row_budget / e) requests (at least 1); admit the first
  ``capacity`` requests of the queue (FIFO), then, while their rows exceed the
  budget, give back the last admitted one; the admitted requests are packed back
  to back: draft_offsets is the exclusive prefix sum of their k.

Everything is exact integer arithmetic except the EMA, which is float64 here and
in the library, with the operations in the same order.
"""

from __future__ import annotations

import math

MAX_K = 16


def rows_of(k: int) -> int:
    """Logit rows a request of draft length k occupies in a round."""
    return 2 * int(k) + 1


def ema_update(e: float, x: float, alpha: float) -> float:
    """One EMA step: alpha * x + (1 - alpha) * e (float64, this order)."""
    return alpha * x + (1.0 - alpha) * e


def capacity(row_budget: int, e: float, n_queue: int) -> int:
    """Requests the next round may take: floor(row_budget / e), at least 1, at most the queue."""
    if n_queue <= 0:
        return 0
    c = math.floor(row_budget / e)
    return max(1, min(n_queue, c))


def plan(row_budget: int, e: float, queue_k):
    """One round.  Returns (admitted, draft_offsets, capacity, rows)."""
    queue_k = [int(k) for k in queue_k]
    cap = capacity(row_budget, e, len(queue_k))
    admitted = cap
    rows = sum(rows_of(k) for k in queue_k[:admitted])
    while admitted > 0 and rows > row_budget:
        admitted -= 1
        rows -= rows_of(queue_k[admitted])
    offsets = [0]
    for k in queue_k[:admitted]:
        offsets.append(offsets[-1] + k)
    return admitted, offsets, cap, rows


class Packer:
    """The packer's state across rounds (row budget, alpha, EMA estimate)."""

    def __init__(self, row_budget: int, alpha: float, initial_rows_per_request: float):
        self.row_budget = int(row_budget)
        self.alpha = float(alpha)
        self.e = float(initial_rows_per_request)

    def plan(self, queue_k):
        return plan(self.row_budget, self.e, queue_k)

    def observe(self, rows: int, requests: int):
        if requests > 0:
            self.e = ema_update(self.e, rows / requests, self.alpha)


def simulate(row_budget, alpha, e0, arrivals, rounds):
    """Serve a stream: ``arrivals[r]`` lists the predicted k of requests arriving before round r.

    Each round plans from the queue, observes the admitted batch, and keeps the
    rest queued in order.  Returns per-round (admitted, offsets, capacity, rows, e_after).
    """
    p = Packer(row_budget, alpha, e0)
    queue = []
    out = []
    for r in range(rounds):
        if r < len(arrivals):
            queue.extend(int(k) for k in arrivals[r])
        admitted, offsets, cap, rows = p.plan(queue)
        p.observe(rows, admitted)
        queue = queue[admitted:]
        out.append((admitted, offsets, cap, rows, p.e))
    return out
