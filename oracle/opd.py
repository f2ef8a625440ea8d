"""Plain float64 CPU oracle: greedy verification of packed draft blocks and the
on-policy-distillation (OPD) loss with its gradient.

TEST INFRASTRUCTURE ONLY -- imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the product path.

Sources.  "the AdaFlash article" is the page "AdaFlash: Adaptive Speculative
Decoding with Online Self-Improvement for High-Concurrency LLM Inference";
"the AdaFlash README" is the page "AdaFlash: Adaptive Speculative Decoding via
On-Policy Distilled Diffusion Drafters".

The method reaches closed-form results (a softmax, a clipped sum, an argmax, a
prefix length), so every function below is that definition written out in
float64 with numpy primitives, one row at a time, without blocking, fusion or
online rescaling.  Inputs are the exact stored values of the logits (bfloat16
and float32 widen to float64 exactly).

Readings taken where the pages leave a step open (each is also listed in the
design notes):

* acceptance is greedy: draft token j is accepted while it equals the target
  row's argmax, the argmax taking the lowest index among equal maxima;
* the acceptance rate divides by the request's own k_i, rounded once to float32;
* the clip bounds each vocabulary term from above only: min(p_v r_v, c);
* the mixture weight of the hard-label term is an argument (``beta``, 1 by
  default) and the loss is the mean over all draft rows of the batch;
* the gradient treats the target and its argmax as constants and lets it pass
  through a term that sits exactly at the bound (m_v = [p_v r_v <= c]).

Pinned by ``tests/test_oracle_pins.py`` (brute force, closed forms, invariants,
finite differences, planted answers); no part is "parity unpinned".
"""

from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# per-row definitions
# ---------------------------------------------------------------------------


def log_sum_exp(x: np.ndarray) -> float:
    """log sum_v exp(x_v), in the max-shifted form m + log sum exp(x - m).

    The normaliser of a softmax over the vocabulary; the draft distribution p and
    the target distribution q of the AdaFlash article, section "On-Policy
    Distillation (OPD) for Domain Adaptation", are softmaxes of logit rows.
    """
    x = np.asarray(x, dtype=np.float64)
    m = float(np.max(x))
    return m + float(np.log(np.sum(np.exp(x - m))))


def first_argmax(x: np.ndarray) -> int:
    """Smallest index v with x_v equal to the row maximum.

    The target's greedy choice at a position (the token the target "verifies";
    AdaFlash article, opening section).  Ties go to the lowest index (a reading:
    the pages name no rule).
    """
    x = np.asarray(x)
    return int(np.flatnonzero(x == np.max(x))[0])


def greedy_accept(tokens: np.ndarray, target_choice: np.ndarray):
    """Accepted prefix length and bonus token of one request.

    ``tokens``: the k draft tokens; ``target_choice``: the target's argmax at the
    k + 1 verified positions (the last is the bonus position).  The draft model
    proposes and the target verifies in parallel (AdaFlash article, opening
    section); greedy reading: token j is accepted while it equals the target's
    choice, the accepted prefix stops at the first mismatch, and the token the
    target picks right after the prefix is emitted as the bonus.
    """
    k = len(tokens)
    L = k
    for j in range(k):
        if int(tokens[j]) != int(target_choice[j]):
            L = j
            break
    return L, int(target_choice[L])


def acceptance_rate(L: int, k: int) -> np.float32:
    """The true acceptance rate L / k of a verified draft, rounded once to float32.

    This is the free supervision signal of the length head (AdaFlash article,
    section "2. Adaptive Length Head for Token-Level Variance").
    """
    return np.float32(L) / np.float32(k)


def hard_label_ce(z: np.ndarray, a: int) -> float:
    """Top-1 hard-label cross-entropy -log p_a with p = softmax(z), a = target argmax.

    AdaFlash article, section "On-Policy Distillation (OPD) for Domain
    Adaptation", item "Reverse KL + Top-1 hard labels".
    """
    z = np.asarray(z, dtype=np.float64)
    log_p = z - log_sum_exp(z)
    return float(-log_p[a])


def clipped_reverse_kl_terms(z: np.ndarray, t: np.ndarray):
    """Per-vocabulary terms of the reverse KL(p || q) = sum_v p_v (log p_v - log q_v).

    p = softmax(draft logits z), q = softmax(target logits t).  The reverse
    direction is the one that "emphasizes the target's high-probability modes"
    (AdaFlash article, "Reverse KL + Top-1 hard labels").  Returns (p, r, term)
    with r_v = log p_v - log q_v and term_v = p_v r_v.
    """
    z = np.asarray(z, dtype=np.float64)
    t = np.asarray(t, dtype=np.float64)
    log_p = z - log_sum_exp(z)
    log_q = t - log_sum_exp(t)
    p = np.exp(log_p)
    r = log_p - log_q
    return p, r, p * r


def row_forward(z: np.ndarray, t: np.ndarray, c: float, beta: float = 1.0) -> dict:
    """Everything the forward pass yields for one (draft row, target row) pair.

    kl  = sum_v min(p_v r_v, c): each vocabulary term clipped before the sum
          (AdaFlash article, "Per-vocabulary divergence clipping"; upper clip
          is a reading);
    ce  = -log p_a, a the target argmax ("Top-1 hard labels");
    loss_row = kl + beta * ce (the "mixture" loss of the AdaFlash README,
          "Released Checkpoint"; beta is a reading).
    Also returns lse_z, lse_t, the target argmax a, the number of clipped terms
    and S = sum_v m_v p_v (r_v + 1) (the row constant of the gradient), with
    S_l1 = sum_v m_v p_v |r_v + 1|, the size of S's summands: S is a difference of
    large sums when much mass is clipped, and its error is judged against S_l1.
    """
    z = np.asarray(z, dtype=np.float64)
    t = np.asarray(t, dtype=np.float64)
    p, r, term = clipped_reverse_kl_terms(z, t)
    kl = float(np.sum(np.minimum(term, c)))
    a = first_argmax(t)
    ce = hard_label_ce(z, a)
    m = term <= c
    S = float(np.sum(np.where(m, p * (r + 1.0), 0.0)))
    S_l1 = float(np.sum(np.where(m, p * np.abs(r + 1.0), 0.0)))
    return dict(kl=kl, ce=ce, loss_row=kl + beta * ce, lse_z=log_sum_exp(z), lse_t=log_sum_exp(t),
                argmax=a, n_clipped=int(np.count_nonzero(~m)), S=S, S_l1=S_l1)


def row_grad(z: np.ndarray, t: np.ndarray, c: float, beta: float, g: float = 1.0) -> np.ndarray:
    """d(g * loss_row)/dz for one row, derived from :func:`row_forward`'s definition.

    With dp_v/dz_u = p_v (delta_uv - p_u) and dr_v/dz_u = delta_uv - p_u, the
    unclipped terms give p_u (m_u (r_u + 1) - S), S = sum_v m_v p_v (r_v + 1); a
    clipped term is the constant c.  The cross-entropy gives p_u - delta_{u,a}.
    Target logits and the argmax a are constants (the target model never changes,
    AdaFlash article, "Decoupled training/inference").
    """
    z = np.asarray(z, dtype=np.float64)
    t = np.asarray(t, dtype=np.float64)
    p, r, term = clipped_reverse_kl_terms(z, t)
    m = (term <= c).astype(np.float64)
    S = float(np.sum(m * p * (r + 1.0)))
    a = first_argmax(t)
    onehot = np.zeros_like(p)
    onehot[a] = 1.0
    return g * (p * (m * (r + 1.0) - S) + beta * (p - onehot))


# ---------------------------------------------------------------------------
# packed batches
# ---------------------------------------------------------------------------
# Layout (AdaFlash article, "Variable-length request packing": requests with
# different verification lengths share one batch).  doff is the exclusive prefix
# sum of k_i; request i owns draft rows doff[i] .. doff[i+1]-1 and target rows
# doff[i]+i .. doff[i+1]+i; draft row doff[i]+j pairs with target row doff[i]+i+j
# and target row doff[i+1]+i is the bonus position.


def _requests(doff):
    doff = np.asarray(doff, dtype=np.int64)
    for i in range(len(doff) - 1):
        yield i, int(doff[i]), int(doff[i + 1] - doff[i])


def verify_packed(target_row, tokens, doff, requests=None):
    """Greedy verification of every (or the listed) request.

    ``target_row(s)`` returns target row s as float64.  Returns dicts keyed by
    request: accept_len, bonus_token, accept_rate, and the target argmax of each
    of the request's target rows.
    """
    tokens = np.asarray(tokens)
    out = {}
    for i, d0, k in _requests(doff):
        if requests is not None and i not in requests:
            continue
        s0 = d0 + i
        choice = np.array([first_argmax(target_row(s0 + j)) for j in range(k + 1)], dtype=np.int64)
        L, bonus = greedy_accept(tokens[d0:d0 + k], choice)
        out[i] = dict(accept_len=L, bonus_token=bonus, accept_rate=acceptance_rate(L, k),
                      target_argmax=choice, target_rows=np.arange(s0, s0 + k + 1))
    return out


def opd_loss_fwd(draft_row, target_row, doff, c, beta=1.0, rows=None):
    """Per-draft-row forward results, and the batch loss when every row is given.

    loss = (1 / N_d) * sum_rows (kl + beta * ce): the mean over all draft rows of
    the batch (a reading; every drafted position is on-policy data).
    """
    per_row = {}
    N_d = int(np.asarray(doff)[-1])
    for i, d0, k in _requests(doff):
        for j in range(k):
            d = d0 + j
            if rows is not None and d not in rows:
                continue
            per_row[d] = row_forward(draft_row(d), target_row(d + i), c, beta)
    loss = None
    if rows is None:
        loss = float(sum(per_row[d]["loss_row"] for d in range(N_d)) / N_d) if N_d else 0.0
    return per_row, loss


def opd_loss_bwd(draft_row, target_row, doff, c, beta=1.0, grad_row=None, grad_scale=1.0, rows=None):
    """Gradient of sum_rows g_r * loss_row with respect to each draft logit row.

    g_r = grad_row[r] when given, else grad_scale (grad_scale = 1 / N_d gives the
    gradient of the mean loss).
    """
    out = {}
    for i, d0, k in _requests(doff):
        for j in range(k):
            d = d0 + j
            if rows is not None and d not in rows:
                continue
            g = float(grad_row[d]) if grad_row is not None else float(grad_scale)
            out[d] = row_grad(draft_row(d), target_row(d + i), c, beta, g)
    return out
