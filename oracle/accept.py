"""Greedy acceptance of the draft tokens.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

[P2] section "接受判定:greedy 与 rejection sampling": under greedy the target
argmax of verify row i is compared with draft token i; drafts are accepted
while they match and everything from the first mismatch on is dropped.
[P1] "阶段 3:拒绝采样与 Bitmask": the step returns the number of accepted
drafts and the next input token (the target's token at the first rejected
position, or the bonus token after full acceptance).  [P4] "MAGIC_DRAFT_TOKEN_ID":
a draft row made entirely of the sentinel id (42) carries no real proposal and
accepts nothing.
"""
from __future__ import annotations

import numpy as np


def accept_greedy(draft: np.ndarray, target_argmax: np.ndarray, magic_draft_id: int = -1):
    """draft [B, K] int64, target_argmax [B, K+1] int64.

    Returns (num_accepted [B] int32, next_tokens [B] int64).
    """
    draft = np.asarray(draft, dtype=np.int64)
    tgt = np.asarray(target_argmax, dtype=np.int64)
    B, K = draft.shape
    n_acc = np.zeros(B, dtype=np.int32)
    nxt = np.zeros(B, dtype=np.int64)
    for b in range(B):
        if magic_draft_id >= 0 and K > 0 and all(int(t) == magic_draft_id for t in draft[b]):
            n = 0
        else:
            n = 0
            while n < K and draft[b, n] == tgt[b, n]:
                n += 1
        n_acc[b] = n
        nxt[b] = tgt[b, n]
    return n_acc, nxt


FIX_SHIFT = 32   # weights are compared at 2^-32 resolution


def _fixed_weights(weights) -> list:
    """floor(max(w, 0) * 2^32) of each single-precision weight, as exact integers."""
    w = np.asarray(weights, dtype=np.float32).astype(np.float64)   # exact widening
    return [int(np.floor(max(x, 0.0) * 2.0 ** FIX_SHIFT)) for x in w.tolist()]


def _scaled_floor(u: float, total: int) -> int:
    """floor(u * total) exactly, for a single-precision u in [0, 1)."""
    m, e = np.frexp(np.float64(np.float32(u)))     # u = m * 2^e, m in [0.5, 1)
    mant = int(m * 2 ** 24)                        # the 24-bit significand, exact
    shift = 24 - int(e)
    return (mant * total) >> shift if mant else 0


def _sample_index(weights: np.ndarray, u: float) -> int:
    """Inverse-CDF draw: the smallest t with W(t) > floor(u * W(V-1)), where W(t)
    is the running sum of floor(w * 2^32) over tokens 0..t (exact integers, so
    the draw does not depend on the order of the additions).  -1 when the total
    weight is zero."""
    w = _fixed_weights(weights)
    total = sum(w)
    if total == 0:
        return -1
    target = _scaled_floor(u, total)
    run = 0
    for t, x in enumerate(w):
        run += x
        if run > target:
            return t
    raise AssertionError("unreachable: target < total")


def accept_stochastic(draft, draft_probs, target_probs, u_accept, u_sample):
    """Rejection-sampling acceptance of a chain of K drafts ([P2] "接受判定:greedy 与
    rejection sampling": the draft distribution q and the target distribution p,
    each draft accepted with probability min(1, p/q); a rejected position draws a
    token from the corrected distribution instead).  The pages do not print the
    corrected distribution; the reading adopted is the standard one of
    speculative sampling, max(0, p - q) normalised, and after K accepted drafts the
    next token is drawn from p of row K.

    draft [B, K] int64; draft_probs q [B, K, V] float32; target_probs p [B, K+1, V]
    float32; u_accept [B, K] and u_sample [B] float32 uniforms in [0, 1) (the
    random numbers are inputs).

    Step i accepts d = draft[b, i] when u_accept[b, i] * q[b, i, d] < p[b, i, d]
    (the accept test u < p/q without a division).  The product and the comparison
    are single precision, as in the kernel, since they decide an integer; a draft
    id outside [0, V) is rejected.  At the first rejected step n the next token is
    the inverse-CDF draw (u_sample) from r = max(0, p[b,n] - q[b,n]) (single
    precision differences, float64 sums); if r has no mass, from p[b,n].  After K
    accepted steps it is the draw from p[b,K].  A distribution with no mass at all
    gives token 0.

    Returns (num_accepted [B] int32, next_tokens [B] int64).
    """
    draft = np.asarray(draft, dtype=np.int64)
    q = np.asarray(draft_probs, dtype=np.float32)
    p = np.asarray(target_probs, dtype=np.float32)
    ua = np.asarray(u_accept, dtype=np.float32)
    us = np.asarray(u_sample, dtype=np.float32)
    B, K = draft.shape
    V = p.shape[2]
    n_acc = np.zeros(B, dtype=np.int32)
    nxt = np.zeros(B, dtype=np.int64)
    for b in range(B):
        n = 0
        while n < K:
            d = int(draft[b, n])
            if not (0 <= d < V):
                break
            if not (np.float32(ua[b, n] * q[b, n, d]) < p[b, n, d]):
                break
            n += 1
        if n < K:
            r = np.maximum(np.float32(0.0), (p[b, n] - q[b, n]).astype(np.float32))
            t = _sample_index(r, us[b])
            if t < 0:
                t = _sample_index(p[b, n], us[b])
        else:
            t = _sample_index(p[b, K], us[b])
        n_acc[b] = n
        nxt[b] = max(t, 0)
    return n_acc, nxt
