"""Per-row top-k selection (index_topk = 2048).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

[P3] section "Indexer 的结构与计算流程": the fused index kernel returns the
top-k indices with shape (total_seq_len, index_topk); [P2] "验证段的逐层算子"
op 6: each query selects its own 2048 positions.  The pages do not fix the
order of the output nor the tie rule; the reading adopted: the output is a
set, equal scores are ordered by lower position first, and when a row sees
fewer than k positions all of them are taken and the tail is padded with -1.
"""
from __future__ import annotations

import numpy as np


def topk_select(scores: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest scores, ties to the lower index, -1 padded.

    Done by a stable sort of the positions on (-score, position).
    Returned in ascending position order (the content is compared as a set).
    """
    scores = np.asarray(scores, dtype=np.float64)
    V = len(scores)
    order = sorted(range(V), key=lambda s: (-scores[s], s)) if V <= 4096 else \
        np.lexsort((np.arange(V), -scores))
    take = np.sort(np.asarray(order[:min(k, V)], dtype=np.int64))
    out = np.full(k, -1, dtype=np.int64)
    out[:len(take)] = take
    return out


def kth_score(scores: np.ndarray, k: int) -> float:
    """The k-th largest score (or the smallest if fewer than k)."""
    s = np.sort(np.asarray(scores, dtype=np.float64))[::-1]
    return float(s[min(k, len(s)) - 1])
