"""Lightning-indexer scores for the verify / draft query rows.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

[P3] section "Indexer 的结构与计算流程": per token the indexer has
index_n_heads query heads of index_head_dim, one key per cached position
(one KV head), and weights_proj gives one weight per head; q and k are FP8
with block-128 scales.  [P2] section "验证段的逐层算子" (ops 5-6): every verify
query scores the whole visible history and picks its own top 2048.

The score of query row r against cached position s is

    I[r, s] = sum_h  w[r, h] * ReLU( qs[r, h] * ks[s] * sum_d q[r, h, d] * k[s, d] )

(the per-head ReLU then the head weight then the head sum; the pages give the
components but not the formula, this is the reading adopted).  Row r sits at
position p_r of its request and sees positions 0..p_r (chain causal mask,
[P2] "验证输入是怎么拼出来的").  Without FP8 (the float32 configuration) the
scales are 1.
"""
from __future__ import annotations

import numpy as np

from .fp8 import decode_e4m3


def dequant_q(q_codes, q_scale):
    """[R, H, D] codes + [R, H] scales -> float64 (block 128 = one scale per head
    vector when D == 128)."""
    return decode_e4m3(q_codes) * np.asarray(q_scale, dtype=np.float64)[..., None]


def indexer_scores_row(q_r: np.ndarray, w_r: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """Scores of one query row against `keys` (already dequantized, float64).

    q_r [H, D], w_r [H], keys [V, D] -> [V].
    """
    q_r = np.asarray(q_r, dtype=np.float64)
    w_r = np.asarray(w_r, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    dots = keys @ q_r.T                      # [V, H]   (library matmul)
    return np.maximum(dots, 0.0) @ w_r       # ReLU per head, weight, sum over heads


def indexer_scores(q, q_scale, w, k_cache, k_scale, cache_start, row_req, row_pos,
                   fp8: bool, rows=None):
    """Scores for the selected rows (all rows by default).

    q: [R, H, D] (uint8 codes if fp8 else float), q_scale: [R, H] or None,
    w: [R, H] float32, k_cache: [T, D] pool, k_scale: [T] or None,
    cache_start: [B] int64 pool offset of each request, row_req: [R] request id,
    row_pos: [R] position p_r.  Returns a dict row -> float64 array of p_r + 1.
    """
    R = len(row_req)
    rows = range(R) if rows is None else rows
    out = {}
    for r in rows:
        b = int(row_req[r])
        p = int(row_pos[r])
        base = int(cache_start[b])
        if fp8:
            q_r = decode_e4m3(q[r]) * np.asarray(q_scale[r], dtype=np.float64)[:, None]
            keys = decode_e4m3(k_cache[base:base + p + 1]) * \
                np.asarray(k_scale[base:base + p + 1], dtype=np.float64)[:, None]
        else:
            q_r = np.asarray(q[r], dtype=np.float64)
            keys = np.asarray(k_cache[base:base + p + 1], dtype=np.float64)
        out[r] = indexer_scores_row(q_r, w[r], keys)
    return out
