"""Algorithmic bytes and flops of each step of the path (the roofline model).

Per request b with r_b query rows, visible positions V_r, H_I indexer heads
of D_I, H_Q query heads, latent 576 (value 512), top-k k:

* indexer  bytes = sum_b V_b * (D_I + 4)             key codes + float32 scale, read once per request
                 + R * H_I * (D_I + 4) + R * H_I * 4 query codes + scales, head weights
           flops = sum_r 2 * H_I * D_I * V_r
* sparse MLA bytes = sum_b |union_i S_{b,i}| * 1152   distinct latent rows gathered per request
                 + R * H_Q * (576 + 512) * 2 + R * k * 4   query, output, indices
           flops = sum_r H_Q * |S_r| * 2 * (576 + 512)
* write-back bytes = sum_b accept_len_b * (1152 + 132) * 2
* merge    bytes = 8 * (S + B*K) * 2 + offsets

The page numbers these formulas reproduce (the indexer read per draft step
with and without index sharing, the accepted-KV move) are checked in
tests/test_roofline_model.py against [P2] "附:长上下文下草稿段的索引器账"
and "KV 交账:接受段的搬移与拒绝段的回收".
"""
from __future__ import annotations

import numpy as np

LATENT_ROW_BYTES = 576 * 2
IDX_KEY_BYTES = 128 + 4


def indexer_bytes(visible_per_request, R, H_I, D_I):
    return int(np.sum(visible_per_request)) * (D_I + 4) + R * H_I * (D_I + 4) + R * H_I * 4


def indexer_flops(visible_per_row, H_I, D_I):
    return 2.0 * H_I * D_I * float(np.sum(visible_per_row))


FP8_LATENT_ROW_BYTES = 656   # 512 E4M3 codes + 4 float32 scales + 64 bf16 rope values


def mla_bytes(union_rows_per_request, R, H_Q, k, row_bytes=LATENT_ROW_BYTES):
    return int(np.sum(union_rows_per_request)) * row_bytes + R * H_Q * (576 + 512) * 2 + R * k * 4


def accept_stochastic_bytes(B, K, V, n_accepted):
    """The K gathered (q, p) pairs and draft ids per request, the uniforms, and the two rows of V
    probabilities the draw scans (residual: p and q of the rejected row; p of row K after full
    acceptance, one row)."""
    n_accepted = np.asarray(n_accepted)
    rows = np.where(n_accepted < K, 2, 1)
    return int(B * K * (8 + 8 + 4) + B * 4 + int(np.sum(rows)) * V * 4 + B * 12)


def mla_flops(selected_per_row, H_Q):
    return float(np.sum(selected_per_row)) * H_Q * 2 * (576 + 512)


def writeback_bytes(accept_len, row_bytes=LATENT_ROW_BYTES + IDX_KEY_BYTES):
    return int(np.sum(accept_len)) * row_bytes * 2


def draft_indexer_read(L, layers=21, key_bytes=128, steps=4, shared=True):
    """Indexer key bytes read by the draft forwards of one decode step at
    context L: once with index sharing, once per draft forward without."""
    return (1 if shared else steps) * layers * key_bytes * L


def accepted_kv_move(batch, accept_len, layers, bytes_per_token_layer):
    return batch * accept_len * layers * bytes_per_token_layer
