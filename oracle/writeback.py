"""KV write-back of the accepted segment (accepted-KV move / draft_extend).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

[P2] section "KV 交账:接受段的搬移与拒绝段的回收": after acceptance only the
first accept_len rows (bonus included) of the 6-row window belong to the
request; they are copied into the destination cache slots and the rejected
rows are not.  [P2] "draft_extend:把接受段写回草稿层" and "草稿层 KV 的账":
the draft layer writes only the accepted segment, at least 1 row (the bonus
token when the first draft is rejected) and at most the whole window.

Both caches of the layer move together: the 576-wide latent row and the
indexer key (128 FP8 bytes plus its float32 scale).  The copy is byte exact.
"""
from __future__ import annotations

import numpy as np


def kv_writeback(src_latent, src_idxk, src_idxs, accept_len, dst_latent, dst_idxk,
                 dst_idxs, dst_start):
    """src_latent [B, W, 576] (any dtype), src_idxk [B, W, 128] uint8,
    src_idxs [B, W] float32, accept_len [B] int, dst_* pools, dst_start [B].

    Returns copies of the three destination pools with rows
    dst_start[b] + i (i < accept_len[b]) replaced by source row i."""
    out_l = np.array(dst_latent, copy=True)
    out_k = np.array(dst_idxk, copy=True)
    out_s = np.array(dst_idxs, copy=True)
    B = len(accept_len)
    for b in range(B):
        for i in range(int(accept_len[b])):
            t = int(dst_start[b]) + i
            out_l[t] = src_latent[b, i]
            out_k[t] = src_idxk[b, i]
            out_s[t] = src_idxs[b, i]
    return out_l, out_k, out_s
