"""index_share_for_mtp_iteration: reuse of the draft step-0 top-k.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

[P1] section "阶段 5:Draft 后续步骤(复用 top-k)": the draft indexer runs only at
step 0; later steps gather the step-0 selection at the accepted position of
each request (gather_accepted_hidden_states(step0_topk, merged_offsets,
num_accepted, ...)) and pass it as prev_topk_indices; the MLA cache length
grows by one per step while the indexer cache length stays fixed.
[P2] "索引器复用的收益与边界": the multi-row step-0 top-k is compacted to one
row per request (compact_topk_indices).

Readings adopted: the reused row of request b is the row at local index
num_accepted[b] of its step-0 segment (row 0 when num_accepted is absent), and
draft step j (j >= 1) attends over that set plus the j positions appended
since step 0 (P_b + 1 .. P_b + j, P_b being the step-0 position).
"""
from __future__ import annotations

import numpy as np


def topk_share_gather(step0_topk: np.ndarray, row_offsets: np.ndarray, num_accepted=None):
    """step0_topk [R0, k], row_offsets [B+1] (segment of each request in the
    step-0 rows), num_accepted [B] or None -> shared [B, k]."""
    step0_topk = np.asarray(step0_topk)
    ro = np.asarray(row_offsets, dtype=np.int64)
    B = len(ro) - 1
    out = np.empty((B, step0_topk.shape[1]), dtype=step0_topk.dtype)
    for b in range(B):
        local = 0 if num_accepted is None else int(num_accepted[b])
        out[b] = step0_topk[ro[b] + local]
    return out


def shared_step_positions(shared_row: np.ndarray, P_b: int, j: int):
    """Positions attended at draft step j: the shared set plus P_b+1..P_b+j."""
    sel = [int(s) for s in np.asarray(shared_row).tolist() if int(s) >= 0]
    return sel + [P_b + 1 + i for i in range(j)]
