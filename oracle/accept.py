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
