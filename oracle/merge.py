"""Ragged merge of prompt tokens and draft tokens.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

[P4] section "Token 合并:RaggedTokenMerger 与 ragged_token_merger": inputs
prompt_tokens [S] int64, prompt_offsets [B+1] uint32 (exclusive prefix sum),
draft_tokens [B, K] int64; outputs merged_tokens [S + B*K] and merged_offsets
[B+1] with merged_offsets[i] = prompt_offsets[i] + i*K.  Each request's
segment holds its prompt tokens followed by its K draft tokens (the same order
as the verify batch "bonus token then drafts" of [P2] section
"验证输入是怎么拼出来的").  K = 0 (prefill, no drafts) is the identity.
"""
from __future__ import annotations

import numpy as np


def host_merged_offsets(prompt_offsets: np.ndarray, K: int) -> np.ndarray:
    """CPU mirror of the merged offsets: out[i] = prompt_offsets[i] + i*K."""
    po = np.asarray(prompt_offsets, dtype=np.int64)
    out = np.empty_like(po)
    for i in range(len(po)):
        out[i] = po[i] + i * K
    return out.astype(np.uint32)


def merge_tokens(prompt_tokens: np.ndarray, prompt_offsets: np.ndarray,
                 draft_tokens: np.ndarray):
    """Concatenate, per request, the prompt tokens then the K draft tokens."""
    prompt_tokens = np.asarray(prompt_tokens, dtype=np.int64)
    po = np.asarray(prompt_offsets, dtype=np.int64)
    draft_tokens = np.asarray(draft_tokens, dtype=np.int64)
    B = len(po) - 1
    K = draft_tokens.shape[1] if draft_tokens.ndim == 2 else 0
    S = int(po[-1])
    mo = host_merged_offsets(po, K).astype(np.int64)
    out = np.zeros(S + B * K, dtype=np.int64)
    for b in range(B):
        n = int(po[b + 1] - po[b])
        for j in range(n):
            out[mo[b] + j] = prompt_tokens[po[b] + j]
        for i in range(K):
            out[mo[b] + n + i] = draft_tokens[b, i]
    return out, mo.astype(np.uint32)
