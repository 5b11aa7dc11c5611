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


# --------------------------------------------------------------------- cross-layer sharing

def resolve_indexer_types(n_layers: int, explicit=None, pattern=None, freq=None, offset=None):
    """Per-layer indexer schedule, 'full' or 'shared' ([P3] "跨层共享的 indexer 调度"):
    an explicit per-layer list first; else a pattern string where F is full and
    S shared; else, when a frequency or an offset is given, layer i is full when
    max(i - offset + 1, 0) % freq == 0 (freq 1 and offset 2 by default); with no
    schedule information every layer is full.  The first layer must be full,
    since no earlier selection exists for it to reuse."""
    if explicit is not None and len(explicit) > 0:
        types = [str(t) for t in explicit]
    elif pattern:
        types = ["full" if c == "F" else "shared" if c == "S" else "?" for c in pattern]
        if "?" in types:
            raise ValueError("pattern characters must be F or S")
    elif freq is not None or offset is not None:
        f = 1 if freq is None else int(freq)
        o = 2 if offset is None else int(offset)
        types = ["full" if max(i - o + 1, 0) % f == 0 else "shared" for i in range(n_layers)]
    else:
        types = ["full"] * n_layers
    if len(types) != n_layers:
        raise ValueError("schedule length must equal the layer count")
    if any(t not in ("full", "shared") for t in types):
        raise ValueError("schedule entries must be full or shared")
    if n_layers > 0 and types[0] != "full":
        raise ValueError("the first layer must be full")
    return types


def source_layers(types):
    """For each layer, the layer whose indexer selection it attends over: itself
    when full, else the most recent full layer before it."""
    src, last = [], -1
    for i, t in enumerate(types):
        if t == "full":
            last = i
        src.append(last)
    return src


def seeded_step_positions(seed_row, P_b: int):
    """Positions attended at the first draft step of the next round when the
    draft indexer's selection is seeded by draft_extend ([P2] "draft_extend:把接受段写回草稿层",
    seed_dsa_topk_from_draft_extend): the selection of the last accepted row,
    which sits at position P_b - 1, plus the step's own position P_b (its key is
    written before attention and it lies past every seeded position)."""
    sel = [int(s) for s in np.asarray(seed_row).tolist() if int(s) >= 0]
    return sel + [P_b]
