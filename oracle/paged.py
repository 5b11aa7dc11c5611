"""Paged (slotted) KV cache: where a position lives, the window's slot plan,
the accepted-KV move and the write-back by slot.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

[P2] section "输入准备:prepare_for_draft": the cache is a pool of token slots
and each request reaches its positions through a token table
(req_to_token); before the draft loop, assign_draft_cache_locs_contiguous_func
reads, once per iteration, the slots of the W window positions that follow
the committed length (seq_len .. seq_len + W - 1) into out_cache_loc, and the
draft steps, the verify forward and draft_extend all write into that window.
The same section speaks of page_size > 1 (pages of consecutive slots).
Reading adopted: a block table per request, block_table[b][j] = the pool page
holding positions j*page_size .. (j+1)*page_size - 1 of request b, so that
position s lives in slot block_table[b][s // page_size] * page_size +
s % page_size; page_size 1 is the token table itself.  A negative page entry,
or a position past the table's width, means no slot.

[P2] section "KV 交账:接受段的搬移与拒绝段的回收": fill_front_out_cache_loc
takes the first accept_len slots of the window (the target slots),
fill_accept_out_cache_loc takes the window slots of the accepted rows
(accept_index), and move_kv_cache copies the KV of the latter into the
former.  It is a move: every destination receives the bytes its source held
before the move began, whatever the overlap between the two slot lists.
"""
from __future__ import annotations

import numpy as np


def slot_of(block_table, page_size: int, b: int, s: int) -> int:
    """Pool slot of position s of request b, or -1 when s is negative, lies
    past the table's width, or its page entry is negative."""
    if s < 0 or s // page_size >= len(block_table[b]):
        return -1
    page = int(block_table[b][s // page_size])
    if page < 0:
        return -1
    return page * page_size + s % page_size


def assign_cache_locs(block_table, page_size: int, start_pos, W: int) -> np.ndarray:
    """out_cache_loc [B, W] int64: the slots of positions start_pos[b] + j,
    j < W (the window planned once per iteration)."""
    B = len(start_pos)
    out = np.empty((B, W), dtype=np.int64)
    for b in range(B):
        for j in range(W):
            out[b, j] = slot_of(block_table, page_size, b, int(start_pos[b]) + j)
    return out


def gather_positions(pool, block_table, page_size: int, b: int, positions) -> np.ndarray:
    """The pool rows holding the given positions of request b (a copy)."""
    return np.stack([np.asarray(pool[slot_of(block_table, page_size, b, int(s))]) for s in positions])


def kv_move_accepted(pools, out_cache_loc, accept_index, accept_len):
    """move_kv_cache over the accepted rows.

    pools: a list of arrays [T, ...] (the latent pool, the indexer key pool,
    the key-scale pool: every cache of the layer moves together).
    out_cache_loc [B, W] int64 window slots; accept_index [B, W] int32, the
    window column of the i-th accepted row (entries past accept_len unused);
    accept_len [B] int.  Destination of row i: out_cache_loc[b, i] (the front
    slots); source: out_cache_loc[b, accept_index[b, i]].

    Returns copies of the pools after the move: all sources are read from the
    state before the move, then the destinations are written."""
    out = [np.array(p, copy=True) for p in pools]
    moves = []
    for b in range(len(accept_len)):
        for i in range(int(accept_len[b])):
            dst = int(out_cache_loc[b, i])
            src = int(out_cache_loc[b, int(accept_index[b, i])])
            moves.append((dst, src))
    before = [[np.array(p[src], copy=True) for (_, src) in moves] for p in pools]
    for k, p in enumerate(out):
        for m, (dst, _) in enumerate(moves):
            p[dst] = before[k][m]
    return out


def kv_writeback_slots(src_latent, src_idxk, src_idxs, accept_len, dst_latent, dst_idxk, dst_idxs,
                       dst_slots):
    """The accepted-segment write-back by slot: row i (i < accept_len[b]) of
    request b's window goes to pool slot dst_slots[b, i] (the window slots
    planned for the layer).  Returns copies of the three pools."""
    out_l = np.array(dst_latent, copy=True)
    out_k = np.array(dst_idxk, copy=True)
    out_s = np.array(dst_idxs, copy=True)
    for b in range(len(accept_len)):
        for i in range(int(accept_len[b])):
            t = int(dst_slots[b, i])
            out_l[t] = src_latent[b, i]
            out_k[t] = src_idxk[b, i]
            out_s[t] = src_idxs[b, i]
    return out_l, out_k, out_s
