"""Sparse MLA decode over the selected latent rows.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

[P2] section "GLM-5.3 的草稿层到底长什么样": the MLA latent has
kv_lora_rank = 512 plus qk_rope_head_dim = 64, i.e. 576 values per token;
[P2] "验证段的逐层算子" op 7 and [P3] "稀疏 MLA 的前向路径": attention runs
only over the positions the indexer selected.  With the absorbed query
(q_nope already multiplied into the latent space, 512, plus q_rope, 64) the
key of position s is the whole latent row c[s, 0:576] and the value is
c[s, 0:512].  For query row r and head h:

    logit_j = scale * q[r, h, :] . c[s_j, :]          over the valid s_j
    o[r, h] = sum_j softmax(logit)_j * c[s_j, 0:512]
    lse[r, h] = log sum_j exp(logit_j)

Entries equal to -1 are padding and are skipped.  Appended positions (the
shared-index draft steps, [P1] "阶段 5:Draft 后续步骤(复用 top-k)") are
base+1 .. base+n_append and are attended in addition to the selected set.
The softmax scale is not on the pages; the caller passes it (1/sqrt(576) in
the workloads).  All arithmetic is float64; a row with no valid index has
o = 0 and lse = -inf.
"""
from __future__ import annotations

import numpy as np

D_LATENT = 576
D_V = 512


def _f64(x, index) -> np.ndarray:
    """x[index] as float64 numpy (x: numpy array or CPU torch tensor, e.g. bf16)."""
    if hasattr(x, "detach"):
        import torch
        return x[torch.as_tensor(index, dtype=torch.long)].double().numpy() if isinstance(index, list) \
            else x[index].double().numpy()
    return np.asarray(x[index], dtype=np.float64)


def row_index_list(idx_r: np.ndarray, n_append: int = 0, base: int | None = None):
    """The positions attended by one row: the valid selected ones, then the
    appended base+1..base+n_append."""
    sel = [int(s) for s in np.asarray(idx_r).tolist() if int(s) >= 0]
    if n_append:
        sel += [int(base) + 1 + j for j in range(n_append)]
    return sel


def sparse_mla(q, latent, cache_start, row_req, idx, scale, n_append=0,
               append_base=None, rows=None, heads=None, d_v=D_V):
    """q [R, H, 576], latent [T, 576] pool, cache_start [B], row_req [R],
    idx [R, k] positions within the request (-1 = padding).

    Returns dict row -> (o [H, d_v] float64, lse [H] float64) for the chosen
    rows (all by default) and heads (all by default)."""
    R, H = q.shape[0], q.shape[1]
    rows = range(R) if rows is None else rows
    heads = range(H) if heads is None else heads
    out = {}
    for r in rows:
        b = int(row_req[r])
        base = int(cache_start[b])
        pos = row_index_list(idx[r], n_append,
                             None if append_base is None else append_base[r])
        C = _f64(latent, [base + s for s in pos]).reshape(len(pos), D_LATENT)
        heads_l = list(heads)
        if len(pos) == 0:
            out[r] = (np.zeros((len(heads_l), d_v)), np.full(len(heads_l), -np.inf))
            continue
        Q = _f64(q, r)[heads_l]                                    # [h, 576]
        logits = scale * (Q @ C.T)                                 # [h, n]
        m = np.max(logits, axis=1, keepdims=True)
        e = np.exp(logits - m)
        ssum = np.sum(e, axis=1)
        o = (e @ C[:, :d_v]) / ssum[:, None]
        lse = m[:, 0] + np.log(ssum)
        out[r] = (o, lse)
    return out


# --------------------------------------------------------------------- FP8 latent cache

FP8_DS_MLA_BYTES = 656   # per token: 512 E4M3 codes + 4 float32 scales + 64 bf16 rope values


def pack_fp8_ds_mla(latent) -> np.ndarray:
    """The 656-byte token layout of the FP8 latent cache ([P2] "草稿层 KV 的账":
    656 bytes per token per layer, the fp8_ds_mla layout; the page gives only
    the total).  Reading adopted: bytes 0..511 the E4M3 codes of latent values
    0..511 in four blocks of 128 (value = code * scale of its block, the
    indexer's block-128 quantizer: scale = amax/448, round to nearest even,
    saturating), bytes 512..527 the four float32 scales, bytes 528..655 the 64
    rope values 512..575 as bf16 (round to nearest even from float32).

    latent [T, 576] (float32 values or a CPU torch tensor) -> uint8 [T, 656]."""
    from .fp8 import quantize_block128
    x = np.asarray(latent.float() if hasattr(latent, "float") else latent, dtype=np.float32)
    T = x.shape[0]
    codes, scales = quantize_block128(x[:, :512])             # [T, 512] uint8, [T, 4] float32
    rope = x[:, 512:576]
    bits = rope.view(np.uint32).astype(np.uint64)
    # bf16 by round to nearest even: add 0x7fff plus the lowest kept bit, keep the high half
    rbits = ((bits + 0x7FFF + ((bits >> 16) & 1)) >> 16).astype(np.uint16)
    out = np.empty((T, FP8_DS_MLA_BYTES), dtype=np.uint8)
    out[:, :512] = codes
    out[:, 512:528] = np.ascontiguousarray(scales, dtype=np.float32).view(np.uint8).reshape(T, 16)
    out[:, 528:656] = np.ascontiguousarray(rbits).view(np.uint8).reshape(T, 128)
    return out


def unpack_fp8_ds_mla(packed) -> np.ndarray:
    """uint8 [T, 656] -> float64 [T, 576]: code * scale for 0..511 (exact in
    float64), the bf16 rope values for 512..575."""
    from .fp8 import decode_e4m3
    pk = np.ascontiguousarray(np.asarray(packed, dtype=np.uint8))
    T = pk.shape[0]
    codes = pk[:, :512]
    scales = pk[:, 512:528].copy().view(np.float32).reshape(T, 4).astype(np.float64)
    vals = decode_e4m3(codes).reshape(T, 4, 128) * scales[:, :, None]
    rope = (pk[:, 528:656].copy().view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.concatenate([vals.reshape(T, 512), rope.reshape(T, 64)], axis=1)
