"""The decode step of the DSA layer composed from the oracle functions.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Order ([P1] "UnifiedMTPGlm5_2 前向传播详解"; [P2] "三段前向的分工"): merge,
verify (indexer scores, top-k, sparse MLA per verify row), greedy acceptance,
write-back of the accepted segment into the draft-layer caches, then the draft
loop with index_share_for_mtp_iteration (indexer + top-k at draft step 0 only,
MLA at every step over the shared set plus the appended positions).
Every stage can be restricted to a subset of rows so that full-size
workloads are checked on a sample.
"""
from __future__ import annotations

import numpy as np

from . import accept, fp8, indexer, merge, mla, share, topk, writeback


def _np(x):
    if hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16":
        x = x.float()
    return x.numpy() if hasattr(x, "numpy") else np.asarray(x)


def _rows(src, name, a, b):
    """Rows [a, b) of an input tensor: regenerated on their own when the
    source can do that (the workload's on-demand tensors), else sliced."""
    return _np(src.rows(name, a, b)) if hasattr(src, "rows") else _np(src[name][a:b])


def _take(src, name, index):
    """Input rows at the given indices, as float64."""
    if hasattr(src, "take"):
        return _np(src.take(name, index)).astype(np.float64)
    return mla._f64(src[name], list(index))


class OracleStep:
    """Oracle of one decode step for a workload (see the workloads module).

    `t` holds the raw inputs of the target layer (q_idx, w_idx, k_idx, latent,
    q_mla) and `d` those of the draft layer."""

    def __init__(self, w, d=None, latent_fp8: bool = False):
        self.w = w
        self.latent_fp8 = latent_fp8   # latent rows stored as 656-byte FP8 rows (mla.pack_fp8_ds_mla)
        self.spec = w.spec
        self.fp8 = not w.spec.latent_f32
        self.t = w.tensors
        self.d = d
        self._kq = {}      # cached per-request quantized keys: (pool name, b) -> (codes, scales)

    # ------------------------------------------------------------ helpers
    def lat(self, rows):
        """Latent rows (float64) as the cache holds them: exact, or through the FP8 row layout."""
        rows = np.asarray(rows, dtype=np.float64)
        if not self.latent_fp8:
            return rows
        return mla.unpack_fp8_ds_mla(mla.pack_fp8_ds_mla(rows.astype(np.float32)))

    def keys(self, name: str, b: int, upto: int):
        """Dequantized indexer keys of request b, positions 0..upto-1 (float64)."""
        base = int(self.w.cache_start[b])
        src = self.t if name in self.t else self.d
        x = _rows(src, name, base, base + upto).astype(np.float32)
        if not self.fp8:
            return x.astype(np.float64)
        codes, scales = fp8.quantize_block128(x)
        return fp8.decode_e4m3(codes) * scales.astype(np.float64)

    def query(self, src, name, r):
        x = _rows(src, name, r, r + 1)[0].astype(np.float32)
        if not self.fp8:
            return x.astype(np.float64)
        codes, scales = fp8.quantize_block128(x)          # one scale per head vector
        return fp8.decode_e4m3(codes) * scales.astype(np.float64)

    # ------------------------------------------------------------ stages
    def merge(self):
        return merge.merge_tokens(self.w.prompt_tokens, self.w.prompt_offsets, self.w.draft_tokens)

    def verify_scores(self, rows, layer: int = 0):
        w = self.w
        out = {}
        for r in rows:
            b = int(w.row_req[r])
            p = int(w.row_pos[r])
            keys = self.keys(_ln("k_idx", layer), b, p + 1)
            out[r] = indexer.indexer_scores_row(self.query(self.t, _ln("q_idx", layer), r),
                                                _rows(self.t, _ln("w_idx", layer), r, r + 1)[0], keys)
        return out

    def verify_topk(self, scores):
        return {r: topk.topk_select(s, self.spec.topk) for r, s in scores.items()}

    def verify_mla(self, idx_rows, heads=None, layer: int = 0):
        """idx_rows: dict row -> selected positions.  The selected latent rows
        of the row's request are gathered, then attended with the oracle's
        sparse MLA definition."""
        w = self.w
        res = {}
        for r, idx in idx_rows.items():
            b = int(w.row_req[r])
            base = int(w.cache_start[b])
            pos = mla.row_index_list(idx)
            C = self.lat(_take(self.t, _ln("latent", layer), [base + s for s in pos]).reshape(len(pos), mla.D_LATENT))
            q = _rows(self.t, _ln("q_mla", layer), r, r + 1).astype(np.float64)
            one = mla.sparse_mla(q, C, np.array([0]), np.array([0]), np.arange(len(pos))[None], _scale(),
                                 heads=heads)
            res[r] = one[0]
        return res

    def accept(self):
        return accept.accept_greedy(self.w.draft_tokens, self.w.target_argmax, magic_draft_id=42)

    def next_pos(self, num_accepted):
        """Position of the draft step-0 row: write-back start + accepted rows."""
        W = self.spec.K + 1
        acc_len = np.clip(np.asarray(num_accepted) + 1, 1, W)
        return self.w.L + acc_len

    def draft_keys(self, num_accepted, b: int, upto: int):
        """Dequantized draft indexer keys of request b after the write-back."""
        base = int(self.w.cache_start[b])
        x = _rows(self.d, "d_k_idx", base, base + upto).astype(np.float32).copy()
        W = self.spec.K + 1
        n = int(min(max(num_accepted[b] + 1, 1), W))
        start = int(self.w.L[b])
        src = _rows(self.d, "src_k_idx", b, b + 1)[0].astype(np.float32)
        for i in range(n):
            if start + i < upto:
                x[start + i] = src[i]
        # the accepted rows are written back byte for byte: their codes and
        # scales are those of the window rows, quantized per token
        if not self.fp8:
            return x.astype(np.float64)
        codes, scales = fp8.quantize_block128(x)
        return fp8.decode_e4m3(codes) * scales.astype(np.float64)

    def draft_latent_rows(self, num_accepted, b: int, positions):
        """Draft latent rows (float64) of request b at `positions` after the write-back."""
        base = int(self.w.cache_start[b])
        W = self.spec.K + 1
        n = int(min(max(num_accepted[b] + 1, 1), W))
        start = int(self.w.L[b])
        out = _take(self.d, "d_latent", [base + int(s) for s in positions]).reshape(len(positions), -1).copy()
        src = _rows(self.d, "src_latent", b, b + 1)[0].astype(np.float64)
        for j, s in enumerate(positions):
            if start <= s < start + n:
                out[j] = src[s - start]
        return self.lat(out)

    def draft_step0(self, num_accepted, reqs):
        """Step-0 indexer scores and top-k of the draft row of each request."""
        P = self.next_pos(num_accepted)
        sc, tk = {}, {}
        for b in reqs:
            keys = self.draft_keys(num_accepted, b, int(P[b]) + 1)
            s = indexer.indexer_scores_row(self.query(self.d, "d_q_idx", b), _rows(self.d, "d_w_idx", b, b + 1)[0],
                                           keys)
            sc[b] = s
            tk[b] = topk.topk_select(s, self.spec.topk)
        return sc, tk

    def draft_mla(self, num_accepted, shared, j: int, reqs, heads=None):
        """Draft step j attention of each request over the shared set plus the
        positions appended since step 0 ([P1] "阶段 5")."""
        P = self.next_pos(num_accepted)
        res = {}
        for b in reqs:
            pos = share.shared_step_positions(shared[b], int(P[b]), j)
            C = self.draft_latent_rows(num_accepted, b, pos)
            q = _rows(self.d, f"d_q_mla{j}", b, b + 1).astype(np.float64)
            # attend over the gathered rows with the same oracle definition
            one = mla.sparse_mla(q, C, np.array([0]), np.array([0]),
                                 np.arange(len(pos))[None], _scale(), heads=heads)
            res[b] = one[0]
        return res


    # ------------------------------------------------------------ cross-layer and cross-phase reuse
    def layered_verify(self, types, rows, heads=None):
        """A verify step over len(types) layers with the full/shared schedule
        ([P3] "跨层共享的 indexer 调度"): a full layer runs its own indexer and
        top-k, a shared layer attends over the selection of the most recent full
        layer.  Returns ({layer: {row: selection}}, {layer: {row: (o, lse)}})."""
        src = share.source_layers(types)
        sel, out = {}, {}
        for l, t in enumerate(types):
            if t == "full":
                sel[l] = self.verify_topk(self.verify_scores(rows, layer=l))
            out[l] = self.verify_mla(sel[src[l]], heads=heads, layer=l)
        return sel, out

    def extend_rows(self, b: int):
        W = self.spec.K + 1
        return list(range(b * W, (b + 1) * W))

    def draft_extend(self, num_accepted, reqs, heads=None, selections=None):
        """draft_extend's attention in the draft layer after the write-back: each
        of the K+1 window rows of request b sits at position L_b + i and runs the
        indexer, the top-k and sparse MLA over the written-back caches (over
        selections[(b, i)] instead of its own top-k where given).
        Returns (scores {(b,i)}, selection {(b,i)}, outputs {(b,i)})."""
        W = self.spec.K + 1
        sc, tk, out = {}, {}, {}
        for b in reqs:
            L = int(self.w.L[b])
            for i in range(W):
                x = b * W + i
                keys = self.draft_keys(num_accepted, b, L + i + 1)
                s = indexer.indexer_scores_row(self.query(self.d, "x_q_idx", x), _rows(self.d, "x_w_idx", x, x + 1)[0],
                                               keys)
                sc[(b, i)] = s
                tk[(b, i)] = topk.topk_select(s, self.spec.topk)
                chosen = tk[(b, i)] if selections is None or (b, i) not in selections else selections[(b, i)]
                pos = mla.row_index_list(chosen)
                C = self.draft_latent_rows(num_accepted, b, pos)
                q = _rows(self.d, "x_q_mla", x, x + 1).astype(np.float64)
                out[(b, i)] = mla.sparse_mla(q, C, np.array([0]), np.array([0]), np.arange(len(pos))[None],
                                             _scale(), heads=heads)[0]
        return sc, tk, out

    def seeded_draft_mla(self, num_accepted, seed, j: int, reqs, heads=None):
        """Draft step j of the next round with the selection seeded by draft_extend
        (seed_dsa_topk_from_draft_extend): the seed (the last accepted row's
        selection, position P_b - 1) plus the positions P_b .. P_b + j."""
        P = self.next_pos(num_accepted)
        res = {}
        for b in reqs:
            pos = share.seeded_step_positions(seed[b], int(P[b])) + [int(P[b]) + 1 + i for i in range(j)]
            C = self.draft_latent_rows(num_accepted, b, pos)
            q = _rows(self.d, f"d_q_mla{j}", b, b + 1).astype(np.float64)
            res[b] = mla.sparse_mla(q, C, np.array([0]), np.array([0]), np.arange(len(pos))[None], _scale(),
                                    heads=heads)[0]
        return res


def _ln(name: str, layer: int) -> str:
    return name if layer == 0 else f"{name}@{layer}"


def _scale():
    import math
    return 1.0 / math.sqrt(576.0)
