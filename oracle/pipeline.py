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
    return x.numpy() if hasattr(x, "numpy") else np.asarray(x)


class OracleStep:
    """Oracle of one decode step for a workload (see the workloads module).

    `t` holds the raw inputs of the target layer (q_idx, w_idx, k_idx, latent,
    q_mla) and `d` those of the draft layer."""

    def __init__(self, w, d=None):
        self.w = w
        self.spec = w.spec
        self.fp8 = not w.spec.latent_f32
        self.t = w.tensors
        self.d = d
        self._kq = {}      # cached per-request quantized keys: (pool name, b) -> (codes, scales)

    # ------------------------------------------------------------ helpers
    def keys(self, name: str, b: int, upto: int):
        """Dequantized indexer keys of request b, positions 0..upto-1 (float64)."""
        base = int(self.w.cache_start[b])
        raw = self.t[name] if name in self.t else self.d[name]
        x = _np(raw[base:base + upto]).astype(np.float32)
        if not self.fp8:
            return x.astype(np.float64)
        codes, scales = fp8.quantize_block128(x)
        return fp8.decode_e4m3(codes) * scales.astype(np.float64)

    def query(self, raw_q, r):
        x = _np(raw_q[r]).astype(np.float32)
        if not self.fp8:
            return x.astype(np.float64)
        codes, scales = fp8.quantize_block128(x)          # one scale per head vector
        return fp8.decode_e4m3(codes) * scales.astype(np.float64)

    # ------------------------------------------------------------ stages
    def merge(self):
        return merge.merge_tokens(self.w.prompt_tokens, self.w.prompt_offsets, self.w.draft_tokens)

    def verify_scores(self, rows):
        w = self.w
        out = {}
        for r in rows:
            b = int(w.row_req[r])
            p = int(w.row_pos[r])
            keys = self.keys("k_idx", b, p + 1)
            out[r] = indexer.indexer_scores_row(self.query(self.t["q_idx"], r), _np(self.t["w_idx"][r]), keys)
        return out

    def verify_topk(self, scores):
        return {r: topk.topk_select(s, self.spec.topk) for r, s in scores.items()}

    def verify_mla(self, idx_rows, heads=None):
        """idx_rows: dict row -> selected positions (from the oracle's own top-k)."""
        w = self.w
        res = {}
        for r, idx in idx_rows.items():
            res.update(mla.sparse_mla(self.t["q_mla"], self.t["latent"], w.cache_start, w.row_req,
                                      {r: idx}, scale=_scale(), rows=[r], heads=heads))
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
        x = _np(self.d["d_k_idx"][base:base + upto]).astype(np.float32).copy()
        W = self.spec.K + 1
        n = int(min(max(num_accepted[b] + 1, 1), W))
        start = int(self.w.L[b])
        src = _np(self.d["src_k_idx"][b]).astype(np.float32)
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
        out = mla._f64(self.d["d_latent"], [base + int(s) for s in positions]).reshape(len(positions), -1)
        src = _np(self.d["src_latent"][b].float()) if hasattr(self.d["src_latent"], "float") \
            else _np(self.d["src_latent"][b])
        for j, s in enumerate(positions):
            if start <= s < start + n:
                out[j] = src[s - start]
        return out

    def draft_step0(self, num_accepted, reqs):
        """Step-0 indexer scores and top-k of the draft row of each request."""
        P = self.next_pos(num_accepted)
        sc, tk = {}, {}
        for b in reqs:
            keys = self.draft_keys(num_accepted, b, int(P[b]) + 1)
            s = indexer.indexer_scores_row(self.query(self.d["d_q_idx"], b), _np(self.d["d_w_idx"][b]), keys)
            sc[b] = s
            tk[b] = topk.topk_select(s, self.spec.topk)
        return sc, tk

    def draft_mla(self, num_accepted, shared, j: int, reqs, heads=None):
        """Draft step j attention of each request over the shared set plus the
        positions appended since step 0 ([P1] "阶段 5")."""
        P = self.next_pos(num_accepted)
        q = self.d[f"d_q_mla{j}"]
        res = {}
        for b in reqs:
            pos = share.shared_step_positions(shared[b], int(P[b]), j)
            C = self.draft_latent_rows(num_accepted, b, pos)
            # attend over the gathered rows with the same oracle definition
            one = mla.sparse_mla(mla._f64(q, b)[None], C, np.array([0]), np.array([0]),
                                 np.arange(len(pos))[None], _scale(), heads=heads)
            res[b] = one[0]
        return res


def _scale():
    import math
    return 1.0 / math.sqrt(576.0)
