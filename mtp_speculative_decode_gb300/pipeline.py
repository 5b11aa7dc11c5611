"""One MTP decode step of the DSA layer on the GPU, as a sequence of C-ABI calls.

Order of the step ([P1] "UnifiedMTPGlm5_2 前向传播详解", [P2] "三段前向的分工"):

1. merge_tokens: prompt (bonus) token + K drafts per request -> verify rows
2. quantize_fp8_block128 of the indexer queries (dynamic FP8, block 128)
3. indexer_topk over the target caches for every verify row
4. sparse_mla_decode over the selected latent rows
5. accept_greedy against the target argmax
6. kv_writeback of the accepted segment into the draft-layer caches
7. the draft loop with index_share_for_mtp_iteration: indexer + top-k at draft
   step 0 only, then sparse MLA at steps 0..n-1 over the shared selection plus
   the positions appended since step 0.

All device buffers are allocated once in __init__ (torch), so a step issues
only kernel launches of libmtpsd on one stream: no allocation, no host sync.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np
import torch

from . import _native as N
from . import api
from . import workloads as W


def _dev_u32(x, device):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.uint32)).to(device)


def _gen(src, name, device):
    """An input tensor on the device: generated there chunk by chunk when the
    source is the workload's on-demand set, else copied."""
    if hasattr(src, "to_device"):
        return src.to_device(name, device)
    return _dev(src[name], device)


def _dev(x, device, dtype=None):
    t = torch.as_tensor(x)
    if dtype is not None:
        t = t.to(dtype)
    return t.to(device).contiguous()


class DecodeStep:
    """One decode step on the GPU.  seeded=True replaces the draft step-0 indexer by draft_extend's attention
    over the K+1 window rows of the draft layer, whose selection at the last accepted row seeds every draft
    step of the next round (seed_dsa_topk_from_draft_extend)."""

    def __init__(self, w: W.Workload, device="cuda", draft: Optional[Dict[str, torch.Tensor]] = None,
                 seeded: bool = False, latent_fp8: bool = False, page_size: Optional[int] = None):
        self.w = w
        self.seeded = seeded
        self.page_size = page_size     # paged caches: every pool reached through one shared block table
        self.paged = None
        self.latent_fp8 = latent_fp8   # latent caches as 656-byte FP8 rows ([P2] "草稿层 KV 的账")
        spec = w.spec
        self.spec = spec
        self.device = device
        self.fp8 = not spec.latent_f32
        B, K, R = spec.B, spec.K, w.R
        self.B, self.K, self.R = B, K, R
        t = w.tensors
        # --- resident caches (target layer)
        self.cache_start = _dev(w.cache_start, device, torch.int64)
        self.latent = self._latent(_gen(t, "latent", device))
        if self.fp8:
            k_raw = _gen(t, "k_idx", device)
            self.k_cache, k_scale = api.quantize_fp8_block128(k_raw)
            self.k_scale = k_scale.reshape(-1).contiguous()
            del k_raw
        else:
            self.k_cache = _gen(t, "k_idx", device)
            self.k_scale = None
        # --- verify rows (host-known layout)
        self.row_pos = _dev(w.row_pos, device, torch.int64)
        self.max_visible = int(w.L.max()) + w.r
        # --- per-step inputs
        self.prompt_tokens = _dev(w.prompt_tokens, device, torch.int64)
        self.prompt_offsets = _dev_u32(w.prompt_offsets, device)
        self.draft_tokens = _dev(w.draft_tokens, device, torch.int64)
        self.target_argmax = _dev(w.target_argmax, device, torch.int64)
        self.q_idx_raw = _gen(t, "q_idx", device)
        self.w_idx = _gen(t, "w_idx", device)
        self.q_mla = _gen(t, "q_mla", device)
        # --- outputs / intermediates
        S = w.prompt_tokens.shape[0]
        self.merged_tokens = torch.empty(S + B * K, dtype=torch.int64, device=device)
        self.merged_offsets = torch.empty(B + 1, dtype=torch.uint32, device=device)
        if spec.verify:
            # verify rows are the merged segments (1 input token + K drafts each)
            host_mo = api.host_merged_offsets(w.prompt_offsets, K)
            self.row_offsets = _dev_u32(host_mo, device)
        else:
            self.row_offsets = _dev_u32(np.arange(B + 1), device)
        if self.fp8:
            self.q_idx = torch.empty(self.q_idx_raw.shape, dtype=torch.uint8, device=device)
            self.q_scale = torch.empty(self.q_idx_raw.shape[:2], dtype=torch.float32, device=device)
        else:
            self.q_idx, self.q_scale = self.q_idx_raw, None
        self.topk_idx = torch.empty(R, spec.topk, dtype=torch.int32, device=device)
        self.out = torch.empty(R, spec.H_Q, 512, dtype=self.q_mla.dtype, device=device)
        mla_dt = N.MTPSD_FP8_DS_MLA if latent_fp8 else (1 if self.fp8 else 0)
        self.mla_dtype = mla_dt
        self.lse = torch.empty(R, spec.H_Q, dtype=torch.float32, device=device)
        self.num_accepted = torch.empty(B, dtype=torch.int32, device=device)
        self.next_tokens = torch.empty(B, dtype=torch.int64, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        # the indexer's score matrix (read back by the top-k) and its small work plan
        self.scores = torch.empty(R, api.scores_ld(self.max_visible), dtype=torch.float32, device=device)
        self.ws_plan = torch.empty(max(api.indexer_plan_bytes(B, R), 256), dtype=torch.uint8, device=device)
        self.ws_topk = torch.empty(max(api.topk_workspace_size(R, self.max_visible, spec.topk), 256), dtype=torch.uint8,
                                   device=device)
        n = api.sparse_mla_workspace_size(R, spec.H_Q, spec.topk, 0, self.mla_dtype)
        self.ws_mla = torch.empty(max(n, 256), dtype=torch.uint8, device=device)
        # --- draft layer
        self.has_draft = spec.draft_steps > 0
        if self.has_draft:
            d = draft if draft is not None else W.draft_tensors(w)
            self.d_latent = self._latent(_gen(d, "d_latent", device))
            if self.fp8:
                kr = _gen(d, "d_k_idx", device)
                self.d_k_cache, ks = api.quantize_fp8_block128(kr)
                self.d_k_scale = ks.reshape(-1).contiguous()
                sr = _gen(d, "src_k_idx", device)
                self.src_idxk, ss = api.quantize_fp8_block128(sr)
                self.src_idxs = ss.reshape(B, -1).contiguous()
                del kr, sr
            else:
                # float32 keys move as raw bytes, without a scale
                self.d_k_cache = _gen(d, "d_k_idx", device)
                self.d_k_scale = None
                self.src_idxk = _gen(d, "src_k_idx", device).view(torch.uint8)
                self.src_idxs = None
            src = _gen(d, "src_latent", device)
            self.src_latent = self._latent(src.reshape(-1, 576)).reshape(src.shape[0], src.shape[1], -1) \
                if latent_fp8 else src
            self.dst_pos = _dev(w.L, device, torch.int64)    # accepted segment starts at L_b
            self.next_pos = torch.empty(B, dtype=torch.int64, device=device)
            self.d_q_idx_raw = _gen(d, "d_q_idx", device)
            self.d_w_idx = _gen(d, "d_w_idx", device)
            if self.fp8:
                self.d_q_idx = torch.empty(self.d_q_idx_raw.shape, dtype=torch.uint8, device=device)
                self.d_q_scale = torch.empty(self.d_q_idx_raw.shape[:2], dtype=torch.float32, device=device)
            else:
                self.d_q_idx, self.d_q_scale = self.d_q_idx_raw, None
            self.d_q_mla = [_gen(d, f"d_q_mla{j}", device) for j in range(spec.draft_steps)]
            self.d_row_offsets = _dev_u32(np.arange(B + 1), device)
            self.d_max_visible = int(w.L.max()) + (K + 1) + 1
            self.d_topk = torch.empty(B, spec.topk, dtype=torch.int32, device=device)
            self.shared_idx = torch.empty(B, spec.topk, dtype=torch.int32, device=device)
            self.d_out = [torch.empty(B, spec.H_Q, 512, dtype=self.q_mla.dtype, device=device)
                          for _ in range(spec.draft_steps)]
            self.d_lse = [torch.empty(B, spec.H_Q, dtype=torch.float32, device=device)
                          for _ in range(spec.draft_steps)]
            self.d_scores = torch.empty(B, api.scores_ld(self.d_max_visible), dtype=torch.float32, device=device)
            self.ws_dplan = torch.empty(max(api.indexer_plan_bytes(B, B), 256), dtype=torch.uint8, device=device)
            self.ws_dtopk = torch.empty(max(api.topk_workspace_size(B, self.d_max_visible, spec.topk), 256),
                                        dtype=torch.uint8, device=device)
            n = max(api.sparse_mla_workspace_size(B, spec.H_Q, spec.topk, j, self.mla_dtype)
                    for j in range(spec.draft_steps))
            self.ws_dmla = torch.empty(max(n, 256), dtype=torch.uint8, device=device)
            if seeded:
                self._init_extend(d, device)
        if page_size:
            if seeded:
                raise ValueError("paged caches are built for the shared-index draft loop, not the seeded one")
            self._init_paged(page_size, device)

    def _init_paged(self, ps: int, device, seed: int = 1234):
        """Moves every cache into a paged pool ([P2] "输入准备:prepare_for_draft": token slots reached through a
        per-request table; page_size > 1 groups them into pages).  Request b's positions 0..cap_b-1 (its region of
        the contiguous layout) take ceil(cap_b / ps) pages drawn at random from a pool with one spare page; the
        target and draft layers share the table (each keeps its own pools).  Set-up only: the step then reads
        and writes the caches through the table."""
        w = self.w
        B = self.B
        T = int(self.latent.shape[0])
        cs = np.asarray(w.cache_start, dtype=np.int64)
        caps = np.diff(np.concatenate([cs, [T]]))
        need = -(-caps // ps)
        n_pages = int(need.sum()) + 1
        perm = np.random.default_rng(seed).permutation(n_pages).astype(np.int32)
        bt = np.full((B, int(need.max())), -1, dtype=np.int32)
        src, dst = [], []
        o = 0
        for b in range(B):
            bt[b, :need[b]] = perm[o:o + need[b]]
            o += int(need[b])
            s = np.arange(caps[b], dtype=np.int64)
            src.append(cs[b] + s)
            dst.append(bt[b, s // ps].astype(np.int64) * ps + s % ps)
        src_t = torch.from_numpy(np.concatenate(src)).to(device)
        dst_t = torch.from_numpy(np.concatenate(dst)).to(device)
        rows = n_pages * ps

        def to_pages(x):
            y = torch.zeros((rows,) + tuple(x.shape[1:]), dtype=x.dtype, device=device)
            y[dst_t] = x[src_t]
            return y

        self.latent = to_pages(self.latent)
        self.k_cache = to_pages(self.k_cache)
        if self.k_scale is not None:
            self.k_scale = to_pages(self.k_scale)
        if self.has_draft:
            self.d_latent = to_pages(self.d_latent)
            self.d_k_cache = to_pages(self.d_k_cache)
            if self.d_k_scale is not None:
                self.d_k_scale = to_pages(self.d_k_scale)
        del src_t, dst_t
        self.block_table_host = bt
        self.block_table = _dev(bt, device, torch.int32)
        self.paged = (self.block_table, ps)
        self.cache_start = None       # positions resolve through the table
        Wn = self.K + 1
        self.win_start = _dev(w.L, device, torch.int64)          # the window follows the committed length
        self.out_cache_loc = torch.empty(B, Wn, dtype=torch.int64, device=device)
        # a chain of drafts accepts a prefix of the window: row i comes from window column i
        self.accept_index = _dev(np.tile(np.arange(Wn, dtype=np.int32), (B, 1)), device, torch.int32)

    def _latent(self, x):
        """A latent pool as the step stores it: as generated, or packed into FP8 rows."""
        return api.pack_latent_fp8(x) if self.latent_fp8 else x

    def _init_extend(self, d, device):
        """Buffers of draft_extend's attention: K+1 rows per request at positions L_b .. L_b + K."""
        spec, w = self.spec, self.w
        B, Wn = spec.B, spec.K + 1
        Rx = B * Wn
        self.x_row_offsets = _dev_u32(np.arange(0, Rx + 1, Wn), device)
        self.x_row_pos = _dev((np.repeat(w.L, Wn) + np.tile(np.arange(Wn), B)).astype(np.int64), device, torch.int64)
        self.x_max_visible = int(w.L.max()) + Wn
        self.x_q_idx_raw = _gen(d, "x_q_idx", device)
        self.x_w_idx = _gen(d, "x_w_idx", device)
        if self.fp8:
            self.x_q_idx = torch.empty(self.x_q_idx_raw.shape, dtype=torch.uint8, device=device)
            self.x_q_scale = torch.empty(self.x_q_idx_raw.shape[:2], dtype=torch.float32, device=device)
        else:
            self.x_q_idx, self.x_q_scale = self.x_q_idx_raw, None
        self.x_q_mla = _gen(d, "x_q_mla", device)
        self.x_scores = torch.empty(Rx, api.scores_ld(self.x_max_visible), dtype=torch.float32, device=device)
        self.ws_xplan = torch.empty(max(api.indexer_plan_bytes(B, Rx), 256), dtype=torch.uint8, device=device)
        self.ws_xtopk = torch.empty(max(api.topk_workspace_size(Rx, self.x_max_visible, spec.topk), 256),
                                    dtype=torch.uint8, device=device)
        self.x_topk = torch.empty(Rx, spec.topk, dtype=torch.int32, device=device)
        self.x_out = torch.empty(Rx, spec.H_Q, 512, dtype=self.q_mla.dtype, device=device)
        self.x_lse = torch.empty(Rx, spec.H_Q, dtype=torch.float32, device=device)
        n = api.sparse_mla_workspace_size(Rx, spec.H_Q, spec.topk, 0, self.mla_dtype)
        self.ws_xmla = torch.empty(max(n, 256), dtype=torch.uint8, device=device)
        self.seed_pos = torch.empty(B, dtype=torch.int64, device=device)
        n = max(api.sparse_mla_workspace_size(B, spec.H_Q, spec.topk, j + 1, self.mla_dtype)
                for j in range(spec.draft_steps))
        self.ws_dmla = torch.empty(max(n, 256, self.ws_dmla.numel() if hasattr(self, "ws_dmla") else 0),
                                   dtype=torch.uint8, device=device)

    # ------------------------------------------------------------------ phases
    def merge(self, stream=None):
        api.merge_tokens(self.prompt_tokens, self.prompt_offsets, self.draft_tokens, self.merged_tokens,
                         self.merged_offsets, stream=stream)

    def verify_scores(self, stream=None):
        """FP8 quantization of the indexer queries, then the indexer score GEMM."""
        if self.fp8:
            api.quantize_fp8_block128(self.q_idx_raw, self.q_idx, self.q_scale, stream=stream)
        api.indexer_scores(self.q_idx, self.q_scale, self.w_idx, self.k_cache, self.k_scale, self.cache_start,
                           self.row_offsets, self.row_pos, self.max_visible, scores=self.scores,
                           workspace=self.ws_plan, dev_status=self.status, stream=stream, paged=self.paged)

    def verify_topk(self, stream=None):
        api.topk(self.scores, self.row_pos, self.max_visible, self.spec.topk, out_idx=self.topk_idx,
                 dev_status=self.status, stream=stream, row_len_add=1, workspace=self.ws_topk)

    def verify_indexer(self, stream=None):
        self.verify_scores(stream)
        self.verify_topk(stream)

    def verify_mla(self, stream=None):
        api.sparse_mla_decode(self.q_mla, self.latent, self.cache_start, self.row_offsets, self.row_pos,
                              self.topk_idx, W.SOFTMAX_SCALE, out=self.out, lse=self.lse, workspace=self.ws_mla,
                              dev_status=self.status, stream=stream, paged=self.paged)

    def accept(self, stream=None):
        api.accept_greedy(self.draft_tokens, self.target_argmax, 42, self.num_accepted, self.next_tokens,
                          stream=stream)

    def plan(self, stream=None):
        """Paged caches: the slots of the window positions L .. L + K (assign_cache_locs), shared by the
        layers."""
        api.assign_cache_locs(self.block_table, self.page_size, self.win_start, self.K + 1, self.out_cache_loc,
                              dev_status=self.status, stream=stream)

    def move(self, stream=None):
        """Paged caches: the target layer's accepted KV moves to the window's front slots (a chain of drafts
        accepts the window's prefix, which is already in place)."""
        api.kv_move_accepted(self.latent, self.k_cache.view(torch.uint8), self.k_scale,
                             self.out_cache_loc, self.accept_index, self.num_accepted, dev_status=self.status,
                             stream=stream)

    def writeback(self, stream=None):
        if self.page_size:
            api.kv_writeback_slots(self.src_latent, self.src_idxk, self.src_idxs, self.num_accepted, self.d_latent,
                                   self.d_k_cache.view(torch.uint8), self.d_k_scale, self.out_cache_loc,
                                   self.dst_pos, self.next_pos, dev_status=self.status, stream=stream)
            return
        api.kv_writeback(self.src_latent, self.src_idxk, self.src_idxs, self.num_accepted, self.d_latent,
                         self.d_k_cache.view(torch.uint8), self.d_k_scale, self.cache_start, self.dst_pos,
                         next_pos=self.next_pos, dev_status=self.status, stream=stream)

    def draft_scores(self, stream=None):
        """Draft step 0: FP8 quantization of the draft indexer query, then the score GEMM at the position
        after the written-back segment."""
        if self.fp8:
            api.quantize_fp8_block128(self.d_q_idx_raw, self.d_q_idx, self.d_q_scale, stream=stream)
        api.indexer_scores(self.d_q_idx, self.d_q_scale, self.d_w_idx, self.d_k_cache, self.d_k_scale,
                           self.cache_start, self.d_row_offsets, self.next_pos, self.d_max_visible,
                           scores=self.d_scores, workspace=self.ws_dplan, dev_status=self.status, stream=stream,
                           paged=self.paged)

    def draft_topk(self, stream=None):
        """Draft step 0 selection, then the share gather that steps 1.. reuse."""
        api.topk(self.d_scores, self.next_pos, self.d_max_visible, self.spec.topk, out_idx=self.d_topk,
                 dev_status=self.status, stream=stream, row_len_add=1, workspace=self.ws_dtopk)
        api.topk_share_gather(self.d_topk, self.d_row_offsets, None, self.shared_idx, dev_status=self.status,
                              stream=stream)

    def draft_indexer(self, stream=None):
        self.draft_scores(stream)
        self.draft_topk(stream)

    def draft_mla(self, j: int, stream=None):
        api.sparse_mla_decode(self.d_q_mla[j], self.d_latent, self.cache_start, self.d_row_offsets, self.next_pos,
                              self.shared_idx, W.SOFTMAX_SCALE, n_append=j,
                              append_base=self.next_pos if j else None, row_pos_add=j, out=self.d_out[j],
                              lse=self.d_lse[j], workspace=self.ws_dmla, dev_status=self.status, stream=stream,
                              paged=self.paged)

    def extend_scores(self, stream=None):
        """draft_extend: FP8 quantization of the window rows' draft indexer queries, then the score GEMM over
        the written-back draft-layer keys."""
        if self.fp8:
            api.quantize_fp8_block128(self.x_q_idx_raw, self.x_q_idx, self.x_q_scale, stream=stream)
        api.indexer_scores(self.x_q_idx, self.x_q_scale, self.x_w_idx, self.d_k_cache, self.d_k_scale,
                           self.cache_start, self.x_row_offsets, self.x_row_pos, self.x_max_visible,
                           scores=self.x_scores, workspace=self.ws_xplan, dev_status=self.status, stream=stream)

    def extend_topk(self, stream=None):
        """draft_extend's selection per window row, and the seed: the selection of row num_accepted (the last
        accepted position) with that row's position."""
        api.topk(self.x_scores, self.x_row_pos, self.x_max_visible, self.spec.topk, out_idx=self.x_topk,
                 dev_status=self.status, stream=stream, row_len_add=1, workspace=self.ws_xtopk)
        api.topk_share_gather(self.x_topk, self.x_row_offsets, self.num_accepted, self.shared_idx,
                              dev_status=self.status, stream=stream, row_pos=self.x_row_pos, shared_pos=self.seed_pos)

    def extend_mla(self, stream=None):
        api.sparse_mla_decode(self.x_q_mla, self.d_latent, self.cache_start, self.x_row_offsets, self.x_row_pos,
                              self.x_topk, W.SOFTMAX_SCALE, out=self.x_out, lse=self.x_lse, workspace=self.ws_xmla,
                              dev_status=self.status, stream=stream)

    def seeded_draft_mla(self, j: int, stream=None):
        """Draft step j of the next round: the seed plus positions P .. P + j (P = seed position + 1)."""
        api.sparse_mla_decode(self.d_q_mla[j], self.d_latent, self.cache_start, self.d_row_offsets, self.seed_pos,
                              self.shared_idx, W.SOFTMAX_SCALE, n_append=j + 1, append_base=self.seed_pos,
                              row_pos_add=j + 1, out=self.d_out[j], lse=self.d_lse[j], workspace=self.ws_dmla,
                              dev_status=self.status, stream=stream)

    def phases(self):
        """The step as an ordered list of (name, callable(stream)): what step() runs."""
        ph = []
        if self.spec.verify:
            ph.append(("merge", self.merge))
            if self.page_size:
                ph.append(("plan", self.plan))
            ph += [("verify_scores", self.verify_scores), ("verify_topk", self.verify_topk),
                   ("verify_mla", self.verify_mla)]
        elif self.page_size:
            ph.append(("plan", self.plan))
        ph.append(("accept", self.accept))
        if self.page_size:
            ph.append(("move", self.move))
        if self.has_draft and self.seeded:
            ph += [("writeback", self.writeback), ("extend_scores", self.extend_scores),
                   ("extend_topk", self.extend_topk), ("extend_mla", self.extend_mla)]
            ph += [(f"draft_mla{j}", (lambda stream=None, j=j: self.seeded_draft_mla(j, stream)))
                   for j in range(self.spec.draft_steps)]
        elif self.has_draft:
            ph += [("writeback", self.writeback), ("draft_scores", self.draft_scores), ("draft_topk", self.draft_topk)]
            ph += [(f"draft_mla{j}", (lambda stream=None, j=j: self.draft_mla(j, stream)))
                   for j in range(self.spec.draft_steps)]
        return ph

    def step(self, stream=None):
        """The whole hot path once."""
        for _, fn in self.phases():
            fn(stream)

    def launches_per_step(self) -> int:
        """Kernel launches of one step (for the benchmark's launch count)."""
        n = 0
        quant = 1 if self.fp8 else 0
        _, H_I, D_I = self.q_idx_raw.shape
        dt = N.MTPSD_FP8_E4M3 if self.fp8 else N.MTPSD_F32
        scores = api.indexer_scores_launch_count(H_I, D_I, dt)
        k = self.spec.topk
        if self.spec.verify:
            n += 1 + quant + scores + api.topk_launch_count(self.max_visible, k) + self._mla_launches(k, 0, self.R)
        n += 1
        if self.page_size:
            n += 2    # the window's slot plan and the accepted-KV move
        if self.has_draft and self.seeded:
            Rx = self.B * (self.K + 1)
            n += 1 + quant + scores + api.topk_launch_count(self.x_max_visible, k) + 1 + self._mla_launches(k, 0, Rx)
            n += sum(self._mla_launches(k, j + 1, self.B) for j in range(self.spec.draft_steps))
        elif self.has_draft:
            n += 1 + quant + scores + api.topk_launch_count(self.d_max_visible, k) + 1
            n += sum(self._mla_launches(k, j, self.B) for j in range(self.spec.draft_steps))
        return n

    def _mla_launches(self, n_idx, n_append, R):
        return api.sparse_mla_launch_count(R, self.spec.H_Q, n_idx, n_append, self.mla_dtype)


class LayeredVerify:
    """A verify step over several DSA layers with the cross-layer indexer schedule ([P3] "跨层共享的 indexer
    调度"): a full layer runs its indexer and top-k over its own key cache, a shared layer attends over the
    selection of the most recent full layer.  Every layer has its own latent cache and queries; the rows are
    the verify rows of the workload (merged once)."""

    def __init__(self, w: W.Workload, types, device="cuda"):
        if not types or types[0] != "full":
            raise ValueError("the first layer must be full")
        self.w, self.types, self.device = w, list(types), device
        spec = w.spec
        self.spec = spec
        self.fp8 = not spec.latent_f32
        B, K, R = spec.B, spec.K, w.R
        self.B, self.K, self.R = B, K, R
        t = w.tensors
        self.cache_start = _dev(w.cache_start, device, torch.int64)
        self.row_pos = _dev(w.row_pos, device, torch.int64)
        self.row_offsets = _dev_u32(api.host_merged_offsets(w.prompt_offsets, K), device)
        self.max_visible = int(w.L.max()) + w.r
        self.prompt_tokens = _dev(w.prompt_tokens, device, torch.int64)
        self.prompt_offsets = _dev_u32(w.prompt_offsets, device)
        self.draft_tokens = _dev(w.draft_tokens, device, torch.int64)
        self.merged_tokens = torch.empty(w.prompt_tokens.shape[0] + B * K, dtype=torch.int64, device=device)
        self.merged_offsets = torch.empty(B + 1, dtype=torch.uint32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.scores = torch.empty(R, api.scores_ld(self.max_visible), dtype=torch.float32, device=device)
        self.ws_plan = torch.empty(max(api.indexer_plan_bytes(B, R), 256), dtype=torch.uint8, device=device)
        self.ws_topk = torch.empty(max(api.topk_workspace_size(R, self.max_visible, spec.topk), 256),
                                   dtype=torch.uint8, device=device)
        n = api.sparse_mla_workspace_size(R, spec.H_Q, spec.topk, 0, 1 if self.fp8 else 0)
        self.ws_mla = torch.empty(max(n, 256), dtype=torch.uint8, device=device)
        self.layers = []
        src = -1
        for l, typ in enumerate(self.types):
            L = {"type": typ}
            L["latent"] = _gen(t, W.layer_name("latent", l), device)
            L["q_mla"] = _gen(t, W.layer_name("q_mla", l), device)
            if typ == "full":
                src = l
                kr = _gen(t, W.layer_name("k_idx", l), device)
                if self.fp8:
                    L["k_cache"], ks = api.quantize_fp8_block128(kr)
                    L["k_scale"] = ks.reshape(-1).contiguous()
                else:
                    L["k_cache"], L["k_scale"] = kr, None
                L["q_idx_raw"] = _gen(t, W.layer_name("q_idx", l), device)
                L["w_idx"] = _gen(t, W.layer_name("w_idx", l), device)
                if self.fp8:
                    L["q_idx"] = torch.empty(L["q_idx_raw"].shape, dtype=torch.uint8, device=device)
                    L["q_scale"] = torch.empty(L["q_idx_raw"].shape[:2], dtype=torch.float32, device=device)
                else:
                    L["q_idx"], L["q_scale"] = L["q_idx_raw"], None
                L["topk"] = torch.empty(R, spec.topk, dtype=torch.int32, device=device)
            L["src"] = src
            L["out"] = torch.empty(R, spec.H_Q, 512, dtype=L["q_mla"].dtype, device=device)
            L["lse"] = torch.empty(R, spec.H_Q, dtype=torch.float32, device=device)
            self.layers.append(L)

    def merge(self, stream=None):
        api.merge_tokens(self.prompt_tokens, self.prompt_offsets, self.draft_tokens, self.merged_tokens,
                         self.merged_offsets, stream=stream)

    def scores_of(self, l, stream=None):
        L = self.layers[l]
        if self.fp8:
            api.quantize_fp8_block128(L["q_idx_raw"], L["q_idx"], L["q_scale"], stream=stream)
        api.indexer_scores(L["q_idx"], L["q_scale"], L["w_idx"], L["k_cache"], L["k_scale"], self.cache_start,
                           self.row_offsets, self.row_pos, self.max_visible, scores=self.scores,
                           workspace=self.ws_plan, dev_status=self.status, stream=stream)

    def topk_of(self, l, stream=None):
        api.topk(self.scores, self.row_pos, self.max_visible, self.spec.topk, out_idx=self.layers[l]["topk"],
                 dev_status=self.status, stream=stream, row_len_add=1, workspace=self.ws_topk)

    def mla_of(self, l, stream=None):
        L = self.layers[l]
        api.sparse_mla_decode(L["q_mla"], L["latent"], self.cache_start, self.row_offsets, self.row_pos,
                              self.layers[L["src"]]["topk"], W.SOFTMAX_SCALE, out=L["out"], lse=L["lse"],
                              workspace=self.ws_mla, dev_status=self.status, stream=stream)

    def phases(self):
        ph = [("merge", self.merge)]
        for l, L in enumerate(self.layers):
            if L["type"] == "full":
                ph += [(f"L{l}_scores", (lambda stream=None, l=l: self.scores_of(l, stream))),
                       (f"L{l}_topk", (lambda stream=None, l=l: self.topk_of(l, stream)))]
            ph.append((f"L{l}_mla", (lambda stream=None, l=l: self.mla_of(l, stream))))
        return ph

    def step(self, stream=None):
        for _, fn in self.phases():
            fn(stream)

    def launches_per_step(self) -> int:
        _, H_I, D_I = self.layers[0]["q_idx_raw"].shape
        dt = N.MTPSD_FP8_E4M3 if self.fp8 else N.MTPSD_F32
        k = self.spec.topk
        n = 1
        for L in self.layers:
            if L["type"] == "full":
                n += (1 if self.fp8 else 0) + api.indexer_scores_launch_count(H_I, D_I, dt) + \
                    api.topk_launch_count(self.max_visible, k)
            n += api.sparse_mla_launch_count(self.R, self.spec.H_Q, k, 0, 1 if self.fp8 else 0)
        return n


class StochasticAccept:
    """Rejection-sampling acceptance over a vocabulary-sized batch ([P2] the acceptance rule of speculative
    sampling): draft tokens and their draft probabilities q, target probabilities p of the K+1 rows, and the
    uniforms of the accept tests and of the draw, all resident on the device."""

    def __init__(self, B: int, K: int, V: int, device="cuda", seed: int = 7):
        self.B, self.K, self.V = B, K, V
        self.draft, self.q, self.p, self.u_accept, self.u_sample = W.stochastic_inputs_device(seed, B, K, V, device)
        self.num_accepted = torch.empty(B, dtype=torch.int32, device=device)
        self.next_tokens = torch.empty(B, dtype=torch.int64, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def accept(self, stream=None):
        api.accept_stochastic(self.draft, self.q, self.p, self.u_accept, self.u_sample, self.num_accepted,
                              self.next_tokens, dev_status=self.status, stream=stream)

    def phases(self):
        return [("accept_stochastic", self.accept)]

    def step(self, stream=None):
        self.accept(stream)

    def launches_per_step(self) -> int:
        return 1
