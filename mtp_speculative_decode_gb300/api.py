"""Python binding of libmtpsd: the C-ABI calls under the same names, taking
torch CUDA tensors.  Argument marshalling only: every step runs in the
library's CUDA kernels on the current torch stream (or the stream given).
Outputs not passed in are allocated with torch before the call."""
from __future__ import annotations

import ctypes as C
from typing import Optional

import numpy as np
import torch

from . import _native as N
from ._native import check, lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t: torch.Tensor, name: str, dtype, ndim: Optional[int] = None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


class Workspace:
    """A reusable device scratch buffer, grown outside the timed path."""

    def __init__(self, device="cuda"):
        self.device = device
        self.buf = torch.empty(0, dtype=torch.uint8, device=device)

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf.numel() < nbytes:
            self.buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)
        return self.buf


_default_ws = {}


def _ws(workspace: Optional[torch.Tensor], nbytes: int, device) -> torch.Tensor:
    if workspace is not None:
        return workspace
    key = str(device)
    if key not in _default_ws:
        _default_ws[key] = Workspace(device)
    return _default_ws[key].get(nbytes)


def _paged(paged):
    """(block_table [B, n] int32 CUDA tensor, page_size) -> a PagedKV (None stays None)."""
    if paged is None:
        return None
    bt, page_size = paged
    _need(bt, "block_table", torch.int32, 2)
    return N.PagedKV(block_table=bt.data_ptr(), bt_stride=bt.shape[1], page_size=int(page_size))


def _byref(x):
    return None if x is None else C.byref(x)


# --------------------------------------------------------------------------- merge

def merge_tokens(prompt_tokens, prompt_offsets, draft_tokens, merged_tokens=None, merged_offsets=None,
                 stream=None):
    _need(prompt_tokens, "prompt_tokens", torch.int64, 1)
    _need(prompt_offsets, "prompt_offsets", torch.uint32, 1)
    _need(draft_tokens, "draft_tokens", torch.int64, 2)
    B, K = draft_tokens.shape
    S = prompt_tokens.numel()
    if prompt_offsets.numel() != B + 1:
        raise ValueError("prompt_offsets must have B+1 entries")
    if merged_tokens is None:
        merged_tokens = torch.empty(S + B * K, dtype=torch.int64, device=prompt_tokens.device)
    if merged_offsets is None:
        merged_offsets = torch.empty(B + 1, dtype=torch.uint32, device=prompt_tokens.device)
    check("mtpsd_merge_tokens", lib().mtpsd_merge_tokens(
        _ptr(prompt_tokens), S, _ptr(prompt_offsets), _ptr(draft_tokens), B, K,
        _ptr(merged_tokens), _ptr(merged_offsets), _stream(stream)))
    return merged_tokens, merged_offsets


def host_merged_offsets(prompt_offsets: np.ndarray, K: int) -> np.ndarray:
    po = np.ascontiguousarray(prompt_offsets, dtype=np.uint32)
    out = np.empty_like(po)
    lib().mtpsd_host_merged_offsets(po.ctypes.data_as(C.c_void_p), len(po) - 1, K,
                                    out.ctypes.data_as(C.c_void_p))
    return out


def pack_latent_fp8(latent, packed=None, stream=None):
    """latent [T, 576] bf16 or float32 -> the FP8 latent cache rows [T, 656] uint8."""
    f32 = latent.dtype == torch.float32
    _need(latent, "latent", torch.float32 if f32 else torch.bfloat16, 2)
    if latent.shape[1] != 576:
        raise ValueError("latent rows must have 576 values")
    T = latent.shape[0]
    if packed is None:
        packed = torch.empty(T, 656, dtype=torch.uint8, device=latent.device)
    check("mtpsd_pack_latent_fp8", lib().mtpsd_pack_latent_fp8(
        _ptr(latent), N.MTPSD_F32 if f32 else N.MTPSD_BF16, T, _ptr(packed), _stream(stream)))
    return packed


def resolve_indexer_types(n_layers: int, explicit=None, pattern=None, freq=None, offset=None):
    """Per-layer indexer schedule as a list of "full" / "shared" (an explicit list is checked and
    returned; otherwise the library resolves the pattern or the frequency and offset)."""
    if explicit is not None and len(explicit) > 0:
        types = [str(t) for t in explicit]
        if len(types) != n_layers or any(t not in ("full", "shared") for t in types) or types[0] != "full":
            raise ValueError("an explicit schedule needs one full/shared entry per layer, the first full")
        return types
    out = np.zeros(max(n_layers, 1), dtype=np.int32)
    check("mtpsd_resolve_indexer_types", lib().mtpsd_resolve_indexer_types(
        n_layers, pattern.encode() if pattern else None, 0 if freq is None else int(freq),
        -1 if offset is None else int(offset), out.ctypes.data_as(C.c_void_p)))
    return ["full" if x else "shared" for x in out[:n_layers]]


# --------------------------------------------------------------------------- FP8

def quantize_fp8_block128(x, codes=None, scales=None, stream=None):
    _need(x, "x", torch.float32)
    if x.numel() % 128:
        raise ValueError("x must hold a multiple of 128 values")
    nb = x.numel() // 128
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(x.shape[:-1] + (x.shape[-1] // 128,), dtype=torch.float32, device=x.device)
    check("mtpsd_quantize_fp8_block128", lib().mtpsd_quantize_fp8_block128(
        _ptr(x), nb, _ptr(codes), _ptr(scales), _stream(stream)))
    return codes, scales


# --------------------------------------------------------------------------- indexer + top-k

def scores_ld(max_visible: int) -> int:
    return int(lib().mtpsd_scores_ld(max_visible))


def indexer_topk_workspace_size(B, R, max_visible, topk) -> int:
    return int(lib().mtpsd_indexer_topk_workspace_size(B, R, max_visible, topk))


def indexer_plan_bytes(B, R) -> int:
    return int(lib().mtpsd_indexer_topk_plan_bytes(B, R))


def indexer_topk_aux_bytes(B, R, max_visible, topk) -> int:
    return int(lib().mtpsd_indexer_topk_aux_bytes(B, R, max_visible, topk))


def topk_workspace_size(R, max_len, k) -> int:
    return int(lib().mtpsd_topk_workspace_size(R, max_len, k))


def _indexer_args(q, q_scale, weights, k_cache, k_scale, cache_start, row_offsets, row_pos, topk, max_visible,
                  topk_idx, topk_score, scores, ws, dev_status):
    fp8 = q.dtype == torch.uint8
    _need(q, "q", torch.uint8 if fp8 else torch.float32, 3)
    _need(k_cache, "k_cache", q.dtype, 2)
    _need(weights, "weights", torch.float32, 2)
    if cache_start is not None:
        _need(cache_start, "cache_start", torch.int64, 1)
    _need(row_offsets, "row_offsets", torch.uint32, 1)
    _need(row_pos, "row_pos", torch.int64, 1)
    if fp8:
        _need(q_scale, "q_scale", torch.float32)
        _need(k_scale, "k_scale", torch.float32)
    if scores is not None:
        _need(scores, "scores", torch.float32, 2)
        if scores.shape[0] != q.shape[0] or scores.shape[1] != scores_ld(max_visible):
            raise ValueError("scores must be [R, scores_ld(max_visible)]")
    R, H, D = q.shape
    return N.IndexerArgs(B=row_offsets.numel() - 1, R=R, n_heads=H, head_dim=D, topk=topk,
                         dtype=N.MTPSD_FP8_E4M3 if fp8 else N.MTPSD_F32,
                         q=q.data_ptr(), q_scale=q_scale.data_ptr() if fp8 else None,
                         weights=weights.data_ptr(), k_cache=k_cache.data_ptr(),
                         k_scale=k_scale.data_ptr() if fp8 else None, pool_tokens=k_cache.shape[0],
                         cache_start=None if cache_start is None else cache_start.data_ptr(),
                         row_offsets=row_offsets.data_ptr(),
                         row_pos=row_pos.data_ptr(), max_visible=max_visible,
                         topk_idx=None if topk_idx is None else topk_idx.data_ptr(),
                         topk_score=None if topk_score is None else topk_score.data_ptr(),
                         scores=None if scores is None else scores.data_ptr(),
                         workspace=ws.data_ptr(), workspace_bytes=ws.numel(),
                         dev_status=None if dev_status is None else dev_status.data_ptr())


def indexer_topk(q, q_scale, weights, k_cache, k_scale, cache_start, row_offsets, row_pos, topk: int,
                 max_visible: int, topk_idx=None, topk_score=None, scores=None, workspace=None,
                 dev_status=None, stream=None, paged=None):
    """paged = (block_table [B, n] int32, page_size) reads the caches through the block table
    (cache_start is then ignored and may be None)."""
    R = q.shape[0]
    B = row_offsets.numel() - 1
    if topk_idx is None:
        topk_idx = torch.empty(R, topk, dtype=torch.int32, device=q.device)
    nbytes = indexer_topk_aux_bytes(B, R, max_visible, topk) if scores is not None else \
        indexer_topk_workspace_size(B, R, max_visible, topk)
    ws = _ws(workspace, nbytes, q.device)
    a = _indexer_args(q, q_scale, weights, k_cache, k_scale, cache_start, row_offsets, row_pos, topk, max_visible,
                      topk_idx, topk_score, scores, ws, dev_status)
    if paged is None:
        check("mtpsd_indexer_topk", lib().mtpsd_indexer_topk(C.byref(a), _stream(stream)))
    else:
        check("mtpsd_indexer_topk_paged", lib().mtpsd_indexer_topk_paged(C.byref(a), _byref(_paged(paged)),
                                                                           _stream(stream)))
    return topk_idx


def indexer_scores(q, q_scale, weights, k_cache, k_scale, cache_start, row_offsets, row_pos, max_visible: int,
                   scores=None, workspace=None, dev_status=None, stream=None, paged=None):
    """The score matrix [R, scores_ld(max_visible)] alone (row r valid up to row_pos[r])."""
    R = q.shape[0]
    B = row_offsets.numel() - 1
    if scores is None:
        scores = torch.empty(R, scores_ld(max_visible), dtype=torch.float32, device=q.device)
    ws = _ws(workspace, indexer_plan_bytes(B, R), q.device)
    a = _indexer_args(q, q_scale, weights, k_cache, k_scale, cache_start, row_offsets, row_pos, 1, max_visible,
                      None, None, scores, ws, dev_status)
    if paged is None:
        check("mtpsd_indexer_scores", lib().mtpsd_indexer_scores(C.byref(a), _stream(stream)))
    else:
        check("mtpsd_indexer_scores_paged", lib().mtpsd_indexer_scores_paged(C.byref(a), _byref(_paged(paged)),
                                                                             _stream(stream)))
    return scores


def topk(scores, row_len, max_len: int, k: int, out_idx=None, out_score=None, dev_status=None, stream=None,
         row_len_add: int = 0, workspace=None):
    """Top-k per row; row r's valid prefix has row_len[r] + row_len_add scores."""
    _need(scores, "scores", torch.float32, 2)
    _need(row_len, "row_len", torch.int64, 1)
    R, ld = scores.shape
    if out_idx is None:
        out_idx = torch.empty(R, k, dtype=torch.int32, device=scores.device)
    nbytes = topk_workspace_size(R, max_len, k)
    ws = _ws(workspace, nbytes, scores.device) if nbytes else None
    check("mtpsd_topk", lib().mtpsd_topk(
        _ptr(scores), ld, R, _ptr(row_len), row_len_add, max_len, k, _ptr(out_idx), _ptr(out_score), _ptr(ws),
        0 if ws is None else ws.numel(), _ptr(dev_status), _stream(stream)))
    return out_idx


# --------------------------------------------------------------------------- sparse MLA

def sparse_mla_workspace_size(R, H, n_idx, n_append, dtype) -> int:
    return int(lib().mtpsd_sparse_mla_workspace_size(R, H, n_idx, n_append, dtype))


def indexer_topk_launch_count(H, D, dtype, max_visible, topk) -> int:
    """Kernel launches of one indexer_topk call (aligned q and k_cache)."""
    return int(lib().mtpsd_indexer_topk_launch_count(H, D, dtype, max_visible, topk))


def topk_launch_count(max_len, k) -> int:
    """Kernel launches of one topk call (aligned score rows)."""
    return int(lib().mtpsd_topk_launch_count(max_len, k))


def indexer_scores_launch_count(H, D, dtype) -> int:
    """Kernel launches of one indexer_scores call (aligned q and k_cache)."""
    return int(lib().mtpsd_indexer_scores_launch_count(H, D, dtype))


def sparse_mla_launch_count(R, H, n_idx, n_append, dtype) -> int:
    """Kernel launches of one sparse_mla_decode call (16-byte aligned output)."""
    return int(lib().mtpsd_sparse_mla_launch_count(R, H, n_idx, n_append, dtype))


def sparse_mla_decode(q, latent, cache_start, row_offsets, row_pos, idx, softmax_scale: float,
                      n_append: int = 0, append_base=None, row_pos_add: int = 0, out=None, lse=None,
                      workspace=None, dev_status=None, stream=None, paged=None):
    """paged = (block_table [B, n] int32, page_size) gathers through the block table (cache_start is
    then ignored and may be None)."""
    bf16 = q.dtype == torch.bfloat16
    _need(q, "q", torch.bfloat16 if bf16 else torch.float32, 3)
    fp8kv = latent.dtype == torch.uint8     # the packed FP8 latent cache (656-byte rows)
    if fp8kv:
        _need(latent, "latent", torch.uint8, 2)
        if not bf16 or latent.shape[1] != 656:
            raise ValueError("an FP8 latent cache needs bf16 queries and 656-byte rows")
    else:
        _need(latent, "latent", q.dtype, 2)
    if cache_start is not None:
        _need(cache_start, "cache_start", torch.int64, 1)
    _need(row_offsets, "row_offsets", torch.uint32, 1)
    _need(row_pos, "row_pos", torch.int64, 1)
    _need(idx, "idx", torch.int32, 2)
    if append_base is not None:
        _need(append_base, "append_base", torch.int64, 1)
    R, H, DL = q.shape
    dt = N.MTPSD_FP8_DS_MLA if fp8kv else (N.MTPSD_BF16 if bf16 else N.MTPSD_F32)
    if out is None:
        out = torch.empty(R, H, 512, dtype=q.dtype, device=q.device)
    nbytes = sparse_mla_workspace_size(R, H, idx.shape[1], n_append, dt)
    ws = _ws(workspace, nbytes, q.device) if nbytes else workspace
    a = N.MlaArgs(B=row_offsets.numel() - 1, R=R, n_heads=H, d_latent=DL, d_v=512, n_idx=idx.shape[1],
                  n_append=n_append, dtype=dt, softmax_scale=softmax_scale, row_pos_add=row_pos_add,
                  q=q.data_ptr(), latent=latent.data_ptr(), pool_tokens=latent.shape[0],
                  cache_start=None if cache_start is None else cache_start.data_ptr(),
                  row_offsets=row_offsets.data_ptr(), row_pos=row_pos.data_ptr(), idx=idx.data_ptr(),
                  append_base=None if append_base is None else append_base.data_ptr(),
                  out=out.data_ptr(), lse=None if lse is None else lse.data_ptr(),
                  workspace=None if ws is None else ws.data_ptr(),
                  workspace_bytes=0 if ws is None else ws.numel(),
                  dev_status=None if dev_status is None else dev_status.data_ptr())
    if paged is None:
        check("mtpsd_sparse_mla_decode", lib().mtpsd_sparse_mla_decode(C.byref(a), _stream(stream)))
    else:
        check("mtpsd_sparse_mla_decode_paged", lib().mtpsd_sparse_mla_decode_paged(
            C.byref(a), _byref(_paged(paged)), _stream(stream)))
    return out


# --------------------------------------------------------------------------- accept / write-back / share

def accept_greedy(draft, target_argmax, magic_draft_id: int = -1, num_accepted=None, next_tokens=None,
                  stream=None):
    _need(draft, "draft", torch.int64, 2)
    _need(target_argmax, "target_argmax", torch.int64, 2)
    B, K = draft.shape
    if target_argmax.shape != (B, K + 1):
        raise ValueError("target_argmax must be [B, K+1]")
    if num_accepted is None:
        num_accepted = torch.empty(B, dtype=torch.int32, device=draft.device)
    if next_tokens is None:
        next_tokens = torch.empty(B, dtype=torch.int64, device=draft.device)
    check("mtpsd_accept_greedy", lib().mtpsd_accept_greedy(
        _ptr(draft), _ptr(target_argmax), B, K, magic_draft_id, _ptr(num_accepted), _ptr(next_tokens),
        _stream(stream)))
    return num_accepted, next_tokens


def accept_stochastic(draft, draft_probs, target_probs, u_accept, u_sample, num_accepted=None, next_tokens=None,
                      dev_status=None, stream=None):
    """Rejection-sampling acceptance: draft [B, K] int64, draft_probs [B, K, V] and target_probs [B, K+1, V]
    float32, u_accept [B, K] and u_sample [B] float32 uniforms."""
    _need(draft, "draft", torch.int64, 2)
    _need(draft_probs, "draft_probs", torch.float32, 3)
    _need(target_probs, "target_probs", torch.float32, 3)
    _need(u_accept, "u_accept", torch.float32, 2)
    _need(u_sample, "u_sample", torch.float32, 1)
    B, K = draft.shape
    V = target_probs.shape[2]
    if target_probs.shape != (B, K + 1, V) or draft_probs.shape != (B, K, V) or u_accept.shape != (B, K) \
            or u_sample.shape != (B,):
        raise ValueError("shapes must be draft [B,K], draft_probs [B,K,V], target_probs [B,K+1,V], "
                         "u_accept [B,K], u_sample [B]")
    if num_accepted is None:
        num_accepted = torch.empty(B, dtype=torch.int32, device=draft.device)
    if next_tokens is None:
        next_tokens = torch.empty(B, dtype=torch.int64, device=draft.device)
    check("mtpsd_accept_stochastic", lib().mtpsd_accept_stochastic(
        _ptr(draft), _ptr(draft_probs), _ptr(target_probs), _ptr(u_accept), _ptr(u_sample), B, K, V,
        _ptr(num_accepted), _ptr(next_tokens), _ptr(dev_status), _stream(stream)))
    return num_accepted, next_tokens


def kv_writeback(src_latent, src_idxk, src_idxs, num_accepted, dst_latent, dst_idxk, dst_idxs, cache_start, dst_pos,
                 next_pos=None, dev_status=None, stream=None):
    bf16 = src_latent.dtype == torch.bfloat16
    fp8kv = src_latent.dtype == torch.uint8   # packed FP8 latent rows (656 bytes)
    _need(src_latent, "src_latent", src_latent.dtype if fp8kv else (torch.bfloat16 if bf16 else torch.float32), 3)
    _need(dst_latent, "dst_latent", src_latent.dtype, 2)
    _need(num_accepted, "num_accepted", torch.int32, 1)
    _need(cache_start, "cache_start", torch.int64, 1)
    _need(dst_pos, "dst_pos", torch.int64, 1)
    B, W, _ = src_latent.shape
    idx_dim = 0
    if src_idxk is not None:
        _need(src_idxk, "src_idxk", torch.uint8, 3)
        _need(dst_idxk, "dst_idxk", torch.uint8, 2)
        idx_dim = src_idxk.shape[2]
    if src_idxs is not None:
        _need(src_idxs, "src_idxs", torch.float32)
        _need(dst_idxs, "dst_idxs", torch.float32)
    check("mtpsd_kv_writeback", lib().mtpsd_kv_writeback(
        _ptr(src_latent), _ptr(src_idxk), _ptr(src_idxs), B, W,
        N.MTPSD_FP8_DS_MLA if fp8kv else (N.MTPSD_BF16 if bf16 else N.MTPSD_F32), idx_dim,
        _ptr(num_accepted), _ptr(dst_latent), _ptr(dst_idxk), _ptr(dst_idxs), _ptr(cache_start), _ptr(dst_pos),
        dst_latent.shape[0], _ptr(next_pos), _ptr(dev_status), _stream(stream)))
    return next_pos


def topk_share_gather(step0_topk, row_offsets, num_accepted=None, shared_idx=None, dev_status=None, stream=None,
                      row_pos=None, shared_pos=None):
    """shared_idx[b] = step0_topk[row_offsets[b] + num_accepted[b]] (row 0 without num_accepted); with
    row_pos, shared_pos[b] receives the position of that row."""
    _need(step0_topk, "step0_topk", torch.int32, 2)
    _need(row_offsets, "row_offsets", torch.uint32, 1)
    if num_accepted is not None:
        _need(num_accepted, "num_accepted", torch.int32, 1)
    B = row_offsets.numel() - 1
    k = step0_topk.shape[1]
    if shared_idx is None:
        shared_idx = torch.empty(B, k, dtype=torch.int32, device=step0_topk.device)
    if row_pos is not None:
        _need(row_pos, "row_pos", torch.int64, 1)
        if shared_pos is None:
            shared_pos = torch.empty(B, dtype=torch.int64, device=step0_topk.device)
    check("mtpsd_topk_share_gather", lib().mtpsd_topk_share_gather(
        _ptr(step0_topk), _ptr(row_offsets), _ptr(num_accepted), B, k, _ptr(shared_idx), _ptr(row_pos),
        _ptr(shared_pos if row_pos is not None else None), _ptr(dev_status), _stream(stream)))
    return shared_idx


# --------------------------------------------------------------------------- paged caches

def _latent_dtype(t):
    if t.dtype == torch.uint8:
        return N.MTPSD_FP8_DS_MLA
    return N.MTPSD_BF16 if t.dtype == torch.bfloat16 else N.MTPSD_F32


def assign_cache_locs(block_table, page_size: int, start_pos, W: int, out_cache_loc=None, dev_status=None,
                      stream=None):
    """out_cache_loc [B, W] int64: the slots of positions start_pos[b] + j (j < W), -1 where none."""
    _need(start_pos, "start_pos", torch.int64, 1)
    B = start_pos.numel()
    if out_cache_loc is None:
        out_cache_loc = torch.empty(B, W, dtype=torch.int64, device=start_pos.device)
    pk = _paged((block_table, page_size))
    check("mtpsd_assign_cache_locs", lib().mtpsd_assign_cache_locs(
        C.byref(pk), B, _ptr(start_pos), W, _ptr(out_cache_loc), _ptr(dev_status), _stream(stream)))
    return out_cache_loc


def kv_move_accepted(latent, idxk, idxs, out_cache_loc, accept_index, num_accepted, dev_status=None, stream=None):
    """Moves the accepted rows' KV (window slots out_cache_loc[b, accept_index[b, i]]) to the front slots
    out_cache_loc[b, i], i < num_accepted[b] + 1, in every cache of the layer (in place)."""
    _need(latent, "latent", latent.dtype, 2)
    _need(out_cache_loc, "out_cache_loc", torch.int64, 2)
    _need(accept_index, "accept_index", torch.int32, 2)
    _need(num_accepted, "num_accepted", torch.int32, 1)
    B, W = out_cache_loc.shape
    idx_dim = 0
    if idxk is not None:
        _need(idxk, "idxk", torch.uint8, 2)
        idx_dim = idxk.shape[1]
    if idxs is not None:
        _need(idxs, "idxs", torch.float32, 1)
    check("mtpsd_kv_move_accepted", lib().mtpsd_kv_move_accepted(
        _ptr(latent), _latent_dtype(latent), _ptr(idxk), idx_dim, _ptr(idxs), latent.shape[0],
        _ptr(out_cache_loc), _ptr(accept_index), _ptr(num_accepted), B, W, _ptr(dev_status), _stream(stream)))


def kv_writeback_slots(src_latent, src_idxk, src_idxs, num_accepted, dst_latent, dst_idxk, dst_idxs, dst_slots,
                       dst_pos=None, next_pos=None, dev_status=None, stream=None):
    """The accepted rows (num_accepted + 1, clamped to [1, W]) of each window to pool slots dst_slots [B, W];
    with dst_pos, next_pos[b] = dst_pos[b] + the rows written."""
    _need(src_latent, "src_latent", src_latent.dtype, 3)
    _need(dst_latent, "dst_latent", src_latent.dtype, 2)
    _need(num_accepted, "num_accepted", torch.int32, 1)
    _need(dst_slots, "dst_slots", torch.int64, 2)
    B, W, _ = src_latent.shape
    idx_dim = 0
    if src_idxk is not None:
        _need(src_idxk, "src_idxk", torch.uint8, 3)
        _need(dst_idxk, "dst_idxk", torch.uint8, 2)
        idx_dim = src_idxk.shape[2]
    if src_idxs is not None:
        _need(src_idxs, "src_idxs", torch.float32)
        _need(dst_idxs, "dst_idxs", torch.float32)
    check("mtpsd_kv_writeback_slots", lib().mtpsd_kv_writeback_slots(
        _ptr(src_latent), _ptr(src_idxk), _ptr(src_idxs), B, W, _latent_dtype(src_latent), idx_dim,
        _ptr(num_accepted), _ptr(dst_latent), _ptr(dst_idxk), _ptr(dst_idxs), _ptr(dst_slots), dst_latent.shape[0],
        _ptr(dst_pos), _ptr(next_pos), _ptr(dev_status), _stream(stream)))
    return next_pos
