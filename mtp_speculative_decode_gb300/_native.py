"""ctypes declarations of libmtpsd.so (the C ABI in include/mtpsd.h).

Loading fails loudly when the library has not been built: there is no
fallback implementation of any step.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmtpsd.so")

MTPSD_OK = 0
MTPSD_EINVAL = -1
MTPSD_EUNSUPPORTED = -2
MTPSD_ECUDA = -3
MTPSD_EWORKSPACE = -4

MTPSD_F32 = 0
MTPSD_BF16 = 1
MTPSD_FP8_E4M3 = 2
MTPSD_FP8_DS_MLA = 3

NOALLOC_SCRATCH_BYTES = 16 << 20   # MTPSD_NOALLOC_SCRATCH_BYTES

STATUS_INDEX_RANGE = 1
STATUS_WRITE_RANGE = 2
STATUS_WAIT_TIMEOUT = 4
STATUS_ROW_RANGE = 8

vp = C.c_void_p
i32 = C.c_int32
i64 = C.c_int64


class IndexerArgs(C.Structure):
    _fields_ = [
        ("B", i32), ("R", i32), ("n_heads", i32), ("head_dim", i32), ("topk", i32), ("dtype", i32),
        ("q", vp), ("q_scale", vp), ("weights", vp), ("k_cache", vp), ("k_scale", vp),
        ("pool_tokens", i64), ("cache_start", vp), ("row_offsets", vp), ("row_pos", vp),
        ("max_visible", i64), ("topk_idx", vp), ("topk_score", vp), ("scores", vp),
        ("workspace", vp), ("workspace_bytes", C.c_size_t), ("dev_status", vp),
    ]


class MlaArgs(C.Structure):
    _fields_ = [
        ("B", i32), ("R", i32), ("n_heads", i32), ("d_latent", i32), ("d_v", i32), ("n_idx", i32),
        ("n_append", i32), ("dtype", i32), ("softmax_scale", C.c_float), ("row_pos_add", i64),
        ("q", vp), ("latent", vp), ("pool_tokens", i64), ("cache_start", vp), ("row_offsets", vp),
        ("row_pos", vp), ("idx", vp), ("append_base", vp), ("out", vp), ("lse", vp),
        ("workspace", vp), ("workspace_bytes", C.c_size_t), ("dev_status", vp),
    ]


class PagedKV(C.Structure):
    _fields_ = [("block_table", vp), ("bt_stride", i32), ("page_size", i32)]


# name -> (restype, argtypes); every symbol include/mtpsd.h declares
SIGNATURES = {
    "mtpsd_merge_tokens": (C.c_int, [vp, i64, vp, vp, i32, i32, vp, vp, vp]),
    "mtpsd_host_merged_offsets": (None, [vp, i32, i32, vp]),
    "mtpsd_resolve_indexer_types": (C.c_int, [i32, C.c_char_p, i32, i32, vp]),
    "mtpsd_quantize_fp8_block128": (C.c_int, [vp, i64, vp, vp, vp]),
    "mtpsd_pack_latent_fp8": (C.c_int, [vp, i32, i64, vp, vp]),
    "mtpsd_scores_ld": (i64, [i64]),
    "mtpsd_indexer_topk_workspace_size": (C.c_size_t, [i32, i32, i64, i32]),
    "mtpsd_indexer_topk_plan_bytes": (C.c_size_t, [i32, i32]),
    "mtpsd_indexer_topk_aux_bytes": (C.c_size_t, [i32, i32, i64, i32]),
    "mtpsd_indexer_topk": (C.c_int, [C.POINTER(IndexerArgs), vp]),
    "mtpsd_indexer_topk_noalloc": (C.c_int, [C.POINTER(IndexerArgs), vp]),
    "mtpsd_indexer_scores": (C.c_int, [C.POINTER(IndexerArgs), vp]),
    "mtpsd_indexer_scores_launch_count": (i32, [i32, i32, i32]),
    "mtpsd_topk_workspace_size": (C.c_size_t, [i32, i64, i32]),
    "mtpsd_topk_launch_count": (i32, [i64, i32]),
    "mtpsd_topk": (C.c_int, [vp, i64, i32, vp, i64, i64, i32, vp, vp, vp, C.c_size_t, vp, vp]),
    "mtpsd_sparse_mla_workspace_size": (C.c_size_t, [i32, i32, i32, i32, i32]),
    "mtpsd_sparse_mla_launch_count": (i32, [i32, i32, i32, i32, i32]),
    "mtpsd_indexer_topk_launch_count": (i32, [i32, i32, i32, i64, i32]),
    "mtpsd_sparse_mla_decode": (C.c_int, [C.POINTER(MlaArgs), vp]),
    "mtpsd_accept_greedy": (C.c_int, [vp, vp, i32, i32, i64, vp, vp, vp]),
    "mtpsd_accept_stochastic": (C.c_int, [vp, vp, vp, vp, vp, i32, i32, i64, vp, vp, vp, vp]),
    "mtpsd_kv_writeback": (C.c_int, [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, i64, vp, vp, vp]),
    "mtpsd_assign_cache_locs": (C.c_int, [C.POINTER(PagedKV), i32, vp, i32, vp, vp, vp]),
    "mtpsd_kv_move_accepted": (C.c_int, [vp, i32, vp, i32, vp, i64, vp, vp, vp, i32, i32, vp, vp]),
    "mtpsd_kv_writeback_slots": (C.c_int, [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, i64, vp, vp, vp, vp]),
    "mtpsd_indexer_topk_paged": (C.c_int, [C.POINTER(IndexerArgs), C.POINTER(PagedKV), vp]),
    "mtpsd_indexer_scores_paged": (C.c_int, [C.POINTER(IndexerArgs), C.POINTER(PagedKV), vp]),
    "mtpsd_sparse_mla_decode_paged": (C.c_int, [C.POINTER(MlaArgs), C.POINTER(PagedKV), vp]),
    "mtpsd_topk_share_gather": (C.c_int, [vp, vp, vp, i32, i32, vp, vp, vp, vp, vp]),
    "mtpsd_check_bounded_wait": (C.c_int, [i64, vp, vp, vp]),
    "mtpsd_last_error": (C.c_char_p, []),
    "mtpsd_version": (i32, []),
}

_lib = None


def lib() -> C.CDLL:
    """The loaded library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m mtp_speculative_decode_gb300.build` "
                "(there is no fallback implementation)")
        handle = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


class MtpsdError(RuntimeError):
    def __init__(self, fn: str, code: int):
        msg = lib().mtpsd_last_error()
        super().__init__(f"{fn} failed with code {code}: {msg.decode() if msg else ''}")
        self.code = code


def check(fn: str, code: int) -> None:
    if code != MTPSD_OK:
        raise MtpsdError(fn, code)
