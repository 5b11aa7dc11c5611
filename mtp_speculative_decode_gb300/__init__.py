"""GB300-native decode-time DSA sparse attention for MTP speculative decoding.

The compute path is libmtpsd.so (hand-written CUDA for sm_103a behind the C
ABI of include/mtpsd.h); this package is its thin Python binding plus the
seeded synthetic workloads used by the tests and the benchmark."""
from .api import (Workspace, accept_greedy, accept_stochastic, assign_cache_locs, host_merged_offsets,
                  indexer_scores, indexer_topk, indexer_topk_workspace_size, kv_move_accepted, kv_writeback,
                  kv_writeback_slots, merge_tokens, pack_latent_fp8, quantize_fp8_block128, scores_ld,
                  sparse_mla_decode, sparse_mla_workspace_size, topk, topk_share_gather)

__all__ = [
    "Workspace", "accept_greedy", "accept_stochastic", "assign_cache_locs", "host_merged_offsets",
    "indexer_scores", "indexer_topk", "indexer_topk_workspace_size", "kv_move_accepted", "kv_writeback",
    "kv_writeback_slots", "merge_tokens", "pack_latent_fp8", "quantize_fp8_block128", "scores_ld",
    "sparse_mla_decode", "sparse_mla_workspace_size", "topk", "topk_share_gather",
]
