"""CPU oracle for the decode-time DSA step under MTP speculative decoding.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (the C-ABI library and its Python binding) never
imports, calls or links anything here, and this package imports nothing from
the product path.

Every function is a plain, slow restatement of what the source pages define,
in float64 unless noted, written for a reader to check against the pages by
eye.  Page titles used in citations:

* [P1] "MAX 中 GLM-5.2 (DeepSeek-V3.2 Sparse) 的统一 MTP 推测解码架构解析"
* [P2] "GLM-5.3 推理全链路(十四):MTP 的三段前向——草稿、验证与 draft_extend 的算子与通信账"
* [P3] "MAX Pipeline 中的 DeepSeek-V3.2 架构实现解析:稀疏注意力、Lightning Indexer 与 MoE 并行推理"
* [P4] "MAX 推测解码配置指南:解读 max.pipelines.speculative 模块"

Pinning (what each function is checked against, other than itself) lives in
``tests/test_oracle_*.py``.  Parity status per function:

* fp8.decode_e4m3 / quantize_block128 — pinned (exhaustive vs a library codec)
* merge.merge_tokens / host_merged_offsets — pinned (hand-worked example)
* indexer.indexer_scores — pinned (hand-worked values, brute force loops,
  special cases)
* topk.topk_select — pinned (brute force over all subsets on tiny inputs)
* mla.sparse_mla — pinned (dense softmax attention when k >= context,
  single-index and q = 0 closed forms)
* accept.accept_greedy — pinned (hand-worked cases)
* writeback.kv_writeback — pinned (byte-level cases)
* share.topk_share_gather / shared_index_list — pinned (equals rerunning the
  indexer when the context is shorter than k)
* accept.accept_stochastic — pinned (hand-worked chains, the emitted
  distribution equals the target's, exact fixed-point draw)
* share.resolve_indexer_types / source_layers / seeded_step_positions —
  pinned (the pages' layer counts, hand-worked schedules and positions)
* mla.pack_fp8_ds_mla / unpack_fp8_ds_mla — pinned (hand-worked token, round
  trip)
* paged.slot_of / assign_cache_locs / gather_positions / kv_move_accepted /
  kv_writeback_slots — pinned (hand-worked block tables, a paged pool built
  page by page reads back the contiguous cache, a swap that an in-place copy
  gets wrong, the contiguous write-back as a special case)
"""
