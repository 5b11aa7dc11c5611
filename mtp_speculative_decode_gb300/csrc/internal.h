// Internal launchers of libmtpsd (called by api.cu after argument checks).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mtpsd {

// Block-table indirection of a paged cache (bt == nullptr: contiguous, pool row cache_start[b] + s).
// Position s of request b lives in slot bt[b * stride + (s >> shift)] << shift | (s & (2^shift - 1)).
struct Paging {
  const int32_t* bt = nullptr;
  int32_t stride = 0;
  int32_t shift = 0;
};

// 2D tensor map with the 128-byte swizzle (map: a 64-byte aligned CUtensorMap).
// dtype_u8_or_bf16: 0 = uint8 elements, 1 = bf16 elements.
bool tma_available();
bool make_tma_store_map(void* map, bool f32, const void* base, int rank, const uint64_t* dims,
                        const uint64_t* strides, const uint32_t* box);
bool make_tma_2d(void* map, int dtype_u8_or_bf16, const void* base, uint64_t inner_elems, uint64_t rows,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, bool l2_256);
bool make_tma_1d_f32(void* map, const void* base, uint64_t n_elems, uint32_t box_elems);
bool make_tma_2d_plain_u8(void* map, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_bytes);

int launch_merge_tokens(const int64_t* prompt, int64_t S, const uint32_t* po, const int64_t* draft,
                        int B, int K, int64_t* out, uint32_t* mo, cudaStream_t st);
int launch_quantize_fp8(const float* x, int64_t n_blocks, uint8_t* codes, float* scales, cudaStream_t st);
int launch_pack_latent_fp8(const void* latent, bool f32_in, int64_t T, uint8_t* out, cudaStream_t st);
int launch_accept_greedy(const int64_t* draft, const int64_t* tgt, int B, int K, int64_t magic,
                         int32_t* n_acc, int64_t* next, cudaStream_t st);
int launch_kv_writeback(const void* src_l, const uint8_t* src_k, const float* src_s, int B, int W,
                        int lat_bytes, int idx_bytes, const int32_t* n_acc, void* dst_l, uint8_t* dst_k,
                        float* dst_s, const int64_t* cache_start, const int64_t* dst_pos, int64_t pool, int64_t* next_pos,
                        int32_t* status, cudaStream_t st, const int64_t* dst_slots = nullptr);
int launch_assign_cache_locs(const Paging& pg, int B, const int64_t* start_pos, int W, int64_t* out, int32_t* status,
                             cudaStream_t st);
int launch_kv_move(void* lat, int lat_bytes, uint8_t* idxk, int idx_bytes, float* idxs, int64_t pool,
                   const int64_t* loc, const int32_t* acc_idx, const int32_t* n_acc, int B, int W, int32_t* status,
                   cudaStream_t st);
int launch_accept_stochastic(const int64_t* draft, const float* q, const float* p, const float* ua, const float* us,
                             int B, int K, int64_t V, int32_t* n_acc, int64_t* next, int32_t* status, cudaStream_t st);
int launch_bounded_wait_check(int64_t limit_ns, int32_t* status, int64_t* out, cudaStream_t st);
int launch_share_gather(const int32_t* s0, const uint32_t* ro, const int32_t* n_acc, int B, int k,
                        int32_t* out, const int64_t* row_pos, int64_t* shared_pos, int32_t* status, cudaStream_t st);

// indexer scores into a [R, ld] float matrix (positions > row_pos are not written)
struct IndexerPlan {
  int B, R, H, D, dtype;
  const void* q; const float* q_scale; const float* w;
  const void* k; const float* k_scale; int64_t pool;
  const int64_t* cache_start; const uint32_t* row_offsets; const int64_t* row_pos;
  int64_t max_visible; float* scores; int64_t ld;
  void* plan_ws;           // workspace for the tensor-core kernel's work plan (indexer_tc_plan_bytes)
  int32_t* status;
  Paging pg;
};
int launch_indexer_scores(const IndexerPlan& p, cudaStream_t st);
size_t indexer_tc_plan_bytes(int B, int R);
int indexer_launch_count(int H, int D, int dtype);
bool indexer_tc_supported(const IndexerPlan& p);
int launch_indexer_scores_tc(const IndexerPlan& p, cudaStream_t st);

// top-k over rows of a score matrix; row length = row_len[r] + len_add
struct TopkPlan {
  const float* scores; int64_t ld; int R; const int64_t* row_len; int64_t len_add;
  int64_t max_len; int k; int32_t* out_idx; float* out_score; int32_t* status;
  void* ws; size_t ws_bytes;   // candidate lists of the split path (rows longer than 40960 keys)
};
int launch_topk(const TopkPlan& p, cudaStream_t st);
size_t topk_workspace_bytes(int R, int64_t max_len, int k);
int topk_launch_count(int64_t max_len, int k, bool aligned);

// sparse MLA
struct MlaPlan {
  int B, R, H, d_latent, d_v, n_idx, n_append, dtype;
  float scale; int64_t row_pos_add;
  const void* q; const void* latent; int64_t pool;
  const int64_t* cache_start; const uint32_t* row_offsets; const int64_t* row_pos;
  const int32_t* idx; const int64_t* append_base;
  void* out; float* lse;
  void* ws; size_t ws_bytes;
  int32_t* status;
  Paging pg;
};
size_t mla_workspace_bytes(int R, int H, int n_idx, int n_append, int dtype);
bool mla_tc_supported(const MlaPlan& p);
int mla_tc_per_split(int R, int H, int64_t total);
int mla_tc_ml_halves();
bool mla_tc_fuse(int n_splits);
int mla_launch_count(int R, int H, int n_idx, int n_append, int dtype);
// Persistent launch of the tensor-core kernel over bf16 rows: `clusters` clusters of two CTAs each take
// pq consecutive pairs of the flattened (row, head group, pair) list (ppr pairs per row and head group,
// hgn head groups, tp pairs in total); `cut`: some row is split between clusters, which leaves float32
// pieces in the workspace and adds the piece merge launch.
struct MlaPersist {
  int clusters, pq, ppr, hgn;
  int64_t tp;
  bool cut;
};
bool mla_tc_persist_plan(int R, int H, int64_t total, int dtype, MlaPersist* pl);
size_t mla_tc_persist_bytes(const MlaPersist& pl);
// Launches the tensor-core kernel; *combined tells whether it also merged the split partials.  With
// pl: the persistent launch (and the piece merge), the pieces in part_o / part_ml.
int launch_sparse_mla_tc(const MlaPlan& p, int n_splits, int per_split, float* part_o, float* part_ml,
                         cudaStream_t st, bool* combined, const MlaPersist* pl = nullptr);
int launch_sparse_mla(const MlaPlan& p, cudaStream_t st);

}  // namespace mtpsd
