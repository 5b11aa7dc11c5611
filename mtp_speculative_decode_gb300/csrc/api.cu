// C ABI of libmtpsd: host-side argument checks, workspace carving and
// dispatch to the kernels.  Nothing here allocates device memory.
#include <stdarg.h>
#include <stdio.h>

#include "common.cuh"
#include "internal.h"

namespace mtpsd {

static thread_local char g_err[512] = "";

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

static int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

static bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Checks a paged-cache descriptor (NULL: contiguous caches) and converts it.
static int check_paged(const mtpsd_paged_kv* pk, Paging* out, const char* who) {
  *out = Paging();
  if (!pk) return MTPSD_OK;
  if (!pk->block_table || pk->bt_stride < 1) return fail(MTPSD_EINVAL, "%s: paged caches need block_table and bt_stride >= 1", who);
  const int32_t ps = pk->page_size;
  if (ps < 1 || ps > 65536 || (ps & (ps - 1))) return fail(MTPSD_EINVAL, "%s: page_size must be a power of two in 1..65536", who);
  out->bt = pk->block_table;
  out->stride = pk->bt_stride;
  while ((1 << out->shift) < ps) ++out->shift;
  return MTPSD_OK;
}

}  // namespace mtpsd

using namespace mtpsd;

extern "C" {

const char* mtpsd_last_error(void) { return g_err; }

int32_t mtpsd_version(void) { return 102; }

int mtpsd_merge_tokens(const int64_t* prompt_tokens, int64_t S, const uint32_t* prompt_offsets,
                       const int64_t* draft_tokens, int32_t B, int32_t K, int64_t* merged_tokens,
                       uint32_t* merged_offsets, void* stream) {
  g_err[0] = 0;
  if (B < 1 || K < 0 || S < 0) return fail(MTPSD_EINVAL, "merge_tokens: need B >= 1, K >= 0, S >= 0");
  if (!prompt_offsets || !merged_offsets || (S > 0 && !prompt_tokens) || (K > 0 && !draft_tokens) ||
      (S + (int64_t)B * K > 0 && !merged_tokens))
    return fail(MTPSD_EINVAL, "merge_tokens: null pointer");
  if (S + (int64_t)B * K > 0xffffffffLL) return fail(MTPSD_EINVAL, "merge_tokens: merged length exceeds uint32 offsets");
  return launch_merge_tokens(prompt_tokens, S, prompt_offsets, draft_tokens, B, K, merged_tokens, merged_offsets,
                             (cudaStream_t)stream);
}

void mtpsd_host_merged_offsets(const uint32_t* prompt_offsets, int32_t B, int32_t K, uint32_t* out) {
  for (int32_t i = 0; i <= B; ++i) out[i] = prompt_offsets[i] + (uint32_t)((int64_t)i * K);
}

int mtpsd_resolve_indexer_types(int32_t n_layers, const char* pattern, int32_t freq, int32_t offset,
                                int32_t* is_full) {
  g_err[0] = 0;
  if (n_layers < 0 || (n_layers > 0 && !is_full)) return fail(MTPSD_EINVAL, "resolve_indexer_types: bad arguments");
  if (pattern && pattern[0]) {
    int32_t n = 0;
    for (const char* c = pattern; *c; ++c, ++n) {
      if (*c != 'F' && *c != 'S') return fail(MTPSD_EINVAL, "resolve_indexer_types: pattern characters must be F or S");
      if (n < n_layers) is_full[n] = *c == 'F';
    }
    if (n != n_layers) return fail(MTPSD_EINVAL, "resolve_indexer_types: pattern length %d != %d layers", n, n_layers);
  } else if (freq > 0 || offset >= 0) {
    const int32_t f = freq > 0 ? freq : 1, o = offset >= 0 ? offset : 2;
    for (int32_t i = 0; i < n_layers; ++i) is_full[i] = ((i - o + 1 > 0 ? i - o + 1 : 0) % f) == 0;
  } else {
    for (int32_t i = 0; i < n_layers; ++i) is_full[i] = 1;
  }
  if (n_layers > 0 && !is_full[0]) return fail(MTPSD_EINVAL, "resolve_indexer_types: the first layer must be full");
  return MTPSD_OK;
}

int mtpsd_quantize_fp8_block128(const float* x, int64_t n_blocks, uint8_t* codes, float* scales, void* stream) {
  g_err[0] = 0;
  if (n_blocks < 0) return fail(MTPSD_EINVAL, "quantize: n_blocks < 0");
  if (n_blocks == 0) return MTPSD_OK;
  if (!x || !codes || !scales) return fail(MTPSD_EINVAL, "quantize: null pointer");
  if (!aligned(x, 16) || !aligned(codes, 4))
    return fail(MTPSD_EINVAL, "quantize: x must be 16-byte and codes 4-byte aligned");
  return launch_quantize_fp8(x, n_blocks, codes, scales, (cudaStream_t)stream);
}

int mtpsd_pack_latent_fp8(const void* latent, int32_t dtype, int64_t T, uint8_t* packed, void* stream) {
  g_err[0] = 0;
  if (T < 0) return fail(MTPSD_EINVAL, "pack_latent_fp8: T < 0");
  if (dtype != MTPSD_BF16 && dtype != MTPSD_F32) return fail(MTPSD_EUNSUPPORTED, "pack_latent_fp8: dtype must be MTPSD_BF16 or MTPSD_F32");
  if (T == 0) return MTPSD_OK;
  if (!latent || !packed) return fail(MTPSD_EINVAL, "pack_latent_fp8: null pointer");
  if (!aligned(latent, 16) || !aligned(packed, 16)) return fail(MTPSD_EINVAL, "pack_latent_fp8: buffers must be 16-byte aligned");
  return launch_pack_latent_fp8(latent, dtype == MTPSD_F32, T, packed, (cudaStream_t)stream);
}

int64_t mtpsd_scores_ld(int64_t max_visible) { return (int64_t)align_up((size_t)(max_visible > 0 ? max_visible : 1), 4); }

size_t mtpsd_indexer_topk_plan_bytes(int32_t B, int32_t R) { return (B < 0 || R < 0) ? 0 : indexer_tc_plan_bytes(B, R); }

size_t mtpsd_indexer_topk_workspace_size(int32_t B, int32_t R, int64_t max_visible, int32_t topk) {
  if (B < 0 || R < 0) return 0;
  size_t scores = (size_t)R * (size_t)mtpsd_scores_ld(max_visible) * sizeof(float);
  return align_up(scores, 256) + indexer_tc_plan_bytes(B, R) + align_up(topk_workspace_bytes(R, max_visible, topk), 256);
}

size_t mtpsd_indexer_topk_aux_bytes(int32_t B, int32_t R, int64_t max_visible, int32_t topk) {
  if (B < 0 || R < 0) return 0;
  return indexer_tc_plan_bytes(B, R) + align_up(topk_workspace_bytes(R, max_visible, topk), 256);
}

}  // extern "C"

namespace mtpsd {
// Checks the indexer arguments and launches the score kernels (plan + tensor-core GEMM, or the CUDA-core
// kernel) into `*scores_out` (args->scores, else the head of the workspace).  need_scores: the call
// requires a caller score buffer (mtpsd_indexer_scores).
static int indexer_scores_checked(const mtpsd_indexer_args* a, const mtpsd_paged_kv* paged, bool need_scores,
                                  bool need_topk, cudaStream_t st, float** scores_out, void** topk_ws,
                                  size_t* topk_ws_bytes) {
  if (!a) return fail(MTPSD_EINVAL, "indexer: null args");
  Paging pg;
  if (int rc = check_paged(paged, &pg, "indexer")) return rc;
  if (a->B < 1 || a->R < 0 || a->n_heads < 1)
    return fail(MTPSD_EINVAL, "indexer: need B >= 1, R >= 0, n_heads >= 1");
  if (a->max_visible < 0 || a->max_visible > 0x7fffffffLL)
    return fail(MTPSD_EINVAL, "indexer: max_visible out of range");
  if (a->dtype == MTPSD_FP8_E4M3) {
    if (a->head_dim != 128) return fail(MTPSD_EUNSUPPORTED, "indexer: FP8 needs head_dim 128 (one block-128 scale per head)");
    if (!a->q_scale || !a->k_scale) return fail(MTPSD_EINVAL, "indexer: FP8 needs q_scale and k_scale");
  } else if (a->dtype == MTPSD_F32) {
    if (a->head_dim < 1 || a->head_dim > 256) return fail(MTPSD_EUNSUPPORTED, "indexer: float32 head_dim 1..256");
  } else {
    return fail(MTPSD_EUNSUPPORTED, "indexer: dtype must be MTPSD_FP8_E4M3 or MTPSD_F32");
  }
  if ((size_t)a->n_heads * a->head_dim > 16384) return fail(MTPSD_EUNSUPPORTED, "indexer: n_heads*head_dim > 16384");
  if (need_topk && (a->topk < 1 || a->topk > 4096)) return fail(MTPSD_EINVAL, "indexer_topk: need 1 <= topk <= 4096");
  if (need_scores && !a->scores) return fail(MTPSD_EINVAL, "indexer_scores: args->scores is required");
  if (a->R == 0) return MTPSD_OK;
  if (!a->q || !a->weights || !a->k_cache || (!pg.bt && !a->cache_start) || !a->row_offsets || !a->row_pos ||
      (need_topk && !a->topk_idx))
    return fail(MTPSD_EINVAL, "indexer: null pointer");
  // the workspace holds the scores (unless the caller gives a buffer), the work plan, and for the top-k
  // of rows longer than 40960 keys its candidate lists
  const size_t score_part = a->scores ? 0 : align_up((size_t)a->R * mtpsd_scores_ld(a->max_visible) * sizeof(float), 256);
  const size_t topk_part = need_topk ? align_up(topk_workspace_bytes(a->R, a->max_visible, a->topk), 256) : 0;
  size_t need = score_part + indexer_tc_plan_bytes(a->B, a->R) + topk_part;
  if (!a->workspace || a->workspace_bytes < need)
    return fail(MTPSD_EWORKSPACE, "indexer: workspace of %zu bytes needed, %zu given", need, a->workspace_bytes);
  if (!aligned(a->workspace, 256)) return fail(MTPSD_EINVAL, "indexer: workspace must be 256-byte aligned");
  if (a->scores && !aligned(a->scores, 16)) return fail(MTPSD_EINVAL, "indexer: scores must be 16-byte aligned");
  const int64_t ld = mtpsd_scores_ld(a->max_visible);
  float* scores = a->scores ? a->scores : (float*)a->workspace;
  IndexerPlan p;
  p.B = a->B; p.R = a->R; p.H = a->n_heads; p.D = a->head_dim; p.dtype = a->dtype;
  p.q = a->q; p.q_scale = a->q_scale; p.w = a->weights; p.k = a->k_cache; p.k_scale = a->k_scale;
  p.pool = a->pool_tokens; p.cache_start = a->cache_start; p.row_offsets = a->row_offsets; p.row_pos = a->row_pos;
  p.max_visible = a->max_visible; p.scores = scores; p.ld = ld;
  p.plan_ws = (char*)a->workspace + score_part;
  p.status = a->dev_status;
  p.pg = pg;
  *scores_out = scores;
  *topk_ws = (char*)a->workspace + score_part + indexer_tc_plan_bytes(a->B, a->R);
  *topk_ws_bytes = topk_part;
  return indexer_tc_supported(p) ? launch_indexer_scores_tc(p, st) : launch_indexer_scores(p, st);
}
}  // namespace mtpsd

extern "C" {

int mtpsd_indexer_scores_paged(const mtpsd_indexer_args* a, const mtpsd_paged_kv* paged, void* stream) {
  g_err[0] = 0;
  float* scores = nullptr;
  void* tws = nullptr;
  size_t twb = 0;
  return indexer_scores_checked(a, paged, true, false, (cudaStream_t)stream, &scores, &tws, &twb);
}

int mtpsd_indexer_scores(const mtpsd_indexer_args* a, void* stream) {
  return mtpsd_indexer_scores_paged(a, nullptr, stream);
}

int32_t mtpsd_indexer_scores_launch_count(int32_t n_heads, int32_t head_dim, int32_t dtype) {
  return indexer_launch_count(n_heads, head_dim, dtype) - 1;
}

int mtpsd_indexer_topk(const mtpsd_indexer_args* a, void* stream) { return mtpsd_indexer_topk_paged(a, nullptr, stream); }

int mtpsd_indexer_topk_paged(const mtpsd_indexer_args* a, const mtpsd_paged_kv* paged, void* stream) {
  g_err[0] = 0;
  cudaStream_t st = (cudaStream_t)stream;
  float* scores = nullptr;
  void* tws = nullptr;
  size_t twb = 0;
  int rc = indexer_scores_checked(a, paged, false, true, st, &scores, &tws, &twb);
  if (rc || a->R == 0) return rc;
  TopkPlan t;
  t.scores = scores; t.ld = mtpsd_scores_ld(a->max_visible); t.R = a->R; t.row_len = a->row_pos; t.len_add = 1;
  t.max_len = a->max_visible; t.k = a->topk; t.out_idx = a->topk_idx; t.out_score = a->topk_score;
  t.status = a->dev_status; t.ws = tws; t.ws_bytes = twb;
  return launch_topk(t, st);
}

int32_t mtpsd_indexer_topk_launch_count(int32_t n_heads, int32_t head_dim, int32_t dtype, int64_t max_visible,
                                        int32_t topk) {
  if (topk < 1 || topk > 4096) return 0;
  return indexer_launch_count(n_heads, head_dim, dtype) - 1 + topk_launch_count(max_visible, topk, true);
}

size_t mtpsd_topk_workspace_size(int32_t R, int64_t max_len, int32_t topk) {
  if (R < 0 || topk < 1 || topk > 4096) return 0;
  return topk_workspace_bytes(R, max_len, topk);
}

int32_t mtpsd_topk_launch_count(int64_t max_len, int32_t topk) {
  if (topk < 1 || topk > 4096) return 0;
  return topk_launch_count(max_len, topk, true);
}

int mtpsd_topk(const float* scores, int64_t ld, int32_t R, const int64_t* row_len, int64_t row_len_add,
               int64_t max_len, int32_t topk, int32_t* out_idx, float* out_score, void* workspace,
               size_t workspace_bytes, int32_t* dev_status, void* stream) {
  g_err[0] = 0;
  if (R < 0 || topk < 1 || topk > 4096 || max_len < 0 || max_len > 0x7fffffffLL || ld < max_len)
    return fail(MTPSD_EINVAL, "topk: need R >= 0, 1 <= topk <= 4096, 0 <= max_len <= ld");
  if (row_len_add < -0x7fffffffLL || row_len_add > 0x7fffffffLL) return fail(MTPSD_EINVAL, "topk: row_len_add out of range");
  if (R == 0) return MTPSD_OK;
  if (!scores || !row_len || !out_idx) return fail(MTPSD_EINVAL, "topk: null pointer");
  const size_t need = topk_workspace_bytes(R, max_len, topk);
  if (need && (!workspace || workspace_bytes < need))
    return fail(MTPSD_EWORKSPACE, "topk: workspace of %zu bytes needed, %zu given", need, workspace_bytes);
  if (need && !aligned(workspace, 256)) return fail(MTPSD_EINVAL, "topk: workspace must be 256-byte aligned");
  TopkPlan t;
  t.scores = scores; t.ld = ld; t.R = R; t.row_len = row_len; t.len_add = row_len_add; t.max_len = max_len;
  t.k = topk; t.out_idx = out_idx; t.out_score = out_score; t.status = dev_status;
  t.ws = workspace; t.ws_bytes = workspace_bytes;
  return launch_topk(t, (cudaStream_t)stream);
}

size_t mtpsd_sparse_mla_workspace_size(int32_t R, int32_t n_heads, int32_t n_idx, int32_t n_append, int32_t dtype) {
  if (R <= 0 || n_heads <= 0 || n_idx < 0 || n_append < 0) return 0;
  return mla_workspace_bytes(R, n_heads, n_idx, n_append, dtype);
}

int32_t mtpsd_sparse_mla_launch_count(int32_t R, int32_t n_heads, int32_t n_idx, int32_t n_append, int32_t dtype) {
  if (R <= 0 || n_heads <= 0 || n_idx < 0 || n_append < 0) return 0;
  return mla_launch_count(R, n_heads, n_idx, n_append, dtype);
}

int mtpsd_sparse_mla_decode(const mtpsd_mla_args* a, void* stream) { return mtpsd_sparse_mla_decode_paged(a, nullptr, stream); }

int mtpsd_sparse_mla_decode_paged(const mtpsd_mla_args* a, const mtpsd_paged_kv* paged, void* stream) {
  g_err[0] = 0;
  if (!a) return fail(MTPSD_EINVAL, "sparse_mla_decode: null args");
  Paging pg;
  if (int rc = check_paged(paged, &pg, "sparse_mla_decode")) return rc;
  if (a->B < 1 || a->R < 0 || a->n_heads < 1 || a->n_idx < 0 || a->n_append < 0)
    return fail(MTPSD_EINVAL, "sparse_mla_decode: need B >= 1, R >= 0, n_heads >= 1, n_idx >= 0, n_append >= 0");
  if (a->d_latent != 576 || a->d_v != 512)
    return fail(MTPSD_EUNSUPPORTED, "sparse_mla_decode: d_latent must be 576 and d_v 512");
  if ((int64_t)a->n_idx + a->n_append > 65536) return fail(MTPSD_EUNSUPPORTED, "sparse_mla_decode: more than 65536 positions per row");
  if (a->dtype == MTPSD_BF16 || a->dtype == MTPSD_FP8_DS_MLA) {
    if (a->n_heads % 16) return fail(MTPSD_EUNSUPPORTED, "sparse_mla_decode: bf16 needs n_heads % 16 == 0");
  } else if (a->dtype != MTPSD_F32) {
    return fail(MTPSD_EUNSUPPORTED, "sparse_mla_decode: dtype must be MTPSD_BF16, MTPSD_FP8_DS_MLA or MTPSD_F32");
  }
  if (a->n_append > 0 && !a->append_base) return fail(MTPSD_EINVAL, "sparse_mla_decode: n_append > 0 needs append_base");
  if (a->R == 0) return MTPSD_OK;
  if (!a->q || !a->latent || (!pg.bt && !a->cache_start) || !a->row_offsets || !a->row_pos || !a->out || (a->n_idx > 0 && !a->idx))
    return fail(MTPSD_EINVAL, "sparse_mla_decode: null pointer");
  if (a->dtype != MTPSD_F32 && (!aligned(a->q, 16) || !aligned(a->latent, 16) || !aligned(a->out, 4)))
    return fail(MTPSD_EINVAL, "sparse_mla_decode: q and latent must be 16-byte aligned");
  MlaPlan p;
  p.B = a->B; p.R = a->R; p.H = a->n_heads; p.d_latent = a->d_latent; p.d_v = a->d_v; p.n_idx = a->n_idx;
  p.n_append = a->n_append; p.dtype = a->dtype; p.scale = a->softmax_scale; p.row_pos_add = a->row_pos_add;
  p.q = a->q; p.latent = a->latent; p.pool = a->pool_tokens; p.cache_start = a->cache_start;
  p.row_offsets = a->row_offsets; p.row_pos = a->row_pos; p.idx = a->idx; p.append_base = a->append_base;
  p.out = a->out; p.lse = a->lse; p.ws = a->workspace; p.ws_bytes = a->workspace_bytes; p.status = a->dev_status;
  p.pg = pg;
  return launch_sparse_mla(p, (cudaStream_t)stream);
}

int mtpsd_accept_greedy(const int64_t* draft, const int64_t* target_argmax, int32_t B, int32_t K,
                        int64_t magic_draft_id, int32_t* num_accepted, int64_t* next_tokens, void* stream) {
  g_err[0] = 0;
  if (B < 0 || K < 0) return fail(MTPSD_EINVAL, "accept_greedy: need B >= 0, K >= 0");
  if (B == 0) return MTPSD_OK;
  if ((K > 0 && !draft) || !target_argmax || !num_accepted || !next_tokens)
    return fail(MTPSD_EINVAL, "accept_greedy: null pointer");
  return launch_accept_greedy(draft, target_argmax, B, K, magic_draft_id, num_accepted, next_tokens,
                              (cudaStream_t)stream);
}

int mtpsd_accept_stochastic(const int64_t* draft, const float* draft_probs, const float* target_probs,
                            const float* u_accept, const float* u_sample, int32_t B, int32_t K, int64_t V,
                            int32_t* num_accepted, int64_t* next_tokens, int32_t* dev_status, void* stream) {
  g_err[0] = 0;
  if (B < 0 || K < 0 || V < 1 || V > 0x7fffffffLL) return fail(MTPSD_EINVAL, "accept_stochastic: need B >= 0, K >= 0, 1 <= V < 2^31");
  if (B == 0) return MTPSD_OK;
  if ((K > 0 && (!draft || !draft_probs || !u_accept)) || !target_probs || !u_sample || !num_accepted || !next_tokens)
    return fail(MTPSD_EINVAL, "accept_stochastic: null pointer");
  return launch_accept_stochastic(draft, draft_probs, target_probs, u_accept, u_sample, B, K, V, num_accepted,
                                  next_tokens, dev_status, (cudaStream_t)stream);
}

int mtpsd_kv_writeback(const void* src_latent, const uint8_t* src_idxk, const float* src_idxs, int32_t B, int32_t W,
                       int32_t latent_dtype, int32_t idx_dim, const int32_t* num_accepted, void* dst_latent,
                       uint8_t* dst_idxk, float* dst_idxs, const int64_t* cache_start, const int64_t* dst_pos, int64_t pool_tokens,
                       int64_t* next_pos, int32_t* dev_status, void* stream) {
  g_err[0] = 0;
  if (B < 0 || W < 1 || pool_tokens < 0 || B > 65535) return fail(MTPSD_EINVAL, "kv_writeback: need 0 <= B <= 65535, W >= 1");
  int lat_bytes;
  if (latent_dtype == MTPSD_BF16) lat_bytes = 576 * 2;
  else if (latent_dtype == MTPSD_F32) lat_bytes = 576 * 4;
  else if (latent_dtype == MTPSD_FP8_DS_MLA) lat_bytes = 656;
  else return fail(MTPSD_EUNSUPPORTED, "kv_writeback: latent dtype must be MTPSD_BF16, MTPSD_F32 or MTPSD_FP8_DS_MLA");
  if (idx_dim != 0 && idx_dim % 16) return fail(MTPSD_EUNSUPPORTED, "kv_writeback: idx_dim must be a multiple of 16");
  if (B == 0) return MTPSD_OK;
  if (!src_latent || !dst_latent || !num_accepted || !cache_start || !dst_pos) return fail(MTPSD_EINVAL, "kv_writeback: null pointer");
  if (idx_dim && (!src_idxk || !dst_idxk)) return fail(MTPSD_EINVAL, "kv_writeback: null indexer key pointer");
  if ((src_idxs == nullptr) != (dst_idxs == nullptr)) return fail(MTPSD_EINVAL, "kv_writeback: give both key scale pointers or neither");
  if (!aligned(src_latent, 16) || !aligned(dst_latent, 16) || (idx_dim && (!aligned(src_idxk, 16) || !aligned(dst_idxk, 16))))
    return fail(MTPSD_EINVAL, "kv_writeback: latent and key buffers must be 16-byte aligned");
  return launch_kv_writeback(src_latent, src_idxk, src_idxs, B, W, lat_bytes, idx_dim, num_accepted, dst_latent,
                             dst_idxk, dst_idxs, cache_start, dst_pos, pool_tokens, next_pos, dev_status, (cudaStream_t)stream);
}

int mtpsd_kv_writeback_slots(const void* src_latent, const uint8_t* src_idxk, const float* src_idxs, int32_t B, int32_t W,
                             int32_t latent_dtype, int32_t idx_dim, const int32_t* num_accepted, void* dst_latent,
                             uint8_t* dst_idxk, float* dst_idxs, const int64_t* dst_slots, int64_t pool_tokens,
                             const int64_t* dst_pos, int64_t* next_pos, int32_t* dev_status, void* stream) {
  g_err[0] = 0;
  if (B < 0 || W < 1 || pool_tokens < 0 || B > 65535) return fail(MTPSD_EINVAL, "kv_writeback_slots: need 0 <= B <= 65535, W >= 1");
  int lat_bytes;
  if (latent_dtype == MTPSD_BF16) lat_bytes = 576 * 2;
  else if (latent_dtype == MTPSD_F32) lat_bytes = 576 * 4;
  else if (latent_dtype == MTPSD_FP8_DS_MLA) lat_bytes = 656;
  else return fail(MTPSD_EUNSUPPORTED, "kv_writeback_slots: latent dtype must be MTPSD_BF16, MTPSD_F32 or MTPSD_FP8_DS_MLA");
  if (idx_dim != 0 && idx_dim % 16) return fail(MTPSD_EUNSUPPORTED, "kv_writeback_slots: idx_dim must be a multiple of 16");
  if (B == 0) return MTPSD_OK;
  if (!src_latent || !dst_latent || !num_accepted || !dst_slots) return fail(MTPSD_EINVAL, "kv_writeback_slots: null pointer");
  if ((dst_pos == nullptr) != (next_pos == nullptr)) return fail(MTPSD_EINVAL, "kv_writeback_slots: give dst_pos and next_pos together or neither");
  if (idx_dim && (!src_idxk || !dst_idxk)) return fail(MTPSD_EINVAL, "kv_writeback_slots: null indexer key pointer");
  if ((src_idxs == nullptr) != (dst_idxs == nullptr)) return fail(MTPSD_EINVAL, "kv_writeback_slots: give both key scale pointers or neither");
  if (!aligned(src_latent, 16) || !aligned(dst_latent, 16) || (idx_dim && (!aligned(src_idxk, 16) || !aligned(dst_idxk, 16))))
    return fail(MTPSD_EINVAL, "kv_writeback_slots: latent and key buffers must be 16-byte aligned");
  return launch_kv_writeback(src_latent, src_idxk, src_idxs, B, W, lat_bytes, idx_dim, num_accepted, dst_latent,
                             dst_idxk, dst_idxs, nullptr, dst_pos, pool_tokens, next_pos, dev_status, (cudaStream_t)stream,
                             dst_slots);
}

int mtpsd_assign_cache_locs(const mtpsd_paged_kv* paged, int32_t B, const int64_t* start_pos, int32_t W,
                            int64_t* out_cache_loc, int32_t* dev_status, void* stream) {
  g_err[0] = 0;
  if (!paged) return fail(MTPSD_EINVAL, "assign_cache_locs: paged descriptor required");
  Paging pg;
  if (int rc = check_paged(paged, &pg, "assign_cache_locs")) return rc;
  if (B < 0 || W < 1) return fail(MTPSD_EINVAL, "assign_cache_locs: need B >= 0, W >= 1");
  if ((int64_t)B * W > 0x7fffffffLL) return fail(MTPSD_EINVAL, "assign_cache_locs: B*W too large");
  if (B == 0) return MTPSD_OK;
  if (!start_pos || !out_cache_loc) return fail(MTPSD_EINVAL, "assign_cache_locs: null pointer");
  return launch_assign_cache_locs(pg, B, start_pos, W, out_cache_loc, dev_status, (cudaStream_t)stream);
}

int mtpsd_kv_move_accepted(void* latent, int32_t latent_dtype, uint8_t* idxk, int32_t idx_dim, float* idxs,
                           int64_t pool_tokens, const int64_t* out_cache_loc, const int32_t* accept_index,
                           const int32_t* num_accepted, int32_t B, int32_t W, int32_t* dev_status, void* stream) {
  g_err[0] = 0;
  if (B < 0 || W < 1 || W > 16 || pool_tokens < 0) return fail(MTPSD_EINVAL, "kv_move_accepted: need B >= 0, 1 <= W <= 16");
  int lat_bytes;
  if (latent_dtype == MTPSD_BF16) lat_bytes = 576 * 2;
  else if (latent_dtype == MTPSD_F32) lat_bytes = 576 * 4;
  else if (latent_dtype == MTPSD_FP8_DS_MLA) lat_bytes = 656;
  else return fail(MTPSD_EUNSUPPORTED, "kv_move_accepted: latent dtype must be MTPSD_BF16, MTPSD_F32 or MTPSD_FP8_DS_MLA");
  if (idx_dim < 0 || idx_dim > 512 || idx_dim % 16) return fail(MTPSD_EUNSUPPORTED, "kv_move_accepted: idx_dim must be a multiple of 16 up to 512");
  if (B == 0) return MTPSD_OK;
  if (!latent || !out_cache_loc || !accept_index || !num_accepted || (idx_dim && !idxk))
    return fail(MTPSD_EINVAL, "kv_move_accepted: null pointer");
  if (!aligned(latent, 16) || (idx_dim && !aligned(idxk, 16)))
    return fail(MTPSD_EINVAL, "kv_move_accepted: latent and key buffers must be 16-byte aligned");
  return launch_kv_move(latent, lat_bytes, idxk, idx_dim, idxs, pool_tokens, out_cache_loc, accept_index, num_accepted, B, W,
                        dev_status, (cudaStream_t)stream);
}

int mtpsd_topk_share_gather(const int32_t* step0_topk, const uint32_t* row_offsets, const int32_t* num_accepted,
                            int32_t B, int32_t k, int32_t* shared_idx, const int64_t* row_pos, int64_t* shared_pos,
                            int32_t* dev_status, void* stream) {
  g_err[0] = 0;
  if (B < 0 || k < 1) return fail(MTPSD_EINVAL, "topk_share_gather: need B >= 0, k >= 1");
  if (B == 0) return MTPSD_OK;
  if (!step0_topk || !row_offsets || !shared_idx) return fail(MTPSD_EINVAL, "topk_share_gather: null pointer");
  if ((row_pos == nullptr) != (shared_pos == nullptr))
    return fail(MTPSD_EINVAL, "topk_share_gather: give row_pos and shared_pos together or neither");
  if ((k & 3) == 0 && (!aligned(step0_topk, 16) || !aligned(shared_idx, 16)))
    return fail(MTPSD_EINVAL, "topk_share_gather: buffers must be 16-byte aligned when k % 4 == 0");
  return launch_share_gather(step0_topk, row_offsets, num_accepted, B, k, shared_idx, row_pos, shared_pos, dev_status,
                             (cudaStream_t)stream);
}

int mtpsd_check_bounded_wait(int64_t limit_ns, int32_t* dev_status, int64_t* result, void* stream) {
  g_err[0] = 0;
  if (limit_ns < 1 || limit_ns > 1000000000LL) return fail(MTPSD_EINVAL, "check_bounded_wait: limit_ns must be 1..1e9");
  if (!dev_status || !result) return fail(MTPSD_EINVAL, "check_bounded_wait: null pointer");
  if (!aligned(result, 8)) return fail(MTPSD_EINVAL, "check_bounded_wait: result must be 8-byte aligned");
  return launch_bounded_wait_check(limit_ns, dev_status, result, (cudaStream_t)stream);
}

}  // extern "C"
