/*
 * mtpsd — decode-time DSA sparse attention for MTP speculative decoding on
 * one NVIDIA GB300 (sm_103a).  C ABI of libmtpsd.so.
 *
 * Source pages cited below (title, section):
 *   [P1] "MAX 中 GLM-5.2 (DeepSeek-V3.2 Sparse) 的统一 MTP 推测解码架构解析"
 *   [P2] "GLM-5.3 推理全链路(十四):MTP 的三段前向——草稿、验证与 draft_extend 的算子与通信账"
 *   [P3] "MAX Pipeline 中的 DeepSeek-V3.2 架构实现解析:稀疏注意力、Lightning Indexer 与 MoE 并行推理"
 *   [P4] "MAX 推测解码配置指南:解读 max.pipelines.speculative 模块"
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer argument is a DEVICE pointer owned by the caller, unless the
 *   comment says "host".  The library never allocates device memory and never
 *   frees caller memory; scratch space is a caller-provided workspace whose
 *   size the matching *_workspace_size() query returns.
 * - Every call that takes a stream is asynchronous on that stream (a
 *   cudaStream_t passed as void*; NULL = the legacy default stream), makes no
 *   host<->device copy and does not synchronize.
 * - Return value: MTPSD_OK (0) or a negative MTPSD_E* code.  Argument and
 *   shape checks run on the host before any launch; on failure nothing is
 *   launched and mtpsd_last_error() describes the problem (thread-local).
 * - Device-side range violations (an index outside the visible context, a
 *   write outside the pool) skip the offending element and OR a MTPSD_STATUS_*
 *   bit into *dev_status (an int32 the caller zeroes; NULL = not reported).
 *   Kernels never trap.  Every device-side wait is bounded: on expiry the
 *   kernel ORs MTPSD_STATUS_WAIT_TIMEOUT, releases what it holds and returns.
 * - Cache layout: a flat pool of tokens; request b owns the contiguous pool
 *   rows starting at cache_start[b] (int64); position s of request b is pool
 *   row cache_start[b] + s.
 * - Query rows are grouped by request: the rows of request b are
 *   row_offsets[b] .. row_offsets[b+1]-1 (uint32 [B+1], exclusive prefix sum,
 *   the same convention as merged_offsets of mtpsd_merge_tokens).  Row r sits
 *   at position row_pos[r] of its request and sees positions 0..row_pos[r]
 *   (chain causal mask, [P2] "验证输入是怎么拼出来的"; the row's own key is
 *   already in the cache, [P2] "验证段的逐层算子" op 3).
 */
#ifndef MTPSD_H
#define MTPSD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* return codes */
#define MTPSD_OK 0
#define MTPSD_EINVAL (-1)        /* bad argument, shape or alignment */
#define MTPSD_EUNSUPPORTED (-2)  /* valid but not implemented (dtype, head dim) */
#define MTPSD_ECUDA (-3)         /* a CUDA runtime call or launch failed */
#define MTPSD_EWORKSPACE (-4)    /* workspace missing or too small */

/* element types */
#define MTPSD_F32 0
#define MTPSD_BF16 1
#define MTPSD_FP8_E4M3 2
#define MTPSD_FP8_DS_MLA 3  /* latent cache rows of 656 bytes: 512 E4M3 codes (four blocks of 128), the four
                               float32 block scales, the 64 rope values as bf16 ([P2] "草稿层 KV 的账") */

/* bits ORed into *dev_status */
#define MTPSD_STATUS_INDEX_RANGE 1   /* a selected index outside 0..row_pos (skipped) */
#define MTPSD_STATUS_WRITE_RANGE 2   /* a write-back row outside the pool (skipped) */
#define MTPSD_STATUS_WAIT_TIMEOUT 4  /* a bounded device wait expired (kernel gave up) */
#define MTPSD_STATUS_ROW_RANGE 8     /* a row position outside its request's pool rows (skipped) */

/* ------------------------------------------------------------------------
 * Ragged token merge.  [P4] "Token 合并:RaggedTokenMerger 与 ragged_token_merger"
 * and [P1] "阶段 1:Token 合并".
 *   prompt_tokens  [S] int64        prompt_offsets [B+1] uint32 (exclusive prefix sum)
 *   draft_tokens   [B, K] int64     (row-major; K may be 0)
 *   merged_tokens  [S + B*K] int64  merged_offsets [B+1] uint32
 * merged_offsets[i] = prompt_offsets[i] + i*K; request b's merged segment is
 * its prompt tokens followed by its K drafts.  S is the host-known total
 * (= prompt_offsets[B]).  B >= 1, K >= 0.
 */
int mtpsd_merge_tokens(const int64_t* prompt_tokens, int64_t S, const uint32_t* prompt_offsets,
                       const int64_t* draft_tokens, int32_t B, int32_t K,
                       int64_t* merged_tokens, uint32_t* merged_offsets, void* stream);

/* Host mirror of the merged offsets, so a caller building a CUDA graph needs
 * no device->host copy ([P4], compute_host_merged_offsets).  All host pointers:
 * prompt_offsets [B+1], out [B+1]. */
void mtpsd_host_merged_offsets(const uint32_t* prompt_offsets, int32_t B, int32_t K, uint32_t* out);

/* Cross-layer indexer schedule ([P3] "跨层共享的 indexer 调度"), host only: is_full[i] = 1 when
 * layer i runs its own indexer (full), 0 when it reuses the selection of the most recent full layer
 * (shared).  From pattern (a string of F and S, one per layer) when given and non-empty; else, when
 * freq > 0 or offset >= 0, layer i is full when max(i - offset + 1, 0) % freq == 0 (freq 1 and offset
 * 2 by default: pass freq 0 or offset -1 to take a default); else every layer is full.  The first
 * layer must be full (MTPSD_EINVAL otherwise).  GLM-5.x's 21 full of 78 layers ([P2] "验证段的逐层算子")
 * is freq 4, offset 2.  An explicit per-layer list needs no call. */
int mtpsd_resolve_indexer_types(int32_t n_layers, const char* pattern, int32_t freq, int32_t offset,
                                int32_t* is_full);

/* ------------------------------------------------------------------------
 * Dynamic FP8 E4M3 quantization with one float32 scale per block of 128
 * contiguous values.  [P3] "Indexer 的结构与计算流程" (q and k quantized to FP8
 * with block size 128) and "双 KV 缓存" (float32 scale per token).
 *   x [n_blocks*128] float32 -> codes [n_blocks*128] uint8, scales [n_blocks] float32
 * scale = amax/448 (1 when amax == 0), code = round-to-nearest-even,
 * saturating, of x/scale (float32 division).
 */
int mtpsd_quantize_fp8_block128(const float* x, int64_t n_blocks, uint8_t* codes, float* scales,
                                void* stream);

/* ------------------------------------------------------------------------
 * FP8 latent cache rows.  [P2] "草稿层 KV 的账" (656 bytes per token per layer, the
 * fp8_ds_mla layout): latent [T, 576] (MTPSD_BF16 or MTPSD_F32) -> packed
 * [T, 656] uint8: bytes 0..511 the E4M3 codes of values 0..511 in four blocks of
 * 128 (the block-128 quantizer above), bytes 512..527 the four float32 scales,
 * bytes 528..655 the 64 rope values 512..575 as bf16 (round to nearest even).
 * latent 16-byte aligned; packed 16-byte aligned.
 */
int mtpsd_pack_latent_fp8(const void* latent, int32_t dtype, int64_t T, uint8_t* packed, void* stream);

/* ------------------------------------------------------------------------
 * Lightning-indexer scores and per-row top-k in one call.
 * [P3] "Indexer 的结构与计算流程" (index heads, weights_proj, FP8 block-128,
 * the fused mla_fp8_index_top_k output of shape (total_seq_len, index_topk));
 * [P2] "验证段的逐层算子" ops 5-6 (every verify query scores the history and
 * picks its own 2048).  Score of row r at position s (0 <= s <= row_pos[r]):
 *   I[r,s] = sum_h w[r,h] * ReLU( q_scale[r,h] * k_scale[s] * sum_d q[r,h,d]*k[s,d] )
 * (float32 configuration: the scales are 1).  topk_idx[r, :] holds the
 * positions of the topk largest I[r, .] (ties to the lower position), in
 * ascending position order, padded with -1 when row_pos[r]+1 < topk.
 */
typedef struct {
  int32_t B;               /* requests */
  int32_t R;               /* query rows, = row_offsets[B] */
  int32_t n_heads;         /* indexer heads H (64 in the FP8 production shape) */
  int32_t head_dim;        /* D: 128 for MTPSD_FP8_E4M3 (one scale per head vector); any multiple of 4 up to 256 for MTPSD_F32 */
  int32_t topk;            /* k, 1..4096 */
  int32_t dtype;           /* MTPSD_FP8_E4M3 or MTPSD_F32 (q, k_cache) */
  const void* q;           /* [R, H, D] uint8 codes or float32 */
  const float* q_scale;    /* [R, H] (FP8 only, else NULL) */
  const float* weights;    /* [R, H] per-head weights (weights_proj output) */
  const void* k_cache;     /* [pool_tokens, D] uint8 codes or float32 */
  const float* k_scale;    /* [pool_tokens] (FP8 only, else NULL) */
  int64_t pool_tokens;
  const int64_t* cache_start; /* [B] */
  const uint32_t* row_offsets; /* [B+1] */
  const int64_t* row_pos;  /* [R] */
  int64_t max_visible;     /* host-known bound >= row_pos[r]+1 for every r; sizes the score buffer */
  int32_t* topk_idx;       /* [R, topk] out */
  float* topk_score;       /* [R, topk] out, nullable (score of each selected position, -inf on padding) */
  float* scores;           /* [R, ld] out, nullable: the raw scores, ld = mtpsd_scores_ld(max_visible) */
  void* workspace;
  size_t workspace_bytes;
  int32_t* dev_status;     /* nullable */
} mtpsd_indexer_args;

/* Row stride (floats) of the score matrix for a given max_visible. */
int64_t mtpsd_scores_ld(int64_t max_visible);
/* Workspace bytes of mtpsd_indexer_topk: the score matrix (R x mtpsd_scores_ld(max_visible) floats,
 * 256-byte padded), the work plan (mtpsd_indexer_topk_plan_bytes) and, when max_visible exceeds
 * 40960, the top-k candidate lists (mtpsd_topk_workspace_size, 256-byte padded).  When args->scores
 * is given (16-byte aligned) the scores go there and the workspace needs only
 * mtpsd_indexer_topk_aux_bytes(B, R, max_visible, topk) = plan + candidate lists. */
size_t mtpsd_indexer_topk_workspace_size(int32_t B, int32_t R, int64_t max_visible, int32_t topk);
size_t mtpsd_indexer_topk_plan_bytes(int32_t B, int32_t R);
size_t mtpsd_indexer_topk_aux_bytes(int32_t B, int32_t R, int64_t max_visible, int32_t topk);
int mtpsd_indexer_topk(const mtpsd_indexer_args* args, void* stream);
/* Kernel launches one mtpsd_indexer_topk call with R > 0 makes on the current device: the score
 * launches (2 on the tensor-core path: group plan and FP8 score GEMM, which needs MTPSD_FP8_E4M3,
 * head_dim 128, 32 or 64 heads and 16-byte aligned q and k_cache, as this count assumes; else 1) plus
 * those of the top-k (mtpsd_topk_launch_count(max_visible, topk)). */
int32_t mtpsd_indexer_topk_launch_count(int32_t n_heads, int32_t head_dim, int32_t dtype, int64_t max_visible,
                                        int32_t topk);

/* The scoring half of mtpsd_indexer_topk, for callers that select (or time the
 * selection) themselves: writes the score matrix args->scores [R, ld] (ld =
 * mtpsd_scores_ld(max_visible); row r holds positions 0..row_pos[r], the rest of
 * the row is not written) and launches nothing else.  args->scores is required
 * (16-byte aligned); topk, topk_idx and topk_score are ignored; the workspace
 * needs mtpsd_indexer_topk_plan_bytes(B, R).  mtpsd_topk over the result with
 * row_len[r] = row_pos[r] + 1 gives exactly what mtpsd_indexer_topk returns. */
int mtpsd_indexer_scores(const mtpsd_indexer_args* args, void* stream);
/* Kernel launches of one mtpsd_indexer_scores call with R > 0 (2 on the tensor-core path, else 1). */
int32_t mtpsd_indexer_scores_launch_count(int32_t n_heads, int32_t head_dim, int32_t dtype);

/* ------------------------------------------------------------------------
 * Allocation-free variant of mtpsd_indexer_topk (the source pages have no
 * counterpart: this is a deployment convenience of this library).
 *
 * For callers that cannot allocate device memory: a plugin or C host whose
 * allocator owns the device memory and hands out no scratch, a serving loop
 * that forbids allocation after start-up, or a caller holding only the raw
 * input/output pointers.  Same arguments and results as mtpsd_indexer_topk,
 * but args->workspace and args->workspace_bytes are ignored: the score
 * scratch lives in a static device array of MTPSD_NOALLOC_SCRATCH_BYTES
 * inside the library, which every GPU that loads the library holds until the
 * process exits.  The caller still passes every input and output.
 * - A call needing more than MTPSD_NOALLOC_SCRATCH_BYTES of scratch
 *   (mtpsd_indexer_topk_workspace_size(B, R, max_visible, topk), about
 *   R * max_visible * 4 bytes; only mtpsd_indexer_topk_aux_bytes(...) when
 *   args->scores is given, since the scores then go to the caller's buffer)
 *   returns MTPSD_EWORKSPACE before any launch.
 * - The first call on a device (the current device) looks up the array's
 *   device address; make that first call before any stream capture.
 * - All calls share the one array, which keeps the last call's contents
 *   (nothing in it needs to start at zero).  Calls that overlap on the GPU
 *   (on different streams without ordering) race on it.
 * - Calls no cudaMalloc / cudaFree or other allocating routine.
 */
#define MTPSD_NOALLOC_SCRATCH_BYTES (16u << 20) /* 16 MiB */
int mtpsd_indexer_topk_noalloc(const mtpsd_indexer_args* args, void* stream);

/* ------------------------------------------------------------------------
 * Standalone per-row top-k over a score matrix (the selection half of the
 * call above, for callers that produce scores themselves).
 *   scores [R, ld] float32, row_len [R] int64: row r's valid prefix has
 *   row_len[r] + row_len_add scores (pass row_pos with row_len_add = 1 for the
 *   indexer's visible lengths), clamped to max_len (flagged
 *   MTPSD_STATUS_INDEX_RANGE when a length exceeds it)
 *   -> out_idx [R, topk] (ascending positions, -1 padded), out_score nullable.
 * Rows of up to 40960 keys take one CTA each (16-byte aligned rows, ld % 4 == 0).
 * Longer rows are split: one CTA per 16384-key segment selects that segment's
 * exact top-k, and merge levels over groups of 16384/topk such lists follow
 * (one launch per level, mtpsd_topk_launch_count); their candidate lists live
 * in the workspace (mtpsd_topk_workspace_size, 256-byte aligned; 0 bytes when
 * max_len <= 40960).  Unaligned score rows take a one-CTA-per-row radix kernel.
 * NaN scores are not supported.
 */
size_t mtpsd_topk_workspace_size(int32_t R, int64_t max_len, int32_t topk);
int32_t mtpsd_topk_launch_count(int64_t max_len, int32_t topk);
int mtpsd_topk(const float* scores, int64_t ld, int32_t R, const int64_t* row_len, int64_t row_len_add,
               int64_t max_len, int32_t topk, int32_t* out_idx, float* out_score, void* workspace,
               size_t workspace_bytes, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * Sparse MLA decode over the selected latent rows.
 * [P2] "GLM-5.3 的草稿层到底长什么样" (kv_lora_rank 512 + qk_rope 64 = 576),
 * "验证段的逐层算子" op 7; [P3] "稀疏 MLA 的前向路径".  With the absorbed query
 * the key of position s is latent[s, 0:576] and its value latent[s, 0:512]:
 *   o[r,h]   = sum_j softmax_j(scale * q[r,h,:].latent[s_j,:]) * latent[s_j, 0:512]
 *   lse[r,h] = log sum_j exp(scale * q[r,h,:].latent[s_j,:])     (natural log)
 * over the valid positions s_j of idx[r, 0:n_idx] (-1 = padding, skipped) and,
 * when n_append > 0, the appended positions append_base[r]+1 .. append_base[r]+n_append
 * ([P1] "阶段 5:Draft 后续步骤(复用 top-k)": the MLA cache grows by one per draft
 * step while the shared indexer selection stays fixed).  Every position must
 * satisfy 0 <= s <= row_pos[r] + row_pos_add; others are skipped and flagged.
 * A row with no valid position gets o = 0 and lse = -inf.
 */
typedef struct {
  int32_t B;
  int32_t R;
  int32_t n_heads;         /* query heads H: a multiple of 16 for MTPSD_BF16, any for MTPSD_F32 */
  int32_t d_latent;        /* 576 */
  int32_t d_v;             /* 512 */
  int32_t n_idx;           /* selected entries per row (row stride of idx) */
  int32_t n_append;        /* appended positions per row (0 = none) */
  int32_t dtype;           /* MTPSD_BF16 or MTPSD_F32: q, latent and out; MTPSD_FP8_DS_MLA: bf16 q and out,
                              latent rows of 656 bytes (the FP8 cache; dequantized tile by tile in shared memory) */
  float softmax_scale;
  int64_t row_pos_add;     /* added to row_pos[r] (draft step j of a shared loop passes j) */
  const void* q;           /* [R, H, d_latent] */
  const void* latent;      /* [pool_tokens, d_latent] */
  int64_t pool_tokens;
  const int64_t* cache_start;  /* [B] */
  const uint32_t* row_offsets; /* [B+1] */
  const int64_t* row_pos;      /* [R] */
  const int32_t* idx;          /* [R, n_idx] */
  const int64_t* append_base;  /* [R] or NULL when n_append == 0 */
  void* out;                   /* [R, H, d_v] */
  float* lse;                  /* [R, H] nullable */
  void* workspace;
  size_t workspace_bytes;
  int32_t* dev_status;         /* nullable */
} mtpsd_mla_args;

size_t mtpsd_sparse_mla_workspace_size(int32_t R, int32_t n_heads, int32_t n_idx, int32_t n_append,
                                       int32_t dtype);
/* Kernel launches one mtpsd_sparse_mla_decode call with these sizes makes on the current device: 1, or 2
 * when the selected list is split and the split partials are merged by a second kernel (they are merged
 * inside the first when the splits of a row fit one thread-block cluster).  With many rows of bf16
 * latent (where a measured cost model favours it; environment MTPSD_MLA_PERSIST=0 turns it off, =1
 * forces it) the tensor-core kernel runs persistently, one cluster per pair of SMs, each taking an equal
 * run of 64-position pairs across rows; a row cut between two clusters leaves float32 pieces in the
 * workspace that a second kernel merges.  The count assumes the tensor-core kernel, which needs q,
 * latent, out and workspace 16-byte aligned (TMA loads and stores); other calls run the portable
 * kernel.  0 for sizes that launch nothing.  The workspace size covers every plan. */
int32_t mtpsd_sparse_mla_launch_count(int32_t R, int32_t n_heads, int32_t n_idx, int32_t n_append, int32_t dtype);
int mtpsd_sparse_mla_decode(const mtpsd_mla_args* args, void* stream);

/* ------------------------------------------------------------------------
 * Greedy acceptance.  [P2] "接受判定:greedy 与 rejection sampling" (accept
 * while draft == target argmax, stop at the first mismatch); [P1] "阶段 3:拒绝
 * 采样与 Bitmask" (outputs num_accepted and next_tokens); [P4] MAGIC_DRAFT_TOKEN_ID.
 *   draft [B, K] int64, target_argmax [B, K+1] int64
 *   -> num_accepted [B] int32 (n_b), next_tokens [B] int64 (= target_argmax[b, n_b])
 * magic_draft_id >= 0: a draft row made entirely of that id accepts 0
 * (42 is the pages' sentinel); -1 disables the check.
 */
int mtpsd_accept_greedy(const int64_t* draft, const int64_t* target_argmax, int32_t B, int32_t K,
                        int64_t magic_draft_id, int32_t* num_accepted, int64_t* next_tokens,
                        void* stream);

/* ------------------------------------------------------------------------
 * Rejection-sampling acceptance.  [P2] "接受判定:greedy 与 rejection sampling":
 * draft i is accepted with probability min(1, p/q) (q the draft distribution,
 * p the target distribution of verify row i); the first rejected position
 * draws its token from the corrected distribution max(0, p - q) normalised
 * (the standard speculative-sampling correction; p itself if that has no
 * mass); after K accepted drafts the next token is drawn from p of row K.
 *   draft [B, K] int64, draft_probs q [B, K, V] float32,
 *   target_probs p [B, K+1, V] float32 (probabilities in [0, 1]),
 *   u_accept [B, K], u_sample [B] float32 uniforms in [0, 1) (the caller draws them)
 *   -> num_accepted [B] int32 (n_b), next_tokens [B] int64.
 * Draft i is accepted when u_accept[b,i] * q[b,i,d] < p[b,i,d] (single
 * precision product); a draft id outside [0, V) is rejected and flagged
 * MTPSD_STATUS_INDEX_RANGE.  The draw is an exact inverse CDF on fixed-point
 * weights floor(max(w, 0) * 2^32): the smallest token whose running sum
 * exceeds floor(u_sample * total), with exact integer sums (a row with no
 * mass at all gives token 0).  Reads two rows of V per request beyond the K
 * gathered entries.
 */
int mtpsd_accept_stochastic(const int64_t* draft, const float* draft_probs, const float* target_probs,
                            const float* u_accept, const float* u_sample, int32_t B, int32_t K, int64_t V,
                            int32_t* num_accepted, int64_t* next_tokens, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * Accepted-segment KV write-back.  [P2] "KV 交账:接受段的搬移与拒绝段的回收"
 * and "draft_extend:把接受段写回草稿层" / "草稿层 KV 的账": only the accepted
 * rows (bonus included: num_accepted[b]+1 rows, at least 1, at most W) of the
 * W-row window are copied, byte for byte, to positions dst_pos[b] + i of
 * request b (pool rows cache_start[b] + dst_pos[b] + i); rejected rows are not
 * written.  Both caches of the layer move together.
 *   src_latent [B, W, 576] (latent_dtype: MTPSD_BF16 or MTPSD_F32), or [B, W, 656] packed
 *   bytes (MTPSD_FP8_DS_MLA)
 *   src_idxk [B, W, idx_dim] uint8, src_idxs [B, W] float32
 *   dst_latent [pool_tokens, 576], dst_idxk [pool_tokens, idx_dim], dst_idxs [pool_tokens]
 *   cache_start [B], dst_pos [B] int64
 *   next_pos [B] int64 out, nullable: dst_pos[b] + num_accepted[b] + 1, the
 *   position of the next draft row.
 * idx_dim is the key size in bytes per token (128 for FP8 keys, a multiple
 * of 16), or 0 to move the latent only (then src_idxk/dst_idxk may be NULL).
 * src_idxs/dst_idxs may both be NULL when the keys carry no scale (float32
 * keys).  A destination row outside the pool is skipped and flagged
 * MTPSD_STATUS_WRITE_RANGE.
 */
int mtpsd_kv_writeback(const void* src_latent, const uint8_t* src_idxk, const float* src_idxs,
                       int32_t B, int32_t W, int32_t latent_dtype, int32_t idx_dim,
                       const int32_t* num_accepted, void* dst_latent, uint8_t* dst_idxk,
                       float* dst_idxs, const int64_t* cache_start, const int64_t* dst_pos,
                       int64_t pool_tokens, int64_t* next_pos, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * Paged (slotted) KV caches.  [P2] "输入准备:prepare_for_draft": the caches
 * are pools of token slots and each request reaches its positions through a
 * token table (req_to_token; page_size > 1 groups consecutive slots into
 * pages).  Here a request's table is one row of a block table:
 *   block_table [B, bt_stride] int32 (device): page ids, -1 = no page;
 *   position s of request b lives in pool slot
 *     block_table[b, s / page_size] * page_size + s % page_size,
 *   and has no slot when s < 0, s / page_size >= bt_stride or the entry is
 *   negative.  page_size 1 is the token table itself.
 * The slots of different requests are disjoint (a slot belongs to one request).
 */
typedef struct {
  const int32_t* block_table;  /* [B, bt_stride] page ids (device) */
  int32_t bt_stride;           /* entries per request (>= 1) */
  int32_t page_size;           /* tokens per page: a power of two, 1 .. 65536 */
} mtpsd_paged_kv;

/* The window's slot plan (assign_draft_cache_locs in [P2] "输入准备:prepare_for_draft"):
 *   out_cache_loc[b, j] = slot of position start_pos[b] + j, j < W (int64 [B, W]), or -1
 *   when that position has no slot (flagged MTPSD_STATUS_ROW_RANGE).
 * start_pos [B] int64 (the committed length: the window follows it). */
int mtpsd_assign_cache_locs(const mtpsd_paged_kv* paged, int32_t B, const int64_t* start_pos, int32_t W,
                            int64_t* out_cache_loc, int32_t* dev_status, void* stream);

/* The accepted-KV move (move_kv_cache over fill_front_out_cache_loc /
 * fill_accept_out_cache_loc, [P2] "KV 交账:接受段的搬移与拒绝段的回收"):
 * for i < accept_len = num_accepted[b] + 1 (the bonus row included; clamped
 * to [0, W]), row i of request b moves from window slot
 * out_cache_loc[b, accept_index[b, i]] to the front slot out_cache_loc[b, i],
 * in every cache of the layer at once.  It is a move: each destination
 * receives what its source held before the call, whatever the overlap of the
 * two slot lists of a request (rows whose source is their destination are
 * left alone; a chain of drafts, accept_index[b, i] = i, moves nothing).
 *   latent [pool_tokens, 576] (latent_dtype MTPSD_BF16 / MTPSD_F32) or [pool_tokens, 656]
 *   bytes (MTPSD_FP8_DS_MLA); idxk [pool_tokens, idx_dim] uint8 (idx_dim a multiple of 16,
 *   0 = none, idxk may then be NULL); idxs [pool_tokens] float32 or NULL.
 *   out_cache_loc [B, W] int64, accept_index [B, W] int32 (window columns), num_accepted [B] int32.
 * A window column outside [0, W) is skipped and flagged MTPSD_STATUS_INDEX_RANGE; a slot
 * outside the pool is skipped and flagged MTPSD_STATUS_WRITE_RANGE.  W <= 16. */
int mtpsd_kv_move_accepted(void* latent, int32_t latent_dtype, uint8_t* idxk, int32_t idx_dim, float* idxs,
                           int64_t pool_tokens, const int64_t* out_cache_loc, const int32_t* accept_index,
                           const int32_t* num_accepted, int32_t B, int32_t W, int32_t* dev_status, void* stream);

/* mtpsd_kv_writeback by slot: the accepted rows (num_accepted[b] + 1, at
 * least 1, at most W) of request b's window go to pool slots
 * dst_slots[b, 0 ..] (int64 [B, W], the window slots planned by
 * mtpsd_assign_cache_locs: the token table is shared by the layers, each
 * layer has its own pools); rejected rows are not written.  dst_pos [B]
 * int64 and next_pos [B] int64 (both or neither, nullable): next_pos[b] =
 * dst_pos[b] + the rows written, the position of the next draft row when
 * dst_pos is the window's first position.  Other arguments as
 * mtpsd_kv_writeback; a slot outside the pool is skipped and flagged
 * MTPSD_STATUS_WRITE_RANGE. */
int mtpsd_kv_writeback_slots(const void* src_latent, const uint8_t* src_idxk, const float* src_idxs,
                             int32_t B, int32_t W, int32_t latent_dtype, int32_t idx_dim,
                             const int32_t* num_accepted, void* dst_latent, uint8_t* dst_idxk,
                             float* dst_idxs, const int64_t* dst_slots, int64_t pool_tokens,
                             const int64_t* dst_pos, int64_t* next_pos, int32_t* dev_status, void* stream);

/* mtpsd_indexer_topk, mtpsd_indexer_scores and mtpsd_sparse_mla_decode over
 * paged caches: position s of request b is read from the slot the block
 * table gives (args->cache_start is ignored and may be NULL); a visible
 * position without a slot reads as zero keys (score 0 x its scale: 0) in the
 * indexer and is skipped in the attention, both flagged
 * MTPSD_STATUS_ROW_RANGE.  Everything else is as the contiguous calls,
 * including workspaces and launch counts.  The tensor-core indexer reads
 * pages of at least 8 tokens (a 128-position key tile as page-sized TMA
 * boxes) when the pool is a whole number of pages; smaller pages take the
 * CUDA-core score kernel, one launch fewer than
 * mtpsd_indexer_topk_launch_count.  paged NULL = the contiguous call. */
int mtpsd_indexer_topk_paged(const mtpsd_indexer_args* args, const mtpsd_paged_kv* paged, void* stream);
int mtpsd_indexer_scores_paged(const mtpsd_indexer_args* args, const mtpsd_paged_kv* paged, void* stream);
int mtpsd_sparse_mla_decode_paged(const mtpsd_mla_args* args, const mtpsd_paged_kv* paged, void* stream);

/* ------------------------------------------------------------------------
 * index_share_for_mtp_iteration gather.  [P1] "阶段 5:Draft 后续步骤(复用
 * top-k)" (gather_accepted_hidden_states over step0_topk at num_accepted);
 * [P2] "索引器复用的收益与边界" (compact_topk_indices: one row per request).
 *   step0_topk [R0, k] int32, row_offsets [B+1] uint32 (rows of each request
 *   in the step-0 output), num_accepted [B] int32 or NULL (row 0 of each
 *   segment) -> shared_idx[b, :] = step0_topk[row_offsets[b] + num_accepted[b], :].
 * A local row outside the request's segment is clamped to its last row and
 * flagged MTPSD_STATUS_INDEX_RANGE.
 * row_pos [R0] int64 and shared_pos [B] int64 (both or neither, nullable):
 * shared_pos[b] = row_pos of the reused row (-1 for an empty segment), the
 * position whose selection is shared; a later step appends positions after it.
 * This serves seed_dsa_topk_from_draft_extend ([P2] "draft_extend:把接受段写回草稿层"):
 * the selection of the last accepted row of draft_extend seeds the next
 * round's draft steps.
 */
int mtpsd_topk_share_gather(const int32_t* step0_topk, const uint32_t* row_offsets,
                            const int32_t* num_accepted, int32_t B, int32_t k, int32_t* shared_idx,
                            const int64_t* row_pos, int64_t* shared_pos, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * Check of the device-side bounded wait (the source pages have no
 * counterpart: it makes the library's failure path testable without a fault).
 * Every tensor-core kernel waits on its mbarrier phases through one helper
 * that gives up after a limit (2 s in the kernels), flags
 * MTPSD_STATUS_WAIT_TIMEOUT, lets the kernel release what it holds and return.
 * This call launches one small kernel in which two warps wait, with that
 * helper (CTA-scope and cluster-scope acquire), on a barrier phase that
 * nothing completes, with the given limit (1 ns .. 1 s).  Afterwards
 * *dev_status has MTPSD_STATUS_WAIT_TIMEOUT set and result [4] int64 (device)
 * holds, per warp, the nanoseconds waited and 1 if the wait succeeded (0:
 * it gave up, as it must).  The device stays usable.
 */
int mtpsd_check_bounded_wait(int64_t limit_ns, int32_t* dev_status, int64_t* result, void* stream);

/* ------------------------------------------------------------------------ */
const char* mtpsd_last_error(void);
int32_t mtpsd_version(void); /* 100*major + minor */

#ifdef __cplusplus
}
#endif
#endif /* MTPSD_H */
