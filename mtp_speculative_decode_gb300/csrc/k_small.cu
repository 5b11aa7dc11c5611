// Small fused kernels of the MTP decode step: ragged merge, FP8 block-128
// quantization, greedy acceptance, accepted-segment KV write-back and the
// step-0 top-k share gather.  All are HBM/latency bound; each is one launch.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"
#include "mbar.cuh"

namespace mtpsd {

// ---------------------------------------------------------------------------
// Ragged merge ([P4] "Token 合并").  One thread per output token; the owning
// request is found by binary search on merged offsets po[b] + b*K.
__global__ void merge_tokens_kernel(const int64_t* __restrict__ prompt, const uint32_t* __restrict__ po,
                                    const int64_t* __restrict__ draft, int B, int K, int64_t total,
                                    int64_t* __restrict__ out, uint32_t* __restrict__ mo) {
  griddep_wait();                // the previous kernel's writes are visible from here on
  griddep_launch_dependents();
  int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t <= B && t < (int64_t)B + 1) mo[t] = po[t] + (uint32_t)(t * K);
  for (; t < total; t += (int64_t)gridDim.x * blockDim.x) {
    int lo = 0, hi = B;  // request b: po[b] + b*K <= t < po[b+1] + (b+1)*K
    while (hi - lo > 1) {
      int mid = (lo + hi) >> 1;
      if ((int64_t)po[mid] + (int64_t)mid * K <= t) lo = mid; else hi = mid;
    }
    int b = lo;
    int64_t start = (int64_t)po[b] + (int64_t)b * K;
    int64_t n = (int64_t)po[b + 1] - po[b];
    int64_t j = t - start;
    out[t] = (j < n) ? prompt[po[b] + j] : draft[(int64_t)b * K + (j - n)];
  }
}

int launch_merge_tokens(const int64_t* prompt, int64_t S, const uint32_t* po, const int64_t* draft,
                        int B, int K, int64_t* out, uint32_t* mo, cudaStream_t st) {
  int64_t total = S + (int64_t)B * K;
  int64_t work = total > B + 1 ? total : B + 1;
  int blocks = (int)((work + 255) / 256);
  if (blocks > 4 * num_sms()) blocks = 4 * num_sms();
  if (blocks < 1) blocks = 1;
  // the first B+1 threads also write merged offsets; make sure they exist
  if ((int64_t)blocks * 256 < B + 1) blocks = (int)((B + 1 + 255) / 256);
  launch_k(merge_tokens_kernel, blocks, 256, 0, st, prompt, po, draft, B, K, total, out, mo);
  return check_launch("merge_tokens");
}

// ---------------------------------------------------------------------------
// FP8 block-128 quantization ([P3] "Indexer 的结构与计算流程").  One warp per
// block of 128 floats (one float4 per lane): amax by shuffle, IEEE float32
// division for the scale and the scaled value, then a saturating RNE
// conversion to E4M3.
__global__ void quantize_fp8_kernel(const float4* __restrict__ x, int64_t n_blocks,
                                    uint32_t* __restrict__ codes, float* __restrict__ scales) {
  griddep_wait();                // the previous kernel's writes are visible from here on
  griddep_launch_dependents();
  int lane = threadIdx.x & 31;
  int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t blk = warp; blk < n_blocks; blk += nwarps) {
    float4 v = x[blk * 32 + lane];
    float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float scale = m > 0.f ? __fdiv_rn(m, 448.0f) : 1.0f;
    uint32_t c0 = __nv_cvt_float_to_fp8(__fdiv_rn(v.x, scale), __NV_SATFINITE, __NV_E4M3);
    uint32_t c1 = __nv_cvt_float_to_fp8(__fdiv_rn(v.y, scale), __NV_SATFINITE, __NV_E4M3);
    uint32_t c2 = __nv_cvt_float_to_fp8(__fdiv_rn(v.z, scale), __NV_SATFINITE, __NV_E4M3);
    uint32_t c3 = __nv_cvt_float_to_fp8(__fdiv_rn(v.w, scale), __NV_SATFINITE, __NV_E4M3);
    codes[blk * 32 + lane] = c0 | (c1 << 8) | (c2 << 16) | (c3 << 24);
    if (lane == 0) scales[blk] = scale;
  }
}

int launch_quantize_fp8(const float* x, int64_t n_blocks, uint8_t* codes, float* scales, cudaStream_t st) {
  if (n_blocks == 0) return MTPSD_OK;
  int64_t warps = n_blocks;
  int64_t blocks = (warps * 32 + 255) / 256;
  if (blocks > 16 * num_sms()) blocks = 16 * num_sms();
  launch_k(quantize_fp8_kernel, (int)blocks, 256, 0, st, (const float4*)x, n_blocks, (uint32_t*)codes, scales);
  return check_launch("quantize_fp8_block128");
}

// ---------------------------------------------------------------------------
// FP8 latent cache rows ([P2] "草稿层 KV 的账": 656 bytes per token).  One warp
// per token: the 512 latent values in four blocks of 128, each quantized like
// the indexer keys (amax/448 scale, IEEE division, saturating RNE E4M3), the
// four float32 scales, then the 64 rope values as bf16.
template <bool F32IN>
__global__ void pack_latent_fp8_kernel(const void* __restrict__ latent, int64_t T, uint8_t* __restrict__ out) {
  griddep_wait();                // the previous kernel's writes are visible from here on
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t t = warp; t < T; t += nwarps) {
    uint8_t* o = out + t * 656;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float v[4];
      if constexpr (F32IN) {
        const float4 f = *(const float4*)((const float*)latent + t * 576 + 128 * k + 4 * lane);
        v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
      } else {
        const uint2 u = *(const uint2*)((const __nv_bfloat16*)latent + t * 576 + 128 * k + 4 * lane);
        v[0] = __uint_as_float(u.x << 16); v[1] = __uint_as_float(u.x & 0xffff0000u);
        v[2] = __uint_as_float(u.y << 16); v[3] = __uint_as_float(u.y & 0xffff0000u);
      }
      float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
      for (int sh = 16; sh; sh >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, sh));
      const float scale = m > 0.f ? __fdiv_rn(m, 448.0f) : 1.0f;
      uint32_t c = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        c |= (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(v[e], scale), __NV_SATFINITE, __NV_E4M3) << (8 * e);
      *(uint32_t*)(o + 128 * k + 4 * lane) = c;
      if (lane == 0) *(float*)(o + 512 + 4 * k) = scale;
    }
    uint32_t r;   // rope values 2 lane, 2 lane + 1 as bf16
    if constexpr (F32IN) {
      const float2 f = *(const float2*)((const float*)latent + t * 576 + 512 + 2 * lane);
      __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
      r = *(uint32_t*)&b;
    } else {
      r = *(const uint32_t*)((const __nv_bfloat16*)latent + t * 576 + 512 + 2 * lane);
    }
    *(uint32_t*)(o + 528 + 4 * lane) = r;
  }
}

int launch_pack_latent_fp8(const void* latent, bool f32_in, int64_t T, uint8_t* out, cudaStream_t st) {
  if (T == 0) return MTPSD_OK;
  int64_t blocks = (T * 32 + 255) / 256;
  if (blocks > 16 * num_sms()) blocks = 16 * num_sms();
  if (f32_in) launch_k(pack_latent_fp8_kernel<true>, (int)blocks, 256, 0, st, latent, T, out);
  else launch_k(pack_latent_fp8_kernel<false>, (int)blocks, 256, 0, st, latent, T, out);
  return check_launch("pack_latent_fp8");
}

// ---------------------------------------------------------------------------
// Greedy acceptance ([P2] "接受判定", [P1] "阶段 3").  One thread per request.
__global__ void accept_greedy_kernel(const int64_t* __restrict__ draft, const int64_t* __restrict__ tgt,
                                     int B, int K, int64_t magic, int32_t* __restrict__ n_acc,
                                     int64_t* __restrict__ next) {
  griddep_wait();                // the previous kernel's writes are visible from here on
  griddep_launch_dependents();
  int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int64_t* d = draft + (int64_t)b * K;
  const int64_t* t = tgt + (int64_t)b * (K + 1);
  int n = 0;
  bool all_magic = (magic >= 0) && (K > 0);
  for (int i = 0; i < K; ++i) all_magic = all_magic && (d[i] == magic);
  if (!all_magic) {
    while (n < K && d[n] == t[n]) ++n;
  }
  n_acc[b] = n;
  next[b] = t[n];
}

int launch_accept_greedy(const int64_t* draft, const int64_t* tgt, int B, int K, int64_t magic,
                         int32_t* n_acc, int64_t* next, cudaStream_t st) {
  launch_k(accept_greedy_kernel, (B + 127) / 128, 128, 0, st, draft, tgt, B, K, magic, n_acc, next);
  return check_launch("accept_greedy");
}

// ---------------------------------------------------------------------------
// Accepted-segment write-back ([P2] "KV 交账", "draft_extend").  One CTA per
// (request, window row); rows beyond num_accepted+1 return at once.  The
// latent row (1152 B bf16 / 2304 B f32) and the 128-byte indexer key move as
// 16-byte vectors; the float32 scale by one thread.
__global__ void kv_writeback_kernel(const uint4* __restrict__ src_l, const uint4* __restrict__ src_k,
                                    const float* __restrict__ src_s, int W, int lat_vec, int idx_vec,
                                    const int32_t* __restrict__ n_acc, uint4* __restrict__ dst_l,
                                    uint4* __restrict__ dst_k, float* __restrict__ dst_s,
                                    const int64_t* __restrict__ cache_start, const int64_t* __restrict__ dst_pos,
                                    int64_t pool,
                                    int64_t* __restrict__ next_pos, int32_t* __restrict__ status,
                                    const int64_t* __restrict__ dst_slots) {
  griddep_wait();                // the previous kernel's writes are visible from here on
  griddep_launch_dependents();
  int b = blockIdx.y;
  int i = blockIdx.x;
  int n = n_acc[b] + 1;                 // accept_len, bonus included
  if (n < 1) n = 1;
  if (n > W) n = W;
  if (i == 0 && threadIdx.x == 0 && next_pos) next_pos[b] = dst_pos[b] + n;
  if (i >= n) return;
  // destination: the planned window slot (paged caches) or the row after the request's committed ones
  int64_t t = dst_slots ? dst_slots[(int64_t)b * W + i] : cache_start[b] + dst_pos[b] + i;
  if (t < 0 || t >= pool) {
    if (threadIdx.x == 0) flag_status(status, MTPSD_STATUS_WRITE_RANGE);
    return;
  }
  int64_t srow = (int64_t)b * W + i;
  for (int v = threadIdx.x; v < lat_vec; v += blockDim.x) dst_l[t * lat_vec + v] = src_l[srow * lat_vec + v];
  for (int v = threadIdx.x; v < idx_vec; v += blockDim.x) dst_k[t * idx_vec + v] = src_k[srow * idx_vec + v];
  if (dst_s && threadIdx.x == 0) dst_s[t] = src_s[srow];
}

int launch_kv_writeback(const void* src_l, const uint8_t* src_k, const float* src_s, int B, int W,
                        int lat_bytes, int idx_bytes, const int32_t* n_acc, void* dst_l, uint8_t* dst_k,
                        float* dst_s, const int64_t* cache_start, const int64_t* dst_pos, int64_t pool,
                        int64_t* next_pos,
                        int32_t* status, cudaStream_t st, const int64_t* dst_slots) {
  dim3 grid(W, B);
  launch_k(kv_writeback_kernel, grid, 64, 0, st, (const uint4*)src_l, (const uint4*)src_k, src_s, W, lat_bytes / 16,
                                           idx_bytes / 16, n_acc, (uint4*)dst_l, (uint4*)dst_k, dst_s,
                                           cache_start, dst_pos, pool, next_pos, status, dst_slots);
  return check_launch("kv_writeback");
}

// ---------------------------------------------------------------------------
// Step-0 top-k share gather ([P1] "阶段 5").  One CTA per request copies one
// k-wide row with 16-byte vectors when k % 4 == 0.
__global__ void share_gather_kernel(const int32_t* __restrict__ s0, const uint32_t* __restrict__ ro,
                                    const int32_t* __restrict__ n_acc, int k, int32_t* __restrict__ out,
                                    const int64_t* __restrict__ row_pos, int64_t* __restrict__ shared_pos,
                                    int32_t* __restrict__ status) {
  griddep_wait();                // the previous kernel's writes are visible from here on
  griddep_launch_dependents();
  int b = blockIdx.x;
  int64_t first = ro[b], last = (int64_t)ro[b + 1] - 1;
  if (last < first) {  // empty segment: nothing to share
    for (int j = threadIdx.x; j < k; j += blockDim.x) out[(int64_t)b * k + j] = -1;
    if (shared_pos && threadIdx.x == 0) shared_pos[b] = -1;
    return;
  }
  int64_t local = n_acc ? n_acc[b] : 0;
  int64_t row = first + local;
  if (row > last || local < 0) {
    if (threadIdx.x == 0) flag_status(status, MTPSD_STATUS_INDEX_RANGE);
    row = local < 0 ? first : last;
  }
  if (shared_pos && threadIdx.x == 0) shared_pos[b] = row_pos[row];
  if ((k & 3) == 0) {
    const int4* src = (const int4*)(s0 + row * k);
    int4* dst = (int4*)(out + (int64_t)b * k);
    for (int j = threadIdx.x; j < k / 4; j += blockDim.x) dst[j] = src[j];
  } else {
    for (int j = threadIdx.x; j < k; j += blockDim.x) out[(int64_t)b * k + j] = s0[row * k + j];
  }
}

int launch_share_gather(const int32_t* s0, const uint32_t* ro, const int32_t* n_acc, int B, int k,
                        int32_t* out, const int64_t* row_pos, int64_t* shared_pos, int32_t* status, cudaStream_t st) {
  launch_k(share_gather_kernel, B, 128, 0, st, s0, ro, n_acc, k, out, row_pos, shared_pos, status);
  return check_launch("topk_share_gather");
}

// ---------------------------------------------------------------------------
// Check of the bounded mbarrier wait that every tensor-core kernel uses: warp 0
// waits at CTA scope and warp 1 at cluster scope on one barrier phase that
// nothing completes, with the caller's limit.  Each gives up (the first at the
// limit, the other at the limit or on the abort flag the first set), flags
// MTPSD_STATUS_WAIT_TIMEOUT and records [waited ns, 1 if the wait succeeded].
__global__ void bounded_wait_check_kernel(unsigned long long limit_ns, int32_t* status, int64_t* out) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"((uint32_t)__cvta_generic_to_shared(&bar)));
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t t0 = mbar::globaltimer_ns();
  const bool ok = warp == 0 ? mbar::wait<false>(&bar, 0, &abort_flag, status, limit_ns)
                            : mbar::wait<true>(&bar, 0, &abort_flag, status, limit_ns);
  const uint64_t t1 = mbar::globaltimer_ns();
  if (lane == 0) {
    out[2 * warp] = (int64_t)(t1 - t0);
    out[2 * warp + 1] = ok ? 1 : 0;
  }
}

int launch_bounded_wait_check(int64_t limit_ns, int32_t* status, int64_t* out, cudaStream_t st) {
  launch_k(bounded_wait_check_kernel, 1, 64, 0, st, (unsigned long long)limit_ns, status, out);
  return check_launch("bounded_wait_check");
}

}  // namespace mtpsd
