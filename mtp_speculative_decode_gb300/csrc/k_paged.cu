// Paged (slotted) KV caches: the window's slot plan and the accepted-KV move.
//
// [P2] "输入准备:prepare_for_draft": the caches are pools of token slots reached
// through a per-request token table (page_size > 1: pages of consecutive
// slots); once per iteration the slots of the W window positions after the
// committed length are planned into out_cache_loc.
// [P2] "KV 交账:接受段的搬移与拒绝段的回收": the KV of the accepted rows
// (their window slots) moves to the first accept_len window slots.
// Both are latency-bound one-launch kernels.
#include "common.cuh"
#include "internal.h"

namespace mtpsd {

// One thread per (request, window column).
__global__ void assign_cache_locs_kernel(const int32_t* __restrict__ bt, int32_t stride, int32_t shift, int B,
                                         const int64_t* __restrict__ start_pos, int W, int64_t* __restrict__ out,
                                         int32_t* __restrict__ status) {
  griddep_wait();                // the previous kernel's writes are visible from here on
  griddep_launch_dependents();
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)B * W) return;
  const int b = (int)(t / W), j = (int)(t % W);
  const int64_t slot = paged_slot(bt, stride, shift, b, start_pos[b] + j);
  if (slot < 0) flag_status(status, MTPSD_STATUS_ROW_RANGE);
  out[t] = slot;
}

int launch_assign_cache_locs(const Paging& pg, int B, const int64_t* start_pos, int W, int64_t* out, int32_t* status,
                             cudaStream_t st) {
  const int64_t n = (int64_t)B * W;
  launch_k(assign_cache_locs_kernel, (unsigned)((n + 255) / 256), 256, 0, st, pg.bt, pg.stride, pg.shift, B,
           start_pos, W, out, status);
  return check_launch("assign_cache_locs");
}

// One CTA per request.  The slots of different requests are disjoint, so the
// move of a request is self-contained: every source row of the request is
// first copied into shared memory, then (after one barrier) every destination
// is written, which makes the result independent of any overlap between the
// request's source and destination slot lists.  Shared row i: the latent
// bytes, the key bytes, then the key scale (16-byte slot).
__global__ void kv_move_kernel(uint4* __restrict__ lat, int lat_vec, uint4* __restrict__ idxk, int idx_vec,
                               float* __restrict__ idxs, int64_t pool, const int64_t* __restrict__ loc,
                               const int32_t* __restrict__ acc_idx, const int32_t* __restrict__ n_acc, int W,
                               int32_t* __restrict__ status) {
  griddep_wait();                // the previous kernel's writes are visible from here on
  griddep_launch_dependents();
  extern __shared__ uint4 stage[];
  __shared__ int64_t dst_of[16];   // destination slot of row i, or -1 (nothing to do)
  __shared__ int64_t src_of[16];
  const int b = blockIdx.x;
  const int row_vec = lat_vec + idx_vec + 1;
  int n = n_acc[b] + 1;            // accept_len, the bonus row included
  n = n < 0 ? 0 : (n > W ? W : n);
  if (threadIdx.x < n) {
    const int i = threadIdx.x;
    const int c = acc_idx[(int64_t)b * W + i];
    int64_t d = -1, s = -1;
    if (c < 0 || c >= W) {
      flag_status(status, MTPSD_STATUS_INDEX_RANGE);
    } else {
      d = loc[(int64_t)b * W + i];
      s = loc[(int64_t)b * W + c];
      if (d < 0 || d >= pool || s < 0 || s >= pool) {
        flag_status(status, MTPSD_STATUS_WRITE_RANGE);
        d = -1;
      } else if (d == s) {
        d = -1;   // already in place
      }
    }
    dst_of[i] = d;
    src_of[i] = s;
  }
  __syncthreads();
  for (int i = 0; i < n; ++i) {
    if (dst_of[i] < 0) continue;
    const int64_t s = src_of[i];
    uint4* row = stage + (int64_t)i * row_vec;
    for (int v = threadIdx.x; v < lat_vec; v += blockDim.x) row[v] = lat[s * lat_vec + v];
    for (int v = threadIdx.x; v < idx_vec; v += blockDim.x) row[lat_vec + v] = idxk[s * idx_vec + v];
    if (idxs && threadIdx.x == 0) row[lat_vec + idx_vec].x = __float_as_uint(idxs[s]);
  }
  __syncthreads();
  for (int i = 0; i < n; ++i) {
    const int64_t d = dst_of[i];
    if (d < 0) continue;
    const uint4* row = stage + (int64_t)i * row_vec;
    for (int v = threadIdx.x; v < lat_vec; v += blockDim.x) lat[d * lat_vec + v] = row[v];
    for (int v = threadIdx.x; v < idx_vec; v += blockDim.x) idxk[d * idx_vec + v] = row[lat_vec + v];
    if (idxs && threadIdx.x == 0) idxs[d] = __uint_as_float(row[lat_vec + idx_vec].x);
  }
}

int launch_kv_move(void* lat, int lat_bytes, uint8_t* idxk, int idx_bytes, float* idxs, int64_t pool,
                   const int64_t* loc, const int32_t* acc_idx, const int32_t* n_acc, int B, int W, int32_t* status,
                   cudaStream_t st) {
  const int lat_vec = lat_bytes / 16, idx_vec = idx_bytes / 16;
  const size_t smem = (size_t)W * (lat_vec + idx_vec + 1) * 16;
  static std::atomic<uint64_t> attr{0};
  if (smem > 48 * 1024 && !set_smem_limit_once(kv_move_kernel, 64 * 1024, attr)) {
    set_error("kv_move_accepted: cudaFuncSetAttribute failed");
    return MTPSD_ECUDA;
  }
  launch_k(kv_move_kernel, B, 256, smem, st, (uint4*)lat, lat_vec, (uint4*)idxk, idx_vec, idxs, pool, loc, acc_idx,
           n_acc, W, status);
  return check_launch("kv_move_accepted");
}

}  // namespace mtpsd
