// Per-row top-k without a full sort: radix select of the k-th largest score
// key, then an ordered compaction.
//
// [P3] "Indexer 的结构与计算流程": the fused index kernel returns the top
// index_topk positions per query row; [P2] "验证段的逐层算子" op 6: each row
// selects its own.  Ties at the k-th score go to the lower position; the
// output lists the selected positions in ascending order, -1 padded.
//
// One CTA of 1024 threads per row.  Scores map to order-preserving uint32
// keys; four 8-bit radix passes (most significant first) over the row find
// the k-th largest key T with warp-aggregated shared-memory histograms.  The
// row's keys stay in shared memory when they fit (<= TOPK_SMEM_KEYS), else
// each pass re-reads the row from L2.  A final pass in which every thread owns
// a contiguous segment writes the keys > T and the first (k - #greater) keys
// == T in position order, so the output is sorted and deterministic.
#include "common.cuh"
#include "internal.h"

namespace mtpsd {

constexpr int TOPK_THREADS = 1024;
constexpr int TOPK_SMEM_KEYS = 48 * 1024;   // 192 KB of keys

__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int w = (lane < (TOPK_THREADS / 32)) ? warp_sums[lane] : 0;
    int incl = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    warp_sums[lane] = incl - w;
    if (lane == 31) *total = incl;
  }
  __syncthreads();
  int res = warp_sums[wid] + x - v;
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(TOPK_THREADS, 1) topk_kernel(TopkPlan p, int64_t cache_cap) {
  extern __shared__ uint32_t keys_s[];
  __shared__ int hist[256];
  __shared__ int warp_sums[32];
  __shared__ int total_s;
  __shared__ uint32_t prefix_s;
  __shared__ int remaining_s;

  const int r = blockIdx.x;
  int64_t V = p.row_len[r] + (p.len_plus_one ? 1 : 0);
  if (V > p.max_len) {
    if (threadIdx.x == 0) flag_status(p.status, MTPSD_STATUS_INDEX_RANGE);
    V = p.max_len;
  }
  if (V < 0) V = 0;
  const int k = p.k;
  int32_t* out = p.out_idx + (int64_t)r * k;
  float* outs = p.out_score ? p.out_score + (int64_t)r * k : nullptr;
  const float* row = p.scores + (int64_t)r * p.ld;

  if (V <= k) {  // everything visible is selected
    for (int64_t i = threadIdx.x; i < k; i += blockDim.x) {
      out[i] = i < V ? (int32_t)i : -1;
      if (outs) outs[i] = i < V ? row[i] : -INFINITY;
    }
    return;
  }

  const bool cached = V <= cache_cap;
  if (cached)
    for (int64_t i = threadIdx.x; i < V; i += blockDim.x) keys_s[i] = float_key(row[i]);

  uint32_t prefix = 0, mask = 0;
  int remaining = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const int64_t Vr = (V + 31) & ~31LL;   // whole warps stay converged for match_any
    for (int64_t i = threadIdx.x; i < Vr; i += blockDim.x) {
      bool in = i < V;
      uint32_t key = 0;
      if (in) {
        key = cached ? keys_s[i] : float_key(row[i]);
        in = (key & mask) == prefix;
      }
      uint32_t bin = in ? ((key >> shift) & 255u) : 256u;
      uint32_t peers = __match_any_sync(0xffffffffu, bin);
      int leader = __ffs(peers) - 1;
      if (in && (int)(threadIdx.x & 31) == leader) atomicAdd(&hist[bin], __popc(peers));
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // find the bin holding the remaining-th largest key, scanning from the top
      const int lane = threadIdx.x;
      int cum = 0;   // keys in bins above the current group
      int chosen = -1, above = 0;
      for (int g = 7; g >= 0 && chosen < 0; --g) {
        int bin = g * 32 + (31 - lane);     // lane 0 = highest bin of the group
        int c = hist[bin];
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        bool hit = (cum + incl >= remaining) && (cum + incl - c < remaining);
        unsigned ball = __ballot_sync(0xffffffffu, hit);
        if (ball) {
          int src = __ffs(ball) - 1;
          chosen = __shfl_sync(0xffffffffu, bin, src);
          above = __shfl_sync(0xffffffffu, cum + incl - c, src);
        }
        cum += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (chosen < 0) chosen = 0;   // unreachable when V > k
      if (lane == 0) {
        prefix_s = prefix | ((uint32_t)chosen << shift);
        remaining_s = remaining - above;
      }
    }
    __syncthreads();
    prefix = prefix_s;
    remaining = remaining_s;
    mask |= 255u << shift;
  }
  const uint32_t T = prefix;     // the k-th largest key
  const int need_eq = remaining; // how many keys equal to T are taken (lowest positions first)

  // ordered compaction: thread t owns positions [t*seg, (t+1)*seg)
  const int64_t seg = (V + TOPK_THREADS - 1) / TOPK_THREADS;
  const int64_t a = min((int64_t)threadIdx.x * seg, V), e = min(a + seg, V);
  int n_gt = 0, n_eq = 0;
  for (int64_t i = a; i < e; ++i) {
    uint32_t key = cached ? keys_s[i] : float_key(row[i]);
    n_gt += key > T;
    n_eq += key == T;
  }
  int eq_before = block_exclusive_scan(n_eq, warp_sums, &total_s);
  int take_eq = max(0, min(n_eq, need_eq - eq_before));
  int out_pos = block_exclusive_scan(n_gt + take_eq, warp_sums, &total_s);
  for (int64_t i = a; i < e; ++i) {
    uint32_t key = cached ? keys_s[i] : float_key(row[i]);
    bool take = key > T;
    if (key == T && take_eq > 0) {
      take = true;
      --take_eq;
    }
    if (take && out_pos < k) {
      out[out_pos] = (int32_t)i;
      if (outs) outs[out_pos] = key_float(key);
      ++out_pos;
    }
  }
}

int launch_topk(const TopkPlan& p, cudaStream_t st) {
  if (p.R == 0) return MTPSD_OK;
  int64_t cache_keys = p.max_len <= TOPK_SMEM_KEYS ? p.max_len : 0;
  size_t smem = (size_t)cache_keys * sizeof(uint32_t);
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  topk_kernel<<<p.R, TOPK_THREADS, smem, st>>>(p, cache_keys);
  return check_launch("topk");
}

}  // namespace mtpsd
