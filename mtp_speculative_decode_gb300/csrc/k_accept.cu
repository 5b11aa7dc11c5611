// Rejection-sampling acceptance of a chain of K drafts.
//
// [P2] "接受判定:greedy 与 rejection sampling": the draft distribution q and
// the target distribution p; draft i is accepted with probability min(1, p/q),
// and a rejected position draws its token from the corrected distribution.
// The corrected distribution is the speculative-sampling one, max(0, p - q)
// normalised; after K accepted drafts the next token is drawn from p of row K.
// The random numbers are inputs (one uniform per draft for the accept test, one
// per request for the draw).
//
// One CTA of 1024 threads per request.  Warp 0 tests the drafts in order,
// u * q[d] < p[d] in single precision (a draft id outside the vocabulary is
// rejected and flagged), and the first rejection fixes the row to draw from.
// The draw is an exact inverse CDF: each weight becomes floor(w * 2^32) as an
// unsigned 64-bit integer, so the running sums are exact in any order; every
// thread sums a contiguous segment of the row, one exclusive block scan gives
// the total and each segment's start, and the thread whose segment holds the
// first running sum above floor(u * total) rescans it to find the token.
#include "common.cuh"
#include "internal.h"

namespace mtpsd {

constexpr int ACC_THREADS = 1024;

// floor(u * total) for a single-precision u in [0, 1), exact: u = mant * 2^(e - 24) with a 24-bit mant.
__device__ __forceinline__ uint64_t scaled_floor(float u, uint64_t total) {
  if (!(u > 0.f)) return 0;
  int e;
  const float m = frexpf(u, &e);                     // u = m * 2^e, m in [0.5, 1)
  const uint64_t mant = (uint64_t)(m * 16777216.0f);  // m * 2^24: an integer below 2^24, exact
  const int shift = 24 - e;                           // >= 25 for u < 1
  const uint64_t lo = mant * total, hi = __umul64hi(mant, total);
  if (shift >= 128) return 0;
  if (shift >= 64) return hi >> (shift - 64);
  return (lo >> shift) | (hi << (64 - shift));
}

// floor(max(w, 0) * 2^32): the scaling by a power of two is exact, the conversion truncates.
__device__ __forceinline__ uint64_t fixed_weight(float w) { return __float2ull_rz(fmaxf(w, 0.f) * 4294967296.0f); }

__device__ __forceinline__ uint64_t block_excl_scan_u64(uint64_t v, uint64_t* warp_sums, uint64_t* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  uint64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[wid] = x;
  __syncthreads();
  if (wid == 0) {
    const uint64_t w = lane < nw ? warp_sums[lane] : 0ull;
    uint64_t incl = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    warp_sums[lane] = incl - w;
    if (lane == 31) *total = incl;
  }
  __syncthreads();
  const uint64_t res = warp_sums[wid] + x - v;
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(ACC_THREADS) accept_stochastic_kernel(
    const int64_t* __restrict__ draft, const float* __restrict__ q, const float* __restrict__ p,
    const float* __restrict__ ua, const float* __restrict__ us, int K, int64_t V, int32_t* __restrict__ n_acc,
    int64_t* __restrict__ next, int32_t* __restrict__ status) {
  griddep_wait();                // the previous kernel's writes are visible from here on
  griddep_launch_dependents();
  __shared__ int s_n;
  __shared__ long long s_tok;
  __shared__ uint64_t warp_sums[32];
  __shared__ uint64_t s_total;
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  if (tid < 32) {
    int rej = K;   // first rejected draft
    for (int i0 = 0; i0 < K; i0 += 32) {
      const int i = i0 + lane;
      bool reject = false;
      if (i < K) {
        const int64_t d = draft[(int64_t)b * K + i];
        if (d < 0 || d >= V) {
          reject = true;
          flag_status(status, MTPSD_STATUS_INDEX_RANGE);
        } else {
          const float qq = q[((int64_t)b * K + i) * V + d];
          const float pp = p[((int64_t)b * (K + 1) + i) * V + d];
          reject = !(__fmul_rn(ua[(int64_t)b * K + i], qq) < pp);
        }
      }
      const unsigned m = __ballot_sync(0xffffffffu, reject);
      if (m) {
        rej = i0 + __ffs(m) - 1;
        break;
      }
    }
    if (lane == 0) {
      s_n = rej;
      s_tok = -1;
    }
  }
  __syncthreads();
  const int n = s_n;
  const float* prow = p + ((int64_t)b * (K + 1) + n) * V;
  const float* qrow = n < K ? q + ((int64_t)b * K + n) * V : nullptr;
  const float u = us[b];
  const int64_t seg = (V + ACC_THREADS - 1) / ACC_THREADS;
  const int64_t a0 = min((int64_t)tid * seg, V), a1 = min(a0 + seg, V);
  // pass 0 draws from the residual (or from p of row K after full acceptance); pass 1 from p of the
  // rejected row when the residual has no mass
  for (int pass = 0; pass < 2; ++pass) {
    if (pass == 1 && !qrow) break;
    const bool resid = qrow != nullptr && pass == 0;
    uint64_t part = 0;
    for (int64_t t = a0; t < a1; ++t) part += fixed_weight(resid ? prow[t] - qrow[t] : prow[t]);
    const uint64_t before = block_excl_scan_u64(part, warp_sums, &s_total);
    const uint64_t total = s_total;   // block-uniform
    if (total == 0) continue;
    const uint64_t target = scaled_floor(u, total);
    if (before <= target && target < before + part) {   // the first running sum above target is here
      uint64_t run = before;
      for (int64_t t = a0; t < a1; ++t) {
        run += fixed_weight(resid ? prow[t] - qrow[t] : prow[t]);
        if (run > target) {
          s_tok = t;
          break;
        }
      }
    }
    break;
  }
  __syncthreads();
  if (tid == 0) {
    n_acc[b] = n;
    next[b] = s_tok >= 0 ? (int64_t)s_tok : 0;
  }
}

int launch_accept_stochastic(const int64_t* draft, const float* q, const float* p, const float* ua, const float* us,
                             int B, int K, int64_t V, int32_t* n_acc, int64_t* next, int32_t* status,
                             cudaStream_t st) {
  launch_k(accept_stochastic_kernel, B, ACC_THREADS, 0, st, draft, q, p, ua, us, K, V, n_acc, next, status);
  return check_launch("accept_stochastic");
}

}  // namespace mtpsd
