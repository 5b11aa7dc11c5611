// Lightning-indexer scores on CUDA cores (float32 accumulation).
//
// [P3] "Indexer 的结构与计算流程":
//   I[r,s] = sum_h w[r,h] * ReLU(q_scale[r,h] * k_scale[s] * q[r,h,:].k[s,:])
// This kernel serves the float32 configuration and any FP8 shape the
// tensor-core kernel (k_indexer_tc.cu) does not take.  One CTA owns a tile of
// 64 positions of one request and loops over that request's rows, so each key
// tile is read from HBM once for all rows of the request.
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace mtpsd {

constexpr int IDX_TILE = 64;

template <bool FP8>
__global__ void __launch_bounds__(256) indexer_scores_kernel(IndexerPlan p) {
  griddep_wait();                // the previous kernel's writes are visible from here on
  griddep_launch_dependents();
  extern __shared__ float smem[];
  const int H = p.H, D = p.D, DP = p.D + 1;
  float* ks = smem;                      // [64][D+1] dequantized keys
  float* qs = ks + IDX_TILE * DP;        // [H][D] dequantized query of the current row
  float* ws = qs + H * D;                // [H] head weights
  float* part = ws + H;                  // [4][64] partial sums

  const int b = blockIdx.y;
  const int tile = blockIdx.x;
  const uint32_t r0 = p.row_offsets[b], r1 = p.row_offsets[b + 1];
  if (r1 <= r0) return;
  int64_t vmax = 0;
  for (uint32_t r = r0; r < r1; ++r) vmax = max(vmax, p.row_pos[r] + 1);
  vmax = min(vmax, p.max_visible);
  const int64_t s0 = (int64_t)tile * IDX_TILE;
  if (s0 >= vmax) return;
  // pool row of each position of the tile (-1: not visible, or no row)
  __shared__ int64_t rows_s[IDX_TILE];
  if (threadIdx.x < IDX_TILE) {
    const int64_t s = s0 + threadIdx.x;
    int64_t row = -1;
    if (s < vmax) {
      row = p.pg.bt ? paged_slot(p.pg.bt, p.pg.stride, p.pg.shift, b, s) : p.cache_start[b] + s;
      if (row >= p.pool) row = -1;
      if (row < 0 && p.pg.bt) flag_status(p.status, MTPSD_STATUS_ROW_RANGE);
    }
    rows_s[threadIdx.x] = row;
  }
  __syncthreads();

  // key tile -> shared (dequantized to float)
  for (int e = threadIdx.x; e < IDX_TILE * D; e += blockDim.x) {
    int i = e / D, d = e % D;
    int64_t row = rows_s[i];
    float v = 0.f;
    if (row >= 0) {
      if (FP8) {
        __nv_fp8_e4m3 c;
        c.__x = ((const uint8_t*)p.k)[row * D + d];
        v = float(c) * p.k_scale[row];
      } else {
        v = ((const float*)p.k)[row * D + d];
      }
    }
    ks[i * DP + d] = v;
  }

  const int pos = threadIdx.x & (IDX_TILE - 1);
  const int hg = threadIdx.x / IDX_TILE;       // 4 head groups
  const int hpg = (H + 3) / 4;
  for (uint32_t r = r0; r < r1; ++r) {
    __syncthreads();
    for (int e = threadIdx.x; e < H * D; e += blockDim.x) {
      int h = e / D;
      float v;
      if (FP8) {
        __nv_fp8_e4m3 c;
        c.__x = ((const uint8_t*)p.q)[(int64_t)r * H * D + e];
        v = float(c) * p.q_scale[(int64_t)r * H + h];
      } else {
        v = ((const float*)p.q)[(int64_t)r * H * D + e];
      }
      qs[e] = v;
    }
    for (int h = threadIdx.x; h < H; h += blockDim.x) ws[h] = p.w[(int64_t)r * H + h];
    __syncthreads();
    float acc = 0.f;
    const float* kr = ks + pos * DP;
    for (int h = hg * hpg; h < min(H, (hg + 1) * hpg); ++h) {
      const float* qh = qs + h * D;
      float dot = 0.f;
      for (int d = 0; d < D; ++d) dot = fmaf(qh[d], kr[d], dot);
      acc = fmaf(ws[h], fmaxf(dot, 0.f), acc);
    }
    part[hg * IDX_TILE + pos] = acc;
    __syncthreads();
    if (threadIdx.x < IDX_TILE) {
      int64_t s = s0 + threadIdx.x;
      if (s <= p.row_pos[r] && s < p.max_visible) {
        float v = part[threadIdx.x] + part[IDX_TILE + threadIdx.x] + part[2 * IDX_TILE + threadIdx.x] +
                  part[3 * IDX_TILE + threadIdx.x];
        p.scores[(int64_t)r * p.ld + s] = v;
      }
    }
  }
}

int launch_indexer_scores(const IndexerPlan& p, cudaStream_t st) {
  int64_t tiles = ceil_div(p.max_visible, IDX_TILE);
  if (tiles <= 0) return MTPSD_OK;
  if (tiles > 2147483647LL) {
    set_error("indexer: too many position tiles");
    return MTPSD_EINVAL;
  }
  size_t smem = sizeof(float) * ((size_t)IDX_TILE * (p.D + 1) + (size_t)p.H * p.D + p.H + 4 * IDX_TILE);
  dim3 grid((unsigned)tiles, p.B);
  if (p.dtype == MTPSD_FP8_E4M3) {
    if (smem > 48 * 1024)
      cudaFuncSetAttribute(indexer_scores_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    launch_k(indexer_scores_kernel<true>, grid, 256, smem, st, p);
  } else {
    if (smem > 48 * 1024)
      cudaFuncSetAttribute(indexer_scores_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    launch_k(indexer_scores_kernel<false>, grid, 256, smem, st, p);
  }
  return check_launch("indexer_scores");
}

}  // namespace mtpsd
