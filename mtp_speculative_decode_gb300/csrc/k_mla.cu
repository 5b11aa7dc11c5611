// Sparse MLA decode over the selected latent rows.
//
// [P2] "GLM-5.3 的草稿层到底长什么样": latent = kv_lora_rank 512 + rope 64;
// [P2] "验证段的逐层算子" op 7 and [P3] "稀疏 MLA 的前向路径": attention runs
// only over the positions chosen by the indexer.  With the absorbed query the
// key of position s is latent[s, 0:576] and its value latent[s, 0:512]:
//   o[r,h] = sum_j softmax_j(scale * q[r,h,:].c[s_j,:]) * c[s_j, 0:512]
//
// bf16 path (sparse_mla_bf16_kernel): one CTA per (row, group of 64 heads,
// split of the selected list).  The selected latent rows of a 32-position
// tile are gathered with 16-byte cp.async into a double-buffered shared tile;
// QK^T and PV run on tensor cores (mma.sync m16n8k16 bf16, fp32 accumulate)
// with the 16x576 query fragments and the 32x576 key tile streamed from
// shared memory by ldmatrix; the online softmax keeps the running max / sum
// per head (the two warps that share a head block exchange the tile max
// through shared memory).  Split CTAs write unnormalised partials that
// mla_combine_kernel merges with their log-sum-exp weights.
// float32 path (sparse_mla_f32_kernel): CUDA cores, one CTA per (row, head).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace mtpsd {

constexpr int MLA_DL = 576;
constexpr int MLA_DV = 512;
constexpr int MLA_HG = 64;            // heads per CTA
constexpr int MLA_NT = 32;            // positions per tile
constexpr int MLA_ROWB = MLA_DL * 2 + 16;   // padded shared row (bytes): conflict-free ldmatrix
constexpr int MLA_PROWB = MLA_NT * 2 + 16;  // padded P row (bytes)
constexpr int MLA_MAX_SPLIT = 2048;   // positions per split CTA
constexpr float LOG2E = 1.4426950408889634f;

// pool row of logical entry j of row r, or -1 (padding / out of range)
__device__ __forceinline__ int64_t mla_pool_row(const MlaPlan& p, int r, int b, int64_t j, int64_t limit) {
  int64_t s;
  if (j < p.n_idx) {
    s = p.idx[(int64_t)r * p.n_idx + j];
    if (s == -1) return -1;
  } else {
    s = p.append_base[r] + 1 + (j - p.n_idx);
  }
  if (s < 0 || s > limit) {
    flag_status(p.status, MTPSD_STATUS_INDEX_RANGE);
    return -1;
  }
  int64_t row = p.pg.bt ? paged_slot(p.pg.bt, p.pg.stride, p.pg.shift, b, s) : p.cache_start[b] + s;
  if (row < 0 || row >= p.pool) {
    flag_status(p.status, MTPSD_STATUS_ROW_RANGE);
    return -1;
  }
  return row;
}

__device__ __forceinline__ void cp_async16(uint32_t smem, const void* gmem, bool valid) {
  int sz = valid ? 16 : 0;   // zero-fill invalid rows
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem), "l"(gmem), "r"(sz));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& a0, uint32_t& a1, uint32_t& a2, uint32_t& a3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& a0, uint32_t& a1, uint32_t& a2, uint32_t& a3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3) : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

struct MlaSplit {
  int n_splits;
  int64_t per_split;   // positions per split (multiple of MLA_NT)
};

// Shared memory layout of the bf16 kernel (FP8KV adds the staging tiles of the packed rows).
constexpr int MLA_FP8_ROW = 656;          // packed FP8 latent row: 512 codes, 4 float32 scales, 64 bf16 rope
template <bool FP8KV>
struct MlaSmemT {
  static constexpr int Q = 0;                                     // [64][ROWB]
  static constexpr int C = Q + MLA_HG * MLA_ROWB;                 // [2][32][ROWB]
  static constexpr int P = C + 2 * MLA_NT * MLA_ROWB;             // [64][PROWB]
  static constexpr int RED = P + MLA_HG * MLA_PROWB;              // [2][64] float
  static constexpr int LSUM = RED + 2 * MLA_HG * 4;               // [2][64] float
  static constexpr int ROWS = LSUM + 2 * MLA_HG * 4;              // [MAX_SPLIT] int64
  static constexpr int STG = ROWS + MLA_MAX_SPLIT * 8;            // FP8KV: [2][32][656] packed rows
  static constexpr int BYTES = STG + (FP8KV ? 2 * MLA_NT * MLA_FP8_ROW : 0);
};
using MlaSmem = MlaSmemT<false>;

// One tile of packed FP8 rows (staging) -> bf16 rows of the compute tile: value = code * block scale
// (E4M3 -> f16 is exact; the product is formed in float32 and rounded to bf16), rope copied.
__device__ __forceinline__ void mla_dequant_tile(const uint8_t* stg, uint8_t* c) {
  for (int w = threadIdx.x; w < MLA_NT * 64; w += blockDim.x) {   // 64 groups of 8 codes per row
    const int i = w >> 6, grp = w & 63;
    const uint8_t* src = stg + i * MLA_FP8_ROW;
    const uint2 codes = *(const uint2*)(src + grp * 8);
    const float sc = *(const float*)(src + 512 + (grp >> 4) * 4);
    uint32_t outw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t word = e < 2 ? codes.x : codes.y;
      const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)((word >> (16 * (e & 1))) & 0xffffu);
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
      const float2 f = __half22float2(*(const __half2*)&hr);
      const __nv_bfloat162 bv = __floats2bfloat162_rn(f.x * sc, f.y * sc);
      outw[e] = *(const uint32_t*)&bv;
    }
    *(uint4*)(c + i * MLA_ROWB + grp * 16) = make_uint4(outw[0], outw[1], outw[2], outw[3]);
  }
  for (int w = threadIdx.x; w < MLA_NT * 8; w += blockDim.x) {    // rope: 8 chunks of 16 bytes per row
    const int i = w >> 3, ch = w & 7;
    *(uint4*)(c + i * MLA_ROWB + 1024 + ch * 16) = *(const uint4*)(stg + i * MLA_FP8_ROW + 528 + ch * 16);
  }
}

template <bool FP8KV>
__global__ void __launch_bounds__(256, 1) sparse_mla_bf16_kernel(MlaPlan p, MlaSplit sp, float* __restrict__ part_o,
                                                                  float* __restrict__ part_ml) {
  using MlaSmem = MlaSmemT<FP8KV>;
  griddep_wait();                // the previous kernel's writes are visible from here on
  griddep_launch_dependents();
  extern __shared__ __align__(128) uint8_t sm[];
  const int r = blockIdx.x;
  const int hg = blockIdx.y;
  const int split = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int mi = warp & 3, vi = warp >> 2;     // head block (16 heads), value half (256 dims)
  const int g = lane >> 2, t4 = lane & 3;
  const int H = p.H;
  const int h0 = hg * MLA_HG;

  const int b = request_of_row(p.row_offsets, p.B, (uint32_t)r);
  const int64_t limit = p.row_pos[r] + p.row_pos_add;
  const int64_t total = (int64_t)p.n_idx + p.n_append;
  const int64_t j0 = (int64_t)split * sp.per_split;
  const int64_t j1 = min(total, j0 + sp.per_split);
  const int n_tiles = (int)ceil_div(max(j1 - j0, (int64_t)0), MLA_NT);

  int64_t* rows_s = (int64_t*)(sm + MlaSmem::ROWS);
  float* red = (float*)(sm + MlaSmem::RED);
  float* lsum = (float*)(sm + MlaSmem::LSUM);
  for (int64_t j = j0 + tid; j < j0 + (int64_t)n_tiles * MLA_NT; j += blockDim.x)
    rows_s[j - j0] = j < j1 ? mla_pool_row(p, r, b, j, limit) : -1;

  // query block -> shared (heads beyond H zero-filled)
  const __nv_bfloat16* qg = (const __nv_bfloat16*)p.q + ((int64_t)r * H) * MLA_DL;
  for (int c = tid; c < MLA_HG * (MLA_DL / 8); c += blockDim.x) {
    int h = c / (MLA_DL / 8), ch = c % (MLA_DL / 8);
    bool ok = (h0 + h) < H;
    const void* src = ok ? (const void*)(qg + (int64_t)(h0 + h) * MLA_DL + ch * 8) : (const void*)qg;
    cp_async16(smem_u32(sm + MlaSmem::Q + h * MLA_ROWB + ch * 16), src, ok);
  }
  cp_async_commit();
  __syncthreads();   // rows_s visible

  const __nv_bfloat16* lat = (const __nv_bfloat16*)p.latent;
  auto gather = [&](int tile, int buf) {
    if constexpr (FP8KV) {   // packed rows into the staging tile (invalid rows zero-filled: scale 0)
      const uint8_t* lat8 = (const uint8_t*)p.latent;
      for (int c = tid; c < MLA_NT * (MLA_FP8_ROW / 16); c += blockDim.x) {
        int i = c / (MLA_FP8_ROW / 16), ch = c % (MLA_FP8_ROW / 16);
        int64_t row = rows_s[(int64_t)tile * MLA_NT + i];
        const void* src = row >= 0 ? (const void*)(lat8 + row * MLA_FP8_ROW + ch * 16) : (const void*)lat8;
        cp_async16(smem_u32(sm + MlaSmem::STG + (buf * MLA_NT + i) * MLA_FP8_ROW + ch * 16), src, row >= 0);
      }
    } else {
      for (int c = tid; c < MLA_NT * (MLA_DL / 8); c += blockDim.x) {
        int i = c / (MLA_DL / 8), ch = c % (MLA_DL / 8);
        int64_t row = rows_s[(int64_t)tile * MLA_NT + i];
        const void* src = row >= 0 ? (const void*)(lat + row * MLA_DL + ch * 8) : (const void*)lat;
        cp_async16(smem_u32(sm + MlaSmem::C + (buf * MLA_NT + i) * MLA_ROWB + ch * 16), src, row >= 0);
      }
    }
    cp_async_commit();
  };

  float o[32][4];
#pragma unroll
  for (int n = 0; n < 32; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};   // rows g, g+8 (log2 units)
  float l_run[2] = {0.f, 0.f};
  const float sl2 = p.scale * LOG2E;

  if (n_tiles > 0) gather(0, 0);
  for (int tile = 0; tile < n_tiles; ++tile) {
    const int buf = tile & 1;
    if (tile + 1 < n_tiles) {
      gather(tile + 1, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if constexpr (FP8KV) {
      mla_dequant_tile(sm + MlaSmem::STG + buf * MLA_NT * MLA_FP8_ROW, sm + MlaSmem::C + buf * MLA_NT * MLA_ROWB);
      __syncthreads();
    }

    // ---- S = Q_blk(16 heads) . C_half(16 positions)^T over 576
    float s[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
    const uint32_t qa = smem_u32(sm + MlaSmem::Q + (mi * 16 + (lane & 15)) * MLA_ROWB + (lane >> 4) * 16);
    const int mat = lane >> 3;
    const uint32_t cb = smem_u32(sm + MlaSmem::C + (buf * MLA_NT + vi * 16 + (mat >> 1) * 8 + (lane & 7)) * MLA_ROWB +
                                 (mat & 1) * 16);
#pragma unroll 4
    for (int kk = 0; kk < MLA_DL / 16; ++kk) {
      uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
      ldsm_x4(qa + kk * 32, a0, a1, a2, a3);
      ldsm_x4(cb + kk * 32, b0, b1, b2, b3);
      mma_bf16(s[0], a0, a1, a2, a3, b0, b1);
      mma_bf16(s[1], a0, a1, a2, a3, b2, b3);
    }
    // mask invalid positions, scale to log2 units
    const int64_t* trow = rows_s + (int64_t)tile * MLA_NT + vi * 16;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < 2; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        int col = n * 8 + t4 * 2 + (e & 1);
        float v = trow[col] >= 0 ? s[n][e] * sl2 : -INFINITY;
        s[n][e] = v;
        mx[e >> 1] = fmaxf(mx[e >> 1], v);
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
    }
    if (t4 == 0) {
      red[vi * MLA_HG + mi * 16 + g] = mx[0];
      red[vi * MLA_HG + mi * 16 + g + 8] = mx[1];
    }
    __syncthreads();
    float alpha[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float other = red[(vi ^ 1) * MLA_HG + mi * 16 + g + i * 8];
      float m_new = fmaxf(m_run[i], fmaxf(mx[i], other));
      alpha[i] = (m_new == -INFINITY) ? 1.f : exp2f(m_run[i] - m_new);
      m_run[i] = m_new;
    }
    // P = exp2(s - m), bf16 into shared; row sums
    float ps[2] = {0.f, 0.f};
    uint8_t* prow = sm + MlaSmem::P;
#pragma unroll
    for (int n = 0; n < 2; ++n) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float m = m_run[i];
        float e0 = (m == -INFINITY) ? 0.f : exp2f(s[n][2 * i] - m);
        float e1 = (m == -INFINITY) ? 0.f : exp2f(s[n][2 * i + 1] - m);
        __nv_bfloat162 pr = __floats2bfloat162_rn(e0, e1);
        // the sum uses the rounded values that PV multiplies
        float2 pf = __bfloat1622float2(pr);
        ps[i] += pf.x + pf.y;
        int hrow = mi * 16 + g + i * 8;
        int col = vi * 16 + n * 8 + t4 * 2;
        *(__nv_bfloat162*)(prow + hrow * MLA_PROWB + col * 2) = pr;
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      ps[i] += __shfl_xor_sync(0xffffffffu, ps[i], 1);
      ps[i] += __shfl_xor_sync(0xffffffffu, ps[i], 2);
      l_run[i] = l_run[i] * alpha[i] + ps[i];
    }
#pragma unroll
    for (int n = 0; n < 32; ++n) {
      o[n][0] *= alpha[0];
      o[n][1] *= alpha[0];
      o[n][2] *= alpha[1];
      o[n][3] *= alpha[1];
    }
    __syncthreads();   // P complete

    // ---- O(16 heads x 256 dims) += P(16 x 32) . V(32 x 256)
    const uint32_t pa = smem_u32(sm + MlaSmem::P + (mi * 16 + (lane & 15)) * MLA_PROWB + (lane >> 4) * 16);
    const uint32_t vb = smem_u32(sm + MlaSmem::C + (buf * MLA_NT + (mat & 1) * 8 + (lane & 7)) * MLA_ROWB +
                                 (vi * 256 + (mat >> 1) * 8) * 2);
#pragma unroll
    for (int kk = 0; kk < MLA_NT / 16; ++kk) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(pa + kk * 32, a0, a1, a2, a3);
#pragma unroll
      for (int nn = 0; nn < 16; ++nn) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + kk * 16 * MLA_ROWB + nn * 32, b0, b1, b2, b3);
        mma_bf16(o[2 * nn], a0, a1, a2, a3, b0, b1);
        mma_bf16(o[2 * nn + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    __syncthreads();   // tile buffer and P free
  }
  if (n_tiles == 0) {
    cp_async_wait<0>();
  }

  // combine the two value-half warps' row sums (each saw half the positions)
  if (t4 == 0) {
    lsum[vi * MLA_HG + mi * 16 + g] = l_run[0];
    lsum[vi * MLA_HG + mi * 16 + g + 8] = l_run[1];
  }
  __syncthreads();
  float l_tot[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) l_tot[i] = l_run[i] + lsum[(vi ^ 1) * MLA_HG + mi * 16 + g + i * 8];

#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int h = h0 + mi * 16 + g + i * 8;
    if (h >= H) continue;
    if (sp.n_splits == 1) {
      const float inv = l_tot[i] > 0.f ? 1.f / l_tot[i] : 0.f;
      __nv_bfloat16* og = (__nv_bfloat16*)p.out + ((int64_t)r * H + h) * MLA_DV + vi * 256;
#pragma unroll
      for (int n = 0; n < 32; ++n) {
        __nv_bfloat162 v = __floats2bfloat162_rn(o[n][2 * i] * inv, o[n][2 * i + 1] * inv);
        *(__nv_bfloat162*)(og + n * 8 + t4 * 2) = v;
      }
      if (p.lse && vi == 0 && t4 == 0)
        p.lse[(int64_t)r * H + h] = l_tot[i] > 0.f ? (m_run[i] + log2f(l_tot[i])) / LOG2E : -INFINITY;
    } else {
      float* po = part_o + (((int64_t)r * H + h) * sp.n_splits + split) * MLA_DV + vi * 256;
#pragma unroll
      for (int n = 0; n < 32; ++n)
        *(float2*)(po + n * 8 + t4 * 2) = make_float2(o[n][2 * i], o[n][2 * i + 1]);
      if (vi == 0 && t4 == 0) {
        float* ml = part_ml + (((int64_t)r * H + h) * sp.n_splits + split) * 2;
        ml[0] = m_run[i];
        ml[1] = l_tot[i];
      }
    }
  }
}

// Merge split partials: o = sum_s 2^(m_s - m) o_s / sum_s 2^(m_s - m) l_s.  The partials carry
// `halves` (max, sum) pairs per split: with 2, the two halves of the value dims were accumulated
// with their own maxima and sums, and each half is merged with its own.
template <typename OutT>
__global__ void mla_combine_kernel(MlaPlan p, int n_splits, int halves, const float* __restrict__ part_o,
                                   const float* __restrict__ part_ml) {
  griddep_wait();                // the previous kernel's writes are visible from here on
  griddep_launch_dependents();
  const int64_t rh = blockIdx.x;   // r * H + h
  const float* ml = part_ml + rh * n_splits * halves * 2;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  for (int v = 0; v < halves; ++v) {
    for (int s = 0; s < n_splits; ++s) m[v] = fmaxf(m[v], ml[(s * halves + v) * 2]);
    for (int s = 0; s < n_splits; ++s) {
      const float ms = ml[(s * halves + v) * 2];
      if (ms != -INFINITY) l[v] += exp2f(ms - m[v]) * ml[(s * halves + v) * 2 + 1];
    }
  }
  const int dh = p.d_v / halves;
  for (int d = threadIdx.x; d < p.d_v; d += blockDim.x) {
    const int v = halves == 2 && d >= dh ? 1 : 0;
    float acc = 0.f;
    for (int s = 0; s < n_splits; ++s) {
      const float ms = ml[(s * halves + v) * 2];
      if (ms != -INFINITY) acc += exp2f(ms - m[v]) * part_o[(rh * n_splits + s) * p.d_v + d];
    }
    const float inv = l[v] > 0.f ? 1.f / l[v] : 0.f;
    OutT* og = (OutT*)p.out + rh * p.d_v + d;
    if constexpr (sizeof(OutT) == 2) *og = __float2bfloat16_rn(acc * inv);
    else *og = acc * inv;
  }
  if (threadIdx.x == 0 && p.lse) p.lse[rh] = l[0] > 0.f ? (m[0] + log2f(l[0])) / LOG2E : -INFINITY;
}

// The same merge for 512 value dims with 16-byte accesses: four heads per
// 256-thread block, 64 threads per head, 8 dims per thread; one weight
// 2^(m_s - m) per split.
template <typename OutT>
__global__ void __launch_bounds__(256) mla_combine512_kernel(MlaPlan p, int n_splits, int halves,
                                                             const float* __restrict__ part_o,
                                                             const float* __restrict__ part_ml) {
  griddep_wait();                // the previous kernel's writes are visible from here on
  griddep_launch_dependents();
  const int64_t rh = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 6);
  if (rh >= (int64_t)p.R * p.H) return;
  const int t = threadIdx.x & 63;
  // dims 8t..8t+7 lie in value half t / 32 when the halves carry their own (max, sum)
  const int ms_stride = halves * 2;
  const float* ml = part_ml + rh * n_splits * ms_stride + (halves == 2 ? (t >> 5) * 2 : 0);
  float m = -INFINITY;
  for (int s = 0; s < n_splits; ++s) m = fmaxf(m, ml[s * ms_stride]);
  float l = 0.f;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int s = 0; s < n_splits; ++s) {
    const float ms = ml[s * ms_stride];
    if (ms == -INFINITY) continue;
    const float w = exp2f(ms - m);
    l += w * ml[s * ms_stride + 1];
    const float4* src = (const float4*)(part_o + (rh * n_splits + s) * MLA_DV) + 2 * t;
    const float4 a = src[0], b = src[1];
    acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
    acc[4] += w * b.x; acc[5] += w * b.y; acc[6] += w * b.z; acc[7] += w * b.w;
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  if constexpr (sizeof(OutT) == 2) {
    uint32_t w4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 v = __floats2bfloat162_rn(acc[2 * i] * inv, acc[2 * i + 1] * inv);
      w4[i] = *(uint32_t*)&v;
    }
    *((uint4*)((__nv_bfloat16*)p.out + rh * MLA_DV) + t) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
  } else {
    float4* dst = (float4*)((float*)p.out + rh * MLA_DV) + 2 * t;
    dst[0] = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    dst[1] = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
  }
  if (t == 0 && p.lse) p.lse[rh] = l > 0.f ? (m + log2f(l)) / LOG2E : -INFINITY;
}

template <typename OutT>
static int launch_combine(const MlaPlan& p, int n_splits, int halves, const float* part_o, const float* part_ml,
                          cudaStream_t st) {
  const int64_t rh = (int64_t)p.R * p.H;
  if (p.d_v == MLA_DV && ((uintptr_t)p.out % 16) == 0) {
    launch_k(mla_combine512_kernel<OutT>, (unsigned)((rh + 3) / 4), 256, 0, st, p, n_splits, halves, part_o, part_ml);
  } else {
    launch_k(mla_combine_kernel<OutT>, (unsigned)rh, 128, 0, st, p, n_splits, halves, part_o, part_ml);
  }
  return check_launch("sparse_mla_combine");
}

// float32 path: one CTA per (row, head, split); logits of the split in shared.
__global__ void __launch_bounds__(256) sparse_mla_f32_kernel(MlaPlan p, MlaSplit sp, float* __restrict__ part_o,
                                                              float* __restrict__ part_ml) {
  griddep_wait();                // the previous kernel's writes are visible from here on
  griddep_launch_dependents();
  extern __shared__ float fsm[];
  const int r = blockIdx.x, h = blockIdx.y, split = blockIdx.z;
  const int H = p.H, DL = p.d_latent, DV = p.d_v;
  const int b = request_of_row(p.row_offsets, p.B, (uint32_t)r);
  const int64_t limit = p.row_pos[r] + p.row_pos_add;
  const int64_t total = (int64_t)p.n_idx + p.n_append;
  const int64_t j0 = (int64_t)split * sp.per_split;
  const int64_t j1 = min(total, j0 + sp.per_split);
  const int n = (int)max(j1 - j0, (int64_t)0);
  float* qs = fsm;                 // [DL]
  float* logit = qs + DL;          // [n]
  int64_t* rows = (int64_t*)(logit + ((n + 1) & ~1));
  __shared__ float red[32];
  const float* q = (const float*)p.q + ((int64_t)r * H + h) * DL;
  const float* lat = (const float*)p.latent;
  for (int d = threadIdx.x; d < DL; d += blockDim.x) qs[d] = q[d];
  for (int j = threadIdx.x; j < n; j += blockDim.x) rows[j] = mla_pool_row(p, r, b, j0 + j, limit);
  __syncthreads();
  const float sl2 = p.scale * LOG2E;
  // one warp per logit
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int j = warp; j < n; j += nw) {
    float acc = 0.f;
    if (rows[j] >= 0) {
      const float* c = lat + rows[j] * DL;
      for (int d = lane; d < DL; d += 32) acc = fmaf(qs[d], c[d], acc);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) logit[j] = rows[j] >= 0 ? acc * sl2 : -INFINITY;
  }
  __syncthreads();
  float m = -INFINITY;
  for (int j = threadIdx.x; j < n; j += blockDim.x) m = fmaxf(m, logit[j]);
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  m = -INFINITY;
  for (int w = 0; w < nw; ++w) m = fmaxf(m, red[w]);
  __syncthreads();
  float l = 0.f;
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    float e = (m == -INFINITY || logit[j] == -INFINITY) ? 0.f : exp2f(logit[j] - m);
    logit[j] = e;
    l += e;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  if (lane == 0) red[warp] = l;
  __syncthreads();
  l = 0.f;
  for (int w = 0; w < nw; ++w) l += red[w];
  for (int d = threadIdx.x; d < DV; d += blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < n; ++j)
      if (rows[j] >= 0) acc = fmaf(logit[j], lat[rows[j] * DL + d], acc);
    if (sp.n_splits == 1) {
      ((float*)p.out)[((int64_t)r * H + h) * DV + d] = l > 0.f ? acc / l : 0.f;
    } else {
      part_o[(((int64_t)r * H + h) * sp.n_splits + split) * DV + d] = acc;
    }
  }
  if (threadIdx.x == 0) {
    if (sp.n_splits == 1) {
      if (p.lse) p.lse[(int64_t)r * H + h] = l > 0.f ? (m + log2f(l)) / LOG2E : -INFINITY;
    } else {
      float* ml = part_ml + (((int64_t)r * H + h) * sp.n_splits + split) * 2;
      ml[0] = m;
      ml[1] = l;
    }
  }
}

static MlaSplit choose_split(int R, int H, int n_idx, int n_append, int dtype) {
  int64_t total = (int64_t)n_idx + n_append;
  MlaSplit sp;
  int64_t ctas = (int64_t)R * (dtype != MTPSD_F32 ? ceil_div(H, MLA_HG) : H);
  int64_t want = ctas >= 2 * num_sms() ? 1 : ceil_div(2 * num_sms(), ctas);
  int64_t by_len = ceil_div(total, 256);
  int64_t ns = want < by_len ? want : by_len;
  int64_t min_ns = ceil_div(total, MLA_MAX_SPLIT);
  if (ns < min_ns) ns = min_ns;
  if (ns < 1) ns = 1;
  sp.per_split = ceil_div(ceil_div(total, ns), MLA_NT) * MLA_NT;
  if (sp.per_split < MLA_NT) sp.per_split = MLA_NT;
  sp.n_splits = (int)ceil_div(total, sp.per_split);
  if (sp.n_splits < 1) sp.n_splits = 1;
  return sp;
}

static bool use_tc(int H, int dtype) {
  MlaPlan q{};
  q.H = H; q.dtype = dtype; q.d_latent = MLA_DL; q.d_v = MLA_DV;
  return mla_tc_supported(q);
}

// splits of the selected list for the tensor-core kernel
static MlaSplit plan_split_tc(int R, int H, int n_idx, int n_append) {
  int64_t total = (int64_t)n_idx + n_append;
  MlaSplit sp;
  sp.per_split = mla_tc_per_split(R, H, total);
  sp.n_splits = total > 0 ? (int)ceil_div(total, sp.per_split) : 1;
  return sp;
}

// splits of the selected list for the kernel that will run: the tensor-core kernel's own plan, or the
// portable kernels' (at most MLA_MAX_SPLIT positions per split)
static MlaSplit plan_split(int R, int H, int n_idx, int n_append, int dtype, bool tc) {
  return tc ? plan_split_tc(R, H, n_idx, n_append) : choose_split(R, H, n_idx, n_append, dtype);
}

int mla_launch_count(int R, int H, int n_idx, int n_append, int dtype) {
  if (R <= 0) return 0;
  const bool tc = use_tc(H, dtype);
  MlaPersist pl;
  if (tc && mla_tc_persist_plan(R, H, (int64_t)n_idx + n_append, dtype, &pl)) return pl.cut ? 2 : 1;
  MlaSplit sp = plan_split(R, H, n_idx, n_append, dtype, tc);
  if (sp.n_splits <= 1) return 1;
  if (tc && mla_tc_fuse(sp.n_splits)) return 1;
  return 2;
}

static size_t split_bytes(int R, int H, const MlaSplit& sp) {
  if (sp.n_splits == 1) return 0;
  size_t rh = (size_t)R * H * sp.n_splits;
  return rh * MLA_DV * sizeof(float) + rh * 4 * sizeof(float) + 256;   // up to two (max, sum) pairs per split
}

// Covers both kernels: a call whose buffers miss the tensor-core kernel's alignment runs the portable one.
size_t mla_workspace_bytes(int R, int H, int n_idx, int n_append, int dtype) {
  size_t n = split_bytes(R, H, plan_split(R, H, n_idx, n_append, dtype, false));
  if (use_tc(H, dtype)) {
    const size_t t = split_bytes(R, H, plan_split(R, H, n_idx, n_append, dtype, true));
    if (t > n) n = t;
    MlaPersist pl;
    if (mla_tc_persist_plan(R, H, (int64_t)n_idx + n_append, dtype, &pl) && mla_tc_persist_bytes(pl) > n)
      n = mla_tc_persist_bytes(pl);
  }
  return n;
}

int launch_sparse_mla(const MlaPlan& p, cudaStream_t st) {
  if (p.R == 0) return MTPSD_OK;
  // the kernel is decided once, and the split plan is that kernel's
  const bool tc = mla_tc_supported(p);
  MlaPersist pl;
  if (tc && mla_tc_persist_plan(p.R, p.H, (int64_t)p.n_idx + p.n_append, p.dtype, &pl)) {
    const size_t need = mla_tc_persist_bytes(pl);
    if (need && (!p.ws || p.ws_bytes < need)) {
      set_error("sparse_mla_decode: workspace of %zu bytes needed, %zu given", need, p.ws_bytes);
      return MTPSD_EWORKSPACE;
    }
    return launch_sparse_mla_tc(p, 1, 0, nullptr, nullptr, st, nullptr, &pl);
  }
  MlaSplit sp = plan_split(p.R, p.H, p.n_idx, p.n_append, p.dtype, tc);
  float* part_o = nullptr;
  float* part_ml = nullptr;
  if (sp.n_splits > 1) {
    size_t need = split_bytes(p.R, p.H, sp);
    if (!p.ws || p.ws_bytes < need) {
      set_error("sparse_mla_decode: workspace of %zu bytes needed, %zu given", need, p.ws_bytes);
      return MTPSD_EWORKSPACE;
    }
    part_o = (float*)p.ws;
    part_ml = part_o + (size_t)p.R * p.H * sp.n_splits * MLA_DV;
  }
  if (tc) {   // bf16 or the FP8 latent rows (dequantized by the producers)
    bool combined = false;
    int rc = launch_sparse_mla_tc(p, sp.n_splits, (int)sp.per_split, part_o, part_ml, st, &combined);
    if (rc) return rc;
    if (sp.n_splits > 1 && !combined) {
      return launch_combine<__nv_bfloat16>(p, sp.n_splits, mla_tc_ml_halves(), part_o, part_ml, st);
    }
    return MTPSD_OK;
  }
  if (p.dtype == MTPSD_BF16 || p.dtype == MTPSD_FP8_DS_MLA) {
    const bool fp8kv = p.dtype == MTPSD_FP8_DS_MLA;
    static std::atomic<uint64_t> attr{0}, attr8{0};
    if (!(fp8kv ? set_smem_limit_once(sparse_mla_bf16_kernel<true>, MlaSmemT<true>::BYTES, attr8)
                : set_smem_limit_once(sparse_mla_bf16_kernel<false>, MlaSmem::BYTES, attr))) {
      set_error("sparse_mla_bf16: cudaFuncSetAttribute failed");
      return MTPSD_ECUDA;
    }
    dim3 grid(p.R, (unsigned)ceil_div(p.H, MLA_HG), sp.n_splits);
    if (fp8kv)
      launch_k(sparse_mla_bf16_kernel<true>, grid, 256, MlaSmemT<true>::BYTES, st, p, sp, part_o, part_ml);
    else
      launch_k(sparse_mla_bf16_kernel<false>, grid, 256, MlaSmem::BYTES, st, p, sp, part_o, part_ml);
    int rc = check_launch("sparse_mla_bf16");
    if (rc) return rc;
    if (sp.n_splits > 1) {
      return launch_combine<__nv_bfloat16>(p, sp.n_splits, 1, part_o, part_ml, st);
    }
    return MTPSD_OK;
  }
  // float32
  size_t smem = sizeof(float) * (p.d_latent + ((sp.per_split + 1) & ~1)) + sizeof(int64_t) * sp.per_split;
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(sparse_mla_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  dim3 grid(p.R, p.H, sp.n_splits);
  launch_k(sparse_mla_f32_kernel, grid, 256, smem, st, p, sp, part_o, part_ml);
  int rc = check_launch("sparse_mla_f32");
  if (rc) return rc;
  if (sp.n_splits > 1) {
    return launch_combine<float>(p, sp.n_splits, 1, part_o, part_ml, st);
  }
  return MTPSD_OK;
}

}  // namespace mtpsd
