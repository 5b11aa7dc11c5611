// Per-row top-k without a full sort: radix select of the k-th largest score
// key, then an ordered compaction.
//
// [P3] "Indexer 的结构与计算流程": the fused index kernel returns the top
// index_topk positions per query row; [P2] "验证段的逐层算子" op 6: each row
// selects its own.  Ties at the k-th score go to the lower position; the
// output lists the selected positions in ascending order, -1 padded.
//
// Rows of up to 40960 keys use the register kernel below.  Longer rows: one
// CTA of 1024 threads per row.  Scores map to order-preserving uint32
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

// Exclusive prefix sum over the block (T = int, or uint32_t for the packed two-field counts below,
// whose upper field may reach bit 31: unsigned addition carries no sign).
template <typename T>
__device__ __forceinline__ T block_exclusive_scan(T v, T* warp_sums, T* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  T x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[wid] = x;
  __syncthreads();
  if (wid == 0) {
    T w = (lane < nw) ? warp_sums[lane] : T(0);
    T incl = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      T y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    warp_sums[lane] = incl - w;
    if (lane == 31) *total = incl;
  }
  __syncthreads();
  T res = warp_sums[wid] + x - v;
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(TOPK_THREADS, 1) topk_kernel(TopkPlan p, int64_t cache_cap) {
  griddep_wait();                // the previous kernel's writes are visible from here on
  griddep_launch_dependents();
  extern __shared__ uint32_t keys_s[];
  __shared__ int hist[256];
  __shared__ int warp_sums[32];
  __shared__ int total_s;
  __shared__ uint32_t prefix_s;
  __shared__ int remaining_s;

  const int r = blockIdx.x;
  int64_t V = p.row_len[r] + p.len_add;
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

// Rows of up to 40960 keys: each thread holds KPT consecutive keys in
// registers (positions t*KPT .. t*KPT+KPT-1) and the CTA finds the k-th
// largest key T exactly by a bitwise search: the bits shared by all visible
// keys are T's, and below them T grows by bit b when at least k keys are
// >= T | 2^b (one counting round per bit: a warp reduction, one barrier, and
// a second warp reduction over the per-warp counts).  The ordered compaction
// is the same as above.  With XT, the row may run past KPT*NTH by at most NTH
// keys: thread t also holds the tail key at position KPT*NTH + t (so a row of
// 8198 keys takes 16 keys per thread and a tail of 6, not 20 per thread), and
// the tail keys, whose positions follow every regular one, are compacted after
// them.
//
// Longer rows are split (MODE 1, then 2 or 3, one launch per level).  Level 1 cuts a
// row into segments of SPLIT_SEG keys, one CTA each, and every CTA selects its
// segment's exact top-k under the same order (larger key first, ties to the
// lower position) as a list of k (key, position) entries in position order; a
// segment with fewer than k keys lists all of them, then -1 positions.  Level
// l >= 2 merges groups of G = SPLIT_SEG / k consecutive lists of level l-1 the
// same way.  Every element of a row's top-k is in the top-k of its segment (and
// of its group) under that order, so every level is exact; the lists of a row
// stay in position order (segment u's positions precede segment u+1's), so the
// compaction, which writes in list order, keeps the output ascending.  The level
// at which a row has one list left writes the row's final output.  MODE 3 is MODE 2
// held to 64 registers, so that two CTAs share an SM when there are more rows than SMs.
// 16384-key segments on 512 threads (32 keys each): two CTAs fit one SM, so one CTA's loads and barriers
// overlap the other's counting (one 1024-thread CTA per SM over 32768-key segments was 18 % slower on
// 768 rows of up to 118 K keys, and 256-thread CTAs over 8192-key segments 15 % slower).
constexpr int SPLIT_SEG = 16384;
constexpr int SPLIT_KPT = 32;
constexpr int SPLIT_NTH = 512;
static_assert(SPLIT_SEG == SPLIT_KPT * SPLIT_NTH && SPLIT_SEG >= 2 * 4096, "segments hold two lists of the largest k");

struct SplitLevel {
  int level;                     // 1: segments of the score rows; >= 2: merges of the previous lists
  int G;                         // lists merged per CTA at levels >= 2
  const uint32_t* in_key;        // previous level's lists, in_stride entries per row
  const int32_t* in_pos;
  int64_t in_stride;
  uint32_t* out_key;             // this level's lists (when not final), out_stride entries per row
  int32_t* out_pos;
  int64_t out_stride;
};

// Shape of a row of V keys at a level: n lists, the last holding last_valid valid entries (every
// other list holds k); n_prev / prev_last_valid describe level - 1 (0 at level 1).
__host__ __device__ __forceinline__ void split_shape(int64_t V, int k, int G, int level, int& n, int& last_valid,
                                                     int& n_prev, int& prev_last_valid) {
  n = V > 0 ? (int)((V + SPLIT_SEG - 1) / SPLIT_SEG) : 1;
  const int64_t tail = V - (int64_t)(n - 1) * SPLIT_SEG;
  last_valid = (int)(tail < k ? (tail > 0 ? tail : 0) : k);
  n_prev = 0;
  prev_last_valid = 0;
  for (int l = 2; l <= level; ++l) {
    n_prev = n;
    prev_last_valid = last_valid;
    const int nn = (n + G - 1) / G;
    const int m = n - (nn - 1) * G;   // lists in the last group
    const int cnt = (m - 1) * k + prev_last_valid;
    last_valid = cnt < k ? cnt : k;
    n = nn;
  }
}

template <int KPT, int NTH, bool XT, int MODE>
__global__ void __launch_bounds__(NTH, MODE == 3 ? 2 : 0) topk_reg_kernel(TopkPlan p, SplitLevel sl) {
  griddep_wait();                // the previous kernel's writes are visible from here on
  griddep_launch_dependents();
  static_assert(MODE == 0 || !XT, "tail keys only for whole rows");
  __shared__ int wsum[2][32];
  __shared__ int warp_sums[32];
  __shared__ int total_s;
  __shared__ uint32_t uwarp_sums[32];
  __shared__ uint32_t utotal_s;
  const int r = blockIdx.x;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  constexpr int NW = NTH / 32;
  int64_t Vrow = p.row_len[r] + p.len_add;
  if (Vrow > p.max_len) {
    if (threadIdx.x == 0 && (MODE == 0 || (sl.level == 1 && blockIdx.y == 0))) flag_status(p.status, MTPSD_STATUS_INDEX_RANGE);
    Vrow = p.max_len;
  }
  if (Vrow < 0) Vrow = 0;
  const int k = p.k;
  // this CTA's keys: V of them, from a score row (MODE 0, 1) or a list of (key, position) (MODE 2, 3)
  const float* row = nullptr;
  const uint32_t* krow = nullptr;
  const int32_t* prow = nullptr;
  int64_t pos_base = 0, lim = 0;
  int V;
  bool fin = true;
  int32_t* opos = p.out_idx + (int64_t)r * k;                       // final: positions and scores
  float* oscore = p.out_score ? p.out_score + (int64_t)r * k : nullptr;
  uint32_t* okey = nullptr;                                         // intermediate: keys and positions
  if constexpr (MODE == 0) {
    V = (int)Vrow;
    row = p.scores + (int64_t)r * p.ld;
    lim = p.ld;
  } else {
    int n, lv, np, plv;
    split_shape(Vrow, k, sl.G, sl.level, n, lv, np, plv);
    const int u = blockIdx.y;
    if (MODE >= 2 && np <= 1) return;   // the row was finished at an earlier level
    if (u >= n) return;
    fin = n == 1;
    if constexpr (MODE == 1) {
      pos_base = (int64_t)u * SPLIT_SEG;
      V = (int)min((int64_t)SPLIT_SEG, Vrow - pos_base);
      if (V < 0) V = 0;
      row = p.scores + (int64_t)r * p.ld + pos_base;
      lim = p.ld - pos_base;
    } else {
      const int m = u < n - 1 ? sl.G : np - (n - 1) * sl.G;   // lists in this group
      V = u < n - 1 ? sl.G * k : (m - 1) * k + plv;
      krow = sl.in_key + (int64_t)r * sl.in_stride + (int64_t)u * sl.G * k;
      prow = sl.in_pos + (int64_t)r * sl.in_stride + (int64_t)u * sl.G * k;
      lim = (int64_t)m * k;
    }
    if (!fin) {
      okey = sl.out_key + (int64_t)r * sl.out_stride + (int64_t)u * k;
      opos = sl.out_pos + (int64_t)r * sl.out_stride + (int64_t)u * k;
      oscore = nullptr;
    }
  }
  auto pos_of = [&](int i) -> int32_t {
    if constexpr (MODE >= 2) return prow[i];
    else return (int32_t)(pos_base + i);
  };
  auto emit = [&](int slot, int i, uint32_t kv) {
    opos[slot] = pos_of(i);
    if (okey) okey[slot] = kv;
    else if (oscore) oscore[slot] = key_float(kv);
  };
  if (V <= k) {  // everything is selected
    for (int i = threadIdx.x; i < k; i += blockDim.x) {
      if (i < V) {
        uint32_t kv;
        if constexpr (MODE >= 2) kv = krow[i];
        else kv = float_key(row[i]);
        emit(i, i, kv);
      } else {
        opos[i] = -1;
        if (okey) okey[i] = 0u;
        else if (oscore) oscore[i] = -INFINITY;
      }
    }
    return;
  }
  // keys of this thread's entries; 0 (below every finite key) past the end
  const int a = threadIdx.x * KPT;
  uint32_t key[KPT];
  if constexpr (MODE >= 2) {
    if ((k & 3) == 0) {   // 16-byte aligned lists (k and the row stride are multiples of 4)
#pragma unroll
      for (int i = 0; i < KPT; i += 4) {
        uint4 f = make_uint4(0u, 0u, 0u, 0u);
        if (a + i < lim) f = *(const uint4*)(krow + a + i);
        key[i] = a + i < V ? f.x : 0u;
        key[i + 1] = a + i + 1 < V ? f.y : 0u;
        key[i + 2] = a + i + 2 < V ? f.z : 0u;
        key[i + 3] = a + i + 3 < V ? f.w : 0u;
      }
    } else {
#pragma unroll
      for (int i = 0; i < KPT; ++i) key[i] = a + i < V ? krow[a + i] : 0u;
    }
  } else {
#pragma unroll
    for (int i = 0; i < KPT; i += 4) {
      float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
      if (a + i < lim) f = *(const float4*)(row + a + i);   // ld is a multiple of 4 and rows are 16-byte aligned
      key[i] = a + i < V ? float_key(f.x) : 0u;
      key[i + 1] = a + i + 1 < V ? float_key(f.y) : 0u;
      key[i + 2] = a + i + 2 < V ? float_key(f.z) : 0u;
      key[i + 3] = a + i + 3 < V ? float_key(f.w) : 0u;
    }
  }
  const int ax = KPT * NTH + threadIdx.x;   // this thread's tail position (XT)
  const bool xv = XT && ax < V;
  const uint32_t xkey = xv ? float_key(row[ax]) : 0u;
  // bits shared by every visible key (the sign and most exponent bits of these
  // scores) are T's as well; the search starts below them
  uint32_t kand = ~0u, kor = 0u;
#pragma unroll
  for (int i = 0; i < KPT; ++i)
    if (a + i < V) {
      kand &= key[i];
      kor |= key[i];
    }
  if (xv) {
    kand &= xkey;
    kor |= xkey;
  }
  kand = __reduce_and_sync(0xffffffffu, kand);
  kor = __reduce_or_sync(0xffffffffu, kor);
  if (lane == 0) {
    wsum[0][wid] = (int)kand;
    wsum[1][wid] = (int)kor;
  }
  __syncthreads();
  kand = __reduce_and_sync(0xffffffffu, lane < NW ? (uint32_t)wsum[0][lane] : ~0u);
  kor = __reduce_or_sync(0xffffffffu, lane < NW ? (uint32_t)wsum[1][lane] : 0u);
  __syncthreads();   // wsum is reused below
  const uint32_t diff = kand ^ kor;
  const int b0 = diff ? 31 - __clz(diff) : -1;   // highest bit where visible keys differ
  uint32_t T = b0 >= 31 ? 0u : (b0 < 0 ? kand : (kand & (~0u << (b0 + 1))));
  // Eleven bits at a time, the last level taking what is left (1 to 11 bits): a 2048-bin histogram of
  // the level's bits of the keys that share T's bits above it (keys above that prefix are only
  // counted), then the bin where the count from the top reaches k; after the last level T is the k-th
  // largest key.  Thread t owns bins BPT*t .. BPT*t+BPT-1.  The keys past the row's end are 0, below
  // every key of a finite score, and there are more than k valid keys, so counting them (in the lowest
  // bin, when the prefix is 0) never moves the k-th largest: no validity test per key.  The increment is
  // a predicated shared-memory reduction, so that the per-key work has no branch.
  constexpr int BPT = 2048 / NTH;
  __shared__ int hist[2048];
  __shared__ int dsel;
  const uint32_t hist_s = (uint32_t)__cvta_generic_to_shared(hist);
  int bl = b0;
#pragma unroll 1
  while (bl >= 0) {
    const int nb = bl >= 10 ? 11 : bl + 1;   // bits of this level: bl - nb + 1 .. bl
    const int sh = bl + 1 - nb;
    const uint32_t bmask = (1u << nb) - 1u;
    const uint32_t sh1 = (uint32_t)(bl + 1);   // the prefix above the level (32: none)
#pragma unroll
    for (int e = 0; e < BPT; ++e) hist[threadIdx.x * BPT + e] = 0;
    __syncthreads();
    const uint32_t preT = __funnelshift_rc(T, 0u, sh1);
    int above = 0;
    auto put = [&](uint32_t kv) {
      const uint32_t pre = __funnelshift_rc(kv, 0u, sh1);
      above += pre > preT ? 1 : 0;
      const uint32_t addr = hist_s + (((kv >> sh) & bmask) << 2);
      asm volatile("{\n .reg .pred q;\n setp.eq.u32 q, %1, %2;\n @q red.shared.add.u32 [%0], 1;\n}\n"
                   ::"r"(addr), "r"(pre), "r"(preT) : "memory");
    };
#pragma unroll
    for (int i = 0; i < KPT; ++i) put(key[i]);
    if constexpr (XT) put(xkey);
    __syncthreads();
    int hv[BPT], lsum = 0;
#pragma unroll
    for (int e = 0; e < BPT; ++e) {
      hv[e] = hist[threadIdx.x * BPT + e];
      lsum += hv[e];
    }
    // both fields stay below 65536 (at most 41984 keys, padding included): one unsigned scan carries
    // the bin counts in the low half and the keys above the prefix in the high half
    const uint32_t pk = block_exclusive_scan<uint32_t>((uint32_t)lsum | ((uint32_t)above << 16), uwarp_sums, &utotal_s);
    const int tot = (int)(utotal_s & 0xffffu), A = (int)(utotal_s >> 16);
    const int U = A + tot - (int)(pk & 0xffffu) - lsum;   // keys in the bins above this thread's, and above the prefix
    if (U < k && k <= U + lsum) {
      int run = U, d = threadIdx.x * BPT;
#pragma unroll
      for (int e = BPT - 1; e >= 0; --e) {
        run += hv[e];
        if (run >= k) {
          d = threadIdx.x * BPT + e;
          break;
        }
      }
      dsel = d;
    }
    __syncthreads();
    T |= (uint32_t)dsel << sh;
    bl -= nb;
  }
  int n_gt = 0, n_eq = 0;
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    n_gt += key[i] > T;
    n_eq += key[i] == T;
  }
  if constexpr (XT) {
    // counts of the regular keys and of the tail keys, each as two 16-bit fields (> T, == T) of an
    // unsigned word: every total is below 65536 (at most 40960 keys), so one scan carries both fields
    // without a carry, and the upper field may use bit 31 (32768 or more equal keys)
    const int xg = xkey > T, xe = xv && xkey == T;
    const uint32_t pr = block_exclusive_scan<uint32_t>((uint32_t)n_gt | ((uint32_t)n_eq << 16), uwarp_sums, &utotal_s);
    const uint32_t tr = utotal_s;
    const uint32_t px = block_exclusive_scan<uint32_t>((uint32_t)xg | ((uint32_t)xe << 16), uwarp_sums, &utotal_s);
    const uint32_t tx = utotal_s;
    const int gt_before = (int)(pr & 0xffffu), eq_before = (int)(pr >> 16);
    const int tot_gt = (int)(tr & 0xffffu) + (int)(tx & 0xffffu);
    const int tot_eq_r = (int)(tr >> 16);
    const int need_eq = k - tot_gt;   // equal keys taken, lowest positions first: regular ones, then the tail
    int take_eq = max(0, min(n_eq, need_eq - eq_before));
    int out_pos = gt_before + min(eq_before, need_eq);
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
      bool take = key[i] > T;
      if (key[i] == T && take_eq > 0) {
        take = true;
        --take_eq;
      }
      if (take && out_pos < k) {
        emit(out_pos, a + i, key[i]);
        ++out_pos;
      }
    }
    const int need_eq_x = max(0, need_eq - tot_eq_r);
    const int gx_before = (int)(px & 0xffffu), ex_before = (int)(px >> 16);
    const int x_pos = (int)(tr & 0xffffu) + min(tot_eq_r, need_eq) + gx_before + min(ex_before, need_eq_x);
    if ((xg || (xe && ex_before < need_eq_x)) && x_pos < k) emit(x_pos, ax, xkey);
    return;
  }
  const int gt_before = block_exclusive_scan(n_gt, warp_sums, &total_s);
  const int need_eq = k - total_s;   // equal keys taken, lowest positions first
  const int eq_before = block_exclusive_scan(n_eq, warp_sums, &total_s);
  int take_eq = max(0, min(n_eq, need_eq - eq_before));
  int out_pos = gt_before + min(eq_before, need_eq);
  if constexpr (MODE >= 2) {
    // merged lists carry their positions: eight of this thread's are loaded together before they are
    // emitted, instead of one dependent load per emitted entry
#pragma unroll
    for (int c0 = 0; c0 < KPT; c0 += 8) {
      int32_t pv[8];
      if ((k & 3) == 0 && a + c0 + 8 <= lim) {
        const int4 v0 = *(const int4*)(prow + a + c0), v1 = *(const int4*)(prow + a + c0 + 4);
        pv[0] = v0.x; pv[1] = v0.y; pv[2] = v0.z; pv[3] = v0.w;
        pv[4] = v1.x; pv[5] = v1.y; pv[6] = v1.z; pv[7] = v1.w;
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) pv[j] = a + c0 + j < lim ? prow[a + c0 + j] : -1;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = c0 + j;
        bool take = key[i] > T;
        if (key[i] == T && take_eq > 0) {
          take = true;
          --take_eq;
        }
        if (take && out_pos < k) {
          opos[out_pos] = pv[j];
          if (okey) okey[out_pos] = key[i];
          else if (oscore) oscore[out_pos] = key_float(key[i]);
          ++out_pos;
        }
      }
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    bool take = key[i] > T;
    if (key[i] == T && take_eq > 0) {
      take = true;
      --take_eq;
    }
    if (take && out_pos < k) {
      emit(out_pos, a + i, key[i]);
      ++out_pos;
    }
  }
}

template <int NTH, bool XT>
static int launch_topk_reg(const TopkPlan& p, int kpt, cudaStream_t st) {
  const SplitLevel none = {};
  switch (kpt) {
#define MTPSD_TOPK_CASE(K) \
  case K: launch_k(topk_reg_kernel<K, NTH, XT, 0>, p.R, NTH, 0, st, p, none); break;
    MTPSD_TOPK_CASE(4) MTPSD_TOPK_CASE(8) MTPSD_TOPK_CASE(12) MTPSD_TOPK_CASE(16) MTPSD_TOPK_CASE(20)
    MTPSD_TOPK_CASE(24) MTPSD_TOPK_CASE(28) MTPSD_TOPK_CASE(32) MTPSD_TOPK_CASE(36) MTPSD_TOPK_CASE(40)
#undef MTPSD_TOPK_CASE
    default: return -1;
  }
  return check_launch("topk");
}

// Levels of the split top-k for rows up to max_len keys: lists per row at each level (the largest
// row's), until one list is left.  Returns the number of levels (>= 2 when max_len > SPLIT_SEG).
static int split_levels(int64_t max_len, int k, int* n_at, int max_levels) {
  const int G = SPLIT_SEG / k;
  int n = (int)((max_len + SPLIT_SEG - 1) / SPLIT_SEG);
  if (n < 1) n = 1;
  int L = 0;
  n_at[L++] = n;
  while (n > 1 && L < max_levels) {
    n = (n + G - 1) / G;
    n_at[L++] = n;
  }
  return L;
}

static bool split_path(const TopkPlan& p) {
  const bool aligned = ((uintptr_t)p.scores % 16) == 0 && (p.ld % 4) == 0;
  return aligned && p.max_len > 40960;
}

// Workspace of the split top-k: two list buffers per row (levels alternate between them), each list
// k entries of a uint32 key and an int32 position; row strides are multiples of 4 entries.
size_t topk_workspace_bytes(int R, int64_t max_len, int k) {
  if (R <= 0 || k < 1 || max_len <= 40960) return 0;
  int n_at[8];
  const int L = split_levels(max_len, k, n_at, 8);
  if (L < 2) return 0;
  const int64_t strideA = ((int64_t)n_at[0] * k + 3) & ~3LL;
  const int64_t strideB = L > 2 ? (((int64_t)n_at[1] * k + 3) & ~3LL) : 0;
  const size_t a = ((size_t)R * strideA * 8 + 255) / 256 * 256;
  const size_t b = ((size_t)R * strideB * 8 + 255) / 256 * 256;
  return a + b;
}

int topk_launch_count(int64_t max_len, int k, bool aligned) {
  if (!aligned || max_len <= 40960) return 1;
  int n_at[8];
  return split_levels(max_len, k, n_at, 8);
}

static int launch_topk_split(const TopkPlan& p, cudaStream_t st) {
  int n_at[8];
  const int L = split_levels(p.max_len, p.k, n_at, 8);
  const size_t need = topk_workspace_bytes(p.R, p.max_len, p.k);
  if (!p.ws || p.ws_bytes < need) {
    set_error("topk: rows longer than 40960 keys need a workspace of %zu bytes (%zu given)", need, p.ws_bytes);
    return MTPSD_EWORKSPACE;
  }
  const int64_t strideA = ((int64_t)n_at[0] * p.k + 3) & ~3LL;
  const int64_t strideB = L > 2 ? (((int64_t)n_at[1] * p.k + 3) & ~3LL) : 0;
  uint32_t* keyA = (uint32_t*)p.ws;
  int32_t* posA = (int32_t*)(keyA + (size_t)p.R * strideA);
  char* bbase = (char*)p.ws + ((size_t)p.R * strideA * 8 + 255) / 256 * 256;
  uint32_t* keyB = (uint32_t*)bbase;
  int32_t* posB = (int32_t*)(keyB + (size_t)p.R * strideB);
  SplitLevel sl = {};
  sl.G = SPLIT_SEG / p.k;
  for (int l = 1; l <= L; ++l) {
    // level l writes buffer A when odd, B when even, and reads the other one
    const bool odd = (l & 1) != 0;
    sl.level = l;
    sl.out_key = odd ? keyA : keyB;
    sl.out_pos = odd ? posA : posB;
    sl.out_stride = odd ? strideA : strideB;
    sl.in_key = odd ? keyB : keyA;
    sl.in_pos = odd ? posB : posA;
    sl.in_stride = odd ? strideB : strideA;
    const dim3 grid(p.R, n_at[l - 1]);
    if (l == 1)
      launch_k(topk_reg_kernel<SPLIT_KPT, SPLIT_NTH, false, 1>, grid, SPLIT_NTH, 0, st, p, sl);
    else if (p.R > num_sms())   // more rows than SMs: two CTAs per SM (64 registers) outrun one faster CTA
      launch_k(topk_reg_kernel<SPLIT_KPT, SPLIT_NTH, false, 3>, grid, SPLIT_NTH, 0, st, p, sl);
    else
      launch_k(topk_reg_kernel<SPLIT_KPT, SPLIT_NTH, false, 2>, grid, SPLIT_NTH, 0, st, p, sl);
    const int rc = check_launch("topk_split");
    if (rc) return rc;
  }
  return MTPSD_OK;
}

int launch_topk(const TopkPlan& p, cudaStream_t st) {
  if (p.R == 0) return MTPSD_OK;
  const bool aligned = ((uintptr_t)p.scores % 16) == 0 && (p.ld % 4) == 0;
  if (aligned && p.max_len <= 40960) {
    // 512 threads per row up to 16384 keys, unless there are too few rows to fill the SMs: then
    // 1024 threads hold fewer keys each and every counting round is shorter
    const int nth = (p.max_len <= 16384 && p.R > num_sms() / 2) ? 512 : 1024;
    // keys per thread in registers (a multiple of 4 for the 16-byte loads), plus one tail key per
    // thread when that covers the rest of the row
    const int kdown = (int)(p.max_len / nth) & ~3;
    const bool xt = kdown >= 4 && p.max_len - (int64_t)kdown * nth <= nth && p.max_len > (int64_t)kdown * nth;
    int kpt = xt ? kdown : (int)((p.max_len + nth - 1) / nth);
    kpt = (kpt + 3) & ~3;
    if (kpt < 4) kpt = 4;
    if (nth == 512 && kpt <= 32) return xt ? launch_topk_reg<512, true>(p, kpt, st) : launch_topk_reg<512, false>(p, kpt, st);
    if (nth == 1024 && kpt <= 40) return xt ? launch_topk_reg<1024, true>(p, kpt, st) : launch_topk_reg<1024, false>(p, kpt, st);
  }
  if (split_path(p)) return launch_topk_split(p, st);
  // unaligned score rows: one CTA per row, radix passes
  int64_t cache_keys = p.max_len <= TOPK_SMEM_KEYS ? p.max_len : 0;
  size_t smem = (size_t)cache_keys * sizeof(uint32_t);
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  launch_k(topk_kernel, p.R, TOPK_THREADS, smem, st, p, cache_keys);
  return check_launch("topk");
}

}  // namespace mtpsd
