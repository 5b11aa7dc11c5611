// FP8 lightning-indexer score GEMM on the 5th-generation tensor cores
// (tcgen05.mma kind::f8f6f4 + TMEM accumulators + TMA-staged operands).
//
// [P3] "Indexer 的结构与计算流程":
//   I[r,s] = sum_h w[r,h] * ReLU(q_scale[r,h] * k_scale[s] * q[r,h,:].k[s,:])
// Since the scales are positive they commute with the ReLU:
//   I[r,s] = k_scale[s] * sum_h (w[r,h] q_scale[r,h]) * ReLU(q8[r,h,:].k8[s,:])
// so the tensor cores see only FP8 codes and the scales enter the epilogue.
//
// Shape of one MMA: M = 128 cached positions (the A operand: a 128 x 128 B
// key tile, K-major, loaded by TMA with the 128-byte swizzle), N = 64 * c
// query columns (c units of 64 (row, head) columns, c <= 4: the B operand,
// K-major), K = 128 FP8 values in 4 steps of 32.  Putting the positions on M
// makes the head sum of the epilogue thread-local: TMEM lane = position,
// columns = (row, head).
//
// TMEM is a ring of 8 slots of 64 columns; a unit is the 64 columns of one
// slot: one row of 64 heads, or two rows of 32.  A key tile of a group of n
// units takes the next n slots of the ring (their MMAs cover up to 4 adjacent
// slots at once, split where the ring wraps), so a one-row group moves 8 tiles
// ahead of the epilogue and a six-row group 1.3.
//
// Roles (448 threads, one persistent CTA per SM):
//   warps 0-11  epilogue, 3 warpgroups: unit u is taken by warpgroup u % 3, so
//               three units drain at once.  Each warp reads its 32 lanes x 64
//               columns (tcgen05.ld), applies ReLU and the weights (w * q_scale)
//               as (x + |x|) * (w q_scale / 2), two FMA-pipe instructions per
//               value, then the head sum and k_scale, and stores one score per
//               lane and row (coalesced).
//   warp 12     TMA producer: the group's query rows, a 6-stage ring of key
//               tiles, and a 16-stage ring of the tiles' key scales (132 floats
//               from a 4-aligned start, so the copy's first coordinate is
//               16-byte aligned; the epilogue indexes from the remainder).
//   warp 13     TMEM allocation and the MMA issue.
// The producer and MMA roles run with the whole warp (uniform loop state,
// bounded waits taken by all lanes) and one elected lane issues.
// Work: the rows of each request are cut into groups of up to 512/H rows
// (the query block kept in shared memory); each group scans
// ceil(max visible / 128) key tiles; the flattened (group, tile) list is split
// into equal contiguous ranges, one per CTA, so a CTA reloads the query block
// only when its range crosses a group boundary.
// Every mbarrier wait is bounded (2 s): on expiry the kernel flags
// MTPSD_STATUS_WAIT_TIMEOUT, drains its own copies in flight, frees TMEM and
// returns.
#include <cuda.h>

#include <algorithm>
#include <stdlib.h>
#include <string.h>

#include "common.cuh"
#include "internal.h"
#include "mbar.cuh"

namespace mtpsd {
namespace itc {

constexpr int TILE_M = 128;
constexpr int KB = 128;                   // bytes per key / query head vector
constexpr int NSTAGE = 6;                 // key tiles in flight
constexpr int NKS = 16;                   // key-scale tiles in flight
constexpr int KS_BOX = TILE_M + 4;        // key scales per copy (a 4-aligned start)
constexpr int KS_STRIDE = 640;            // bytes per key-scale slot (128-byte aligned)
constexpr int NSLOT = 8;                  // TMEM slots
constexpr int SLOT_COLS = 64;
constexpr int MAX_CHUNK = 4;              // slots per MMA
constexpr int Q_ROWS = 512;               // query head vectors held in shared memory
constexpr int EPI_WG = 3;
constexpr int EPI_WARPS = 4 * EPI_WG;
constexpr int PRODUCER_WARP = EPI_WARPS;
constexpr int MMA_WARP = EPI_WARPS + 1;
constexpr int THREADS = 32 * (EPI_WARPS + 2);
constexpr int MAX_GROUP_ROWS = Q_ROWS / 32;
constexpr int SPLIT_STAGE_COLS = 256;                  // TMEM columns of one head half (8 rows x 32 heads)
constexpr int SPLIT_HALF_BYTES = 8 * 32 * KB;          // query bytes of one head half (8 rows x 32 heads)
static_assert(2 * SPLIT_HALF_BYTES == Q_ROWS * KB && 2 * SPLIT_STAGE_COLS == NSLOT * SLOT_COLS, "split layout");

constexpr int OFF_K = 0;
constexpr int OFF_Q = OFF_K + NSTAGE * TILE_M * KB;      // 98304
constexpr int OFF_KS = OFF_Q + Q_ROWS * KB;              // [NKS][KS_STRIDE]
constexpr int OFF_WQ = OFF_KS + NKS * KS_STRIDE;         // per epilogue warp: [Q_ROWS] float
constexpr int OFF_VIS = OFF_WQ + EPI_WARPS * Q_ROWS * 4; // per epilogue warp: [MAX_GROUP_ROWS] int64
constexpr int OFF_BAR = OFF_VIS + EPI_WARPS * MAX_GROUP_ROWS * 8;
constexpr int NCH = 2 * NSLOT;            // chunk barriers (a chunk holds >= 1 of the <= NSLOT units in flight)
constexpr int N_BARS = 2 * NSTAGE + 2 + NCH + NSLOT + 2 * NKS + 1;
constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;         // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
static_assert((OFF_KS % 128) == 0 && (KS_STRIDE % 128) == 0, "key-scale slots are 128-byte aligned");
static_assert(KS_BOX * 4 <= KS_STRIDE && (KS_BOX * 4) % 16 == 0, "key-scale box");

constexpr unsigned long long WAIT_LIMIT_NS = mbar::DEFAULT_LIMIT_NS;

struct Params {
  const float* q_scale;
  const float* w;
  const int64_t* cache_start;
  const int64_t* row_pos;
  int64_t pool;
  int64_t max_visible;
  float* scores;
  int64_t ld;
  int H;
  const int* g_b;
  const int* g_row0;
  const int* g_nrows;
  const int* g_vmax;
  const int* g_tile0;      // [n_groups + 1]
  const int* n_groups;
  int32_t* status;
  const float* k_scale;    // key scales (PAGED kernels copy them box by box)
  const int32_t* bt;       // block table of a paged cache (PAGED kernels only)
  int32_t bt_stride;
  int32_t pg_shift;        // log2(page size), >= 3
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(bar)) : "memory");
}
// Bounded wait (the shared helper with this kernel's limit): false when it gave up (time limit or
// another role aborted).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int32_t* status) {
  return mbar::wait<false>(bar, parity, abort_flag, status, WAIT_LIMIT_NS);
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"((uint64_t)src), "r"(bytes), "r"(saddr(bar))
               : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"((uint64_t)map), "r"(x), "r"(y), "r"(saddr(bar))
      : "memory");
}

// One lane of a converged warp (the lowest), as a warp-uniform branch: the
// producer and MMA roles run with the whole warp so that their loop state
// stays in uniform registers, and only the elected lane issues.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile("{\n .reg .b32 rx;\n .reg .pred px;\n elect.sync rx|px, 0xffffffff;\n selp.b32 %0, 1, 0, px;\n}\n"
               : "=r"(pred));
  return pred != 0;
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row atoms of
// 1024 bytes (stride byte offset 1024), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_byte_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_byte_addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;                 // leading byte offset (unused with this swizzle)
  d |= (uint64_t)(1024 >> 4) << 32;       // stride byte offset
  d |= (uint64_t)1 << 46;                 // version
  d |= (uint64_t)2 << 61;                 // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f8f6f4, A = B = E4M3, D = F32, both K-major, M = 128, N = 64 * c.
__device__ __forceinline__ uint32_t idesc(int c) {
  return (1u << 4) | ((uint32_t)(64 * c) >> 3 << 17) | ((128u >> 4) << 24);
}
// The same with N given in columns (a multiple of 16, at most 256).
__device__ __forceinline__ uint32_t idesc_n(int n) { return (1u << 4) | ((uint32_t)n >> 3 << 17) | ((128u >> 4) << 24); }

__device__ __forceinline__ void mma_fp8(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t id, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(id), "r"(accumulate));
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// (group, tile) cursor over the flattened work list.  CACHE: the current group's tile count is kept in
// a register, so advancing within a group touches no memory (one-row groups: a global load per tile in
// every role's loop put its latency on each role's critical path); without it the count is reloaded
// (the head-halves kernel, whose epilogue has no register to spare).
template <bool CACHE>
struct CursorT {
  int g, tile, len;
  // called by all 32 lanes of a warp: the last g with g_tile0[g] <= it (which skips groups without
  // tiles), found with rounds of 32 parallel loads
  __device__ void start(const Params& p, int n_groups, int it) {
    g = request_of_row_warp((const uint32_t*)p.g_tile0, n_groups, (uint32_t)it);
    tile = it - p.g_tile0[g];
    if (CACHE) len = p.g_tile0[g + 1] - p.g_tile0[g];
  }
  __device__ void next(const Params& p, int n_groups) {
    ++tile;
    if (CACHE) {
      while (g + 1 <= n_groups - 1 && tile >= len) {
        tile -= len;
        ++g;
        len = p.g_tile0[g + 1] - p.g_tile0[g];
      }
    } else {
      while (g + 1 <= n_groups - 1 && tile >= p.g_tile0[g + 1] - p.g_tile0[g]) {
        tile -= p.g_tile0[g + 1] - p.g_tile0[g];
        ++g;
      }
    }
  }
};

// ------------------------------------------------------------------- kernels
// Group plan: one block of up to 1024 threads (one request per thread, in passes of blockDim
// requests).  For each request, its rows are cut into groups of at most group_rows rows; each group
// scans ceil(vmax/128) tiles, vmax being the largest visible length of its rows (clamped to
// max_visible).  The group and tile offsets are exclusive prefix sums over the requests (warp
// shuffles, then one warp over the warp totals).
__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

__global__ void __launch_bounds__(1024) plan_kernel(const uint32_t* __restrict__ ro, const int64_t* __restrict__ row_pos,
                                                    int B, int64_t max_visible, int group_rows, int* g_b,
                                                    int* g_row0, int* g_nrows, int* g_vmax, int* g_tile0,
                                                    int* n_groups) {
  griddep_wait();                // the previous kernel's writes are visible from here on
  griddep_launch_dependents();
  __shared__ int s_wg[32], s_wt[32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  int carry_g = 0, carry_t = 0;
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int r0 = 0, r1 = 0, ng = 0, nt = 0;
    if (b < B) {
      r0 = (int)ro[b];
      r1 = (int)ro[b + 1];
      for (int a = r0; a < r1; a += group_rows) {
        const int e = min(r1, a + group_rows);
        int64_t vm = 0;
        for (int r = a; r < e; ++r) vm = max(vm, min(row_pos[r] + 1, max_visible));
        ++ng;
        nt += (int)((vm + TILE_M - 1) / TILE_M);
      }
    }
    const int ig = warp_incl_scan(ng, lane), it = warp_incl_scan(nt, lane);
    if (lane == 31) {
      s_wg[wid] = ig;
      s_wt[wid] = it;
    }
    __syncthreads();
    if (wid == 0) {
      const int vg = lane < nw ? s_wg[lane] : 0, vt = lane < nw ? s_wt[lane] : 0;
      const int sg = warp_incl_scan(vg, lane), stt = warp_incl_scan(vt, lane);
      if (lane < nw) {
        s_wg[lane] = sg - vg;     // exclusive offsets of the warps
        s_wt[lane] = stt - vt;
      }
    }
    __syncthreads();
    int gpos = carry_g + s_wg[wid] + ig - ng;
    int tpos = carry_t + s_wt[wid] + it - nt;
    for (int a = r0; a < r1; a += group_rows) {   // no rows: no groups (b >= B too)
      const int e = min(r1, a + group_rows);
      int64_t vm = 0;
      for (int r = a; r < e; ++r) vm = max(vm, min(row_pos[r] + 1, max_visible));
      g_b[gpos] = b;
      g_row0[gpos] = a;
      g_nrows[gpos] = e - a;
      g_vmax[gpos] = (int)vm;
      g_tile0[gpos] = tpos;
      ++gpos;
      tpos += (int)((vm + TILE_M - 1) / TILE_M);
    }
    // pass totals: the last warp's exclusive offset plus its inclusive total
    const int last = nw - 1;
    __shared__ int s_tot[2];
    if (threadIdx.x == blockDim.x - 1) {
      s_tot[0] = s_wg[last] + ig;
      s_tot[1] = s_wt[last] + it;
    }
    __syncthreads();
    carry_g += s_tot[0];
    carry_t += s_tot[1];
    __syncthreads();   // s_wg / s_wt / s_tot are rewritten by the next pass
  }
  if (threadIdx.x == 0) {
    g_tile0[carry_g] = carry_t;
    *n_groups = carry_g;
  }
}

// PAGED: the cache is paged (pages of 2^pg_shift >= 8 tokens).  A key tile of 128 positions is then
// loaded as 128 / SUB boxes of SUB = min(page, 128) rows, each from the slot its page entry gives (1024-byte
// aligned destinations keep the 128-byte swizzle), and the key scales of each box as one bulk copy; lane k of
// the producer handles box k.  A box without a page (or outside the pool) loads zeros: its keys through an
// out-of-range TMA row, its scales written as zeros by the lane itself.
// SPLIT (64 heads, groups of up to 8 rows): every key tile is scored in two halves, heads 0..31 then heads
// 32..63 of all the group's rows, each half in its own 256-column TMEM stage (N = 32 x rows), so that the MMAs
// of one half run while the epilogue drains the other.  A six-row tile has 384 accumulator columns, and
// without the split the next tile's MMAs could only start after the epilogue had read most of this one:
// every tile paid a full MMA -> epilogue -> MMA round trip.  The query block is held as [half][row][32 heads];
// epilogue warpgroup w takes the row pairs (2j, 2j+1) with j = w and j = w + 3 in both halves and carries the
// first half's partial head sums in registers to the second.
template <int H, bool PAGED, bool SPLIT>
__global__ void __launch_bounds__(THREADS, 1) indexer_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                                                const __grid_constant__ CUtensorMap tmap_q,
                                                                const __grid_constant__ CUtensorMap tmap_ks,
                                                                Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(sm + OFF_BAR);
  uint64_t* k_full = bars;
  uint64_t* k_empty = bars + NSTAGE;
  uint64_t* q_full = bars + 2 * NSTAGE;
  uint64_t* q_empty = q_full + 1;
  uint64_t* chunk_full = q_full + 2;          // MMA chunk c done: chunk_full[c % NCH], phase c / NCH
  uint64_t* slot_empty = chunk_full + NCH;
  uint64_t* ks_full = slot_empty + NSLOT;
  uint64_t* ks_empty = ks_full + NKS;
  uint64_t* drain = ks_empty + NKS;
  uint32_t* tmem_slot = (uint32_t*)(sm + OFF_MISC);
  volatile int* abort_flag = (volatile int*)(sm + OFF_MISC + 4);
  // per-warp copies of the group's weights and visible lengths: each epilogue
  // warp fills and reads its own, so only __syncwarp orders them
  float* wq = (float*)(sm + OFF_WQ) + (threadIdx.x >> 5) * Q_ROWS;
  int64_t* vis = (int64_t*)(sm + OFF_VIS) + (threadIdx.x >> 5) * MAX_GROUP_ROWS;
  constexpr int ROWS_PER_UNIT = SLOT_COLS / H;   // 1 (H = 64) or 2 (H = 32)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The set-up below touches no global memory, so it overlaps the previous kernel's tail
  // (programmatic dependent launch); the plan it wrote is read after griddep_wait().
  if (threadIdx.x == 0) {
    for (int i = 0; i < NSTAGE; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < NCH; ++i) mbar_init(&chunk_full[i], 1);
    // the four warps of the unit's warpgroup; SPLIT: every epilogue warp, once per half
    for (int i = 0; i < NSLOT; ++i) mbar_init(&slot_empty[i], SPLIT ? EPI_WARPS : 4);
    for (int i = 0; i < NKS; ++i) {
      mbar_init(&ks_full[i], 1);
      mbar_init(&ks_empty[i], EPI_WARPS);    // every epilogue warp, once per tile
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == MMA_WARP) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tmem_slot)),
                 "r"(NSLOT * SLOT_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (warp == PRODUCER_WARP && elect_one()) {
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmap_k) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmap_q) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmap_ks) : "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_wait();                // the previous kernel's writes are visible from here on
  griddep_launch_dependents();
  const int n_groups = *p.n_groups;
  const int total = n_groups > 0 ? p.g_tile0[n_groups] : 0;
  const int it0 = (int)(((int64_t)blockIdx.x * total) / gridDim.x);
  const int it1 = (int)(((int64_t)(blockIdx.x + 1) * total) / gridDim.x);
  if (it0 >= it1) {   // no work: uniform per CTA; the TMEM allocated above is released
    if (warp == MMA_WARP)
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(NSLOT * SLOT_COLS));
    return;
  }

  if (warp == PRODUCER_WARP) {
    int n_load = 0, gq = 0, cur_g = -1;
    int64_t cstart = 0, cur_vmax = 0;
    bool ok = true;
    CursorT<!SPLIT> c;
    c.start(p, n_groups, it0);
    // PAGED: this lane's box of a (group, tile): its page entry, loaded one tile ahead of its use
    const int sub = PAGED ? min(TILE_M, 1 << p.pg_shift) : TILE_M;
    const int n_sub = TILE_M / sub;
    auto page_of = [&](int g, int tile) -> int32_t {
      if (lane >= n_sub) return -1;
      const int64_t pg = ((int64_t)tile * TILE_M + lane * sub) >> p.pg_shift;
      if (pg >= p.bt_stride) return -1;
      return __ldg(p.bt + (int64_t)p.g_b[g] * p.bt_stride + pg);
    };
    int32_t pe_cur = PAGED ? page_of(c.g, c.tile) : 0;
    for (int it = it0; it < it1 && ok; ++it, c.next(p, n_groups)) {
      const int g = c.g;
      int32_t pe_next = -1;
      if (PAGED && it + 1 < it1) {
        CursorT<!SPLIT> cn = c;
        cn.next(p, n_groups);
        pe_next = page_of(cn.g, cn.tile);
      }
      if (g != cur_g) {
        if (gq > 0) ok = __all_sync(0xffffffffu, mbar_wait(q_empty, (gq - 1) & 1, abort_flag, p.status));
        if (!ok) break;
        const int nrows = p.g_nrows[g], row0 = p.g_row0[g];
        if (PAGED) cur_vmax = p.g_vmax[g];
        else cstart = p.cache_start[p.g_b[g]];
        if (elect_one()) {
          mbar_expect_tx(q_full, (uint32_t)(nrows * H * KB));
          if (SPLIT) {   // [half][row][32 heads]: two boxes of 32 head vectors per row
            for (int i = 0; i < nrows; ++i)
              for (int h = 0; h < 2; ++h)
                tma_load_2d(saddr(sm + OFF_Q + h * SPLIT_HALF_BYTES + i * 32 * KB), &tmap_q, 0, (row0 + i) * H + h * 32,
                            q_full);
          } else {
            for (int i = 0; i < nrows; ++i)
              tma_load_2d(saddr(sm + OFF_Q + i * H * KB), &tmap_q, 0, (row0 + i) * H, q_full);
          }
        }
        __syncwarp();
        ++gq;
        cur_g = g;
      }
      const int stage = n_load % NSTAGE, round = n_load / NSTAGE;
      const int kslot = n_load % NKS, kround = n_load / NKS;
      if (round > 0) ok = __all_sync(0xffffffffu, mbar_wait(&k_empty[stage], (round - 1) & 1, abort_flag, p.status));
      if (ok && kround > 0)
        ok = __all_sync(0xffffffffu, mbar_wait(&ks_empty[kslot], (kround - 1) & 1, abort_flag, p.status));
      if (!ok) break;
      if (PAGED) {
        const int64_t s = (int64_t)c.tile * TILE_M + lane * sub;
        int64_t slot = (lane < n_sub && pe_cur >= 0)
                           ? (((int64_t)pe_cur << p.pg_shift) | (s & ((1LL << p.pg_shift) - 1))) : -1;
        if (slot + sub > p.pool) slot = -1;
        if (lane < n_sub && slot < 0 && s < cur_vmax) flag_status(p.status, MTPSD_STATUS_ROW_RANGE);
        float* ks_dst = (float*)(sm + OFF_KS + kslot * KS_STRIDE) + lane * sub;
        if (lane < n_sub && slot < 0)
          for (int i = 0; i < sub; ++i) ks_dst[i] = 0.f;   // generic-proxy zeros, ordered by the arrive below
        const uint32_t ks_bytes = (uint32_t)sub * 4u *
                                  (uint32_t)__popc(__ballot_sync(0xffffffffu, lane < n_sub && slot >= 0));
        __syncwarp();
        if (elect_one()) {
          mbar_expect_tx(&k_full[stage], TILE_M * KB);
          mbar_expect_tx(&ks_full[kslot], ks_bytes);
        }
        __syncwarp();
        if (lane < n_sub) {
          tma_load_2d(saddr(sm + OFF_K + stage * TILE_M * KB + lane * sub * KB), &tmap_k, 0,
                      slot >= 0 ? (int)slot : (int)p.pool, &k_full[stage]);
          if (slot >= 0) bulk_load(saddr(ks_dst), p.k_scale + slot, (uint32_t)sub * 4u, &ks_full[kslot]);
        }
        pe_cur = pe_next;
      } else {
        const int64_t y = cstart + (int64_t)c.tile * TILE_M;
        if (elect_one()) {
          mbar_expect_tx(&k_full[stage], TILE_M * KB);
          tma_load_2d(saddr(sm + OFF_K + stage * TILE_M * KB), &tmap_k, 0, (int)y, &k_full[stage]);
          // key scales of the tile from a 4-aligned start (16-byte aligned copy); elements past the pool
          // read as zero
          mbar_expect_tx(&ks_full[kslot], KS_BOX * 4);
          tma_load_2d(saddr(sm + OFF_KS + kslot * KS_STRIDE), &tmap_ks, (int)(y & ~(int64_t)3), 0, &ks_full[kslot]);
        }
      }
      __syncwarp();
      ++n_load;
    }
    if (*abort_flag && lane == 0) {   // drain this CTA's copies still in flight (bounded)
      volatile int dummy = 0;
      for (int s = 0; s < NSTAGE; ++s) {
        const int issued = n_load / NSTAGE + (s < n_load % NSTAGE ? 1 : 0);   // loads of stage s
        if (issued > 0) mbar_wait(&k_full[s], (issued - 1) & 1, &dummy, p.status);
      }
      for (int s = 0; s < NKS; ++s) {
        const int issued = n_load / NKS + (s < n_load % NKS ? 1 : 0);
        if (issued > 0) mbar_wait(&ks_full[s], (issued - 1) & 1, &dummy, p.status);
      }
      if (gq > 0) mbar_wait(q_full, (gq - 1) & 1, &dummy, p.status);
    }
  } else if (warp == MMA_WARP && SPLIT) {
    // per key tile: half h (heads 32h .. 32h+31 of every row) into TMEM stage h, N = 32 x rows
    int n_cons = 0, gq = 0, cur_g = -1, nrows = 0;
    bool ok = true;
    CursorT<!SPLIT> c;
    c.start(p, n_groups, it0);
    for (int it = it0; it < it1 && ok; ++it, c.next(p, n_groups)) {
      const int g = c.g;
      if (g != cur_g) {
        if (cur_g >= 0) {
          if (elect_one()) mma_commit(q_empty);
          __syncwarp();
        }
        ok = __all_sync(0xffffffffu, mbar_wait(q_full, gq & 1, abort_flag, p.status));
        if (!ok) break;
        ++gq;
        cur_g = g;
        nrows = p.g_nrows[g];
      }
      const int stage = n_cons % NSTAGE, round = n_cons / NSTAGE;
      ok = __all_sync(0xffffffffu, mbar_wait(&k_full[stage], round & 1, abort_flag, p.status));
      if (!ok) break;
      const uint32_t a_base = saddr(sm + OFF_K + stage * TILE_M * KB);
      const uint32_t id = idesc_n(32 * nrows);
      for (int h = 0; h < 2 && ok; ++h) {
        // stage h was last used by the previous tile's half h
        if (n_cons > 0) ok = __all_sync(0xffffffffu, mbar_wait(&slot_empty[h], (n_cons - 1) & 1, abort_flag, p.status));
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) {
          const uint32_t b_base = saddr(sm + OFF_Q + h * SPLIT_HALF_BYTES);
          const uint32_t d = tmem_base + (uint32_t)(h * SPLIT_STAGE_COLS);
#pragma unroll
          for (int kk = 0; kk < KB / 32; ++kk)
            mma_fp8(d, sw128_desc(a_base + kk * 32), sw128_desc(b_base + kk * 32), id, kk > 0 ? 1u : 0u);
          mma_commit(&chunk_full[h]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (elect_one()) mma_commit(&k_empty[stage]);
      __syncwarp();
      ++n_cons;
    }
    if (elect_one()) mma_commit(drain);
    __syncwarp();
    volatile int dummy = 0;
    mbar_wait(drain, 0, &dummy, p.status);
  } else if (warp == MMA_WARP) {
    int n_cons = 0, gq = 0, cur_g = -1, units = 0;
    int u = 0;        // running unit (slot use) index
    int nchunk = 0;   // running MMA chunk index
    bool ok = true;
    CursorT<!SPLIT> c;
    c.start(p, n_groups, it0);
    for (int it = it0; it < it1 && ok; ++it, c.next(p, n_groups)) {
      const int g = c.g;
      if (g != cur_g) {
        if (cur_g >= 0) {
          if (elect_one()) mma_commit(q_empty);
          __syncwarp();
        }
        ok = __all_sync(0xffffffffu, mbar_wait(q_full, gq & 1, abort_flag, p.status));
        if (!ok) break;
        ++gq;
        cur_g = g;
        units = (p.g_nrows[g] * H + SLOT_COLS - 1) / SLOT_COLS;
      }
      const int stage = n_cons % NSTAGE, round = n_cons / NSTAGE;
      // Every wait of the tile comes before its first MMA: once about four MMAs are queued, the issuing
      // warp's memory instructions (these barrier probes included) stall until the queue drains, so
      // waits between MMA batches would let the tensor pipe run dry once per batch.
      ok = __all_sync(0xffffffffu, mbar_wait(&k_full[stage], round & 1, abort_flag, p.status));
      for (int v = 0; v < units && ok; ++v) {
        const int ur = (u + v) / NSLOT;   // previous uses of the unit's slot
        if (ur > 0)
          ok = __all_sync(0xffffffffu, mbar_wait(&slot_empty[(u + v) % NSLOT], (ur - 1) & 1, abort_flag, p.status));
      }
      if (!ok) break;
      tc_fence_after();
      const uint32_t a_base = saddr(sm + OFF_K + stage * TILE_M * KB);
      for (int v0 = 0; v0 < units; ++nchunk) {
        // the next up-to-4 units that sit in adjacent slots (the ring does not wrap inside one MMA)
        const int s0 = (u + v0) % NSLOT;
        int cnt = units - v0;
        if (cnt > MAX_CHUNK) cnt = MAX_CHUNK;
        if (cnt > NSLOT - s0) cnt = NSLOT - s0;
        if (elect_one()) {
          const uint32_t b_base = saddr(sm + OFF_Q + v0 * SLOT_COLS * KB);
          const uint32_t d = tmem_base + (uint32_t)(s0 * SLOT_COLS);
          const uint32_t id = idesc(cnt);
#pragma unroll
          for (int kk = 0; kk < KB / 32; ++kk)
            mma_fp8(d, sw128_desc(a_base + kk * 32), sw128_desc(b_base + kk * 32), id, kk > 0 ? 1u : 0u);
          mma_commit(&chunk_full[nchunk % NCH]);
        }
        __syncwarp();
        v0 += cnt;
      }
      if (elect_one()) mma_commit(&k_empty[stage]);
      __syncwarp();
      u += units;
      ++n_cons;
    }
    // all issued MMAs complete before TMEM is released
    if (elect_one()) mma_commit(drain);
    __syncwarp();
    volatile int dummy = 0;
    mbar_wait(drain, 0, &dummy, p.status);
  } else if (SPLIT) {
    // ------------------------------------------------------------ epilogue of the head halves
    const int wg = warp >> 2;
    const int quarter = warp & 3;
    const int pos_in_tile = quarter * 32 + lane;
    int cur_g = -1, nrows = 0, row0 = 0, n_tile = 0, ks_off = 0;
    int64_t vmax = 0, cstart = 0;
    bool ok = true;
    CursorT<!SPLIT> c;
    c.start(p, n_groups, it0);
    for (int it = it0; it < it1 && ok; ++it, c.next(p, n_groups), ++n_tile) {
      const int g = c.g;
      if (g != cur_g) {
        __syncwarp();
        nrows = p.g_nrows[g];
        row0 = p.g_row0[g];
        vmax = p.g_vmax[g];
        cstart = PAGED ? 0 : p.cache_start[p.g_b[g]];
        ks_off = (int)(cstart & 3);
        {
          float wv[Q_ROWS / 32], qv[Q_ROWS / 32];
#pragma unroll
          for (int k = 0; k < Q_ROWS / 32; ++k) {
            const int e = lane + 32 * k;
            const bool in = e < nrows * H;
            wv[k] = in ? p.w[(int64_t)row0 * H + e] : 0.f;
            qv[k] = in ? p.q_scale[(int64_t)row0 * H + e] : 0.f;
          }
#pragma unroll
          for (int k = 0; k < Q_ROWS / 32; ++k)
            if (lane + 32 * k < nrows * H) wq[lane + 32 * k] = 0.5f * (wv[k] * qv[k]);
        }
        for (int i = lane; i < nrows; i += 32) vis[i] = min(p.row_pos[row0 + i] + 1, p.max_visible);
        __syncwarp();
        cur_g = g;
      }
      const int kslot = n_tile % NKS, kround = n_tile / NKS;
      ok = __all_sync(0xffffffffu, mbar_wait(&ks_full[kslot], kround & 1, abort_flag, p.status));
      if (!ok) break;
      const int64_t s = (int64_t)c.tile * TILE_M + pos_in_tile;
      const float ks = (s < vmax) ? ((const float*)(sm + OFF_KS + kslot * KS_STRIDE))[ks_off + pos_in_tile] : 0.f;
      // this warpgroup's row pairs: j = wg (k = 0) and j = wg + 3 (k = 1), rows 2j and 2j + 1
      const int n_pairs = (nrows + 1) >> 1;
      const int n_mine = (wg < n_pairs ? 1 : 0) + (wg + EPI_WG < n_pairs ? 1 : 0);
      float part[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
      for (int h = 0; h < 2 && ok; ++h) {
        ok = __all_sync(0xffffffffu, mbar_wait(&chunk_full[h], n_tile & 1, abort_flag, p.status));
        if (!ok) break;
        tc_fence_after();
        if (n_mine == 0) {   // nothing to read: release the stage at once
          __syncwarp();
          if (lane == 0) mbar_arrive(&slot_empty[h]);
          continue;
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int j = wg + EPI_WG * k;
          if (k >= n_mine) break;
          float x[64];   // x[0..31]: row 2j, x[32..63]: row 2j + 1 (heads 32h ..)
          const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) +
                                 (uint32_t)(h * SPLIT_STAGE_COLS + j * 64);
          tmem_ld32(taddr, x);
          tmem_ld32(taddr + 32, x + 32);
          tmem_ld_wait();
          if (k == n_mine - 1) {   // the warp's last read of this stage
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&slot_empty[h]);
          }
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int i = 2 * j + r;   // row within the group
            if (i >= nrows) break;
            const float4* wr = (const float4*)(wq + i * H + h * 32);
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int m = 0; m < 8; ++m) {
              const float4 ww = wr[m];
              acc[0] = fmaf(ww.x, x[32 * r + 4 * m + 0] + fabsf(x[32 * r + 4 * m + 0]), acc[0]);
              acc[1] = fmaf(ww.y, x[32 * r + 4 * m + 1] + fabsf(x[32 * r + 4 * m + 1]), acc[1]);
              acc[2] = fmaf(ww.z, x[32 * r + 4 * m + 2] + fabsf(x[32 * r + 4 * m + 2]), acc[2]);
              acc[3] = fmaf(ww.w, x[32 * r + 4 * m + 3] + fabsf(x[32 * r + 4 * m + 3]), acc[3]);
            }
            const float sc = (acc[0] + acc[1]) + (acc[2] + acc[3]);
            if (h == 0) {
              part[k][r] = sc;
            } else if (s < vis[i]) {
              p.scores[(int64_t)(row0 + i) * p.ld + s] = (part[k][r] + sc) * ks;
            }
          }
        }
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&ks_empty[kslot]);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int wg = warp >> 2;              // this warpgroup takes units u with u % EPI_WG == wg
    const int quarter = warp & 3;          // TMEM lanes 32*quarter .. +31
    const int pos_in_tile = quarter * 32 + lane;
    int cur_g = -1, nrows = 0, row0 = 0, units = 0, n_tile = 0, ks_off = 0;
    int u = 0, nchunk = 0;   // running unit and MMA chunk indices (the MMA warp's chunking, replayed)
    int64_t vmax = 0, cstart = 0;
    bool ok = true;
    CursorT<!SPLIT> c;
    c.start(p, n_groups, it0);
    for (int it = it0; it < it1 && ok; ++it, c.next(p, n_groups), ++n_tile) {
      const int g = c.g;
      if (g != cur_g) {
        __syncwarp();   // the warp is done with the previous group's copies
        nrows = p.g_nrows[g];
        row0 = p.g_row0[g];
        vmax = p.g_vmax[g];
        cstart = PAGED ? 0 : p.cache_start[p.g_b[g]];
        ks_off = (int)(cstart & 3);   // paged: the scale slot holds the tile's 128 scales from its start
        units = (nrows * H + SLOT_COLS - 1) / SLOT_COLS;
        {   // all of the group's (row, head) weights in flight at once
          float wv[Q_ROWS / 32], qv[Q_ROWS / 32];
#pragma unroll
          for (int k = 0; k < Q_ROWS / 32; ++k) {
            const int e = lane + 32 * k;
            const bool in = e < nrows * H;
            wv[k] = in ? p.w[(int64_t)row0 * H + e] : 0.f;
            qv[k] = in ? p.q_scale[(int64_t)row0 * H + e] : 0.f;
          }
          // halved: the epilogue forms 2 ReLU(x) = x + |x| (exact) on the FMA pipe
#pragma unroll
          for (int k = 0; k < Q_ROWS / 32; ++k)
            if (lane + 32 * k < nrows * H) wq[lane + 32 * k] = 0.5f * (wv[k] * qv[k]);
        }
        for (int i = lane; i < nrows; i += 32) vis[i] = min(p.row_pos[row0 + i] + 1, p.max_visible);
        __syncwarp();
        cur_g = g;
      }
      const int kslot = n_tile % NKS, kround = n_tile / NKS;
      // every epilogue warp waits for the tile's key scales (so that its release below can never count
      // toward an earlier use of the slot), reads them if it owns a unit, and releases them
      ok = __all_sync(0xffffffffu, mbar_wait(&ks_full[kslot], kround & 1, abort_flag, p.status));
      if (!ok) break;
      const int64_t s = (int64_t)c.tile * TILE_M + pos_in_tile;
      const float ks = (s < vmax) ? ((const float*)(sm + OFF_KS + kslot * KS_STRIDE))[ks_off + pos_in_tile] : 0.f;
      // chunks of the tile, as the MMA warp forms them: unit v is in chunk nchunk + chunk_of(v)
      auto chunk_of = [&](int v) -> int {
        int c = 0;
#pragma unroll
        for (int v0 = 0, k = 0; k < NSLOT; ++k) {
          if (v0 >= units) break;
          const int s0 = (u + v0) % NSLOT;
          int cnt = units - v0;
          if (cnt > MAX_CHUNK) cnt = MAX_CHUNK;
          if (cnt > NSLOT - s0) cnt = NSLOT - s0;
          if (v < v0 + cnt) break;
          v0 += cnt;
          ++c;
        }
        return c;
      };
      const int nch_tile = units > 0 ? chunk_of(units - 1) + 1 : 0;
      // first unit of this tile that belongs to this warpgroup
      int v = (wg - u % EPI_WG + EPI_WG) % EPI_WG;
      for (; v < units; v += EPI_WG) {
        const int uu = u + v;
        const int slot = uu % NSLOT;
        const int ch = nchunk + chunk_of(v);
        // warp-uniform outcome: tcgen05.ld below is a warp-collective instruction
        ok = __all_sync(0xffffffffu, mbar_wait(&chunk_full[ch % NCH], (ch / NCH) & 1, abort_flag, p.status));
        if (!ok) break;
        tc_fence_after();
        float x[64];
        const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(slot * SLOT_COLS);
        tmem_ld32(taddr, x);
        tmem_ld32(taddr + 32, x + 32);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&slot_empty[slot]);
#pragma unroll
        for (int j = 0; j < ROWS_PER_UNIT; ++j) {
          const int i = v * ROWS_PER_UNIT + j;   // row within the group
          if (i >= nrows) break;
          // ReLU(x) w = (x + |x|) (w / 2): an FADD with the free |.| operand modifier and an FFMA, both
          // on the FMA pipe (x + |x| is 2x or +0 exactly, so the products equal those of max(x, 0) w)
          const float4* wr = (const float4*)(wq + i * H);
          float acc[4] = {0.f, 0.f, 0.f, 0.f};   // heads h = 4k + m go to acc[m]
          const int hb = j * H;   // first column of row i within the unit
#pragma unroll
          for (int m = 0; m < H / 4; ++m) {
            const float4 ww = wr[m];
            acc[0] = fmaf(ww.x, x[hb + 4 * m + 0] + fabsf(x[hb + 4 * m + 0]), acc[0]);
            acc[1] = fmaf(ww.y, x[hb + 4 * m + 1] + fabsf(x[hb + 4 * m + 1]), acc[1]);
            acc[2] = fmaf(ww.z, x[hb + 4 * m + 2] + fabsf(x[hb + 4 * m + 2]), acc[2]);
            acc[3] = fmaf(ww.w, x[hb + 4 * m + 3] + fabsf(x[hb + 4 * m + 3]), acc[3]);
          }
          const float sc = (acc[0] + acc[1]) + (acc[2] + acc[3]);
          if (s < vis[i]) p.scores[(int64_t)(row0 + i) * p.ld + s] = sc * ks;
        }
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&ks_empty[kslot]);
      u += units;
      nchunk += nch_tile;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(NSLOT * SLOT_COLS));
  }
}

}  // namespace itc

// ------------------------------------------------------------------ host side
static bool make_map_rows128(CUtensorMap* map, const void* base, int64_t rows, uint32_t box_rows) {
  return make_tma_2d(map, 0, base, 128, (uint64_t)rows, 128, 128, box_rows, true);
}

static bool tc_device_ok() { return cc_major() == 10; }

size_t indexer_tc_plan_bytes(int B, int R) {
  size_t n = (size_t)B + (size_t)R + 2;
  return ((5 * n + 1) * sizeof(int) + 255) / 256 * 256;
}

bool indexer_tc_supported(const IndexerPlan& p) {
  const char* env = getenv("MTPSD_INDEXER");
  if (env && strcmp(env, "generic") == 0) return false;
  if (p.dtype != MTPSD_FP8_E4M3 || p.D != 128) return false;
  if (p.H != 64 && p.H != 32) return false;
  if (((uintptr_t)p.k % 16) || ((uintptr_t)p.q % 16) || ((uintptr_t)p.k_scale % 16)) return false;
  if (p.pool < 1 || p.pool > 0x7fffffffLL || (int64_t)p.R * p.H > 0x7fffffffLL) return false;
  if (p.max_visible > 0x7fffffffLL - itc::TILE_M) return false;
  if (!p.plan_ws) return false;
  // paged caches: pages of at least 8 tokens (1024-byte aligned swizzled key boxes, 32-byte scale copies)
  // that tile the pool
  if (p.pg.bt && (p.pg.shift < 3 || (p.pool & ((1LL << p.pg.shift) - 1)) != 0)) return false;
  return tc_device_ok() && tma_available();
}

int indexer_launch_count(int H, int D, int dtype) {
  const char* env = getenv("MTPSD_INDEXER");
  const bool tc = !(env && strcmp(env, "generic") == 0) && dtype == MTPSD_FP8_E4M3 && D == 128 &&
                  (H == 64 || H == 32) && tc_device_ok() && tma_available();
  return tc ? 3 : 2;
}

int launch_indexer_scores_tc(const IndexerPlan& p, cudaStream_t st) {
  using namespace itc;
  CUtensorMap mk, mq, mks;
  const bool paged = p.pg.bt != nullptr;
  const uint32_t key_box = paged ? (uint32_t)std::min<int64_t>(TILE_M, 1LL << p.pg.shift) : (uint32_t)TILE_M;
  // head halves: groups average five or more rows (64 heads), so a tile's accumulators would fill most of TMEM
  const char* env_split = getenv("MTPSD_INDEXER_SPLIT");
  const bool split = p.H == 64 && (env_split ? env_split[0] == '1' : (int64_t)p.R >= 5LL * p.B);
  if (!make_map_rows128(&mk, p.k, p.pool, key_box) ||
      !make_map_rows128(&mq, p.q, (int64_t)p.R * p.H, split ? 32u : (uint32_t)p.H) ||
      !make_tma_1d_f32(&mks, p.k_scale, (uint64_t)p.pool, KS_BOX)) {
    set_error("indexer: cuTensorMapEncodeTiled failed");
    return MTPSD_ECUDA;
  }
  const size_t n = (size_t)p.B + (size_t)p.R + 2;
  int* w = (int*)p.plan_ws;
  int* g_b = w;
  int* g_row0 = g_b + n;
  int* g_nrows = g_row0 + n;
  int* g_vmax = g_nrows + n;
  int* g_tile0 = g_vmax + n;
  int* n_groups = g_tile0 + n;
  const int group_rows = Q_ROWS / p.H;
  const int plan_threads = p.B >= 1024 ? 1024 : ((p.B + 31) / 32) * 32 + (p.B == 0 ? 32 : 0);
  launch_k(plan_kernel, 1, plan_threads, 0, st, p.row_offsets, p.row_pos, p.B, p.max_visible, group_rows, g_b, g_row0, g_nrows,
                                  g_vmax, g_tile0, n_groups);
  int rc = check_launch("indexer_tc_plan");
  if (rc) return rc;
  Params kp;
  kp.q_scale = p.q_scale; kp.w = p.w; kp.cache_start = p.cache_start;
  kp.row_pos = p.row_pos; kp.pool = p.pool; kp.max_visible = p.max_visible; kp.scores = p.scores; kp.ld = p.ld;
  kp.H = p.H; kp.g_b = g_b; kp.g_row0 = g_row0; kp.g_nrows = g_nrows; kp.g_vmax = g_vmax; kp.g_tile0 = g_tile0;
  kp.n_groups = n_groups; kp.status = p.status;
  kp.k_scale = p.k_scale; kp.bt = p.pg.bt; kp.bt_stride = p.pg.stride; kp.pg_shift = p.pg.shift;
  static std::atomic<uint64_t> attr[6];
  auto kern = p.H == 64 ? (split ? (paged ? indexer_tc_kernel<64, true, true> : indexer_tc_kernel<64, false, true>)
                                 : (paged ? indexer_tc_kernel<64, true, false> : indexer_tc_kernel<64, false, false>))
                        : (paged ? indexer_tc_kernel<32, true, false> : indexer_tc_kernel<32, false, false>);
  const int which = p.H == 64 ? (split ? 4 : 0) + (paged ? 1 : 0) : 2 + (paged ? 1 : 0);
  if (!set_smem_limit_once(kern, SMEM_BYTES, attr[which])) {
    set_error("indexer_tc: cudaFuncSetAttribute failed");
    return MTPSD_ECUDA;
  }
  launch_k(kern, num_sms(), THREADS, SMEM_BYTES, st, mk, mq, mks, kp);
  return check_launch("indexer_tc");
}

}  // namespace mtpsd
