// Sparse MLA decode on the 5th-generation tensor cores (tcgen05 kind::f16,
// bf16 operands, fp32 accumulators in TMEM).
//
// [P2] "验证段的逐层算子" op 7 / [P3] "稀疏 MLA 的前向路径": per query row r and
// head h, softmax attention over the selected latent rows c[s_j, 0:576] with
// values c[s_j, 0:512].
//
// The latent rows are bf16 (1152 bytes), or the 656-byte FP8 rows of [P2]
// "草稿层 KV 的账" (512 E4M3 codes in four blocks of 128 with float32 scales,
// then the 64 rope values as bf16): the FP8 instantiation stages each
// producer warp's rows in shared memory and dequantizes them into the same
// bf16 operand layout (below, at the producers).
//
// A cluster of two CTAs owns (row, 128-head group, split of the selected
// list); the 128 heads are the MMA's M.  The two CTAs split the 576 latent
// dims instead of duplicating them, so every selected row is gathered once:
//   rank 0: dims 0..255 and the rope dims 512..575 (5 chunks of 64 dims);
//           its value dims are 0..255
//   rank 1: dims 256..511 (4 chunks); its value dims are 256..511
// Each CTA forms the partial scores of its dims, S_k = Q[:, D_k] C[:, D_k]^T,
// in TMEM.  Its sender warps scale them to log2 units, round them to fp16
// and stage them in shared memory; lane 0 of each sender warp then moves the
// warp's 32 heads into the other CTA's receive slot with one bulk copy per
// half pair (positions 0..31 and 32..63, 2 KB each), each completing bytes on
// its own mbarrier of that CTA.  Its softmax warps take each half as it lands:
// add it to their own fp32 partial, S = S_own + S_other, and exponentiate
// against the current reference max in the same pass, for this CTA's 256
// value dims.  The two CTAs see the other half rounded differently, so each
// value half keeps its own running (max, sum); split partials carry one
// (max, sum) per half.
//   TMEM  [  0,128) this CTA's first 256 query dims (A operand, bf16 pairs)
//         [128,192) [192,256) two partial-score buffers of 64 positions
//                   (fp32), P aliased in their first 32 columns (bf16 pairs)
//         [256,512) O: 128 heads x this CTA's 256 value dims (fp32)
//   SMEM  rank 0's rope query dims (16 KB, 128-byte swizzle); a ring of four
//         pair buffers of 64 gathered positions (40 KB each), laid out per
//         64-dim chunk (64 rows x 128 B, 128-byte swizzle), which are both the
//         K-major B operand of the scores (N = 64 positions) and, for chunks
//         0..3, the MN-major B operand of O += P V (K = positions, N = 256);
//         two receive slots for the other CTA's fp16 partial scores and one
//         staging slot for this CTA's (16 KB each: two halves of 8 KB, each
//         row = head with 32 positions in 64 bytes, 16-byte piece c at
//         (c ^ ((head >> 1) & 3))).  After the last pair the drained ring
//         stages O as 128-byte-swizzled boxes of 32 heads for TMA stores (bf16
//         output, or float32 split partials).
// Per pair: QK^T is 16 MMAs with A from TMEM (+4 with A from shared memory on
// rank 0), M=128, N=64, K=16; PV is 4 MMAs (M=128, N=256, K=16) with A = P
// from TMEM.  The MMA warp issues, in this fixed order, QK(P+1) (its buffer
// was last read by PV(P-1), issued before it) and PV(P) once the softmax
// published P, and sleeps in its waits: a polling or a blocked issue there
// takes issue slots and memory-instruction slots from the softmax warp that
// shares its scheduler.  The softmax (thread = head) applies a lazy max: O
// is rescaled, and the pair's exponentials taken again, only when a head's
// max grows by more than 2^8.
//
// Roles (416 threads): warps 0-3 softmax/epilogue (TMEM lanes = heads);
// warps 4-7 send the partial scores (thread = head of TMEM quadrant warp%4).
// Per-thread DSMEM stores (st.async) drain at about 13 bytes per cycle per
// SM and hold up the memory instructions of every warp on the issuing
// scheduler, so the senders only stage and bulk copies cross to the other SM.
// A shared-to-cluster bulk copy completes only on the receiver's mbarrier, so
// the receiver's first softmax thread reports each landed pair back (a relaxed
// remote arrival on stg_free) and the senders restage only after it.  Warps
// 8-11 produce, with the selection entries queued four tiles ahead: each turns its 8 positions of every
// 32-row tile into pool rows and gathers this CTA's chunks of them with TMA
// tile::gather4 loads (4 rows x 64 dims per instruction; invalid positions
// read as zeros through an out-of-range row); the first also loads rank 0's
// rope query dims; warp 12 allocates TMEM and issues the MMAs.  A receive
// slot is refilled (pair P+2) only after the other CTA's softmax warps have
// consumed it (one remote arrival per warp).  The producer and MMA roles run
// with the whole warp so that descriptors and coordinates stay in uniform
// registers, and one elected lane issues.  Every mbarrier wait is bounded
// (2 s) and flags MTPSD_STATUS_WAIT_TIMEOUT on expiry; a CTA whose partner
// stops sending times out the same way.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"
#include "mbar.cuh"

namespace mtpsd {
namespace mtc {

constexpr int DL = 576, DV = 512, DVH = 256;
constexpr int HG = 128;                 // heads per CTA (MMA M)
constexpr int NT = 32;                  // positions per gathered tile
constexpr int NP = 64;                  // positions per MMA step (a pair of tiles)
constexpr int NPAIR = 4;                // pair buffers in the ring
constexpr int NSTAGE = 2 * NPAIR;       // 32-row tiles in the ring
constexpr int NCH_MAX = 5;              // 64-dim chunks one CTA gathers (rank 0)
constexpr int QTM = 256;                // query dims held in TMEM
constexpr int CHUNK_BYTES = NP * 128;   // 8192: one chunk of a pair buffer
constexpr int PAIR_STRIDE = NCH_MAX * CHUNK_BYTES;   // 40960
constexpr int XSLOT_BYTES = HG * NP * 2;             // 16384: one pair's fp16 partial scores
constexpr int XHALF_BYTES = XSLOT_BYTES / 2;         // 8192: positions 0..31 or 32..63 of the pair
constexpr int OFF_QR = 0;                                    // rope query dims (rank 0)
constexpr int OFF_C = OFF_QR + HG * 128;                     // 16384
constexpr int OFF_X = OFF_C + NPAIR * PAIR_STRIDE;           // 180224: [2] receive slots
constexpr int OFF_STG = OFF_X + 2 * XSLOT_BYTES;             // 212992: own fp16 partials staged for the copy
constexpr int OFF_MASK = OFF_STG + XSLOT_BYTES;              // 229376: [NSTAGE][4] uint32 validity bits
constexpr int OFF_BAR = OFF_MASK + NSTAGE * 4 * 4;
// barriers: c_full[NSTAGE], c_empty[NPAIR], s_full[2], p_full[2], pv_done[2], x_full[2][2], s_read[2], x_free[2],
// stg_free, q_ready, drain
constexpr int N_BARS = NSTAGE + NPAIR + 14 + 3;
constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;               // tmem base, abort flag
constexpr int SMEM_USED = OFF_MISC + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;                 // alignment slack
constexpr int THREADS = 416;
constexpr int SEND_WARP = 4, PROD_WARP = 8, N_PROD = 4, MMA_WARP = 12;
constexpr int TM_Q = 0, TM_S0 = 128, TM_O = 256;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float RESCALE_LOG2 = 8.0f;
constexpr unsigned long long WAIT_LIMIT_NS = mbar::DEFAULT_LIMIT_NS;
constexpr int MAX_FUSED_SPLITS_K = 4;     // splits of a row that share one cluster and merge in the kernel
// FP8 latent rows (656 bytes: 512 E4M3 codes, 4 float32 block scales, 64 bf16 rope values).  The ring
// then has three pair buffers, and the fourth pair's space holds each producer warp's staging ring of
// FD tiles: per tile its 8 rows' codes for this CTA's 256 dims ([group][half][4 rows][128 B]), their
// 16-byte scale records ([group][4 rows][16 B], each group at a 128-byte boundary) and, on rank 0,
// their rope bytes ([group][4 rows][128 B]).
constexpr int FP8_ROW = 656;
constexpr int FD = 3;
constexpr int F_CODES = 2 * 2 * 512;
constexpr int F_SCL = 2 * 128;
constexpr int F_ROPE = 2 * 512;
constexpr int F_TILE = F_CODES + F_SCL + F_ROPE;
constexpr int OFF_F = OFF_C + 3 * PAIR_STRIDE;           // the fourth pair buffer
static_assert(4 * FD * F_TILE + 4 * FD * 8 <= PAIR_STRIDE && (F_TILE % 128) == 0 && (OFF_F % 1024) == 0,
              "FP8 staging fits the fourth pair buffer");
static_assert(SMEM_BYTES <= 232448, "shared memory");

struct Params {
  int B, R, H, n_idx, n_append;
  float sl2;                  // softmax scale * log2(e)
  int64_t row_pos_add;
  const __nv_bfloat16* q;
  const __nv_bfloat16* latent;
  int64_t pool;
  const int64_t* cache_start;
  const int32_t* bt;          // block table of a paged cache, or null (contiguous)
  int32_t bt_stride;
  int32_t pg_shift;           // log2(page size)
  const uint32_t* row_offsets;
  const int64_t* row_pos;
  const int32_t* idx;
  const int64_t* append_base;
  __nv_bfloat16* out;
  float* lse;
  float* part_o;              // split partials (unnormalised O), or null
  float* part_ml;
  int n_splits;
  int per_split;              // positions per split (multiple of NP)
  int fused_combine;          // the splits of a row share one cluster and merge their partials in-kernel
  // Persistent launch: cluster c takes the pairs [c pq, min(tp, (c + 1) pq)) of the flattened list of
  // (row, head group, pair) units, row by row; a row cut between clusters leaves one float32 piece per
  // cluster (slot 0: the cluster's first unit, slot 1: its last) for the piece merge.
  int pq;                     // pairs per cluster
  int ppr;                    // pairs per (row, head group)
  int hgn;                    // head groups, H / 128
  int64_t tp;                 // pairs in total
  int32_t* status;
};

// One (row, head group) range of pairs that a cluster processes.
struct Item {
  int r, h0;                  // query row and first head
  int64_t j0, j1;             // positions [j0, j1) of the row's list (selected, then appended)
  int n_pairs;
  int g0;                     // the CTA's running pair index of the first pair (ring and barrier phases)
  int slot;                   // -1: the whole row (normalised output); else the piece slot of a cut row
};

template <bool PERSIST>
__device__ __forceinline__ int n_items_of(const Params& p) {
  if (!PERSIST) return 1;
  const int64_t a0 = (int64_t)blockIdx.x * p.pq, a1 = min(p.tp, a0 + (int64_t)p.pq);
  return a1 > a0 ? (int)((a1 - 1) / p.ppr - a0 / p.ppr + 1) : 0;
}
template <bool PERSIST>
__device__ __forceinline__ Item item_of(const Params& p, int i) {
  Item I;
  const int64_t total = (int64_t)p.n_idx + p.n_append;
  if (!PERSIST) {   // one (row, head group, split) per cluster
    I.r = blockIdx.x;
    I.h0 = (int)(blockIdx.y >> 1) * HG;
    I.j0 = (int64_t)blockIdx.z * p.per_split;
    I.j1 = min(total, I.j0 + (int64_t)p.per_split);
    I.n_pairs = I.j1 > I.j0 ? (int)((I.j1 - I.j0 + NP - 1) / NP) : 0;   // a last half pair: zero rows
    I.g0 = 0;
    I.slot = -1;
    return I;
  }
  const int64_t a0 = (int64_t)blockIdx.x * p.pq, a1 = min(p.tp, a0 + (int64_t)p.pq);
  const int64_t u = a0 / p.ppr + i;
  const int64_t ua = u * p.ppr, ub = ua + p.ppr;
  const int64_t pa = max(a0, ua), pb = min(a1, ub);
  I.r = (int)(u / p.hgn);
  I.h0 = (int)(u % p.hgn) * HG;
  I.j0 = (pa - ua) * NP;
  I.j1 = min(total, (pb - ua) * NP);
  I.n_pairs = (int)(pb - pa);
  I.g0 = (int)(pa - a0);
  I.slot = (pa == ua && pb == ub) ? -1 : (i == 0 ? 0 : 1);
  return I;
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"((uint32_t)__cvta_generic_to_shared(b)),
               "r"(bytes) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"((uint64_t)map), "r"(x), "r"(y), "r"((uint32_t)__cvta_generic_to_shared(bar)) : "memory");
}
// TMA stores of one shared-memory box (bulk async-group of the issuing thread)
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
               ::"l"((uint64_t)map), "r"(x), "r"(y), "r"(src) : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];"
               ::"l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(src) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}
// 4 rows (y0..y3) x one box of columns starting at x
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int x, int y0, int y1, int y2,
                                            int y3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4, %5, %6}], [%7];" ::"r"(dst),
      "l"((uint64_t)map), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"((uint32_t)__cvta_generic_to_shared(bar))
      : "memory");
}

__device__ __forceinline__ uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t c) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(c));
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(b)) : "memory");
}
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t par, volatile int* abort_flag, int32_t* status) {
  return mbar::wait<false>(b, par, abort_flag, status, WAIT_LIMIT_NS);
}
// One lane of a converged warp (the lowest), as a warp-uniform branch: the
// issuing role runs with all 32 lanes so that addresses and descriptors stay
// in uniform registers, and only the elected lane issues TMA / MMA.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile("{\n .reg .b32 rx;\n .reg .pred px;\n elect.sync rx|px, 0xffffffff;\n selp.b32 %0, 1, 0, px;\n}\n"
               : "=r"(pred));
  return pred != 0;
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void commit(uint64_t* b) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(b)) : "memory");
}

// K-major (or MN-major) 128-byte-swizzle descriptor.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// kind::f16 instruction descriptors: D = F32, A = B = BF16, A K-major.
constexpr uint32_t IDESC_QK = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(NP >> 3) << 17) | ((uint32_t)(HG >> 4) << 24);
constexpr uint32_t IDESC_PV =
    (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((uint32_t)(DVH >> 3) << 17) | ((uint32_t)(HG >> 4) << 24);

__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
               ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
               ::"r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

#define TM_REGS32(r) \
  "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), \
  "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),      \
  "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),     \
  "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
#define TM_IN32(r) \
  "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), \
  "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),  \
  "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),   \
  "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])

__device__ __forceinline__ void tm_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
               "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : TM_REGS32(r) : "r"(taddr));
}
__device__ __forceinline__ void tm_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
               "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
               ::"r"(taddr), TM_IN32(r) : "memory");
}
__device__ __forceinline__ void tm_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
               ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
               "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
               : "memory");
}
__device__ __forceinline__ void tm_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tm_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 2^x with the hardware approximation (PTX ex2.approx.ftz.f32); -inf -> +0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);   // .x (low half) = lo
  return *(uint32_t*)&v;
}

// The same wait with cluster-scope acquire, for barriers whose bytes the other CTA completes.
__device__ __forceinline__ bool mbar_wait_cl(uint64_t* b, uint32_t par, volatile int* abort_flag, int32_t* status) {
  return mbar::wait<true>(b, par, abort_flag, status, WAIT_LIMIT_NS);
}
// shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t map_rank(uint32_t cta_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(cta_addr), "r"(rank));
  return r;
}
// 16 bytes into the other CTA's shared memory; completes 16 bytes on its barrier
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                            uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
               "r"(a), "r"(b), "r"(c), "r"(d), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// (lo, hi) -> fp16 pair with lo in the low half; out-of-range values saturate to +-65504
__device__ __forceinline__ uint32_t pack_f16_sat(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
// Arrive on a barrier of the other CTA.  Relaxed: the callers arrive after the values they read have
// been consumed (so the reads are complete), and a release at cluster scope costs thousands of cycles.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// fp16 pair -> two floats (exact)
__device__ __forceinline__ float2 f16x2_to_f32(uint32_t u) {
  __half2 h = *(__half2*)&u;
  return __half22float2(h);
}

// Position of an entry, or -1 (padding, past the split, or out of range: flagged).
__device__ __forceinline__ int64_t entry_pos(const Params& p, int64_t s, int64_t limit) {
  if (s == -1 || s == -2) return -1;
  if (s < 0 || s > limit) {
    flag_status(p.status, MTPSD_STATUS_INDEX_RANGE);
    return -1;
  }
  return s;
}
// Block-table entry of position s of request b (paged caches), or -1 when s has no page: the load is
// issued a tile before its value is used (entry_row), so its latency hides behind that tile.
__device__ __forceinline__ int32_t page_entry(const Params& p, int b, int64_t s) {
  if (!p.bt || s < 0 || (s >> p.pg_shift) >= p.bt_stride) return -1;
  return __ldg(p.bt + (int64_t)b * p.bt_stride + (s >> p.pg_shift));
}
// Pool row of position s (-1: padding / flagged), from the request's first row (contiguous) or its
// page entry (paged); a row outside the pool, or a position without a page, is flagged.
template <bool PAGED>
__device__ __forceinline__ int64_t entry_row(const Params& p, int64_t s, int64_t base, int32_t page) {
  if (s < 0) return -1;
  const int64_t row = PAGED ? (page < 0 ? -1 : (((int64_t)page << p.pg_shift) | (s & ((1LL << p.pg_shift) - 1))))
                            : base + s;
  if (row < 0 || row >= p.pool) {
    flag_status(p.status, MTPSD_STATUS_ROW_RANGE);
    return -1;
  }
  return row;
}

// Merge of the S split partials of heads [hlo, hhi) for one value half (the fused combine):
// o = sum_s 2^(m_s - m) o_s / sum_s 2^(m_s - m) l_s, 8 value dims per thread.  Warp w takes heads
// hlo + w + 13 i; the loads of HB heads are issued together before their arithmetic.
template <int S>
__device__ __noinline__ void merge_splits(const Params& p, int r, int h0, int hlo, int hhi, uint32_t rank) {
  constexpr int NW = THREADS / 32, HB = S == 2 ? 3 : (S == 3 ? 2 : 1);
  const int warp = threadIdx.x >> 5, d8 = threadIdx.x & 31;   // dims 8*d8 .. +7 of the half
  for (int i0 = 0; hlo + warp + NW * i0 < hhi; i0 += HB) {
    float2 mlv[HB][S];
    float4 ov[HB][S][2];
#pragma unroll
    for (int i = 0; i < HB; ++i) {
      const int hh = hlo + warp + NW * (i0 + i);
      if (hh < hhi) {
        const int64_t rh = (int64_t)r * p.H + h0 + hh;
#pragma unroll
        for (int t = 0; t < S; ++t) {
          mlv[i][t] = *(const float2*)(p.part_ml + ((rh * S + t) * 2 + rank) * 2);
          const float4* src = (const float4*)(p.part_o + (rh * S + t) * DV + rank * DVH) + 2 * d8;
          ov[i][t][0] = src[0];
          ov[i][t][1] = src[1];
        }
      }
    }
#pragma unroll
    for (int i = 0; i < HB; ++i) {
      const int hh = hlo + warp + NW * (i0 + i);
      if (hh >= hhi) break;
      const int64_t rh = (int64_t)r * p.H + h0 + hh;
      float m = -INFINITY;
#pragma unroll
      for (int t = 0; t < S; ++t) m = fmaxf(m, mlv[i][t].x);
      float l = 0.f;
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int t = 0; t < S; ++t) {
        if (mlv[i][t].x == -INFINITY) continue;
        const float w = ex2(mlv[i][t].x - m);
        l += w * mlv[i][t].y;
        const float4 a = ov[i][t][0], c = ov[i][t][1];
        acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
        acc[4] += w * c.x; acc[5] += w * c.y; acc[6] += w * c.z; acc[7] += w * c.w;
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint32_t w4[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) w4[k] = pack_bf16(acc[2 * k] * inv, acc[2 * k + 1] * inv);
      *((uint4*)(p.out + rh * DV + rank * DVH) + d8) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      if (rank == 0 && d8 == 0 && p.lse) p.lse[rh] = l > 0.f ? (m + log2f(l)) / LOG2E : -INFINITY;
    }
  }
}

// This CTA's 256 query dims of head h0 + h (thread = head = TMEM lane) -> TMEM columns [0,128) as bf16
// pairs, then the thread's arrival on q_ready.  Two rounds of 16 loads of 16 bytes, each round's loads
// in flight together.
__device__ __forceinline__ void load_q_tmem(const Params& p, uint32_t taddr, int r, int h0, int h, uint32_t rank,
                                            uint64_t* q_ready) {
  const bool head_ok = (h0 + h) < p.H;
  const uint4* src = (const uint4*)(p.q + ((int64_t)r * p.H + h0 + h) * DL + rank * QTM);
#pragma unroll
  for (int c2 = 0; c2 < QTM / 128; ++c2) {
    uint4 x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = head_ok ? src[c2 * 16 + i] : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      uint32_t v[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 y = x[cc * 8 + i];
        v[4 * i] = y.x; v[4 * i + 1] = y.y; v[4 * i + 2] = y.z; v[4 * i + 3] = y.w;
      }
      tm_st32(taddr + TM_Q + (2 * c2 + cc) * 32, v);
    }
  }
  tm_wait_st();
  fence_before();
  mbar_arrive(q_ready);
}
// The lines of those query dims (and on rank 0 of the rope dims) into L2, ahead of load_q_tmem and the
// rope copy.
__device__ __forceinline__ void prefetch_q_l2(const Params& p, int r, int h0, int h, uint32_t rank) {
  if (h0 + h >= p.H) return;
  const char* row = (const char*)(p.q + ((int64_t)r * p.H + h0 + h) * DL);
#pragma unroll
  for (int k = 0; k < 4; ++k) asm volatile("prefetch.global.L2 [%0];" ::"l"(row + rank * QTM * 2 + k * 128));
  if (rank == 0) asm volatile("prefetch.global.L2 [%0];" ::"l"(row + 2 * QTM * 2));
}

// PAGED: positions resolve to pool rows through the block table (the producers look a tile ahead).
// FP8KV: the latent pool holds 656-byte FP8 rows; tm_lat is a uint8 map of them with 128-byte boxes and
// tm_sc one with 16-byte boxes (the scale records); the producers dequantize into the pair buffers.
// PERSIST: one cluster per pair of SMs, each working through its range of pairs item by item (Params):
// every role keeps its running pair index across the items, so every ring slot and barrier phase
// advances as within one row; the sender warps load the next item's queries once the last QK of the
// previous item has completed, and the softmax warps write each item's O from registers (the gather
// ring is busy with the next item's rows).
template <bool PAGED, bool FP8KV, bool PERSIST>
__global__ void __launch_bounds__(THREADS, 1) sparse_mla_tc_kernel(const __grid_constant__ CUtensorMap tm_lat,
                                                                   const __grid_constant__ CUtensorMap tm_q,
                                                                   const __grid_constant__ CUtensorMap tm_st,
                                                                   const __grid_constant__ CUtensorMap tm_sc, Params p) {
  static_assert(!(FP8KV && PERSIST), "the persistent launch takes bf16 rows");
  constexpr int NPAIR_K = FP8KV ? 3 : NPAIR;   // pair buffers of the ring
  constexpr int NSTAGE_K = 2 * NPAIR_K;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(sm + OFF_BAR);
  uint64_t* c_full = bars;                 // per tile stage: the producers' bytes landed
  uint64_t* c_empty = bars + NSTAGE;       // per pair buffer: its PV completed (NPAIR_K used)
  uint64_t* s_full = c_empty + NPAIR;      // partial scores of the pair in score buffer s are in TMEM
  uint64_t* f_full = (uint64_t*)(sm + OFF_F + 4 * FD * F_TILE);   // FP8KV: [producer][FD] staging tiles landed
  uint64_t* p_full = s_full + 2;
  uint64_t* pv_done = p_full + 2;
  uint64_t* x_full = pv_done + 2;          // [slot][half]: half of receive slot s holds the other CTA's scores
  uint64_t* s_read = x_full + 4;           // the senders have read score buffer s
  uint64_t* x_free = s_read + 2;           // the other CTA has consumed what this CTA sent into its slot s
  uint64_t* stg_free = x_free + 2;         // the other CTA received the last staged pair (staging reusable)
  uint64_t* q_ready = stg_free + 1;
  uint64_t* drain = q_ready + 1;
  uint32_t* tmem_slot = (uint32_t*)(sm + OFF_MISC);
  volatile int* abort_flag = (volatile int*)(sm + OFF_MISC + 4);
  uint32_t* mask_s = (uint32_t*)(sm + OFF_MASK);   // [stage][producer]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // cluster (1, 2, S): rank = value half + 2 * split; the other half of the same split is crank ^ 1
  const uint32_t crank = cluster_rank();
  const uint32_t rank = crank & 1u;        // = the value half this CTA owns
  const uint32_t peer = crank ^ 1u;
  const int nch = rank == 0 ? 5 : 4;       // 64-dim chunks this CTA gathers
  const int split = blockIdx.z;
  const int n_items = n_items_of<PERSIST>(p);

  if (threadIdx.x == 0) {
    for (int i = 0; i < NSTAGE; ++i) mbar_init(&c_full[i], N_PROD);
    for (int i = 0; i < NPAIR; ++i) mbar_init(&c_empty[i], 1);
    if (FP8KV)
      for (int i = 0; i < 4 * FD; ++i) mbar_init(&f_full[i], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&pv_done[i], 1);
      mbar_init(&x_full[2 * i], 1);
      mbar_init(&x_full[2 * i + 1], 1);
      mbar_init(&s_read[i], 128);
      mbar_init(&x_free[i], 4);           // one arrival per softmax warp of the other CTA
    }
    // 128 softmax threads (query dims in TMEM), plus on rank 0 the first producer (rope dims by TMA)
    mbar_init(stg_free, 1);                 // one arrival by the other CTA's first softmax thread
    mbar_init(q_ready, rank == 0 ? 129 : 128);
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == MMA_WARP) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tmem_slot)), "r"(512));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (warp == PROD_WARP && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tm_lat) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tm_q) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tm_st) : "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  cluster_sync();                          // both CTAs' barriers exist before any remote arrival
  // Everything above touches no global memory and overlaps the previous kernel's tail (programmatic
  // dependent launch); its writes are visible from here on.
  griddep_wait();
  griddep_launch_dependents();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    // ------------------------------------------------ softmax / epilogue: thread = head
    const int h = threadIdx.x;                 // 0..127 = TMEM lane
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    if (!PERSIST) {   // the queries of the one item (the persistent launch: the sender warps, per item)
      const Item I0 = item_of<PERSIST>(p, 0);
      load_q_tmem(p, tmem + lane_off, I0.r, I0.h0, h, rank, q_ready);
    }
    // receive slot layout: two halves (positions 0..31, 32..63) that arrive separately; head h's 32
    // fp16 scores of a half are 4 pieces of 16 bytes at h*64, piece c at (c ^ ((h >> 1) & 3)), so that
    // eight consecutive heads touch all 32 banks
    const uint32_t x_own = saddr(sm + OFF_X) + (uint32_t)h * 64u;
    const uint32_t xfree_peer = map_rank(saddr(x_free), peer);
    const uint32_t stgfree_peer = map_rank(saddr(stg_free), peer);
    const uint32_t swz = (uint32_t)((h >> 1) & 3);
    bool ok = true;
    for (int it = 0; it < n_items && ok; ++it) {
      const Item I = item_of<PERSIST>(p, it);
      const int r = I.r, h0 = I.h0, n_pairs = I.n_pairs;
      const bool head_ok = (h0 + h) < p.H;
      float m_ref = -INFINITY, l = 0.f;
      // P: the CTA's running pair index (ring slots and barrier phases)
      for (int P = I.g0; P < I.g0 + n_pairs && ok; ++P) {
        const int s = P & 1;
        const uint32_t par = (P >> 1) & 1;
        const int st0 = 2 * (P % NPAIR_K);
        const uint32_t cpar = (P / NPAIR_K) & 1;
        if (h == 0) {
          mbar_arrive_expect_tx(&x_full[2 * s], XHALF_BYTES);
          mbar_arrive_expect_tx(&x_full[2 * s + 1], XHALF_BYTES);
        }
        ok = __all_sync(0xffffffffu, mbar_wait(&s_full[s], par, abort_flag, p.status));
        // the validity bits were written by the producers before they released the two tiles
        ok = ok && __all_sync(0xffffffffu, mbar_wait(&c_full[st0], cpar, abort_flag, p.status));
        ok = ok && __all_sync(0xffffffffu, mbar_wait(&c_full[st0 + 1], cpar, abort_flag, p.status));
        if (!ok) break;
        fence_after();
        const uint32_t* m0 = mask_s + st0 * 4;
        const uint32_t* m1 = mask_s + (st0 + 1) * 4;
        const uint64_t mask =
            (uint64_t)(m0[0] | m0[1] | m0[2] | m0[3]) | ((uint64_t)(m1[0] | m1[1] | m1[2] | m1[3]) << 32);
        // S = this CTA's partial (fp32, TMEM) + the other's (fp16, receive slot), in log2 units, and in the
        // same pass p = 2^(S - m_ref) against the current reference max (lazy max: the reference moves only
        // when a head's max grows by more than 2^RESCALE_LOG2, and then the pass runs again from TMEM and
        // the slot, which stay intact until P is published and the slot released).  The two halves of the
        // pair (positions 0..31, 32..63) are processed as they land.  The mask is the same for the whole
        // CTA, so the branch is uniform; a pair without padding skips the per-position select.  Masked
        // positions (-inf) give exact zeros.  The sum is taken over the fp32 values (their bf16 rounding
        // in P is unbiased and below the output tolerance).
        const bool full = mask == ~0ull;
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        float psum[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pk[32];
        auto half_pass = [&](const int half, const bool masked, const float mo) {
          uint32_t sr[32];
          tm_ld32(tmem + lane_off + TM_S0 + s * 64 + half * 32, sr);
          tm_wait_ld();
          const uint32_t xo = x_own + (uint32_t)s * XSLOT_BYTES + (uint32_t)half * XHALF_BYTES;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t px[4];
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(px[0]), "=r"(px[1]), "=r"(px[2]), "=r"(px[3])
                         : "r"(xo + ((c ^ swz) << 4))
                         : "memory");
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int j = 8 * c + 2 * i;   // within the half
              const float2 o = f16x2_to_f32(px[i]);
              float v0 = fmaf(__uint_as_float(sr[j]), p.sl2, o.x);
              float v1 = fmaf(__uint_as_float(sr[j + 1]), p.sl2, o.y);
              if (masked) {
                v0 = ((mask >> (32 * half + j)) & 1ull) ? v0 : -INFINITY;
                v1 = ((mask >> (32 * half + j + 1)) & 1ull) ? v1 : -INFINITY;
              }
              mx[i] = fmaxf(mx[i], fmaxf(v0, v1));
              const float e0 = ex2(v0 - mo), e1 = ex2(v1 - mo);
              pk[16 * half + (j >> 1)] = pack_bf16(e0, e1);
              psum[i] += e0 + e1;
            }
          }
        };
        const float mo0 = m_ref == -INFINITY ? 0.f : m_ref;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          ok = __all_sync(0xffffffffu, mbar_wait_cl(&x_full[2 * s + half], par, abort_flag, p.status));
          if (!ok) break;
          if (half == 1 && h == 0) mbar_arrive_remote(stgfree_peer);   // the other CTA may restage
          if (full) half_pass(half, false, mo0);
          else half_pass(half, true, mo0);
        }
        if (!ok) break;
        const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        // A head whose max grew past the reference takes a new one.  The decision is made per warp: the
        // TMEM loads and stores below are warp-collective, so every thread of a warp in which any head
        // moves runs them (the others keep their reference and scale O by 1).
        const bool grow = mt > m_ref + RESCALE_LOG2 || (m_ref == -INFINITY && mt > -INFINITY);
        if (__any_sync(0xffffffffu, grow)) {
          const float m_new = grow ? mt : m_ref;
          const bool scale_o = grow && m_ref > -INFINITY;   // O already holds this head's earlier pairs
          if (__any_sync(0xffffffffu, scale_o)) {
            const float alpha = scale_o ? ex2(m_ref - m_new) : 1.f;
            // O must not be touched while the previous PV is still accumulating
            mbar_wait(&pv_done[(P - 1) & 1], ((P - 1) >> 1) & 1, abort_flag, p.status);
            fence_after();
            l *= alpha;
#pragma unroll 1
            for (int c = 0; c < DVH / 32; ++c) {
              uint32_t o[32];
              tm_ld32(tmem + lane_off + TM_O + c * 32, o);
              tm_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tm_st32(tmem + lane_off + TM_O + c * 32, o);
            }
            tm_wait_st();
          }
          m_ref = m_new;
          // this pair's exponentials again, against the (possibly) new reference
          const float mo1 = m_ref == -INFINITY ? 0.f : m_ref;
#pragma unroll
          for (int i = 0; i < 4; ++i) psum[i] = 0.f;
          if (full) {
            half_pass(0, false, mo1);
            half_pass(1, false, mo1);
          } else {
            half_pass(0, true, mo1);
            half_pass(1, true, mo1);
          }
        }
        // slot s may be written again (pair P+2) once all four warps have consumed it
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(xfree_peer + (uint32_t)s * 8u);
        l += (psum[0] + psum[1]) + (psum[2] + psum[3]);
        // P overwrites the scores: the senders must have read them
        ok = __all_sync(0xffffffffu, mbar_wait(&s_read[s], par, abort_flag, p.status));
        if (!ok) break;
        tm_st32(tmem + lane_off + TM_S0 + s * 64, pk);
        tm_wait_st();
        fence_before();
        mbar_arrive(&p_full[s]);
      }
      // ------------------------------------------------ epilogue
      if (ok && n_pairs > 0) {
        const int last = I.g0 + n_pairs - 1;
        ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[last & 1], (last >> 1) & 1, abort_flag, p.status));
      }
      if (ok) fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      if constexpr (PERSIST) {
        // O leaves from registers (the gather ring already holds the next item's rows): each thread
        // writes its head's 256 value dims, 512 contiguous bytes of bf16, or 1 KB of float32 for a piece
        // of a cut row with the piece's (max, sum)
        if (!ok) break;
        const int64_t rh = (int64_t)r * p.H + h0 + h;
        if (I.slot < 0) {
          uint4* dst = (uint4*)(p.out + rh * DV + rank * DVH);
#pragma unroll 1
          for (int c = 0; c < DVH / 32; ++c) {
            uint32_t o[32];
            tm_ld32(tmem + lane_off + TM_O + c * 32, o);
            tm_wait_ld();
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              w[i] = pack_bf16(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
            if (head_ok) {
#pragma unroll
              for (int q = 0; q < 4; ++q)
                dst[c * 4 + q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
            }
          }
          if (head_ok && rank == 0 && p.lse) p.lse[rh] = l > 0.f ? (m_ref + log2f(l)) / LOG2E : -INFINITY;
        } else {
          const int64_t pc = ((int64_t)blockIdx.x * 2 + I.slot) * HG + h;   // piece row of this head
          uint4* dst = (uint4*)(p.part_o + pc * DV + rank * DVH);
#pragma unroll 1
          for (int c = 0; c < DVH / 32; ++c) {
            uint32_t o[32];
            tm_ld32(tmem + lane_off + TM_O + c * 32, o);
            tm_wait_ld();
#pragma unroll
            for (int q = 0; q < 8; ++q) dst[c * 8 + q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
          }
          float* ml = p.part_ml + (pc * 2 + rank) * 2;
          ml[0] = l > 0.f ? m_ref : -INFINITY;
          ml[1] = l;
        }
      } else {
        // O leaves through shared memory (the drained gather ring): each warp writes its 32 heads as
        // boxes of 32 rows x 128 bytes with the 128-byte swizzle (16-byte piece c of row i at c ^ (i & 7),
        // so the eight rows of a quarter warp hit all banks), then one lane stores them with TMA.
        const bool have_o = n_pairs > 0 && ok;
        const uint32_t row_off = (uint32_t)lane * 128u;
        const uint32_t sw = (uint32_t)(lane & 7);
        if (p.n_splits == 1) {
          const uint32_t stg = saddr(sm + OFF_C) + (uint32_t)warp * 16384u;   // 4 boxes of 64 bf16 columns
#pragma unroll 1
          for (int c = 0; c < DVH / 32; ++c) {
            uint32_t o[32];
            if (have_o) {
              tm_ld32(tmem + lane_off + TM_O + c * 32, o);
              tm_wait_ld();
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = 0u;
            }
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              w[i] = pack_bf16(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
            const uint32_t box = stg + (uint32_t)(c >> 1) * 4096u + row_off;
#pragma unroll
            for (int q = 0; q < 4; ++q)
              st_shared_v4(box + ((((uint32_t)(c & 1) * 4u + q) ^ sw) << 4), w[4 * q], w[4 * q + 1], w[4 * q + 2],
                           w[4 * q + 3]);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // visible to the TMA store
          __syncwarp();
          if (ok && lane == 0) {
#pragma unroll
            for (int bx = 0; bx < DVH / 64; ++bx)
              tma_store_2d(&tm_st, stg + (uint32_t)bx * 4096u, (int)rank * DVH + bx * 64, r * p.H + h0 + warp * 32);
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");   // the staging is read before exit
          }
          __syncwarp();
          if (head_ok && rank == 0 && p.lse)
            p.lse[(int64_t)r * p.H + h0 + h] = l > 0.f ? (m_ref + log2f(l)) / LOG2E : -INFINITY;
        } else {
          const uint32_t stg = saddr(sm + OFF_C) + (uint32_t)warp * 32768u;   // 8 boxes of 32 float columns
#pragma unroll 1
          for (int c = 0; c < DVH / 32; ++c) {
            uint32_t o[32];
            if (have_o) {
              tm_ld32(tmem + lane_off + TM_O + c * 32, o);
              tm_wait_ld();
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = 0u;
            }
            const uint32_t box = stg + (uint32_t)c * 4096u + row_off;
#pragma unroll
            for (int q = 0; q < 8; ++q)
              st_shared_v4(box + (((uint32_t)q ^ sw) << 4), o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (ok && lane == 0) {
#pragma unroll
            for (int c = 0; c < DVH / 32; ++c)
              tma_store_3d(&tm_st, stg + (uint32_t)c * 4096u, (int)rank * DVH + c * 32, split,
                           r * p.H + h0 + warp * 32);
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            // the partials are complete in global memory, and ordered before this thread's later
            // generic accesses (the cluster barrier that releases them to the merging CTAs)
            asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
            asm volatile("fence.proxy.async.global;" ::: "memory");
          }
          __syncwarp();
          if (head_ok) {   // each value half carries its own (max, sum)
            float* ml = p.part_ml + ((((int64_t)r * p.H + h0 + h) * p.n_splits + split) * 2 + rank) * 2;
            ml[0] = l > 0.f ? m_ref : -INFINITY;
            ml[1] = l;
          }
        }
      }
    }
  } else if (warp < SEND_WARP + 4) {
    // ------------------------------------------------ senders: thread = head of TMEM quadrant warp % 4
    // Each reads the partial scores of its head, scales them to log2 units, rounds them to fp16 and
    // stages them in its rows of the staging slot (same layout as a receive slot); lane 0 of each warp
    // then copies the warp's 32 rows of each half (2 KB) into the other CTA's receive slot with one bulk
    // copy per half, completing bytes on that half's x_full, so that the first half is on its way
    // while the second is converted.  The staging slot is rewritten only after the other CTA reported
    // that the previous pair landed (stg_free): a shared-to-cluster bulk copy has no completion
    // this CTA can wait on.
    const int h = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t x_peer0 = map_rank(saddr(sm + OFF_X), peer);
    const uint32_t xfull_peer = map_rank(saddr(x_full), peer);
    const uint32_t stg0 = saddr(sm + OFF_STG);
    const uint32_t stg_row = stg0 + (uint32_t)h * 64u;
    const uint32_t swz = (uint32_t)((h >> 1) & 3);
    const uint32_t off = (uint32_t)(warp & 3) * 32u * 64u;   // this warp's rows within a half
    bool ok = true;
    int q_issued = 0;   // rope query loads issued by this warp (rank 0, first sender warp)
    for (int it = 0; it < n_items && ok; ++it) {
      const Item I = item_of<PERSIST>(p, it);
      if (PERSIST) {
        // The item's queries.  TMEM columns [0,128) and the rope dims in shared memory are free: this warp
        // waited for the previous item's last QK to complete (its s_full) in its last pair.
        if (rank == 0 && warp == SEND_WARP) {
          if (elect_one()) {
            mbar_arrive_expect_tx(q_ready, HG * 128);
            tma_load_2d(saddr(sm + OFF_QR), &tm_q, 512, I.r * p.H + I.h0, q_ready);
          }
          __syncwarp();
          ++q_issued;
        }
        load_q_tmem(p, tmem + lane_off, I.r, I.h0, h, rank, q_ready);
        if (it + 1 < n_items) {   // the next item's queries into L2 while this one runs
          const Item In = item_of<PERSIST>(p, it + 1);
          prefetch_q_l2(p, In.r, In.h0, h, rank);
        }
      }
      // P: the CTA's running pair index
      for (int P = I.g0; P < I.g0 + I.n_pairs && ok; ++P) {
        const int s = P & 1;
        const uint32_t par = (P >> 1) & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(&s_full[s], par, abort_flag, p.status));
        if (!ok) break;
        fence_after();
        uint32_t sr[64];
        tm_ld32(tmem + lane_off + TM_S0 + s * 64, sr);
        tm_ld32(tmem + lane_off + TM_S0 + s * 64 + 32, sr + 32);
        tm_wait_ld();
        fence_before();
        mbar_arrive(&s_read[s]);
        // the other CTA received pair P-1 (so its copies have read the staging slot)
        if (P >= 1) ok = __all_sync(0xffffffffu, mbar_wait_cl(stg_free, (P - 1) & 1, abort_flag, p.status));
        if (!ok) break;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t hx[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            hx[j] = pack_f16_sat(__uint_as_float(sr[32 * half + 2 * j]) * p.sl2,
                                 __uint_as_float(sr[32 * half + 2 * j + 1]) * p.sl2);
          const uint32_t row = stg_row + (uint32_t)half * XHALF_BYTES;
#pragma unroll
          for (int c = 0; c < 4; ++c)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + ((c ^ swz) << 4)),
                         "r"(hx[4 * c]), "r"(hx[4 * c + 1]), "r"(hx[4 * c + 2]), "r"(hx[4 * c + 3])
                         : "memory");
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // visible to the bulk copy
          // the other CTA has consumed what was sent into its slot s two pairs ago
          if (half == 0 && P >= 2)
            ok = __all_sync(0xffffffffu, mbar_wait_cl(&x_free[s], ((P - 2) >> 1) & 1, abort_flag, p.status));
          else
            __syncwarp();
          if (!ok) break;
          if (lane == 0) {
            const uint32_t ho = (uint32_t)s * XSLOT_BYTES + (uint32_t)half * XHALF_BYTES + off;
            asm volatile(
                "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                ::"r"(x_peer0 + ho), "r"(stg0 + (uint32_t)half * XHALF_BYTES + off), "r"(32 * 64),
                "r"(xfull_peer + (uint32_t)(2 * s + half) * 8u)
                : "memory");
          }
          __syncwarp();
        }
      }
    }
    if (PERSIST && q_issued > 0 && *abort_flag && lane == 0) {   // the last rope load lands before exit
      volatile int dummy = 0;
      mbar_wait(q_ready, (q_issued - 1) & 1, &dummy, p.status);
    }
  } else if (warp < PROD_WARP + N_PROD) {
    // ------------------------------------------------ producers
    // Producer pw gathers the 4-row groups g = pw and g = pw + 4 of every
    // 32-row tile: lane l (< 8) owns position 4*g + (l & 3) of group
    // g = pw + 4*(l >> 2); the other lanes mirror lanes 0..7.  The selection
    // entries are loaded PF tiles ahead (a register queue), so that the second
    // tile of a pair issues right after the first instead of waiting for an L2 load.
    const int pw = warp - PROD_WARP;
    const int ln = lane & 7;
    const int my_pos = 4 * (pw + 4 * (ln >> 2)) + (ln & 3);
    const int32_t oob = (int32_t)p.pool;   // a row outside the tensor map: TMA reads zeros
    // first latent column of local chunk c
    auto chunk_x = [&](int c) -> int { return rank == 0 ? (c < 4 ? c * 64 : 512) : 256 + c * 64; };
    if (!PERSIST && rank == 0 && pw == 0 && elect_one()) {
      // rope query dims of the 128 heads: one box of 64 dims x 128 rows (the persistent launch: the
      // sender warps, per item)
      const Item I0 = item_of<PERSIST>(p, 0);
      mbar_arrive_expect_tx(q_ready, HG * 128);
      tma_load_2d(saddr(sm + OFF_QR), &tm_q, 512, I0.r * p.H + I0.h0, q_ready);
    }
    __syncwarp();
    bool pok = true;   // no abort seen
    int issued = 0;    // bf16 rows: the CTA's running index of the next tile to issue
    for (int it = 0; it < n_items && pok; ++it) {
      const Item I = item_of<PERSIST>(p, it);
      const int r = I.r;
      const int64_t j0 = I.j0, j1 = I.j1;
      const int n_tiles = 2 * I.n_pairs;   // a last half pair is filled with zero rows
      const int T0 = 2 * I.g0;             // the CTA's running index of the item's first tile
      const int32_t* idx_row = p.idx + (int64_t)r * p.n_idx;
      // raw selected entry of position j (or a clamped dummy when j is an appended / past-the-split position)
      auto raw = [&](int64_t j) -> int32_t { return p.n_idx > 0 ? idx_row[min(j, (int64_t)p.n_idx - 1)] : 0; };
      // the first entries and the row's visible limit are loaded while the warp looks up the request
      constexpr int PF = 4;
      int32_t rq[PF];
#pragma unroll
      for (int i = 0; i < PF; ++i) rq[i] = i < n_tiles ? raw(j0 + (int64_t)i * NT + my_pos) : 0;
      const int64_t limit = p.row_pos[r] + p.row_pos_add;
      const int64_t abase = p.n_append > 0 ? p.append_base[r] + 1 : 0;   // first appended position
      const int breq = request_of_row_warp(p.row_offsets, p.B, (uint32_t)r);
      const int64_t base = PAGED ? 0 : p.cache_start[breq];
      // checked position of this lane's entry in tile t, from its raw selected entry
      auto tile_pos = [&](int t, int32_t rv) -> int64_t {
        const int64_t j = j0 + (int64_t)t * NT + my_pos;
        return entry_pos(p, j >= j1 ? -2 : (j < p.n_idx ? (int64_t)rv : abase + (j - p.n_idx)), limit);
      };
      // PAGED: tile t's position and page entry are taken one iteration ahead (the page load in flight)
      int64_t s_next = 0;
      int32_t pg_next = -1;
      if (PAGED) {
        s_next = n_tiles > 0 ? tile_pos(0, rq[0]) : -1;
        pg_next = page_entry(p, breq, s_next);
      }
      if constexpr (FP8KV) {
        // ---- FP8 rows: gather this warp's 8 rows of tile ti into staging slot ti % FD (FD tiles ahead of
        // the dequantization), then per tile t: dequantize them into the pair buffer, publish the validity
        // bits and arrive on the tile's c_full (one arrival per producer warp).
        uint8_t* fstg = sm + OFF_F + pw * FD * F_TILE;
        uint64_t* ffull = f_full + pw * FD;
        uint32_t mq[FD];
        int ti = 0, done = 0;
        bool ok = true;
        auto issue_tile = [&](int tt) {
          const int32_t craw = rq[0];
#pragma unroll
          for (int i = 0; i + 1 < PF; ++i) rq[i] = rq[i + 1];
          rq[PF - 1] = tt + PF < n_tiles ? raw(j0 + (int64_t)(tt + PF) * NT + my_pos) : 0;
          const int64_t sp = tile_pos(tt, craw);
          const int64_t row = entry_row<PAGED>(p, sp, base, PAGED ? page_entry(p, breq, sp) : -1);
          const bool valid = row >= 0 && lane < 8;
          mq[tt % FD] = __reduce_or_sync(0xffffffffu, valid ? (1u << my_pos) : 0u);
          const int yv = row >= 0 ? (int)row : oob;
          int y[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) y[i] = __shfl_sync(0xffffffffu, yv, i);
          const int k = tt % FD;
          const uint32_t sb = saddr(fstg + k * F_TILE);
          if (elect_one()) {
            mbar_arrive_expect_tx(&ffull[k], (uint32_t)(F_CODES + 2 * 64 + (rank == 0 ? F_ROPE : 0)));
#pragma unroll
            for (int gi = 0; gi < 2; ++gi) {
              const int* yg = y + 4 * gi;
#pragma unroll
              for (int hf = 0; hf < 2; ++hf)
                tma_gather4(sb + (gi * 2 + hf) * 512, &tm_lat, (int)rank * 256 + hf * 128, yg[0], yg[1], yg[2], yg[3],
                            &ffull[k]);
              tma_gather4(sb + F_CODES + gi * 128, &tm_sc, 512, yg[0], yg[1], yg[2], yg[3], &ffull[k]);
              if (rank == 0)
                tma_gather4(sb + F_CODES + F_SCL + gi * 512, &tm_lat, 528, yg[0], yg[1], yg[2], yg[3], &ffull[k]);
            }
          }
          __syncwarp();
        };
        for (int t = 0; t < n_tiles && ok; ++t) {
          while (ti < n_tiles && ti < t + FD) issue_tile(ti++);
          const int k = t % FD;
          ok = __all_sync(0xffffffffu, mbar_wait(&ffull[k], (t / FD) & 1, abort_flag, p.status));
          const int st = t % NSTAGE_K, P = t >> 1, q = P % NPAIR_K, R = P / NPAIR_K;
          if (ok && R > 0) ok = __all_sync(0xffffffffu, mbar_wait(&c_empty[q], (R - 1) & 1, abort_flag, p.status));
          if (!ok) break;
          const uint8_t* sb = fstg + k * F_TILE;
          uint8_t* pair = sm + OFF_C + q * PAIR_STRIDE;
          // One row half (128 codes, contiguous in staging) per step: lane l takes codes 4l .. 4l+3, so the
          // staging reads are conflict-free; they land as 8 bytes of bf16 in chunk (2 half + l / 16), 16-byte
          // slot (l % 16) / 2, at the 128-byte swizzle the MMAs read.
#pragma unroll 4
          for (int it = 0; it < 16; ++it) {
            const int row8 = it >> 1, hf = it & 1, gi = row8 >> 2, rig = row8 & 3;
            const int pos = (t & 1) * NT + 4 * (pw + 4 * gi) + rig;   // position within the pair
            const uint32_t w4 = *(const uint32_t*)(sb + (gi * 2 + hf) * 512 + rig * 128 + lane * 4);
            const float sc = *(const float*)(sb + F_CODES + gi * 128 + rig * 16 + ((int)rank * 2 + hf) * 4);
            uint32_t ow[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const __nv_fp8x2_storage_t pr = (__nv_fp8x2_storage_t)((w4 >> (16 * e)) & 0xffffu);
              const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pr, __NV_E4M3);   // exact
              const float2 f = __half22float2(*(const __half2*)&hr);
              const __nv_bfloat162 bv = __floats2bfloat162_rn(f.x * sc, f.y * sc);
              ow[e] = *(const uint32_t*)&bv;
            }
            const int cc = hf * 2 + (lane >> 4), kk = (lane & 15) >> 1;
            *(uint2*)(pair + cc * CHUNK_BYTES + pos * 128 + ((kk ^ (pos & 7)) << 4) + (lane & 1) * 8) =
                make_uint2(ow[0], ow[1]);
          }
          if (rank == 0) {   // rope bytes (bf16 already) into chunk 4, swizzled
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int id = lane * 2 + e, row8 = id >> 3, kk = id & 7, gi = row8 >> 2, rig = row8 & 3;
              const int pos = (t & 1) * NT + 4 * (pw + 4 * gi) + rig;
              *(uint4*)(pair + 4 * CHUNK_BYTES + pos * 128 + ((kk ^ (pos & 7)) << 4)) =
                  *(const uint4*)(sb + F_CODES + F_SCL + gi * 512 + rig * 128 + kk * 16);
            }
          }
          // the MMAs (async proxy) read what these generic stores wrote, and the next gathers into this
          // staging slot come after its reads
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            mask_s[st * 4 + pw] = mq[k];
            mbar_arrive(&c_full[st]);
          }
          __syncwarp();
          done = t + 1;
        }
        pok = ok;
        if (*abort_flag && lane == 0) {   // wait (bounded) for this warp's staging copies still in flight
          volatile int dummy = 0;
          for (int tt = done; tt < ti; ++tt) mbar_wait(&ffull[tt % FD], (tt / FD) & 1, &dummy, p.status);
          if (rank == 0 && pw == 0) mbar_wait(q_ready, 0, &dummy, p.status);
        }
      } else {
        for (int t = 0; t < n_tiles; ++t) {
          int64_t s_cur;
          int32_t pg_cur = -1;
          if (PAGED) {
#pragma unroll
            for (int i = 0; i + 1 < PF; ++i) rq[i] = rq[i + 1];
            rq[PF - 1] = t + PF < n_tiles ? raw(j0 + (int64_t)(t + PF) * NT + my_pos) : 0;
            s_cur = s_next;
            pg_cur = pg_next;
            s_next = t + 1 < n_tiles ? tile_pos(t + 1, rq[0]) : -1;
            pg_next = page_entry(p, breq, s_next);
          } else {
            const int32_t craw = rq[0];
#pragma unroll
            for (int i = 0; i + 1 < PF; ++i) rq[i] = rq[i + 1];
            rq[PF - 1] = t + PF < n_tiles ? raw(j0 + (int64_t)(t + PF) * NT + my_pos) : 0;
            s_cur = craw;   // resolved after the wait below, as its position
          }
          const int tg = T0 + t;   // running tile index: ring stage and pair buffer
          const int st = tg % NSTAGE_K, P = tg >> 1, q = P % NPAIR_K, R = P / NPAIR_K;
          if (R > 0 && !__all_sync(0xffffffffu, mbar_wait(&c_empty[q], (R - 1) & 1, abort_flag, p.status))) {
            pok = false;
            break;
          }
          if (!PAGED) s_cur = tile_pos(t, (int32_t)s_cur);
          const int64_t row = entry_row<PAGED>(p, s_cur, base, pg_cur);
          const bool valid = row >= 0 && lane < 8;
          const uint32_t bits = __reduce_or_sync(0xffffffffu, valid ? (1u << my_pos) : 0u);
          if (lane == 0) mask_s[st * 4 + pw] = bits;
          const int yv = row >= 0 ? (int)row : oob;
          int y[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) y[i] = __shfl_sync(0xffffffffu, yv, i);
          const uint32_t dst = saddr(sm + OFF_C + q * PAIR_STRIDE + (t & 1) * (NT * 128));
          if (elect_one()) {
            mbar_arrive_expect_tx(&c_full[st], (uint32_t)nch * 1024u);
#pragma unroll
            for (int gi = 0; gi < 2; ++gi) {
              const int g = pw + 4 * gi;
#pragma unroll
              for (int c = 0; c < NCH_MAX; ++c)
                if (c < nch)
                  tma_gather4(dst + c * CHUNK_BYTES + g * 512, &tm_lat, chunk_x(c), y[4 * gi], y[4 * gi + 1],
                              y[4 * gi + 2], y[4 * gi + 3], &c_full[st]);
            }
          }
          __syncwarp();
          issued = tg + 1;
        }
      }
    }
    if (!FP8KV && *abort_flag && lane == 0) {   // wait (bounded) for this CTA's copies still in flight
      volatile int dummy = 0;
      for (int st = 0; st < NSTAGE_K; ++st) {
        const int n = issued / NSTAGE_K + (st < issued % NSTAGE_K ? 1 : 0);
        if (n > 0) mbar_wait(&c_full[st], (n - 1) & 1, &dummy, p.status);
      }
      if (!PERSIST && rank == 0 && pw == 0) mbar_wait(q_ready, 0, &dummy, p.status);
    }
  } else {
    // ------------------------------------------------ MMA issue (warp 12; one elected lane issues)
    const uint64_t qr_desc = desc_sw128(saddr(sm + OFF_QR), 16, 1024);
    const uint64_t c_desc0 = desc_sw128(saddr(sm + OFF_C), 16, 1024);
    const uint64_t v_desc0 = desc_sw128(saddr(sm + OFF_C), CHUNK_BYTES, 1024);
    const int nk = nch * 4;
    // The MMAs follow a fixed order: QK(0), then for every pair P, QK(P+1) (its S buffer was last read
    // by PV(P-1), issued before it: the MMAs execute in issue order) and PV(P) once the softmax
    // published P.  The waits suspend the warp (try_wait) instead of polling, so the softmax warp that
    // shares this scheduler keeps its issue slots.
    auto issue_qk = [&](int nq) -> bool {
      const int bq = nq % NPAIR_K;
      const uint32_t par = (nq / NPAIR_K) & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&c_full[2 * bq], par, abort_flag, p.status) &&
                                       mbar_wait(&c_full[2 * bq + 1], par, abort_flag, p.status)))
        return false;
      fence_after();
      const uint64_t cd = c_desc0 + (uint64_t)((bq * PAIR_STRIDE) >> 4);
      const uint32_t d = tmem + TM_S0 + (nq & 1) * 64;
      if (elect_one()) {
        // partial S over this CTA's chunks: 0..3 with A from TMEM, rank 0's rope chunk with A from shared memory
#pragma unroll
        for (int k = 0; k < NCH_MAX * 4; ++k) {
          if (k < nk) {
            const uint32_t boff = (uint32_t)((k >> 2) * CHUNK_BYTES + (k & 3) * 32);   // chunk, 32-byte K step
            if (k < QTM / 16)
              mma_ts(d, tmem + TM_Q + k * 8, cd + (boff >> 4), IDESC_QK, k > 0 ? 1u : 0u);
            else
              mma_ss(d, qr_desc + (uint64_t)(((k & 3) * 32) >> 4), cd + (boff >> 4), IDESC_QK, 1u);
          }
        }
        commit(&s_full[nq & 1]);
      }
      __syncwarp();
      return true;
    };
    // The pairs of all items run in one sequence (np: the CTA's running pair index), in the order above
    // except at an item boundary: the first QK of an item waits for its queries (q_ready), which the
    // sender warps load once the previous item's last QK completed, so the previous item's last PV is
    // issued before it (its epilogue does not wait for the new queries; measured faster than the other
    // order).  The first PV of an item overwrites O.
    const int n_total = PERSIST ? (int)(min(p.tp, (int64_t)(blockIdx.x + 1) * p.pq) - (int64_t)blockIdx.x * p.pq)
                                : item_of<PERSIST>(p, 0).n_pairs;
    int q_item = 0, q_start = 0;   // the next item whose queries the QKs wait for, and its first pair
    auto qk = [&](int g) -> bool {
      if (g == q_start) {
        if (!__all_sync(0xffffffffu, mbar_wait(q_ready, q_item & 1, abort_flag, p.status))) return false;
        fence_after();
        ++q_item;
        q_start = q_item < n_items ? item_of<PERSIST>(p, q_item).g0 : INT_MAX;
      }
      return issue_qk(g);
    };
    bool ok = true;
    if (n_total == 0 && n_items > 0)   // nothing to compute: the query copies still land before exit
      ok = __all_sync(0xffffffffu, mbar_wait(q_ready, 0, abort_flag, p.status));
    if (ok && n_total > 0) ok = qk(0);
    int p_item = 0, p_start = 0;   // the item of the next PV and its first pair
    for (int np = 0; np < n_total && ok; ++np) {
      const bool boundary = np + 1 == q_start;   // np + 1 is the first pair of the next item
      if (np + 1 < n_total && !boundary && !qk(np + 1)) {
        ok = false;
        break;
      }
      const bool first = np == p_start;
      if (first) {
        ++p_item;
        p_start = p_item < n_items ? item_of<PERSIST>(p, p_item).g0 : INT_MAX;
      }
      // O += P(np) V(np): A = P from TMEM, B = chunks 0..3 of the pair buffer as MN-major (N = 256 dims)
      const int sp = np & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&p_full[sp], (np >> 1) & 1, abort_flag, p.status))) {
        ok = false;
        break;
      }
      fence_after();
      const int bp = np % NPAIR_K;
      const uint64_t vd = v_desc0 + (uint64_t)((bp * PAIR_STRIDE) >> 4);
      if (elect_one()) {
#pragma unroll
        for (int k = 0; k < NP / 16; ++k)
          mma_ts(tmem + TM_O, tmem + TM_S0 + sp * 64 + k * 8, vd + (uint64_t)((k * 16 * 128) >> 4), IDESC_PV,
                 (!first || k > 0) ? 1u : 0u);
        commit(&pv_done[sp]);
        commit(&c_empty[bp]);
      }
      __syncwarp();
      if (np + 1 < n_total && boundary && !qk(np + 1)) ok = false;
    }
    if (elect_one()) commit(drain);
    __syncwarp();
    volatile int dummy = 0;
    mbar_wait(drain, 0, &dummy, p.status);
  }

  fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
  }
  // the other CTA no longer writes into this CTA's shared memory; with a fused combine, every split of
  // this row has also written its partials (the barrier releases and acquires at cluster scope)
  cluster_sync();
  if (!PERSIST && p.fused_combine) {
    const Item I0 = item_of<PERSIST>(p, 0);
    const int hlo = split * HG / p.n_splits, hhi = (split + 1) * HG / p.n_splits;
    switch (p.n_splits) {
      case 2: merge_splits<2>(p, I0.r, I0.h0, hlo, hhi, rank); break;
      case 3: merge_splits<3>(p, I0.r, I0.h0, hlo, hhi, rank); break;
      default: merge_splits<4>(p, I0.r, I0.h0, hlo, hhi, rank); break;
    }
  }
}

// Merge of the pieces of the rows cut between clusters of the persistent launch.  CTA (c, y) takes heads
// 4y .. 4y + 3 of the row (unit) cut at pair (c + 1) pq when that is the first cut inside it; the unit's
// pieces are those of the clusters whose ranges overlap it (slot 0 when the unit is the cluster's first,
// else slot 1).  Per head and value half, o = sum_k 2^(m_k - m) o_k / sum_k 2^(m_k - m) l_k; thread =
// (head, 8 value dims).  Every piece is read without a condition (a piece without mass holds zeros and
// weighs 0), so the loads of all pieces are in flight together.
constexpr int MERGE_HEADS = 4;
struct PieceMerge {
  __nv_bfloat16* out;
  float* lse;
  const float* part_o;
  const float* part_ml;
  int H, pq, ppr, hgn;
  int64_t tp;
};
__global__ void __launch_bounds__(64 * MERGE_HEADS) mla_piece_merge_kernel(PieceMerge a) {
  griddep_wait();                // the persistent kernel's pieces are visible from here on
  griddep_launch_dependents();
  const int64_t cut = (int64_t)(blockIdx.x + 1) * a.pq;
  if (cut >= a.tp || cut % a.ppr == 0) return;
  const int64_t u = cut / a.ppr, ua = u * a.ppr, ub = ua + a.ppr;
  if (ua / a.pq != (int64_t)blockIdx.x) return;   // an earlier cut of this unit merges it
  const int c_first = (int)(ua / a.pq), c_last = (int)((ub - 1) / a.pq);
  const int r = (int)(u / a.hgn), h0 = (int)(u % a.hgn) * HG;
  const int hh = blockIdx.y * MERGE_HEADS + (threadIdx.x >> 6);
  const int d8 = threadIdx.x & 63, half = d8 >> 5;   // value dims 8 d8 .. 8 d8 + 7
  auto piece = [&](int c) -> int64_t {   // piece row of head hh from cluster c
    return ((int64_t)c * 2 + ((int64_t)c * a.pq / a.ppr == u ? 0 : 1)) * HG + hh;
  };
  float m = -INFINITY;
#pragma unroll 4
  for (int c = c_first; c <= c_last; ++c) m = fmaxf(m, a.part_ml[(piece(c) * 2 + half) * 2]);
  float l = 0.f;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int c = c_first; c <= c_last; ++c) {
    const int64_t pc = piece(c);
    const float2 ml = *(const float2*)(a.part_ml + (pc * 2 + half) * 2);   // (max, sum) of the piece
    const float4* src = (const float4*)(a.part_o + pc * DV) + 2 * d8;
    const float4 x = src[0], y = src[1];
    const float w = ml.x == -INFINITY ? 0.f : ex2(ml.x - m);
    l += w * ml.y;
    acc[0] += w * x.x; acc[1] += w * x.y; acc[2] += w * x.z; acc[3] += w * x.w;
    acc[4] += w * y.x; acc[5] += w * y.y; acc[6] += w * y.z; acc[7] += w * y.w;
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const int64_t rh = (int64_t)r * a.H + h0 + hh;
  uint32_t w4[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) w4[k] = pack_bf16(acc[2 * k] * inv, acc[2 * k + 1] * inv);
  *((uint4*)(a.out + rh * DV) + d8) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
  if (d8 == 0 && a.lse) a.lse[rh] = l > 0.f ? (m + log2f(l)) / LOG2E : -INFINITY;
}

}  // namespace mtc

bool mla_tc_supported(const MlaPlan& p) {
  if ((p.dtype != MTPSD_BF16 && p.dtype != MTPSD_FP8_DS_MLA) || p.d_latent != 576 || p.d_v != 512) return false;
  if (p.H % mtc::HG != 0) return false;
  if (cc_major() != 10) return false;
  const char* env = getenv("MTPSD_MLA");
  if (env && env[0] == 'm') return false;   // "mma": the mma.sync kernel
  if (p.pool > 0x7ffffffeLL || (int64_t)p.R * p.H > 0x7fffffffLL) return false;
  if (((uintptr_t)p.latent % 16) || ((uintptr_t)p.q % 16)) return false;
  // the output and the split partials (workspace) are written by TMA stores
  if (((uintptr_t)p.out % 16) || ((uintptr_t)p.ws % 16)) return false;
  return tma_available();
}

namespace {
// Largest split count whose splits share one cluster (2 CTAs per split, 8 CTAs at most).
constexpr int MAX_FUSED_SPLITS = mtc::MAX_FUSED_SPLITS_K;

cudaLaunchConfig_t mla_tc_config(dim3 grid, int cluster_z, cudaStream_t st, cudaLaunchAttribute* attrs) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(mtc::THREADS);
  cfg.dynamicSmemBytes = mtc::SMEM_BYTES;
  cfg.stream = st;
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = 1;
  attrs[0].val.clusterDim.y = 2;
  attrs[0].val.clusterDim.z = cluster_z;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return cfg;
}
bool mla_tc_prepare() {
  static std::atomic<uint64_t> attr[6];
  return set_smem_limit_once(mtc::sparse_mla_tc_kernel<false, false, false>, mtc::SMEM_BYTES, attr[0]) &&
         set_smem_limit_once(mtc::sparse_mla_tc_kernel<true, false, false>, mtc::SMEM_BYTES, attr[1]) &&
         set_smem_limit_once(mtc::sparse_mla_tc_kernel<false, true, false>, mtc::SMEM_BYTES, attr[2]) &&
         set_smem_limit_once(mtc::sparse_mla_tc_kernel<true, true, false>, mtc::SMEM_BYTES, attr[3]) &&
         set_smem_limit_once(mtc::sparse_mla_tc_kernel<false, false, true>, mtc::SMEM_BYTES, attr[4]) &&
         set_smem_limit_once(mtc::sparse_mla_tc_kernel<true, false, true>, mtc::SMEM_BYTES, attr[5]);
}
// CTAs of this kernel that run at once with clusters of 2 x cluster_z CTAs (cached per device; -1 in
// the cache stands for "none fit").
int mla_tc_resident_ctas(int cluster_z) {
  static std::atomic<int> cache[kMaxCachedDevices][MAX_FUSED_SPLITS + 1];
  const int dev = current_device();
  const bool cacheable = dev >= 0 && dev < kMaxCachedDevices;
  if (cacheable) {
    const int v = cache[dev][cluster_z].load(std::memory_order_relaxed);
    if (v) return v < 0 ? 0 : v;
  }
  int n = 0, clusters = 0;
  cudaLaunchAttribute attrs[1];
  cudaLaunchConfig_t cfg = mla_tc_config(dim3(1, 2, cluster_z), cluster_z, 0, attrs);
  if (mla_tc_prepare() &&
      cudaOccupancyMaxActiveClusters(&clusters, (void*)mtc::sparse_mla_tc_kernel<false, false, false>, &cfg) == cudaSuccess &&
      clusters > 0)
    n = 2 * cluster_z * clusters;
  else
    n = cluster_z == 1 ? (num_sms() & ~1) : 0;
  cudaGetLastError();
  if (cacheable) cache[dev][cluster_z].store(n > 0 ? n : -1, std::memory_order_relaxed);
  return n;
}
}  // namespace

// The splits of a row share one cluster (and merge in the kernel) when there are few of them and
// such clusters fit on the device.
bool mla_tc_fuse(int n_splits) {
  return n_splits >= 2 && n_splits <= MAX_FUSED_SPLITS && mla_tc_resident_ctas(n_splits) > 0;
}

static int64_t split_plan(int R, int H, int64_t total, double* cost_out);

// The persistent launch for bf16 rows, where it is modelled faster than the split launch
// (MTPSD_MLA_PERSIST=0 turns it off, =1 takes it whenever it applies): every resident cluster gets the
// same number of consecutive pairs, so no wave is partly empty.  Measured on GB300, an item costs as
// much beyond its pairs as a row of the split launch does (four whole rows per cluster ran exactly as
// long as four waves), about PERSIST_ITEM_PAIRS pairs, and the piece merge about PERSIST_MERGE_PAIRS;
// the gain is the last wave's idle clusters.  The model counts every pair alike; ragged rows (short
// contexts leave masked pairs) are balanced by the split launch's dynamic CTA scheduling and not by the
// equal runs, so the persistent launch needs a PERSIST_MARGIN lead: the 384 uniform draft_extend rows
// take it (measured 311 -> 283 us), the 768 ragged verify rows of the decode workload do not (measured
// neutral to 10 us slower).
constexpr double PERSIST_ITEM_PAIRS = 4.5;
constexpr double PERSIST_MERGE_PAIRS = 10.0;
constexpr double PERSIST_MARGIN = 0.97;
bool mla_tc_persist_plan(int R, int H, int64_t total, int dtype, MlaPersist* pl) {
  if (dtype != MTPSD_BF16 || total <= 0 || R <= 0 || H % mtc::HG != 0) return false;
  const char* env = getenv("MTPSD_MLA_PERSIST");
  if (env && env[0] == '0') return false;
  const int slots = mla_tc_resident_ctas(1) / 2;
  if (slots < 1) return false;
  const int hgn = H / mtc::HG;
  const int64_t ppr = (total + mtc::NP - 1) / mtc::NP;
  const int64_t units = (int64_t)R * hgn;
  const int64_t tp = units * ppr;
  if (tp > 0x3fffffffLL) return false;   // the running pair index is an int
  const int64_t pq = (tp + slots - 1) / slots;
  pl->clusters = (int)((tp + pq - 1) / pq);
  pl->pq = (int)pq;
  pl->ppr = (int)ppr;
  pl->hgn = hgn;
  pl->tp = tp;
  pl->cut = false;
  for (int c = 0; c + 1 < pl->clusters; ++c)
    if (((int64_t)(c + 1) * pq) % ppr != 0) pl->cut = true;
  if (env && env[0] == '1') return true;
  double split_cost = 0.0;
  split_plan(R, H, total, &split_cost);
  const double items = (double)((pq + ppr - 1) / ppr + 1);
  const double cost = (double)pq + 4.0 + items * PERSIST_ITEM_PAIRS + (pl->cut ? PERSIST_MERGE_PAIRS : 0.0);
  return cost < PERSIST_MARGIN * split_cost;
}

// Pieces of the persistent launch: two per cluster (its first and its last unit), each 128 heads x 512
// float32 values, then per piece, head and value half a (max, sum) pair.
size_t mla_tc_persist_bytes(const MlaPersist& pl) {
  if (!pl.cut) return 0;
  const size_t rows = (size_t)pl.clusters * 2 * mtc::HG;
  return (rows * mtc::DV * sizeof(float) + 255) / 256 * 256 + rows * 4 * sizeof(float);
}

// Splits of the selected list that balance whole waves of resident clusters.
// Returns the positions per split (a multiple of NP).
// The split count s with the least modelled time, in units of one pair's time: waves of resident CTAs,
// each taking its split's pairs plus about four pairs of start-up.
static int64_t split_plan(int R, int H, int64_t total, double* cost_out) {
  const int64_t tiles = (total + mtc::NP - 1) / mtc::NP;
  const int64_t units = (int64_t)R * (H / mtc::HG) * 2;
  int64_t best = 1;
  double best_cost = 1e30;
  for (int64_t s = best; s <= best + 64 && s <= tiles; ++s) {
    const int64_t per = (tiles + s - 1) / s;
    const int slots = mla_tc_fuse((int)s) ? mla_tc_resident_ctas((int)s) : mla_tc_resident_ctas(1);
    const int64_t waves = (units * s + slots - 1) / slots;
    const double cost = (double)waves * (per + 4.0);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = s;
    }
  }
  if (cost_out) *cost_out = best_cost;
  return best;
}
int mla_tc_per_split(int R, int H, int64_t total) {
  const int64_t tiles = (total + mtc::NP - 1) / mtc::NP;
  const int64_t best = split_plan(R, H, total, nullptr);
  const int64_t per = ((tiles + best - 1) / best) * mtc::NP;
  return (int)(per > 0 ? per : mtc::NP);
}

// (max, sum) pairs per split that the kernel writes: one per value half
int mla_tc_ml_halves() { return 2; }

int launch_sparse_mla_tc(const MlaPlan& p, int n_splits, int per_split, float* part_o, float* part_ml,
                         cudaStream_t st, bool* combined, const MlaPersist* pl) {
  using namespace mtc;
  if (pl) {   // one item list per cluster; pieces of cut rows in the workspace
    n_splits = 1;
    per_split = 0;
    part_o = pl->cut ? (float*)p.ws : nullptr;
    part_ml = pl->cut ? (float*)((char*)p.ws + ((size_t)pl->clusters * 2 * HG * DV * sizeof(float) + 255) / 256 * 256)
                      : nullptr;
  }
  Params k;
  k.B = p.B; k.R = p.R; k.H = p.H; k.n_idx = p.n_idx; k.n_append = p.n_append;
  k.sl2 = p.scale * LOG2E; k.row_pos_add = p.row_pos_add;
  k.q = (const __nv_bfloat16*)p.q; k.latent = (const __nv_bfloat16*)p.latent; k.pool = p.pool;
  k.cache_start = p.cache_start; k.bt = p.pg.bt; k.bt_stride = p.pg.stride; k.pg_shift = p.pg.shift;
  k.row_offsets = p.row_offsets; k.row_pos = p.row_pos; k.idx = p.idx;
  k.append_base = p.append_base; k.out = (__nv_bfloat16*)p.out; k.lse = p.lse; k.part_o = part_o; k.part_ml = part_ml;
  k.n_splits = n_splits; k.per_split = per_split; k.status = p.status;
  k.fused_combine = !pl && mla_tc_fuse(n_splits) ? 1 : 0;
  if (combined) *combined = k.fused_combine != 0;
  k.pq = pl ? pl->pq : 0;
  k.ppr = pl ? pl->ppr : 0;
  k.hgn = pl ? pl->hgn : 0;
  k.tp = pl ? pl->tp : 0;
  alignas(64) CUtensorMap tm_lat, tm_q, tm_st, tm_sc;
  const bool fp8 = p.dtype == MTPSD_FP8_DS_MLA;
  // epilogue stores: boxes of 32 heads x 128 bytes, into out [R*H, 512] bf16 or into the split
  // partials [R*H, splits, 512] float32
  const uint64_t rh = (uint64_t)p.R * p.H;
  const uint64_t out_dims[2] = {(uint64_t)DV, rh}, out_strides[1] = {(uint64_t)DV * 2};
  const uint32_t out_box[2] = {64, 32};
  const uint64_t po_dims[3] = {(uint64_t)DV, (uint64_t)n_splits, rh};
  const uint64_t po_strides[2] = {(uint64_t)DV * 4, (uint64_t)DV * 4 * n_splits};
  const uint32_t po_box[3] = {32, 1, 32};
  const bool st_ok = n_splits == 1 ? make_tma_store_map(&tm_st, false, p.out, 2, out_dims, out_strides, out_box)
                                   : make_tma_store_map(&tm_st, true, part_o, 3, po_dims, po_strides, po_box);
  // latent gathers: bf16 rows in 64-value (128-byte) boxes, swizzled for the MMAs; FP8 rows as bytes
  // without swizzle, in 128-byte boxes (codes, rope) and 16-byte boxes (the scale records)
  const bool lat_ok = fp8 ? (make_tma_2d_plain_u8(&tm_lat, p.latent, FP8_ROW, (uint64_t)p.pool, 128) &&
                             make_tma_2d_plain_u8(&tm_sc, p.latent, FP8_ROW, (uint64_t)p.pool, 16))
                          : make_tma_2d(&tm_lat, 1, p.latent, DL, (uint64_t)p.pool, DL * 2, 64, 1, false);
  if (!fp8) tm_sc = tm_lat;   // unused
  if (!st_ok || !lat_ok || !make_tma_2d(&tm_q, 1, p.q, DL, (uint64_t)p.R * p.H, DL * 2, 64, HG, true)) {
    set_error("sparse_mla: cuTensorMapEncodeTiled failed");
    return MTPSD_ECUDA;
  }
  if (!mla_tc_prepare()) {
    set_error("sparse_mla_tc: cudaFuncSetAttribute failed");
    return MTPSD_ECUDA;
  }
  cudaLaunchAttribute attrs[2];
  const dim3 grid = pl ? dim3(pl->clusters, 2, 1) : dim3(p.R, (p.H / HG) * 2, n_splits);
  cudaLaunchConfig_t cfg = mla_tc_config(grid, k.fused_combine ? n_splits : 1, st, attrs);
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see launch_k()
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 2;
  cudaError_t e;
  if (pl)
    e = p.pg.bt ? cudaLaunchKernelEx(&cfg, sparse_mla_tc_kernel<true, false, true>, tm_lat, tm_q, tm_st, tm_sc, k)
                : cudaLaunchKernelEx(&cfg, sparse_mla_tc_kernel<false, false, true>, tm_lat, tm_q, tm_st, tm_sc, k);
  else if (fp8)
    e = p.pg.bt ? cudaLaunchKernelEx(&cfg, sparse_mla_tc_kernel<true, true, false>, tm_lat, tm_q, tm_st, tm_sc, k)
                : cudaLaunchKernelEx(&cfg, sparse_mla_tc_kernel<false, true, false>, tm_lat, tm_q, tm_st, tm_sc, k);
  else
    e = p.pg.bt ? cudaLaunchKernelEx(&cfg, sparse_mla_tc_kernel<true, false, false>, tm_lat, tm_q, tm_st, tm_sc, k)
                : cudaLaunchKernelEx(&cfg, sparse_mla_tc_kernel<false, false, false>, tm_lat, tm_q, tm_st, tm_sc, k);
  if (e != cudaSuccess) {
    set_error("sparse_mla_tc: launch failed: %s", cudaGetErrorString(e));
    return MTPSD_ECUDA;
  }
  int rc = check_launch("sparse_mla_tc");
  if (rc || !pl || !pl->cut) return rc;
  PieceMerge a;
  a.out = (__nv_bfloat16*)p.out;
  a.lse = p.lse;
  a.part_o = part_o;
  a.part_ml = part_ml;
  a.H = p.H;
  a.pq = pl->pq;
  a.ppr = pl->ppr;
  a.hgn = pl->hgn;
  a.tp = pl->tp;
  launch_k(mla_piece_merge_kernel, dim3((unsigned)(pl->clusters - 1), HG / MERGE_HEADS), 64 * MERGE_HEADS, 0, st, a);
  return check_launch("sparse_mla_piece_merge");
}

}  // namespace mtpsd
