// MLA decode attention on the fifth-generation tensor cores (tcgen05 with
// TMEM accumulators), fed by TMA tensor copies, sm_103a.
//
// Irminsul: MLA-Native Position-Independent Caching for Agentic LLM Serving,
// 2.1-2.2: every query head h attends to the shared latent rows
// row_t = [cKV_t (512) | k_r,t (64)], with the query absorbed into the latent
// space, q_h = [q_nope,h (512) | q_rope,h (64)].  A chunk token's rope key is
// used rotated by its chunk's delta, which needs no rotated copy: either the
// query's rope part is rotated by R(-delta) instead (q . R(delta) k =
// (R(-delta) q) . k, R orthogonal), or the stored key is rotated on its way
// through shared memory:
//   s_h,t = scale * [q_nope,h | q_rope,h] . [cKV_t | R(delta_t) k_r,t] + bias_t,
//   out_h = sum_t softmax(s_h)_t cKV_t      (512 dims, before W_UV).
// bias: LegoLink's pseudo-sink suppression (EPIC Guide: Position-Independent
// Caching for LLM Serving, LegoLink "1. Identifying and Neutralizing
// Pseudo-Sinks"): a constant logit offset on the first k tokens of every
// chunk not at position 0.
//
// A tile is up to four plan stages of one (layer, key), one per 16-row slot:
// 64 positions, the M of the score product.  A stage is up to 16 consecutive
// positions read from consecutive rows of one source, with at most two
// deltas (positions from its split on take the second), so a stage of
// consecutive rows runs across a chunk boundary.  Per tile, with warps by
// role:
//   * three producer warps read the tile's record (formed on the host, the
//     same in every layer) and load its rows into a ring of two tiles with
//     3-D TMA tile copies, one per 64-dim plane (128-byte swizzle) and per run
//     of stages that read consecutive rows (boxes of 16 to 64 rows);
//   * the query warp writes the query operands: q_nope at each key's first
//     tile, and the rope part --
//       16 heads per CTA: for each delta new to the tile's four entries,
//       R(-delta) q_rope as bf16 hi and lo rows;
//       32 heads: q_rope as given, at the key's first tile, and for every
//       tile the cos / sin of its stage deltas (lane f: frequency f);
//   * (32 heads) softmax warps 0-7 first rotate the rope keys: the two warps
//     of lane quadrant s take stage s, half of the dims each; threads t and
//     t + 16 rotate half of row t % 16's k_r each by its delta in fp32, swap
//     halves, and write its bf16 hi (t < 16) or lo part (t >= 16) into TMEM,
//     so that the quadrant's lanes hold an
//     A operand of 128 rows (stage s's hi rows in lanes 32 s .. + 15, its lo
//     rows in lanes 32 s + 16 .. + 31, two dims per column);
//   * two score issuers (one warp each) issue S = rows [q_nope | rope]^T into
//     TMEM: M = 64, 32 k-steps over the latent (even and odd into separate
//     partial sums), then the rope k-steps: 16 heads, 4 over the rope plane
//     against every entry's hi and lo rows; 32 heads, 4 of M = 128 with A
//     the rotated-key operand in TMEM, into one column per head, the hi
//     rows' part in lanes 0-15 of each lane quadrant and the lo rows' in
//     lanes 16-31;
//   * two value issuers issue O^T += V^T P^T once P is written: M = 128
//     latent dims (four M-tiles, two each), N = 2 x heads (P's hi and lo rows
//     side by side), K = the 16 positions of a stage; V^T is the same shared
//     planes read as an MN-major operand;
//   * softmax warp w, for stage w % 4's positions (TMEM lanes
//     32 (w % 4) .. + 15 of the M = 64 scores) and half of the heads, read
//     with the 16x256b shape so that each thread holds two positions, adds
//     the nope partial sums and the rope columns (16 heads: of each
//     position's entry; 32 heads: both lane halves), keeps a running max per head that is raised only
//     when a score passes it by more than kTcLazy (log2 units; O and l are
//     then rescaled), writes P = exp2(s - m) as bf16 hi and lo rows, and at
//     the key's last tile in this CTA writes the record (O, m, l) that
//     k_attend_merge combines.
// Rotating the query costs one pass over the heads per new delta and keeps
// the key path untouched: the better trade at 16 heads.  At 32 heads that
// pass is twice as long and sits on the score product's chain, and rotating
// the keys (a fixed 64 rows per tile, spread over the softmax warps) wins.
// The hi + lo splits keep about 16 significant bits of the rotated operand
// and of P; rows and q are bf16 already and every product accumulates in
// fp32 in TMEM.  Every wait is bounded: a wait that runs out raises
// PIC_DEV_TIMEOUT and tells the other roles to stop, and the CTA frees its
// TMEM before it leaves.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "pic_device.cuh"
#include "pic_internal.h"

namespace pic {
namespace {

using namespace dev;


constexpr int kMlaLatentDims = 512;
constexpr int kMlaRowDims = 576;                           // latent + 64-d rope key
constexpr int kTcStagesPerTile = 4;
constexpr int kTcPlanes = 9;                               // 8 latent planes + the rope plane
constexpr int kTcPlaneBytes = 64 * 128;                    // 64 rows x 64 dims x bf16
constexpr int kTcTileBytes = kTcPlanes * kTcPlaneBytes;    // 73,728
constexpr int kTcStageBytes = 16 * 128;                    // one stage's rows in one plane
constexpr float kTcLazy = 8.0f;
// warps 0-7 softmax (warp w: TMEM lane quadrant w % 4, heads of half w / 4),
// then a producer, the score-product issuer (it also holds the TMEM
// allocation), the query warp, the value-product issuer, a second
// score-product issuer, two more producers and a second value-product
// issuer.  A thread issuing alone puts out a small tcgen05.mma about every
// 55-70 cycles whatever its shape (a converged warp issuing from its elected
// lane, about every 29), and one warp issues TMA copies one lane after
// another (~35 ns each), so both are spread over warps.
constexpr int kTcSoftmaxWarps = 8;
constexpr int kTcProducer = 8, kTcMma = 9, kTcQuery = 10, kTcPv = 11, kTcMma2 = 12, kTcPv2 = 13, kTcProducer2 = 14;
__host__ __device__ constexpr int tc_score_issuers(int) { return 2; }
__host__ __device__ constexpr int tc_producers(int) { return 3; }
__host__ __device__ constexpr int tc_value_issuers(int) { return 2; }
__host__ __device__ constexpr int tc_threads(int hc) {
  return 32 * (9 + tc_score_issuers(hc) + tc_producers(hc) + tc_value_issuers(hc));
}
// TMEM columns: two score buffers of tc_score_cols(HC) (the latent score as
// NP = 2 partial sums, 2 HC columns, then the rope columns: HC, or with
// rotated queries NE x 2 x HC), then O^T: four
// M-tiles of 2 HC columns (the hi and lo parts of P side by side).  An M = 64
// score puts rows 16 q .. 16 q + 15 in lanes 0-15 of lane quadrant q; an
// M = 128 product row r in lane r.
// 16 heads per CTA rotate the query (NE entries), 32 the rope keys.
__host__ __device__ constexpr bool tc_rot_keys(int hc) { return hc >= 32; }
__host__ __device__ constexpr uint32_t tc_score_cols(int hc) {
  return tc_rot_keys(hc) ? 3u * static_cast<uint32_t>(hc) : 192u;
}
__host__ __device__ constexpr uint32_t tc_tmem_cols(int) { return 512u; }
constexpr int kTcFirst = 1, kTcLast = 2, kTcEnd = 4;       // tile flags

struct TcTile {
  int32_t ns;      // stages present
  int32_t layer;   // local layer
  int32_t key;
  int32_t flags;   // kTcFirst: first tile of the key in this CTA; kTcLast: its last; kTcEnd: the CTA's last
  int32_t n_tok[kTcStagesPerTile];   // positions of each stage
  int32_t sink[kTcStagesPerTile];    // their sink bits
  int32_t split[kTcStagesPerTile];   // first position of the stage's second delta (16: none)
  int32_t delta[kTcStagesPerTile];   // rotated keys: shift of the stage's positions [0, split)
  int32_t delta2[kTcStagesPerTile];  // and of [split, n_tok)
  int32_t entry[kTcStagesPerTile];   // rotated queries: entry of [0, split)
  int32_t entry2[kTcStagesPerTile];  // and of [split, n_tok)
  int32_t fresh;                     // entries this tile (re)writes
  int32_t ent_delta[kTcStagesPerTile];
  int32_t pad[3];
};

// Shared-memory layout (offsets from a 1024-byte aligned base).
template <int HC>
struct TcLayout {
  static constexpr bool kKeys = tc_rot_keys(HC);
  static constexpr int NE = kKeys ? 1 : 4;                      // entries of rotated query rows
  static constexpr int kRing = 0;                               // 2 tiles
  static constexpr int kQn = kRing + 2 * kTcTileBytes;         // q_nope: 8 planes x HC rows x 128 B
  static constexpr int kQnPlane = HC * 128;
  // the rope B operand: rotated keys, q_rope (HC rows); rotated queries, NE
  // entries x 2 halves of the heads x (HC / 2 hi + HC / 2 lo) rows; 128 B a row
  static constexpr int kRope = kQn + 8 * kQnPlane;
  static constexpr int kRopeBytes = kKeys ? (HC * 128 < 1024 ? 1024 : HC * 128) : NE * 2 * HC * 128;
  static constexpr int kPt = kRope + kRopeBytes;                // P^T: 2 buffers x (HC hi + HC lo) rows
  static constexpr int kPtBytes = 2 * HC * 128;
  static constexpr int kWmax = kPt + 2 * kPtBytes;              // float [2][4][HC]
  static constexpr int kLred = kWmax + 2 * 4 * HC * 4;          // float [4][HC]
  // rotated keys: cos / sin of each slot's stage deltas, float2 [2][4][2][32]
  static constexpr int kCs = kLred + 4 * HC * 4;
  static constexpr int kTiles = kCs + (kKeys ? 2 * 4 * 2 * 32 * 8 : 0);  // TcTile [2]
  static constexpr int kBars = kTiles + 2 * static_cast<int>(sizeof(TcTile));
  // full[2] empty[2] meta[2] q_ready[2] rot_done[2] s_full[2] p_full[2] pv_done[2] done[4]
  static constexpr int kNumBars = 20;
  static constexpr int kMisc = kBars + kNumBars * 8;            // tmem slot, abort flag
  static constexpr int kTotal = kMisc + 16;
  static constexpr int kAlloc = kTotal + 1024;                  // room to align the base
  static_assert(kQn % 1024 == 0 && kRope % 1024 == 0 && kPt % 1024 == 0 &&
                    kPtBytes % 1024 == 0,
                "operands sit on 1024-byte swizzle atoms");
  static_assert(kAlloc <= 227 * 1024, "shared memory");
};

// byte offset of element (row r, col c) of a 128B-swizzled tile of 128-byte rows
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + (((c >> 3) ^ (r & 7)) << 4) + (c & 7) * 2);
}

// tcgen05 shared-memory matrix descriptor: start, leading / stride byte
// offsets, version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}
// instruction descriptor of kind::f16: bf16 A and B, fp32 D, M x N, A K- or MN-major
__host__ __device__ constexpr uint32_t idesc(int M, int N, int a_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
// Both run on a whole converged warp and issue from its elected lane (the
// same lane every time, as the commit tracks that thread's products).  Issued
// this way, from operands the warp holds in common, a 64 x 16 product goes out
// about twice as often as from a branch taken by one lane.
__device__ __forceinline__ void tc_mma_elect(uint32_t d, uint64_t a, uint64_t b, uint32_t id, bool acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(id), "r"(acc ? 1u : 0u));
}
// the same with A in TMEM (M rows in lanes, two 16-bit elements per column)
__device__ __forceinline__ void tc_mma_tmem_a_elect(uint32_t d, uint32_t a, uint64_t b, uint32_t id, bool acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(b), "r"(id), "r"(acc ? 1u : 0u));
}
__device__ __forceinline__ void tc_commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float* v) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(r[j]);
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
               "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
               "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
               : "memory");
}

// N columns (8, or a multiple of 16) of this warp's TMEM lanes
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float* v) {
  if constexpr (N == 8) {
    tmem_ld8(taddr, v);
  } else {
#pragma unroll
    for (int j = 0; j < N; j += 16) tmem_ld16(taddr + j, v + j);
  }
}
template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const float* v) {
  if constexpr (N == 8) {
    tmem_st8(taddr, v);
  } else {
#pragma unroll
    for (int j = 0; j < N; j += 16) tmem_st16(taddr + j, v + j);
  }
}

// 16 TMEM lanes from a lane quadrant's base, G groups of 8 columns (shape
// 16x256b).  Per group g, thread t gets lanes t / 4 and t / 4 + 8 at columns
// 8 g + 2 (t % 4) and + 1, as v[4 g .. 4 g + 3] = (t / 4, c), (t / 4, c + 1),
// (t / 4 + 8, c), (t / 4 + 8, c + 1) (the layout measured on GB300).
template <int G>
__device__ __forceinline__ void tmem_ld16x256(uint32_t taddr, float* v) {
  uint32_t r[4 * G];
  if constexpr (G == 1) {
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
  } else if constexpr (G == 2) {
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
  } else {
    static_assert(G == 4, "16x256b groups");
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
  }
#pragma unroll
  for (int j = 0; j < 4 * G; ++j) v[j] = __uint_as_float(r[j]);
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// bounded wait that also gives up once another role has aborted
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, const volatile int* abort_flag,
                                              uint32_t spins) {
  for (uint32_t i = 0; i < spins; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
  }
  return false;
}

// named barrier 1 over the eight softmax warps (256 threads), returning the
// OR of every thread's predicate
__device__ __forceinline__ bool softmax_bar_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, 256, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v ? 1u : 0u)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(x);
  lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}
// the same for a pair, packed: x in the low halves, y in the high
__device__ __forceinline__ void split2_bf16(float x, float y, uint32_t& hi, uint32_t& lo) {
  hi = bf_pack(x, y);
  lo = bf_pack(x - bf_lo(hi), y - bf_hi(hi));
}

// grid: persistent CTAs, CTA c owns units [U c / G, U (c + 1) / G) of the
// (layer, tile) list; block: tc_threads(HC) threads (the warp roles above).
template <int PAIRING, int HC>
__global__ void __launch_bounds__(tc_threads(HC), 1)
    k_attend_mla_tc(const AttnParams P, const __grid_constant__ TcMaps maps) {
  // the merge that reads this kernel's records may be scheduled from now on
  // (it waits for this grid's completion before it reads anything)
  asm volatile("griddepcontrol.launch_dependents;");
  using L = TcLayout<HC>;
  constexpr bool NEOX = (PAIRING == kNeox);
  constexpr bool KEYS = L::kKeys;  // rotate the rope keys (else the query)
  constexpr int NE = L::NE;
  constexpr uint32_t kIdS = idesc(64, HC, 0);       // scores: latent k-steps
  constexpr uint32_t kIdK = idesc(128, HC, 0);      // rope k-steps over the rotated keys' hi and lo rows
  constexpr uint32_t kIdR = idesc(64, NE * 2 * HC, 0);  // rope k-steps against every entry (rotated queries)
  constexpr uint32_t kIdPV = idesc(128, 2 * HC, 1);  // O^T += V^T P^T, P's hi and lo rows side by side
  constexpr int kSI = tc_score_issuers(HC);
  constexpr int kNP = tc_producers(HC);
  constexpr int kVI = tc_value_issuers(HC);
  // the latent score accumulates in NP partial sums (k-step mod NP; with two
  // score issuers, one each), then one rope column per head
  constexpr int NP = 2;
  constexpr uint32_t kSCols = tc_score_cols(HC);
  constexpr uint32_t kRopeCol = NP * HC;
  constexpr uint32_t kOCol = 2 * kSCols;
  constexpr uint32_t kOColsPerTile = 2 * HC;
  constexpr uint32_t kCols = tc_tmem_cols(HC);
  // rotated keys: their A operand after O^T, 128 lanes x 32 columns (64 bf16 dims)
  constexpr uint32_t kRopeACol = kOCol + 4 * kOColsPerTile;
  static_assert(kRopeCol + (KEYS ? HC : NE * 2 * HC) <= kSCols && kOCol + 4 * kOColsPerTile <= kCols, "TMEM columns");
  static_assert(!KEYS || kRopeACol + 32 <= kCols, "TMEM columns: rotated-key operand");
  static_assert(KEYS || NE * 2 * HC == 128, "rope entry columns");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t base_u32 = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* full = bars + 0;        // a tile's rows landed (by tile parity, as below)
  uint64_t* empty = bars + 2;       // its value product finished: the ring slot is free
  uint64_t* meta_ready = bars + 4;  // its metadata is written
  uint64_t* q_ready = bars + 6;     // its query operands are written
  uint64_t* rot_done = bars + 8;    // its rope keys are rotated
  uint64_t* s_full = bars + 10;     // its score product finished
  uint64_t* p_full = bars + 12;     // its P is written
  uint64_t* pv_done = bars + 14;    // its value product finished
  uint64_t* done = bars + 16;       // each issuer's products all finished
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  TcTile* tiles = reinterpret_cast<TcTile*>(smem + L::kTiles);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t U = P.n_units, G = gridDim.x;
  const int64_t u_begin = U * blockIdx.x / G, u_end = U * (blockIdx.x + 1) / G;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&full[b], kNP);  // each producer warp arrives with the bytes of its copies
      mbar_init(&empty[b], kVI);  // every value issuer commits
      mbar_init(&meta_ready[b], 1);
      mbar_init(&q_ready[b], 1);
      mbar_init(&rot_done[b], kTcSoftmaxWarps);
      mbar_init(&s_full[b], kSI);  // every score issuer commits
      mbar_init(&p_full[b], kTcSoftmaxWarps);
      mbar_init(&pv_done[b], kVI);
    }
    for (int b = 0; b < 4; ++b) mbar_init(&done[b], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kTcMma) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                 "r"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  auto fail = [&]() {
    atomicOr(P.status, kDevTimeout);
    *abort_flag = 1;
  };
  const uint32_t spins = P.max_spins != 0 ? P.max_spins : kMaxSpins;
  const bool has_work = u_begin < u_end;

  const int prod = warp == kTcProducer ? 0 : (warp >= kTcProducer2 && warp < kTcProducer2 + kNP - 1) ? warp - kTcProducer2 + 1 : -1;
  if (prod >= 0 && has_work) {
    // ------------------------------------------------------------ producer
    // Starts the copies of the CTA's tiles, which the host formed (TcTileRec,
    // the same in every layer): the next tile's record is read while the
    // current slot drains, and consecutive stages that read consecutive rows
    // of one source share one TMA box of 16, 32, 48 or 64 rows.
    const int tpl = P.tc_tiles_per_layer;
    const int32_t* recs = reinterpret_cast<const int32_t*>(P.tc_tiles);
    constexpr int kRecInts = static_cast<int>(sizeof(TcTileRec) / 4);  // 44: lane l reads ints l and 32 + l
    auto load_rec = [&](int64_t ti, int& a, int& b) {
      a = 0;
      b = 0;
      if (ti < u_end) {
        const int64_t k = ti - (ti / tpl) * tpl;
        a = __ldg(recs + k * kRecInts + lane);
        if (lane < kRecInts - 32) b = __ldg(recs + k * kRecInts + 32 + lane);
      }
    };
    int ra, rb;  // the current tile's record
    load_rec(u_begin, ra, rb);
    int i = 0;
    bool failed = false;
    int issued = 0;
    for (int64_t ti = u_begin; ti < u_end; ++ti, ++i) {
      const int rt = i & 1;
      int na, nb;
      load_rec(ti + 1, na, nb);  // the next tile's, used in the next iteration
      const int layer = static_cast<int>(ti / tpl);
      const int ns = __shfl_sync(0xffffffffu, ra, 0), key = __shfl_sync(0xffffffffu, ra, 1);
      const int rflags = __shfl_sync(0xffffffffu, ra, 2), rfresh = __shfl_sync(0xffffffffu, ra, 3);
      // lane s < 4 holds stage s (lanes 4-31 a copy of stage lane % 4) and entry s
      const int s4 = lane & 3;
      const int my_n = __shfl_sync(0xffffffffu, ra, 4 + s4), my_sink = __shfl_sync(0xffffffffu, ra, 8 + s4);
      const int my_e0 = __shfl_sync(0xffffffffu, ra, 12 + s4), my_e1 = __shfl_sync(0xffffffffu, ra, 16 + s4);
      const int my_split = __shfl_sync(0xffffffffu, ra, 20 + s4), my_row = __shfl_sync(0xffffffffu, ra, 24 + s4);
      const int my_src = __shfl_sync(0xffffffffu, ra, 28 + s4), my_ed = __shfl_sync(0xffffffffu, rb, s4);
      const int my_d = __shfl_sync(0xffffffffu, rb, 4 + s4), my_d2 = __shfl_sync(0xffffffffu, rb, 8 + s4);
      const bool first = ti == u_begin || (rflags & kTcRecKeyFirst);
      const bool end = ti == u_end - 1;
      const int flags = (first ? kTcFirst : 0) | ((end || (rflags & kTcRecKeyLast)) ? kTcLast : 0) | (end ? kTcEnd : 0);
      // rotated queries: at the CTA's first tile every entry it uses is new to the query warp
      uint32_t used = lane < ns ? ((1u << my_e0) | (my_split < my_n ? (1u << my_e1) : 0u)) : 0u;
      used = __reduce_or_sync(0xffffffffu, used);
      const int fresh = ti == u_begin ? static_cast<int>(used) : rfresh;
      // The copies are planned before the slot is free, so that once it is
      // only the announcements and the copies themselves remain.  Stage k
      // continues stage k - 1's box when that stage is full and its rows go on.
      const int prow = __shfl_up_sync(0xffffffffu, my_row, 1);
      const int pflags = __shfl_up_sync(0xffffffffu, my_src, 1);
      const int pn = __shfl_up_sync(0xffffffffu, my_n, 1);
      const bool cont = lane > 0 && lane < ns && pn == 16 && pflags == my_src && my_row == prow + 16;
      const uint32_t cmask = __ballot_sync(0xffffffffu, cont);
      const bool leader = lane < ns && !cont;
      const uint32_t lmask = __ballot_sync(0xffffffffu, leader);
      const int ngroups = __popc(lmask);
      const int my_len = leader ? __ffs(~(cmask >> (lane + 1))) : 0;  // this stage and the ones continuing it
      const int z = P.layer_begin + layer;
      // copy q (box q / 9, plane q % 9; at most 36) goes to producer warp
      // q % kNP, lane (q / kNP) % 32; each warp announces its own bytes
      constexpr int kRounds = (4 * kTcPlanes + 32 * kNP - 1) / (32 * kNP);
      int cp_row[kRounds], cp_len[kRounds], cp_pl[kRounds];
      uint32_t cp_dst[kRounds];
      const CUtensorMap* cp_map[kRounds];
      uint32_t bytes = 0;
#pragma unroll
      for (int r = 0; r < kRounds; ++r) {
        const int q = prod + kNP * (lane + 32 * r);
        const int g = q / kTcPlanes;
        uint32_t m = lmask;
        for (int x = 0; x < g && m; ++x) m &= m - 1;  // drop the first g leaders
        const int src = m ? __ffs(m) - 1 : 0;
        cp_row[r] = __shfl_sync(0xffffffffu, my_row, src);
        const int fl = __shfl_sync(0xffffffffu, my_src, src);
        cp_len[r] = __shfl_sync(0xffffffffu, my_len, src);
        cp_pl[r] = g < ngroups ? q - g * kTcPlanes : kTcPlanes;
        cp_dst[r] = base_u32 + L::kRing + rt * kTcTileBytes + src * kTcStageBytes + cp_pl[r] * kTcPlaneBytes;
        cp_map[r] = cp_pl[r] < kTcPlanes ? ((fl & kAttnFromCache) ? &maps.cache[cp_len[r] - 1] : &maps.pool[cp_len[r] - 1])
                                         : nullptr;
        bytes += cp_pl[r] < kTcPlanes ? static_cast<uint32_t>(cp_len[r]) * kTcStageBytes : 0u;
      }
      bytes = __reduce_add_sync(0xffffffffu, bytes);
      // the slot's previous tile (i - 2) must be done before its metadata and rows are replaced
      if (i >= 2 && !__all_sync(0xffffffffu, wait_or_abort(&empty[rt], ((i >> 1) - 1) & 1, abort_flag, spins))) {
        failed = true;
        break;
      }
      if (prod == 0) {
        TcTile& t = tiles[rt];
        if (lane < 4) {
          t.n_tok[lane] = my_n;
          t.sink[lane] = my_sink;
          t.split[lane] = my_split;
          t.delta[lane] = my_d;
          t.delta2[lane] = my_d2;
          t.entry[lane] = my_e0;
          t.entry2[lane] = my_e1;
          t.ent_delta[lane] = my_ed;
        }
        if (lane == 0) {
          t.ns = ns;
          t.layer = layer;
          t.key = key;
          t.flags = flags;
          t.fresh = fresh;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&meta_ready[rt]);
      }
      // test hook (pic_debug_stall_next_launch): CTA 0 leaves this tile's rows
      // unrequested, so the waits for them run out and take the failure path
      const bool stalled = P.debug_stall != 0 && blockIdx.x == 0 && i == P.debug_stall - 1;
      if (!stalled) {
        if (lane == 0) mbar_arrive_expect_tx(&full[rt], bytes);
        __syncwarp();
#pragma unroll
        for (int r = 0; r < kRounds; ++r)
          if (cp_pl[r] < kTcPlanes) tma_load_3d(cp_dst[r], cp_map[r], 64 * cp_pl[r], cp_row[r], z, &full[rt]);
      }
      issued = i + 1;
      ra = na;
      rb = nb;
    }
    if (failed) {
      if (lane == 0) fail();
      // wait (bounded) for the copies of the last two tiles issued
      if (lane == 0)
        for (int k = (issued > 2 ? issued - 2 : 0); k < issued; ++k) mbar_wait_bounded(&full[k & 1], (k >> 1) & 1, spins);
    }
  } else if (warp == kTcQuery && has_work) {
    if constexpr (KEYS) {
      // --------------------------------------------------------------- query
      // For every tile, cos / sin of its stage deltas for the softmax warps'
      // key rotation (lane f: frequency f), written while the rows are still
      // on their way.  At each key's first tile in this CTA it also writes
      // the query operands, q_nope (8 planes) and q_rope (one plane), once
      // the previous tile's score product no longer reads them.  Arrives on
      // every tile.
      const float2 fq = __ldg(P.freq + lane);
      for (int i = 0;; ++i) {
        const int rt = i & 1;
        if (!__all_sync(0xffffffffu, wait_or_abort(&meta_ready[rt], (i >> 1) & 1, abort_flag, spins))) {
          if (lane == 0) fail();
          break;
        }
        const int t_flags = tiles[rt].flags, t_layer = tiles[rt].layer, t_key = tiles[rt].key;
        // the slot's previous tile (i - 2) was rotated before its softmax,
        // which ended before this tile's metadata was written
        float2* cs = reinterpret_cast<float2*>(smem + L::kCs) + rt * 256;
        for (int st = 0; st < tiles[rt].ns; ++st) {
          const int d1 = tiles[rt].delta[st], d2 = tiles[rt].delta2[st];
          float c = 1.0f, sn = 0.0f;
          if (d1 != 0) shift_cossin(d1, fq, c, sn);
          cs[st * 64 + lane] = make_float2(c, sn);
          if (tiles[rt].split[st] < tiles[rt].n_tok[st]) {
            c = 1.0f;
            sn = 0.0f;
            if (d2 != 0) shift_cossin(d2, fq, c, sn);
            cs[st * 64 + 32 + lane] = make_float2(c, sn);
          }
        }
        if (t_flags & kTcFirst) {
          if (i >= 1 &&
              !__all_sync(0xffffffffu, wait_or_abort(&s_full[(i - 1) & 1], ((i - 1) >> 1) & 1, abort_flag, spins))) {
            if (lane == 0) fail();
            break;
          }
          const int req = t_key / P.head_groups, hg = t_key - req * P.head_groups;
          const uint16_t* qh = P.q + ((static_cast<int64_t>(t_layer) * P.n_req + req) * P.num_q_heads + hg * HC) *
                                         static_cast<int64_t>(kMlaRowDims);
          // 72 16-byte pieces per head: 64 of q_nope, 8 of q_rope
          for (int c = lane; c < HC * 72; c += 32) {
            const int h = c / 72, ch = c - h * 72;
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(qh + h * kMlaRowDims) + ch);
            const int off = ch < 64 ? L::kQn + (ch >> 3) * L::kQnPlane : L::kRope;
            *reinterpret_cast<uint4*>(smem + off + sw128(h, (ch & 7) * 8)) = v;
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_ready[rt]);
        if (t_flags & kTcEnd) break;
      }
    } else {
      // --------------------------------------------------------------- query
      // Writes each tile's query operands: q_nope on a key change, and for each
      // fresh delta entry R(-delta) q_rope as bf16 hi and lo rows, once no
      // earlier score product still reads what they replace.
      float qa[HC], qb[HC];  // this lane's rope pair of every head (lane f: frequency f)
      uint32_t used_prev = 0;  // entries the previous tile read
  #pragma unroll
      for (int h = 0; h < HC; ++h) qa[h] = qb[h] = 0.0f;
      const int ia = NEOX ? lane : 2 * lane, ib = NEOX ? lane + 32 : 2 * lane + 1;
      for (int i = 0;; ++i) {
        const int rt = i & 1;
        if (!__all_sync(0xffffffffu, wait_or_abort(&meta_ready[rt], (i >> 1) & 1, abort_flag, spins))) {
          if (lane == 0) fail();
          break;
        }
        const TcTile t = tiles[rt];
        const bool key_change = (t.flags & kTcFirst) != 0;
        uint32_t used = 0;  // entries this tile reads
  #pragma unroll
        for (int st = 0; st < kTcStagesPerTile; ++st)
          if (st < t.ns) used |= (1u << t.entry[st]) | (t.split[st] < t.n_tok[st] ? (1u << t.entry2[st]) : 0u);
        if (key_change || t.fresh) {
          // Tile i - 2's score product is done (its value product freed the
          // slot tile i loads into); tile i - 1's may still read q_nope and its
          // entries, so wait for it when either is about to be rewritten.
          const bool clash = key_change || (static_cast<uint32_t>(t.fresh) & used_prev) != 0u;
          if (i >= 1 && clash &&
              !__all_sync(0xffffffffu, wait_or_abort(&s_full[(i - 1) & 1], ((i - 1) >> 1) & 1, abort_flag, spins))) {
            if (lane == 0) fail();
            break;
          }
          if (key_change) {
            const int req = t.key / P.head_groups, hg = t.key - req * P.head_groups;
            const uint16_t* qh = P.q + ((static_cast<int64_t>(t.layer) * P.n_req + req) * P.num_q_heads + hg * HC) *
                                           static_cast<int64_t>(kMlaRowDims);
            for (int c = lane; c < HC * 64; c += 32) {
              const int h = c >> 6, ch = c & 63;
              const uint4 v = __ldg(reinterpret_cast<const uint4*>(qh + h * kMlaRowDims) + ch);
              *reinterpret_cast<uint4*>(smem + L::kQn + (ch >> 3) * L::kQnPlane + sw128(h, (ch & 7) * 8)) = v;
            }
  #pragma unroll
            for (int h = 0; h < HC; ++h) {
              qa[h] = __uint_as_float(static_cast<uint32_t>(__ldg(qh + h * kMlaRowDims + kMlaLatentDims + ia)) << 16);
              qb[h] = __uint_as_float(static_cast<uint32_t>(__ldg(qh + h * kMlaRowDims + kMlaLatentDims + ib)) << 16);
            }
          }
          // lane f rotates frequency f of every head: pairs (2f, 2f + 1) interleaved, (f, f + 32) neox
          uint8_t* rp = smem + L::kRope;
  #pragma unroll
          for (int e = 0; e < NE; ++e) {
            if (!((t.fresh >> e) & 1)) continue;
            float cs = 1.0f, sn = 0.0f;
            if (t.ent_delta[e] != 0) shift_cossin(t.ent_delta[e], __ldg(P.freq + lane), cs, sn);
  #pragma unroll
            for (int h = 0; h < HC; ++h) {
              __nv_bfloat16 ah, al, bh, bl;
              split_bf16(qa[h] * cs + qb[h] * sn, ah, al);
              split_bf16(qb[h] * cs - qa[h] * sn, bh, bl);
              // per entry and half of the heads: the half's hi rows, then its lo rows
              constexpr int HH = HC / 2;
              const int rh = e * 2 * HC + (h / HH) * 2 * HH + h % HH, rl = rh + HH;
              if (NEOX) {
                *reinterpret_cast<__nv_bfloat16*>(rp + sw128(rh, ia)) = ah;
                *reinterpret_cast<__nv_bfloat16*>(rp + sw128(rh, ib)) = bh;
                *reinterpret_cast<__nv_bfloat16*>(rp + sw128(rl, ia)) = al;
                *reinterpret_cast<__nv_bfloat16*>(rp + sw128(rl, ib)) = bl;
              } else {  // (2f, 2f + 1) are adjacent: one 4-byte store per part
                *reinterpret_cast<__nv_bfloat162*>(rp + sw128(rh, ia)) = __halves2bfloat162(ah, bh);
                *reinterpret_cast<__nv_bfloat162*>(rp + sw128(rl, ia)) = __halves2bfloat162(al, bl);
              }
            }
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_ready[rt]);
        used_prev = used;
        if (t.flags & kTcEnd) break;
      }
    }
  } else if ((warp == kTcMma || warp == kTcMma2 || warp == kTcPv || warp == kTcPv2) && has_work) {
    // --------------------------------------------------- MMA issuers
    // Each issuer runs its loop on the whole warp (the waits, the operand
    // addresses) and issues the products and commits from the elected lane.
    const uint32_t ring = base_u32 + L::kRing;
    // A descriptor is affine in its start address (start / 16 sits in the
    // low bits, and no start here reaches 256 KB), so each product builds its
    // base descriptors once and steps them by constants.
    if (warp == kTcMma || warp == kTcMma2) {
      // S of tile i once its rows are in and its TMEM buffer is free (the
      // softmax of tile i - 2 has written P, so it is done reading that
      // buffer); at a key's first tile also once the query operands are
      // written.  The first issuer takes the even latent k-steps and then the
      // rope k-steps: rotated keys, once the softmax warps have rotated them,
      // four of M = 128 with A their hi and lo rows in TMEM; rotated queries, once
      // the query warp has written this tile's entries, over the rope plane
      // against every entry.  The second issuer takes the odd latent k-steps.
      // Each writes its own latent partial sums (k-step mod NP).
      const int par = warp == kTcMma ? 0 : 1;
      const uint64_t dq = sdesc(base_u32 + L::kQn, 16, 1024), dr = sdesc(base_u32 + L::kRope, 16, 1024);
      for (int i = 0;; ++i) {
        const int rt = i & 1;
        bool ok = wait_or_abort(&full[rt], (i >> 1) & 1, abort_flag, spins) &&
                  (i < 2 || wait_or_abort(&p_full[rt], ((i - 2) >> 1) & 1, abort_flag, spins));
        const int flags = ok ? tiles[rt].flags : 0;
        if (ok && (flags & kTcFirst)) ok = wait_or_abort(&q_ready[rt], (i >> 1) & 1, abort_flag, spins);
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) fail();
          break;
        }
        tc_fence_after();
        const uint64_t da = sdesc(ring + rt * kTcTileBytes, 16, 1024);
        const uint32_t d = tmem + rt * kSCols;
#pragma unroll
        for (int k2 = 0; k2 < 32 / kSI; ++k2) {
          const int ks = kSI * k2 + par;
          tc_mma_elect(d + (ks % NP) * HC, da + (((ks >> 2) * kTcPlaneBytes + (ks & 3) * 32) >> 4),
                       dq + (((ks >> 2) * L::kQnPlane + (ks & 3) * 32) >> 4), kIdS, ks >= NP);
        }
        if (par == 0) {
          if constexpr (KEYS) {
            if (!__all_sync(0xffffffffu, wait_or_abort(&rot_done[rt], (i >> 1) & 1, abort_flag, spins))) {
              if (lane == 0) fail();
              break;
            }
            tc_fence_after();
            // one M = 128 product per k-step, A from TMEM (8 columns a k-step):
            // the hi rows' partial score lands in lanes 32 w .. 32 w + 15, the
            // lo rows' in lanes 32 w + 16 .. 32 w + 31
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              tc_mma_tmem_a_elect(d + kRopeCol, tmem + kRopeACol + 8 * ks, dr + ((ks * 32) >> 4), kIdK, ks > 0);
          } else {
            if (!(flags & kTcFirst)) {
              if (!__all_sync(0xffffffffu, wait_or_abort(&q_ready[rt], (i >> 1) & 1, abort_flag, spins))) {
                if (lane == 0) fail();
                break;
              }
              tc_fence_after();
            }
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              tc_mma_elect(d + kRopeCol, da + ((8 * kTcPlaneBytes + ks * 32) >> 4), dr + ((ks * 32) >> 4), kIdR, ks > 0);
          }
        }
        tc_commit_elect(&s_full[rt]);
        if (flags & kTcEnd) break;
      }
      tc_commit_elect(&done[par]);
      mbar_wait_bounded(&done[par], 0);
    } else {
      // O^T += V^T P^T of tile i once its P is written; its metadata stays in
      // the slot until this product ends.  With two issuers each takes two of
      // the four latent M-tiles.
      const uint32_t pt = base_u32 + L::kPt;
      const int vi = warp == kTcPv ? 0 : 1;
      for (int i = 0;; ++i) {
        const int rt = i & 1;
        if (!__all_sync(0xffffffffu, wait_or_abort(&p_full[rt], (i >> 1) & 1, abort_flag, spins))) {
          if (lane == 0) fail();
          break;
        }
        const int t_ns = tiles[rt].ns, t_flags = tiles[rt].flags;
        tc_fence_after();
        // V^T as an MN-major A: 64 latent dims per 128-byte row, rows 1,024
        // bytes per 8 positions (SBO), the next 64 dims one plane on (LBO)
        const uint64_t dv = sdesc(ring + rt * kTcTileBytes, kTcPlaneBytes, 1024);
        const uint64_t dp = sdesc(pt + rt * L::kPtBytes, 16, 1024);
        const bool first = (t_flags & kTcFirst) != 0;
        // the four latent M-tiles are independent accumulators: innermost
#pragma unroll
        for (int w = 0; w < kTcStagesPerTile; ++w) {
          if (w >= t_ns) break;
          const uint64_t bd = dp + ((w * 32) >> 4);
#pragma unroll
          for (int m4 = 0; m4 < 4 / kVI; ++m4) {
            const int mt = vi * (4 / kVI) + m4;
            tc_mma_elect(tmem + kOCol + mt * kOColsPerTile, dv + ((2 * mt * kTcPlaneBytes + w * kTcStageBytes) >> 4),
                         bd, kIdPV, !(first && w == 0));
          }
        }
        tc_commit_elect(&empty[rt]);
        tc_commit_elect(&pv_done[rt]);
        if (t_flags & kTcEnd) break;
      }
      tc_commit_elect(&done[2 + vi]);
      mbar_wait_bounded(&done[2 + vi], 0);
    }
  } else if (warp < kTcSoftmaxWarps && has_work) {
    // ------------------------------------------------------------ softmax
    // Warp (w, half): stage w's 16 positions (TMEM lanes 32w .. 32w + 15 of
    // the M = 64 scores), heads [h0, h0 + HH); O^T lanes 32w .. 32w + 31.
    // The scores are read with the 16x256b shape, so every thread holds two
    // positions (q0 and q0 + 8) of NH of the warp's heads: its value r is
    // position q0 + 8 ((r >> 1) & 1) of head slot 2 (r >> 2) + (r & 1), and
    // slot j is head 8 (j >> 1) + c0 + (j & 1) of the warp's HH.
    constexpr int HH = HC / 2;
    constexpr int NG = HH / 8;  // 8-column groups of the warp's heads
    constexpr int NR = 4 * NG;  // scores a thread holds
    constexpr int NH = 2 * NG;  // heads a thread holds
    const int w = warp & 3, half = warp >> 2, h0 = half * HH;
    const int q0 = lane >> 2, c0 = 2 * (lane & 3);
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * w) << 16);
    float* wmax = reinterpret_cast<float*>(smem + L::kWmax);
    float* lred = reinterpret_cast<float*>(smem + L::kLred);
    float m_run[NH], l_part[NH];
#pragma unroll
    for (int j = 0; j < NH; ++j) {
      m_run[j] = -INFINITY;
      l_part[j] = 0.0f;
    }
    // this warp's O^T columns of M-tile mt: part 0 the product of P's hi rows, part 1 of its lo rows
    auto o_col = [&](int mt, int part) { return tl + kOCol + mt * kOColsPerTile + part * HC + h0; };
    for (int i = 0;; ++i) {
      const int rt = i & 1;
      const uint32_t ph = (i >> 1) & 1;
      // every softmax warp reaches each barrier reduction below, so a wait
      // that runs out in one warp ends all eight together
      // rotated keys: also the tile's cos / sin table (the query warp)
      const bool landed_rows =
          __all_sync(0xffffffffu, wait_or_abort(&full[rt], ph, abort_flag, spins) &&
                                      (!KEYS || wait_or_abort(&q_ready[rt], ph, abort_flag, spins)));
      if (KEYS && landed_rows) {
        // rotate stage w's rope keys by their deltas, R(delta) k_r in fp32,
        // into the rotated-key operand in TMEM: an A operand of 128 rows whose
        // lanes 32 w .. + 15 hold the stage's keys as bf16 hi parts and lanes
        // 32 w + 16 .. + 31 the lo parts, two dims per column; warp half h
        // writes dims 32 h .. 32 h + 31.  Thread t writes lane 32 w + t.  The
        // operand is free: this warp has seen the previous tile's scores, so
        // its rope product, the operand's last reader, has ended.
        const TcTile& tr0 = tiles[rt];
        if (w < tr0.ns) {
          const int n0 = tr0.n_tok[w], sp0 = tr0.split[w];
          const int j = lane & 15, row = 16 * w + j, x7 = row & 7;
          const bool live = j < n0;
          const uint8_t* rope =
              smem + L::kRing + rt * kTcTileBytes + 8 * kTcPlaneBytes + (row >> 3) * 1024 + x7 * 128;
          const float4* cs = reinterpret_cast<const float4*>(reinterpret_cast<const float2*>(smem + L::kCs) +
                                                             rt * 256 + w * 64 + (j >= sp0 ? 32 : 0));
          // Threads t and t + 16 share row t % 16: each rotates half of the
          // warp's 16 columns (thread part p = t / 16 takes columns 8 p ..
          // 8 p + 7) and hands the other thread the part that one writes.
          const int p = lane >> 4;
          uint32_t own[8], other[8];  // this thread's part, and the partner's part, of columns 8 p + m
#pragma unroll
          for (int cc2 = 0; cc2 < 2; ++cc2) {
            const int c = 2 * p + cc2;  // output dims 32 half + 8 c .. + 7: columns 4 c .. 4 c + 3
            float o[8];
            if (NEOX) {
              // frequency d pairs dims (d, d + 32): half 0 writes d, half 1 d + 32, d = 8 c .. 8 c + 7
              uint4 xa = *reinterpret_cast<const uint4*>(rope + ((c ^ x7) << 4));
              uint4 xb = *reinterpret_cast<const uint4*>(rope + (((4 + c) ^ x7) << 4));
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float4 cc = cs[4 * c + k];  // (cos, sin) of frequencies 8 c + 2 k, 8 c + 2 k + 1
                const float2 a = bf_pair(word(xa, k)), b = bf_pair(word(xb, k));
                o[2 * k] = half ? a.x * cc.y + b.x * cc.x : a.x * cc.x - b.x * cc.y;
                o[2 * k + 1] = half ? a.y * cc.w + b.y * cc.z : a.y * cc.z - b.y * cc.w;
              }
            } else {
              // dims (2 f, 2 f + 1) pair, frequency f = 16 half + 4 c + k
              uint4 x = *reinterpret_cast<const uint4*>(rope + (((4 * half + c) ^ x7) << 4));
#pragma unroll
              for (int k2 = 0; k2 < 2; ++k2) {
                const float4 cc = cs[8 * half + 2 * c + k2];  // (cos, sin) of two frequencies
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const float2 ab = bf_pair(word(x, 2 * k2 + e));
                  const float cf = e ? cc.z : cc.x, sf = e ? cc.w : cc.y;
                  o[4 * k2 + 2 * e] = ab.x * cf - ab.y * sf;
                  o[4 * k2 + 2 * e + 1] = ab.x * sf + ab.y * cf;
                }
              }
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              uint32_t hi, lo;
              split2_bf16(o[2 * k], o[2 * k + 1], hi, lo);
              own[4 * cc2 + k] = p ? lo : hi;
              other[4 * cc2 + k] = p ? hi : lo;
            }
          }
          uint32_t out[16];
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            const uint32_t got = __shfl_xor_sync(0xffffffffu, other[m], 16);  // the partner's columns, this part
            out[m] = live ? (p ? got : own[m]) : 0u;
            out[8 + m] = live ? (p ? own[m] : got) : 0u;
          }
          float outf[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) outf[k] = __uint_as_float(out[k]);
          tmem_st16(tmem + (static_cast<uint32_t>(32 * w) << 16) + kRopeACol + 16 * half, outf);
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&rot_done[rt]);
      }
      const bool got = landed_rows && __all_sync(0xffffffffu, wait_or_abort(&s_full[rt], ph, abort_flag, spins));
      // this warp's fields of the tile record (read now: the slot's record is
      // replaced once the tile's value product has finished; after a wait
      // that ran out they are not used) and its scores
      const TcTile& tr = tiles[rt];
      const int t_flags = tr.flags, t_layer = tr.layer, t_key = tr.key;
      const bool present = w < tr.ns;
      const int n_tok = present ? tr.n_tok[w] : 0;
      const int entry = present ? tr.entry[w] : 0;
      const int entry2 = present ? tr.entry2[w] : 0;
      const int split = present ? tr.split[w] : 16;
      const int sink = present ? tr.sink[w] : 0;
      float s[NR];
      bool need = false;
      if (got) {
        tc_fence_after();
        if (t_flags & kTcFirst) {
#pragma unroll
          for (int j = 0; j < NH; ++j) {
            m_run[j] = -INFINITY;
            l_part[j] = 0.0f;
          }
        }
        if constexpr (KEYS) {
          // the latent partial sums and the rope column of the warp's heads:
          // the hi rows' part in lanes 0-15 of the quadrant, the lo rows' in 16-31
          float sp[NP][NR], rr[NR], rl[NR];
          const uint32_t sc = tl + rt * kSCols + h0;
          tmem_ld16x256<NG>(sc + kRopeCol, rr);
          tmem_ld16x256<NG>(sc + kRopeCol + (16u << 16), rl);
  #pragma unroll
          for (int pp = 0; pp < NP; ++pp) tmem_ld16x256<NG>(sc + pp * HC, sp[pp]);
          tmem_wait_ld();
  #pragma unroll
          for (int r = 0; r < NR; ++r) {
            float v = sp[0][r];
  #pragma unroll
            for (int pp = 1; pp < NP; ++pp) v += sp[pp][r];
            s[r] = v + (rr[r] + rl[r]);
          }
        } else {
          // latent partial sums; the rope hi then lo columns of the slot's first
          // delta and then, when the slot holds a second one from position split
          // on, of that one (read into the same registers)
          float sp[NP][NR], rr[2 * NR], nope[NR];
          const uint32_t sc = tl + rt * kSCols + h0;
          tmem_ld16x256<2 * NG>(sc + kRopeCol + entry * 2 * HC + h0, rr);
  #pragma unroll
          for (int pp = 0; pp < NP; ++pp) tmem_ld16x256<NG>(sc + pp * HC, sp[pp]);
          tmem_wait_ld();
  #pragma unroll
          for (int r = 0; r < NR; ++r) {
            nope[r] = sp[0][r];
  #pragma unroll
            for (int pp = 1; pp < NP; ++pp) nope[r] += sp[pp][r];
            s[r] = (nope[r] + rr[r]) + rr[NR + r];
          }
          if (split < n_tok) {  // the same for the whole warp
            tmem_ld16x256<2 * NG>(sc + kRopeCol + entry2 * 2 * HC + h0, rr);
            tmem_wait_ld();
  #pragma unroll
            for (int r = 0; r < NR; ++r)
              if (q0 + 8 * ((r >> 1) & 1) >= split) s[r] = (nope[r] + rr[r]) + rr[NR + r];
          }
        }
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          const int q = q0 + 8 * ((r >> 1) & 1);
          const bool live = q < n_tok;
          const float bias = (live && ((sink >> q) & 1)) ? P.sink_log2 : 0.0f;
          s[r] = live ? s[r] * P.scale_log2 + bias : -INFINITY;
          need |= s[r] > m_run[2 * (r >> 2) + (r & 1)] + kTcLazy;
        }
      }
      // One reduction carries both rare events, a wait that ran out and a
      // score that raises a head's running max; a second one tells them apart.
      if (softmax_bar_or(!got || need)) {
        if (softmax_bar_or(!got)) {
          if (lane == 0 && !got) fail();
          break;
        }
        float* wm = wmax + (rt * 4 + w) * HC + h0;
#pragma unroll
        for (int j = 0; j < NH; ++j) {
          const int r = 4 * (j >> 1) + (j & 1);
          float v = fmaxf(s[r], s[r + 2]);
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
          if (q0 == 0) wm[8 * (j >> 1) + c0 + (j & 1)] = v;
        }
        softmax_bar_or(false);
        const volatile float* vm = wmax + rt * 4 * HC + h0;
        float alpha[NH];
        bool rescale = false;
#pragma unroll
        for (int j = 0; j < NH; ++j) {
          const int h = 8 * (j >> 1) + c0 + (j & 1);
          const float tm = fmaxf(fmaxf(vm[h], vm[HC + h]), fmaxf(vm[2 * HC + h], vm[3 * HC + h]));
          const float mn = fmaxf(m_run[j], tm);
          alpha[j] = (mn == -INFINITY) ? 1.0f : exp2f(m_run[j] - mn);
          rescale |= alpha[j] != 1.0f;
          m_run[j] = mn;
          l_part[j] *= alpha[j];
        }
        // every warp takes the same branch: the barrier below is reached by all or none
        const bool rescale_any = softmax_bar_or(rescale);
        if (!(t_flags & kTcFirst) && rescale_any) {
          // O holds this key's earlier tiles: wait for the last product into it, then scale in place
          const bool landed = wait_or_abort(&pv_done[(i - 1) & 1], ((i - 1) >> 1) & 1, abort_flag, spins);
          if (softmax_bar_or(!landed)) {
            if (lane == 0 && !landed) fail();
            break;
          }
          // every lane scales all HH heads of its O^T rows: head h's factor is
          // held by lane (h % 8) / 2 in slot 2 (h / 8) + (h & 1)
          float alpha_all[HH];
#pragma unroll
          for (int h = 0; h < HH; ++h)
            alpha_all[h] = __shfl_sync(0xffffffffu, alpha[2 * (h >> 3) + (h & 1)], (h & 7) >> 1);
          tc_fence_after();
#pragma unroll
          for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
            for (int part = 0; part < 2; ++part) {
              float o[HH];
              tmem_ld<HH>(o_col(mt, part), o);
              tmem_wait_ld();
#pragma unroll
              for (int c = 0; c < HH; ++c) o[c] *= alpha_all[c];
              tmem_st<HH>(o_col(mt, part), o);
            }
          }
          tmem_wait_st();
        }
      }
      float p[NR];
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        const int q = q0 + 8 * ((r >> 1) & 1);
        const int j = 2 * (r >> 2) + (r & 1);
        p[r] = q < n_tok ? exp2f(s[r] - m_run[j]) : 0.0f;
        l_part[j] += p[r];
      }
      if (present) {
        uint8_t* ring_t = smem + L::kRing + rt * kTcTileBytes;
        // rows past the stage's tokens may hold anything: zero their values (planes
        // 4 half .. 4 half + 3) so that P = 0 meets finite V
        const int dead = 16 - n_tok;
        for (int c = lane; c < dead * 32; c += 32) {
          const int r = 16 * w + n_tok + (c >> 5), pl = 4 * half + ((c >> 3) & 3), ch = c & 7;
          *reinterpret_cast<uint4*>(ring_t + pl * kTcPlaneBytes + (r >> 3) * 1024 + (r & 7) * 128 +
                                    ((ch ^ (r & 7)) << 4)) = make_uint4(0, 0, 0, 0);
        }
        uint8_t* ptb = smem + L::kPt + rt * L::kPtBytes;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          const int row = h0 + 8 * (r >> 2) + c0 + (r & 1), col = 16 * w + q0 + 8 * ((r >> 1) & 1);
          __nv_bfloat16 hi, lo;
          split_bf16(p[r], hi, lo);
          *reinterpret_cast<__nv_bfloat16*>(ptb + sw128(row, col)) = hi;
          *reinterpret_cast<__nv_bfloat16*>(ptb + sw128(HC + row, col)) = lo;
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[rt]);

      if (t_flags & kTcLast) {
        // the key's last tile in this CTA: write its record (O, m, l)
        const bool landed = wait_or_abort(&pv_done[rt], ph, abort_flag, spins);
        if (softmax_bar_or(!landed)) {
          if (lane == 0 && !landed) fail();
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int j = 0; j < NH; ++j) {
          float v = l_part[j];
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (q0 == 0) lred[w * HC + h0 + 8 * (j >> 1) + c0 + (j & 1)] = v;
        }
        softmax_bar_or(false);
        const AttnKey kk = P.keys[static_cast<int64_t>(t_layer) * P.n_keys + t_key];
        const int blk_floats = attn_block_floats(HC, kMlaLatentDims);
        float* blk =
            P.records + static_cast<int64_t>(kk.rec_base + (static_cast<int>(blockIdx.x) - kk.first_cta)) * blk_floats;
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
          float o[HH], ol[HH];
          tmem_ld<HH>(o_col(mt, 0), o);
          tmem_ld<HH>(o_col(mt, 1), ol);
          tmem_wait_ld();
          const int d = mt * 128 + 32 * w + lane;
#pragma unroll
          for (int h = 0; h < HH; ++h) blk[(h0 + h) * kMlaLatentDims + d] = o[h] + ol[h];
        }
        if (w == 0) {
          // lane h < HH writes head h0 + h: its running max from the lane that holds it
          float mv = 0.0f;
#pragma unroll
          for (int h = 0; h < HH; ++h) {
            const float v = __shfl_sync(0xffffffffu, m_run[2 * (h >> 3) + (h & 1)], (h & 7) >> 1);
            if (lane == h) mv = v;
          }
          if (lane < HH) {
            const volatile float* vl = lred + h0;
            blk[HC * kMlaLatentDims + h0 + lane] = mv;
            blk[HC * kMlaLatentDims + HC + h0 + lane] =
                (vl[lane] + vl[HC + lane]) + (vl[2 * HC + lane] + vl[3 * HC + lane]);
          }
        }
        tc_fence_before();
      }
      if (t_flags & kTcEnd) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kTcMma) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols) : "memory");
  }
}

template <int PAIRING, int HC>
cudaError_t launch_tc(const AttnParams& p, const TcMaps& maps, int grid, size_t smem, cudaStream_t s) {
  auto kern = k_attend_mla_tc<PAIRING, HC>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<grid, tc_threads(HC), smem, s>>>(p, maps);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_attend_merge_mla(p, HC, s);
}

}  // namespace

bool attend_mla_tc_config(int hc, size_t* smem_bytes) {
  if (hc == 16) {
    *smem_bytes = TcLayout<16>::kAlloc;
  } else if (hc == 32) {
    *smem_bytes = TcLayout<32>::kAlloc;
  } else {
    return false;
  }
  return *smem_bytes <= 227 * 1024;
}

cudaError_t launch_attend_mla_tc(const AttnParams& p, const TcMaps& maps, int pairing, int hc, int grid,
                                 size_t smem_bytes, cudaStream_t s) {
  if (p.n_units <= 0 || grid <= 0) return cudaSuccess;
  if (pairing == kNeox) {
    if (hc == 16) return launch_tc<kNeox, 16>(p, maps, grid, smem_bytes, s);
    if (hc == 32) return launch_tc<kNeox, 32>(p, maps, grid, smem_bytes, s);
  } else {
    if (hc == 16) return launch_tc<kInterleaved, 16>(p, maps, grid, smem_bytes, s);
    if (hc == 32) return launch_tc<kInterleaved, 32>(p, maps, grid, smem_bytes, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pic
