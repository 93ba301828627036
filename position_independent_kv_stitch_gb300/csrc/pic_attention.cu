// Decode attention over a stitched context, with the delta-rotation fused into
// the key path (GQA, sm_103a).
//
// Irminsul: MLA-Native Position-Independent Caching for Agentic LLM Serving,
// 2.2 "delta-Rotation Rule" and 4. Results: the rotation R(delta) k can be
// applied on the HBM -> on-chip path of attention instead of writing a rotated
// copy, so no extra HBM traffic is spent.  Every context position is read from
// where it lives -- a chunk token from its source rows (pool, or the blocks of
// a block-resident chunk), an inline token from the request's paged cache --
// and one decode step of attention runs over them:
//   scores = scale * q . R(delta) k + bias,  p = softmax,  out = sum p v
// (bias: LegoLink's pseudo-sink suppression, EPIC Guide: Position-Independent
// Caching for LLM Serving, LegoLink "1. Identifying and Neutralizing
// Pseudo-Sinks" -- the first k tokens of every chunk not at position 0 get a
// negative logit offset).  q . R(delta) k = (R(-delta) q) . k because R is
// orthogonal, so the query is rotated once per delta and keys are used as
// stored.
//
// Structure (one pass over K and V: HBM-bound):
//   * Persistent CTAs, each owning a contiguous range of (layer, stage)
//     units; a stage is <= 16 consecutive positions of one request that share
//     one delta.  Warp HB (the producer) copies every position's K and V rows
//     (all heads of the group) into a ring of shared-memory slots with
//     cp.async.bulk, one row per copy into a row pitch padded by 16 bytes (so
//     the eight rows an ldmatrix reads fall in distinct banks), tracked by
//     mbarriers; its descriptor loads run two stages ahead.
//   * Warp h < HB (a consumer) owns KV head h and keeps an online softmax per
//     query head across the CTA's stages of one key (request x head group),
//     flushed to a record when the range leaves the key; a second kernel
//     merges the records of each key (flash-decoding).
//   * The two products of a stage are small matrix products, run on the
//     tensor cores with mma.sync m16n8k16 (bf16 in, fp32 accumulate):
//     S = Q K^T (rows: query heads, 16 positions) and O += P V.  Tensor cores
//     are used here to cut the instruction count per byte (a 16-position
//     stage costs ~150 instructions per warp instead of ~1,000 FMA-path
//     ones), not for their FLOPs.  Q and P are fp32 values; each is split
//     into bf16 hi + lo parts placed in rows g and g + 8 of the same A tile,
//     so one product carries both and the sum of the two rows keeps about
//     16 significant bits (K and V are bf16 already, products accumulate in
//     fp32).
// Every mbarrier wait is bounded: on timeout the warp raises PIC_DEV_TIMEOUT,
// the producer waits (bounded) for the copies it issued, and the CTA exits.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <cstdint>

#include "pic_device.cuh"
#include "pic_internal.h"

namespace pic {
namespace {

using namespace dev;

constexpr unsigned kFullMask = 0xffffffffu;
constexpr size_t kSmemBudget = 227 * 1024;  // dynamic shared memory per CTA on sm_103a
constexpr int kMetaFirst = 1;               // stage opens its key in this CTA
constexpr int kMetaLast = 2;                // stage closes its key in this CTA

struct StageMeta {  // written by the producer before the stage's arrive
  int32_t layer;    // local layer
  int32_t key;
  int32_t delta;
  int32_t n_tok;
  uint32_t sink_mask;
  int32_t flags;
  int32_t pad[2];
};
static_assert(sizeof(StageMeta) == 32, "StageMeta layout");

constexpr int ST = kAttnStageTokens;

// The producer's descriptor rings: stage descriptors of units u .. u + 4
// and token rows of units u .. u + 2, filled by cp.async so that the loads
// stay in flight several stages ahead without holding registers.
struct ProdState {
  AttnStage desc[8];      // unit v at [v & 7]
  AttnTok tok[4][32];     // unit v at [v & 3], one row per lane
};
static_assert(sizeof(ProdState) == 1152, "ProdState layout");
constexpr int kDescAhead = 4;  // descriptors are requested this many units ahead

// Shared memory: barriers | metas | producer rings | per consumer warp (raw
// q bf16 [G][D], rotated q fp32 [G][D]) | ring of stages (ST K rows, then ST
// V rows).
struct SmemLayout {
  size_t meta, prod, warp, warp_bytes, qrot, ring, row_pitch, stage_bytes, total;
};
__host__ __device__ inline SmemLayout smem_layout(int D, int G, int HB, int ring) {
  SmemLayout L{};
  L.meta = 4 * kAttnMaxStages * sizeof(uint64_t);  // full and empty barriers of the K and V halves
  L.prod = L.meta + kAttnMaxStages * sizeof(StageMeta);
  L.warp = (L.prod + 2 * sizeof(ProdState) + 127) / 128 * 128;  // one descriptor ring per producer
  L.qrot = static_cast<size_t>(G) * D * 2;
  L.warp_bytes = (L.qrot + static_cast<size_t>(G) * D * 4 + 127) / 128 * 128;
  L.ring = (L.warp + HB * L.warp_bytes + 127) / 128 * 128;
  L.row_pitch = static_cast<size_t>(HB) * D * 2 + 16;
  L.stage_bytes = 2 * ST * L.row_pitch;
  L.total = L.ring + ring * L.stage_bytes;
  return L;
}

// ------------------------------------------------------------- tensor cores

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// c += A B for one 16x8x16 tile: A row-major bf16 (4 regs), B column-major bf16 (2 regs)
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// (x, y) as bf16 pairs: hi = RN(x, y), lo = RN of what hi left out
__device__ __forceinline__ void split_bf16x2(float x, float y, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x - hf.x, y - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

__device__ __forceinline__ void cp_async16(void* sdst, const void* gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(smem_u32(sdst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async8(void* sdst, const void* gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(sdst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// unit v's stage descriptor (stage j of its layer; lane 0) and, once that
// is in shared memory, its token rows (one per lane)
__device__ __forceinline__ void fetch_desc(const AttnParams& P, ProdState* ps, int64_t v, int j, int lane) {
  if (lane == 0) cp_async16(&ps->desc[v & 7], P.stages + j);
}
__device__ __forceinline__ void fetch_toks(const AttnParams& P, ProdState* ps, int64_t v, int lane) {
  const AttnStage& d = ps->desc[v & 7];
  if (lane < d.n_tok) cp_async8(&ps->tok[v & 3][lane], P.toks + d.tok_off + lane);
}
// (stage, layer) of the unit k units after (j, layer)
__device__ __forceinline__ int advance_stage(int j, int k, int n_stages) {
  j += k;
  while (j >= n_stages) j -= n_stages;
  return j;
}

// grid: persistent CTAs; block: 32 * (HB + 2) threads (HB consumers, a K and a V producer).
template <int PAIRING, int D, int G>
__global__ void __launch_bounds__(32 * (kAttnMaxHeads + 2), 1) k_attend(const AttnParams P) {
  // the merge that reads this kernel's records may be scheduled from now on
  // (it waits for this grid's completion before it reads anything)
  asm volatile("griddepcontrol.launch_dependents;");
  constexpr bool NEOX = (PAIRING == kNeox);
  constexpr int HALF = D / 2;
  constexpr int KS = D / 16;   // k-steps of Q K^T
  constexpr int NT = D / 8;    // n-tiles of P V
  constexpr int BLK = attn_block_floats(G, D);

  extern __shared__ __align__(128) uint8_t smem[];
  const int HB = P.heads_per_cta;
  const int NS = P.ring;
  const SmemLayout L = smem_layout(D, G, HB, NS);
  // Each ring slot holds a stage's K rows then its V rows; the halves have
  // their own barriers, so a slot's K half is refilled as soon as every
  // consumer has its scores, while its V half is still being read.
  uint64_t* full_k = reinterpret_cast<uint64_t*>(smem);
  uint64_t* full_v = full_k + kAttnMaxStages;
  uint64_t* empty_k = full_v + kAttnMaxStages;
  uint64_t* empty_v = empty_k + kAttnMaxStages;
  StageMeta* meta = reinterpret_cast<StageMeta*>(smem + L.meta);
  uint8_t* ring = smem + L.ring;
  const size_t srow = static_cast<size_t>(HB) * D * 2;  // bytes of one position's rows
  const uint32_t pitch = static_cast<uint32_t>(L.row_pitch);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t U = P.n_units, N = gridDim.x;
  const int64_t u_begin = U * blockIdx.x / N, u_end = U * (blockIdx.x + 1) / N;

  // Rows past a stage's positions keep what an earlier stage left there; the
  // ring starts zeroed so that they always hold finite values (their
  // probabilities are 0, and 0 * v must stay 0 in the tensor-core sums).
  for (size_t i = threadIdx.x; i < static_cast<size_t>(NS) * L.stage_bytes / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(ring)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full_k[s], 1);
      mbar_init(&full_v[s], 1);
      mbar_init(&empty_k[s], HB);
      mbar_init(&empty_v[s], HB);
    }
    fence_mbar_init();
  }
  fence_proxy_async_smem();  // the zeros are ordered before the bulk copies into the ring
  __syncthreads();

  if (warp >= HB) {
    // ----------------------------------------------------------- producers
    // Warp HB fills the K halves of the slots (and writes each stage's
    // meta), warp HB + 1 the V halves; each walks every unit of the CTA.
    // Descriptors run ahead: each iteration requests unit u + 4's stage and
    // unit u + 2's token rows (whose stage arrived two iterations ago), and
    // waits only for the requests of two iterations ago.
    const bool vq = warp == HB + 1;
    uint64_t* fb = vq ? full_v : full_k;
    uint64_t* eb = vq ? empty_v : empty_k;
    ProdState* ps = reinterpret_cast<ProdState*>(smem + L.prod) + (vq ? 1 : 0);
    const int n_st = P.n_stages;
    int j = static_cast<int>(u_begin % n_st);       // stage of unit u within its layer
    int layer = static_cast<int>(u_begin / n_st);
    for (int k = 0; k < kDescAhead && u_begin + k < u_end; ++k)
      fetch_desc(P, ps, u_begin + k, advance_stage(j, k, n_st), lane);
    cp_async_commit();
    cp_async_wait<0>();
    __syncwarp();
    for (int k = 0; k < 2 && u_begin + k < u_end; ++k) fetch_toks(P, ps, u_begin + k, lane);
    cp_async_commit();
    cp_async_wait<0>();
    // per-layer bases of the four source tensors
    int base_layer = -1;
    const uint8_t *kp = nullptr, *vp = nullptr, *kc = nullptr, *vc = nullptr;
    int prev_layer = -1, prev_key = -1;
    // Unit u is prepared (its meta, this lane's source rows) before its slot
    // frees up, so a released slot is refilled with a handful of
    // instructions.  The unit's rows arrived two iterations ago, the stage
    // after it three.
    StageMeta pm{};
    int pn = 0;
    const uint8_t* pks = nullptr;
    const uint8_t* pvs = nullptr;
    auto prepare = [&](int64_t u) {
      cp_async_wait<1>();
      __syncwarp();
      const AttnStage cur = ps->desc[u & 7];
      const AttnStage nx = ps->desc[(u + 1) & 7];
      pm.layer = layer;
      pm.key = cur.key;
      pm.delta = cur.delta;
      pm.n_tok = cur.n_tok;
      pm.sink_mask = cur.sink_mask;
      pm.flags = 0;
      if (layer != prev_layer || cur.key != prev_key) pm.flags |= kMetaFirst;
      if (u + 1 == u_end || j + 1 == n_st || nx.key != cur.key) pm.flags |= kMetaLast;
      prev_layer = layer;
      prev_key = cur.key;
      if (layer != base_layer) {
        const int64_t l_abs = P.layer_begin + layer;
        kp = P.k_pool + l_abs * P.pool_layer_stride;
        vp = P.v_pool + l_abs * P.pool_layer_stride;
        kc = P.k_cache + l_abs * P.cache_layer_stride;
        vc = P.v_cache + l_abs * P.cache_layer_stride;
        base_layer = layer;
      }
      pn = cur.n_tok;
      if (lane < pn) {
        const AttnTok tok = ps->tok[u & 3][lane];
        const bool from_cache = (tok.flags & kAttnFromCache) != 0;
        const int64_t off = static_cast<int64_t>(tok.row) * P.row_bytes +
                            static_cast<int64_t>(cur.key % P.head_groups) * srow;
        pks = (from_cache ? kc : kp) + off;
        pvs = (from_cache ? vc : vp) + off;
      }
    };
    prepare(u_begin);
    int64_t it = 0;
    bool failed = false;
    int slot = 0;
    uint32_t round = 0;   // how many times the ring has wrapped
    for (int64_t u = u_begin; u < u_end; ++u, ++it) {
      // every lane polls; the warp leaves together if any lane gave up
      if (round > 0 && !__all_sync(kFullMask, mbar_wait_bounded(&eb[slot], (round - 1) & 1u))) {
        failed = true;
        break;
      }
      if (!vq && lane == 0) meta[slot] = pm;
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&fb[slot], static_cast<uint32_t>(pn * srow));
      __syncwarp();
      if (lane < pn) {
        // one copy per position, into the padded row pitch of this half
        uint8_t* d = ring + slot * L.stage_bytes + (vq ? ST * L.row_pitch : 0) + lane * L.row_pitch;
        bulk_load(d, vq ? pvs : pks, static_cast<uint32_t>(srow), &fb[slot]);
      }
      // ring entries being refilled held units u - 4 (stage) and u - 2 (rows): both done
      if (u + kDescAhead < u_end) fetch_desc(P, ps, u + kDescAhead, advance_stage(j, kDescAhead, n_st), lane);
      if (u + 2 < u_end) fetch_toks(P, ps, u + 2, lane);
      cp_async_commit();
      if (j + 1 == n_st) {
        j = 0;
        ++layer;
      } else {
        ++j;
      }
      if (++slot == NS) {
        slot = 0;
        ++round;
      }
      if (u + 1 < u_end) prepare(u + 1);
    }
    if (failed) {
      if (lane == 0) atomicOr(P.status, kDevTimeout);
      // wait (bounded) for every copy this warp issued before leaving
      const int64_t issued = it;
      for (int64_t k = (issued > NS ? issued - NS : 0); k < issued; ++k)
        mbar_wait_bounded(&fb[k % NS], static_cast<uint32_t>((k / NS) & 1));
    }
    cp_async_wait<0>();  // no descriptor copy may outlive the CTA
    return;
  }

  // -------------------------------------------------------------- consumer
  const int h = warp;              // KV head within the group
  const int g = lane >> 2;         // query-head row of the fragments (rows g and g + 8)
  const int tq = lane & 3;         // column pair within the fragments
  const bool row_live = g < G;
  uint8_t* wbuf = smem + L.warp + h * L.warp_bytes;
  uint16_t* q_raw = reinterpret_cast<uint16_t*>(wbuf);
  float* q_rot = reinterpret_cast<float*>(wbuf + L.qrot);
  // ldmatrix row addresses of this lane: K (non-transposed) and V (transposed)
  const int mi = lane >> 3, ri = lane & 7;
  const uint32_t k_lane = static_cast<uint32_t>((ri + ((mi & 2) ? 8 : 0)) * pitch + h * D * 2 + (mi & 1) * 16);
  const uint32_t v_lane = static_cast<uint32_t>((ri + ((mi & 1) ? 8 : 0)) * pitch + h * D * 2 + (mi & 2) * 8);
  const uint32_t ring_u32 = smem_u32(ring);

  float o[NT][4];
  uint32_t qa[KS][4];
  float m_run = -FLT_MAX, l_part = 0.0f;
  int cur_delta = 0;
  bool have_rot = false;
  int slot = 0;
  uint32_t round = 0;
  for (int64_t u = u_begin; u < u_end; ++u) {
    if (!__all_sync(kFullMask, mbar_wait_bounded(&full_k[slot], round & 1u))) {
      if (lane == 0) atomicOr(P.status, kDevTimeout);
      return;
    }
    const StageMeta m = meta[slot];
    if (m.flags & kMetaFirst) {
      m_run = -FLT_MAX;
      l_part = 0.0f;
#pragma unroll
      for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.0f;
      // this head's G query rows, bf16, contiguous
      const int hg = m.key % P.head_groups;
      const int req = m.key / P.head_groups;
      const uint4* qsrc = reinterpret_cast<const uint4*>(
          P.q + ((static_cast<int64_t>(m.layer) * P.n_req + req) * P.num_q_heads + (hg * HB + h) * G) * D);
      for (int i = lane; i < G * D / 8; i += 32) reinterpret_cast<uint4*>(q_raw)[i] = __ldg(qsrc + i);
      have_rot = false;
      __syncwarp();
    }
    if (!have_rot || m.delta != cur_delta) {
      // R(-delta) q: each lane takes frequencies f = lane, lane + 32, ...
      for (int f = lane; f < HALF; f += 32) {
        float cs = 1.0f, sn = 0.0f;
        if (m.delta != 0) shift_cossin(m.delta, __ldg(P.freq + f), cs, sn);
        const int a = NEOX ? f : 2 * f, b = NEOX ? f + HALF : 2 * f + 1;
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          const float qa_ = __uint_as_float(static_cast<uint32_t>(q_raw[gg * D + a]) << 16);
          const float qb_ = __uint_as_float(static_cast<uint32_t>(q_raw[gg * D + b]) << 16);
          q_rot[gg * D + a] = qa_ * cs + qb_ * sn;
          q_rot[gg * D + b] = qb_ * cs - qa_ * sn;
        }
      }
      __syncwarp();
      // A fragments of [q_hi; q_lo]: row g holds hi, row g + 8 lo
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        if (row_live) {
          const float2 x = *reinterpret_cast<const float2*>(q_rot + g * D + 16 * kk + 2 * tq);
          const float2 y = *reinterpret_cast<const float2*>(q_rot + g * D + 16 * kk + 8 + 2 * tq);
          split_bf16x2(x.x, x.y, qa[kk][0], qa[kk][1]);
          split_bf16x2(y.x, y.y, qa[kk][2], qa[kk][3]);
        } else {
          qa[kk][0] = qa[kk][1] = qa[kk][2] = qa[kk][3] = 0u;
        }
      }
      __syncwarp();
      cur_delta = m.delta;
      have_rot = true;
    }

    const uint32_t kbase = ring_u32 + static_cast<uint32_t>(slot * L.stage_bytes);
    const uint32_t vbase = kbase + ST * pitch;
    // ---- S = [q_hi; q_lo] K^T over the stage's 16 positions (two n-tiles)
    // (even and odd k-steps accumulate separately: two short dependency chains)
    float s0[2][4] = {}, s1[2][4] = {};
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kbase + k_lane + kk * 32, b0, b1, b2, b3);
      mma_bf16(s0[kk & 1], qa[kk], b0, b1);
      mma_bf16(s1[kk & 1], qa[kk], b2, b3);
    }
    // the K half is free for the next stage as soon as every consumer has its scores
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_k[slot]);
    // this lane's scores: head g, positions 2tq, 2tq + 1, 8 + 2tq, 9 + 2tq
    float sc[4] = {(s0[0][0] + s0[0][2]) + (s0[1][0] + s0[1][2]), (s0[0][1] + s0[0][3]) + (s0[1][1] + s0[1][3]),
                   (s1[0][0] + s1[0][2]) + (s1[1][0] + s1[1][2]), (s1[0][1] + s1[0][3]) + (s1[1][1] + s1[1][3])};
    float mt = -FLT_MAX;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = (i < 2 ? 0 : 8) + 2 * tq + (i & 1);
      const bool live = row_live && t < m.n_tok;
      const float bias = ((m.sink_mask >> t) & 1u) ? P.sink_log2 : 0.0f;
      sc[i] = live ? sc[i] * P.scale_log2 + bias : -FLT_MAX;
      mt = fmaxf(mt, sc[i]);
    }
    mt = fmaxf(mt, __shfl_xor_sync(kFullMask, mt, 1));
    mt = fmaxf(mt, __shfl_xor_sync(kFullMask, mt, 2));
    const float m_new = fmaxf(m_run, mt);
    const float alpha = exp2f(m_run - m_new);
    float p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = sc[i] > -FLT_MAX ? exp2f(sc[i] - m_new) : 0.0f;
    l_part = l_part * alpha + ((p[0] + p[1]) + (p[2] + p[3]));
    m_run = m_new;
    // A fragment of [p_hi; p_lo] over the 16 positions
    uint32_t pa[4];
    split_bf16x2(p[0], p[1], pa[0], pa[1]);
    split_bf16x2(p[2], p[3], pa[2], pa[3]);

    if (!__all_sync(kFullMask, mbar_wait_bounded(&full_v[slot], round & 1u))) {
      if (lane == 0) atomicOr(P.status, kDevTimeout);
      return;
    }
    // ---- O = alpha O + [p_hi; p_lo] V (alpha is 1 once the running max settles)
    if (!__all_sync(kFullMask, alpha == 1.0f)) {
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        o[j][0] *= alpha;
        o[j][1] *= alpha;
        o[j][2] *= alpha;
        o[j][3] *= alpha;
      }
    }
#pragma unroll
    for (int j = 0; j < NT; j += 2) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(vbase + v_lane + j * 16, b0, b1, b2, b3);
      mma_bf16(o[j], pa, b0, b1);
      mma_bf16(o[j + 1], pa, b2, b3);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_v[slot]);
    if (++slot == NS) {
      slot = 0;
      ++round;
    }

    if (m.flags & kMetaLast) {
      // the four lanes of a query head hold its sums over different positions
      float l_tot = l_part;
      l_tot += __shfl_xor_sync(kFullMask, l_tot, 1);
      l_tot += __shfl_xor_sync(kFullMask, l_tot, 2);
      const AttnKey kk = P.keys[static_cast<int64_t>(m.layer) * P.n_keys + m.key];
      float* blk = P.records + (static_cast<int64_t>(kk.rec_base + (blockIdx.x - kk.first_cta)) * HB + h) * BLK;
      if (row_live) {
#pragma unroll
        for (int j = 0; j < NT; ++j)
          *reinterpret_cast<float2*>(blk + g * D + 8 * j + 2 * tq) = make_float2(o[j][0] + o[j][2], o[j][1] + o[j][3]);
        if (tq == 0) {
          blk[G * D + g] = m_run;
          blk[G * D + G + g] = l_tot;
        }
      }
    }
  }
}

// One thread block per (request, query head, layer): merges the records of
// its key (flash-decoding).  Statistics are in log2 units.  The records'
// maxima and sums are reduced across the block's threads; each record's
// weight exp2(m_k - M) is kept in shared memory for the weighted sum over
// the output dims.
constexpr int kMergeThreads = 128;

__device__ __forceinline__ float block_reduce(float v, bool is_max, float* red) {
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(kFullMask, v, o);
    v = is_max ? fmaxf(v, w) : v + w;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // red is free
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = red[0];
  for (int w = 1; w < kMergeThreads / 32; ++w) v = is_max ? fmaxf(v, red[w]) : v + red[w];
  return v;
}

template <int D>
__global__ void __launch_bounds__(kMergeThreads) k_attend_merge(const AttnParams P, int group) {
  __shared__ float s_e[kAttnMaxCtas];  // exp2(m_k - M) per record
  __shared__ float s_red[kMergeThreads / 32];
  // launched as a programmatic dependent of the attention kernel: wait until
  // that grid has completed and its records are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int r = blockIdx.x, gq = blockIdx.y, lz = blockIdx.z;
  const int hk = gq / group, g = gq % group;
  const int HB = P.heads_per_cta;
  const int hg = hk / HB, h = hk % HB;
  const int64_t lk = static_cast<int64_t>(lz) * P.n_keys + static_cast<int64_t>(r) * P.head_groups + hg;
  const int rec0 = P.keys[lk].rec_base, rec1 = P.keys[lk + 1].rec_base;
  const int BLK = attn_block_floats(group, D);
  const float* base = P.records + static_cast<int64_t>(h) * BLK;
  const int64_t stride = static_cast<int64_t>(HB) * BLK;
  float mloc = -FLT_MAX;
  for (int k = rec0 + threadIdx.x; k < rec1; k += kMergeThreads) mloc = fmaxf(mloc, base[k * stride + group * D + g]);
  const float M = block_reduce(mloc, true, s_red);
  float tloc = 0.0f;
  for (int k = rec0 + threadIdx.x; k < rec1; k += kMergeThreads) {
    const float e = exp2f(base[k * stride + group * D + g] - M);
    s_e[k - rec0] = e;
    tloc += e * base[k * stride + group * D + group + g];
  }
  const float tot = block_reduce(tloc, false, s_red);  // its barriers also publish s_e
  const float inv = 1.0f / tot;
  for (int d = threadIdx.x; d < D; d += kMergeThreads) {
    float acc = 0.0f;
    for (int k = rec0; k < rec1; ++k) acc += s_e[k - rec0] * base[k * stride + g * D + d];
    P.out[((static_cast<int64_t>(lz) * P.n_req + r) * P.num_q_heads + gq) * D + d] = acc * inv;
  }
  if (threadIdx.x == 0 && P.lse != nullptr)
    P.lse[(static_cast<int64_t>(lz) * P.n_req + r) * P.num_q_heads + gq] = (M + log2f(tot)) * 0.69314718055994531f;
}

// The merge after an attention kernel, as its programmatic dependent: the
// merge's CTAs may be scheduled while the attention kernel's last CTAs still
// run (each attention CTA allows it once it has started), so the launch
// latency hides behind the attention kernel's tail; the merge's first
// instruction waits for that kernel's completion and memory.
template <int D>
cudaError_t launch_merge(const AttnParams& p, int group, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_req, p.num_q_heads, p.n_layers);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_attend_merge<D>, p, group);
}

template <int PAIRING, int D, int G>
cudaError_t launch_g(const AttnParams& p, int grid, size_t smem, cudaStream_t s) {
  auto kern = k_attend<PAIRING, D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<grid, 32 * (p.heads_per_cta + 2), smem, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_merge<D>(p, G, s);
}

template <int PAIRING, int D, int G>
int occupancy_g(int heads_per_cta, size_t smem) {
  auto kern = k_attend<PAIRING, D, G>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 32 * (heads_per_cta + 2), smem) != cudaSuccess) return 0;
  return n;
}

// Returns FN<pairing, head_dim, group>(args...) for the runtime triple, FAIL
// when it has no instance.
#define PIC_ATTN_DISPATCH(FN, FAIL, ...)                              \
  do {                                                                \
    if (pairing == kNeox) {                                           \
      if (head_dim == 64) {                                           \
        if (group == 1) return FN<kNeox, 64, 1>(__VA_ARGS__);         \
        if (group == 2) return FN<kNeox, 64, 2>(__VA_ARGS__);         \
        if (group == 4) return FN<kNeox, 64, 4>(__VA_ARGS__);         \
        if (group == 8) return FN<kNeox, 64, 8>(__VA_ARGS__);         \
      } else if (head_dim == 128) {                                   \
        if (group == 1) return FN<kNeox, 128, 1>(__VA_ARGS__);        \
        if (group == 2) return FN<kNeox, 128, 2>(__VA_ARGS__);        \
        if (group == 4) return FN<kNeox, 128, 4>(__VA_ARGS__);        \
        if (group == 8) return FN<kNeox, 128, 8>(__VA_ARGS__);        \
      }                                                               \
    } else {                                                          \
      if (head_dim == 64) {                                           \
        if (group == 1) return FN<kInterleaved, 64, 1>(__VA_ARGS__);  \
        if (group == 2) return FN<kInterleaved, 64, 2>(__VA_ARGS__);  \
        if (group == 4) return FN<kInterleaved, 64, 4>(__VA_ARGS__);  \
        if (group == 8) return FN<kInterleaved, 64, 8>(__VA_ARGS__);  \
      } else if (head_dim == 128) {                                   \
        if (group == 1) return FN<kInterleaved, 128, 1>(__VA_ARGS__); \
        if (group == 2) return FN<kInterleaved, 128, 2>(__VA_ARGS__); \
        if (group == 4) return FN<kInterleaved, 128, 4>(__VA_ARGS__); \
        if (group == 8) return FN<kInterleaved, 128, 8>(__VA_ARGS__); \
      }                                                               \
    }                                                                 \
    return FAIL;                                                      \
  } while (0)


// ------------------------------------------------------------------ MLA

// Decode attention for MLA models (Irminsul 2.1-2.2): every query head
// attends to the same latent rows, row_t = [cKV_t (512) | k_r,t (64)], with
// the query already absorbed into the latent space, q_h = [q_nope,h (512) |
// q_rope,h (64)]:
//   s_h,t = scale * (q_nope,h . cKV_t + q_rope,h . R(delta) k_r,t) + bias_t
//         = scale * [q_nope,h | R(-delta) q_rope,h] . row_t + bias_t,
//   out_h = sum_t softmax(s_h)_t cKV_t     (512 dims, before the up-projection).
// Only the 64-d rope part of the query is rotated (once per delta); the
// latent is used as stored, as Irminsul's delta-rotation requires.
//
// One latent row per position: the producer warp copies each position's
// 1,152-byte row once (it serves as key and, its first 512 dims, as value).
// The score tile of 16 heads x 16 positions and the 16 x 512 output are
// shared by four consumer warps: warp quarter q computes the partial scores
// over k-steps [9q, 9q + 9) of the 36 and owns output dims [128q, 128q + 128).
// Partial scores meet in shared memory (two buffers, by stage parity) behind
// an mbarrier per head group, waited on with a bound like every other wait;
// each warp then runs the same softmax on the summed scores.
constexpr int kMlaLatent = 512;
constexpr int kMlaRopeDims = 64;
constexpr int kMlaRow = kMlaLatent + kMlaRopeDims;  // 576 dims per latent row
constexpr int kMlaQKS = kMlaRow / 16 / 4;           // k-steps of Q K^T per warp quarter (9)
constexpr int kMlaRopeKS0 = kMlaLatent / 16;        // first rope k-step (32)
constexpr int kMlaQNT = kMlaLatent / 8 / 4;         // n-tiles of P V per warp quarter (16)
constexpr int kMlaHeadsPerGroup = 16;
constexpr int kMlaMaxStages = 12;                   // ring depth bound (smaller stages than GQA's)
constexpr size_t kMlaSmemHalf = 112 * 1024;         // shared memory per CTA when two share an SM

constexpr int kMlaQPitch = kMlaQKS * 16 * 2 + 16;  // bytes per head row of a warp's q slice (304)
constexpr int kMlaRopePitch = kMlaRopeDims * 2 + 16; // bytes per head row of a rotated rope tile (144)

struct MlaLayout {
  size_t meta, gbar, prod, sbuf, qs, rope, ring, row_pitch, stage_bytes, total;
};
__host__ __device__ inline MlaLayout mla_layout(int ng, int ring) {
  MlaLayout L{};
  L.meta = 2 * kMlaMaxStages * sizeof(uint64_t);
  L.gbar = L.meta + kMlaMaxStages * sizeof(StageMeta);
  L.prod = (L.gbar + 8 * sizeof(uint64_t) + 127) / 128 * 128;
  L.sbuf = (L.prod + sizeof(ProdState) + 127) / 128 * 128;
  // per head group: 2 stage parities x 4 quarters x 16 heads x 16 positions
  L.qs = (L.sbuf + static_cast<size_t>(ng) * 2 * 4 * 256 * sizeof(float) + 127) / 128 * 128;
  // per consumer warp: its q slice, 16 heads x 144 dims (bf16)
  L.rope = L.qs + static_cast<size_t>(ng) * 4 * 16 * kMlaQPitch;
  // per head group: the rotated rope part of q as bf16 hi and lo tiles, 16 heads x 64 dims each
  L.ring = (L.rope + static_cast<size_t>(ng) * 2 * 16 * kMlaRopePitch + 127) / 128 * 128;
  L.row_pitch = kMlaRow * 2 + 16;  // +16 bytes: the 8 rows an ldmatrix reads fall in distinct banks
  L.stage_bytes = ST * L.row_pitch;
  L.total = L.ring + ring * L.stage_bytes;
  return L;
}

// grid: persistent CTAs; block: 32 * (4 NG + 1) threads (NG groups of 16 heads).
template <int PAIRING, int NG>
__global__ void __launch_bounds__(32 * (4 * NG + 1), NG == 1 ? 2 : 1) k_attend_mla(const AttnParams P) {
  // the merge that reads this kernel's records may be scheduled from now on
  // (it waits for this grid's completion before it reads anything)
  asm volatile("griddepcontrol.launch_dependents;");
  constexpr bool NEOX = (PAIRING == kNeox);
  constexpr int NCW = 4 * NG;                          // consumer warps
  constexpr int HC = kMlaHeadsPerGroup * NG;           // query heads per CTA (and per record)
  const int BLK = attn_block_floats(HC, kMlaLatent);   // floats of one record

  extern __shared__ __align__(128) uint8_t smem[];
  const int NS = P.ring;
  const MlaLayout L = mla_layout(NG, NS);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMlaMaxStages;
  StageMeta* meta = reinterpret_cast<StageMeta*>(smem + L.meta);
  uint64_t* gbar = reinterpret_cast<uint64_t*>(smem + L.gbar);
  float* sbuf = reinterpret_cast<float*>(smem + L.sbuf);
  uint8_t* ring = smem + L.ring;
  const uint32_t pitch = static_cast<uint32_t>(L.row_pitch);
  const uint32_t rowb = static_cast<uint32_t>(P.row_bytes);  // 1,152

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t U = P.n_units, N = gridDim.x;
  const int64_t u_begin = U * blockIdx.x / N, u_end = U * (blockIdx.x + 1) / N;

  for (size_t i = threadIdx.x; i < static_cast<size_t>(NS) * L.stage_bytes / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(ring)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NCW);
    }
    for (int gi = 0; gi < NG; ++gi) mbar_init(&gbar[gi], 4);
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  __syncthreads();

  if (warp == NCW) {
    // ------------------------------------------------------------ producer
    ProdState* ps = reinterpret_cast<ProdState*>(smem + L.prod);
    const int n_st = P.n_stages;
    int j = static_cast<int>(u_begin % n_st);
    int layer = static_cast<int>(u_begin / n_st);
    for (int k = 0; k < kDescAhead && u_begin + k < u_end; ++k)
      fetch_desc(P, ps, u_begin + k, advance_stage(j, k, n_st), lane);
    cp_async_commit();
    cp_async_wait<0>();
    __syncwarp();
    for (int k = 0; k < 2 && u_begin + k < u_end; ++k) fetch_toks(P, ps, u_begin + k, lane);
    cp_async_commit();
    cp_async_wait<0>();
    int base_layer = -1;
    const uint8_t *kp = nullptr, *kc = nullptr;
    int prev_layer = -1, prev_key = -1;
    StageMeta pm{};
    int pn = 0;
    const uint8_t* pks = nullptr;
    auto prepare = [&](int64_t u) {
      cp_async_wait<1>();
      __syncwarp();
      const AttnStage cur = ps->desc[u & 7];
      const AttnStage nx = ps->desc[(u + 1) & 7];
      pm.layer = layer;
      pm.key = cur.key;
      pm.delta = cur.delta;
      pm.n_tok = cur.n_tok;
      pm.sink_mask = cur.sink_mask;
      pm.flags = 0;
      if (layer != prev_layer || cur.key != prev_key) pm.flags |= kMetaFirst;
      if (u + 1 == u_end || j + 1 == n_st || nx.key != cur.key) pm.flags |= kMetaLast;
      prev_layer = layer;
      prev_key = cur.key;
      if (layer != base_layer) {
        const int64_t l_abs = P.layer_begin + layer;
        kp = P.k_pool + l_abs * P.pool_layer_stride;
        kc = P.k_cache + l_abs * P.cache_layer_stride;
        base_layer = layer;
      }
      pn = cur.n_tok;
      if (lane < pn) {
        const AttnTok tok = ps->tok[u & 3][lane];
        pks = ((tok.flags & kAttnFromCache) ? kc : kp) + static_cast<int64_t>(tok.row) * P.row_bytes;
      }
    };
    prepare(u_begin);
    int64_t it = 0;
    bool failed = false;
    int slot = 0;
    uint32_t round = 0;
    for (int64_t u = u_begin; u < u_end; ++u, ++it) {
      if (round > 0 && !__all_sync(kFullMask, mbar_wait_bounded(&empty[slot], (round - 1) & 1u))) {
        failed = true;
        break;
      }
      if (lane == 0) meta[slot] = pm;
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(pn) * rowb);
      __syncwarp();
      if (lane < pn) bulk_load(ring + slot * L.stage_bytes + lane * L.row_pitch, pks, rowb, &full[slot]);
      if (u + kDescAhead < u_end) fetch_desc(P, ps, u + kDescAhead, advance_stage(j, kDescAhead, n_st), lane);
      if (u + 2 < u_end) fetch_toks(P, ps, u + 2, lane);
      cp_async_commit();
      if (j + 1 == n_st) {
        j = 0;
        ++layer;
      } else {
        ++j;
      }
      if (++slot == NS) {
        slot = 0;
        ++round;
      }
      if (u + 1 < u_end) prepare(u + 1);
    }
    if (failed) {
      if (lane == 0) atomicOr(P.status, kDevTimeout);
      const int64_t issued = it;
      for (int64_t k = (issued > NS ? issued - NS : 0); k < issued; ++k)
        mbar_wait_bounded(&full[k % NS], static_cast<uint32_t>((k / NS) & 1));
    }
    cp_async_wait<0>();
    return;
  }
  if (warp > NCW) return;

  // -------------------------------------------------------------- consumer
  const int grp = warp >> 2;        // head group within the CTA: heads 16 grp .. 16 grp + 15
  const int qr = warp & 3;          // quarter: k-steps [9 qr, 9 qr + 9), output dims [128 qr, 128 qr + 128)
  const int g = lane >> 2, tq = lane & 3;
  const int mi = lane >> 3, ri = lane & 7;
  const uint32_t k_lane = static_cast<uint32_t>((ri + ((mi & 2) ? 8 : 0)) * pitch + (mi & 1) * 16);
  const uint32_t v_lane =
      static_cast<uint32_t>((ri + ((mi & 1) ? 8 : 0)) * pitch + (mi & 2) * 8 + qr * (kMlaLatent / 4) * 2);
  const uint32_t ring_u32 = smem_u32(ring);
  float* my_sbuf = sbuf + grp * (2 * 4 * 256);
  // this warp's q slice (16 heads x its 144 dims) and the group's rotated rope tiles
  uint8_t* qs = smem + L.qs + static_cast<size_t>(warp) * 16 * kMlaQPitch;
  uint8_t* rope_hl = smem + L.rope + static_cast<size_t>(grp) * 2 * 16 * kMlaRopePitch;
  // ldmatrix row address of this lane for an A tile (16 rows x 16 cols)
  const uint32_t a_lane = static_cast<uint32_t>((ri + ((mi & 1) ? 8 : 0)) * kMlaQPitch + ((mi & 2) ? 16 : 0));
  const uint32_t r_lane = static_cast<uint32_t>((ri + ((mi & 1) ? 8 : 0)) * kMlaRopePitch + ((mi & 2) ? 16 : 0));
  const uint32_t qs_u32 = smem_u32(qs), rope_u32 = smem_u32(rope_hl);
  constexpr int R0 = kMlaRopeKS0 - kMlaQKS * 3;  // first rope k-step within quarter 3's slice (5)

  float o[kMlaQNT][4];
  float m_run[2] = {-FLT_MAX, -FLT_MAX}, l_part[2] = {0.0f, 0.0f};
  int cur_delta = 0;
  bool have_rot = false;
  int slot = 0;
  uint32_t round = 0;
  uint32_t gphase = 0;
  for (int64_t u = u_begin; u < u_end; ++u) {
    if (!__all_sync(kFullMask, mbar_wait_bounded(&full[slot], round & 1u))) {
      if (lane == 0) atomicOr(P.status, kDevTimeout);
      return;
    }
    const StageMeta m = meta[slot];
    if (m.flags & kMetaFirst) {
      m_run[0] = m_run[1] = -FLT_MAX;
      l_part[0] = l_part[1] = 0.0f;
#pragma unroll
      for (int jn = 0; jn < kMlaQNT; ++jn) o[jn][0] = o[jn][1] = o[jn][2] = o[jn][3] = 0.0f;
      const int hg = m.key % P.head_groups;
      const int req = m.key / P.head_groups;
      const uint16_t* qh0 = P.q + ((static_cast<int64_t>(m.layer) * P.n_req + req) * P.num_q_heads + hg * HC +
                                   grp * kMlaHeadsPerGroup) * kMlaRow + kMlaQKS * 16 * qr;
      __syncwarp();  // the slice's previous readers are done
      // 16 heads x 144 dims = 16 x 18 chunks of 16 bytes
      for (int i = lane; i < 16 * kMlaQKS * 2; i += 32) {
        const int row = i / (kMlaQKS * 2), c = i % (kMlaQKS * 2);
        *reinterpret_cast<uint4*>(qs + row * kMlaQPitch + c * 16) =
            __ldg(reinterpret_cast<const uint4*>(qh0 + row * kMlaRow) + c);
      }
      __syncwarp();
      have_rot = false;
    }
    if (qr == 3 && (!have_rot || m.delta != cur_delta)) {
      // R(-delta) on the rope part: lane f takes frequency f for all 16 heads
      // (pairs (2f, 2f + 1) interleaved, (f, f + 32) neox)
      const int f = lane;
      const int ia = NEOX ? f : 2 * f, ib = NEOX ? f + 32 : 2 * f + 1;
      float cs = 1.0f, sn = 0.0f;
      if (m.delta != 0) shift_cossin(m.delta, __ldg(P.freq + f), cs, sn);
      const uint16_t* src = reinterpret_cast<const uint16_t*>(qs) + R0 * 16;
#pragma unroll 4
      for (int row = 0; row < 16; ++row) {
        const uint16_t* qrow = src + row * (kMlaQPitch / 2);
        const float a = __uint_as_float(static_cast<uint32_t>(qrow[ia]) << 16);
        const float b = __uint_as_float(static_cast<uint32_t>(qrow[ib]) << 16);
        const float ra = a * cs + b * sn, rb = b * cs - a * sn;
        const __nv_bfloat16 ha = __float2bfloat16_rn(ra), hb = __float2bfloat16_rn(rb);
        const __nv_bfloat16 la = __float2bfloat16_rn(ra - __bfloat162float(ha));
        const __nv_bfloat16 lb = __float2bfloat16_rn(rb - __bfloat162float(hb));
        __nv_bfloat16* hi_row = reinterpret_cast<__nv_bfloat16*>(rope_hl + row * kMlaRopePitch);
        __nv_bfloat16* lo_row = reinterpret_cast<__nv_bfloat16*>(rope_hl + (16 + row) * kMlaRopePitch);
        hi_row[ia] = ha;
        hi_row[ib] = hb;
        lo_row[ia] = la;
        lo_row[ib] = lb;
      }
      __syncwarp();
      cur_delta = m.delta;
      have_rot = true;
    }

    const uint32_t kbase = ring_u32 + static_cast<uint32_t>(slot * L.stage_bytes);
    // ---- partial S over this quarter's k-steps (two n-tiles of 8 positions;
    // even and odd k-steps accumulate separately: two short dependency chains)
    float s[2][4] = {}, s2[2][4] = {};
    const int nope_ks = qr < 3 ? kMlaQKS : R0;
#pragma unroll
    for (int kk = 0; kk < kMlaQKS; ++kk) {
      if (kk < nope_ks) {
        uint32_t a[4], b0, b1, b2, b3;
        ldsm_x4(qs_u32 + a_lane + kk * 32, a[0], a[1], a[2], a[3]);
        ldsm_x4(kbase + k_lane + (kMlaQKS * qr + kk) * 32, b0, b1, b2, b3);
        if (kk & 1) {
          mma_bf16(s2[0], a, b0, b1);
          mma_bf16(s2[1], a, b2, b3);
        } else {
          mma_bf16(s[0], a, b0, b1);
          mma_bf16(s[1], a, b2, b3);
        }
      }
    }
    if (qr == 3) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        uint32_t ah[4], al[4], b0, b1, b2, b3;
        ldsm_x4(rope_u32 + r_lane + r * 32, ah[0], ah[1], ah[2], ah[3]);
        ldsm_x4(rope_u32 + 16 * kMlaRopePitch + r_lane + r * 32, al[0], al[1], al[2], al[3]);
        ldsm_x4(kbase + k_lane + (kMlaRopeKS0 + r) * 32, b0, b1, b2, b3);
        mma_bf16(s[0], ah, b0, b1);
        mma_bf16(s[1], ah, b2, b3);
        mma_bf16(s2[0], al, b0, b1);
        mma_bf16(s2[1], al, b2, b3);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) s[nt][i] += s2[nt][i];
    // ---- exchange partial scores within the head group
    float* part = my_sbuf + (gphase & 1) * (4 * 256);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      *reinterpret_cast<float2*>(part + qr * 256 + g * 16 + 8 * nt + 2 * tq) = make_float2(s[nt][0], s[nt][1]);
      *reinterpret_cast<float2*>(part + qr * 256 + (g + 8) * 16 + 8 * nt + 2 * tq) = make_float2(s[nt][2], s[nt][3]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&gbar[grp]);
    if (!__all_sync(kFullMask, mbar_wait_bounded(&gbar[grp], gphase & 1u))) {
      if (lane == 0) atomicOr(P.status, kDevTimeout);
      return;
    }
    ++gphase;
    float sc[2][4];  // [row g / g + 8][positions 2tq, 2tq + 1, 8 + 2tq, 9 + 2tq]
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const float2 v = *reinterpret_cast<const float2*>(part + qq * 256 + (g + 8 * rr) * 16 + 8 * nt + 2 * tq);
          acc.x += v.x;
          acc.y += v.y;
        }
        sc[rr][2 * nt] = acc.x;
        sc[rr][2 * nt + 1] = acc.y;
      }
    // ---- online softmax per head (rows g and g + 8), identical in the four quarters
    float p[2][4], alpha[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      float mt = -FLT_MAX;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = (i < 2 ? 0 : 8) + 2 * tq + (i & 1);
        const bool live = t < m.n_tok;
        const float bias = ((m.sink_mask >> t) & 1u) ? P.sink_log2 : 0.0f;
        sc[rr][i] = live ? sc[rr][i] * P.scale_log2 + bias : -FLT_MAX;
        mt = fmaxf(mt, sc[rr][i]);
      }
      mt = fmaxf(mt, __shfl_xor_sync(kFullMask, mt, 1));
      mt = fmaxf(mt, __shfl_xor_sync(kFullMask, mt, 2));
      const float m_new = fmaxf(m_run[rr], mt);
      alpha[rr] = exp2f(m_run[rr] - m_new);
#pragma unroll
      for (int i = 0; i < 4; ++i) p[rr][i] = sc[rr][i] > -FLT_MAX ? exp2f(sc[rr][i] - m_new) : 0.0f;
      l_part[rr] = l_part[rr] * alpha[rr] + ((p[rr][0] + p[rr][1]) + (p[rr][2] + p[rr][3]));
      m_run[rr] = m_new;
    }
    if (!__all_sync(kFullMask, alpha[0] == 1.0f && alpha[1] == 1.0f)) {
#pragma unroll
      for (int jn = 0; jn < kMlaQNT; ++jn) {
        o[jn][0] *= alpha[0];
        o[jn][1] *= alpha[0];
        o[jn][2] *= alpha[1];
        o[jn][3] *= alpha[1];
      }
    }
    // A fragments of P (rows: heads g, g + 8; cols: the 16 positions), hi and lo parts
    uint32_t ph[4], pl[4];
    split_bf16x2(p[0][0], p[0][1], ph[0], pl[0]);
    split_bf16x2(p[1][0], p[1][1], ph[1], pl[1]);
    split_bf16x2(p[0][2], p[0][3], ph[2], pl[2]);
    split_bf16x2(p[1][2], p[1][3], ph[3], pl[3]);
    // ---- O += P V over this quarter's 128 latent dims
#pragma unroll
    for (int jn = 0; jn < kMlaQNT; jn += 2) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(kbase + v_lane + jn * 16, b0, b1, b2, b3);
      mma_bf16(o[jn], ph, b0, b1);
      mma_bf16(o[jn], pl, b0, b1);
      mma_bf16(o[jn + 1], ph, b2, b3);
      mma_bf16(o[jn + 1], pl, b2, b3);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    if (++slot == NS) {
      slot = 0;
      ++round;
    }

    if (m.flags & kMetaLast) {
      const AttnKey kk = P.keys[static_cast<int64_t>(m.layer) * P.n_keys + m.key];
      float* blk = P.records + static_cast<int64_t>(kk.rec_base + (blockIdx.x - kk.first_cta)) * BLK;
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int hrow = grp * kMlaHeadsPerGroup + g + 8 * rr;  // head within the record
#pragma unroll
        for (int jn = 0; jn < kMlaQNT; ++jn)
          *reinterpret_cast<float2*>(blk + hrow * kMlaLatent + qr * (kMlaLatent / 4) + 8 * jn + 2 * tq) =
              make_float2(o[jn][2 * rr], o[jn][2 * rr + 1]);
        float l_tot = l_part[rr];
        l_tot += __shfl_xor_sync(kFullMask, l_tot, 1);
        l_tot += __shfl_xor_sync(kFullMask, l_tot, 2);
        if (qr == 0 && tq == 0) {
          blk[HC * kMlaLatent + hrow] = m_run[rr];
          blk[HC * kMlaLatent + HC + hrow] = l_tot;
        }
      }
    }
  }
}

template <int PAIRING, int NG>
cudaError_t launch_mla_g(const AttnParams& p, int grid, size_t smem, cudaStream_t s) {
  auto kern = k_attend_mla<PAIRING, NG>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<grid, 32 * (4 * NG + 1), smem, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_merge<kMlaLatent>(p, kMlaHeadsPerGroup * NG, s);
}

template <int PAIRING, int NG>
int occupancy_mla_g(size_t smem) {
  auto kern = k_attend_mla<PAIRING, NG>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 32 * (4 * NG + 1), smem) != cudaSuccess) return 0;
  return n;
}

#define PIC_MLA_DISPATCH(FN, FAIL, ...)                                     \
  do {                                                                      \
    if (pairing == kNeox) {                                                 \
      if (ng == 1) return FN<kNeox, 1>(__VA_ARGS__);                        \
      if (ng == 2) return FN<kNeox, 2>(__VA_ARGS__);                        \
    } else {                                                                \
      if (ng == 1) return FN<kInterleaved, 1>(__VA_ARGS__);                 \
      if (ng == 2) return FN<kInterleaved, 2>(__VA_ARGS__);                 \
    }                                                                       \
    return FAIL;                                                            \
  } while (0)

}  // namespace

bool attend_config(int head_dim, int group, int heads_per_cta, int* ring, size_t* smem_bytes) {
  if (heads_per_cta < 1 || heads_per_cta > kAttnMaxHeads) return false;
  const SmemLayout base = smem_layout(head_dim, group, heads_per_cta, 0);
  if (base.total + 2 * base.stage_bytes > kSmemBudget) return false;
  int n = static_cast<int>((kSmemBudget - base.total) / base.stage_bytes);
  if (n > kAttnMaxStages) n = kAttnMaxStages;
  *ring = n;
  *smem_bytes = smem_layout(head_dim, group, heads_per_cta, n).total;
  return true;
}

int attend_ctas_per_sm(int pairing, int head_dim, int group, int heads_per_cta, size_t smem_bytes) {
  PIC_ATTN_DISPATCH(occupancy_g, 0, heads_per_cta, smem_bytes);
}

cudaError_t launch_attend(const AttnParams& p, int pairing, int head_dim, int group, int grid, size_t smem_bytes,
                          cudaStream_t s) {
  if (p.n_units <= 0 || grid <= 0) return cudaSuccess;
  PIC_ATTN_DISPATCH(launch_g, cudaErrorInvalidValue, p, grid, smem_bytes, s);
}

}  // namespace pic

namespace pic {

bool attend_mla_config(int ng, int* ring, size_t* smem_bytes) {
  if (ng != 1 && ng != 2) return false;
  // one group of 16 heads: two CTAs per SM (half the shared memory each, so
  // eight consumer warps share an SM); two groups: one CTA
  const size_t budget = ng == 1 ? kMlaSmemHalf : kSmemBudget;
  const MlaLayout base = mla_layout(ng, 0);
  if (base.total + 3 * base.stage_bytes > budget) return false;
  int n = static_cast<int>((budget - base.total) / base.stage_bytes);
  if (n > kMlaMaxStages) n = kMlaMaxStages;
  *ring = n;
  *smem_bytes = mla_layout(ng, n).total;
  return true;
}

int attend_mla_ctas_per_sm(int pairing, int ng, size_t smem_bytes) {
  PIC_MLA_DISPATCH(occupancy_mla_g, 0, smem_bytes);
}

cudaError_t launch_attend_mla(const AttnParams& p, int pairing, int ng, int grid, size_t smem_bytes,
                              cudaStream_t s) {
  if (p.n_units <= 0 || grid <= 0) return cudaSuccess;
  PIC_MLA_DISPATCH(launch_mla_g, cudaErrorInvalidValue, p, grid, smem_bytes, s);
}

cudaError_t launch_attend_merge_mla(const AttnParams& p, int heads_per_record, cudaStream_t s) {
  return launch_merge<kMlaLatent>(p, heads_per_record, s);
}

}  // namespace pic
