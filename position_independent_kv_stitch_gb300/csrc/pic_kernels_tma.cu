// Bulk-copy (TMA) pipelined variant of the stitch / in-place kernels, sm_103a.
//
// CTAs stride over work units (unit = run x a few consecutive layers, runs
// fastest, so CTAs running together touch neighbouring memory); each CTA
// moves its units' tiles (one tile = one run x one layer) through a ring of
// shared-memory stages:
//   * one thread issues cp.async.bulk global -> shared copies of a unit's
//     whole source rows (a run's rows are contiguous in the pool and in the
//     paged block), tracked by one mbarrier per stage, keeping NS - 1 units
//     of loads in flight;
//   * all threads rotate only the RoPE slice of the key rows in shared
//     memory (EPIC Guide: Position-Independent Caching for LLM Serving,
//     "Mathematical Foundations" 2: k_target = R_dp k_cached, one dp per
//     chunk; Irminsul, 2.1: for MLA only the 64-d k_r, the 512-d latent is
//     reused verbatim);
//   * the same thread issues cp.async.bulk shared -> global stores of the
//     whole tile into the paged cache.
// Values and MLA latents never pass through registers, and the bytes in
// flight no longer depend on register count.  cos/sin are recomputed only
// when the tile's delta changes (the layers of a unit share it).
//
// Every mbarrier wait is bounded: on timeout the CTA raises PIC_DEV_TIMEOUT
// in the workspace header, waits (bounded) for the copies it issued, and
// exits; no wait can hang the GPU.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "pic_device.cuh"
#include "pic_internal.h"

namespace pic {
namespace {

using namespace dev;

constexpr int kTmaThreads = 256;

// What the producer learned about a unit, for the consumers of its stage.
struct StageMeta {
  uint8_t* dst_k;
  uint8_t* dst_v;
  int32_t delta;
  int32_t ntok;
  int32_t valid;     // destination block resolved inside the cache
  int32_t layer;
  int32_t idx_off;
  int32_t idx_count;
  int32_t idx_start;
  int32_t has_v;     // the tile carries a value tile too (not for in-place runs)
};

// MODE 0: GQA/MLA stitch with values (K + V tiles); 1: stitch without values
// (MLA rows); 2: in place (K rows of the cache, read and written back).
// HOOK: the instance launched only under pic_debug_stall_next_launch (the
// stall test hook and a launch-specific wait bound); the production
// instances carry neither.
template <int PAIRING, int RD, int MODE, bool HOOK = false>
__global__ void __launch_bounds__(kTmaThreads, 1) k_tma_pipeline(const KernelParams P, const TmaConfig C) {
  constexpr bool NEOX = (PAIRING == kNeox);
  constexpr bool HAS_V = (MODE == 0);
  constexpr bool INPLACE = (MODE == 2);
  constexpr int VPR = RD / 8;
  constexpr int TPR = NEOX ? VPR / 2 : VPR;
  constexpr int NF = NEOX ? 8 : 4;
  constexpr int HSTEP = kTmaThreads / TPR;
  static_assert(kTmaThreads % TPR == 0, "thread slots must tile the block");

  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stages = smem;
  StageMeta* meta = reinterpret_cast<StageMeta*>(smem + static_cast<size_t>(C.stages) * C.stage_bytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(meta + C.stages);

  const int tid = threadIdx.x;
  // Units = run x group of lg_size consecutive layers.  Strided order
  // (P.contiguous == 0): u = group * n_runs + run and CTA c takes units
  // c, c + G, ..., so CTAs running together touch neighbouring runs of one
  // layer group.  Contiguous order: u = run * n_lgroups + group and CTA c owns
  // [c*U/G, (c+1)*U/G), so a run's layers follow one another.  A unit's tiles
  // are its layers, one tile = one run x one layer.
  const int64_t n_units = static_cast<int64_t>(P.n_runs) * P.n_lgroups;
  const int64_t G = gridDim.x;
  const int64_t c_begin = n_units * blockIdx.x / G;
  const int64_t c_end = n_units * (blockIdx.x + 1) / G;
  auto ceil_div = [](int64_t x, int64_t y) -> int64_t { return x <= 0 ? 0 : (x + y - 1) / y; };
  auto count_congruent = [&](int64_t a, int64_t b, int64_t m, int64_t r) -> int64_t {
    return ceil_div(b - r, m) - ceil_div(a - r, m);  // #{u in [a, b) : u = r (mod m)}
  };
  int64_t my_units, my_last;
  if (P.contiguous) {
    my_units = c_end - c_begin;
    my_last = count_congruent(c_begin, c_end, P.n_lgroups, P.n_lgroups - 1);
  } else {
    my_units = count_congruent(0, n_units, G, blockIdx.x);
    my_last = count_congruent(static_cast<int64_t>(P.n_lgroups - 1) * P.n_runs, n_units, G, blockIdx.x);
  }
  const int last_len = P.num_layers - (P.n_lgroups - 1) * P.lg_size;  // layers in the last group
  const int n_tiles = static_cast<int>(my_units * P.lg_size - my_last * (P.lg_size - last_len));
  const int tensor_bytes = C.stage_bytes / (HAS_V ? 2 : 1);  // V tile sits after the K tile

  if (tid == 0) {
    for (int s = 0; s < C.stages; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // k-th unit of this CTA -> (run, layer group)
  auto unit_of = [&](int64_t k, int& run, int& grp) {
    if (P.contiguous) {
      const int64_t u = c_begin + k;
      run = static_cast<int>(u / P.n_lgroups);
      grp = static_cast<int>(u - static_cast<int64_t>(run) * P.n_lgroups);
    } else {
      const int64_t u = blockIdx.x + k * G;
      grp = static_cast<int>(u / P.n_runs);
      run = static_cast<int>(u - static_cast<int64_t>(grp) * P.n_runs);
    }
  };
  auto block_of = [&](const RunDesc& d) -> int {
    return __ldg(P.block_tables + static_cast<int64_t>(d.req) * P.max_blocks + d.dst_pos / P.block_size);
  };

  // Producer (thread 0): walks this CTA's tiles in order, fills each stage's
  // metadata and starts its copies.  A unit's descriptor and destination
  // block are looked up once, when its first tile is issued, and reused for
  // its other layers.  (Prefetching them further ahead does not help:
  // mbarrier.arrive has release semantics, so the next arrive would wait for
  // the prefetch anyway.)
  int64_t k_unit = 0;  // unit of the next tile
  int cur_l = 0;       // layer of the next tile inside its unit
  int cached_run = -1;
  int grp = 0;
  RunDesc r{};
  bool valid = false;
  int64_t dst_off = 0;
  auto issue = [&](int t) {
    const int s = t % C.stages;
    if (cur_l == 0) {
      int run;
      unit_of(k_unit, run, grp);
      if (run != cached_run) {
        r = P.runs[run];
        const int blk = block_of(r);
        valid = blk >= 0 && blk < P.num_cache_blocks;
        dst_off = valid ? (static_cast<int64_t>(blk) * P.block_size + r.dst_pos % P.block_size) * P.row_bytes : 0;
        cached_run = run;
        if (!valid) {
          atomicOr(&P.header->status, kDevBadBlock);
          P.header->bad_req = static_cast<uint32_t>(r.req);
          P.header->bad_pos = static_cast<uint32_t>(r.dst_pos);
        }
      }
    }
    const int l = grp * P.lg_size + cur_l;
    if (++cur_l == min(P.lg_size, P.num_layers - grp * P.lg_size)) {  // next tile starts unit k + 1
      cur_l = 0;
      ++k_unit;
    }
    const int ntok = run_ntok(r);
    const int kind = INPLACE ? kRunInPlace : run_kind(r);
    const bool has_v = HAS_V && kind != kRunInPlace;
    StageMeta& m = meta[s];
    m.delta = r.delta;
    m.ntok = ntok;
    m.valid = valid ? 1 : 0;
    m.layer = l;
    m.idx_off = r.idx_off;
    m.idx_count = r.idx_count;
    m.idx_start = r.idx_start;
    m.has_v = has_v ? 1 : 0;
    m.dst_k = P.k_dst + l * P.dst_layer_stride + dst_off;
    m.dst_v = HAS_V ? P.v_dst + l * P.dst_layer_stride + dst_off : nullptr;
    // test hook (pic_debug_stall_next_launch): this tile's barrier never
    // completes, so the waits for it run out and take the failure path below
    if (HOOK && P.debug_stall != 0 && blockIdx.x == 0 && t == P.debug_stall - 1) return;
    if (!valid || ntok == 0) {
      mbar_arrive(&bars[s]);  // nothing to copy: complete the phase
      return;
    }
    const uint32_t bytes = static_cast<uint32_t>(ntok) * static_cast<uint32_t>(P.row_bytes);
    uint8_t* st = stages + static_cast<size_t>(s) * C.stage_bytes;
    // source rows: the pool, blocks of the cache itself, or the destination (in place)
    const int64_t src_off = static_cast<int64_t>(r.src) * P.row_bytes;
    const uint8_t* src_k = kind == kRunInPlace ? m.dst_k
                           : kind == kRunBlocks ? P.k_dst + l * P.dst_layer_stride + src_off
                                                : P.k_src + l * P.src_layer_stride + src_off;
    mbar_arrive_expect_tx(&bars[s], bytes * (has_v ? 2u : 1u));
    bulk_load(st, src_k, bytes, &bars[s]);
    if (has_v) {
      const uint8_t* src_v = kind == kRunBlocks ? P.v_dst + l * P.dst_layer_stride + src_off
                                                : P.v_src + l * P.src_layer_stride + src_off;
      bulk_load(st + tensor_bytes, src_v, bytes, &bars[s]);
    }
  };

  const uint32_t spins = HOOK && P.max_spins != 0 ? P.max_spins : kMaxSpins;
  int issued = 0;
  if (tid == 0) {
    const int pre = min(C.stages - 1, n_tiles);
    for (; issued < pre; ++issued) issue(issued);
  }

  const int slot = tid % TPR;
  const int hrow0 = tid / TPR;
  const int f0 = slot * NF;
  const int lo_off = P.rope_off_bytes + slot * 16;
  const int hi_off = lo_off + RD;
  float c[NF], s[NF];
  int cached_delta = INT_MIN;
  bool aborted = false;
  int t = 0;

  for (; t < n_tiles; ++t) {
    const int sidx = t % C.stages;
    const uint32_t parity = static_cast<uint32_t>(t / C.stages) & 1u;
    const bool ok = mbar_wait_bounded(&bars[sidx], parity, spins);
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    const StageMeta m = meta[sidx];
    uint8_t* st = stages + static_cast<size_t>(sidx) * C.stage_bytes;
    if (!INPLACE && P.ridx != nullptr && m.layer == 0 && m.idx_count > 0) {
      for (int i = tid; i < m.idx_count; i += kTmaThreads) P.ridx[m.idx_off + i] = m.idx_start + i;
    }
    if (m.valid && m.delta != 0) {
      if (m.delta != cached_delta) {
#pragma unroll
        for (int k = 0; k < NF; ++k) shift_cossin(m.delta, __ldg(P.freq + f0 + k), c[k], s[k]);
        cached_delta = m.delta;
      }
      const int nh = m.ntok * P.heads_per_token;
      for (int h = hrow0; h < nh; h += HSTEP) {
        uint8_t* row = st + h * P.head_stride;
        uint4 a = *reinterpret_cast<uint4*>(row + lo_off);
        if (NEOX) {
          uint4 b = *reinterpret_cast<uint4*>(row + hi_off);
          rotate_neox(a, b, c, s);
          *reinterpret_cast<uint4*>(row + hi_off) = b;
        } else {
          rotate_interleaved(a, c, s);
        }
        *reinterpret_cast<uint4*>(row + lo_off) = a;
      }
    }
    fence_proxy_async_smem();  // make the rotated rows visible to the bulk copy engine
    __syncthreads();
    if (tid == 0) {
      if (m.valid && m.ntok > 0) {
        const uint32_t bytes = static_cast<uint32_t>(m.ntok) * static_cast<uint32_t>(P.row_bytes);
        bulk_store(m.dst_k, st, bytes);
        if (HAS_V && m.has_v) bulk_store(m.dst_v, st + tensor_bytes, bytes);
      }
      bulk_commit();
      bulk_wait_read_1();  // the previous unit's stores have read their stage
      if (issued < n_tiles) issue(issued++);
    }
  }

  if (tid == 0) {
    if (aborted) {
      atomicOr(&P.header->status, kDevTimeout);
      // wait (bounded) for loads this CTA started but nobody consumed
      for (int u = t; u < issued; ++u)
        mbar_wait_bounded(&bars[u % C.stages], static_cast<uint32_t>(u / C.stages) & 1u, spins);
    }
    bulk_wait_all();
  }
  if (!INPLACE && P.indptr_dst != nullptr && blockIdx.x == 0) {
    for (int i = tid; i < P.n_indptr; i += kTmaThreads) P.indptr_dst[i] = P.indptr_src[i];
  }
}

template <typename K>
cudaError_t launch_one(K kernel, const KernelParams& p, const TmaConfig& c, int grid, cudaStream_t stream) {
  const size_t smem = tma_smem_bytes(c);
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kernel<<<grid, kTmaThreads, smem, stream>>>(p, c);
  return cudaGetLastError();
}

}  // namespace

size_t tma_smem_bytes(const TmaConfig& c) {
  return static_cast<size_t>(c.stages) * c.stage_bytes + static_cast<size_t>(c.stages) * sizeof(StageMeta) +
         static_cast<size_t>(c.stages) * sizeof(uint64_t);
}

cudaError_t launch_tma(const KernelParams& p, const TmaConfig& c, int mode, int pairing, int rope_dim, int grid,
                       cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  if (p.debug_stall != 0 || p.max_spins != 0) {  // test hook: stitch modes only
#define PIC_TMA_HOOK(MODE_, PAIR_, RD_)                                             \
  if (mode == MODE_ && pairing == PAIR_ && rope_dim == RD_)                         \
    return launch_one(k_tma_pipeline<PAIR_, RD_, MODE_, true>, p, c, grid, stream);
    PIC_TMA_HOOK(0, kNeox, 64) PIC_TMA_HOOK(0, kNeox, 128) PIC_TMA_HOOK(0, kNeox, 256)
    PIC_TMA_HOOK(0, kInterleaved, 64) PIC_TMA_HOOK(0, kInterleaved, 128) PIC_TMA_HOOK(0, kInterleaved, 256)
    PIC_TMA_HOOK(1, kNeox, 64) PIC_TMA_HOOK(1, kInterleaved, 64)
#undef PIC_TMA_HOOK
    return cudaErrorInvalidValue;
  }
#define PIC_TMA_CASE(MODE_, PAIR_, RD_)                                             \
  if (mode == MODE_ && pairing == PAIR_ && rope_dim == RD_)                         \
    return launch_one(k_tma_pipeline<PAIR_, RD_, MODE_>, p, c, grid, stream);
#define PIC_TMA_RD(MODE_, PAIR_) PIC_TMA_CASE(MODE_, PAIR_, 64) PIC_TMA_CASE(MODE_, PAIR_, 128) PIC_TMA_CASE(MODE_, PAIR_, 256)
  PIC_TMA_RD(0, kNeox)
  PIC_TMA_RD(0, kInterleaved)
  PIC_TMA_CASE(1, kNeox, 64)
  PIC_TMA_CASE(1, kInterleaved, 64)
  PIC_TMA_RD(2, kNeox)
  PIC_TMA_RD(2, kInterleaved)
#undef PIC_TMA_RD
#undef PIC_TMA_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pic
