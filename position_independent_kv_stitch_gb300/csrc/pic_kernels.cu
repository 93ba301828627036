// CUDA kernels for position-independent KV stitching on GB300 (sm_103a).
//
// The work is a gather / delta-rotate / paged scatter over bf16 rows: it moves
// bytes and does 6 flops per rotated pair, so HBM bandwidth bounds it and
// tensor cores have nothing to do.  Design:
//   * Work unit = one run (<= block_size consecutive tokens of one chunk that
//     land in one paged block; contiguous in both pool and cache) x a group
//     of consecutive layers.  A persistent grid strides over the units with
//     runs fastest, so CTAs running together stream neighbouring memory and
//     finish within one unit of each other.
//   * Every thread owns a fixed slice of each head row (16-byte vectors), so
//     its RoPE frequencies are fixed: the cos/sin of delta * theta_i are
//     computed in registers when the delta changes and reused for every
//     token, head and layer that shares it (one delta per chunk: EPIC Guide,
//     "Mathematical Foundations: RoPE In-Place Key Transformation", 2. The
//     In-Place Shift Transformation -- R_{n+dp} = R_dp R_n).
//   * Neox half-split pairs (i, i + d/2) live in two vectors d bytes apart; a
//     thread loads both, so no shuffles are needed.  Interleaved pairs
//     (2i, 2i+1) sit inside one vector.
//   * Loads of the pool and stores into the cache are streaming (evict-first):
//     neither is re-read by this launch.
//   * Angles: the host gives f_i = theta_i / (2 pi) as a float pair hi + lo.
//     delta * hi is split exactly into p + e with one FMA (Dekker's
//     TwoProduct), p's integer part is dropped exactly, the small terms are
//     added back, and sincospif turns the fraction of a turn into cos/sin.
//     This keeps |delta| up to 2^24 accurate to ~1e-7 rad, where a plain
//     float delta * theta would be off by up to ~1e-2 rad at delta ~ 1e5.
//   * Device errors (a block-table entry outside the cache) skip the write and
//     raise a bit in the workspace header; no trap, no wait, no spin.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "pic_device.cuh"
#include "pic_internal.h"

namespace pic {
namespace {

using namespace dev;

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ uint4 ld_stream(const uint8_t* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void st_stream(uint8_t* p, uint4 v) {
  __stcs(reinterpret_cast<uint4*>(p), v);
}
__device__ __forceinline__ uint4 ld_plain(const uint8_t* p) {
  return *reinterpret_cast<const uint4*>(p);
}
__device__ __forceinline__ void st_plain(uint8_t* p, uint4 v) {
  *reinterpret_cast<uint4*>(p) = v;
}

// Resolves a run's destination block; false (and a raised status bit) when
// the block table entry does not name a cache block.
__device__ __forceinline__ bool resolve_block(const KernelParams& P, const RunDesc& r, int& blk,
                                              int& row0) {
  const int lb = r.dst_pos / P.block_size;
  row0 = r.dst_pos - lb * P.block_size;
  blk = __ldg(P.block_tables + static_cast<int64_t>(r.req) * P.max_blocks + lb);
  if (blk < 0 || blk >= P.num_cache_blocks) {
    if (threadIdx.x == 0) {
      atomicOr(&P.header->status, kDevBadBlock);
      P.header->bad_req = static_cast<uint32_t>(r.req);
      P.header->bad_pos = static_cast<uint32_t>(r.dst_pos);
    }
    return false;
  }
  return true;
}

__device__ __forceinline__ void emit_recompute(const KernelParams& P, const RunDesc& r, int lg) {
  if (P.ridx != nullptr && lg == 0 && r.idx_count > 0) {
    for (int t = threadIdx.x; t < r.idx_count; t += blockDim.x) P.ridx[r.idx_off + t] = r.idx_start + t;
  }
}

__device__ __forceinline__ void emit_indptr(const KernelParams& P) {
  if (P.indptr_dst != nullptr && blockIdx.x == 0) {
    for (int t = threadIdx.x; t < P.n_indptr; t += blockDim.x) P.indptr_dst[t] = P.indptr_src[t];
  }
}

// ------------------------------------------------ GQA stitch / in-place shift
//
// RD = rope dims of a head row (the whole head for GQA).  STITCH: read the
// pool, write K rotated and V copied into the paged cache.  !STITCH: rotate
// the cache's key rows in place (values untouched).
constexpr int kThreads = 256;

template <int PAIRING, int RD, bool STITCH>
__global__ void __launch_bounds__(kThreads, 2) k_rotate_rows(const KernelParams P) {
  constexpr bool NEOX = (PAIRING == kNeox);
  constexpr int VPR = RD / 8;                    // 16-B vectors in the rope slice
  constexpr int TPR = NEOX ? VPR / 2 : VPR;      // threads per head row
  constexpr int NF = NEOX ? 8 : 4;               // frequencies per thread
  constexpr int HSTEP = kThreads / TPR;          // head rows per block sweep
  constexpr int U = NEOX ? 4 : 8;                // sweeps in flight (16 vectors with V)
  static_assert(kThreads % TPR == 0, "thread slots must tile the block");

  const int slot = threadIdx.x % TPR;
  const int hrow0 = threadIdx.x / TPR;
  const int f0 = slot * NF;
  const int lo_off = P.rope_off_bytes + slot * 16;
  const int hi_off = lo_off + RD;                // neox partner: +RD/2 elements

  // Units are run x layer group.  Either each CTA owns a contiguous range of
  // units (layer group fastest) or CTAs stride over units (run fastest, so
  // CTAs running at the same time touch neighbouring runs of one layer).
  // A run's descriptor, block and cos/sin are set up once per change.
  const int64_t n_units = static_cast<int64_t>(P.n_runs) * P.n_lgroups;
  const int64_t u_first = P.contiguous ? n_units * blockIdx.x / gridDim.x : blockIdx.x;
  const int64_t u_last = P.contiguous ? n_units * (blockIdx.x + 1) / gridDim.x : n_units;
  const int64_t u_step = P.contiguous ? 1 : gridDim.x;
  int cur_run = -1;
  RunDesc r{};
  bool valid = false, has_v = false;
  int ntok = 0;
  int64_t dst_off = 0, src_off = 0, src_ls = 0;
  const uint8_t* ksrc = nullptr;
  const uint8_t* vsrc = nullptr;
  int cached_delta = 0;
  float c[NF], s[NF];
#pragma unroll
  for (int k = 0; k < NF; ++k) { c[k] = 1.0f; s[k] = 0.0f; }

  for (int64_t u = u_first; u < u_last; u += u_step) {
    int run, lg;
    if (P.contiguous) {
      run = static_cast<int>(u / P.n_lgroups);
      lg = static_cast<int>(u - static_cast<int64_t>(run) * P.n_lgroups);
    } else {
      lg = static_cast<int>(u / P.n_runs);
      run = static_cast<int>(u - static_cast<int64_t>(lg) * P.n_runs);
    }
    if (run != cur_run) {
      cur_run = run;
      r = P.runs[run];
      ntok = run_ntok(r);
      int blk, row0;
      valid = resolve_block(P, r, blk, row0);
      dst_off = valid ? (static_cast<int64_t>(blk) * P.block_size + row0) * P.row_bytes : 0;
      // source rows: the pool, blocks of the cache itself, or the destination (in place)
      const int kind = STITCH ? run_kind(r) : kRunInPlace;
      has_v = STITCH && kind != kRunInPlace;
      if (kind == kRunPool) {
        ksrc = P.k_src; vsrc = P.v_src; src_ls = P.src_layer_stride;
        src_off = static_cast<int64_t>(r.src) * P.row_bytes;
      } else {
        ksrc = P.k_dst; vsrc = P.v_dst; src_ls = P.dst_layer_stride;
        src_off = kind == kRunBlocks ? static_cast<int64_t>(r.src) * P.row_bytes : dst_off;
      }
      if (r.delta != 0 && r.delta != cached_delta) {
#pragma unroll
        for (int k = 0; k < NF; ++k) shift_cossin(r.delta, __ldg(P.freq + f0 + k), c[k], s[k]);
        cached_delta = r.delta;
      }
    }
    if (STITCH) emit_recompute(P, r, lg);
    if (!valid) continue;
    const bool rot = (r.delta != 0);
    const int nh = ntok * P.heads_per_token;
    const int l_end = min(P.num_layers, (lg + 1) * P.lg_size);
    for (int l = lg * P.lg_size; l < l_end; ++l) {
      const uint8_t* ks = ksrc + l * src_ls + src_off;
      uint8_t* kd = P.k_dst + l * P.dst_layer_stride + dst_off;
      const uint8_t* vs = has_v ? vsrc + l * src_ls + src_off : nullptr;
      uint8_t* vd = has_v ? P.v_dst + l * P.dst_layer_stride + dst_off : nullptr;

      for (int h0 = hrow0; h0 < nh; h0 += HSTEP * U) {
        uint4 ka[U], kb[U], va[U], vb[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
          const int h = h0 + j * HSTEP;
          if (h < nh) {
            const int64_t o = static_cast<int64_t>(h) * P.head_stride;
            if (STITCH) {
              ka[j] = ld_stream(ks + o + lo_off);
              if (NEOX) kb[j] = ld_stream(ks + o + hi_off);
              if (has_v) {
                va[j] = ld_stream(vs + o + lo_off);
                if (NEOX) vb[j] = ld_stream(vs + o + hi_off);
              }
            } else {
              ka[j] = ld_plain(ks + o + lo_off);
              if (NEOX) kb[j] = ld_plain(ks + o + hi_off);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < U; ++j) {
          const int h = h0 + j * HSTEP;
          if (h < nh) {
            const int64_t o = static_cast<int64_t>(h) * P.head_stride;
            if (rot) {
              if (NEOX) rotate_neox(ka[j], kb[j], c, s);
              else rotate_interleaved(ka[j], c, s);
            }
            if (STITCH) {
              st_stream(kd + o + lo_off, ka[j]);
              if (NEOX) st_stream(kd + o + hi_off, kb[j]);
              if (has_v) {
                st_stream(vd + o + lo_off, va[j]);
                if (NEOX) st_stream(vd + o + hi_off, vb[j]);
              }
            } else {
              st_plain(kd + o + lo_off, ka[j]);
              if (NEOX) st_plain(kd + o + hi_off, kb[j]);
            }
          }
        }
      }
    }
  }
  if (STITCH) emit_indptr(P);
}

// ------------------------------------------------------------- MLA stitch
//
// Row = 512-d latent (64 vectors, copied) + 64-d rope key (8 vectors,
// rotated): Irminsul, 2.1 Structural Insight: MLA Decomposition and 2.2
// "delta-Rotation Rule".  288 threads = 4 rows x 72 vectors, so every thread
// keeps one column (and one set of frequencies) for the whole kernel.
constexpr int kMlaRowVecs = 72;
constexpr int kMlaLatVecs = 64;
constexpr int kMlaRowsPerSweep = 4;
constexpr int kMlaThreads = kMlaRowVecs * kMlaRowsPerSweep;  // 288

template <int PAIRING>
__global__ void __launch_bounds__(kMlaThreads) k_stitch_mla(const KernelParams P) {
  constexpr bool NEOX = (PAIRING == kNeox);
  constexpr int NF = NEOX ? 8 : 4;
  constexpr int U = 4;
  const int col = threadIdx.x % kMlaRowVecs;
  const int trow = threadIdx.x / kMlaRowVecs;
  // rope role: interleaved -> every rope column rotates its own 4 pairs;
  // neox -> columns 64..67 rotate with partners 68..71, which stay idle.
  const bool rope_col = col >= kMlaLatVecs;
  const bool active = !(NEOX && col >= kMlaLatVecs + 4);
  const int rv = col - kMlaLatVecs;
  const int f0 = rope_col ? rv * NF : 0;

  const int64_t n_units = static_cast<int64_t>(P.n_runs) * P.n_lgroups;
  for (int64_t u = blockIdx.x; u < n_units; u += gridDim.x) {
    const int lg = static_cast<int>(u / P.n_runs);
    const RunDesc r = P.runs[u - static_cast<int64_t>(lg) * P.n_runs];
    emit_recompute(P, r, lg);
    int blk, row0;
    if (!resolve_block(P, r, blk, row0)) continue;

    const bool rot = rope_col && (r.delta != 0);
    float c[NF], s[NF];
    if (rot) {
#pragma unroll
      for (int k = 0; k < NF; ++k) shift_cossin(r.delta, __ldg(P.freq + f0 + k), c[k], s[k]);
    }
    const int ntok = run_ntok(r);
    const int kind = run_kind(r);
    const int64_t dst_off = (static_cast<int64_t>(blk) * P.block_size + row0) * P.row_bytes;
    // source rows: the pool, blocks of the cache itself, or the destination
    // (in place: only the rope key moves, the latent stays where it is)
    const uint8_t* sbase = kind == kRunPool ? P.k_src : P.k_dst;
    const int64_t sls = kind == kRunPool ? P.src_layer_stride : P.dst_layer_stride;
    const int64_t src_off = kind == kRunInPlace ? dst_off : static_cast<int64_t>(r.src) * P.row_bytes;
    const bool work = active && !(kind == kRunInPlace && !rope_col);
    const int l_begin = lg * P.lg_size;
    const int l_end = min(P.num_layers, l_begin + P.lg_size);

    for (int l = l_begin; l < l_end && work; ++l) {
      const uint8_t* src = sbase + l * sls + src_off + col * 16;
      uint8_t* dst = P.k_dst + l * P.dst_layer_stride + dst_off + col * 16;
      for (int r0 = trow; r0 < ntok; r0 += kMlaRowsPerSweep * U) {
        uint4 x[U], y[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
          const int row = r0 + j * kMlaRowsPerSweep;
          if (row < ntok) {
            x[j] = ld_stream(src + static_cast<int64_t>(row) * P.row_bytes);
            if (NEOX && rope_col) y[j] = ld_stream(src + static_cast<int64_t>(row) * P.row_bytes + 64);
          }
        }
#pragma unroll
        for (int j = 0; j < U; ++j) {
          const int row = r0 + j * kMlaRowsPerSweep;
          if (row < ntok) {
            if (rot) {
              if (NEOX) rotate_neox(x[j], y[j], c, s);
              else rotate_interleaved(x[j], c, s);
            }
            st_stream(dst + static_cast<int64_t>(row) * P.row_bytes, x[j]);
            if (NEOX && rope_col) st_stream(dst + static_cast<int64_t>(row) * P.row_bytes + 64, y[j]);
          }
        }
      }
    }
  }
  emit_indptr(P);
}

// ---------------------------------------------------------- cos/sin probe

__global__ void k_cossin(const int32_t* __restrict__ deltas, int32_t n, const float2* __restrict__ freq,
                         int32_t half, float* __restrict__ out) {
  const int64_t total = static_cast<int64_t>(n) * half;
  for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t j = t / half;
    const int i = static_cast<int>(t - j * half);
    float c, s;
    shift_cossin(deltas[j], freq[i], c, s);
    out[2 * t] = c;
    out[2 * t + 1] = s;
  }
}

template <typename K>
int occupancy_of(K kernel, int threads) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0) != cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  return n > 0 ? n : 1;
}

}  // namespace

// ---------------------------------------------------------------- launchers

#define PIC_DISPATCH_RD(RD_, PAIR_, STITCH_, FN)                                   \
  do {                                                                             \
    if ((RD_) == 64) { FN(PAIR_, 64, STITCH_); }                                   \
    else if ((RD_) == 128) { FN(PAIR_, 128, STITCH_); }                            \
    else if ((RD_) == 256) { FN(PAIR_, 256, STITCH_); }                            \
    else return cudaErrorInvalidValue;                                             \
  } while (0)

#define PIC_LAUNCH_ROWS(PAIR_, RD_, STITCH_) \
  k_rotate_rows<PAIR_, RD_, STITCH_><<<grid, kThreads, 0, stream>>>(p)

#define PIC_OCC_ROWS(PAIR_, RD_, STITCH_) \
  return occupancy_of(k_rotate_rows<PAIR_, RD_, STITCH_>, kThreads)

cudaError_t launch_stitch_gqa(const KernelParams& p, int pairing, int head_dim, int grid,
                              cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  if (pairing == kNeox) PIC_DISPATCH_RD(head_dim, kNeox, true, PIC_LAUNCH_ROWS);
  else PIC_DISPATCH_RD(head_dim, kInterleaved, true, PIC_LAUNCH_ROWS);
  return cudaGetLastError();
}

cudaError_t launch_rerotate(const KernelParams& p, int pairing, int rope_dim, int grid,
                            cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  if (pairing == kNeox) PIC_DISPATCH_RD(rope_dim, kNeox, false, PIC_LAUNCH_ROWS);
  else PIC_DISPATCH_RD(rope_dim, kInterleaved, false, PIC_LAUNCH_ROWS);
  return cudaGetLastError();
}

cudaError_t launch_stitch_mla(const KernelParams& p, int pairing, int grid, cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  if (pairing == kNeox) k_stitch_mla<kNeox><<<grid, kMlaThreads, 0, stream>>>(p);
  else k_stitch_mla<kInterleaved><<<grid, kMlaThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_cossin(const int32_t* deltas, int32_t n, const float2* freq, int32_t half,
                          float* out, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(n) * half;
  if (total <= 0) return cudaSuccess;
  const int threads = 256;
  const int64_t want = (total + threads - 1) / threads;
  const int grid = static_cast<int>(want < 65535 ? want : 65535);
  k_cossin<<<grid, threads, 0, stream>>>(deltas, n, freq, half, out);
  return cudaGetLastError();
}

int occupancy_stitch_gqa(int pairing, int head_dim) {
  if (pairing == kNeox) PIC_DISPATCH_RD(head_dim, kNeox, true, PIC_OCC_ROWS);
  else PIC_DISPATCH_RD(head_dim, kInterleaved, true, PIC_OCC_ROWS);
  return 1;
}

int occupancy_rerotate(int pairing, int rope_dim) {
  if (pairing == kNeox) PIC_DISPATCH_RD(rope_dim, kNeox, false, PIC_OCC_ROWS);
  else PIC_DISPATCH_RD(rope_dim, kInterleaved, false, PIC_OCC_ROWS);
  return 1;
}

int occupancy_stitch_mla(int pairing) {
  return pairing == kNeox ? occupancy_of(k_stitch_mla<kNeox>, kMlaThreads)
                          : occupancy_of(k_stitch_mla<kInterleaved>, kMlaThreads);
}

}  // namespace pic
