// Decode attention over a stitched context, with the delta-rotation fused into
// the key loads (GQA, sm_103a).
//
// Irminsul: MLA-Native Position-Independent Caching for Agentic LLM Serving,
// 2.2 "delta-Rotation Rule" and 4. Results: the rotation R(delta) k can be
// applied on the HBM -> on-chip load path of attention instead of writing a
// rotated copy, so no extra HBM traffic is spent.  Here every context
// position is read from where it lives -- a chunk token from its source rows
// (pool, or the blocks of a block-resident chunk) with its key rotated by the
// chunk's delta in registers, an inline token from the request's paged cache
// -- and one decode step of attention runs over them:
//   scores = scale * q . R(delta) k + bias,  p = softmax,  out = sum p v
// (bias: LegoLink's pseudo-sink suppression, EPIC Guide: Position-Independent
// Caching for LLM Serving, LegoLink "1. Identifying and Neutralizing
// Pseudo-Sinks" -- the first k tokens of every chunk not at position 0 get a
// negative logit offset).
//
// Flash-decoding split: one CTA per (tile of <= 128 positions, KV head,
// layer) computes the tile's max, sum of exponentials and weighted value sum
// for the query heads of its group; a second kernel merges the tiles.  The work is memory-bound (one pass over K and V, a few FMAs per
// byte) and runs on CUDA cores; tensor cores would idle on a 1-token query.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <cstdint>

#include "pic_internal.h"

namespace pic {
namespace {

constexpr int kAttnThreads = kAttnTileTokens;  // one thread per position of a tile

__device__ __forceinline__ void shift_cossin(int delta, float2 f, float& c, float& s) {
  const float d = static_cast<float>(delta);   // exact for |delta| < 2^24
  const float p = __fmul_rn(d, f.x);
  const float e = __fmaf_rn(d, f.x, -p);       // d * hi == p + e exactly (TwoProduct)
  const float r = __fsub_rn(p, rintf(p));      // exact, |r| <= 1/2 turn
  const float t = __fadd_rn(r, __fmaf_rn(d, f.y, e));
  sincospif(2.0f * t, &s, &c);
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t vword(const uint4& v, int w) {
  return w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w));
}

// Block-wide max / sum over the threads of the CTA through shared scratch.
__device__ __forceinline__ float block_max(float x, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
  __syncthreads();
  float m = red[0];
#pragma unroll
  for (int w = 1; w < kAttnThreads / 32; ++w) m = fmaxf(m, red[w]);
  __syncthreads();
  return m;
}
__device__ __forceinline__ float block_sum(float x, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
  __syncthreads();
  float t = 0.0f;
#pragma unroll
  for (int w = 0; w < kAttnThreads / 32; ++w) t += red[w];
  __syncthreads();
  return t;
}

// grid: (tiles, kv heads, layers).  G = query heads per KV head, D = head dim.
//
// The rotation is applied to the query, not the keys: q . R(d) k =
// (R(-d) q) . k, so each tile rotates its G query heads once per distinct
// delta (<= kAttnMaxSlots) into shared memory and every key is consumed as
// stored.  Thread t owns token t of the tile: it loads the token's head row
// (2*D bytes) and dots it with the rotated query of its delta, read as
// 16-byte broadcasts.  After the tile's softmax statistics, VT = D/8 threads
// share each value row for the weighted sum.  No shuffle or barrier sits in
// a divergent region: every thread of the CTA runs the same reductions.
template <int PAIRING, int D, int G>
__global__ void __launch_bounds__(kAttnThreads) k_attend_tiles(const AttnParams P) {
  constexpr bool NEOX = (PAIRING == kNeox);
  constexpr int HALF = D / 2;
  constexpr int VPR = D / 8;              // 16-B vectors per head row
  constexpr int VT = VPR;                 // value phase: threads per row
  constexpr int VG = kAttnThreads / VT;   // value phase: rows handled at once
  static_assert(kAttnThreads % VT == 0 && 32 % VT == 0, "value threads must tile a warp");

  // The rotated queries are dead once the scores are computed (the softmax
  // reductions' barriers separate the two uses), so the per-warp value sums
  // reuse their shared memory.
  constexpr int QROT = attn_slots(G) * G * D;
  constexpr int PART = (kAttnThreads / 32) * G * D;
  __shared__ __align__(16) float buf[QROT > PART ? QROT : PART];
  float (*q_rot)[G][D] = reinterpret_cast<float (*)[G][D]>(buf);
  float (*part)[G][D] = reinterpret_cast<float (*)[G][D]>(buf);
  __shared__ float p_s[kAttnThreads][G];
  __shared__ AttnTok tok_s[kAttnThreads];
  __shared__ float red[kAttnThreads / 32];

  const int tile = blockIdx.x;
  const int h = blockIdx.y;
  const int layer = P.layer_begin + blockIdx.z;
  const AttnTile T = P.tiles[tile];
  const int tid = threadIdx.x;
  const bool have = tid < T.n_tok;
  if (have) tok_s[tid] = P.toks[T.tok_off + tid];

  // ---- R(-delta) q for every distinct delta of the tile
  const uint16_t* qg = P.q + ((static_cast<int64_t>(blockIdx.z) * P.n_req + T.req) * P.num_q_heads + h * G) * D;
  for (int i = tid; i < T.n_slots * G * HALF; i += kAttnThreads) {
    const int slot = i / (G * HALF), g = (i / HALF) % G, f = i % HALF;
    const int a = NEOX ? f : 2 * f, b = NEOX ? f + HALF : 2 * f + 1;
    const float qa = __uint_as_float(static_cast<uint32_t>(qg[g * D + a]) << 16);
    const float qb = __uint_as_float(static_cast<uint32_t>(qg[g * D + b]) << 16);
    float c = 1.0f, s = 0.0f;
    if (T.deltas[slot] != 0) shift_cossin(T.deltas[slot], __ldg(P.freq + f), c, s);
    q_rot[slot][g][a] = qa * c + qb * s;        // R(-delta): rotate backwards
    q_rot[slot][g][b] = qb * c - qa * s;
  }
  __syncthreads();

  // ---- scores: thread t owns token t of the tile
  float sc[G];
#pragma unroll
  for (int g = 0; g < G; ++g) sc[g] = -FLT_MAX;
  if (have) {
    const AttnTok tk = tok_s[tid];
    const bool from_cache = (tk.flags & kAttnFromCache) != 0;
    const uint8_t* base = from_cache ? P.k_cache + layer * P.cache_layer_stride
                                     : P.k_pool + layer * P.pool_layer_stride;
    const uint8_t* row = base + static_cast<int64_t>(tk.row) * P.row_bytes + h * (D * 2);
    uint4 kv[VPR];
#pragma unroll
    for (int v = 0; v < VPR; ++v) kv[v] = *reinterpret_cast<const uint4*>(row + v * 16);
    const int slot = tk.flags & 0xff;
    float dot[G];
#pragma unroll
    for (int g = 0; g < G; ++g) dot[g] = 0.0f;
#pragma unroll
    for (int v = 0; v < VPR; ++v) {
      float kf[8];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        kf[2 * w] = bf_lo(vword(kv[v], w));
        kf[2 * w + 1] = bf_hi(vword(kv[v], w));
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float4 q0 = *reinterpret_cast<const float4*>(&q_rot[slot][g][v * 8]);
        const float4 q1 = *reinterpret_cast<const float4*>(&q_rot[slot][g][v * 8 + 4]);
        dot[g] += kf[0] * q0.x + kf[1] * q0.y + kf[2] * q0.z + kf[3] * q0.w +
                  kf[4] * q1.x + kf[5] * q1.y + kf[6] * q1.z + kf[7] * q1.w;
      }
    }
    const float bias = (tk.flags & kAttnSink) ? P.sink_bias : 0.0f;
#pragma unroll
    for (int g = 0; g < G; ++g) sc[g] = dot[g] * P.scale + bias;
  }

  // ---- tile softmax statistics per query head
  float m_g[G], l_g[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m_g[g] = block_max(sc[g], red);
    const float pv = have ? __expf(sc[g] - m_g[g]) : 0.0f;
    p_s[tid][g] = pv;
    l_g[g] = block_sum(pv, red);
  }
  __syncthreads();

  // ---- weighted value sum: VT threads per row, VG rows at a time
  const int vv = tid % VT;          // this thread's 16-B vector of the row
  const int r0 = tid / VT;
  float acc[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[g][e] = 0.0f;
  for (int t = r0; t < T.n_tok; t += VG) {
    const AttnTok tk = tok_s[t];
    const bool from_cache = (tk.flags & kAttnFromCache) != 0;
    const uint8_t* base = from_cache ? P.v_cache + layer * P.cache_layer_stride
                                     : P.v_pool + layer * P.pool_layer_stride;
    const uint4 x = *reinterpret_cast<const uint4*>(base + static_cast<int64_t>(tk.row) * P.row_bytes +
                                                    h * (D * 2) + vv * 16);
    float xv[8];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      xv[2 * w] = bf_lo(vword(x, w));
      xv[2 * w + 1] = bf_hi(vword(x, w));
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float pt = p_s[t][g];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[g][e] += pt * xv[e];
    }
  }
  // reduce the VG row groups: lanes of a warp that hold the same vector by
  // shuffles (every lane takes part), then the warps through shared memory
#pragma unroll
  for (int o = VT; o < 32; o <<= 1)
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[g][e] += __shfl_xor_sync(0xffffffffu, acc[g][e], o);
  const int lane = tid & 31, warp = tid >> 5;
  if (lane < VT) {
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < 8; ++e) part[warp][g][vv * 8 + e] = acc[g][e];
  }
  __syncthreads();
  // partial record: [layer][tile][h][g] -> (m, l, acc[D])
  float* out = P.partial + ((static_cast<int64_t>(blockIdx.z) * gridDim.x + tile) * gridDim.y + h) *
                               static_cast<int64_t>(G) * (D + 2);
  for (int i = tid; i < G * D; i += kAttnThreads) {
    const int g = i / D, d = i % D;
    float sum = 0.0f;
#pragma unroll
    for (int w = 0; w < kAttnThreads / 32; ++w) sum += part[w][g][d];
    out[g * (D + 2) + 2 + d] = sum;
  }
  if (tid == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      out[g * (D + 2)] = m_g[g];
      out[g * (D + 2) + 1] = l_g[g];
    }
  }
}

// One thread block per (request, query head, layer): merges its tiles.
template <int D>
__global__ void __launch_bounds__(128) k_attend_combine(const AttnParams P, int group) {
  const int r = blockIdx.x, gq = blockIdx.y, lz = blockIdx.z;
  const int h = gq / group, g = gq % group;
  const int t0 = P.req_tile_begin[r], t1 = P.req_tile_begin[r + 1];
  __shared__ float w_s[kAttnMaxCombine];
  __shared__ float tot_s;
  const int64_t stride_tile = static_cast<int64_t>(P.n_kv_heads) * group * (D + 2);
  const float* base = P.partial + static_cast<int64_t>(lz) * P.n_tiles * stride_tile +
                      static_cast<int64_t>(h) * group * (D + 2) + static_cast<int64_t>(g) * (D + 2);
  float M = -FLT_MAX;
  for (int t = t0; t < t1; ++t) M = fmaxf(M, base[t * stride_tile]);
  if (threadIdx.x == 0) {
    float tot = 0.0f;
    for (int t = t0; t < t1; ++t) {
      const float w = __expf(base[t * stride_tile] - M);
      if (t - t0 < kAttnMaxCombine) w_s[t - t0] = w;
      tot += w * base[t * stride_tile + 1];
    }
    tot_s = tot;
  }
  __syncthreads();
  const float tot = tot_s;
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float s = 0.0f;
    for (int t = t0; t < t1; ++t) {
      const float w = (t - t0 < kAttnMaxCombine) ? w_s[t - t0] : __expf(base[t * stride_tile] - M);
      s += w * base[t * stride_tile + 2 + d];
    }
    P.out[((static_cast<int64_t>(lz) * P.n_req + r) * P.num_q_heads + gq) * D + d] = s / tot;
  }
  if (threadIdx.x == 0 && P.lse != nullptr)
    P.lse[(static_cast<int64_t>(lz) * P.n_req + r) * P.num_q_heads + gq] = M + logf(tot);
}

template <int PAIRING, int D, int G>
cudaError_t launch_tiles(const AttnParams& p, cudaStream_t s) {
  k_attend_tiles<PAIRING, D, G><<<dim3(p.n_tiles, p.n_kv_heads, p.n_layers), kAttnThreads, 0, s>>>(p);
  return cudaGetLastError();
}

template <int PAIRING, int D>
cudaError_t launch_for_d(const AttnParams& p, int group, cudaStream_t s) {
  cudaError_t e;
  switch (group) {
    case 1: e = launch_tiles<PAIRING, D, 1>(p, s); break;
    case 2: e = launch_tiles<PAIRING, D, 2>(p, s); break;
    case 4: e = launch_tiles<PAIRING, D, 4>(p, s); break;
    case 8: e = launch_tiles<PAIRING, D, 8>(p, s); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  k_attend_combine<D><<<dim3(p.n_req, p.num_q_heads, p.n_layers), 128, 0, s>>>(p, group);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attend(const AttnParams& p, int pairing, int head_dim, int group, cudaStream_t s) {
  if (p.n_tiles <= 0 || p.n_layers <= 0) return cudaSuccess;
  if (pairing == kNeox) {
    if (head_dim == 64) return launch_for_d<kNeox, 64>(p, group, s);
    if (head_dim == 128) return launch_for_d<kNeox, 128>(p, group, s);
  } else {
    if (head_dim == 64) return launch_for_d<kInterleaved, 64>(p, group, s);
    if (head_dim == 128) return launch_for_d<kInterleaved, 128>(p, group, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pic
