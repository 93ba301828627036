// Content-defined chunking of token documents, and chunk fingerprints, on the GPU.
//
// Irminsul: MLA-Native Position-Independent Caching for Agentic LLM Serving,
// 2.2 "Content-Hash Keying with CDC": chunk boundaries come from a rolling
// Gear hash over 64-token windows, a chunk ends where the hash falls below a
// threshold, and every chunk is keyed by its xxHash64 fingerprint; "Hybrid
// Strategies (S1/S2)", S1: a chunk that misses the registry is subdivided
// into fixed 128-token windows.
//
// What is computed (the page fixes the window, the cut rule and the hash
// family; the arithmetic below is the plain reading of it):
//   h_i = 2 h_{i-1} + gear[t_i] (mod 2^64), with h = 0 before a document's
//   first token, i.e. h_i = sum_{k=0}^{63} gear[t_{i-k}] 2^k over tokens of
//   the same document: a 64-bit Gear hash forgets what lies 64 tokens back.
//   A chunk ends after token i when h_i < threshold (with min_len: only once
//   the chunk holds min_len tokens; with max_len: always once it holds
//   max_len); the tail of a document is a chunk.
//   fingerprint = XXH64(the chunk's token ids as little-endian int32 bytes),
//   following the published XXH64 specification (four accumulators over
//   32-byte stripes, lane merge, length, 8- and 4-byte tails, avalanche).
//
// Launches (one call of pic_cdc_chunk, all on the caller's stream):
//   k_cdc_docs   checks the document offsets; for every 8192-token tile finds
//                the first document boundary its hash window can see.
//   k_cdc_hash   one CTA per tile: token ids by 16-byte loads, one Gear
//                gather per token, every position's hash, one cut bit each,
//                and the tile's cut count.
//   k_cdc_walk   (min_len > 1 or max_len > 0 only) one warp per document
//                walks its cut candidates and applies the length rules; then
//                k_cdc_tile_count recounts the tiles.
//   k_cdc_scan   one CTA: tile counts -> each tile's first chunk index.
//   k_cdc_emit   one CTA per tile: chunk ends, numbered in position order,
//                and the CSR offset of every document starting in the tile.
//   k_xxh64      four lanes per chunk: XXH64 of the chunk's token bytes.
// Documents are contiguous and each one's last token ends a chunk, so chunks
// numbered in position order are in document order, document d's first
// chunk index is the number of cuts before offsets[d], and chunk c starts
// where chunk c - 1 ends (chunk 0 at offsets[0]).
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstdio>

#include "pic.h"
#include "pic_internal.h"

namespace pic {
namespace {

constexpr int kHashThreads = 256;
constexpr int kTile = kHashThreads * 32;         // tokens per tile: one 32-bit cut word per thread
constexpr int kTileWords = kTile / 32;
constexpr int kHalo = 64;                        // the hash window reaches 63 tokens back
constexpr int kTokPad = kTile + kTile / 32;      // one pad word per 32 tokens: conflict-free row reads
constexpr int kBndWords = (kHalo + kTile + 64) / 32;  // boundary bits over [t0 - 64, t0 + kTile + 64)
constexpr int kWarpThreads = 256;                // CTA size of the per-document kernels
constexpr int kScanThreads = 1024;
constexpr int kScanPerThread = 4;
constexpr int kXxhThreads = 256;
constexpr unsigned kFull = 0xffffffffu;

// XXH64 primes (published specification).
constexpr uint64_t kP1 = 0x9E3779B185EBCA87ull;
constexpr uint64_t kP2 = 0xC2B2AE3D27D4EB4Full;
constexpr uint64_t kP3 = 0x165667B19E3779F9ull;
constexpr uint64_t kP4 = 0x85EBCA77C2B2AE63ull;
constexpr uint64_t kP5 = 0x27D4EB2F165667C5ull;

struct CdcLayout {
  size_t first_doc;   // int32 per tile
  size_t tile_count;  // int64 per tile + 1: cut counts, then each tile's first chunk index and the total
  size_t bits;        // uint32 cut words, kTileWords per tile
  size_t total;
};

CdcLayout cdc_layout(int64_t n_tokens) {
  const int64_t n_tiles = (n_tokens + kTile - 1) / kTile;
  CdcLayout l;
  l.first_doc = kWsAlign;
  l.tile_count = l.first_doc + align_up(static_cast<size_t>(n_tiles) * 4, kWsAlign);
  l.bits = l.tile_count + align_up(static_cast<size_t>(n_tiles + 1) * 8, kWsAlign);
  l.total = l.bits + align_up(static_cast<size_t>(n_tiles) * kTileWords * 4, kWsAlign);
  return l;
}

__device__ __forceinline__ uint64_t rotl64(uint64_t x, int r) { return (x << r) | (x >> (64 - r)); }

__device__ __forceinline__ uint64_t xxh_round(uint64_t acc, uint64_t lane) {
  acc += lane * kP2;
  acc = rotl64(acc, 31);
  return acc * kP1;
}

__device__ __forceinline__ uint64_t xxh_merge(uint64_t acc, uint64_t v) {
  acc ^= xxh_round(0, v);
  return acc * kP1 + kP4;
}

// Bits of cut word w (positions [32w, 32w + 32)) that lie inside [lo, hi).
__device__ __forceinline__ uint32_t word_mask(int64_t w, int64_t lo, int64_t hi) {
  const int64_t base = w << 5;
  const int64_t a = lo > base ? lo - base : 0;
  const int64_t b = hi - base < 32 ? hi - base : 32;
  if (b <= a) return 0u;
  const uint32_t upto = b == 32 ? kFull : ((1u << b) - 1u);
  return upto & ~((1u << a) - 1u);
}

// The kernels of one call run back to back: each after the first is
// launched as a programmatic dependent of the one before it.  A kernel lets
// the next be scheduled once all its CTAs run, and waits for the previous
// kernel's completion (and memory) before it reads anything.
__device__ __forceinline__ void after_previous_kernel() {
  asm volatile("griddepcontrol.launch_dependents;");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ bool docs_bad(const WsHeader* h) {
  return (*reinterpret_cast<const volatile uint32_t*>(&h->status) & PIC_DEV_BAD_DOCS) != 0;
}

// ---------------------------------------------------------------- offsets

// Document d covers tokens [offsets[d], offsets[d + 1]).  Checks that the
// offsets are non-decreasing inside [0, n_tokens], and records for every tile
// k the first document index whose start is >= k * kTile - kHalo (the first
// boundary the tile's hash window can meet).  Index d in [0, n_docs + 1]
// owns the tiles whose window start falls in (offsets[d - 1], offsets[d]],
// with offsets[-1] = -inf and offsets[n_docs + 1] = +inf.
__global__ void k_cdc_docs(const int64_t* __restrict__ offsets, int32_t n_docs, int64_t n_tokens,
                           int32_t* __restrict__ first_doc, int64_t* __restrict__ tile_count, int64_t n_tiles,
                           WsHeader* hdr) {
  asm volatile("griddepcontrol.launch_dependents;");  // the hash pass may be scheduled from now on
  const int64_t n = static_cast<int64_t>(n_docs) + 2;
  for (int64_t d = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; d < n;
       d += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    int64_t cur = d <= n_docs ? offsets[d] : INT64_MAX;
    int64_t prev = d > 0 ? offsets[d - 1] : INT64_MIN;
    if (d <= n_docs && (cur < 0 || cur > n_tokens || (d > 0 && cur < prev)))
      atomicOr(&hdr->status, PIC_DEV_BAD_DOCS);
    // clamp so the tile arithmetic below cannot overflow (bad offsets only)
    cur = cur < -1 ? -1 : (cur > n_tokens + 1 ? n_tokens + 1 : cur);
    prev = prev < -kHalo - 1 ? -kHalo - 1 : (prev > n_tokens + 1 ? n_tokens + 1 : prev);
    // tiles k with prev < k*kTile - kHalo <= cur
    int64_t k_lo = d == 0 ? 0 : (prev + kHalo) / kTile + 1;   // prev + kHalo >= -1: floor is fine for >= 0
    if (d > 0 && prev + kHalo < 0) k_lo = 0;
    int64_t k_hi = d == n_docs + 1 ? n_tiles - 1 : (cur + kHalo) / kTile;
    if (k_hi > n_tiles - 1) k_hi = n_tiles - 1;
    for (int64_t k = k_lo; k <= k_hi; ++k) {
      first_doc[k] = static_cast<int32_t>(d);
      tile_count[k] = 0;
    }
  }
}

// ---------------------------------------------------------------- hash

// Gear hash and cut candidates of one tile per iteration.  Thread j owns the
// 32 positions [t0 + 32j, t0 + 32j + 32) and writes their cut word.
//
// Block decomposition of the rolling hash: let B_j be the hash after thread
// j's 32 positions starting from 0 (reset at a document start inside them),
// and R_j the true hash at the block's last position.  As 2^64 = 0 mod 2^64,
// R_{j-1} = B_{j-1} + (no document start in block j-1 ? B_{j-2} << 32 : 0),
// so every thread starts from the exact hash after reading only two partial
// sums: the serial recurrence runs over 32 positions per thread, not 95.
__global__ void __launch_bounds__(kHashThreads, 2)
k_cdc_hash(const int32_t* __restrict__ tokens, int64_t n_tokens, const int64_t* __restrict__ offsets,
           int32_t n_docs, const uint64_t* __restrict__ gear, uint32_t vocab, uint64_t threshold,
           const int32_t* __restrict__ first_doc, uint32_t* __restrict__ bits,
           unsigned long long* __restrict__ tile_count, int64_t n_tiles, WsHeader* hdr) {
  __shared__ int32_t s_tok[kTokPad];
  __shared__ uint32_t s_bnd[kBndWords];
  __shared__ uint64_t s_part[kHashThreads + 2];  // B_j at index j + 2; halo blocks -2, -1 at 0, 1

  after_previous_kernel();
  if (docs_bad(hdr)) return;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int64_t in_lo = offsets[0];
  const int64_t in_hi = offsets[n_docs];
  bool bad_token = false;

  for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const int64_t t0 = tile * kTile;
    const int64_t r0 = t0 - kHalo;  // position of boundary bit 0
    __syncthreads();                // the previous tile is done with shared memory
    for (int i = tid; i < kBndWords; i += kHashThreads) s_bnd[i] = 0u;

    // token ids of the tile: 16-byte loads, all issued before use
    int4 v[kTile / 4 / kHashThreads];
#pragma unroll
    for (int k = 0; k < kTile / 4 / kHashThreads; ++k) {
      const int64_t p = t0 + 4 * (k * kHashThreads + tid);
      if (p + 4 <= n_tokens) {
        v[k] = __ldcs(reinterpret_cast<const int4*>(tokens + p));
      } else {
        v[k].x = p < n_tokens ? tokens[p] : 0;
        v[k].y = p + 1 < n_tokens ? tokens[p + 1] : 0;
        v[k].z = p + 2 < n_tokens ? tokens[p + 2] : 0;
        v[k].w = p + 3 < n_tokens ? tokens[p + 3] : 0;
      }
    }
    __syncthreads();  // s_bnd cleared
    // document boundaries the tile can see: offsets in [t0 - 64, t0 + kTile + 64)
    for (int64_t d = first_doc[tile] + static_cast<int64_t>(tid); d <= n_docs; d += kHashThreads) {
      const int64_t o = offsets[d];
      if (o >= r0 + 32 * kBndWords) break;  // offsets are non-decreasing
      const int64_t r = o - r0;
      atomicOr(&s_bnd[r >> 5], 1u << (r & 31));
    }
#pragma unroll
    for (int k = 0; k < kTile / 4 / kHashThreads; ++k) {
      const int t = 4 * (k * kHashThreads + tid);
      const int q = t + (t >> 5);
      s_tok[q] = v[k].x;
      s_tok[q + 1] = v[k].y;
      s_tok[q + 2] = v[k].z;
      s_tok[q + 3] = v[k].w;
    }
    __syncthreads();  // s_tok, s_bnd complete

    // own 32 Gear values
    const int64_t p0 = t0 + 32 * static_cast<int64_t>(tid);
    uint64_t g[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const uint32_t tk = static_cast<uint32_t>(s_tok[33 * tid + i]);
      const int64_t p = p0 + i;
      const bool in = p >= in_lo && p < in_hi;
      bad_token |= in && tk >= vocab;
      g[i] = (in && tk < vocab) ? __ldg(gear + tk) : 0ull;
    }
    const uint32_t bw = s_bnd[tid + 2];  // document starts inside this block
    {
      const int lb = bw ? 31 - __clz(bw) : 0;
      uint64_t part = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) part += (i >= lb) ? (g[i] << (31 - i)) : 0ull;
      s_part[tid + 2] = part;
    }
    if (tid < 32) {
      // halo blocks -2 and -1: the 64 tokens before the tile, one per lane each
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const int64_t p = t0 - kHalo + 32 * b + lane;
        uint64_t gv = 0;
        if (p >= in_lo && p < in_hi) {
          const uint32_t tk = static_cast<uint32_t>(tokens[p]);
          if (tk < vocab) gv = __ldg(gear + tk);
        }
        const uint32_t hb = s_bnd[b];
        const int lb = hb ? 31 - __clz(hb) : 0;
        uint64_t c = lane >= lb ? (gv << (31 - lane)) : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(kFull, c, o);
        if (lane == 0) s_part[b] = c;
      }
    }
    __syncthreads();  // every partial sum is in

    // exact hash entering the block, then the 32 positions
    uint64_t h = s_part[tid + 1] + (s_bnd[tid + 1] == 0u ? (s_part[tid] << 32) : 0ull);
    uint32_t cut = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if ((bw >> i) & 1u) h = 0;
      h = 2 * h + g[i];
      cut |= (h < threshold ? 1u : 0u) << i;
    }
    // the last token of a document ends a chunk: p + 1 is a document boundary
    const uint32_t ends = (bw >> 1) | ((s_bnd[tid + 3] & 1u) << 31);
    // positions inside [in_lo, in_hi)
    const int64_t a = in_lo - p0 < 0 ? 0 : (in_lo - p0 > 32 ? 32 : in_lo - p0);
    const int64_t b = in_hi - p0 < 0 ? 0 : (in_hi - p0 > 32 ? 32 : in_hi - p0);
    uint32_t inside = 0;
    if (b > a) inside = (b == 32 ? kFull : ((1u << b) - 1u)) & ~((1u << a) - 1u);
    const uint32_t word = (cut | ends) & inside;
    bits[tile * kTileWords + tid] = word;
    const unsigned n_cut = __reduce_add_sync(kFull, static_cast<unsigned>(__popc(word)));
    if (lane == 0 && n_cut) atomicAdd(&tile_count[tile], static_cast<unsigned long long>(n_cut));
  }
  if (__syncthreads_or(bad_token) && tid == 0) atomicOr(&hdr->status, PIC_DEV_BAD_TOKEN);
}

// ---------------------------------------------------------------- length rules

// One warp per document: applies min_len / max_len along the document.  The
// cut after token i is the first i >= start with (i >= start + max_len - 1) or
// (i is a hash candidate and i >= start + max(min_len, 1) - 1); the document's
// last token always ends a chunk.  The document's cut bits are rewritten; a
// word shared with a neighbouring document is updated with atomics restricted
// to this document's bits.
__global__ void __launch_bounds__(kWarpThreads)
k_cdc_walk(const int64_t* __restrict__ offsets, int32_t n_docs, uint32_t* bits, int32_t min_len,
           int32_t max_len, const WsHeader* hdr) {
  after_previous_kernel();
  if (docs_bad(hdr)) return;
  const int lane = threadIdx.x & 31;
  const int64_t warp = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t lo_len = min_len > 1 ? min_len : 1;
  for (int64_t d = warp; d < n_docs; d += n_warps) {
    const int64_t ds = offsets[d], de = offsets[d + 1];
    if (ds >= de) continue;
    int64_t start = ds;
    const int64_t w_last = (de - 1) >> 5;
    for (int64_t wb = ds >> 5; wb <= w_last; wb += 32) {
      const int64_t w = wb + lane;
      const bool have = w <= w_last;
      const uint32_t dmask = have ? word_mask(w, ds, de) : 0u;
      const uint32_t cand = have ? (bits[w] & dmask) : 0u;
      const int64_t win_end = (wb + 32) << 5;
      uint32_t fin = 0;
      while (start < de) {
        const int64_t lo = start + lo_len - 1;
        int64_t hi = de - 1;
        if (max_len > 0 && start + max_len - 1 < hi) hi = start + max_len - 1;
        const uint32_t m = cand & word_mask(w, lo, INT64_MAX);
        const uint32_t any = __ballot_sync(kFull, m != 0u);
        int64_t c = INT64_MAX;
        if (any) {
          const int f = __ffs(any) - 1;
          const uint32_t mf = __shfl_sync(kFull, m, f);
          c = ((wb + f) << 5) + (__ffs(mf) - 1);
        }
        int64_t cutpos;
        if (c <= hi) cutpos = c;
        else if (hi < win_end) cutpos = hi;
        else break;  // the next cut lies past this window
        if (w == (cutpos >> 5)) fin |= 1u << (cutpos & 31);
        start = cutpos + 1;
      }
      if (have) {
        if (dmask == kFull) {
          bits[w] = fin;
        } else {
          atomicOr(&bits[w], fin);
          atomicAnd(&bits[w], fin | ~dmask);
        }
      }
    }
  }
}

// ---------------------------------------------------------------- counts, scan

// One warp per tile: its cut count (after the length rules rewrote the bits).
__global__ void __launch_bounds__(kWarpThreads)
k_cdc_tile_count(const uint32_t* __restrict__ bits, int64_t* __restrict__ tile_count, int64_t n_tiles,
                 const WsHeader* hdr) {
  after_previous_kernel();
  if (docs_bad(hdr)) return;
  const int lane = threadIdx.x & 31;
  const int64_t warp = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t t = warp; t < n_tiles; t += n_warps) {
    unsigned c = 0;
#pragma unroll
    for (int k = 0; k < kTileWords / 32; ++k) c += __popc(bits[t * kTileWords + k * 32 + lane]);
    c = __reduce_add_sync(kFull, c);
    if (lane == 0) tile_count[t] = c;
  }
}

// Single CTA: tile_count[k] holds tile k's cut count on entry and the number
// of cuts before tile k on exit; tile_count[n_tiles] receives the total.
// With bad offsets it writes indptr = 0 instead; with no tiles (no tokens)
// every offset is 0 and so is every indptr entry.
__global__ void __launch_bounds__(kScanThreads)
k_cdc_scan(int64_t* __restrict__ tile_count, int64_t n_tiles, int64_t* __restrict__ indptr, int32_t n_docs,
           int64_t capacity, WsHeader* hdr) {
  __shared__ int64_t s_warp[kScanThreads / 32];
  __shared__ int64_t s_carry;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  after_previous_kernel();
  if (docs_bad(hdr) || n_tiles == 0) {
    for (int64_t d = tid; d <= n_docs; d += kScanThreads) indptr[d] = 0;
    return;
  }
  if (tid == 0) s_carry = 0;
  __syncthreads();
  for (int64_t base = 0; base < n_tiles; base += kScanThreads * kScanPerThread) {
    int64_t v[kScanPerThread];
    int64_t sum = 0;
#pragma unroll
    for (int k = 0; k < kScanPerThread; ++k) {
      const int64_t i = base + tid * kScanPerThread + k;
      v[k] = i < n_tiles ? tile_count[i] : 0;
      sum += v[k];
    }
    int64_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t t = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) s_warp[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      int64_t x = s_warp[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t t = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += t;
      }
      s_warp[lane] = x;  // inclusive over warps
    }
    __syncthreads();
    int64_t run = s_carry + (wid > 0 ? s_warp[wid - 1] : 0) + incl - sum;
#pragma unroll
    for (int k = 0; k < kScanPerThread; ++k) {
      const int64_t i = base + tid * kScanPerThread + k;
      if (i < n_tiles) tile_count[i] = run;
      run += v[k];
    }
    __syncthreads();
    if (tid == 0) s_carry += s_warp[kScanThreads / 32 - 1];
    __syncthreads();
  }
  if (tid == 0) {
    tile_count[n_tiles] = s_carry;
    if (s_carry > capacity) atomicOr(&hdr->status, PIC_DEV_CAPACITY);
  }
}

// ---------------------------------------------------------------- emission

// One CTA per tile, one thread per cut word.  Chunk index = cuts before the
// tile + rank inside it; ends[index] = one past the cut token.  Every document
// offset inside the tile (offsets[n_docs] included) gets indptr = the number
// of cuts before it.  Nothing at or past `capacity` is written to ends.
__global__ void __launch_bounds__(kHashThreads)
k_cdc_emit(const int64_t* __restrict__ offsets, int32_t n_docs, const uint32_t* __restrict__ bits,
           const int64_t* __restrict__ tile_first, const int32_t* __restrict__ first_doc, int64_t n_tiles,
           int64_t* __restrict__ ends, int64_t capacity, int64_t* __restrict__ indptr, const WsHeader* hdr) {
  __shared__ int32_t s_warp[kHashThreads / 32];
  __shared__ int32_t s_pref[kTileWords];
  __shared__ uint32_t s_word[kTileWords];
  after_previous_kernel();
  if (docs_bad(hdr)) return;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const int64_t t0 = tile * kTile;
    const uint32_t word = bits[tile * kTileWords + tid];
    const int n = __popc(word);
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += t;
    }
    __syncthreads();  // the previous tile is done with shared memory
    if (lane == 31) s_warp[wid] = incl;
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int k = 0; k < kHashThreads / 32; ++k) {
      const int c = s_warp[k];
      before += k < wid ? c : 0;
      total += c;
    }
    const int excl = before + incl - n;
    s_pref[tid] = excl;
    s_word[tid] = word;
    const int64_t base = tile_first[tile];
    int64_t idx = base + excl;
    uint32_t m = word;
    while (m) {
      const int b = __ffs(m) - 1;
      m &= m - 1u;
      if (idx < capacity) ends[idx] = t0 + 32 * tid + b + 1;
      ++idx;
    }
    __syncthreads();  // s_pref, s_word complete
    const bool last = tile == n_tiles - 1;
    for (int64_t d = static_cast<int64_t>(first_doc[tile]) + tid; d <= n_docs; d += kHashThreads) {
      const int64_t o = offsets[d];
      if (o < t0) continue;  // seen by the tile's hash window, but lies in the tile before
      if (o >= t0 + kTile) {
        if (!last) break;    // offsets are non-decreasing
        indptr[d] = base + total;  // o == n_tokens at the end of the last tile
        continue;
      }
      const int r = static_cast<int>(o - t0);
      const int w = r >> 5, bit = r & 31;
      indptr[d] = base + s_pref[w] + __popc(s_word[w] & ((1u << bit) - 1u));
    }
  }
}

// ---------------------------------------------------------------- XXH64

// XXH64 of spans of token ids, in two phases per CTA batch of spans:
//   A: a 4-lane group runs the four stripe accumulators of one span (lane j
//      takes bytes 8j .. 8j + 7 of every 32-byte stripe) and parks them in
//      shared memory; groups take the batch's spans from a shared counter, so
//      long and short spans keep every group busy.
//   B: one thread per span merges the accumulators, hashes the tail (at most
//      seven tokens), adds the length and applies the avalanche.
// Every lane of phase B runs the same code, so the serial finishing steps do
// not leave three of four lanes idle.  Each CTA owns a contiguous range of
// spans.
//   starts == nullptr: span c starts where span c - 1 ends (span 0 at
//   *first_start): the chunks of pic_cdc_chunk.
//   n_dev != nullptr: the span count is *n_dev, clamped to cap.
constexpr int kXxhBatch = 1024;             // spans per CTA batch
constexpr int kXxhGroups = kXxhThreads / 4; // 4-lane groups per CTA
constexpr int kXxhU = 8;                    // stripes per group step

struct SpanInfo {
  const int32_t* p;
  int64_t ntok;
  bool bad;
};

__device__ __forceinline__ SpanInfo span_info(const int32_t* tokens, int64_t n_tokens, const int64_t* starts,
                                              const int64_t* first_start, const int64_t* ends, int64_t c) {
  const int64_t e = ends[c];
  const int64_t s = starts ? starts[c] : (c > 0 ? ends[c - 1] : *first_start);
  SpanInfo r;
  r.bad = s < 0 || e < s || e > n_tokens;
  r.ntok = r.bad ? 0 : e - s;
  r.p = tokens + (r.bad ? 0 : s);
  return r;
}

__global__ void __launch_bounds__(kXxhThreads)
k_xxh64(const int32_t* __restrict__ tokens, int64_t n_tokens, const int64_t* __restrict__ starts,
        const int64_t* __restrict__ first_start, const int64_t* __restrict__ ends,
        const int64_t* __restrict__ n_dev, int64_t n_host, int64_t cap, uint64_t seed, uint64_t* __restrict__ out,
        uint32_t* status, const WsHeader* hdr) {
  __shared__ uint64_t s_acc[4][kXxhBatch];
  __shared__ int s_next;
  after_previous_kernel();
  if (hdr && docs_bad(hdr)) return;
  int64_t n = n_host;
  if (n_dev) {
    n = *n_dev;
    if (n > cap) n = cap;
  }
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int j = lane & 3;
  const int g0 = lane & ~3;
  const unsigned gmask = 0xfu << g0;
  uint64_t v_init = seed;
  if (j == 0) v_init = seed + kP1 + kP2;
  else if (j == 1) v_init = seed + kP2;
  else if (j == 3) v_init = seed - kP1;
  const int64_t c_lo = n * blockIdx.x / gridDim.x, c_hi = n * (blockIdx.x + 1) / gridDim.x;

  for (int64_t b0 = c_lo; b0 < c_hi; b0 += kXxhBatch) {
    const int nb = static_cast<int>(c_hi - b0 < kXxhBatch ? c_hi - b0 : kXxhBatch);
    if (tid == 0) s_next = kXxhGroups;
    __syncthreads();
    // phase A: stripes.  One flat loop: every iteration advances each group's
    // span by up to kXxhU stripes; a group whose span is done parks its
    // accumulators and takes the next span in the same iteration, so the
    // warp never waits at a loop exit for its longest span.
    int k = tid >> 2;
    const int32_t* q = tokens;
    int64_t left = 0;  // stripes still to run on span k
    uint64_t v = v_init;
    if (k < nb) {
      const SpanInfo sp = span_info(tokens, n_tokens, starts, first_start, ends, b0 + k);
      left = sp.ntok >> 3;  // 32 bytes = 8 tokens
      q = sp.p + 2 * j;
    }
    while (__any_sync(kFull, k < nb)) {
      if (k < nb && left > 0) {
        const int m = left < kXxhU ? static_cast<int>(left) : kXxhU;
        uint32_t lo[kXxhU], hi[kXxhU];
#pragma unroll
        for (int u = 0; u < kXxhU; ++u) {
          lo[u] = 0u;
          hi[u] = 0u;
          if (u < m) {
            lo[u] = static_cast<uint32_t>(__ldg(q + 8 * u));
            hi[u] = static_cast<uint32_t>(__ldg(q + 8 * u + 1));
          }
        }
#pragma unroll
        for (int u = 0; u < kXxhU; ++u)
          if (u < m) v = xxh_round(v, lo[u] | (static_cast<uint64_t>(hi[u]) << 32));
        left -= m;
        q += 8 * m;
      }
      if (k < nb && left == 0) {
        s_acc[j][k] = v;
        int nk = 0;
        if (j == 0) nk = atomicAdd(&s_next, 1);
        k = __shfl_sync(gmask, nk, g0);
        v = v_init;
        if (k < nb) {
          const SpanInfo sp = span_info(tokens, n_tokens, starts, first_start, ends, b0 + k);
          left = sp.ntok >> 3;
          q = sp.p + 2 * j;
        }
      }
    }
    __syncthreads();
    // phase B: one thread per span
    for (int k = tid; k < nb; k += kXxhThreads) {
      const int64_t c = b0 + k;
      const SpanInfo sp = span_info(tokens, n_tokens, starts, first_start, ends, c);
      const int64_t stripes = sp.ntok >> 3;
      uint64_t acc;
      if (stripes > 0) {
        const uint64_t v1 = s_acc[0][k], v2 = s_acc[1][k], v3 = s_acc[2][k], v4 = s_acc[3][k];
        acc = rotl64(v1, 1) + rotl64(v2, 7) + rotl64(v3, 12) + rotl64(v4, 18);
        acc = xxh_merge(acc, v1);
        acc = xxh_merge(acc, v2);
        acc = xxh_merge(acc, v3);
        acc = xxh_merge(acc, v4);
      } else {
        acc = seed + kP5;
      }
      acc += static_cast<uint64_t>(sp.ntok) * 4u;
      int64_t t = stripes << 3;
      for (; t + 2 <= sp.ntok; t += 2) {
        const uint64_t w = static_cast<uint32_t>(__ldg(sp.p + t)) |
                           (static_cast<uint64_t>(static_cast<uint32_t>(__ldg(sp.p + t + 1))) << 32);
        acc ^= xxh_round(0, w);
        acc = rotl64(acc, 27) * kP1 + kP4;
      }
      if (t < sp.ntok) {
        acc ^= static_cast<uint64_t>(static_cast<uint32_t>(__ldg(sp.p + t))) * kP1;
        acc = rotl64(acc, 23) * kP2 + kP3;
      }
      acc ^= acc >> 33;
      acc *= kP2;
      acc ^= acc >> 29;
      acc *= kP3;
      acc ^= acc >> 32;
      if (sp.bad) {
        acc = 0;
        atomicOr(status, PIC_DEV_BAD_SPAN);
      }
      out[c] = acc;
    }
    __syncthreads();  // the next batch reuses s_acc and s_next
  }
}

// ---------------------------------------------------------------- host side

// A kernel launched as a programmatic dependent of the previous one on the
// stream (see after_previous_kernel).
template <typename... KArgs, typename... Args>
cudaError_t launch_after(void (*kern)(KArgs...), int grid, int block, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
  return n;
}

pic_status arg_error(pic_status st, const char* msg) { return set_error(nullptr, st, msg); }

pic_status cuda_error(cudaError_t e, const char* what) {
  char msg[256];
  std::snprintf(msg, sizeof(msg), "%s: %s", what, cudaGetErrorString(e));
  return set_error(nullptr, PIC_ERR_CUDA, msg);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int warp_grid(int64_t n_docs, int sms) {
  const int64_t warps_per_cta = kWarpThreads / 32;
  int64_t g = (n_docs + warps_per_cta - 1) / warps_per_cta;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  if (g > cap) g = cap;
  return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace
}  // namespace pic

using namespace pic;

extern "C" size_t pic_cdc_workspace_bytes(int64_t n_tokens) {
  if (n_tokens < 0) return 0;
  return cdc_layout(n_tokens).total;
}

extern "C" pic_status pic_cdc_chunk(const int32_t* d_tokens, int64_t n_tokens, const int64_t* d_doc_offsets,
                                    int32_t n_docs, const uint64_t* d_gear, int32_t vocab, uint64_t threshold,
                                    int32_t min_len, int32_t max_len, uint64_t seed, int64_t* d_chunk_indptr,
                                    int64_t* d_chunk_ends, uint64_t* d_fingerprints, int64_t capacity,
                                    void* d_workspace, size_t workspace_bytes, pic_stream_t stream) {
  if (n_tokens < 0 || n_docs < 0 || capacity < 0 || min_len < 0 || max_len < 0)
    return arg_error(PIC_ERR_INVALID_ARG, "negative size, length rule or capacity");
  if (!d_doc_offsets || !d_chunk_indptr || !d_workspace)
    return arg_error(PIC_ERR_INVALID_ARG, "null document offsets, chunk indptr or workspace");
  if (n_tokens > 0 && (!d_tokens || !d_gear || vocab <= 0))
    return arg_error(PIC_ERR_INVALID_ARG, "tokens need a token buffer and a Gear table of vocab >= 1 entries");
  if (capacity > 0 && !d_chunk_ends) return arg_error(PIC_ERR_INVALID_ARG, "null chunk ends with capacity > 0");
  if (!aligned(d_tokens, 16) || !aligned(d_doc_offsets, 8) || !aligned(d_gear, 8) ||
      !aligned(d_chunk_indptr, 8) || !aligned(d_chunk_ends, 8) || !aligned(d_fingerprints, 8) ||
      !aligned(d_workspace, kWsAlign))
    return arg_error(PIC_ERR_ALIGNMENT,
                     "tokens must be 16-byte aligned, offsets/Gear/outputs 8-byte, the workspace 256-byte");
  const CdcLayout lay = cdc_layout(n_tokens);
  if (workspace_bytes < lay.total) return arg_error(PIC_ERR_CAPACITY, "workspace smaller than pic_cdc_workspace_bytes");

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(d_workspace);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  int32_t* first_doc = reinterpret_cast<int32_t*>(ws + lay.first_doc);
  int64_t* tile_count = reinterpret_cast<int64_t*>(ws + lay.tile_count);
  uint32_t* bits = reinterpret_cast<uint32_t*>(ws + lay.bits);
  const int64_t n_tiles = (n_tokens + kTile - 1) / kTile;
  const int sms = sm_count();

  cudaError_t e = cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s);
  if (e != cudaSuccess) return cuda_error(e, "status reset");
  {
    const int64_t work = (static_cast<int64_t>(n_docs) + 2 > n_tiles ? static_cast<int64_t>(n_docs) + 2 : n_tiles);
    int64_t grid = (work + 255) / 256;
    if (grid > static_cast<int64_t>(sms) * 4) grid = static_cast<int64_t>(sms) * 4;
    k_cdc_docs<<<static_cast<int>(grid < 1 ? 1 : grid), 256, 0, s>>>(d_doc_offsets, n_docs, n_tokens, first_doc,
                                                                      tile_count, n_tiles, hdr);
  }
  e = cudaGetLastError();
  if (n_tiles > 0 && e == cudaSuccess) {
    const int grid = static_cast<int>(n_tiles < static_cast<int64_t>(sms) * 2 ? n_tiles : static_cast<int64_t>(sms) * 2);
    e = launch_after(k_cdc_hash, grid, kHashThreads, s, d_tokens, n_tokens, d_doc_offsets, n_docs, d_gear,
                     static_cast<uint32_t>(vocab), threshold, static_cast<const int32_t*>(first_doc), bits,
                     reinterpret_cast<unsigned long long*>(tile_count), n_tiles, hdr);
    if (e == cudaSuccess && n_docs > 0 && (min_len > 1 || max_len > 0)) {
      e = launch_after(k_cdc_walk, warp_grid(n_docs, sms), kWarpThreads, s, d_doc_offsets, n_docs, bits, min_len,
                       max_len, static_cast<const WsHeader*>(hdr));
      if (e == cudaSuccess)
        e = launch_after(k_cdc_tile_count, warp_grid(n_tiles, sms), kWarpThreads, s,
                         static_cast<const uint32_t*>(bits), tile_count, n_tiles, static_cast<const WsHeader*>(hdr));
    }
  }
  if (e == cudaSuccess)
    e = launch_after(k_cdc_scan, 1, kScanThreads, s, tile_count, n_tiles, d_chunk_indptr, n_docs, capacity, hdr);
  if (n_tiles > 0 && e == cudaSuccess) {
    const int grid = static_cast<int>(n_tiles < static_cast<int64_t>(sms) * 4 ? n_tiles : static_cast<int64_t>(sms) * 4);
    e = launch_after(k_cdc_emit, grid, kHashThreads, s, d_doc_offsets, n_docs, static_cast<const uint32_t*>(bits),
                     static_cast<const int64_t*>(tile_count), static_cast<const int32_t*>(first_doc), n_tiles,
                     d_chunk_ends, capacity, d_chunk_indptr, static_cast<const WsHeader*>(hdr));
    if (e == cudaSuccess && d_fingerprints && capacity > 0)
      // five CTAs per SM: its 45 registers allow them, and the extra warps hide the rounds' latency
      e = launch_after(k_xxh64, sms * 5, kXxhThreads, s, d_tokens, n_tokens, static_cast<const int64_t*>(nullptr),
                       d_doc_offsets, static_cast<const int64_t*>(d_chunk_ends),
                       static_cast<const int64_t*>(tile_count + n_tiles), static_cast<int64_t>(0), capacity, seed,
                       d_fingerprints, &hdr->status, static_cast<const WsHeader*>(hdr));
  }
  if (e != cudaSuccess) return cuda_error(e, "chunking launch");
  return set_error(nullptr, PIC_OK, "");
}

extern "C" pic_status pic_fingerprint_spans(const int32_t* d_tokens, int64_t n_tokens, const int64_t* d_starts,
                                            const int64_t* d_ends, int64_t n_spans, uint64_t seed,
                                            uint64_t* d_out, uint32_t* d_status, pic_stream_t stream) {
  if (n_tokens < 0 || n_spans < 0) return arg_error(PIC_ERR_INVALID_ARG, "negative size");
  if (n_spans > 0 && (!d_starts || !d_ends || !d_out || !d_status))
    return arg_error(PIC_ERR_INVALID_ARG, "null span, output or status pointer");
  if (n_spans > 0 && n_tokens > 0 && !d_tokens) return arg_error(PIC_ERR_INVALID_ARG, "null token buffer");
  if (!aligned(d_tokens, 4) || !aligned(d_starts, 8) || !aligned(d_ends, 8) || !aligned(d_out, 8) ||
      !aligned(d_status, 4))
    return arg_error(PIC_ERR_ALIGNMENT, "tokens and status must be 4-byte aligned, spans and output 8-byte");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (d_status) {
    cudaError_t e = cudaMemsetAsync(d_status, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess) return cuda_error(e, "status reset");
  }
  if (n_spans == 0) return set_error(nullptr, PIC_OK, "");
  const int sms = sm_count();
  int64_t grid = (n_spans + kXxhBatch - 1) / kXxhBatch;
  if (grid > static_cast<int64_t>(sms) * 4) grid = static_cast<int64_t>(sms) * 4;
  k_xxh64<<<static_cast<int>(grid), kXxhThreads, 0, s>>>(d_tokens, n_tokens, d_starts, nullptr, d_ends, nullptr,
                                                          n_spans, n_spans, seed, d_out, d_status, nullptr);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "fingerprint launch");
  return set_error(nullptr, PIC_OK, "");
}

extern "C" pic_status pic_s1_windows(int64_t begin, int64_t end, int32_t window, int64_t* starts,
                                     int64_t* ends, int64_t capacity, int64_t* count) {
  if (begin < 0 || end < begin || window <= 0 || capacity < 0 || !count)
    return arg_error(PIC_ERR_INVALID_ARG, "need 0 <= begin <= end, window >= 1 and a count pointer");
  const int64_t n = (end - begin + window - 1) / window;
  *count = n;
  if (!starts && !ends) return set_error(nullptr, PIC_OK, "");
  if (n > capacity) return arg_error(PIC_ERR_CAPACITY, "more windows than capacity");
  for (int64_t k = 0; k < n; ++k) {
    const int64_t b = begin + k * window;
    if (starts) starts[k] = b;
    if (ends) ends[k] = b + window < end ? b + window : end;
  }
  return set_error(nullptr, PIC_OK, "");
}
