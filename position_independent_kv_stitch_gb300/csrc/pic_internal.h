// Internal interface between the host library (pic_host.cpp) and the CUDA
// kernels (pic_kernels.cu).  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "pic.h"

namespace pic {

// region stitch-schedule: what the stitch and in-place kernels share with the
// host (a measurement record names this region).

// One run: up to block_size consecutive tokens of one segment that land in
// one paged block.  Runs are layer-independent; a kernel work unit is a run
// times a group of consecutive layers.  32 bytes, read once per unit.
struct alignas(32) RunDesc {
  int32_t src;        // kRunPool: pool token row of the first token; kRunBlocks:
                      // absolute cache row (block * block_size + row); kRunInPlace: unused
  int32_t dst_pos;    // absolute position of the run's first token
  int32_t req;        // block-table row
  int32_t ntok_kind;  // tokens in the run (0 .. block_size, low 16 bits) | kind << 16
  int32_t delta;      // position shift of the segment
  int32_t idx_off;    // first recompute-list slot this run writes
  int32_t idx_count;  // recompute positions it writes (segment's first run only)
  int32_t idx_start;  // first recompute position
};
static_assert(sizeof(RunDesc) == 32, "RunDesc layout");

// Where a run's source rows are: copied from the chunk pool, copied from the
// blocks of a block-resident chunk in the cache itself, or the destination
// rows themselves (a mapped chunk's keys rotated in place; values untouched).
// A run of 0 tokens only carries recompute positions.
enum RunKind : int32_t { kRunPool = 0, kRunBlocks = 1, kRunInPlace = 2 };
__host__ __device__ inline int32_t run_ntok(const RunDesc& r) { return r.ntok_kind & 0xffff; }
__host__ __device__ inline int32_t run_kind(const RunDesc& r) { return r.ntok_kind >> 16; }

// Workspace layout: [header 256 B][freq table][indptr][runs], each 256-B aligned.
struct WsHeader {
  uint32_t status;      // PIC_DEV_* bits raised by kernels
  uint32_t bad_req;     // a block-table row that held a bad entry (diagnostic)
  uint32_t bad_pos;     // the position it was asked for
  uint32_t pad[61];
};
static_assert(sizeof(WsHeader) == 256, "WsHeader layout");

constexpr size_t kWsAlign = 256;
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

enum Pairing : int { kNeox = 0, kInterleaved = 1 };

struct KernelParams {
  const RunDesc* runs;
  int32_t n_runs;
  int32_t n_lgroups;        // ceil(num_layers / lg_size)
  int32_t lg_size;          // layers per work unit
  int32_t contiguous;       // 1: CTA c owns units [c*U/G, (c+1)*U/G), layer group fastest;
                            // 0: CTA c takes units c, c+G, ..., run fastest
  int32_t num_layers;
  const float2* freq;       // rope_dim/2 (hi, lo): theta_i / (2 pi) as a float pair
  const uint8_t* k_src;     // pool (stitch) -- unused in place
  const uint8_t* v_src;     // value pool (GQA stitch) or null
  int64_t src_layer_stride;
  uint8_t* k_dst;           // paged key / MLA cache
  uint8_t* v_dst;           // paged value cache (GQA stitch) or null
  int64_t dst_layer_stride;
  const int32_t* block_tables;
  int32_t max_blocks;
  int32_t num_cache_blocks;
  int32_t block_size;
  int32_t heads_per_token;  // head rows per token (GQA heads; 1 for an MLA row)
  int32_t head_stride;      // bytes between head rows
  int32_t row_bytes;        // bytes per token row
  int32_t rope_off_bytes;   // byte offset of the rope slice inside a head row
  int32_t* ridx;            // recompute list output (may be null)
  const int32_t* indptr_src;
  int32_t* indptr_dst;      // recompute CSR offsets output (may be null)
  int32_t n_indptr;
  WsHeader* header;
  // Test hook of the bulk pipeline's failure path (pic_debug_stall_next_launch):
  // debug_stall = t + 1 makes CTA 0 skip tile t's copies and barrier arrival;
  // max_spins bounds every mbarrier wait (0: the default bound).
  int32_t debug_stall;
  uint32_t max_spins;
};

// Shared-memory pipeline shape of the bulk-copy kernels.
struct TmaConfig {
  int32_t stages;       // ring depth (>= 2)
  int32_t stage_bytes;  // bytes per stage (K tile, then V tile when present), multiple of 128
  int32_t tile_tokens;  // most tokens one unit (run x layer) may hold
};
constexpr size_t kTmaStageBudget = 200 * 1024;  // shared memory given to the stages
constexpr int kTmaMaxStages = 16;
constexpr int kTmaTileBytesPerTensor = 32 * 1024;

size_t tma_smem_bytes(const TmaConfig& c);
// mode 0: stitch with values, 1: stitch without values (MLA), 2: in place.
cudaError_t launch_tma(const KernelParams& p, const TmaConfig& c, int mode, int pairing, int rope_dim,
                       int grid, cudaStream_t stream);

// end region stitch-schedule

// region attend-params: what the decode attention kernels share with the host
// (a measurement record names this region).

// ---- decode attention over a stitched context (pic_attention.cu)
//
// Work is cut into stages: <= kAttnStageTokens consecutive positions of one
// request that share one delta.  A persistent CTA owns a contiguous range of
// (layer, stage) units; one consumer warp per KV head keeps an online softmax
// for the group's query heads while the CTA's range stays on one key
// (request x head group); each (layer, key) the range leaves becomes one
// record: per KV head, the max, sum and weighted values of its query heads.
constexpr int kAttnStageTokens = 16;        // positions per stage (one k-step of P.V)
constexpr int kAttnMaxHeads = 8;            // KV heads per CTA: one consumer warp each
constexpr int kAttnMaxStages = 8;           // shared-memory ring depth
constexpr int kAttnMaxCtas = 1024;          // persistent grid bound (workspace sizing)
constexpr int32_t kAttnFromCache = 1 << 8;  // AttnTok.flags: row is a paged-cache row

struct AttnStage {
  int32_t tok_off;     // first entry of the stage in the token list
  int32_t delta;       // every key of the stage is rotated by R(delta) (MLA on tcgen05: the keys
                       // before the stage's split; see TcTileRec)
  int32_t key;         // request * head_groups + head group
  uint16_t n_tok;      // 1 .. kAttnStageTokens
  uint16_t sink_mask;  // bit t: position t is a LegoLink pseudo-sink
};
static_assert(sizeof(AttnStage) == 16, "AttnStage layout");

struct AttnTok {
  int32_t row;    // pool token row, or absolute cache row (block * bs + row)
  int32_t flags;  // kAttnFromCache
};

struct AttnKey {  // per (layer, key), plus one closing entry
  int32_t rec_base;   // first record of this (layer, key)
  int32_t first_cta;  // CTA that writes that record
};

struct AttnParams {
  const AttnStage* stages;  // one layer's stages, key-major
  int32_t n_stages;
  const AttnTok* toks;
  const struct TcTileRec* tc_tiles;  // MLA on tcgen05: one layer's tiles (the same in every layer)
  int32_t tc_tiles_per_layer;        // n_units then counts (layer, tile) units
  const AttnKey* keys;      // [n_layers * n_keys + 1]
  int32_t n_keys;
  int64_t n_units;          // n_layers * n_stages
  const float2* freq;       // RoPE frequencies in turns, (hi, lo)
  const uint16_t* q;        // bf16 [n_layers][n_req][num_q_heads][D]
  int32_t n_req;
  int32_t num_q_heads;
  int32_t n_kv_heads;
  int32_t heads_per_cta;    // HB: KV heads a CTA (and a record) covers
  int32_t head_groups;      // n_kv_heads / HB
  int32_t n_layers;
  int32_t layer_begin;
  float scale_log2;         // softmax scale * log2(e)
  float sink_log2;          // sink bias * log2(e)
  const uint8_t* k_pool;
  const uint8_t* v_pool;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  int64_t pool_layer_stride;
  int64_t cache_layer_stride;
  int32_t row_bytes;        // one token, all KV heads
  int32_t ring;             // stages in the shared-memory ring
  float* records;           // [records][HB][attn_block_floats(G, D)]
  float* out;               // [n_layers][n_req][num_q_heads][D]
  float* lse;               // [n_layers][n_req][num_q_heads] or null
  uint32_t* status;         // PIC_DEV_* bits
  // Test hook (pic_debug_stall_next_launch; the tcgen05 MLA kernel only):
  // debug_stall = t + 1 makes CTA 0 skip tile t's copies and barrier
  // arrivals; max_spins bounds every wait of the launch (0: the default).
  int32_t debug_stall;
  uint32_t max_spins;
};

// floats of one (record, KV head) block: acc[G][D], m[G], l[G], padded to 16 B
__host__ __device__ constexpr int attn_block_floats(int group, int head_dim) {
  return (group * (head_dim + 2) + 3) / 4 * 4;
}
// floats of one record: every KV head of the group
__host__ __device__ constexpr int attn_record_floats(int group, int head_dim, int heads_per_cta) {
  return heads_per_cta * attn_block_floats(group, head_dim);
}
// Ring depth and dynamic shared memory of the attention kernel; false when
// two stages do not fit.
bool attend_config(int head_dim, int group, int heads_per_cta, int* ring, size_t* smem_bytes);
// CTAs of the attention kernel that fit on one SM.
int attend_ctas_per_sm(int pairing, int head_dim, int group, int heads_per_cta, size_t smem_bytes);
cudaError_t launch_attend(const AttnParams& p, int pairing, int head_dim, int group, int grid, size_t smem_bytes,
                          cudaStream_t stream);

// MLA decode attention (same plan, stages and records; one latent row per
// position, query heads in groups of 16, ng groups per CTA).
constexpr int kAttnMlaLatent = 512;
bool attend_mla_config(int ng, int* ring, size_t* smem_bytes);
int attend_mla_ctas_per_sm(int pairing, int ng, size_t smem_bytes);
cudaError_t launch_attend_mla(const AttnParams& p, int pairing, int ng, int grid, size_t smem_bytes,
                              cudaStream_t stream);
// Combines the per-CTA records of an MLA attention into out / lse.
cudaError_t launch_attend_merge_mla(const AttnParams& p, int heads_per_record, cudaStream_t stream);

// MLA decode attention on tcgen05 tensor cores with TMA tensor loads (same
// plan and records; hc = 16 or 32 query heads per CTA).  The maps view the
// pool and the paged cache as [layers][rows][576] bf16 with 128-byte swizzle
// and a box of 64 dims x 16 (g + 1) rows for map g; every stage of the plan
// reads consecutive rows of one of them.
// One tile of the tcgen05 MLA attention, formed on the host: up to four plan
// stages of one key, one per 16-row slot of the shared-memory ring.  A stage
// is up to 16 positions read from consecutive rows of one source and holds
// one or two deltas (positions from split on take the second).  Every layer
// has the same tiles.  With 16 query heads per CTA the kernel rotates the
// query's rope part, once per delta, into one of four entries of rotated
// query rows (entry, entry2, fresh, ent_delta); with 32 it rotates the rope
// keys themselves (delta, delta2).
constexpr int kTcRecKeyFirst = 1;  // the key's first tile in the layer
constexpr int kTcRecKeyLast = 2;   // its last
struct TcTileRec {
  int32_t ns;            // stages
  int32_t key;
  int32_t flags;         // kTcRecKeyFirst | kTcRecKeyLast
  int32_t fresh;         // entries given a new delta since the key's previous tile
  int32_t n_tok[4];
  int32_t sink[4];       // bit t: position t is a LegoLink pseudo-sink
  int32_t entry[4];      // entry of the stage's positions [0, split)
  int32_t entry2[4];     // entry of [split, n_tok)
  int32_t split[4];      // 16: one delta
  int32_t row[4];        // first source row of the stage
  int32_t src[4];        // its source (kAttnFromCache or 0)
  int32_t ent_delta[4];  // the delta each entry holds after this tile
  int32_t delta[4];      // shift of the stage's positions [0, split)
  int32_t delta2[4];     // and of [split, n_tok)
};
static_assert(sizeof(TcTileRec) == 176, "TcTileRec layout: 44 ints");

struct TcMaps {
  CUtensorMap pool[4];
  CUtensorMap cache[4];
};
bool attend_mla_tc_config(int hc, size_t* smem_bytes);
cudaError_t launch_attend_mla_tc(const AttnParams& p, const TcMaps& maps, int pairing, int hc, int grid,
                                 size_t smem_bytes, cudaStream_t stream);

// end region attend-params

// Launchers; each returns the launch's cudaError_t.  `grid` is the number of
// CTAs (persistent, grid-stride over units).
cudaError_t launch_stitch_gqa(const KernelParams& p, int pairing, int head_dim, int grid,
                              cudaStream_t stream);
cudaError_t launch_stitch_mla(const KernelParams& p, int pairing, int grid, cudaStream_t stream);
cudaError_t launch_rerotate(const KernelParams& p, int pairing, int rope_dim, int grid,
                            cudaStream_t stream);
cudaError_t launch_cossin(const int32_t* deltas, int32_t n, const float2* freq, int32_t half,
                          float* out, cudaStream_t stream);

// Stitch whose workspace image is built in caller-supplied host memory and
// copied (pageable copy, no pinned staging) into caller-supplied device
// scratch.  On success it allocates nothing, host or device (only building an
// error message may touch the heap).  Used by the no-alloc entry point
// (pic_noalloc.cu), which owns both buffers.
pic_status stitch_with_scratch(pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req,
                               const void* k_pool, const void* v_pool, int64_t pool_ls,
                               void* k_cache, void* v_cache, int64_t cache_ls,
                               const int32_t* d_bt, int32_t max_blocks, int32_t* d_ridx,
                               int32_t* d_indptr, int64_t recompute_capacity, void* d_scratch,
                               size_t scratch_bytes, uint8_t* host_image, size_t host_image_bytes,
                               uint32_t* d_status_out, cudaStream_t stream);

// Records an error message on ctx (or the calling thread) and returns st.
pic_status set_error(pic_ctx* ctx, pic_status st, const char* msg);

// Pool staging (pic_stage_pool): spans of pool rows of one layer (byte
// offset and length, multiples of 16), copied for every layer and tensor.
struct StageSpan {
  int64_t off;
  int64_t bytes;
};
constexpr int kStageMaxSpans = 1024;  // per launch: the parameters stay below 32 KB
struct StageParams {
  const uint8_t* src[2];  // host pools (K, V)
  uint8_t* dst[2];        // device pools (K, V)
  int64_t src_ls, dst_ls;
  int32_t n_spans, layers, tensors;
  StageSpan spans[kStageMaxSpans];
};
cudaError_t launch_stage_rows(const StageParams& p, int grid, cudaStream_t stream);

// Resident CTAs per SM of the kernel the matching launcher would use.
int occupancy_stitch_gqa(int pairing, int head_dim);
int occupancy_stitch_mla(int pairing);
int occupancy_rerotate(int pairing, int rope_dim);

}  // namespace pic
