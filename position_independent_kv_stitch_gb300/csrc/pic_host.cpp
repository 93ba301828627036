// Host side of libpic: the C ABI declared in include/pic.h.
//
// Holds the content-addressed chunk registry, the prompt composer, the paged
// block allocator and the recompute-list rule, validates every call, builds
// the flat run list each launch consumes and enqueues it on the caller's
// stream.  Sources: "EPIC Guide: Position-Independent Caching for LLM
// Serving" (runtime: chunk registry, prompt composer, PagedAttention block
// pool; LegoLink sink tokens), "Irminsul: MLA-Native Position-Independent
// Caching for Agentic LLM Serving" (registry entry (cKV, k_r, base_pos),
// delta = p_target - p_source, first-chunk carve-out).
#include "pic.h"

#include <algorithm>
#include <cstdarg>
#include <cstdlib>
#include <array>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <limits>
#include <new>
#include <set>
#include <string>
#include <unordered_map>
#include <memory>
#include <vector>

#include "pic_internal.h"

using pic::RunDesc;
using pic::WsHeader;

namespace {

constexpr double kPi = 3.14159265358979323846;

thread_local std::string g_thread_error;

struct KeyHash {
  size_t operator()(const std::array<uint8_t, PIC_KEY_BYTES>& k) const {
    uint64_t h = 0xcbf29ce484222325ull;  // FNV-1a over the key bytes
    for (uint8_t b : k) {
      h ^= b;
      h *= 0x100000001b3ull;
    }
    return static_cast<size_t>(h);
  }
};

struct ChunkEntry {
  std::array<uint8_t, PIC_KEY_BYTES> key;
  int64_t pool_token_offset;  // -1 for a block-resident chunk
  int32_t num_tokens;
  int32_t base_pos;           // block-resident: the position its keys are rotated to now
  bool live;
  bool in_blocks = false;     // KV sits in blocks of the paged cache
  std::vector<int32_t> blocks;
  int32_t refs = 0;           // live plans using this block-resident chunk
  const void* mapped_by = nullptr;  // the live plan that has its blocks mapped
};

struct Segment {
  int32_t chunk_id;
  int64_t src_tok;            // pool chunks: first pool token row; else -1
  int32_t num_tokens;
  int32_t dst_pos;
  int32_t delta;
  int32_t n_recompute;        // first n_recompute positions of the segment
  int32_t kind;               // pic::kRunPool / kRunBlocks / kRunInPlace
  std::vector<int32_t> src_blocks;  // kRunBlocks: the chunk's blocks
};

// Paged blocks [0, n): lowest free id first (one deterministic choice).
class BlockAllocator {
 public:
  explicit BlockAllocator(int32_t n) : n_(n), words_((n + 63) / 64, 0), free_count_(n) {}

  int32_t free_count() const { return free_count_; }
  bool is_free(int32_t id) const { return id >= 0 && id < n_ && !(words_[id >> 6] >> (id & 63) & 1ull); }

  // Takes specific free ids (the caller checked is_free).
  void take(const std::vector<int32_t>& ids) {
    for (int32_t id : ids) words_[id >> 6] |= 1ull << (id & 63);
    free_count_ -= static_cast<int32_t>(ids.size());
    hint_ = first_free_from(hint_);
  }

  // Takes the `count` lowest free ids; false (nothing taken) if too few are free.
  bool allocate(int32_t count, std::vector<int32_t>& out) {
    out.clear();
    if (count > free_count_) return false;
    out.reserve(count);
    int32_t b = hint_;
    while (static_cast<int32_t>(out.size()) < count) {
      b = first_free_from(b);
      out.push_back(b);
      ++b;
    }
    for (int32_t id : out) words_[id >> 6] |= 1ull << (id & 63);
    free_count_ -= count;
    hint_ = first_free_from(hint_);
    return true;
  }

  void release(const std::vector<int32_t>& ids) {
    for (int32_t id : ids) {
      words_[id >> 6] &= ~(1ull << (id & 63));
      hint_ = std::min(hint_, id);
    }
    free_count_ += static_cast<int32_t>(ids.size());
  }

 private:
  int32_t first_free_from(int32_t b) const {
    while (b < n_) {
      const uint64_t w = words_[b >> 6];
      if (w == ~0ull) {
        b = ((b >> 6) + 1) << 6;
        continue;
      }
      if (!(w >> (b & 63) & 1ull)) return b;
      ++b;
    }
    return n_;
  }

  int32_t n_;
  std::vector<uint64_t> words_;
  int32_t free_count_;
  int32_t hint_ = 0;  // no free block below this id
};

int vectorized_bytes_ok(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

struct pic_plan {
  pic_ctx* owner;
  uint64_t serial = 0;          // unique within the context: names this plan in caches
  std::vector<Segment> segs;
  std::vector<int32_t> table;   // the request's block table (mapped + fresh blocks)
  std::vector<int32_t> fresh;   // blocks this plan took from the allocator
  int32_t total_tokens;
  int32_t n_recompute;
  bool has_mapped = false;      // some segment rotates a mapped chunk in place
  bool applied = false;         // its in-place rotations have been enqueued
  std::vector<std::pair<int32_t, int32_t>> undo;  // (chunk, position before mapping)
};

// Pinned host staging buffers for workspace images.  A pageable source would
// make cudaMemcpyAsync wait for the stream first; pinned buffers let the next
// call be planned and enqueued while the previous kernel runs.  Each buffer
// records an event after its upload and is reused only once that has fired.
struct StagingSlot {
  uint8_t* host = nullptr;
  size_t cap = 0;
  cudaEvent_t uploaded = nullptr;
};
constexpr int kStagingSlots = 4;

// A device copy of a cached attention plan's read-only image (frequency
// table, stages, tiles, token rows, record keys): a decode loop that attends
// to the same plans uploads it once, not every step.
struct AttnResident {
  void* dev = nullptr;             // stream-ordered allocation on `device`
  size_t cap = 0;
  int device = -1;
  uint64_t owner = 0;              // serial of the cached plan whose image it holds (0: none)
  int32_t layers = 0;              // the image's record keys are for this layer count
  int64_t ctas = 0;                // and grid
  cudaEvent_t last_use = nullptr;  // recorded after every launch that reads it
};

struct pic_ctx {
  pic_model_desc model;
  std::vector<double> theta;          // radians per position, rope_dim/2
  std::vector<float2> freq_turns;     // theta_i / (2 pi) as hi + lo floats
  int32_t num_cache_blocks;
  std::vector<ChunkEntry> chunks;
  std::unordered_map<std::array<uint8_t, PIC_KEY_BYTES>, int32_t, KeyHash> by_key;
  BlockAllocator alloc;
  std::set<pic_plan*> plans;
  std::string err;
  // Kernel variant per mode: the bulk-copy pipeline when a unit fits a
  // shared-memory stage, the register kernel otherwise (or when
  // PIC_KERNEL=regs is set in the environment at pic_create).
  bool tma_stitch = false;
  bool tma_inplace = false;
  pic::TmaConfig tma_stitch_cfg{};
  pic::TmaConfig tma_inplace_cfg{};
  // MLA decode attention on tcgen05 tensor cores (16 or 32 heads per CTA);
  // PIC_ATTEND_KERNEL=mma at pic_create selects the warp-level mma kernel
  bool attend_tc = false;
  StagingSlot staging[kStagingSlots];
  int staging_next = 0;
  int staging_device = -1;
  // pic_debug_stall_next_launch: consumed by the next pic_stitch or pic_attend_decode
  int32_t debug_stall = 0;   // tile + 1, 0 = off
  uint32_t debug_spins = 0;  // 0 = the default wait bound
  uint64_t plan_serial = 0;  // last serial given to a plan
  // The last decode-attention plan of each stage form (one delta per stage,
  // or up to two), reused while the same plans (by serial and in-place
  // state), source and head layout come back: a decode loop attends to the
  // same composed requests every step.
  std::shared_ptr<void> attn_cache[2];
  uint64_t attn_serial = 0;  // last serial given to a cached attention plan
  AttnResident attn_res[2];  // one per cache slot
  // pic_stitch_staged: the stream its pool copies run on, and the event that
  // orders them against the caller's stream (created on first use, per device)
  cudaStream_t copy_stream = nullptr;
  cudaEvent_t copy_event = nullptr;
  int copy_device = -1;
  pic_ctx(int32_t nb) : num_cache_blocks(nb), alloc(nb) {}
};

namespace {

pic_status fail(pic_ctx* ctx, pic_status st, const char* fmt, ...) __attribute__((format(printf, 3, 4)));
pic_status fail(pic_ctx* ctx, pic_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (ctx) ctx->err = buf;
  else g_thread_error = buf;
  return st;
}

pic_status ok(pic_ctx* ctx) {
  if (ctx) ctx->err.clear();
  else g_thread_error.clear();
  return PIC_OK;
}

pic_status cuda_fail(pic_ctx* ctx, cudaError_t e, const char* what) {
  return fail(ctx, PIC_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

int64_t row_bytes_of(const pic_model_desc& m) {
  return static_cast<int64_t>(m.num_kv_heads) * m.head_dim * 2;
}

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
};

pic_status current_device(pic_ctx* ctx, DeviceInfo& di) {
  cudaError_t e = cudaGetDevice(&di.device);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaGetDevice");
  e = cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, di.device);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaDeviceGetAttribute");
  return PIC_OK;
}

bool plan_valid(const pic_ctx* ctx, const pic_plan* p) {
  return p != nullptr && ctx->plans.count(const_cast<pic_plan*>(p)) != 0;
}

// region stitch-schedule: run lists, workspace layout, grids and launches of
// the stitch and in-place kernels (a measurement record names this region).

// Calls f(t, cnt, src) for each run of a segment: at most `cap` tokens that
// land in one destination block and, for copies out of a block-resident
// chunk, come from one of its blocks.  src is the run's first source row
// (pool token row or absolute cache row; unused in place).  A mapped segment
// whose keys need no rotation (delta 0) moves nothing: it yields one run of 0
// tokens when it still has recompute positions to write, else none.
template <typename F>
void for_each_run(const Segment& sg, int32_t bs, int32_t cap, F f) {
  if (sg.num_tokens <= 0) return;
  if (sg.kind == pic::kRunInPlace && sg.delta == 0) {
    if (sg.n_recompute > 0) f(0, 0, 0);
    return;
  }
  for (int32_t t = 0; t < sg.num_tokens;) {
    const int32_t pos = sg.dst_pos + t;
    int32_t cnt = std::min(std::min(bs - pos % bs, sg.num_tokens - t), cap);
    int32_t src = 0;
    if (sg.kind == pic::kRunPool) {
      src = static_cast<int32_t>(sg.src_tok + t);
    } else if (sg.kind == pic::kRunBlocks) {
      cnt = std::min(cnt, bs - t % bs);
      src = sg.src_blocks[t / bs] * bs + t % bs;
    }
    f(t, cnt, src);
    t += cnt;
  }
}

// Runs of an in-place shift segment (source = destination).
void append_shift_runs(std::vector<RunDesc>& runs, int32_t dst_pos, int32_t n, int32_t req, int32_t delta,
                       int32_t bs, int32_t cap) {
  for (int32_t t = 0; t < n;) {
    const int32_t pos = dst_pos + t;
    const int32_t cnt = std::min(std::min(bs - pos % bs, n - t), cap);
    RunDesc r{};
    r.dst_pos = pos;
    r.req = req;
    r.ntok_kind = cnt | (pic::kRunInPlace << 16);
    r.delta = delta;
    runs.push_back(r);
    t += cnt;
  }
}

int64_t runs_in_range(int32_t dst_pos, int32_t n, int32_t bs, int32_t cap) {
  int64_t runs = 0;
  for (int32_t t = 0; t < n;) {
    const int32_t pos = dst_pos + t;
    t += std::min(std::min(bs - pos % bs, n - t), cap);
    ++runs;
  }
  return runs;
}

// Layers per unit: enough units per resident CTA (~16) for an even finish,
// as few as that allows so the per-unit cos/sin work is amortised.
void choose_layer_groups(int64_t n_runs, int32_t L, int64_t resident, int32_t& lg_size,
                         int32_t& n_lgroups) {
  const int64_t want_units = std::max<int64_t>(1, resident * 16);
  int64_t lg = (n_runs * L) / want_units;
  lg = std::max<int64_t>(1, std::min<int64_t>(lg, L));
  lg_size = static_cast<int32_t>(lg);
  n_lgroups = (L + lg_size - 1) / lg_size;
}

struct WsLayout {
  size_t freq_off, indptr_off, runs_off, total;
};

WsLayout ws_layout(size_t half, size_t n_indptr, size_t n_runs) {
  WsLayout w;
  w.freq_off = pic::align_up(sizeof(WsHeader), pic::kWsAlign);
  w.indptr_off = pic::align_up(w.freq_off + half * sizeof(float2), pic::kWsAlign);
  w.runs_off = pic::align_up(w.indptr_off + n_indptr * sizeof(int32_t), pic::kWsAlign);
  w.total = pic::align_up(w.runs_off + n_runs * sizeof(RunDesc), pic::kWsAlign);
  return w;
}

int32_t stitch_cap(const pic_ctx* ctx) {
  return ctx->tma_stitch ? ctx->tma_stitch_cfg.tile_tokens : ctx->model.block_size;
}
int32_t inplace_cap(const pic_ctx* ctx) {
  return ctx->tma_inplace ? ctx->tma_inplace_cfg.tile_tokens : ctx->model.block_size;
}

size_t count_stitch_runs(const pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req) {
  const int32_t bs = ctx->model.block_size, cap = stitch_cap(ctx);
  size_t n = 0;
  for (int32_t r = 0; r < n_req; ++r)
    for (const Segment& sg : plans[r]->segs) for_each_run(sg, bs, cap, [&](int32_t, int32_t, int32_t) { ++n; });
  return n;
}

size_t count_shift_runs(const pic_ctx* ctx, const pic_shift_seg* segs, int32_t n) {
  const int32_t bs = ctx->model.block_size, cap = inplace_cap(ctx);
  size_t runs = 0;
  for (int32_t i = 0; i < n; ++i) {
    if (segs[i].num_tokens <= 0 || segs[i].delta == 0 || segs[i].start_pos < 0) continue;
    runs += static_cast<size_t>(runs_in_range(segs[i].start_pos, segs[i].num_tokens, bs, cap));
  }
  return runs;
}

// Writes the stitch workspace image (frequencies, CSR offsets, runs) into a
// zeroed host buffer laid out as `w`, with no allocation.
void build_stitch_image(const pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req, uint8_t* image,
                        const WsLayout& w) {
  const int32_t bs = ctx->model.block_size, cap = stitch_cap(ctx);
  std::memcpy(image + w.freq_off, ctx->freq_turns.data(), ctx->freq_turns.size() * sizeof(float2));
  int32_t* indptr = reinterpret_cast<int32_t*>(image + w.indptr_off);
  RunDesc* out = reinterpret_cast<RunDesc*>(image + w.runs_off);
  size_t k = 0;
  int64_t idx = 0;
  for (int32_t r = 0; r < n_req; ++r) {
    indptr[r] = static_cast<int32_t>(idx);
    for (const Segment& sg : plans[r]->segs) {
      for_each_run(sg, bs, cap, [&](int32_t t, int32_t cnt, int32_t src) {
        RunDesc& rd = out[k++];
        rd.src = src;
        rd.dst_pos = sg.dst_pos + t;
        rd.req = r;
        rd.ntok_kind = cnt | (sg.kind << 16);
        rd.delta = sg.delta;
        rd.idx_off = static_cast<int32_t>(idx);
        rd.idx_count = t == 0 ? sg.n_recompute : 0;
        rd.idx_start = sg.dst_pos;
      });
      idx += sg.n_recompute;
    }
  }
  indptr[n_req] = static_cast<int32_t>(idx);
}

void set_geometry(const pic_ctx* ctx, pic::KernelParams& p) {
  const pic_model_desc& m = ctx->model;
  p.num_layers = m.num_layers;
  p.num_cache_blocks = ctx->num_cache_blocks;
  p.block_size = m.block_size;
  p.row_bytes = static_cast<int32_t>(row_bytes_of(m));
  if (m.kind == PIC_KIND_GQA) {
    p.heads_per_token = m.num_kv_heads;
    p.head_stride = m.head_dim * 2;
    p.rope_off_bytes = 0;
  } else {
    p.heads_per_token = 1;
    p.head_stride = p.row_bytes;
    p.rope_off_bytes = m.rope_offset * 2;
  }
}

// Schedules, measured on GB300 with all five workloads (the choices with the
// highest sustained HBM throughput):
//  * register kernels: CTAs stride over units of 2 layers, runs fastest, so
//    CTAs running together stream neighbouring memory; about 64 KB of loads
//    in flight per SM is best -- 1 CTA/SM for the stitch (K and V in flight),
//    2 CTAs/SM for the in-place shift (K only);
//  * bulk pipeline: strided units of 2 layers for GQA stitches, 4 for GQA
//    shifts; contiguous units of 4 layers for MLA rows, whose short tiles
//    need the producer's run lookup reused across a run's layers.
constexpr int kRegsLayersPerUnit = 2;

void set_layer_groups(pic::KernelParams& p, int32_t L, int lg) {
  p.lg_size = std::max(1, std::min<int32_t>(lg, L));
  p.n_lgroups = (L + p.lg_size - 1) / p.lg_size;
}

int grid_for(const pic::KernelParams& p, int64_t resident) {
  const int64_t units = static_cast<int64_t>(p.n_runs) * p.n_lgroups;
  // at least one CTA so the CSR offsets are always written
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(resident, units)));
}

// Where a buffer lives, for the kernels: 0 device (or managed) memory, 1
// pinned / registered host memory (reachable over the host link), -1 memory
// the GPU cannot reach (pageable host memory).
int residency(const void* p) {
  if (!p) return 0;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  if (a.type == cudaMemoryTypeHost) return 1;
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return 0;
  return -1;
}

// 1 if any of the buffers is host memory, 0 if all are device memory, -1 if
// one is unreachable (the error is recorded on ctx).
int host_buffers(pic_ctx* ctx, const void* const* ptrs, int n) {
  int any_host = 0;
  for (int i = 0; i < n; ++i) {
    const int r = residency(ptrs[i]);
    if (r < 0) {
      fail(ctx, PIC_ERR_INVALID_ARG,
           "a pool or cache buffer is pageable host memory; pin it (cudaHostAlloc / cudaHostRegister) or use "
           "device memory");
      return -1;
    }
    any_host |= r;
  }
  return any_host;
}

// Picks the kernel for a stitch and launches it on stream s.
// Buffers in host memory always go to the register kernels: they stream
// through the host link with plain loads and stores.
// True when most tokens of the batch are mapped keys rotated in place (K
// only, half the bytes in flight per thread of a K+V copy).
bool mostly_in_place(const pic_plan* const* plans, int32_t n_req) {
  int64_t in_place = 0, copied = 0;
  for (int32_t r = 0; r < n_req; ++r)
    for (const Segment& sg : plans[r]->segs) {
      if (sg.kind == pic::kRunInPlace) in_place += sg.delta != 0 ? sg.num_tokens : 0;
      else copied += sg.num_tokens;
    }
  return in_place > copied;
}

cudaError_t launch_stitch_kernel(const pic_ctx* ctx, pic::KernelParams& p, int sm_count, cudaStream_t s,
                                 bool host_io, bool in_place_heavy) {
  const pic_model_desc& m = ctx->model;
  const bool gqa = m.kind == PIC_KIND_GQA;
  if (ctx->tma_stitch && !host_io) {
    // one CTA per SM (the stages take most of shared memory)
    set_layer_groups(p, m.num_layers, gqa ? 2 : 4);
    p.contiguous = gqa ? 0 : 1;
    return pic::launch_tma(p, ctx->tma_stitch_cfg, gqa ? 0 : 1, m.pairing, m.rope_dim, grid_for(p, sm_count), s);
  }
  if (gqa) {
    set_layer_groups(p, m.num_layers, kRegsLayersPerUnit);
    p.contiguous = 0;
    // ~64 KB of loads in flight per SM: one CTA for K+V copies, two when most
    // runs move keys only (mapped chunks rotated in place)
    const int cps = std::min(in_place_heavy ? 2 : 1, pic::occupancy_stitch_gqa(m.pairing, m.head_dim));
    return pic::launch_stitch_gqa(p, m.pairing, m.head_dim, grid_for(p, static_cast<int64_t>(sm_count) * cps), s);
  }
  const int64_t resident = static_cast<int64_t>(sm_count) * pic::occupancy_stitch_mla(m.pairing);
  choose_layer_groups(static_cast<int64_t>(p.n_runs), m.num_layers, resident, p.lg_size, p.n_lgroups);
  return pic::launch_stitch_mla(p, m.pairing, grid_for(p, resident), s);
}

cudaError_t launch_shift_kernel(const pic_ctx* ctx, pic::KernelParams& p, int sm_count, cudaStream_t s,
                                bool host_io) {
  const pic_model_desc& m = ctx->model;
  if (ctx->tma_inplace && !host_io) {
    set_layer_groups(p, m.num_layers, 4);
    p.contiguous = 0;
    return pic::launch_tma(p, ctx->tma_inplace_cfg, 2, m.pairing, m.rope_dim, grid_for(p, sm_count), s);
  }
  set_layer_groups(p, m.num_layers, kRegsLayersPerUnit);
  p.contiguous = 0;
  const int cps = std::min(2, pic::occupancy_rerotate(m.pairing, m.rope_dim));
  return pic::launch_rerotate(p, m.pairing, m.rope_dim, grid_for(p, static_cast<int64_t>(sm_count) * cps), s);
}

// Chooses the bulk-copy pipeline shape for units of `tensors` row tiles, or
// returns false when the register kernel should be used.
bool tma_config_for(int64_t row_bytes, int32_t block_size, int tensors, int64_t tile_bytes, pic::TmaConfig& c) {
  int64_t tile = std::max<int64_t>(1, tile_bytes / row_bytes);
  tile = std::min<int64_t>(tile, block_size);
  const int64_t per_tensor = static_cast<int64_t>(pic::align_up(static_cast<size_t>(tile * row_bytes), 128));
  const int64_t stage = per_tensor * tensors;
  const int64_t stages = std::min<int64_t>(pic::kTmaMaxStages, static_cast<int64_t>(pic::kTmaStageBudget) / stage);
  if (stages < 2) return false;
  c.stages = static_cast<int32_t>(stages);
  c.stage_bytes = static_cast<int32_t>(stage);
  c.tile_tokens = static_cast<int32_t>(tile);
  return true;
}

// Argument checks shared by pic_stitch and the scratch-backed stitch.
pic_status check_stitch_args(pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req,
                             const void* k_pool, const void* v_pool, int64_t pool_ls,
                             const void* k_cache, const void* v_cache, int64_t cache_ls,
                             const int32_t* d_bt, int32_t max_blocks, const int32_t* d_ridx,
                             const int32_t* d_indptr, int64_t recompute_capacity) {
  const pic_model_desc& m = ctx->model;
  if (n_req < 0 || (n_req > 0 && !plans)) return fail(ctx, PIC_ERR_INVALID_ARG, "bad plan list");
  for (int32_t r = 0; r < n_req; ++r) {
    if (!plan_valid(ctx, plans[r])) return fail(ctx, PIC_ERR_INVALID_ARG, "plans[%d] does not belong to this context", r);
    if (static_cast<int32_t>(plans[r]->table.size()) > max_blocks)
      return fail(ctx, PIC_ERR_CAPACITY, "plans[%d] has %zu blocks, block-table rows hold %d", r,
                  plans[r]->table.size(), max_blocks);
    if (plans[r]->has_mapped) {
      if (plans[r]->applied)
        return fail(ctx, PIC_ERR_INVALID_ARG, "plans[%d] maps chunks whose keys were already rotated in place; "
                    "a plan with mapped chunks is stitched once", r);
      for (int32_t q = 0; q < r; ++q)
        if (plans[q] == plans[r]) return fail(ctx, PIC_ERR_INVALID_ARG, "plans[%d] appears twice", r);
    }
  }
  const bool gqa = m.kind == PIC_KIND_GQA;
  if (!k_pool || !k_cache || !d_bt) return fail(ctx, PIC_ERR_INVALID_ARG, "null pool, cache or block table");
  if (gqa && (!v_pool || !v_cache)) return fail(ctx, PIC_ERR_INVALID_ARG, "GQA needs v_pool and v_cache");
  if (!gqa && (v_pool || v_cache)) return fail(ctx, PIC_ERR_INVALID_ARG, "MLA rows have no separate values (pass NULL)");
  if ((d_ridx == nullptr) != (d_indptr == nullptr))
    return fail(ctx, PIC_ERR_INVALID_ARG, "pass both recompute outputs or neither");
  if (!vectorized_bytes_ok(k_pool) || !vectorized_bytes_ok(k_cache) ||
      (gqa && (!vectorized_bytes_ok(v_pool) || !vectorized_bytes_ok(v_cache))) || (pool_ls & 15) || (cache_ls & 15))
    return fail(ctx, PIC_ERR_ALIGNMENT, "pools, caches and layer strides must be 16-byte aligned");
  const int64_t row_bytes = row_bytes_of(m);
  if (pool_ls < 0 || cache_ls < 0 || (m.num_layers > 1 && (pool_ls == 0 || cache_ls == 0)))
    return fail(ctx, PIC_ERR_INVALID_ARG, "bad layer strides");
  if (m.num_layers > 1 && cache_ls < static_cast<int64_t>(ctx->num_cache_blocks) * m.block_size * row_bytes)
    return fail(ctx, PIC_ERR_RANGE, "cache layer stride smaller than num_cache_blocks * block_size rows");
  int64_t n_rec = 0;
  for (int32_t r = 0; r < n_req; ++r) n_rec += plans[r]->n_recompute;
  if (d_ridx && n_rec > std::numeric_limits<int32_t>::max())
    return fail(ctx, PIC_ERR_RANGE, "recompute list of %lld entries: CSR offsets are int32",
                static_cast<long long>(n_rec));
  if (d_ridx && n_rec > recompute_capacity)
    return fail(ctx, PIC_ERR_CAPACITY, "recompute list has %lld entries, capacity %lld",
                static_cast<long long>(n_rec), static_cast<long long>(recompute_capacity));
  return PIC_OK;
}

void fill_stitch_params(const pic_ctx* ctx, pic::KernelParams& p, uint8_t* ws, const WsLayout& w, size_t n_runs,
                        int32_t n_req, const void* k_pool, const void* v_pool, int64_t pool_ls, void* k_cache,
                        void* v_cache, int64_t cache_ls, const int32_t* d_bt, int32_t max_blocks, int32_t* d_ridx,
                        int32_t* d_indptr) {
  set_geometry(ctx, p);
  p.runs = reinterpret_cast<const RunDesc*>(ws + w.runs_off);
  p.n_runs = static_cast<int32_t>(n_runs);
  p.freq = reinterpret_cast<const float2*>(ws + w.freq_off);
  p.k_src = static_cast<const uint8_t*>(k_pool);
  p.v_src = static_cast<const uint8_t*>(v_pool);
  p.src_layer_stride = pool_ls;
  p.k_dst = static_cast<uint8_t*>(k_cache);
  p.v_dst = static_cast<uint8_t*>(v_cache);
  p.dst_layer_stride = cache_ls;
  p.block_tables = d_bt;
  p.max_blocks = max_blocks;
  p.ridx = d_ridx;
  p.indptr_src = reinterpret_cast<const int32_t*>(ws + w.indptr_off);
  p.indptr_dst = d_indptr;
  p.n_indptr = n_req + 1;
  p.header = reinterpret_cast<WsHeader*>(ws);
}

// end region stitch-schedule

void release_staging(pic_ctx* ctx) {
  for (StagingSlot& sl : ctx->staging) {
    if (sl.uploaded) {
      cudaEventSynchronize(sl.uploaded);
      cudaEventDestroy(sl.uploaded);
    }
    if (sl.host) cudaFreeHost(sl.host);
    sl = StagingSlot{};
  }
  ctx->staging_device = -1;
}

void release_attn_resident(pic_ctx* ctx) {
  bool any = false;
  for (const AttnResident& r : ctx->attn_res) any |= r.dev != nullptr || r.last_use != nullptr;
  if (!any) return;
  int cur = -1;
  cudaGetDevice(&cur);
  for (AttnResident& r : ctx->attn_res) {
    if (r.dev || r.last_use) {
      cudaSetDevice(r.device);
      if (r.last_use) cudaEventSynchronize(r.last_use);
      if (r.dev) cudaFree(r.dev);
      if (r.last_use) cudaEventDestroy(r.last_use);
    }
    r = AttnResident{};
  }
  if (cur >= 0) cudaSetDevice(cur);
}

// Releases the context's copy stream and event.
void release_copy_stream(pic_ctx* ctx) {
  if (!ctx->copy_stream && !ctx->copy_event) return;
  int cur = -1;
  cudaGetDevice(&cur);
  cudaSetDevice(ctx->copy_device);
  if (ctx->copy_stream) {
    cudaStreamSynchronize(ctx->copy_stream);
    cudaStreamDestroy(ctx->copy_stream);
  }
  if (ctx->copy_event) cudaEventDestroy(ctx->copy_event);
  ctx->copy_stream = nullptr;
  ctx->copy_event = nullptr;
  ctx->copy_device = -1;
  if (cur >= 0) cudaSetDevice(cur);
}

// A zeroed pinned buffer of `bytes` for the next upload on `device`.
pic_status acquire_staging(pic_ctx* ctx, int device, size_t bytes, StagingSlot** out) {
  if (ctx->staging_device != device) {
    release_staging(ctx);
    ctx->staging_device = device;
  }
  StagingSlot& sl = ctx->staging[ctx->staging_next];
  ctx->staging_next = (ctx->staging_next + 1) % kStagingSlots;
  cudaError_t e;
  if (sl.uploaded) {
    e = cudaEventSynchronize(sl.uploaded);  // the last upload from this buffer is done
    if (e != cudaSuccess) return cuda_fail(ctx, e, "staging event");
  } else {
    e = cudaEventCreateWithFlags(&sl.uploaded, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaEventCreate");
  }
  if (sl.cap < bytes) {
    if (sl.host) cudaFreeHost(sl.host);
    sl.host = nullptr;
    sl.cap = 0;
    const size_t cap = std::max<size_t>(bytes + bytes / 2, 64 * 1024);
    e = cudaHostAlloc(reinterpret_cast<void**>(&sl.host), cap, cudaHostAllocPortable);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaHostAlloc (staging)");
    sl.cap = cap;
  }
  std::memset(sl.host, 0, bytes);
  *out = &sl;
  return PIC_OK;
}

// Enqueues the upload of a staged image and marks the slot busy until it lands.
pic_status upload_staging(pic_ctx* ctx, StagingSlot* sl, void* d_ws, size_t bytes, cudaStream_t s) {
  cudaError_t e = cudaMemcpyAsync(d_ws, sl->host, bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "workspace upload");
  e = cudaEventRecord(sl->uploaded, s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaEventRecord");
  return PIC_OK;
}

void fill_freq(const pic_ctx* ctx, uint8_t* base, const WsLayout& w) {
  std::memcpy(base + w.freq_off, ctx->freq_turns.data(), ctx->freq_turns.size() * sizeof(float2));
}

// region attend-plan: stages, tiles, records and tensor maps of the decode
// attention (a measurement record names this region).

// Decode attention: every position [0, total) of each request becomes one
// token entry (where its K/V row is), and each request's positions are cut
// into stages of <= kAttnStageTokens consecutive positions sharing one
// delta.  fused: chunk tokens are read from their sources (pool rows,
// block-resident chunk rows) and their keys need R(delta); inline positions
// and mapped chunks already rotated come from the request's paged cache.
// cache: every position from the paged cache, no rotation.  Stages are listed
// key-major (key = request * head_groups + head group) for one layer; the
// kernel walks (layer, stage) units.
struct AttnPlan {
  std::vector<pic::AttnStage> stages;
  std::vector<int4> ext;  // per stage: first token's {row, flags}, second delta, split (16: none)
  std::vector<pic::AttnTok> toks;
  std::vector<int32_t> key_stage_begin;  // [n_keys + 1]
  int32_t heads_per_cta = 0, head_groups = 0, n_keys = 0;
};

bool attn_heads(const pic_model_desc& m, int32_t* hb, int32_t* groups) {
  const int32_t H = m.num_kv_heads;
  if (H >= 1 && H <= pic::kAttnMaxHeads) {
    *hb = H;
    *groups = 1;
    return true;
  }
  if (H > 0 && H % pic::kAttnMaxHeads == 0) {
    *hb = pic::kAttnMaxHeads;
    *groups = H / pic::kAttnMaxHeads;
    return true;
  }
  return false;
}

// How one decode attention maps heads onto CTAs and records.
//   GQA: hb KV heads per CTA (head_groups groups of them per request), group
//        query heads per KV head, values of head_dim dims.
//   MLA: every query head reads the one latent row; a CTA (and a record)
//        covers group = min(H, 32) query heads, 16 per mla_ng quarter-warp
//        set, head_groups = H / group per request; values are the 512 latent
//        dims.
struct AttnHeads {
  int32_t hb = 0, head_groups = 0, group = 0, vdim = 0, mla_ng = 0;
};

bool attn_layout_heads(const pic_model_desc& m, int32_t num_q_heads, AttnHeads* h) {
  if (m.kind == PIC_KIND_MLA) {
    if (num_q_heads != 16 && num_q_heads != 32 && num_q_heads != 64 && num_q_heads != 128) return false;
    h->hb = 1;
    h->group = std::min<int32_t>(num_q_heads, 32);
    h->head_groups = num_q_heads / h->group;
    h->vdim = m.head_dim - m.rope_dim;
    h->mla_ng = h->group / 16;
    return true;
  }
  if (!attn_heads(m, &h->hb, &h->head_groups)) return false;
  if (m.num_kv_heads <= 0 || num_q_heads % m.num_kv_heads != 0) return false;
  h->group = num_q_heads / m.num_kv_heads;
  h->vdim = m.head_dim;
  h->mla_ng = 0;
  return true;
}

// two_deltas (MLA on tcgen05): a stage of consecutive rows may go on across
// one change of delta; the positions from its split on take the second delta.
void attend_plan(const pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req, int32_t source,
                 const AttnHeads& heads, bool two_deltas, AttnPlan* out) {
  const int32_t bs = ctx->model.block_size;
  const int32_t ST = pic::kAttnStageTokens;
  const bool mla = ctx->model.kind == PIC_KIND_MLA;
  out->heads_per_cta = heads.hb;
  out->head_groups = heads.head_groups;
  out->n_keys = n_req * out->head_groups;
  out->key_stage_begin.assign(1, 0);
  std::vector<pic::AttnStage> req_stages;
  std::vector<int4> req_ext;
  for (int32_t r = 0; r < n_req; ++r) {
    const pic_plan* pl = plans[r];
    const int32_t T = pl->total_tokens;
    const int32_t tok_off = static_cast<int32_t>(out->toks.size());
    std::vector<int32_t> deltas(T, 0);
    std::vector<uint8_t> sink(T, 0);
    out->toks.resize(out->toks.size() + T);
    pic::AttnTok* tk = out->toks.data() + tok_off;
    for (int32_t p = 0; p < T; ++p) tk[p] = pic::AttnTok{pl->table[p / bs] * bs + p % bs, pic::kAttnFromCache};
    for (const Segment& sg : pl->segs) {
      for (int32_t t = 0; t < sg.num_tokens; ++t) {
        const int32_t p = sg.dst_pos + t;
        if (sg.dst_pos != 0 && t < sg.n_recompute) sink[p] = 1;
        if (source != PIC_ATTEND_FUSED) continue;
        if (sg.kind == pic::kRunPool) {
          tk[p] = pic::AttnTok{static_cast<int32_t>(sg.src_tok + t), 0};
          deltas[p] = sg.delta;
        } else if (sg.kind == pic::kRunBlocks) {
          tk[p].row = sg.src_blocks[t / bs] * bs + t % bs;
          deltas[p] = sg.delta;
        } else if (!pl->applied) {  // mapped chunk whose keys have not moved yet
          deltas[p] = sg.delta;
        }
      }
    }
    req_stages.clear();
    req_ext.clear();
    for (int32_t p = 0; p < T;) {
      pic::AttnStage st{};
      st.tok_off = tok_off + p;
      st.delta = deltas[p];
      int32_t n = 0, split = ST, d2 = 0;
      // MLA stages also read consecutive rows of one source (one TMA box)
      while (p + n < T && n < ST &&
             (!mla || n == 0 || (tk[p + n].flags == tk[p].flags && tk[p + n].row == tk[p].row + n))) {
        const int32_t d = deltas[p + n];
        if (split == ST) {
          if (d != st.delta) {
            if (!two_deltas) break;
            split = n;  // the one change of delta a stage may hold
            d2 = d;
          }
        } else if (d != d2) {
          break;
        }
        if (sink[p + n]) st.sink_mask |= static_cast<uint16_t>(1u << n);
        ++n;
      }
      st.n_tok = static_cast<uint16_t>(n);
      req_stages.push_back(st);
      req_ext.push_back(make_int4(tk[p].row, tk[p].flags, d2, split));
      p += n;
    }
    for (int32_t hg = 0; hg < out->head_groups; ++hg) {
      for (pic::AttnStage st : req_stages) {
        st.key = r * out->head_groups + hg;
        out->stages.push_back(st);
      }
      out->ext.insert(out->ext.end(), req_ext.begin(), req_ext.end());
      out->key_stage_begin.push_back(static_cast<int32_t>(out->stages.size()));
    }
  }
}

// The attention plan of a call, from the context's one-entry cache when the
// same plans (serials and in-place state), source and head layout were
// planned last; pool_rows: one past the last pool row the plan reads.
struct AttnPlanCache {
  std::vector<uint64_t> key;
  uint64_t serial = 0;
  AttnPlan plan;
  int64_t pool_rows = 0;
  // two-delta plans (MLA on tcgen05): one layer's tiles and each key's first
  // tile (n_keys + 1 entries)
  std::vector<pic::TcTileRec> tiles;
  std::vector<int32_t> key_tile_begin;
};

// The tiles of the tcgen05 MLA attention for one layer (every layer has the
// same stages).  Within a key, stages fill tiles of up to four in order.
// With ne > 0 entries of rotated query rows (16 heads per CTA) each delta of
// a stage takes an entry: the entry that holds it, else a free one (holding
// nothing), else one neither this tile nor the previous one uses (its rewrite
// need not wait for the previous tile's score product), else one this tile
// does not use; a stage that finds no entry starts the next tile, and entries
// start empty at each key.  With ne = 0 (the kernel rotates the keys) tiles
// end only at four stages or at the key's end.
void tc_tiles(const AttnPlan& plan, int ne, std::vector<pic::TcTileRec>* tiles, std::vector<int32_t>* key_tile_begin) {
  tiles->clear();
  key_tile_begin->assign(1, 0);
  for (int32_t k = 0; k < plan.n_keys; ++k) {
    const int32_t end = plan.key_stage_begin[k + 1];
    int32_t ent_delta[4] = {0, 0, 0, 0};
    uint32_t valid = 0, prev_used = 0;
    bool first = true;
    for (int32_t j = plan.key_stage_begin[k]; j < end;) {
      pic::TcTileRec t{};
      t.key = k;
      uint32_t used = 0, fresh = 0;
      auto find = [&](int32_t d, uint32_t skip) {
        for (int x = 0; x < ne; ++x)
          if (((valid >> x) & 1u) && !((skip >> x) & 1u) && ent_delta[x] == d) return x;
        return -1;
      };
      auto pick = [&](uint32_t busy) {
        for (int x = 0; x < ne; ++x)
          if (!((busy >> x) & 1u) && !((valid >> x) & 1u)) return x;
        for (int x = 0; x < ne; ++x)
          if (!((busy >> x) & 1u) && !((prev_used >> x) & 1u)) return x;
        for (int x = 0; x < ne; ++x)
          if (!((busy >> x) & 1u)) return x;
        return -1;
      };
      while (t.ns < 4 && j < end) {
        const pic::AttnStage& st = plan.stages[j];
        const int4 x = plan.ext[j];
        const bool two = x.w < st.n_tok;
        int e1 = 0, e2 = 0;
        if (ne > 0) {
          uint32_t busy = used;
          e1 = find(st.delta, 0u);
          const bool new1 = e1 < 0;
          if (new1) e1 = pick(busy);
          if (e1 < 0) break;
          busy |= 1u << e1;
          e2 = e1;
          bool new2 = false;
          if (two) {
            e2 = find(x.z, new1 ? (1u << e1) : 0u);  // an entry just taken no longer holds what it held
            new2 = e2 < 0;
            if (new2) e2 = pick(busy);
            if (e2 < 0) break;
            busy |= 1u << e2;
          }
          if (new1) ent_delta[e1] = st.delta;
          if (new2) ent_delta[e2] = x.z;
          const uint32_t took = (new1 ? (1u << e1) : 0u) | (new2 ? (1u << e2) : 0u);
          valid |= took;
          fresh |= took;
          used = busy;
        }
        const int s4 = t.ns;
        t.n_tok[s4] = st.n_tok;
        t.sink[s4] = st.sink_mask;
        t.entry[s4] = e1;
        t.entry2[s4] = e2;
        t.split[s4] = two ? x.w : 16;
        t.row[s4] = x.x;
        t.src[s4] = x.y;
        t.delta[s4] = st.delta;
        t.delta2[s4] = two ? x.z : st.delta;
        ++t.ns;
        ++j;
      }
      t.fresh = static_cast<int32_t>(fresh);
      for (int e = 0; e < 4; ++e) t.ent_delta[e] = ent_delta[e];
      t.flags = (first ? pic::kTcRecKeyFirst : 0) | (j >= end ? pic::kTcRecKeyLast : 0);
      first = false;
      prev_used = used;
      tiles->push_back(t);
    }
    key_tile_begin->push_back(static_cast<int32_t>(tiles->size()));
  }
}

const AttnPlanCache& attend_plan_cached(pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req, int32_t source,
                                        const AttnHeads& heads, bool two_deltas) {
  std::vector<uint64_t> key;
  key.reserve(2 * static_cast<size_t>(n_req) + 5);
  for (int32_t r = 0; r < n_req; ++r) {
    key.push_back(plans[r]->serial);
    key.push_back(plans[r]->applied ? 1u : 0u);
  }
  key.push_back(static_cast<uint64_t>(source));
  key.push_back(static_cast<uint64_t>(heads.hb));
  key.push_back(static_cast<uint64_t>(heads.head_groups));
  key.push_back(static_cast<uint64_t>(heads.group));
  key.push_back(two_deltas ? 1u : 0u);
  std::shared_ptr<void>& slot = ctx->attn_cache[two_deltas ? 1 : 0];
  auto* c = static_cast<AttnPlanCache*>(slot.get());
  if (c && c->key == key) return *c;
  auto fresh = std::make_shared<AttnPlanCache>();
  attend_plan(ctx, plans, n_req, source, heads, two_deltas, &fresh->plan);
  for (const pic::AttnTok& t : fresh->plan.toks)
    if (!(t.flags & pic::kAttnFromCache)) fresh->pool_rows = std::max<int64_t>(fresh->pool_rows, int64_t{t.row} + 1);
  // 16 heads per CTA: four entries of rotated query rows; more: rotated keys
  if (two_deltas) tc_tiles(fresh->plan, heads.group == 16 ? 4 : 0, &fresh->tiles, &fresh->key_tile_begin);
  fresh->key = std::move(key);
  fresh->serial = ++ctx->attn_serial;
  slot = fresh;
  return *fresh;
}

struct AttnLayout {
  size_t freq_off, stages_off, tiles_off, toks_off, keys_off, records_off, total;
};

// cuTensorMapEncodeTiled, looked up once through the runtime (no link to the
// driver library).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// A view of MLA rows as [layers][rows][576] bf16, read in boxes of box_rows
// rows x 64 dims with 128-byte swizzle; rows past `rows` read as zeros.
bool encode_mla_rows(CUtensorMap* map, const void* base, int64_t rows, int64_t layers, int64_t layer_stride,
                     uint32_t box_rows) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc || !base || rows <= 0 || layers <= 0 || (layer_stride & 15) || rows > (int64_t{1} << 32)) return false;
  if (layers > 1 && layer_stride < rows * 1152) return false;
  const cuuint64_t dims[3] = {576, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(layers)};
  const cuuint64_t strides[2] = {1152, static_cast<cuuint64_t>(layers > 1 ? layer_stride : rows * 1152)};
  const cuuint32_t box[3] = {64, box_rows, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

AttnLayout attend_layout(const pic_ctx* ctx, size_t n_stages, size_t n_tiles, size_t n_toks, size_t n_key_entries,
                         size_t n_records, const AttnHeads& heads) {
  AttnLayout w;
  w.freq_off = pic::align_up(sizeof(WsHeader), pic::kWsAlign);
  w.stages_off = pic::align_up(w.freq_off + ctx->freq_turns.size() * sizeof(float2), pic::kWsAlign);
  w.tiles_off = pic::align_up(w.stages_off + n_stages * sizeof(pic::AttnStage), pic::kWsAlign);
  w.toks_off = pic::align_up(w.tiles_off + n_tiles * sizeof(pic::TcTileRec), pic::kWsAlign);
  w.keys_off = pic::align_up(w.toks_off + n_toks * sizeof(pic::AttnTok), pic::kWsAlign);
  w.records_off = pic::align_up(w.keys_off + n_key_entries * sizeof(pic::AttnKey), pic::kWsAlign);
  const size_t rec = static_cast<size_t>(pic::attn_record_floats(heads.group, heads.vdim, heads.hb)) * 4;
  w.total = pic::align_up(w.records_off + n_records * rec, pic::kWsAlign);
  return w;
}

// Records of a persistent grid of `ctas` over `layers` x plan.stages units:
// CTA c owns units [U c / N, U (c + 1) / N); each (layer, key) gets one
// record per CTA whose range touches it, written at rec_base + (c - first_cta).
// The same for a grid over (layer, tile) units: key k of a layer covers its
// tiles [key_tile_begin[k], key_tile_begin[k + 1]).
int64_t attend_keys_tiles(const std::vector<int32_t>& key_tile_begin, int32_t layers, int64_t ctas,
                          std::vector<pic::AttnKey>* keys) {
  const int32_t n_keys = static_cast<int32_t>(key_tile_begin.size()) - 1;
  const int64_t tpl = key_tile_begin.back();
  const int64_t U = tpl * layers;
  auto cta_of = [&](int64_t u) { return ((u + 1) * ctas - 1) / U; };
  int64_t rec = 0;
  if (keys) keys->clear();
  for (int32_t l = 0; l < layers; ++l)
    for (int32_t k = 0; k < n_keys; ++k) {
      const int64_t a = l * tpl + key_tile_begin[k], b = l * tpl + key_tile_begin[k + 1];
      const int64_t c0 = cta_of(a), c1 = cta_of(b - 1);
      if (keys) keys->push_back(pic::AttnKey{static_cast<int32_t>(rec), static_cast<int32_t>(c0)});
      rec += c1 - c0 + 1;
    }
  if (keys) keys->push_back(pic::AttnKey{static_cast<int32_t>(rec), 0});
  return rec;
}

int64_t attend_keys(const AttnPlan& plan, int32_t layers, int64_t ctas, std::vector<pic::AttnKey>* keys) {
  const int64_t nsl = static_cast<int64_t>(plan.stages.size());
  const int64_t U = nsl * layers;
  auto cta_of = [&](int64_t u) { return ((u + 1) * ctas - 1) / U; };
  int64_t rec = 0;
  if (keys) keys->clear();
  for (int32_t l = 0; l < layers; ++l)
    for (int32_t k = 0; k < plan.n_keys; ++k) {
      const int64_t a = l * nsl + plan.key_stage_begin[k], b = l * nsl + plan.key_stage_begin[k + 1];
      const int64_t c0 = cta_of(a), c1 = cta_of(b - 1);
      if (keys) keys->push_back(pic::AttnKey{static_cast<int32_t>(rec), static_cast<int32_t>(c0)});
      rec += c1 - c0 + 1;
    }
  if (keys) keys->push_back(pic::AttnKey{static_cast<int32_t>(rec), 0});
  return rec;
}

// end region attend-plan

}  // namespace

// ======================================================================= API

extern "C" {

int32_t pic_abi_version(void) { return PIC_ABI_VERSION; }

const char* pic_status_string(pic_status s) {
  switch (s) {
    case PIC_OK: return "PIC_OK";
    case PIC_ERR_INVALID_ARG: return "PIC_ERR_INVALID_ARG";
    case PIC_ERR_UNKNOWN_CHUNK: return "PIC_ERR_UNKNOWN_CHUNK";
    case PIC_ERR_KEY_CONFLICT: return "PIC_ERR_KEY_CONFLICT";
    case PIC_ERR_OUT_OF_BLOCKS: return "PIC_ERR_OUT_OF_BLOCKS";
    case PIC_ERR_CAPACITY: return "PIC_ERR_CAPACITY";
    case PIC_ERR_RANGE: return "PIC_ERR_RANGE";
    case PIC_ERR_ALIGNMENT: return "PIC_ERR_ALIGNMENT";
    case PIC_ERR_CUDA: return "PIC_ERR_CUDA";
    case PIC_ERR_DEVICE_CHECK: return "PIC_ERR_DEVICE_CHECK";
    case PIC_ERR_UNSUPPORTED: return "PIC_ERR_UNSUPPORTED";
    case PIC_ERR_BUSY: return "PIC_ERR_BUSY";
  }
  return "PIC_ERR_?";
}

const char* pic_last_error(const pic_ctx* ctx) {
  return ctx ? ctx->err.c_str() : g_thread_error.c_str();
}

pic_status pic_create(const pic_model_desc* m, int32_t num_cache_blocks, pic_ctx** out) {
  if (!m || !out) return fail(nullptr, PIC_ERR_INVALID_ARG, "pic_create: null argument");
  if (num_cache_blocks < 0) return fail(nullptr, PIC_ERR_INVALID_ARG, "num_cache_blocks < 0");
  if (m && static_cast<int64_t>(num_cache_blocks) * std::max(1, m->block_size) > std::numeric_limits<int32_t>::max())
    return fail(nullptr, PIC_ERR_RANGE, "num_cache_blocks * block_size must stay below 2^31 rows");
  if (m->num_layers < 1) return fail(nullptr, PIC_ERR_INVALID_ARG, "num_layers must be >= 1");
  if (m->block_size < 1 || m->block_size > 256)
    return fail(nullptr, PIC_ERR_INVALID_ARG, "block_size must be in [1, 256]");
  if (m->pairing != PIC_PAIRING_NEOX_HALF && m->pairing != PIC_PAIRING_INTERLEAVED)
    return fail(nullptr, PIC_ERR_INVALID_ARG, "unknown pairing %d", m->pairing);
  if (m->kind == PIC_KIND_GQA) {
    if (m->num_kv_heads < 1) return fail(nullptr, PIC_ERR_INVALID_ARG, "num_kv_heads must be >= 1");
    if (m->head_dim != 64 && m->head_dim != 128 && m->head_dim != 256)
      return fail(nullptr, PIC_ERR_UNSUPPORTED, "GQA head_dim %d has no kernel (64, 128, 256)", m->head_dim);
    if (m->rope_dim != m->head_dim || m->rope_offset != 0)
      return fail(nullptr, PIC_ERR_UNSUPPORTED, "GQA keys are rotated over the whole head (rope_dim == head_dim, rope_offset 0)");
  } else if (m->kind == PIC_KIND_MLA) {
    if (m->num_kv_heads != 1 || m->head_dim != 576 || m->rope_dim != 64 || m->rope_offset != 512)
      return fail(nullptr, PIC_ERR_UNSUPPORTED, "MLA rows must be 512 latent + 64 rope (num_kv_heads 1, head_dim 576)");
  } else {
    return fail(nullptr, PIC_ERR_INVALID_ARG, "unknown kind %d", m->kind);
  }
  const int32_t half = m->rope_dim / 2;
  std::vector<double> theta(half);
  if (m->inv_freq) {
    for (int32_t i = 0; i < half; ++i) {
      if (!std::isfinite(m->inv_freq[i]) || m->inv_freq[i] < 0)
        return fail(nullptr, PIC_ERR_INVALID_ARG, "inv_freq[%d] is not a finite non-negative number", i);
      theta[i] = m->inv_freq[i];
    }
  } else {
    if (!(m->rope_theta > 1.0) || !std::isfinite(m->rope_theta))
      return fail(nullptr, PIC_ERR_INVALID_ARG, "rope_theta must be > 1");
    // theta_i = b^(-2i/d): EPIC Guide, "Mathematical Foundations", 1.
    for (int32_t i = 0; i < half; ++i)
      theta[i] = std::pow(m->rope_theta, -2.0 * static_cast<double>(i) / m->rope_dim);
    if (m->scaling == PIC_SCALING_LLAMA3) {
      // Llama-3.1 rescaling (public rule; not on the pages).
      const double orig = m->llama3_orig_max_pos, lo = m->llama3_low_freq_factor,
                   hi = m->llama3_high_freq_factor, factor = m->llama3_factor;
      if (!(orig > 0 && lo > 0 && hi > lo && factor > 0))
        return fail(nullptr, PIC_ERR_INVALID_ARG, "bad llama3 scaling parameters");
      const double low_wavelen = orig / lo, high_wavelen = orig / hi;
      for (int32_t i = 0; i < half; ++i) {
        const double wavelen = 2.0 * kPi / theta[i];
        if (wavelen < high_wavelen) continue;
        if (wavelen > low_wavelen) {
          theta[i] = theta[i] / factor;
        } else {
          const double s = (orig / wavelen - lo) / (hi - lo);
          theta[i] = (1.0 - s) * theta[i] / factor + s * theta[i];
        }
      }
    } else if (m->scaling != PIC_SCALING_NONE) {
      return fail(nullptr, PIC_ERR_INVALID_ARG, "unknown scaling %d", m->scaling);
    }
  }
  pic_ctx* ctx = new (std::nothrow) pic_ctx(num_cache_blocks);
  if (!ctx) return fail(nullptr, PIC_ERR_INVALID_ARG, "out of host memory");
  ctx->model = *m;
  {
    // Default: the bulk-copy pipeline for MLA rows (it keeps the 512-d latent
    // out of registers and wins there), the register kernel for GQA rows
    // (faster there).  PIC_KERNEL=regs or =bulk forces one variant.
    const char* kv = std::getenv("PIC_KERNEL");
    const bool regs_only = kv && std::strcmp(kv, "regs") == 0;
    const bool bulk_all = kv && std::strcmp(kv, "bulk") == 0;
    const int64_t tile_bytes = pic::kTmaTileBytesPerTensor;
    const int64_t row = row_bytes_of(*m);
    if (!regs_only && (bulk_all || m->kind == PIC_KIND_MLA)) {
      ctx->tma_stitch = tma_config_for(row, m->block_size, m->kind == PIC_KIND_GQA ? 2 : 1, tile_bytes,
                                       ctx->tma_stitch_cfg);
    }
    // An MLA shift touches only the 64-d rope slice of each row: the register
    // kernel reads just those bytes, whole-row copies would move 9x more.
    if (bulk_all && m->kind == PIC_KIND_GQA) {
      ctx->tma_inplace = tma_config_for(row, m->block_size, 1, tile_bytes, ctx->tma_inplace_cfg);
    }
    const char* ak = std::getenv("PIC_ATTEND_KERNEL");
    ctx->attend_tc = m->kind == PIC_KIND_MLA && !(ak && std::strcmp(ak, "mma") == 0);
  }
  ctx->model.inv_freq = nullptr;
  ctx->theta = theta;
  ctx->freq_turns.resize(half);
  for (int32_t i = 0; i < half; ++i) {
    const double f = theta[i] / (2.0 * kPi);
    const float fh = static_cast<float>(f);
    ctx->freq_turns[i] = make_float2(fh, static_cast<float>(f - static_cast<double>(fh)));
  }
  *out = ctx;
  return ok(nullptr);
}

void pic_destroy(pic_ctx* ctx) {
  if (!ctx) return;
  release_staging(ctx);
  release_attn_resident(ctx);
  release_copy_stream(ctx);
  for (pic_plan* p : ctx->plans) delete p;
  delete ctx;
}

// ------------------------------------------------------------------ registry

pic_status pic_register_chunk(pic_ctx* ctx, const uint8_t* key, int64_t pool_token_offset,
                              int32_t num_tokens, int32_t base_pos, int32_t* chunk_id,
                              int32_t* is_new) {
  if (!ctx) return fail(nullptr, PIC_ERR_INVALID_ARG, "null ctx");
  if (!key || !chunk_id) return fail(ctx, PIC_ERR_INVALID_ARG, "null key or chunk_id");
  if (num_tokens < 0 || pool_token_offset < 0 || base_pos < 0)
    return fail(ctx, PIC_ERR_RANGE, "negative offset, length or base_pos");
  if (pool_token_offset + num_tokens > std::numeric_limits<int32_t>::max())
    return fail(ctx, PIC_ERR_RANGE, "pool rows beyond 2^31 tokens");
  std::array<uint8_t, PIC_KEY_BYTES> k;
  std::memcpy(k.data(), key, PIC_KEY_BYTES);
  auto it = ctx->by_key.find(k);
  if (it != ctx->by_key.end()) {
    const ChunkEntry& e = ctx->chunks[it->second];
    if (e.in_blocks)
      return fail(ctx, PIC_ERR_KEY_CONFLICT, "key already registered as block-resident chunk %d", it->second);
    if (e.num_tokens != num_tokens || e.base_pos != base_pos)
      return fail(ctx, PIC_ERR_KEY_CONFLICT,
                  "key already registered as chunk %d with %d tokens at base %d", it->second,
                  e.num_tokens, e.base_pos);
    *chunk_id = it->second;
    if (is_new) *is_new = 0;
    return ok(ctx);
  }
  const int32_t id = static_cast<int32_t>(ctx->chunks.size());
  ctx->chunks.push_back(ChunkEntry{k, pool_token_offset, num_tokens, base_pos, true});
  ctx->by_key.emplace(k, id);
  *chunk_id = id;
  if (is_new) *is_new = 1;
  return ok(ctx);
}

pic_status pic_register_chunk_blocks(pic_ctx* ctx, const uint8_t* key, const int32_t* blocks,
                                     int32_t num_tokens, int32_t base_pos, int32_t* chunk_id, int32_t* is_new) {
  if (!ctx) return fail(nullptr, PIC_ERR_INVALID_ARG, "null ctx");
  if (!key || !chunk_id || !blocks) return fail(ctx, PIC_ERR_INVALID_ARG, "null key, blocks or chunk_id");
  if (num_tokens <= 0 || base_pos < 0) return fail(ctx, PIC_ERR_RANGE, "num_tokens must be > 0 and base_pos >= 0");
  const int64_t bs = ctx->model.block_size;
  const int64_t nb64 = (static_cast<int64_t>(num_tokens) + bs - 1) / bs;
  // Checked before blocks[] is read: a chunk cannot hold more blocks than the cache has.
  if (nb64 > ctx->num_cache_blocks)
    return fail(ctx, PIC_ERR_RANGE, "chunk of %d tokens needs %lld blocks, the cache has %d", num_tokens,
                static_cast<long long>(nb64), ctx->num_cache_blocks);
  const int32_t nb = static_cast<int32_t>(nb64);
  std::vector<int32_t> ids(blocks, blocks + nb);
  std::array<uint8_t, PIC_KEY_BYTES> k;
  std::memcpy(k.data(), key, PIC_KEY_BYTES);
  auto it = ctx->by_key.find(k);
  if (it != ctx->by_key.end()) {
    const ChunkEntry& e = ctx->chunks[it->second];
    if (!e.in_blocks || e.num_tokens != num_tokens || e.blocks != ids)
      return fail(ctx, PIC_ERR_KEY_CONFLICT, "key already registered as chunk %d with other tokens or blocks",
                  it->second);
    *chunk_id = it->second;
    if (is_new) *is_new = 0;
    return ok(ctx);
  }
  std::vector<int32_t> sorted = ids;
  std::sort(sorted.begin(), sorted.end());
  for (int32_t i = 0; i < nb; ++i) {
    if (!ctx->alloc.is_free(sorted[i]))
      return fail(ctx, PIC_ERR_RANGE, "block %d is outside the cache or not free", sorted[i]);
    if (i > 0 && sorted[i] == sorted[i - 1]) return fail(ctx, PIC_ERR_INVALID_ARG, "block %d listed twice", sorted[i]);
  }
  ctx->alloc.take(ids);
  const int32_t id = static_cast<int32_t>(ctx->chunks.size());
  ChunkEntry e{k, -1, num_tokens, base_pos, true};
  e.in_blocks = true;
  e.blocks = std::move(ids);
  ctx->chunks.push_back(std::move(e));
  ctx->by_key.emplace(k, id);
  *chunk_id = id;
  if (is_new) *is_new = 1;
  return ok(ctx);
}

pic_status pic_lookup_chunk(const pic_ctx* cctx, const uint8_t* key, int32_t* chunk_id) {
  pic_ctx* ctx = const_cast<pic_ctx*>(cctx);
  if (!ctx) return fail(nullptr, PIC_ERR_INVALID_ARG, "null ctx");
  if (!key || !chunk_id) return fail(ctx, PIC_ERR_INVALID_ARG, "null key or chunk_id");
  std::array<uint8_t, PIC_KEY_BYTES> k;
  std::memcpy(k.data(), key, PIC_KEY_BYTES);
  auto it = ctx->by_key.find(k);
  if (it == ctx->by_key.end()) return fail(ctx, PIC_ERR_UNKNOWN_CHUNK, "key not registered");
  *chunk_id = it->second;
  return ok(ctx);
}

pic_status pic_chunk_info(const pic_ctx* cctx, int32_t id, int64_t* pool_token_offset,
                          int32_t* num_tokens, int32_t* base_pos) {
  pic_ctx* ctx = const_cast<pic_ctx*>(cctx);
  if (!ctx) return fail(nullptr, PIC_ERR_INVALID_ARG, "null ctx");
  if (id < 0 || id >= static_cast<int32_t>(ctx->chunks.size()) || !ctx->chunks[id].live)
    return fail(ctx, PIC_ERR_UNKNOWN_CHUNK, "no chunk %d", id);
  const ChunkEntry& e = ctx->chunks[id];
  if (pool_token_offset) *pool_token_offset = e.pool_token_offset;
  if (num_tokens) *num_tokens = e.num_tokens;
  if (base_pos) *base_pos = e.base_pos;
  return ok(ctx);
}

pic_status pic_unregister_chunk(pic_ctx* ctx, int32_t id) {
  if (!ctx) return fail(nullptr, PIC_ERR_INVALID_ARG, "null ctx");
  if (id < 0 || id >= static_cast<int32_t>(ctx->chunks.size()) || !ctx->chunks[id].live)
    return fail(ctx, PIC_ERR_UNKNOWN_CHUNK, "no chunk %d", id);
  ChunkEntry& ce = ctx->chunks[id];
  if (ce.in_blocks) {
    if (ce.refs > 0) return fail(ctx, PIC_ERR_BUSY, "chunk %d is used by %d live request(s)", id, ce.refs);
    ctx->alloc.release(ce.blocks);
    ce.blocks.clear();
  }
  ctx->chunks[id].live = false;
  ctx->by_key.erase(ctx->chunks[id].key);
  return ok(ctx);
}

// ------------------------------------------------------------- plan + table

pic_status pic_build_block_table(pic_ctx* ctx, const pic_request_desc* rq, int32_t* bt_out,
                                 int32_t max_blocks, pic_plan** plan_out) {
  if (!ctx) return fail(nullptr, PIC_ERR_INVALID_ARG, "null ctx");
  if (!rq || !plan_out) return fail(ctx, PIC_ERR_INVALID_ARG, "null request or plan_out");
  if (rq->n_chunks < 0 || (rq->n_chunks > 0 && !rq->chunk_ids))
    return fail(ctx, PIC_ERR_INVALID_ARG, "bad chunk list");
  if (rq->k_nonleading < 0 || rq->k_leading < 0 || rq->start_pos < 0 || rq->total_tokens < 0)
    return fail(ctx, PIC_ERR_RANGE, "negative k, start_pos or total_tokens");
  if (max_blocks < 0 || (max_blocks > 0 && !bt_out))
    return fail(ctx, PIC_ERR_INVALID_ARG, "bad block table output");

  // Compose: EPIC Guide, "Algorithmic Architecture" 2. Modular Prompt Composer.
  const int64_t bs = ctx->model.block_size;
  std::unordered_map<int32_t, int32_t> occurrences;
  for (int32_t j = 0; j < rq->n_chunks; ++j) ++occurrences[rq->chunk_ids[j]];
  std::vector<Segment> segs;
  segs.reserve(rq->n_chunks);
  int64_t pos = rq->start_pos;
  int64_t prev_end = -1;
  int64_t n_recompute = 0;
  for (int32_t j = 0; j < rq->n_chunks; ++j) {
    const int32_t id = rq->chunk_ids[j];
    if (id < 0 || id >= static_cast<int32_t>(ctx->chunks.size()) || !ctx->chunks[id].live)
      return fail(ctx, PIC_ERR_UNKNOWN_CHUNK, "chunk %d (position %d in the request) is not registered", id, j);
    const ChunkEntry& e = ctx->chunks[id];
    if (e.in_blocks && e.mapped_by != nullptr)
      return fail(ctx, PIC_ERR_BUSY, "chunk %d is mapped by a live request; free it first", id);
    const int32_t n = rq->take_tokens ? rq->take_tokens[j] : e.num_tokens;
    if (n < 0 || n > e.num_tokens)
      return fail(ctx, PIC_ERR_RANGE, "take_tokens[%d] = %d outside [0, %d]", j, n, e.num_tokens);
    const int64_t p = rq->dst_pos ? rq->dst_pos[j] : pos;
    if (p < 0 || (prev_end >= 0 && p < prev_end))
      return fail(ctx, PIC_ERR_RANGE, "chunk %d at position %lld overlaps the previous chunk (ends %lld)", j,
                  static_cast<long long>(p), static_cast<long long>(prev_end));
    if (p + n > std::numeric_limits<int32_t>::max())
      return fail(ctx, PIC_ERR_RANGE, "positions beyond int32");
    // delta = p_target - p_source (Irminsul, 2.2 delta-Rotation Rule); for a
    // block-resident chunk p_source is where its keys sit now.
    const int64_t delta = p - e.base_pos;
    if (delta > PIC_MAX_ABS_DELTA || delta < -PIC_MAX_ABS_DELTA)
      return fail(ctx, PIC_ERR_RANGE, "|delta| of chunk %d exceeds 2^24 - 1", j);
    // recompute count: LegoLink sinks of non-leading chunks; Irminsul carve-out at position 0
    const int32_t k = (p == 0) ? rq->k_leading : rq->k_nonleading;
    const int32_t nr = std::min(k, n);
    Segment sg{id, e.in_blocks ? -1 : e.pool_token_offset, n, static_cast<int32_t>(p), static_cast<int32_t>(delta),
               nr, pic::kRunPool, {}};
    if (e.in_blocks) {
      // EPIC runtime figure, step 1 "Virtual Block Mapping": reuse the chunk's
      // blocks when it starts on a block boundary, is taken whole, occurs once
      // here and no other live request uses it; otherwise copy it out.
      const bool map = rq->alias && p % bs == 0 && n == e.num_tokens && occurrences[id] == 1 && e.refs == 0;
      sg.kind = map ? pic::kRunInPlace : pic::kRunBlocks;
      if (!map) sg.src_blocks = e.blocks;
    }
    segs.push_back(std::move(sg));
    n_recompute += nr;
    pos = p + n;
    prev_end = pos;
  }
  const int64_t end = segs.empty() ? rq->start_pos : pos;
  if (rq->total_tokens > 0 && rq->total_tokens < end)
    return fail(ctx, PIC_ERR_RANGE, "total_tokens %d is before the end of the last chunk (%lld)",
                rq->total_tokens, static_cast<long long>(end));
  const int64_t total = rq->total_tokens > 0 ? rq->total_tokens : end;
  const int64_t nblocks = (total + bs - 1) / bs;
  if (nblocks > max_blocks)
    return fail(ctx, PIC_ERR_CAPACITY, "request needs %lld blocks, table holds %d",
                static_cast<long long>(nblocks), max_blocks);
  if (n_recompute > std::numeric_limits<int32_t>::max())
    return fail(ctx, PIC_ERR_RANGE, "recompute list too long");

  // Logical blocks served by mapped chunks keep the chunk's blocks; the rest
  // are fresh, lowest free id first.
  std::vector<int32_t> table(static_cast<size_t>(nblocks), -1);
  for (const Segment& sg : segs) {
    if (sg.kind != pic::kRunInPlace) continue;
    const ChunkEntry& e = ctx->chunks[sg.chunk_id];
    for (size_t b = 0; b < e.blocks.size(); ++b) table[sg.dst_pos / bs + b] = e.blocks[b];
  }
  int32_t need = 0;
  for (int32_t v : table) need += v < 0;
  pic_plan* plan = new (std::nothrow) pic_plan();
  if (!plan) return fail(ctx, PIC_ERR_INVALID_ARG, "out of host memory");
  if (!ctx->alloc.allocate(need, plan->fresh)) {
    delete plan;
    return fail(ctx, PIC_ERR_OUT_OF_BLOCKS, "request needs %d fresh blocks, %d free", need, ctx->alloc.free_count());
  }
  for (size_t i = 0, f = 0; i < table.size(); ++i)
    if (table[i] < 0) table[i] = plan->fresh[f++];
  plan->owner = ctx;
  plan->serial = ++ctx->plan_serial;
  plan->table = std::move(table);
  plan->segs = std::move(segs);
  plan->total_tokens = static_cast<int32_t>(total);
  plan->n_recompute = static_cast<int32_t>(n_recompute);
  // Registry: block-resident chunks gain a user; mapped ones move to their new position.
  for (const Segment& sg : plan->segs) {
    ChunkEntry& e = ctx->chunks[sg.chunk_id];
    if (!e.in_blocks) continue;
    ++e.refs;
    if (sg.kind == pic::kRunInPlace) {
      plan->undo.emplace_back(sg.chunk_id, e.base_pos);
      plan->has_mapped = true;
      e.mapped_by = plan;
      e.base_pos = sg.dst_pos;
    }
  }
  for (int32_t i = 0; i < max_blocks; ++i)
    bt_out[i] = i < static_cast<int32_t>(plan->table.size()) ? plan->table[i] : -1;
  ctx->plans.insert(plan);
  *plan_out = plan;
  return ok(ctx);
}

pic_status pic_free_request(pic_ctx* ctx, pic_plan* plan) {
  if (!ctx) return fail(nullptr, PIC_ERR_INVALID_ARG, "null ctx");
  if (!plan_valid(ctx, plan)) return fail(ctx, PIC_ERR_INVALID_ARG, "plan does not belong to this context");
  if (!plan->applied)
    for (const auto& u : plan->undo) ctx->chunks[u.first].base_pos = u.second;  // rotation never enqueued
  for (const Segment& sg : plan->segs) {
    ChunkEntry& e = ctx->chunks[sg.chunk_id];
    if (!e.in_blocks) continue;
    --e.refs;
    if (sg.kind == pic::kRunInPlace) e.mapped_by = nullptr;
  }
  ctx->alloc.release(plan->fresh);
  ctx->plans.erase(plan);
  delete plan;
  return ok(ctx);
}

pic_status pic_plan_info(const pic_plan* p, int32_t* total_tokens, int32_t* num_blocks,
                         int32_t* num_segments, int32_t* num_recompute) {
  if (!p) return fail(nullptr, PIC_ERR_INVALID_ARG, "null plan");
  if (total_tokens) *total_tokens = p->total_tokens;
  if (num_blocks) *num_blocks = static_cast<int32_t>(p->table.size());
  if (num_segments) *num_segments = static_cast<int32_t>(p->segs.size());
  if (num_recompute) *num_recompute = p->n_recompute;
  return ok(nullptr);
}

pic_status pic_plan_segment(const pic_plan* p, int32_t j, int32_t* chunk_id, int64_t* src_token,
                            int32_t* num_tokens, int32_t* dst_pos, int32_t* delta) {
  if (!p) return fail(nullptr, PIC_ERR_INVALID_ARG, "null plan");
  if (j < 0 || j >= static_cast<int32_t>(p->segs.size()))
    return fail(nullptr, PIC_ERR_RANGE, "segment %d out of range", j);
  const Segment& s = p->segs[j];
  if (chunk_id) *chunk_id = s.chunk_id;
  if (src_token) *src_token = s.src_tok;
  if (num_tokens) *num_tokens = s.num_tokens;
  if (dst_pos) *dst_pos = s.dst_pos;
  if (delta) *delta = s.delta;
  return ok(nullptr);
}

int32_t pic_plan_segment_mode(const pic_plan* p, int32_t j) {
  if (!p || j < 0 || j >= static_cast<int32_t>(p->segs.size())) return -1;
  return p->segs[j].kind;  // PIC_SEG_* values equal the run kinds
}

// -------------------------------------------------------------- recompute

pic_status pic_recompute_indices(const pic_plan* const* plans, int32_t n_req, int32_t* idx_out,
                                 int32_t* indptr_out, int64_t capacity, int64_t* count) {
  if (n_req < 0 || (n_req > 0 && !plans)) return fail(nullptr, PIC_ERR_INVALID_ARG, "bad plan list");
  int64_t total = 0;
  for (int32_t r = 0; r < n_req; ++r) {
    if (!plans[r]) return fail(nullptr, PIC_ERR_INVALID_ARG, "plans[%d] is null", r);
    total += plans[r]->n_recompute;
  }
  if (count) *count = total;
  if (total > std::numeric_limits<int32_t>::max())
    return fail(nullptr, PIC_ERR_RANGE, "recompute list of %lld entries: CSR offsets are int32",
                static_cast<long long>(total));
  if (!idx_out) return ok(nullptr);
  if (total > capacity) return fail(nullptr, PIC_ERR_CAPACITY, "recompute list has %lld entries, capacity %lld",
                                    static_cast<long long>(total), static_cast<long long>(capacity));
  int64_t w = 0;
  for (int32_t r = 0; r < n_req; ++r) {
    if (indptr_out) indptr_out[r] = static_cast<int32_t>(w);
    for (const Segment& s : plans[r]->segs)
      for (int32_t t = 0; t < s.n_recompute; ++t) idx_out[w++] = s.dst_pos + t;
  }
  if (indptr_out) indptr_out[n_req] = static_cast<int32_t>(w);
  return ok(nullptr);
}

// ------------------------------------------------------------------- stitch

size_t pic_workspace_bytes(const pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req) {
  if (!ctx || n_req < 0 || (n_req > 0 && !plans)) return 0;
  for (int32_t r = 0; r < n_req; ++r)
    if (!plans[r]) return 0;
  const size_t runs = count_stitch_runs(ctx, plans, n_req);
  return ws_layout(ctx->freq_turns.size(), static_cast<size_t>(n_req) + 1, runs).total;
}

pic_status pic_stitch(pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req,
                      const void* k_pool, const void* v_pool, int64_t pool_ls, void* k_cache,
                      void* v_cache, int64_t cache_ls, const int32_t* d_bt, int32_t max_blocks,
                      int32_t* d_ridx, int32_t* d_indptr, int64_t recompute_capacity,
                      void* d_ws, size_t ws_bytes, pic_stream_t stream) {
  if (!ctx) return fail(nullptr, PIC_ERR_INVALID_ARG, "null ctx");
  pic_status st = check_stitch_args(ctx, plans, n_req, k_pool, v_pool, pool_ls, k_cache, v_cache, cache_ls,
                                    d_bt, max_blocks, d_ridx, d_indptr, recompute_capacity);
  if (st != PIC_OK) return st;
  if (!d_ws) return fail(ctx, PIC_ERR_INVALID_ARG, "null workspace");
  if (!vectorized_bytes_ok(d_ws)) return fail(ctx, PIC_ERR_ALIGNMENT, "workspace must be 16-byte aligned");
  const size_t n_runs = count_stitch_runs(ctx, plans, n_req);
  const WsLayout w = ws_layout(ctx->freq_turns.size(), static_cast<size_t>(n_req) + 1, n_runs);
  if (ws_bytes < w.total)
    return fail(ctx, PIC_ERR_CAPACITY, "workspace has %zu bytes, needs %zu", ws_bytes, w.total);
  if (n_runs > static_cast<size_t>(std::numeric_limits<int32_t>::max()))
    return fail(ctx, PIC_ERR_RANGE, "too many runs");

  DeviceInfo di;
  st = current_device(ctx, di);
  if (st != PIC_OK) return st;
  const void* bufs[4] = {k_pool, v_pool, k_cache, v_cache};
  const int host_io = host_buffers(ctx, bufs, 4);
  if (host_io < 0) return PIC_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  StagingSlot* sl = nullptr;
  st = acquire_staging(ctx, di.device, w.total, &sl);
  if (st != PIC_OK) return st;
  build_stitch_image(ctx, plans, n_req, sl->host, w);
  st = upload_staging(ctx, sl, d_ws, w.total, s);
  if (st != PIC_OK) return st;

  pic::KernelParams p{};
  fill_stitch_params(ctx, p, static_cast<uint8_t*>(d_ws), w, n_runs, n_req, k_pool, v_pool, pool_ls, k_cache,
                     v_cache, cache_ls, d_bt, max_blocks, d_ridx, d_indptr);
  p.debug_stall = ctx->debug_stall;
  p.max_spins = ctx->debug_spins;
  ctx->debug_stall = 0;
  ctx->debug_spins = 0;
  const cudaError_t e = launch_stitch_kernel(ctx, p, di.sm_count, s, host_io != 0, mostly_in_place(plans, n_req));
  if (e != cudaSuccess) return cuda_fail(ctx, e, "stitch launch");
  for (int32_t r = 0; r < n_req; ++r) const_cast<pic_plan*>(plans[r])->applied = true;
  return ok(ctx);
}

// ---------------------------------------------------- pools in host memory

namespace {

// The pool rows [begin, end) the plans' pool segments read, sorted and
// merged (overlapping or adjacent ranges become one); *rows_read counts
// every row read, repeats included.
std::vector<std::pair<int64_t, int64_t>> pool_read_ranges(const pic_plan* const* plans, int32_t n_req,
                                                          int64_t* rows_read) {
  std::vector<std::pair<int64_t, int64_t>> v;
  int64_t read = 0;
  for (int32_t r = 0; r < n_req; ++r)
    for (const Segment& sg : plans[r]->segs)
      if (sg.kind == pic::kRunPool && sg.num_tokens > 0) {
        v.emplace_back(sg.src_tok, sg.src_tok + sg.num_tokens);
        read += sg.num_tokens;
      }
  std::sort(v.begin(), v.end());
  std::vector<std::pair<int64_t, int64_t>> merged;
  for (const auto& x : v) {
    if (!merged.empty() && x.first <= merged.back().second)
      merged.back().second = std::max(merged.back().second, x.second);
    else
      merged.push_back(x);
  }
  if (rows_read) *rows_read = read;
  return merged;
}

// The rows of `a` outside `b` (both sorted and merged), sorted and merged.
std::vector<std::pair<int64_t, int64_t>> minus_ranges(const std::vector<std::pair<int64_t, int64_t>>& a,
                                                      const std::vector<std::pair<int64_t, int64_t>>& b) {
  std::vector<std::pair<int64_t, int64_t>> out;
  size_t j = 0;
  for (const auto& x : a) {
    int64_t lo = x.first;
    while (j < b.size() && b[j].second <= lo) ++j;
    for (size_t k = j; k < b.size() && b[k].first < x.second; ++k) {
      if (b[k].first > lo) out.emplace_back(lo, b[k].first);
      lo = std::max(lo, b[k].second);
    }
    if (lo < x.second) out.emplace_back(lo, x.second);
  }
  return out;
}

pic_status check_plan_list(pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req) {
  if (n_req < 0 || (n_req > 0 && !plans)) return fail(ctx, PIC_ERR_INVALID_ARG, "bad plan list");
  for (int32_t r = 0; r < n_req; ++r)
    if (!plan_valid(ctx, plans[r])) return fail(ctx, PIC_ERR_INVALID_ARG, "plans[%d] does not belong to this context", r);
  return PIC_OK;
}

}  // namespace

pic_status pic_pool_read_rows(const pic_ctx* cctx, const pic_plan* const* plans, int32_t n_req,
                              const pic_plan* const* staged_plans, int32_t n_staged, int64_t* distinct_rows,
                              int64_t* rows_read) {
  pic_ctx* ctx = const_cast<pic_ctx*>(cctx);
  if (!ctx) return fail(nullptr, PIC_ERR_INVALID_ARG, "null ctx");
  pic_status st = check_plan_list(ctx, plans, n_req);
  if (st != PIC_OK) return st;
  st = check_plan_list(ctx, staged_plans, n_staged);
  if (st != PIC_OK) return st;
  int64_t read = 0, distinct = 0;
  for (const auto& x : minus_ranges(pool_read_ranges(plans, n_req, &read), pool_read_ranges(staged_plans, n_staged, nullptr)))
    distinct += x.second - x.first;
  if (distinct_rows) *distinct_rows = distinct;
  if (rows_read) *rows_read = read;
  return ok(ctx);
}

namespace {

// Host and device pools of a staging call, checked.
struct StagePools {
  const void* host[2];
  void* dev[2];
  int64_t host_ls, dev_ls;
  int tensors;
};

// Checks the pools of a staging call that need no CUDA call (null,
// GQA/MLA values, alignment, strides reaching row `top`).
pic_status check_stage_pools(pic_ctx* ctx, const StagePools& sp, int64_t top) {
  const pic_model_desc& m = ctx->model;
  const bool gqa = m.kind == PIC_KIND_GQA;
  if (!sp.host[0] || !sp.dev[0]) return fail(ctx, PIC_ERR_INVALID_ARG, "null pool");
  if (gqa && (!sp.host[1] || !sp.dev[1])) return fail(ctx, PIC_ERR_INVALID_ARG, "GQA needs both value pools");
  if (!gqa && (sp.host[1] || sp.dev[1])) return fail(ctx, PIC_ERR_INVALID_ARG, "MLA rows have no separate values (pass NULL)");
  for (int k = 0; k < sp.tensors; ++k)
    if (!vectorized_bytes_ok(sp.host[k]) || !vectorized_bytes_ok(sp.dev[k]))
      return fail(ctx, PIC_ERR_ALIGNMENT, "pools and layer strides must be 16-byte aligned");
  if ((sp.host_ls & 15) || (sp.dev_ls & 15))
    return fail(ctx, PIC_ERR_ALIGNMENT, "pools and layer strides must be 16-byte aligned");
  const int64_t row = row_bytes_of(m);
  if (m.num_layers > 1 && (sp.host_ls < top * row || sp.dev_ls < top * row))
    return fail(ctx, PIC_ERR_RANGE, "a layer stride is smaller than the %lld pool rows the plans reach",
                static_cast<long long>(top));
  return PIC_OK;
}

// Where the pools live: pinned host memory and device memory (CUDA calls).
pic_status check_stage_residency(pic_ctx* ctx, const StagePools& sp) {
  for (int k = 0; k < sp.tensors; ++k) {
    if (residency(sp.host[k]) != 1)
      return fail(ctx, PIC_ERR_INVALID_ARG, "host pools must be pinned host memory (cudaHostAlloc / cudaHostRegister)");
    if (residency(sp.dev[k]) != 0) return fail(ctx, PIC_ERR_INVALID_ARG, "device pools must be device memory");
  }
  return PIC_OK;
}

// Enqueues the copy kernel over `ranges` (pool rows), every layer and tensor,
// on stream s: one launch per kStageMaxSpans ranges.  Adds the bytes to *bytes.
pic_status launch_stage_ranges(pic_ctx* ctx, const StagePools& sp, const std::vector<std::pair<int64_t, int64_t>>& ranges,
                               int sm_count, cudaStream_t s, int64_t* bytes) {
  const int64_t row = row_bytes_of(ctx->model);
  const int32_t L = ctx->model.num_layers;
  auto prm = std::make_unique<pic::StageParams>();
  for (int k = 0; k < 2; ++k) {
    prm->src[k] = static_cast<const uint8_t*>(sp.host[k]);
    prm->dst[k] = static_cast<uint8_t*>(sp.dev[k]);
  }
  prm->src_ls = sp.host_ls;
  prm->dst_ls = sp.dev_ls;
  prm->layers = L;
  prm->tensors = sp.tensors;
  for (size_t r0 = 0; r0 < ranges.size(); r0 += pic::kStageMaxSpans) {
    const size_t n = std::min<size_t>(pic::kStageMaxSpans, ranges.size() - r0);
    for (size_t i = 0; i < n; ++i) {
      prm->spans[i].off = ranges[r0 + i].first * row;
      prm->spans[i].bytes = (ranges[r0 + i].second - ranges[r0 + i].first) * row;
      *bytes += prm->spans[i].bytes * L * sp.tensors;
    }
    prm->n_spans = static_cast<int32_t>(n);
    const int64_t items = static_cast<int64_t>(n) * L * sp.tensors;
    const cudaError_t e = pic::launch_stage_rows(*prm, static_cast<int>(std::min<int64_t>(items, sm_count)), s);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "pool staging launch");
  }
  return PIC_OK;
}

// The request groups of a staged stitch: [bounds[g], bounds[g + 1]).
std::vector<int32_t> group_bounds(int32_t n_req, int32_t n_groups) {
  const int32_t G = std::max<int32_t>(1, std::min(n_groups, n_req));
  std::vector<int32_t> b(G + 1);
  for (int32_t g = 0; g <= G; ++g) b[g] = static_cast<int32_t>(static_cast<int64_t>(n_req) * g / G);
  return b;
}

// A group's workspace layout, its offset in the workspace and its runs.
struct GroupLayout {
  WsLayout w;
  size_t off;
  size_t runs;
};

std::vector<GroupLayout> group_layouts(const pic_ctx* ctx, const pic_plan* const* plans, const std::vector<int32_t>& b,
                                       size_t* total) {
  std::vector<GroupLayout> out;
  size_t off = 0;
  for (size_t g = 0; g + 1 < b.size(); ++g) {
    const int32_t n = b[g + 1] - b[g];
    const size_t runs = count_stitch_runs(ctx, plans + b[g], n);
    const WsLayout w = ws_layout(ctx->freq_turns.size(), static_cast<size_t>(n) + 1, runs);
    out.push_back(GroupLayout{w, off, runs});
    off += w.total;
  }
  *total = off;
  return out;
}

}  // namespace

pic_status pic_stage_pool(pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req,
                          const pic_plan* const* staged_plans, int32_t n_staged,
                          const void* host_k_pool, const void* host_v_pool, int64_t host_ls,
                          void* dev_k_pool, void* dev_v_pool, int64_t dev_ls, int64_t* bytes_copied,
                          pic_stream_t stream) {
  if (!ctx) return fail(nullptr, PIC_ERR_INVALID_ARG, "null ctx");
  pic_status st = check_plan_list(ctx, plans, n_req);
  if (st != PIC_OK) return st;
  st = check_plan_list(ctx, staged_plans, n_staged);
  if (st != PIC_OK) return st;
  const StagePools sp{{host_k_pool, host_v_pool}, {dev_k_pool, dev_v_pool}, host_ls, dev_ls,
                      ctx->model.kind == PIC_KIND_GQA ? 2 : 1};
  const auto ranges = minus_ranges(pool_read_ranges(plans, n_req, nullptr), pool_read_ranges(staged_plans, n_staged, nullptr));
  st = check_stage_pools(ctx, sp, ranges.empty() ? 0 : ranges.back().second);
  if (st != PIC_OK) return st;
  DeviceInfo di;
  st = current_device(ctx, di);
  if (st != PIC_OK) return st;
  st = check_stage_residency(ctx, sp);
  if (st != PIC_OK) return st;
  int64_t bytes = 0;
  st = launch_stage_ranges(ctx, sp, ranges, di.sm_count, reinterpret_cast<cudaStream_t>(stream), &bytes);
  if (st != PIC_OK) return st;
  if (bytes_copied) *bytes_copied = bytes;
  return ok(ctx);
}

size_t pic_stitch_staged_workspace_bytes(const pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req,
                                         int32_t n_groups) {
  if (!ctx || n_req < 0 || (n_req > 0 && !plans) || n_groups < 1) return 0;
  for (int32_t r = 0; r < n_req; ++r)
    if (!plans[r]) return 0;
  size_t total = 0;
  group_layouts(ctx, plans, group_bounds(n_req, n_groups), &total);
  return total;
}

pic_status pic_stitch_staged(pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req, int32_t n_groups,
                             const void* host_k_pool, const void* host_v_pool, int64_t host_ls,
                             void* dev_k_pool, void* dev_v_pool, int64_t dev_ls, void* k_cache, void* v_cache,
                             int64_t cache_ls, const int32_t* d_bt, int32_t max_blocks, int32_t* d_ridx,
                             int32_t* d_indptr, int64_t recompute_capacity, void* d_ws, size_t ws_bytes,
                             int64_t* bytes_staged, pic_stream_t stream) {
  if (!ctx) return fail(nullptr, PIC_ERR_INVALID_ARG, "null ctx");
  if (n_groups < 1) return fail(ctx, PIC_ERR_INVALID_ARG, "n_groups must be >= 1");
  pic_status st = check_stitch_args(ctx, plans, n_req, dev_k_pool, dev_v_pool, dev_ls, k_cache, v_cache, cache_ls,
                                    d_bt, max_blocks, d_ridx, d_indptr, recompute_capacity);
  if (st != PIC_OK) return st;
  const StagePools sp{{host_k_pool, host_v_pool}, {dev_k_pool, dev_v_pool}, host_ls, dev_ls,
                      ctx->model.kind == PIC_KIND_GQA ? 2 : 1};
  const auto all = pool_read_ranges(plans, n_req, nullptr);
  st = check_stage_pools(ctx, sp, all.empty() ? 0 : all.back().second);
  if (st != PIC_OK) return st;
  if (!d_ws) return fail(ctx, PIC_ERR_INVALID_ARG, "null workspace");
  if (!vectorized_bytes_ok(d_ws)) return fail(ctx, PIC_ERR_ALIGNMENT, "workspace must be 16-byte aligned");
  const std::vector<int32_t> b = group_bounds(n_req, n_groups);
  size_t need = 0;
  const auto lay = group_layouts(ctx, plans, b, &need);
  if (ws_bytes < need) return fail(ctx, PIC_ERR_CAPACITY, "workspace has %zu bytes, needs %zu", ws_bytes, need);
  for (const GroupLayout& x : lay)
    if (x.runs > static_cast<size_t>(std::numeric_limits<int32_t>::max())) return fail(ctx, PIC_ERR_RANGE, "too many runs");

  DeviceInfo di;
  st = current_device(ctx, di);
  if (st != PIC_OK) return st;
  st = check_stage_residency(ctx, sp);
  if (st != PIC_OK) return st;
  const void* bufs[2] = {k_cache, v_cache};
  const int host_io = host_buffers(ctx, bufs, 2);
  if (host_io < 0) return PIC_ERR_INVALID_ARG;
  if (ctx->copy_device != di.device) {
    release_copy_stream(ctx);
    cudaError_t e = cudaStreamCreateWithFlags(&ctx->copy_stream, cudaStreamNonBlocking);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaStreamCreate (staging)");
    e = cudaEventCreateWithFlags(&ctx->copy_event, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaEventCreate (staging)");
    ctx->copy_device = di.device;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream), cs = ctx->copy_stream;
  // the copies start after the work queued on the caller's stream before this call
  cudaError_t e = cudaEventRecord(ctx->copy_event, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, ctx->copy_event, 0);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "staging stream order");
  uint8_t* ws = static_cast<uint8_t*>(d_ws);
  int64_t bytes = 0;
  int64_t rec_base = 0;  // recompute entries of the groups before
  for (size_t g = 0; g + 1 < b.size(); ++g) {
    const int32_t r0 = b[g], n = b[g + 1] - b[g];
    // group g's rows that no earlier group read, on the copy stream; then the
    // caller's stream waits for them
    st = launch_stage_ranges(ctx, sp, minus_ranges(pool_read_ranges(plans + r0, n, nullptr), pool_read_ranges(plans, r0, nullptr)),
                             di.sm_count, cs, &bytes);
    if (st != PIC_OK) return st;
    e = cudaEventRecord(ctx->copy_event, cs);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ctx->copy_event, 0);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "staging stream order");
    // the group's stitch: its image numbers requests and recompute entries
    // from 0; the recompute offsets move by the earlier groups' entries, and
    // the kernel gets the group's block-table rows and CSR slots
    const WsLayout& w = lay[g].w;
    StagingSlot* sl = nullptr;
    st = acquire_staging(ctx, di.device, w.total, &sl);
    if (st != PIC_OK) return st;
    build_stitch_image(ctx, plans + r0, n, sl->host, w);
    int32_t* indptr = reinterpret_cast<int32_t*>(sl->host + w.indptr_off);
    for (int32_t i = 0; i <= n; ++i) indptr[i] += static_cast<int32_t>(rec_base);
    RunDesc* runs = reinterpret_cast<RunDesc*>(sl->host + w.runs_off);
    for (size_t k = 0; k < lay[g].runs; ++k) runs[k].idx_off += static_cast<int32_t>(rec_base);
    st = upload_staging(ctx, sl, ws + lay[g].off, w.total, s);
    if (st != PIC_OK) return st;
    pic::KernelParams p{};
    fill_stitch_params(ctx, p, ws + lay[g].off, w, lay[g].runs, n, dev_k_pool, dev_v_pool, dev_ls, k_cache, v_cache,
                       cache_ls, d_bt + static_cast<int64_t>(r0) * max_blocks, max_blocks, d_ridx,
                       d_indptr ? d_indptr + r0 : nullptr);
    p.header = reinterpret_cast<WsHeader*>(ws);  // one status word for the whole call: group 0's
    e = launch_stitch_kernel(ctx, p, di.sm_count, s, host_io != 0, mostly_in_place(plans + r0, n));
    if (e != cudaSuccess) return cuda_fail(ctx, e, "stitch launch");
    for (int32_t r = r0; r < r0 + n; ++r) rec_base += plans[r]->n_recompute;
  }
  for (int32_t r = 0; r < n_req; ++r) const_cast<pic_plan*>(plans[r])->applied = true;
  if (bytes_staged) *bytes_staged = bytes;
  return ok(ctx);
}

// ------------------------------------------------------------ in-place shift

size_t pic_rerotate_workspace_bytes(const pic_ctx* ctx, const pic_shift_seg* segs, int32_t n) {
  if (!ctx || n < 0 || (n > 0 && !segs)) return 0;
  return ws_layout(ctx->freq_turns.size(), 0, count_shift_runs(ctx, segs, n)).total;
}

pic_status pic_rerotate_inplace(pic_ctx* ctx, void* k_cache, int64_t cache_ls,
                                const int32_t* d_bt, int32_t n_tables, int32_t max_blocks,
                                const pic_shift_seg* segs, int32_t n_segs, void* d_ws,
                                size_t ws_bytes, pic_stream_t stream) {
  if (!ctx) return fail(nullptr, PIC_ERR_INVALID_ARG, "null ctx");
  const pic_model_desc& m = ctx->model;
  if (n_segs < 0 || (n_segs > 0 && !segs)) return fail(ctx, PIC_ERR_INVALID_ARG, "bad segment list");
  if (!k_cache || !d_bt || !d_ws) return fail(ctx, PIC_ERR_INVALID_ARG, "null cache, block table or workspace");
  if (n_tables < 0 || max_blocks < 0) return fail(ctx, PIC_ERR_INVALID_ARG, "bad block table shape");
  if (!vectorized_bytes_ok(k_cache) || (cache_ls & 15) || !vectorized_bytes_ok(d_ws))
    return fail(ctx, PIC_ERR_ALIGNMENT, "cache, layer stride and workspace must be 16-byte aligned");
  const int64_t row_bytes = row_bytes_of(m);
  if (cache_ls < 0 || (m.num_layers > 1 && cache_ls < static_cast<int64_t>(ctx->num_cache_blocks) * m.block_size * row_bytes))
    return fail(ctx, PIC_ERR_RANGE, "cache layer stride smaller than num_cache_blocks * block_size rows");
  const int32_t bs = m.block_size;
  for (int32_t i = 0; i < n_segs; ++i) {
    const pic_shift_seg& g = segs[i];
    if (g.req < 0 || g.req >= n_tables) return fail(ctx, PIC_ERR_RANGE, "segs[%d].req %d outside [0, %d)", i, g.req, n_tables);
    if (g.start_pos < 0 || g.num_tokens < 0) return fail(ctx, PIC_ERR_RANGE, "segs[%d] has a negative range", i);
    if (static_cast<int64_t>(g.start_pos) + g.num_tokens > static_cast<int64_t>(max_blocks) * bs)
      return fail(ctx, PIC_ERR_RANGE, "segs[%d] ends past the block table", i);
    if (static_cast<int64_t>(g.start_pos) + g.num_tokens > std::numeric_limits<int32_t>::max())
      return fail(ctx, PIC_ERR_RANGE, "segs[%d] ends past int32 positions", i);
    if (g.delta > PIC_MAX_ABS_DELTA || g.delta < -PIC_MAX_ABS_DELTA)
      return fail(ctx, PIC_ERR_RANGE, "segs[%d].delta exceeds 2^24 - 1", i);
  }
  const size_t n_runs = count_shift_runs(ctx, segs, n_segs);
  const WsLayout w = ws_layout(ctx->freq_turns.size(), 0, n_runs);
  if (ws_bytes < w.total) return fail(ctx, PIC_ERR_CAPACITY, "workspace has %zu bytes, needs %zu", ws_bytes, w.total);
  if (n_runs > static_cast<size_t>(std::numeric_limits<int32_t>::max())) return fail(ctx, PIC_ERR_RANGE, "too many runs");

  DeviceInfo di;
  pic_status st = current_device(ctx, di);
  if (st != PIC_OK) return st;
  const void* bufs[1] = {k_cache};
  const int host_io = host_buffers(ctx, bufs, 1);
  if (host_io < 0) return PIC_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  StagingSlot* sl = nullptr;
  st = acquire_staging(ctx, di.device, w.total, &sl);
  if (st != PIC_OK) return st;
  uint8_t* base = sl->host;
  fill_freq(ctx, base, w);
  std::vector<RunDesc> runs;
  runs.reserve(n_runs);
  const int32_t cap = inplace_cap(ctx);
  for (int32_t i = 0; i < n_segs; ++i) {
    const pic_shift_seg& g = segs[i];
    if (g.num_tokens <= 0 || g.delta == 0) continue;  // R_0 = I: nothing to do
    append_shift_runs(runs, g.start_pos, g.num_tokens, g.req, g.delta, bs, cap);
  }
  std::memcpy(base + w.runs_off, runs.data(), runs.size() * sizeof(RunDesc));
  st = upload_staging(ctx, sl, d_ws, w.total, s);
  if (st != PIC_OK) return st;
  if (n_runs == 0) return ok(ctx);

  uint8_t* ws = static_cast<uint8_t*>(d_ws);
  pic::KernelParams p{};
  set_geometry(ctx, p);
  p.runs = reinterpret_cast<const RunDesc*>(ws + w.runs_off);
  p.n_runs = static_cast<int32_t>(n_runs);
  p.freq = reinterpret_cast<const float2*>(ws + w.freq_off);
  p.k_dst = static_cast<uint8_t*>(k_cache);
  p.dst_layer_stride = cache_ls;
  p.block_tables = d_bt;
  p.max_blocks = max_blocks;
  p.header = reinterpret_cast<WsHeader*>(ws);
  const cudaError_t e = launch_shift_kernel(ctx, p, di.sm_count, s, host_io != 0);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "rerotate launch");
  return ok(ctx);
}

// ------------------------------------------------------------- diagnostics

pic_status pic_query_device_status(pic_ctx* ctx, const void* d_ws, pic_stream_t stream,
                                   uint32_t* status_out) {
  if (!d_ws) return fail(ctx, PIC_ERR_INVALID_ARG, "null workspace");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaStreamSynchronize");
  WsHeader h;
  e = cudaMemcpy(&h, d_ws, sizeof(h), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "status read");
  if (status_out) *status_out = h.status;
  if (h.status != 0)
    return fail(ctx, PIC_ERR_DEVICE_CHECK,
                "kernel reported device status 0x%x (bit 0x1: block-table entry outside the cache, table row %u, "
                "position %u; bit 0x2: a bounded wait gave up; 0x4: token id outside the Gear table; "
                "0x8: bad document offsets; 0x10: more chunks than capacity; 0x20: bad span)",
                h.status, h.bad_req, h.bad_pos);
  return ok(ctx);
}

pic_status pic_debug_stall_next_launch(pic_ctx* ctx, int32_t stall_tile, uint32_t max_spins) {
  if (!ctx) return fail(nullptr, PIC_ERR_INVALID_ARG, "null ctx");
  ctx->debug_stall = stall_tile >= 0 ? stall_tile + 1 : 0;
  ctx->debug_spins = stall_tile >= 0 ? max_spins : 0;
  return ok(ctx);
}

int32_t pic_kernel_variant(const pic_ctx* ctx, int32_t mode) {
  if (!ctx || mode < 0 || mode > 2) return -1;
  if (mode == 2) return ctx->attend_tc ? PIC_VARIANT_TENSOR_CORE_TMEM : PIC_VARIANT_WARP_MMA;
  const bool bulk = mode == 0 ? ctx->tma_stitch : ctx->tma_inplace;
  return bulk ? PIC_VARIANT_BULK_PIPELINE : PIC_VARIANT_REGISTERS;
}

pic_status pic_rotation_cossin(pic_ctx* ctx, const int32_t* d_deltas, int32_t n, float* d_out,
                               void* d_ws, size_t ws_bytes, pic_stream_t stream) {
  if (!ctx) return fail(nullptr, PIC_ERR_INVALID_ARG, "null ctx");
  if (n < 0 || (n > 0 && (!d_deltas || !d_out)) || !d_ws)
    return fail(ctx, PIC_ERR_INVALID_ARG, "bad arguments");
  const size_t need = ctx->freq_turns.size() * sizeof(float2);
  if (ws_bytes < need || ws_bytes < 4096) return fail(ctx, PIC_ERR_CAPACITY, "workspace needs 4096 bytes");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(d_ws, ctx->freq_turns.data(), need, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "frequency upload");
  e = pic::launch_cossin(d_deltas, n, static_cast<const float2*>(d_ws),
                         static_cast<int32_t>(ctx->freq_turns.size()), d_out, s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "cos/sin launch");
  return ok(ctx);
}

// ------------------------------------------------------- decode attention
// region attend-launch: workspace and launches of the decode attention (a
// measurement record names this region).

size_t pic_attend_workspace_bytes(const pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req,
                                  int32_t num_q_heads, int32_t num_layers) {
  if (!ctx || n_req < 0 || (n_req > 0 && !plans) || num_q_heads <= 0 || num_layers <= 0) return 0;
  for (int32_t r = 0; r < n_req; ++r)
    if (!plans[r]) return 0;
  AttnHeads heads;
  if (!attn_layout_heads(ctx->model, num_q_heads, &heads)) return 0;
  const bool mla = ctx->model.kind == PIC_KIND_MLA;
  AttnPlan fused, cache;
  attend_plan(ctx, plans, n_req, PIC_ATTEND_FUSED, heads, false, &fused);  // two-delta stages are never more
  attend_plan(ctx, plans, n_req, PIC_ATTEND_CACHE, heads, false, &cache);
  const size_t n_stages = std::max(fused.stages.size(), cache.stages.size());
  // a grid of at most kAttnMaxCtas CTAs adds at most one record per CTA
  const size_t n_keys = static_cast<size_t>(num_layers) * fused.n_keys;
  const size_t records = n_keys + pic::kAttnMaxCtas;
  // the tcgen05 kernel's tiles: at most one per stage
  return attend_layout(ctx, n_stages, mla ? n_stages : 0, fused.toks.size(), n_keys + 1, records, heads).total;
}

pic_status pic_attend_decode(pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req, int32_t source,
                             const void* q, int32_t num_q_heads, float softmax_scale, float sink_bias,
                             const void* k_pool, const void* v_pool, int64_t pool_ls, const void* k_cache,
                             const void* v_cache, int64_t cache_ls, int32_t layer_begin, int32_t num_layers,
                             float* out, float* lse, void* d_ws, size_t ws_bytes, pic_stream_t stream) {
  if (!ctx) return fail(nullptr, PIC_ERR_INVALID_ARG, "null ctx");
  const pic_model_desc& m = ctx->model;
  const bool mla = m.kind == PIC_KIND_MLA;
  AttnHeads heads;
  if (mla) {
    if (m.head_dim != 576 || m.rope_dim != 64 || m.rope_offset != 512)
      return fail(ctx, PIC_ERR_UNSUPPORTED, "MLA decode attention covers 512-dim latents with a 64-dim rope key");
    if (!attn_layout_heads(m, num_q_heads, &heads))
      return fail(ctx, PIC_ERR_UNSUPPORTED, "MLA decode attention takes 16, 32, 64 or 128 query heads");
  } else {
    if (m.head_dim != 64 && m.head_dim != 128)
      return fail(ctx, PIC_ERR_UNSUPPORTED, "decode attention covers GQA heads of 64 or 128 dims");
    int32_t hb = 0, hgroups = 0;
    if (!attn_heads(m, &hb, &hgroups))
      return fail(ctx, PIC_ERR_UNSUPPORTED, "decode attention needs <= %d KV heads or a multiple of %d",
                  pic::kAttnMaxHeads, pic::kAttnMaxHeads);
    if (num_q_heads <= 0 || num_q_heads % m.num_kv_heads != 0)
      return fail(ctx, PIC_ERR_INVALID_ARG, "num_q_heads must be a multiple of num_kv_heads");
    const int32_t group = num_q_heads / m.num_kv_heads;
    if (group != 1 && group != 2 && group != 4 && group != 8)
      return fail(ctx, PIC_ERR_UNSUPPORTED, "query heads per KV head must be 1, 2, 4 or 8");
    attn_layout_heads(m, num_q_heads, &heads);
  }
  if (source != PIC_ATTEND_FUSED && source != PIC_ATTEND_CACHE) return fail(ctx, PIC_ERR_INVALID_ARG, "bad source");
  if (n_req <= 0 || !plans) return fail(ctx, PIC_ERR_INVALID_ARG, "no requests");
  for (int32_t r = 0; r < n_req; ++r)
    if (!plan_valid(ctx, plans[r])) return fail(ctx, PIC_ERR_INVALID_ARG, "plans[%d] does not belong to this context", r);
  if (layer_begin < 0 || num_layers <= 0 || static_cast<int64_t>(layer_begin) + num_layers > m.num_layers)
    return fail(ctx, PIC_ERR_RANGE, "layer range outside the model");
  if (!q || !out || !d_ws || !k_cache || (!mla && !v_cache))
    return fail(ctx, PIC_ERR_INVALID_ARG, "null q, out, cache or workspace");
  if (source == PIC_ATTEND_FUSED && (!k_pool || (!mla && !v_pool)))
    return fail(ctx, PIC_ERR_INVALID_ARG, "fused attention reads the pool: pass k_pool (and v_pool for GQA)");
  if (mla) {
    v_pool = nullptr;  // the latent serves as value
    v_cache = nullptr;
  }
  if (!vectorized_bytes_ok(q) || !vectorized_bytes_ok(out) || !vectorized_bytes_ok(k_cache) ||
      (v_cache && !vectorized_bytes_ok(v_cache)) || (cache_ls & 15) || (k_pool && !vectorized_bytes_ok(k_pool)) ||
      (v_pool && !vectorized_bytes_ok(v_pool)) || (pool_ls & 15) || !vectorized_bytes_ok(d_ws))
    return fail(ctx, PIC_ERR_ALIGNMENT, "q, out, pools, caches, strides and workspace must be 16-byte aligned");
  for (int32_t r = 0; r < n_req; ++r)
    if (plans[r]->total_tokens == 0) return fail(ctx, PIC_ERR_RANGE, "plans[%d] has no context to attend", r);
  // MLA on tcgen05 when the pool and cache can be described as TMA tensors;
  // its stages may hold two deltas, the other kernels' one
  int ring = 0;
  size_t smem = 0;
  pic::TcMaps maps{};
  const bool tc_fits = mla && ctx->attend_tc && pic::attend_mla_tc_config(heads.group, &smem);
  const AttnPlanCache* cached = &attend_plan_cached(ctx, plans, n_req, source, heads, tc_fits);
  bool tc = tc_fits;
  if (tc) {
    // the pool view spans the rows the plan reads; the cache view every cache row
    const int64_t pool_rows = cached->pool_rows;
    const int64_t layers = static_cast<int64_t>(layer_begin) + num_layers;
    for (int g = 0; g < 4 && tc; ++g) {
      const uint32_t box = 16u * static_cast<uint32_t>(g + 1);
      tc = encode_mla_rows(&maps.cache[g], k_cache, static_cast<int64_t>(ctx->num_cache_blocks) * m.block_size,
                           layers, cache_ls, box);
      if (tc && pool_rows > 0) tc = encode_mla_rows(&maps.pool[g], k_pool, pool_rows, layers, pool_ls, box);
      if (tc && pool_rows == 0) maps.pool[g] = maps.cache[g];  // nothing is read from the pool
    }
  }
  if (tc_fits && !tc) cached = &attend_plan_cached(ctx, plans, n_req, source, heads, false);
  const AttnPlan& plan = cached->plan;
  const bool fits = tc || (mla ? pic::attend_mla_config(heads.mla_ng, &ring, &smem)
                               : pic::attend_config(m.head_dim, heads.group, heads.hb, &ring, &smem));
  if (!fits) return fail(ctx, PIC_ERR_UNSUPPORTED, "attention stages do not fit in shared memory");
  // units: (layer, stage), or (layer, tile) for the tcgen05 kernel
  const int64_t units = static_cast<int64_t>(tc ? cached->tiles.size() : plan.stages.size()) * num_layers;
  if (units > INT32_MAX || static_cast<int64_t>(plan.toks.size()) > INT32_MAX)
    return fail(ctx, PIC_ERR_CAPACITY, "attention batch too large");

  DeviceInfo di;
  pic_status st = current_device(ctx, di);
  if (st != PIC_OK) return st;
  const void* bufs[4] = {k_pool, v_pool, k_cache, v_cache};
  for (int i = 0; i < 4; ++i)
    if (bufs[i] && residency(bufs[i]) != 0)
      return fail(ctx, PIC_ERR_UNSUPPORTED, "decode attention reads pools and caches from device memory only");
  const int per_sm = tc ? 1
                   : mla ? pic::attend_mla_ctas_per_sm(m.pairing, heads.mla_ng, smem)
                         : pic::attend_ctas_per_sm(m.pairing, m.head_dim, heads.group, heads.hb, smem);
  if (per_sm <= 0) return fail(ctx, PIC_ERR_CUDA, "attention kernel does not fit on an SM");
  const int64_t ctas = std::min<int64_t>({units, static_cast<int64_t>(di.sm_count) * per_sm, pic::kAttnMaxCtas});
  std::vector<pic::AttnKey> keys;
  const int64_t records = tc ? attend_keys_tiles(cached->key_tile_begin, num_layers, ctas, &keys)
                            : attend_keys(plan, num_layers, ctas, &keys);
  // the tcgen05 kernel reads tiles instead of stages and token rows
  const size_t n_stages = tc ? 0 : plan.stages.size(), n_toks = tc ? 0 : plan.toks.size();
  const AttnLayout w = attend_layout(ctx, n_stages, tc ? cached->tiles.size() : 0, n_toks, keys.size(),
                                     static_cast<size_t>(records), heads);
  if (ws_bytes < w.total) return fail(ctx, PIC_ERR_CAPACITY, "workspace has %zu bytes, needs %zu", ws_bytes, w.total);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The read-only image (everything before the records) stays on the device
  // in the context's buffer for this cache slot while the same plan, layer
  // count and grid come back, so a decode loop uploads nothing per step; it
  // is staged and uploaded when it changes, into the workspace only when no
  // buffer can be had.  The workspace's header (status word) is zeroed.
  const size_t image = w.records_off;
  AttnResident& res = ctx->attn_res[tc ? 1 : 0];
  const bool resident = res.dev && res.device == di.device && res.owner == cached->serial &&
                        res.layers == num_layers && res.ctas == ctas;
  void* img = res.dev;
  if (!resident) {
    StagingSlot* sl = nullptr;
    st = acquire_staging(ctx, di.device, image, &sl);
    if (st != PIC_OK) return st;
    uint8_t* base = sl->host;
    std::memcpy(base + w.freq_off, ctx->freq_turns.data(), ctx->freq_turns.size() * sizeof(float2));
    std::memcpy(base + w.stages_off, plan.stages.data(), n_stages * sizeof(pic::AttnStage));
    if (tc) std::memcpy(base + w.tiles_off, cached->tiles.data(), cached->tiles.size() * sizeof(pic::TcTileRec));
    std::memcpy(base + w.toks_off, plan.toks.data(), n_toks * sizeof(pic::AttnTok));
    std::memcpy(base + w.keys_off, keys.data(), keys.size() * sizeof(pic::AttnKey));
    img = d_ws;
    if (res.device < 0 || res.device == di.device) {
      res.owner = 0;
      // launches on any stream that still read the buffer's old image come first
      if (res.last_use) {
        cudaError_t e = cudaStreamWaitEvent(s, res.last_use, 0);
        if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaStreamWaitEvent");
      }
      if (res.cap < image) {
        if (res.dev) cudaFreeAsync(res.dev, s);
        res.dev = nullptr;
        res.cap = 0;
        void* d = nullptr;
        if (cudaMallocAsync(&d, image, s) == cudaSuccess) {
          res.dev = d;
          res.cap = image;
          res.device = di.device;
        } else {
          cudaGetLastError();  // not sticky: the image goes to the workspace instead
        }
      }
      if (res.dev) img = res.dev;
    }
    st = upload_staging(ctx, sl, img, image, s);
    if (st != PIC_OK) return st;
    if (img == res.dev) {
      res.owner = cached->serial;
      res.layers = num_layers;
      res.ctas = ctas;
    }
  }
  if (img != d_ws) {
    cudaError_t e = cudaMemsetAsync(d_ws, 0, sizeof(WsHeader), s);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "workspace header");
  }
  const uint8_t* im = static_cast<const uint8_t*>(img);

  uint8_t* ws = static_cast<uint8_t*>(d_ws);
  constexpr float kLog2e = 1.4426950408889634f;
  pic::AttnParams p{};
  p.stages = reinterpret_cast<const pic::AttnStage*>(im + w.stages_off);
  p.n_stages = static_cast<int32_t>(n_stages);
  p.toks = reinterpret_cast<const pic::AttnTok*>(im + w.toks_off);
  p.tc_tiles = reinterpret_cast<const pic::TcTileRec*>(im + w.tiles_off);
  p.tc_tiles_per_layer = tc ? static_cast<int32_t>(cached->tiles.size()) : 0;
  p.keys = reinterpret_cast<const pic::AttnKey*>(im + w.keys_off);
  p.n_keys = plan.n_keys;
  p.n_units = units;
  p.freq = reinterpret_cast<const float2*>(im + w.freq_off);
  p.q = static_cast<const uint16_t*>(q);
  p.n_req = n_req;
  p.num_q_heads = num_q_heads;
  p.n_kv_heads = m.num_kv_heads;
  p.heads_per_cta = heads.hb;
  p.head_groups = heads.head_groups;
  p.n_layers = num_layers;
  p.layer_begin = layer_begin;
  p.scale_log2 = softmax_scale * kLog2e;
  p.sink_log2 = sink_bias * kLog2e;
  p.k_pool = static_cast<const uint8_t*>(k_pool);
  p.v_pool = static_cast<const uint8_t*>(v_pool);
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.pool_layer_stride = pool_ls;
  p.cache_layer_stride = cache_ls;
  p.row_bytes = static_cast<int32_t>(row_bytes_of(m));
  p.ring = ring;
  p.records = reinterpret_cast<float*>(ws + w.records_off);
  p.out = out;
  p.lse = lse;
  p.status = &reinterpret_cast<WsHeader*>(ws)->status;
  p.debug_stall = ctx->debug_stall;
  p.max_spins = ctx->debug_spins;
  ctx->debug_stall = 0;
  ctx->debug_spins = 0;
  cudaError_t e;
  if (tc) {
    e = pic::launch_attend_mla_tc(p, maps, m.pairing, heads.group, static_cast<int>(ctas), smem, s);
  } else {
    e = mla ? pic::launch_attend_mla(p, m.pairing, heads.mla_ng, static_cast<int>(ctas), smem, s)
            : pic::launch_attend(p, m.pairing, m.head_dim, heads.group, static_cast<int>(ctas), smem, s);
  }
  if (e != cudaSuccess) return cuda_fail(ctx, e, "attention launch");
  if (img == res.dev) {
    if (!res.last_use) {
      e = cudaEventCreateWithFlags(&res.last_use, cudaEventDisableTiming);
      if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaEventCreate");
    }
    e = cudaEventRecord(res.last_use, s);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaEventRecord");
  }
  return ok(ctx);
}

// end region attend-launch

}  // extern "C"

// ===================================================== scratch-backed stitch
//
// Used only by the no-alloc entry point.  Same checks, workspace image and
// launch as pic_stitch, but the image is written straight into a
// caller-owned host buffer and uploaded with a plain copy from that
// (pageable) buffer into a caller-owned device buffer, so nothing is
// allocated here.  A copy from pageable memory may make the host wait until
// the stream's earlier work has finished.

namespace pic {

pic_status set_error(pic_ctx* ctx, pic_status st, const char* msg) { return fail(ctx, st, "%s", msg); }

pic_status stitch_with_scratch(pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req,
                               const void* k_pool, const void* v_pool, int64_t pool_ls,
                               void* k_cache, void* v_cache, int64_t cache_ls,
                               const int32_t* d_bt, int32_t max_blocks, int32_t* d_ridx,
                               int32_t* d_indptr, int64_t recompute_capacity, void* d_scratch,
                               size_t scratch_bytes, uint8_t* image, size_t image_bytes,
                               uint32_t* d_status_out, cudaStream_t s) {
  if (!ctx) return fail(nullptr, PIC_ERR_INVALID_ARG, "null ctx");
  pic_status st = check_stitch_args(ctx, plans, n_req, k_pool, v_pool, pool_ls, k_cache, v_cache, cache_ls,
                                    d_bt, max_blocks, d_ridx, d_indptr, recompute_capacity);
  if (st != PIC_OK) return st;
  const size_t n_runs = count_stitch_runs(ctx, plans, n_req);
  const WsLayout w = ws_layout(ctx->freq_turns.size(), static_cast<size_t>(n_req) + 1, n_runs);
  const size_t limit = std::min(scratch_bytes, image_bytes);
  if (w.total > limit)
    return fail(ctx, PIC_ERR_CAPACITY,
                "this batch needs %zu bytes of scratch (%zu runs); the static scratch holds %zu bytes. "
                "Split the batch or call pic_stitch with a workspace", w.total, n_runs, limit);
  if (!d_scratch || !image) return fail(ctx, PIC_ERR_INVALID_ARG, "null scratch");

  // Image: zeroed header (the status word must start at 0 on every call),
  // frequencies, CSR offsets, runs written in place.
  std::memset(image, 0, w.total);
  build_stitch_image(ctx, plans, n_req, image, w);

  DeviceInfo di;
  st = current_device(ctx, di);
  if (st != PIC_OK) return st;
  const void* bufs[4] = {k_pool, v_pool, k_cache, v_cache};
  const int host_io = host_buffers(ctx, bufs, 4);
  if (host_io < 0) return PIC_ERR_INVALID_ARG;
  cudaError_t e = cudaMemcpyAsync(d_scratch, image, w.total, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "scratch upload");
  KernelParams p{};
  fill_stitch_params(ctx, p, static_cast<uint8_t*>(d_scratch), w, n_runs, n_req, k_pool, v_pool, pool_ls, k_cache,
                     v_cache, cache_ls, d_bt, max_blocks, d_ridx, d_indptr);
  // The failure-test hook applies to this launch exactly as to pic_stitch's.
  p.debug_stall = ctx->debug_stall;
  p.max_spins = ctx->debug_spins;
  ctx->debug_stall = 0;
  ctx->debug_spins = 0;
  e = launch_stitch_kernel(ctx, p, di.sm_count, s, host_io != 0, mostly_in_place(plans, n_req));
  if (e != cudaSuccess) return cuda_fail(ctx, e, "stitch launch");
  for (int32_t r = 0; r < n_req; ++r) const_cast<pic_plan*>(plans[r])->applied = true;
  if (d_status_out) {
    e = cudaMemcpyAsync(d_status_out, d_scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "status copy");
  }
  return ok(ctx);
}

}  // namespace pic
