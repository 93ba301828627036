/*
 * pic.h -- C ABI of the position-independent KV stitching library (libpic).
 *
 * What the library does.  Each document chunk's KV cache is computed once, at
 * virtual offset 0, and kept in a chunk pool in GPU memory.  A request lists
 * chunks in any order; the library places them at their new absolute
 * positions in the request's paged KV cache.  On the way, the RoPE part of
 * every cached key is re-rotated by the chunk's position shift
 * delta = dst_pos - base_pos, using R(a + b) = R(a) R(b); values (GQA) and
 * the MLA latent are copied bit for bit.  The same pass writes the list of
 * token positions to recompute (the first k tokens of each chunk).
 *
 * Sources (pages, cited by title and section):
 *   [EPIC]     "EPIC Guide: Position-Independent Caching for LLM Serving"
 *              (aifetchly blog, on EPIC, ICML 2025).
 *   [Irminsul] "Irminsul: MLA-Native Position-Independent Caching for Agentic
 *              LLM Serving" (gist.science explainer), Technical Summary.
 *   [SemPIC]   "SemPIC: Learning Semantic Position-Independent KV Caches"
 *              (agihunt summary), cache-hit serving paragraph.
 *
 * Conventions for every function:
 *   - Ownership: the caller owns every device buffer (pools, caches, block
 *     tables, index outputs, workspaces).  The library owns its host-side
 *     registry, block allocator and pic_plan objects, and only two pieces of
 *     device memory: the fixed scratch array of pic_stitch_noalloc, and the
 *     device copy of the decode attention's plan image that pic_attend_decode
 *     keeps per context (freed by pic_destroy).  pic_stitch_staged also keeps
 *     a CUDA stream and an event per context.
 *   - Threads: a context is used by one host thread at a time.
 *   - Streams: all device work is enqueued on the caller's stream and is
 *     asynchronous; host arguments may be reused as soon as a call returns.
 *     (pic_stitch_staged runs its copies on its own stream, ordered between
 *     the caller's earlier and later work.)
 *   - Errors: every call returns a pic_status; on failure nothing was
 *     enqueued and pic_last_error() describes the cause.  CUDA launch
 *     failures are PIC_ERR_CUDA.  Errors a kernel finds on the device (a
 *     block-table entry outside the cache) skip the faulty write and raise a
 *     status word in the workspace, read by pic_query_device_status().
 *     Kernels never trap; their only waits (for their own bulk copies) are
 *     bounded and raise PIC_DEV_TIMEOUT instead of hanging.
 *   - Layouts (bf16 elements, row = one token of one layer):
 *       GQA key/value row: [num_kv_heads][head_dim], RoPE over all of head_dim.
 *       MLA row: [latent_dim + rope_dim] with the rope key last ([Irminsul]
 *       2.1: 512-d cKV latent, 64-d k_r).
 *       Pool:  [num_layers] x (layer stride) of [pool_tokens][row].
 *       Cache: [num_layers] x (layer stride) of [num_cache_blocks][block_size][row].
 *     Base pointers and layer strides must be multiples of 16 bytes.
 *   - Host-resident pools and caches: pool and cache pointers may also be
 *     pinned host memory (cudaHostAlloc, or memory registered with
 *     cudaHostRegister): the kernels then stream them over the host link
 *     directly, with no staging copy (on GB300, NVLink-C2C to Grace memory).
 *     Pageable host memory is refused with PIC_ERR_INVALID_ARG.  Block tables,
 *     recompute outputs and workspaces stay in device memory.
 *   - Positions are int32; |delta| must be below 2^24.
 */
#ifndef PIC_H
#define PIC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; 0 is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st* pic_stream_t;

#define PIC_ABI_VERSION 2
#define PIC_KEY_BYTES 32
#define PIC_MAX_ABS_DELTA ((1 << 24) - 1)

typedef enum pic_status {
  PIC_OK = 0,
  PIC_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad enum, bad plan      */
  PIC_ERR_UNKNOWN_CHUNK = 2, /* chunk id or key not in the registry                  */
  PIC_ERR_KEY_CONFLICT = 3,  /* key already registered with another length/base_pos  */
  PIC_ERR_OUT_OF_BLOCKS = 4, /* block allocator cannot cover the request             */
  PIC_ERR_CAPACITY = 5,      /* an output or workspace buffer is too small           */
  PIC_ERR_RANGE = 6,         /* position, delta or token range out of bounds         */
  PIC_ERR_ALIGNMENT = 7,     /* pointer or stride not a multiple of 16 bytes         */
  PIC_ERR_CUDA = 8,          /* a CUDA runtime call or launch failed                 */
  PIC_ERR_DEVICE_CHECK = 9,  /* a kernel found a bad block-table entry               */
  PIC_ERR_UNSUPPORTED = 10,  /* geometry the library has no kernel for               */
  PIC_ERR_BUSY = 11          /* chunk is mapped by a live request, or in use         */
} pic_status;

enum { PIC_KIND_GQA = 0, PIC_KIND_MLA = 1 };
/* NEOX_HALF pairs dims (i, i + d/2); INTERLEAVED pairs (2i, 2i + 1), the
 * layout [EPIC] "Mathematical Foundations" 1. prints. */
enum { PIC_PAIRING_NEOX_HALF = 0, PIC_PAIRING_INTERLEAVED = 1 };
enum { PIC_SCALING_NONE = 0, PIC_SCALING_LLAMA3 = 1 };

/* Device status word bits (pic_query_device_status). */
#define PIC_DEV_BAD_BLOCK 0x1u /* a block-table entry was < 0 or >= num_cache_blocks */
#define PIC_DEV_TIMEOUT 0x2u   /* a bounded wait inside a kernel gave up (never expected) */
#define PIC_DEV_BAD_TOKEN 0x4u /* chunking: a token id outside [0, vocab); its Gear value taken as 0 */
#define PIC_DEV_BAD_DOCS 0x8u  /* chunking: document offsets not non-decreasing within [0, n_tokens] */
#define PIC_DEV_CAPACITY 0x10u /* chunking: more chunks than capacity; the rest were not written */
#define PIC_DEV_BAD_SPAN 0x20u /* fingerprints: a span outside [0, n_tokens] or with end < start */

/*
 * Model geometry and RoPE settings.
 *   GQA: num_kv_heads >= 1, head_dim in {64, 128, 256}, rope_dim == head_dim,
 *        rope_offset == 0.
 *   MLA: num_kv_heads == 1, head_dim == latent + rope (576), rope_dim == 64,
 *        rope_offset == 512.
 * Frequencies: theta_i = rope_theta^(-2i/rope_dim) ([EPIC] "Mathematical
 * Foundations" 1.), optionally with Llama-3.1 scaling (not on the pages;
 * the public rule), or exactly the rope_dim/2 values in inv_freq when that
 * pointer is non-NULL (copied at pic_create; any other RoPE scaling scheme can
 * be supplied this way).
 */
typedef struct pic_model_desc {
  int32_t kind;              /* PIC_KIND_GQA or PIC_KIND_MLA                       */
  int32_t num_layers;        /* >= 1                                               */
  int32_t num_kv_heads;      /* GQA: heads per row; MLA: 1                         */
  int32_t head_dim;          /* GQA: dims per head; MLA: row width                 */
  int32_t rope_dim;          /* dims rotated per head (even)                       */
  int32_t rope_offset;       /* first rotated dim inside a head                    */
  int32_t pairing;           /* PIC_PAIRING_*                                      */
  int32_t block_size;        /* tokens per paged block, 1 .. 256                   */
  int32_t scaling;           /* PIC_SCALING_*                                      */
  int32_t llama3_orig_max_pos;
  double rope_theta;
  double llama3_factor;
  double llama3_low_freq_factor;
  double llama3_high_freq_factor;
  const double* inv_freq;    /* optional: rope_dim/2 frequencies (radians/token)   */
} pic_model_desc;

typedef struct pic_ctx pic_ctx;
typedef struct pic_plan pic_plan;

/*
 * One request: the prompt's chunks in order ([EPIC] "Algorithmic
 * Architecture" 2. Modular Prompt Composer).
 *   chunk_ids    n_chunks registered ids; a chunk may appear more than once
 *                (each occurrence is its own segment).
 *   take_tokens  NULL = whole chunks; else tokens taken from the start of
 *                each chunk (0 .. num_tokens).
 *   dst_pos      NULL = chunk j starts where chunk j-1 ended, the first at
 *                start_pos; else the absolute position of each chunk's first
 *                token, non-decreasing and non-overlapping (the "offset" of
 *                [EPIC] "Production Deployment Playbook" 2.).  Gaps hold
 *                inline tokens the caller computes itself.
 *   total_tokens logical length the block table must cover; 0 = the end of
 *                the last chunk.  Must not be smaller than that end.
 *   k_nonleading tokens recomputed at the start of every chunk not at
 *                position 0 (LegoLink pseudo-sinks; [EPIC] uses 4).
 *   k_leading    tokens recomputed at the start of a chunk at position 0
 *                ([Irminsul] 2.2 First-Chunk Carve-Out uses 32).
 *   alias        1: map block-resident chunks into the request instead of
 *                copying them when allowed (see pic_register_chunk_blocks);
 *                0: always copy.
 */
typedef struct pic_request_desc {
  const int32_t* chunk_ids;
  const int32_t* take_tokens;
  const int32_t* dst_pos;
  int32_t n_chunks;
  int32_t start_pos;
  int32_t total_tokens;
  int32_t k_nonleading;
  int32_t k_leading;
  int32_t alias;
} pic_request_desc;

/* One in-place shift: rows [start_pos, start_pos + num_tokens) of block-table
 * row `req` are rotated by `delta`. */
typedef struct pic_shift_seg {
  int32_t req;
  int32_t start_pos;
  int32_t num_tokens;
  int32_t delta;
} pic_shift_seg;

/* ---------------------------------------------------------------- context */

/* Creates a context for one model and a paged cache of num_cache_blocks
 * blocks (the allocator's range; the caller's cache tensors must hold at
 * least that many blocks per layer).  Validates the geometry
 * (PIC_ERR_UNSUPPORTED for shapes without a kernel).  Does not touch the GPU;
 * the device of the first launch is used for every later launch.
 * *out is set on success, left untouched otherwise. */
pic_status pic_create(const pic_model_desc* model, int32_t num_cache_blocks, pic_ctx** out);

/* Frees the context, its registry and every plan still alive. NULL is a no-op. */
void pic_destroy(pic_ctx* ctx);

/* Last error message of ctx (or of the calling thread when ctx is NULL);
 * valid until the next call on the same ctx / thread.  Never NULL. */
const char* pic_last_error(const pic_ctx* ctx);

const char* pic_status_string(pic_status status);
int32_t pic_abi_version(void);

/* --------------------------------------------------------------- registry */

/*
 * Content-addressed chunk registry ([EPIC] "Algorithmic Architecture" 1.
 * Content-Addressed Chunk Registry; [Irminsul] 2.2 Registry Lookup:
 * hash -> (cKV, k_r, base_pos)).  key is PIC_KEY_BYTES opaque bytes (a
 * SHA-256 digest, or a zero-padded xxHash64).  The chunk's rows are pool
 * token rows [pool_token_offset, pool_token_offset + num_tokens) of every
 * layer; base_pos is the position they were computed at (0 = offset 0).
 * Registering a known key with the same num_tokens and base_pos returns its
 * id with *is_new = 0 (the pool offset of the first registration is kept);
 * with another num_tokens or base_pos it fails with PIC_ERR_KEY_CONFLICT.
 */
pic_status pic_register_chunk(pic_ctx* ctx, const uint8_t* key, int64_t pool_token_offset,
                              int32_t num_tokens, int32_t base_pos, int32_t* chunk_id,
                              int32_t* is_new);

/*
 * Registers a chunk whose KV already sits in blocks of the paged cache (for
 * instance a document prefilled once into the cache): blocks[j], j <
 * ceil(num_tokens / block_size), holds its tokens [j*bs, (j+1)*bs) in rows
 * 0.. of the block (the last block partly), keys rotated for position
 * base_pos.  The blocks must be free in the allocator; they are taken out of
 * it and belong to the chunk until pic_unregister_chunk.  A chunk needing
 * more blocks than the cache holds fails with PIC_ERR_RANGE before blocks[]
 * is read.
 *
 * Such a chunk can be served to a request without moving its values: the
 * EPIC runtime ([EPIC] "Algorithmic Architecture", runtime figure step 1
 * "Virtual Block Mapping" -- the request reuses the chunk's physical blocks --
 * and step 2, the keys rotated in place by dp).  pic_build_block_table with
 * alias = 1 maps the chunk's blocks into the request's table when the chunk
 * starts on a block boundary, is taken whole, occurs once in the request and
 * no other live request uses it; the stitch then rotates only its keys, in
 * place, by delta = new position - current position, and the chunk's current
 * position becomes the new one (pic_chunk_info reports it).  Otherwise its
 * tokens are copied out of its blocks like a pool chunk.  While a request has
 * a chunk mapped, no other request may use that chunk (PIC_ERR_BUSY): its
 * keys are being moved.  Rows of a mapped chunk's last block past its tokens
 * belong to the request while it lives.
 */
pic_status pic_register_chunk_blocks(pic_ctx* ctx, const uint8_t* key, const int32_t* blocks,
                                     int32_t num_tokens, int32_t base_pos, int32_t* chunk_id,
                                     int32_t* is_new);

/* Registry lookup by key: PIC_ERR_UNKNOWN_CHUNK on a miss. */
pic_status pic_lookup_chunk(const pic_ctx* ctx, const uint8_t* key, int32_t* chunk_id);

/* Reads back a registry entry.  For a block-resident chunk, *pool_token_offset
 * is -1 and *base_pos its current position. */
pic_status pic_chunk_info(const pic_ctx* ctx, int32_t chunk_id, int64_t* pool_token_offset,
                          int32_t* num_tokens, int32_t* base_pos);

/* Removes a chunk from the registry; the id is never reused.  Plans already
 * built from a pool chunk keep working (they hold copies of the entry).  A
 * block-resident chunk still used by a live request is refused with
 * PIC_ERR_BUSY; otherwise its blocks return to the allocator. */
pic_status pic_unregister_chunk(pic_ctx* ctx, int32_t chunk_id);

/* ---------------------------------------------------------- plan + table */

/*
 * Composes one request and allocates its paged blocks.
 *   Segments: dst_pos as described in pic_request_desc, delta = dst_pos -
 *   base_pos ([Irminsul] 2.2 delta-Rotation Rule; [SemPIC] "assign final
 *   logical positions, re-rotate the RoPE keys").
 *   Blocks: ceil(total / block_size) blocks covering positions [0, total),
 *   taken lowest free id first, in logical order (one deterministic choice;
 *   the pages fix none).  block_table_out[0 .. max_blocks) receives the ids,
 *   -1 past the last one.
 * On success *plan_out owns the blocks until pic_free_request.  Fails with
 * PIC_ERR_CAPACITY if max_blocks is too small, PIC_ERR_OUT_OF_BLOCKS if the
 * allocator is exhausted (nothing is allocated then).
 */
pic_status pic_build_block_table(pic_ctx* ctx, const pic_request_desc* request,
                                 int32_t* block_table_out, int32_t max_blocks,
                                 pic_plan** plan_out);

/* Returns the plan's fresh blocks to the allocator (mapped chunk blocks stay
 * with their chunks), releases the chunks it used and frees the plan.  A plan
 * whose in-place rotations were never enqueued puts its mapped chunks back
 * at their old positions. */
pic_status pic_free_request(pic_ctx* ctx, pic_plan* plan);

/* Sizes of a plan (any pointer may be NULL). */
pic_status pic_plan_info(const pic_plan* plan, int32_t* total_tokens, int32_t* num_blocks,
                         int32_t* num_segments, int32_t* num_recompute);

/* Segment j of a plan: where it reads, where it lands and its shift. */
pic_status pic_plan_segment(const pic_plan* plan, int32_t j, int32_t* chunk_id,
                            int64_t* src_token, int32_t* num_tokens, int32_t* dst_pos,
                            int32_t* delta);

/* How segment j is served: PIC_SEG_COPY_POOL, PIC_SEG_COPY_BLOCKS (copied out
 * of a block-resident chunk) or PIC_SEG_MAPPED (the chunk's blocks mapped,
 * keys rotated in place); -1 on bad arguments. */
#define PIC_SEG_COPY_POOL 0
#define PIC_SEG_COPY_BLOCKS 1
#define PIC_SEG_MAPPED 2
int32_t pic_plan_segment_mode(const pic_plan* plan, int32_t j);

/* ---------------------------------------------------------------- stitch */

/* Workspace bytes pic_stitch needs for this batch of plans (device memory,
 * 256-byte aligned, owned by the caller). */
size_t pic_workspace_bytes(const pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req);

/*
 * The hot path: for every layer l, plan r, segment, and token t of it,
 *   K_cache[l][bt[r][p / bs]][p % bs] = R(delta) K_pool[l][src + t]   (rope dims)
 *   V_cache[l][...same slot...]       = V_pool[l][src + t]           (bit copy)
 * with p = dst_pos + t ([EPIC] "Mathematical Foundations" 2. The In-Place
 * Shift Transformation: k_target = R_dp k_cached, "Values ... completely
 * untouched"; runtime figure: chunks land in PagedAttention blocks).  For MLA
 * (v_pool = v_cache = NULL) the latent dims are copied and only the rope
 * dims rotated ([Irminsul] 2.1-2.2).  delta == 0 is a pure bit copy.
 * Rotation arithmetic: fp32, one round-to-nearest-even to bf16.
 * The same launch writes the recompute list as CSR: d_recompute_indptr
 * [n_req + 1] and d_recompute_idx [count] (ascending positions per request;
 * the rule is pic_recompute_indices').
 *   d_block_tables  device int32 [n_req][max_blocks]; row r is plans[r]'s
 *                   table (as pic_build_block_table returned it).
 *   d_recompute_*   may both be NULL when no index output is wanted.
 *   recompute_capacity  elements available in d_recompute_idx.
 *   d_workspace     >= pic_workspace_bytes(...) bytes of device memory.
 * Rows of the cache outside the plans' chunks are not touched.  Plans must
 * not write the same cache slot twice (distinct plans own distinct blocks).
 * Mapped segments (PIC_SEG_MAPPED) are served in the same launch by rotating
 * their keys in place; a plan's in-place rotations run once, so a plan with
 * mapped segments can be stitched only once (PIC_ERR_INVALID_ARG after).
 */
pic_status pic_stitch(pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req,
                      const void* k_pool, const void* v_pool, int64_t pool_layer_stride_bytes,
                      void* k_cache, void* v_cache, int64_t cache_layer_stride_bytes,
                      const int32_t* d_block_tables, int32_t max_blocks,
                      int32_t* d_recompute_idx, int32_t* d_recompute_indptr,
                      int64_t recompute_capacity, void* d_workspace, size_t workspace_bytes,
                      pic_stream_t stream);

/*
 * pic_stitch_noalloc -- pic_stitch without a caller workspace.  The pages
 * have no counterpart to this call; it exists for deployment.
 *
 * Some callers cannot allocate device memory where they stitch: an engine
 * that gave (nearly) all of HBM to its own KV-cache pool, a framework that
 * hands a plugin only the tensors it reads and writes, or a loop that must
 * not pay for cudaMalloc / cudaFree (cudaFree synchronizes the whole
 * device).  This call runs the same kernel and computes the same result
 * as pic_stitch, with the same arguments minus the workspace; it allocates no
 * memory of any kind.  Its scratch (run list, frequency table, status word)
 * is a fixed 4 MiB array of device memory inside the library, which every GPU
 * that loads the library holds until the process exits.
 *   - Limit: a batch whose scratch image exceeds 4 MiB (about 130,000 runs of
 *     up to block_size tokens, i.e. about two million tokens per call at block
 *     size 16) fails with PIC_ERR_CAPACITY before anything is enqueued; split
 *     the batch or use pic_stitch.
 *   - Set-up: the first call on a device (with that device current) looks up
 *     the array's device address; make that first call before any stream
 *     capture.
 *   - Host wait: the scratch image is uploaded from an ordinary (pageable)
 *     host array inside the library, and the CUDA runtime may hold such a
 *     copy, and so this call, until the work already queued on the stream
 *     has finished.  Unlike pic_stitch, the call is therefore not always
 *     asynchronous with respect to the host.
 *   - Sharing: every call uses the same array and leaves its contents behind;
 *     each call rewrites what it needs, including a zeroed status word.  Calls
 *     that overlap on the GPU (different streams) race on it, and calls from
 *     several host threads at once race on its host image: issue one call at a
 *     time.
 *   - d_status: optional device uint32 that receives the device status word
 *     of this launch (PIC_DEV_* bits, 0 = clean); may be NULL.
 */
pic_status pic_stitch_noalloc(pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req,
                              const void* k_pool, const void* v_pool, int64_t pool_layer_stride_bytes,
                              void* k_cache, void* v_cache, int64_t cache_layer_stride_bytes,
                              const int32_t* d_block_tables, int32_t max_blocks,
                              int32_t* d_recompute_idx, int32_t* d_recompute_indptr,
                              int64_t recompute_capacity, uint32_t* d_status, pic_stream_t stream);

/* ---------------------------------------------- pools in host memory */

/*
 * Pool rows a batch reads: *rows_read counts every (segment, token) that
 * copies a row out of the pool, *distinct_rows the pool rows among them,
 * each once (chunks placed more than once, or in several requests, read
 * the same rows), leaving out rows that staged_plans read (may be NULL and
 * 0; the rows pic_stage_pool would copy with the same lists).
 * Block-resident and mapped chunks read no pool rows.  Per layer; multiply
 * by num_layers and the row bytes (twice for GQA: K and V) for bytes.  Host
 * only, no device work.  Either output may be NULL.
 */
pic_status pic_pool_read_rows(const pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req,
                              const pic_plan* const* staged_plans, int32_t n_staged,
                              int64_t* distinct_rows, int64_t* rows_read);

/*
 * pic_stage_pool -- copies the pool rows a batch reads, each once, from a
 * pool in pinned host memory into a device pool of the same layout.  The
 * pages keep chunk caches in GPU memory; this call serves a pool kept in
 * host memory instead.  pic_stitch can read such a pool directly over the
 * host link, but then a row placed n times crosses the link n times.  After
 * this call, pic_stitch with dev_k_pool / dev_v_pool as its pool (on the
 * same stream) reads every row from HBM.
 *   staged_plans, n_staged     plans whose rows an earlier call already
 *        staged into the same device pools (may be NULL and 0): their rows are
 *        skipped.  A caller can so split a batch into groups of requests and
 *        stage group g + 1 on a copy stream while group g is stitched.
 *   host_k_pool, host_v_pool   pinned host memory (cudaHostAlloc or
 *        cudaHostRegister), [num_layers] x host_pool_layer_stride_bytes of
 *        [pool_tokens][row]; v is NULL for MLA.
 *   dev_k_pool, dev_v_pool     device memory with the same token rows,
 *        [num_layers] x dev_pool_layer_stride_bytes; only the rows the plans
 *        read are written, the others are left as they are.
 * The rows are copied by a kernel on `stream` (SM loads over the host link,
 * one CTA per SM), not by a copy engine: a copy engine serves its queue in
 * order, so gigabytes of pool copies queued on it would hold back every
 * small upload behind them, such as a stitch's workspace image on another
 * stream.  *bytes_copied (may be NULL) receives the bytes the launch copies.
 * Layer strides must hold the highest row read (with more than one layer);
 * pointers and strides must be multiples of 16 bytes.  Host pointers that are
 * not pinned, or device pointers that are not device memory, are refused
 * with PIC_ERR_INVALID_ARG before anything is enqueued.  A batch of more than
 * 1,024 row ranges takes one launch per 1,024; a launch the CUDA runtime
 * refuses returns PIC_ERR_CUDA with the earlier launches enqueued.
 */
pic_status pic_stage_pool(pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req,
                          const pic_plan* const* staged_plans, int32_t n_staged,
                          const void* host_k_pool, const void* host_v_pool,
                          int64_t host_pool_layer_stride_bytes, void* dev_k_pool, void* dev_v_pool,
                          int64_t dev_pool_layer_stride_bytes, int64_t* bytes_copied, pic_stream_t stream);

/*
 * pic_stitch_staged -- pic_stage_pool and pic_stitch in one call, pipelined
 * over groups of requests, for a chunk pool in pinned host memory.  The
 * requests are cut into n_groups consecutive groups (at most n_req).  Group
 * g's pool rows, less those of earlier groups, are copied into the device
 * pools on a stream the context owns, while group g - 1 is stitched on
 * `stream`.  So each distinct row crosses the host link once, and the
 * stitches hide behind the copies.  The outputs equal those of
 * pic_stage_pool followed by pic_stitch with the device pools, bit for bit:
 * the cache rows, and one recompute CSR over all requests.
 *   host_* / dev_* pools   as pic_stage_pool; the device pools then hold the
 *                          rows the plans read.
 *   k_cache ... stream     as pic_stitch.
 *   d_workspace            pic_stitch_staged_workspace_bytes(ctx, plans,
 *                          n_req, n_groups) bytes.  Its first 256 bytes hold
 *                          the status word of the whole call, read by
 *                          pic_query_device_status.
 *   *bytes_staged          (may be NULL) bytes the copies move.
 * Stream order: the copies start after the work queued on `stream` before the
 * call, and every stitch and the work queued on `stream` after the call run
 * after the copies they need.  The context keeps the copy stream and an event
 * (created on first use, per device; destroyed by pic_destroy).  Errors as
 * pic_stitch and pic_stage_pool; n_groups < 1 is PIC_ERR_INVALID_ARG.
 */
size_t pic_stitch_staged_workspace_bytes(const pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req,
                                         int32_t n_groups);
pic_status pic_stitch_staged(pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req, int32_t n_groups,
                             const void* host_k_pool, const void* host_v_pool,
                             int64_t host_pool_layer_stride_bytes, void* dev_k_pool, void* dev_v_pool,
                             int64_t dev_pool_layer_stride_bytes, void* k_cache, void* v_cache,
                             int64_t cache_layer_stride_bytes, const int32_t* d_block_tables, int32_t max_blocks,
                             int32_t* d_recompute_idx, int32_t* d_recompute_indptr, int64_t recompute_capacity,
                             void* d_workspace, size_t workspace_bytes, int64_t* bytes_staged,
                             pic_stream_t stream);

/* ------------------------------------------------------- in-place shift */

size_t pic_rerotate_workspace_bytes(const pic_ctx* ctx, const pic_shift_seg* segs,
                                    int32_t n_segs);

/*
 * Re-rotates keys already in the paged cache, in place ([EPIC] runtime
 * figure, step 2 "Fast In-Place RoPE Key Rotation"; "Mathematical
 * Foundations" 2.): for each seg, each position p in [start_pos,
 * start_pos + num_tokens), the key row at bt[req][p / bs], p % bs becomes
 * R(delta) of itself (rope dims only; values and MLA latents untouched).
 *   d_block_tables  device int32 [n_tables][max_blocks].
 *   segs            host array; a cache row must not appear twice (the
 *                   rotations would race).  delta == 0 segments are skipped.
 * Note: if blocks are shared between requests, every sharer sees the
 * rotation.
 */
pic_status pic_rerotate_inplace(pic_ctx* ctx, void* k_cache, int64_t cache_layer_stride_bytes,
                                const int32_t* d_block_tables, int32_t n_tables,
                                int32_t max_blocks, const pic_shift_seg* segs, int32_t n_segs,
                                void* d_workspace, size_t workspace_bytes, pic_stream_t stream);

/* ------------------------------------------------------ recompute list */

/*
 * Host twin of the index list pic_stitch writes.  For each plan, ascending:
 * a segment at position 0 contributes its first min(k_leading, len) positions,
 * every other segment its first min(k_nonleading, len) positions ([EPIC]
 * LegoLink "1. Identifying and Neutralizing Pseudo-Sinks": sink tokens at each
 * chunk start, global token 0 protected; [Irminsul] 2.2 First-Chunk
 * Carve-Out).  idx_out / indptr_out are host arrays (indptr_out has n_req + 1
 * entries); *count receives the total even when capacity is too small
 * (PIC_ERR_CAPACITY, nothing written to idx_out then).  idx_out may be NULL to
 * query the count.  A total above 2^31 - 1 entries (the CSR offsets are
 * int32) fails with PIC_ERR_RANGE, *count still set, nothing written.
 */
pic_status pic_recompute_indices(const pic_plan* const* plans, int32_t n_req, int32_t* idx_out,
                                 int32_t* indptr_out, int64_t capacity, int64_t* count);

/* ---------------------------------------------------- decode attention */

#define PIC_ATTEND_FUSED 0 /* chunk tokens read from their sources, keys rotated on load */
#define PIC_ATTEND_CACHE 1 /* every position read from the request's paged cache          */

/* Workspace bytes of pic_attend_decode for this batch (either source). */
size_t pic_attend_workspace_bytes(const pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req,
                                  int32_t num_q_heads, int32_t num_layers);

/*
 * One decode step of grouped-query attention over each request's context,
 * positions [0, total_tokens) of its plan, for layers [layer_begin,
 * layer_begin + num_layers):
 *   s_t = softmax_scale * q . k_t + (sink_bias if t is a pseudo-sink),
 *   out = sum_t softmax(s)_t v_t,  lse = log sum_t exp(s_t).
 * PIC_ATTEND_FUSED reads chunk tokens where the chunk lives (pool rows, or the
 * blocks of a block-resident chunk) and applies the chunk's R(delta) on the
 * way from HBM to the SMs, so the context needs no stitched copy ([Irminsul]
 * 2.2 and 4: the rotation belongs in the attention kernel's load path, where
 * it costs no HBM traffic).  The kernel rotates the query by R(-delta) once
 * per delta instead of every key, which gives the same scores.  Positions no
 * chunk covers (inline tokens) and mapped chunks whose rotation already ran
 * are read from the paged cache through the plan's block table.
 * PIC_ATTEND_CACHE reads every position from the paged cache (a stitched
 * context).  A pseudo-sink is one of the first k_nonleading tokens of a chunk
 * not at position 0, the positions pic_recompute_indices lists for it
 * ([EPIC] LegoLink "1. Identifying and Neutralizing Pseudo-Sinks"; the listing
 * adds -15 to those logits); sink_bias 0 disables it.
 *   q      device bf16 [num_layers][n_req][num_q_heads][head_dim], already
 *          rotated to the query's position; query head g reads KV head
 *          g / (num_q_heads / num_kv_heads).  16-byte aligned.
 *   out    device float [num_layers][n_req][num_q_heads][head_dim].
 *   lse    device float [num_layers][n_req][num_q_heads] or NULL.
 * GQA models with head_dim 64 or 128, at most 8 KV heads or a multiple of 8,
 * and 1, 2, 4 or 8 query heads per KV head; pools and caches in device
 * memory, 16-byte aligned.
 * MLA models ([Irminsul] 2.1: 512-dim latent + 64-dim rope key per row):
 * every query head attends to the shared latent rows with its query absorbed
 * into the latent space, q = [q_nope (512) | q_rope (64)] (head_dim 576), so
 *   s_t = softmax_scale * (q_nope . cKV_t + q_rope . R(delta) k_r,t) + bias,
 *   out = sum_t softmax(s)_t cKV_t   (out: [num_layers][n_req][num_q_heads][512]);
 * only the rope part is rotated (with 16 heads per CTA the kernel rotates
 * q_rope by R(-delta); with 32 and more it rotates the rope keys on their way
 * through the SM), the latent is used as stored and serves as the value.  16, 32, 64 or 128
 * query heads (64 and 128 run as 2 and 4 groups of 32 that each read the
 * rows); v_pool and v_cache are ignored and may be NULL.  The cache's block tables are the plans' (as
 * pic_build_block_table returned them).  Two launches: a persistent kernel
 * streams the context through shared memory and leaves per-range softmax
 * records in the workspace, a second merges them into out and lse.
 * Device memory: the context keeps a device copy of the plan's read-only
 * image (stages, token rows, record keys: at most about 10 bytes per context
 * position, plus 8 per layer and request) for the last plan of each of two
 * kinds (one delta per stage, or up to two), and uploads
 * it again only when the plans, the layer count or the grid change, so a
 * decode loop over the same plans uploads nothing but a zeroed status word.
 * It is allocated stream-ordered on the call's stream and freed by
 * pic_destroy; a call that replaces it first waits (on the device) for
 * launches on any stream that still read it.  Errors:
 * PIC_ERR_UNSUPPORTED for other geometries or host-resident buffers,
 * PIC_ERR_RANGE for an empty context or a layer range outside the model,
 * PIC_ERR_CAPACITY for a short workspace; a bounded wait that gave up on the
 * device sets PIC_DEV_TIMEOUT in the workspace's status word.
 */
pic_status pic_attend_decode(pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req, int32_t source,
                             const void* q, int32_t num_q_heads, float softmax_scale, float sink_bias,
                             const void* k_pool, const void* v_pool, int64_t pool_layer_stride_bytes,
                             const void* k_cache, const void* v_cache, int64_t cache_layer_stride_bytes,
                             int32_t layer_begin, int32_t num_layers, float* out, float* lse,
                             void* d_workspace, size_t workspace_bytes, pic_stream_t stream);

/* ------------------------------------------- content-defined chunking */

/*
 * Chunk keys from content ([Irminsul] 2.2 "Content-Hash Keying with CDC":
 * boundaries from a rolling Gear hash over 64-token windows, a chunk ends
 * where the hash falls below a threshold, each chunk keyed by its xxHash64
 * fingerprint).  Document d is tokens [offsets[d], offsets[d + 1]) of
 * d_tokens; documents are chunked independently:
 *   h_i = 2 h_{i-1} + gear[t_i] (mod 2^64), h = 0 before the document's first
 *   token (so h_i depends on the 64 tokens t_{i-63} .. t_i only);
 *   a chunk ends after token i when h_i < threshold -- with min_len > 1 only
 *   once it holds min_len tokens, with max_len > 0 always once it holds
 *   max_len -- and the document's last token ends its last chunk.
 *   fingerprint = XXH64 (published specification) of the chunk's token ids as
 *   little-endian int32 bytes, with `seed`.  A registry key (pic_register_chunk)
 *   is the fingerprint's 8 bytes little-endian, zero-padded to 32.
 *   d_tokens       device int32 [n_tokens], 16-byte aligned.
 *   d_doc_offsets  device int64 [n_docs + 1]; checked on the device: offsets
 *                  that are not non-decreasing inside [0, n_tokens] raise
 *                  PIC_DEV_BAD_DOCS and every count comes out 0.
 *   d_gear         device uint64 [vocab]: one random 64-bit value per token id.
 *                  A token outside [0, vocab) counts as Gear value 0 and
 *                  raises PIC_DEV_BAD_TOKEN.
 *   threshold      e.g. 2^64 / mean_len for chunks of mean_len tokens on average.
 * Outputs (device, 8-byte aligned), in document order:
 *   d_chunk_indptr int64 [n_docs + 1]: document d owns chunks
 *                  [indptr[d], indptr[d + 1]); indptr[n_docs] is the total,
 *                  also when it exceeds capacity.
 *   d_chunk_ends   int64 [capacity]: one past each chunk's last token (a
 *                  chunk starts where the previous one of its document ended,
 *                  the first at offsets[d]).
 *   d_fingerprints uint64 [capacity], or NULL for no fingerprints.
 * Chunks past capacity are not written and raise PIC_DEV_CAPACITY; read the
 * total from indptr[n_docs] and call again with a larger buffer.
 * d_workspace: pic_cdc_workspace_bytes(n_tokens) bytes, 256-byte aligned; its
 * status word (PIC_DEV_* bits) is read with pic_query_device_status(NULL, ...).
 * Host-side argument errors return before anything is enqueued.
 */
size_t pic_cdc_workspace_bytes(int64_t n_tokens);
pic_status pic_cdc_chunk(const int32_t* d_tokens, int64_t n_tokens, const int64_t* d_doc_offsets,
                         int32_t n_docs, const uint64_t* d_gear, int32_t vocab, uint64_t threshold,
                         int32_t min_len, int32_t max_len, uint64_t seed, int64_t* d_chunk_indptr,
                         int64_t* d_chunk_ends, uint64_t* d_fingerprints, int64_t capacity,
                         void* d_workspace, size_t workspace_bytes, pic_stream_t stream);

/*
 * XXH64 of arbitrary token spans: d_out[k] = XXH64(token ids [d_starts[k],
 * d_ends[k]) as little-endian int32 bytes, seed) -- the fingerprint
 * pic_cdc_chunk computes, for spans the caller chooses (the S1 windows of a
 * chunk that missed the registry, [Irminsul] "Hybrid Strategies (S1/S2)").
 *   d_tokens  device int32 [n_tokens], 4-byte aligned.
 *   d_starts, d_ends  device int64 [n_spans]; d_out device uint64 [n_spans].
 *   d_status  device uint32, set to 0 and then OR-ed with PIC_DEV_BAD_SPAN for
 *             a span outside [0, n_tokens] or with end < start (its digest
 *             is written as 0).
 */
pic_status pic_fingerprint_spans(const int32_t* d_tokens, int64_t n_tokens, const int64_t* d_starts,
                                 const int64_t* d_ends, int64_t n_spans, uint64_t seed, uint64_t* d_out,
                                 uint32_t* d_status, pic_stream_t stream);

/*
 * S1 fallback windows of a chunk [begin, end) that missed the registry
 * ([Irminsul] "Hybrid Strategies (S1/S2)", S1: fixed 128-token windows):
 * window k is [begin + window*k, min(begin + window*(k + 1), end)).  Host
 * arrays; *count receives the number of windows; starts and ends may both be
 * NULL to query it; PIC_ERR_CAPACITY when count > capacity.
 */
pic_status pic_s1_windows(int64_t begin, int64_t end, int32_t window, int64_t* starts, int64_t* ends,
                          int64_t capacity, int64_t* count);

/* ---------------------------------------------------------- diagnostics */

/*
 * Synchronizes `stream`, then reads and clears nothing: returns the device
 * status word the last launch that used d_workspace left (0 = clean) in
 * *status_out, and PIC_ERR_DEVICE_CHECK when it is non-zero.  ctx may be NULL
 * (a chunking workspace); the message then goes to the calling thread.
 */
pic_status pic_query_device_status(pic_ctx* ctx, const void* d_workspace, pic_stream_t stream,
                                   uint32_t* status_out);

/*
 * Test hook for the failure paths of the kernels that wait on their own
 * copies: the bulk-copy pipeline of pic_stitch (pic_kernel_variant(ctx, 0) ==
 * PIC_VARIANT_BULK_PIPELINE) and the tcgen05 MLA attention of
 * pic_attend_decode (pic_kernel_variant(ctx, 2) ==
 * PIC_VARIANT_TENSOR_CORE_TMEM).  The next of those calls on ctx makes its
 * first CTA skip the copies and the barrier arrival of its tile stall_tile,
 * and bounds every barrier wait of that launch at max_spins tries (0: the
 * library's default bound).  The wait for that tile then runs out: the
 * launch raises PIC_DEV_TIMEOUT in the workspace status word, every thread
 * of the CTA leaves after bounded waits for the copies and products it did
 * start (the attention CTA also frees its tensor memory), and the context
 * stays usable.  Nothing faults or hangs; the other CTAs complete their
 * tiles.  The setting is used by exactly one pic_stitch or pic_attend_decode
 * (whichever kernel it runs) and then cleared; stall_tile < 0 clears it at
 * once.  The pages have no counterpart: this exists to test the library's
 * own failure detection.
 */
pic_status pic_debug_stall_next_launch(pic_ctx* ctx, int32_t stall_tile, uint32_t max_spins);

/*
 * Which kernel a context launches for mode 0 (pic_stitch / pic_stitch_noalloc)
 * or mode 1 (pic_rerotate_inplace): PIC_VARIANT_REGISTERS (16-byte vector
 * loads and stores through registers) or PIC_VARIANT_BULK_PIPELINE (bulk
 * async copies through a shared-memory ring).  The bulk pipeline is used when
 * one work unit fits a stage, unless the environment variable PIC_KERNEL was
 * "regs" at pic_create.  Both compute the same result.
 * Mode 2 (pic_attend_decode): PIC_VARIANT_TENSOR_CORE_TMEM (MLA models:
 * tcgen05 products with TMEM accumulators, rows loaded by TMA tensor copies;
 * chosen unless PIC_ATTEND_KERNEL was "mma" at pic_create) or
 * PIC_VARIANT_WARP_MMA (warp-level mma.sync products; GQA models, and MLA
 * when so chosen).  Both compute the same result to rounding.
 * -1 on bad arguments.
 */
#define PIC_VARIANT_REGISTERS 0
#define PIC_VARIANT_BULK_PIPELINE 1
#define PIC_VARIANT_TENSOR_CORE_TMEM 2
#define PIC_VARIANT_WARP_MMA 3
int32_t pic_kernel_variant(const pic_ctx* ctx, int32_t mode);

/*
 * The cos/sin the kernels use, for testing the angle arithmetic: for each of
 * the n shifts in d_deltas (device int32), writes rope_dim/2 (cos, sin) float
 * pairs of delta * theta_i to d_out (device float [n][rope_dim/2][2]).
 * d_workspace: >= 4096 bytes.
 */
pic_status pic_rotation_cossin(pic_ctx* ctx, const int32_t* d_deltas, int32_t n, float* d_out,
                               void* d_workspace, size_t workspace_bytes, pic_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PIC_H */
