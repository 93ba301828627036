// pic_stitch_noalloc: the stitch for callers that must not allocate.
//
// Some callers cannot allocate GPU memory where they stitch: a serving
// engine that has already handed (nearly) all of HBM to its own KV-cache
// block pool and forbids other allocations, a host framework that gives a
// plugin only the tensors it reads and writes, or a loop that must not pay
// for cudaMalloc / cudaFree (cudaFree synchronizes the whole device).  For
// them this entry point runs the same stitch kernel as pic_stitch, but its
// scratch (the per-launch run list, frequency table and status word) lives
// in a fixed array of device memory that belongs to this library, declared
// below, instead of a caller workspace.  The caller still passes every input
// and output buffer.
//
// The array is a file-scope __device__ variable: each GPU that loads the
// library holds kScratchBytes of it until the process exits.  Host code may
// not use its name as a pointer (on the host it is only a stand-in for the
// symbol), so its device address is looked up once per device with
// cudaGetSymbolAddress and then passed to the kernel like any other pointer.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <mutex>

#include "pic.h"
#include "pic_internal.h"

namespace {

// 4 MiB: room for about 130,000 runs of up to block_size tokens per launch
// (two million tokens at block size 16), with the header, frequency table
// and CSR offsets.
constexpr size_t kScratchBytes = 4u << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Host image of one launch's scratch, uploaded with a pageable copy (which
// the runtime may hold until the stream's earlier work is done).  Static
// too, so nothing is allocated per call.
alignas(256) unsigned char g_host_image[kScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace

extern "C" pic_status pic_stitch_noalloc(pic_ctx* ctx, const pic_plan* const* plans, int32_t n_req,
                                         const void* k_pool, const void* v_pool,
                                         int64_t pool_layer_stride_bytes, void* k_cache,
                                         void* v_cache, int64_t cache_layer_stride_bytes,
                                         const int32_t* d_block_tables, int32_t max_blocks,
                                         int32_t* d_recompute_idx, int32_t* d_recompute_indptr,
                                         int64_t recompute_capacity, uint32_t* d_status,
                                         pic_stream_t stream) {
  if (!ctx) return pic::set_error(nullptr, PIC_ERR_INVALID_ARG, "null ctx");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    char msg[256];
    std::snprintf(msg, sizeof(msg), "cudaGetDevice: %s", cudaGetErrorString(e));
    return pic::set_error(ctx, PIC_ERR_CUDA, msg);
  }
  if (dev < 0 || dev >= kMaxDevices) return pic::set_error(ctx, PIC_ERR_UNSUPPORTED, "device index too large");
  void* scratch = nullptr;
  {
    // First call on this device (with it current): find the array's device address.
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_scratch);
      if (e != cudaSuccess || p == nullptr) {
        char msg[256];
        std::snprintf(msg, sizeof(msg), "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
        return pic::set_error(ctx, PIC_ERR_CUDA, msg);
      }
      g_scratch_addr[dev] = p;
    }
    scratch = g_scratch_addr[dev];
  }
  return pic::stitch_with_scratch(ctx, plans, n_req, k_pool, v_pool, pool_layer_stride_bytes, k_cache,
                                  v_cache, cache_layer_stride_bytes, d_block_tables, max_blocks,
                                  d_recompute_idx, d_recompute_indptr, recompute_capacity, scratch,
                                  kScratchBytes, g_host_image, sizeof(g_host_image), d_status,
                                  reinterpret_cast<cudaStream_t>(stream));
}
