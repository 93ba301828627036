// Device helpers shared by the kernels of libpic (sm_103a): the RoPE angle
// reduction, bf16 <-> fp32 packing and pair rotation, and the PTX of
// mbarriers and bulk (TMA) copies.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace pic {
namespace dev {

constexpr unsigned kDevBadBlock = 0x1u;   // PIC_DEV_BAD_BLOCK
constexpr unsigned kDevTimeout = 0x2u;    // PIC_DEV_TIMEOUT
// Tries of one bounded mbarrier wait.  An unfinished try_wait suspends the
// thread for a few microseconds (about 4 us per try measured on GB300), so a
// wait gives up after about a second; a copy the kernel issued lands within
// microseconds.
constexpr uint32_t kMaxSpins = 1u << 18;

// cos / sin of delta * theta_i.  The host gives f_i = theta_i / (2 pi) as a
// float pair hi + lo; delta * hi is split exactly into p + e with one FMA
// (Dekker's TwoProduct), p's integer part is dropped exactly, the small terms
// are added back, and sincospif turns the fraction of a turn into cos / sin.
__device__ __forceinline__ void shift_cossin(int delta, float2 f, float& c, float& s) {
  const float d = static_cast<float>(delta);   // exact for |delta| < 2^24
  const float p = __fmul_rn(d, f.x);
  const float e = __fmaf_rn(d, f.x, -p);       // d * hi == p + e exactly
  const float r = __fsub_rn(p, rintf(p));      // exact, |r| <= 1/2 turn
  const float t = __fadd_rn(r, __fmaf_rn(d, f.y, e));
  sincospif(2.0f * t, &s, &c);                 // cos / sin of 2 pi t
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float2 bf_pair(uint32_t w) { return make_float2(bf_lo(w), bf_hi(w)); }
__device__ __forceinline__ uint32_t bf_pack(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // round to nearest even
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t& word(uint4& v, int w) {
  return w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w));
}

// Neox pair-vector: a holds x_a of frequencies f0..f0+7, b holds x_b of the same.
__device__ __forceinline__ void rotate_neox(uint4& a, uint4& b, const float* c, const float* s) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint32_t aw = word(a, w), bw = word(b, w);
    const float a0 = bf_lo(aw), a1 = bf_hi(aw), b0 = bf_lo(bw), b1 = bf_hi(bw);
    const float c0 = c[2 * w], s0 = s[2 * w], c1 = c[2 * w + 1], s1 = s[2 * w + 1];
    word(a, w) = bf_pack(a0 * c0 - b0 * s0, a1 * c1 - b1 * s1);
    word(b, w) = bf_pack(a0 * s0 + b0 * c0, a1 * s1 + b1 * c1);
  }
}

// Interleaved vector: word w holds the pair (x, y) of frequency f0 + w.
__device__ __forceinline__ void rotate_interleaved(uint4& v, const float* c, const float* s) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint32_t vw = word(v, w);
    const float x = bf_lo(vw), y = bf_hi(vw);
    word(v, w) = bf_pack(x * c[w] - y * s[w], x * s[w] + y * c[w]);
  }
}

// ------------------------------------------------ mbarriers and bulk copies

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// true when the phase completed, false after max_spins tries
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t max_spins = kMaxSpins) {
  for (uint32_t i = 0; i < max_spins; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
__device__ __forceinline__ void bulk_load(void* sdst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(sdst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_store(void* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_u32(ssrc)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace dev
}  // namespace pic
