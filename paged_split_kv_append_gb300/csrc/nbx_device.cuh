// Device helpers shared by the libnbx kernels: element formats, packed fp32 math,
// mbarrier / bulk-copy wrappers (inline PTX for sm_103a) and bounded waits.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "../../include/nbx.h"

namespace nbx {

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- element formats
// Tags of the pool / query element types. EPV = elements per 16-byte vector.
struct F32 {
  static constexpr int kCode = NBX_F32;
  static constexpr int kBytes = 4;
  static constexpr int kEPV = 4;
};
struct BF16 {
  static constexpr int kCode = NBX_BF16;
  static constexpr int kBytes = 2;
  static constexpr int kEPV = 8;
};
struct E4M3 {
  static constexpr int kCode = NBX_E4M3;
  static constexpr int kBytes = 1;
  static constexpr int kEPV = 16;
};

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  // bf16 is the upper half of a binary32: the low element sits in bits 0..15
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t pair16) {
  // hardware conversion of two E4M3 codes (low byte = element 0) to two halves, exact
  uint32_t h2;
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h2) : "r"(pair16));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// Unpack the 16-byte vector `v` of format T into floats, pairwise: out[k] holds elements 2k, 2k+1.
template <class T>
__device__ __forceinline__ void unpack16(const uint4& v, float2* out);

template <>
__device__ __forceinline__ void unpack16<F32>(const uint4& v, float2* out) {
  out[0] = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
  out[1] = make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
}
template <>
__device__ __forceinline__ void unpack16<BF16>(const uint4& v, float2* out) {
  out[0] = bf16x2_to_float2(v.x);
  out[1] = bf16x2_to_float2(v.y);
  out[2] = bf16x2_to_float2(v.z);
  out[3] = bf16x2_to_float2(v.w);
}
template <>
__device__ __forceinline__ void unpack16<E4M3>(const uint4& v, float2* out) {
  out[0] = e4m3x2_to_float2(v.x & 0xffffu);
  out[1] = e4m3x2_to_float2(v.x >> 16);
  out[2] = e4m3x2_to_float2(v.y & 0xffffu);
  out[3] = e4m3x2_to_float2(v.y >> 16);
  out[4] = e4m3x2_to_float2(v.z & 0xffffu);
  out[5] = e4m3x2_to_float2(v.z >> 16);
  out[6] = e4m3x2_to_float2(v.w & 0xffffu);
  out[7] = e4m3x2_to_float2(v.w >> 16);
}

// Two consecutive elements of format T at p (p aligned to 2 elements), as floats.
template <class T>
__device__ __forceinline__ float2 load_pair(const void* p);
template <>
__device__ __forceinline__ float2 load_pair<F32>(const void* p) {
  return *reinterpret_cast<const float2*>(p);
}
template <>
__device__ __forceinline__ float2 load_pair<BF16>(const void* p) {
  return bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(p));
}
template <>
__device__ __forceinline__ float2 load_pair<E4M3>(const void* p) {
  return e4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(p));
}

// ---------------------------------------------------------------- packed fp32 math
// Blackwell executes two fp32 FMAs per instruction on register pairs (fma.rn.f32x2).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// 2^x with the hardware approximation (relative error ~2^-22; ex2(-inf) = +0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------- status word
__device__ __forceinline__ void raise_status(int32_t* status, int32_t bits) {
  if (status != nullptr) atomicOr(status, bits);
}

// ---------------------------------------------------------------- mbarrier + bulk copy
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait for the phase of `bar` with the given parity to complete. Gives up after
// `limit_ns` nanoseconds of wall time and returns false (the caller records NBX_DEV_TIMEOUT).
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: no wait of a correct run comes near it

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0u && global_timer_ns() - t0 > limit_ns) return false;
  }
}

// One-dimensional bulk copy global -> shared, completing on `bar` (addresses 16-byte aligned,
// bytes a multiple of 16).
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Named barrier over the first `threads` threads of the CTA (id 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ float ld_cg_f32(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

}  // namespace nbx
