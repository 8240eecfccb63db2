// Device helpers shared by the libnbx kernels: element formats, packed fp32 math,
// mbarrier / bulk-copy wrappers (inline PTX for sm_103a) and bounded waits.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "nbx.h"

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
// Blackwell executes two fp32 FMAs per instruction on a 64-bit register pair (fma.rn.f32x2).
// f32x2 holds such a pair (low half = element 0); keeping pairs in 64-bit registers through
// the hot loops avoids repacking around every packed instruction.
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unpack2(f32x2 v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// two bf16 (low half = element 0) -> packed fp32 pair
__device__ __forceinline__ f32x2 bf16x2_to_f32x2(uint32_t w) {
  f32x2 r;
  // low half: byte permute (bytes 0,1 of w to bytes 2,3, zeros below); high half: mask
  asm("{\n\t.reg .b32 lo, hi;\n\tprmt.b32 lo, %1, 0, 0x1044;\n\tand.b32 hi, %1, 0xffff0000;\n\tmov.b64 %0, {lo, hi};\n\t}"
      : "=l"(r)
      : "r"(w));
  return r;
}
__device__ __forceinline__ f32x2 e4m3x2_to_f32x2(uint32_t pair16) {
  const float2 f = e4m3x2_to_float2(pair16);
  return pack2(f.x, f.y);
}

// Unpack the 16-byte vector `v` of format T into packed pairs: out[k] holds elements 2k, 2k+1.
template <class T>
__device__ __forceinline__ void unpack16x2(const uint4& v, f32x2* out);
template <>
__device__ __forceinline__ void unpack16x2<F32>(const uint4& v, f32x2* out) {
  out[0] = (static_cast<f32x2>(v.y) << 32) | v.x;
  out[1] = (static_cast<f32x2>(v.w) << 32) | v.z;
}
template <>
__device__ __forceinline__ void unpack16x2<BF16>(const uint4& v, f32x2* out) {
  out[0] = bf16x2_to_f32x2(v.x);
  out[1] = bf16x2_to_f32x2(v.y);
  out[2] = bf16x2_to_f32x2(v.z);
  out[3] = bf16x2_to_f32x2(v.w);
}
template <>
__device__ __forceinline__ void unpack16x2<E4M3>(const uint4& v, f32x2* out) {
  out[0] = e4m3x2_to_f32x2(v.x & 0xffffu);
  out[1] = e4m3x2_to_f32x2(v.x >> 16);
  out[2] = e4m3x2_to_f32x2(v.y & 0xffffu);
  out[3] = e4m3x2_to_f32x2(v.y >> 16);
  out[4] = e4m3x2_to_f32x2(v.z & 0xffffu);
  out[5] = e4m3x2_to_f32x2(v.z >> 16);
  out[6] = e4m3x2_to_f32x2(v.w & 0xffffu);
  out[7] = e4m3x2_to_f32x2(v.w >> 16);
}

// Programmatic dependent launch: let the next kernel in the stream start its prologue early /
// wait until the kernel this one depends on has finished and its writes are visible.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// max that returns NaN if either input is NaN (fmaxf would drop it)
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// 2^x with the hardware approximation (relative error ~2^-22; ex2(-inf) = +0), results below
// 2^-126 flushed to +0. Every caller weights terms against a largest weight of at least 1 in the
// same sum (a softmax weight against the row maximum, a split against the largest split maximum),
// so a flushed weight is far below the sum's fp32 resolution; without the flush each call carries
// extra instructions for subnormal results.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
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

// Explicit shared-memory accesses on 32-bit shared addresses (volatile: they must stay behind
// the barrier waits that publish the data).
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ void lds2x64(uint32_t a, unsigned long long& x, unsigned long long& y) {
  asm volatile("ld.shared.v2.u64 {%0, %1}, [%2];" : "=l"(x), "=l"(y) : "r"(a));
}
__device__ __forceinline__ void sts64(uint32_t a, unsigned long long v) {
  asm volatile("st.shared.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
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

// try_wait: a thread whose phase has not completed may be suspended until it completes or a
// system-dependent time limit passes, so waiting warps leave the issue slots free. (An explicit
// suspend-time hint of 1 ms measured about 1 % slower on the SIMT partial.)
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

// 16-byte asynchronous copy global -> shared through L2 only (cp.async.cg; both addresses 16-byte
// aligned), tracked per thread.
__device__ __forceinline__ void cp_async16(uint32_t dst_smem, const void* src_gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst_smem), "l"(src_gmem) : "memory");
}
// The same with a source size of 16 or 0 bytes: with `valid` false nothing is read (the source
// address is not dereferenced) and the 16 destination bytes are zeroed.
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst_smem, const void* src_gmem, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst_smem), "l"(src_gmem), "r"(valid ? 16 : 0)
               : "memory");
}
// Arrives on `bar` once every cp.async this thread issued before has completed; the arrival is one
// of the barrier's expected arrivals (.noinc).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Waits for every cp.async this thread issued.
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Orders this thread's generic-proxy shared-memory accesses before later async-proxy accesses (bulk
// copies) of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

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
    if ((i & 3u) == 0u && global_timer_ns() - t0 > limit_ns) return false;
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

// An L2 policy that keeps the lines it writes ahead of ordinary ones. The decode's small
// intermediates (the split plan and work list, the fp32 split partials) are read back by later
// launches of the same call, while the K/V page tiles streaming through L2 in between would
// otherwise push them out to DRAM.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// The same, applied to the given fraction (0, 1] of the lines written.
__device__ __forceinline__ uint64_t l2_keep_policy(float frac) {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, %1;" : "=l"(pol) : "f"(frac));
  return pol;
}
__device__ __forceinline__ void st_global_hint(float* dst, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(dst), "f"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_global_hint(int4* dst, int4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.s32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(dst), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w), "l"(pol)
               : "memory");
}

// Named barrier over the first `threads` threads of the CTA (id 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ float4 ld_cg_f4(const float4* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
  return v;
}

// Counter in shared memory: add with release order / read with acquire order (CTA scope).
__device__ __forceinline__ void red_release_shared_add(int* p, int v) {
  asm volatile("red.release.cta.shared::cta.add.s32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_shared(volatile int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(const_cast<int*>(p))) : "memory");
  return v;
}

__device__ __forceinline__ float ld_cg_f32(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

}  // namespace nbx
