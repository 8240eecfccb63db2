// Kernel 1: the slot-mapping append, cast on store; in decode-step mode the slots come from the
// device lengths and the block table (nbxtensor/ops/paged_decode_attn.py, paged_kv_append_step_kernel:
// the step writes at the layer's device length, so a recorded launch replays unchanged).
//
// nbxtensor/ops/paged_decode_attn.py, paged_kv_append_kernel: one program per (new token,
// KV head) writes its D values to pool[slot / page_tokens, h, slot % page_tokens, :], converted
// to the pool's element type. Here one warp handles one (token, head, K-or-V) row: each lane
// moves 4 consecutive elements per pass (a 16-byte fp32 load or an 8-byte bf16 load, one
// multiply by the reciprocal pool scale, one packed conversion, one 16/8/4-byte store), so a
// row of D elements takes D/128 passes and every access is coalesced.
#include "nbx_device.cuh"
#include "nbx_internal.h"

namespace nbx {
namespace {

template <class In>
__device__ __forceinline__ float4 load4(const void* p);
template <>
__device__ __forceinline__ float4 load4<F32>(const void* p) {
  return *reinterpret_cast<const float4*>(p);
}
template <>
__device__ __forceinline__ float4 load4<BF16>(const void* p) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  const float2 a = bf16x2_to_float2(w.x), b = bf16x2_to_float2(w.y);
  return make_float4(a.x, a.y, b.x, b.y);
}

template <class Out>
__device__ __forceinline__ void store4(void* p, float4 v);
template <>
__device__ __forceinline__ void store4<F32>(void* p, float4 v) {
  *reinterpret_cast<float4*>(p) = v;
}
template <>
__device__ __forceinline__ void store4<BF16>(void* p, float4 v) {
  // round to nearest even (CUDA's conversion)
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 w;
  w.x = *reinterpret_cast<uint32_t*>(&a);
  w.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = w;
}
template <>
__device__ __forceinline__ void store4<E4M3>(void* p, float4 v) {
  // round to nearest even with saturation to the largest finite value (CUDA's conversion)
  const __nv_fp8x2_storage_t a = __nv_cvt_float2_to_fp8x2(make_float2(v.x, v.y), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t b = __nv_cvt_float2_to_fp8x2(make_float2(v.z, v.w), __NV_SATFINITE, __NV_E4M3);
  *reinterpret_cast<uint32_t*>(p) = static_cast<uint32_t>(a) | (static_cast<uint32_t>(b) << 16);
}

template <class In, class Out>
__global__ void __launch_bounds__(256) append_kernel(AppendParams p) {
  // a decode launched next may start its plan now: the plan reads only the lengths and waits for
  // this grid before it writes any of them, and the decode's own kernels wait for the plan
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t rows = static_cast<int64_t>(p.n_tok) * p.h_kv * 2;
  const int64_t pool_positions = static_cast<int64_t>(p.num_pages) * p.page_tokens;
  for (int64_t w = warp; w < rows; w += n_warps) {
    const int which = static_cast<int>(w & 1);            // 0: K, 1: V
    const int64_t th = w >> 1;
    const int64_t t = th / p.h_kv;
    const int h = static_cast<int>(th - t * p.h_kv);
    int64_t slot;
    if (p.lens == nullptr) {
      slot = p.slot_mapping[t];
    } else {   // decode step: the position comes from the device length, the page from the table
      const int64_t b = t / p.rows;
      const int64_t pos = static_cast<int64_t>(p.lens[b]) + (t - b * p.rows);
      if (pos < 0 || pos >= p.max_pos) {
        if (lane == 0 && which == 0 && h == 0) raise_status(p.status, NBX_DEV_BAD_LEN);
        continue;
      }
      const int32_t pg = p.block_table[b * p.max_pages + pos / p.page_tokens];
      if (pg < 0 || pg >= p.num_pages) {
        if (lane == 0 && which == 0 && h == 0) raise_status(p.status, NBX_DEV_BAD_PAGE);
        continue;
      }
      slot = static_cast<int64_t>(pg) * p.page_tokens + pos % p.page_tokens;
    }
    if (slot < 0 || slot >= pool_positions) {
      if (lane == 0 && which == 0 && h == 0) raise_status(p.status, NBX_DEV_BAD_SLOT);
      continue;
    }
    const int64_t page = slot / p.page_tokens;
    const int64_t pos = slot - page * p.page_tokens;
    const char* src = static_cast<const char*>(which ? p.new_v : p.new_k) +
                      ((t * p.h_kv + h) * p.d) * In::kBytes;
    char* dst = static_cast<char*>(which ? p.v_pool : p.k_pool) +
                (((page * p.h_kv + h) * p.page_tokens + pos) * p.d) * Out::kBytes;
    const float inv = which ? p.v_inv : p.k_inv;
    for (int e = lane * 4; e < p.d; e += 128) {
      float4 x = load4<In>(src + static_cast<int64_t>(e) * In::kBytes);
      x.x *= inv;
      x.y *= inv;
      x.z *= inv;
      x.w *= inv;
      store4<Out>(dst + static_cast<int64_t>(e) * Out::kBytes, x);
    }
  }
}

template <class In, class Out>
cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(p.n_tok) * p.h_kv * 2;
  const int threads = 256;
  int64_t blocks = (rows * 32 + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(device_info().sm_count) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  append_kernel<In, Out><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t append_dispatch(const AppendParams& p, int new_dtype, int pool_dtype, cudaStream_t stream) {
  if (new_dtype == NBX_F32) {
    if (pool_dtype == NBX_F32) return launch_append<F32, F32>(p, stream);
    if (pool_dtype == NBX_BF16) return launch_append<F32, BF16>(p, stream);
    return launch_append<F32, E4M3>(p, stream);
  }
  if (pool_dtype == NBX_F32) return launch_append<BF16, F32>(p, stream);
  if (pool_dtype == NBX_BF16) return launch_append<BF16, BF16>(p, stream);
  return launch_append<BF16, E4M3>(p, stream);
}

}  // namespace nbx
