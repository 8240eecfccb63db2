// nbx_paged_decode_attn_noalloc: the paged decode attention with its scratch memory inside the
// library, for callers that cannot allocate device memory.
//
// nbx_paged_decode_attn needs a caller-provided workspace (the split plan, the work list and the
// fp32 split partials). Some callers cannot provide one: code that runs where cudaMalloc is not
// allowed or not wanted (inside an allocator's own callbacks, in a process whose memory budget
// is fixed before the library is loaded, or in a plug-in that has no handle on the host
// application's allocator). For them this entry point takes only the inputs and the output and
// uses a fixed scratch array that lives in the library's own device memory.
//
// The scratch is a file-scope __device__ array of NBX_NOALLOC_SCRATCH_BYTES. Every GPU that loads
// the library holds it until the process exits. In host code the array's name only stands for
// it; its device address is looked up with cudaGetSymbolAddress, once per device, on the first
// call made with that device current. That first call should therefore come before any stream
// capture. The address is kept for the life of the process: it does not survive a
// cudaDeviceReset of that device (or a different context made current on it), after which this
// entry point must not be called in the same process. All calls share the one array and it
// keeps the contents of the last call: the kernels rewrite everything they read (the plan kernel
// zeroes the work counter each call), and calls that overlap on the GPU (two streams, or two
// threads) race on it.
#include <cstdint>
#include <mutex>

#include "nbx_internal.h"

namespace nbx {
namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[NBX_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxScratchDevices = 64;
void* g_scratch_ptr[kMaxScratchDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device, looked up once per device.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxScratchDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace nbx

extern "C" NBX_API int nbx_paged_decode_attn_noalloc(const void* q, int q_dtype, int batch, int rows, int h_q, int d,
                                                      const void* k_pool, const void* v_pool, int pool_dtype,
                                                      int num_pages, int h_kv, int page_tokens,
                                                      const int32_t* block_table, int max_pages,
                                                      const int32_t* seq_lens, int max_seq_len, float scale,
                                                      float k_scale, float v_scale, float* out, int32_t* status,
                                                      void* stream) {
  const size_t need = nbx_paged_decode_workspace_bytes(batch, rows, h_q, h_kv, d, max_seq_len);
  if (need > static_cast<size_t>(NBX_NOALLOC_SCRATCH_BYTES)) return NBX_ERR_WORKSPACE;   // too large for the scratch
  void* scratch = nullptr;
  if (batch > 0 && need > 0) {
    if (nbx::scratch_address(&scratch) != cudaSuccess) return NBX_ERR_CUDA;
  }
  return nbx_paged_decode_attn(q, q_dtype, batch, rows, h_q, d, k_pool, v_pool, pool_dtype, num_pages, h_kv,
                               page_tokens, block_table, max_pages, seq_lens, max_seq_len, scale, k_scale, v_scale,
                               out, scratch, static_cast<size_t>(NBX_NOALLOC_SCRATCH_BYTES), status, stream);
}
