// The C ABI of libnbx: argument checks on the host, then the launches.
//
// Every check that the host can make happens before anything touches the GPU, mirroring
// the wrappers' refusals (nbxtensor/ops/attention_wrappers.py, paged_kv_append and
// paged_decode_attention: shapes that do not fit, non-int32 tables, a page that is not a
// whole number of tiles); the library then launches and returns without synchronising.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "nbx_internal.h"

namespace nbx {

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
bool g_info_ok[kMaxDevices];
std::mutex g_info_mu;
std::atomic<int> g_grid_limit{0};
constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;   // 2 s: no wait of a correct run comes near it
constexpr unsigned long long kMaxProducerDelayNs = 50000000ull;     // 50 ms
std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitLimitNs};
std::atomic<unsigned long long> g_producer_delay_ns{0};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool finite(float x) { return std::isfinite(x); }
}  // namespace

const DeviceInfo& device_info() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) dev = 0;
  std::lock_guard<std::mutex> lock(g_info_mu);
  if (!g_info_ok[dev]) {
    DeviceInfo di;
    di.device = dev;
    di.sm_count = 0;
    di.max_smem_optin = 0;
    cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&di.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (di.sm_count < 1) di.sm_count = 1;
    g_info[dev] = di;
    g_info_ok[dev] = true;
  }
  return g_info[dev];
}

}  // namespace nbx

using namespace nbx;

extern "C" {

NBX_API int nbx_abi_version(void) { return 100; }

NBX_API const char* nbx_status_string(int status) {
  switch (status) {
    case NBX_OK: return "ok";
    case NBX_ERR_NULL: return "a required pointer is NULL";
    case NBX_ERR_SHAPE: return "sizes do not fit together or are outside the supported set";
    case NBX_ERR_DTYPE: return "unsupported dtype code";
    case NBX_ERR_PAGE_ALIGN: return "page_tokens is not a multiple of the 16-position tile";
    case NBX_ERR_WORKSPACE: return "workspace too small";
    case NBX_ERR_CUDA: return "CUDA runtime error";
    case NBX_ERR_ALIGN: return "buffer not 16-byte aligned";
    case NBX_ERR_VALUE: return "scalar argument not finite, or scale not positive";
    default: return "unknown status";
  }
}

NBX_API void nbx_set_decode_grid_limit(int max_ctas) { g_grid_limit.store(max_ctas < 0 ? 0 : max_ctas); }

NBX_API void nbx_set_decode_wait_test(unsigned long long wait_limit_ns, unsigned long long producer_delay_ns) {
  g_wait_limit_ns.store(wait_limit_ns == 0 ? kDefaultWaitLimitNs : wait_limit_ns);
  g_producer_delay_ns.store(producer_delay_ns > kMaxProducerDelayNs ? kMaxProducerDelayNs : producer_delay_ns);
}

NBX_API int nbx_paged_kv_append(const void* new_k, const void* new_v, int new_dtype, int n_tok, int h_kv, int d,
                                void* k_pool, void* v_pool, int pool_dtype, int num_pages, int page_tokens,
                                const int32_t* slot_mapping, float k_scale, float v_scale, int32_t* status,
                                void* stream) {
  if (n_tok < 0 || h_kv < 1 || d < 16 || d > 1024 || (d % 16) != 0 || num_pages < 1 || page_tokens < 1)
    return NBX_ERR_SHAPE;
  if (new_dtype != NBX_F32 && new_dtype != NBX_BF16) return NBX_ERR_DTYPE;
  if (pool_dtype != NBX_F32 && pool_dtype != NBX_BF16 && pool_dtype != NBX_E4M3) return NBX_ERR_DTYPE;
  if (!finite(k_scale) || !finite(v_scale) || !(k_scale > 0.f) || !(v_scale > 0.f)) return NBX_ERR_VALUE;
  if (n_tok == 0) return NBX_OK;
  if (!new_k || !new_v || !k_pool || !v_pool || !slot_mapping) return NBX_ERR_NULL;
  if (!aligned16(new_k) || !aligned16(new_v) || !aligned16(k_pool) || !aligned16(v_pool)) return NBX_ERR_ALIGN;
  AppendParams p = {};
  p.new_k = new_k;
  p.new_v = new_v;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.slot_mapping = slot_mapping;
  p.status = status;
  p.n_tok = n_tok;
  p.h_kv = h_kv;
  p.d = d;
  p.num_pages = num_pages;
  p.page_tokens = page_tokens;
  p.k_inv = 1.0f / k_scale;
  p.v_inv = 1.0f / v_scale;
  const cudaError_t e = append_dispatch(p, new_dtype, pool_dtype, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NBX_OK : NBX_ERR_CUDA;
}

static bool decode_shape_ok(int batch, int rows, int h_q, int h_kv, int d, int max_seq_len) {
  if (batch < 0 || rows < 1 || h_q < 1 || h_kv < 1 || (h_q % h_kv) != 0) return false;
  if (d != 64 && d != 128 && d != 256) return false;
  if (max_seq_len < 0) return false;
  return true;
}

NBX_API int nbx_paged_decode_partial_kernel(int q_dtype, int pool_dtype, int rows, int h_q, int h_kv, int d,
                                            int num_pages, int page_tokens) {
  if (!decode_shape_ok(1, rows, h_q, h_kv, d, 0) || num_pages < 1 || page_tokens < 1) return NBX_ERR_SHAPE;
  if ((page_tokens % NBX_TILE_POSITIONS) != 0) return NBX_ERR_PAGE_ALIGN;
  if (q_dtype != NBX_F32 && q_dtype != NBX_BF16) return NBX_ERR_DTYPE;
  if (pool_dtype != NBX_F32 && pool_dtype != NBX_BF16 && pool_dtype != NBX_E4M3) return NBX_ERR_DTYPE;
  DecodeParams p = {};
  p.rows = rows;
  p.h_q = h_q;
  p.h_kv = h_kv;
  p.group = h_q / h_kv;
  p.d = d;
  p.num_pages = num_pages;
  p.page_tokens = page_tokens;
  p.qk_scale_log2 = 1.f;   // a positive softmax scale
  if (!mma_path_applies(p, q_dtype, pool_dtype)) return NBX_PARTIAL_SIMT;
  return pool_dtype == NBX_E4M3 ? NBX_PARTIAL_TCGEN05_FP8 : NBX_PARTIAL_TCGEN05;
}

NBX_API size_t nbx_paged_decode_workspace_bytes(int batch, int rows, int h_q, int h_kv, int d, int max_seq_len) {
  if (!decode_shape_ok(batch, rows, h_q, h_kv, d, max_seq_len)) return 0;
  WorkspaceLayout w;
  if (!workspace_layout(batch, rows, h_q, h_kv, d, max_seq_len, &w)) return 0;
  return w.total;
}

NBX_API size_t nbx_paged_decode_workspace_bytes_for(int q_dtype, int pool_dtype, int batch, int rows, int h_q,
                                                    int h_kv, int d, int max_seq_len, int page_tokens) {
  if (!decode_shape_ok(batch, rows, h_q, h_kv, d, max_seq_len)) return 0;
  (void)q_dtype;
  (void)pool_dtype;
  (void)page_tokens;
  WorkspaceLayout w;
  if (!workspace_layout(batch, rows, h_q, h_kv, d, max_seq_len, &w)) return 0;
  return w.total;
}

// The decode call behind every decode entry point. `identity` reads the pools as one page per
// sequence through an identity block table the plan kernel writes into the workspace; `lens_out`
// and `len_add` make it a decode step's (attend with seq_lens + len_add, write that length back).
static int decode_call(const void* q, int q_dtype, int batch, int rows, int h_q, int d, const void* k_pool,
                       const void* v_pool, int pool_dtype, int num_pages, int h_kv, int page_tokens,
                       const int32_t* block_table, int max_pages, const int32_t* seq_lens, int max_seq_len,
                       float scale, float k_scale, float v_scale, float* out, void* workspace,
                       size_t workspace_bytes, int32_t* status, cudaStream_t stream, bool identity,
                       int32_t* lens_out, int len_add, const float* fs_q_norm = nullptr,
                       const float* fs_kv_max = nullptr) {
  if (!decode_shape_ok(batch, rows, h_q, h_kv, d, max_seq_len)) return NBX_ERR_SHAPE;
  if (num_pages < 1 || page_tokens < 1 || max_pages < 1) return NBX_ERR_SHAPE;
  if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_pages) * page_tokens) return NBX_ERR_SHAPE;
  if ((page_tokens % NBX_TILE_POSITIONS) != 0) return NBX_ERR_PAGE_ALIGN;
  if (q_dtype != NBX_F32 && q_dtype != NBX_BF16) return NBX_ERR_DTYPE;
  if (pool_dtype != NBX_F32 && pool_dtype != NBX_BF16 && pool_dtype != NBX_E4M3) return NBX_ERR_DTYPE;
  if (!finite(scale) || !finite(k_scale) || !finite(v_scale) || !(k_scale > 0.f) || !(v_scale > 0.f))
    return NBX_ERR_VALUE;
  if (batch == 0) return NBX_OK;
  if (!q || !k_pool || !v_pool || (!identity && !block_table) || !seq_lens || !out || !workspace) return NBX_ERR_NULL;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out)) return NBX_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return NBX_ERR_ALIGN;
  WorkspaceLayout w;
  if (!workspace_layout(batch, rows, h_q, h_kv, d, max_seq_len, &w)) return NBX_ERR_SHAPE;
  if (workspace_bytes < w.total) return NBX_ERR_WORKSPACE;

  char* ws = static_cast<char*>(workspace);
  DecodeParams p = {};
  p.q = q;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.ident_bt = identity ? reinterpret_cast<int32_t*>(ws + w.ident_bt) : nullptr;
  p.block_table = identity ? p.ident_bt : block_table;
  p.seq_lens = seq_lens;
  p.lens_out = lens_out;
  p.len_add = len_add;
  p.out = out;
  p.status = status;
  p.header = reinterpret_cast<int32_t*>(ws + w.header);
  p.plan = reinterpret_cast<SeqPlan*>(ws + w.plan);
  p.entries = reinterpret_cast<Entry*>(ws + w.entries);
  p.m_part = reinterpret_cast<float*>(ws + w.m_part);
  p.l_part = reinterpret_cast<float*>(ws + w.l_part);
  p.acc_part = reinterpret_cast<float*>(ws + w.acc_part);
  p.batch = batch;
  p.rows = rows;
  p.h_q = h_q;
  p.h_kv = h_kv;
  p.group = h_q / h_kv;
  p.d = d;
  p.num_pages = num_pages;
  p.page_tokens = page_tokens;
  p.max_pages = max_pages;
  p.max_seq_len = max_seq_len;
  p.max_splits = w.max_splits;
  p.row_blocks = w.row_blocks;
  p.qk_scale_log2 = scale * k_scale * kLog2eHost;
  p.v_scale = v_scale;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.fs_q_norm = fs_q_norm;
  p.fs_kv_max = fs_kv_max;
  p.fs_scale_log2 = scale * kLog2eHost;
  p.k_scale_host = k_scale;
  p.producer_delay_ns = g_producer_delay_ns.load();
  {
    const double part_bytes = static_cast<double>(batch) * rows * h_q * w.max_splits * d * 4.0;
    p.keep_frac = static_cast<float>(part_bytes <= 67108864.0 ? 1.0 : 67108864.0 / part_bytes);
  }
  const cudaError_t e = decode_dispatch(p, q_dtype, pool_dtype, g_grid_limit.load(), stream);
  return e == cudaSuccess ? NBX_OK : NBX_ERR_CUDA;
}

NBX_API int nbx_paged_decode_attn(const void* q, int q_dtype, int batch, int rows, int h_q, int d,
                                  const void* k_pool, const void* v_pool, int pool_dtype, int num_pages, int h_kv,
                                  int page_tokens, const int32_t* block_table, int max_pages,
                                  const int32_t* seq_lens, int max_seq_len, float scale, float k_scale,
                                  float v_scale, float* out, void* workspace, size_t workspace_bytes,
                                  int32_t* status, void* stream) {
  return decode_call(q, q_dtype, batch, rows, h_q, d, k_pool, v_pool, pool_dtype, num_pages, h_kv, page_tokens,
                     block_table, max_pages, seq_lens, max_seq_len, scale, k_scale, v_scale, out, workspace,
                     workspace_bytes, status, static_cast<cudaStream_t>(stream), false, nullptr, 0);
}

NBX_API int nbx_paged_decode_attn_fixed_shift(const void* q, int q_dtype, int batch, int rows, int h_q, int d,
                                              const void* k_pool, const void* v_pool, int pool_dtype, int num_pages,
                                              int h_kv, int page_tokens, const int32_t* block_table, int max_pages,
                                              const int32_t* seq_lens, int max_seq_len, float scale, float k_scale,
                                              float v_scale, float* out, void* workspace, size_t workspace_bytes,
                                              const float* q_norm, const float* kv_max, int32_t* status,
                                              void* stream) {
  if (batch > 0 && (q_norm == nullptr || kv_max == nullptr)) return NBX_ERR_NULL;
  return decode_call(q, q_dtype, batch, rows, h_q, d, k_pool, v_pool, pool_dtype, num_pages, h_kv, page_tokens,
                     block_table, max_pages, seq_lens, max_seq_len, scale, k_scale, v_scale, out, workspace,
                     workspace_bytes, status, static_cast<cudaStream_t>(stream), false, nullptr, 0, q_norm, kv_max);
}

NBX_API int nbx_paged_decode_bounds(const void* q, int q_dtype, int batch, int rows, int h_q, int d, const void* k_pool,
                                    const void* v_pool, int pool_dtype, int num_pages, int h_kv, int page_tokens,
                                    const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                                    int max_seq_len, float k_scale, float v_scale, float* q_norm, float* kv_max,
                                    int32_t* status, void* stream) {
  if (!decode_shape_ok(batch, rows, h_q, h_kv, d, max_seq_len)) return NBX_ERR_SHAPE;
  if (num_pages < 1 || page_tokens < 1 || max_pages < 1) return NBX_ERR_SHAPE;
  if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_pages) * page_tokens) return NBX_ERR_SHAPE;
  if (q_dtype != NBX_F32 && q_dtype != NBX_BF16) return NBX_ERR_DTYPE;
  if (pool_dtype != NBX_F32 && pool_dtype != NBX_BF16 && pool_dtype != NBX_E4M3) return NBX_ERR_DTYPE;
  if (!finite(k_scale) || !finite(v_scale) || !(k_scale > 0.f) || !(v_scale > 0.f)) return NBX_ERR_VALUE;
  if (batch == 0) return NBX_OK;
  if (!q || !k_pool || !v_pool || !block_table || !seq_lens || !q_norm || !kv_max) return NBX_ERR_NULL;
  DecodeParams p = {};
  p.q = q;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.status = status;
  p.batch = batch;
  p.rows = rows;
  p.h_q = h_q;
  p.h_kv = h_kv;
  p.d = d;
  p.num_pages = num_pages;
  p.page_tokens = page_tokens;
  p.max_pages = max_pages;
  p.max_seq_len = max_seq_len;
  p.v_scale = v_scale;
  p.k_scale_host = k_scale;
  const cudaError_t e = bounds_dispatch(p, q_dtype, pool_dtype, q_norm, kv_max, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NBX_OK : NBX_ERR_CUDA;
}

NBX_API int nbx_decode_fixed_shift_gate(int n_keys, double v_max_bound, int* c_out, int* gate_out) {
  if (n_keys < 1 || !(v_max_bound >= 1.0) || !std::isfinite(v_max_bound) || !c_out || !gate_out) return NBX_ERR_VALUE;
  int lg_n = 0;
  while ((1ll << lg_n) < n_keys) ++lg_n;   // ceil(log2 n)
  const int lg_v = static_cast<int>(std::ceil(std::log2(v_max_bound)));
  *c_out = 127 - lg_n - lg_v;
  const int w = *c_out + 125;
  *gate_out = w >= 0 ? w / 2 : -((1 - w) / 2);   // floor(w / 2)
  return NBX_OK;
}

NBX_API int nbx_decode_attn_contiguous(const void* q, int q_dtype, int batch, int rows, int h_q, int d,
                                       const void* k_cache, const void* v_cache, int cache_dtype, int h_kv,
                                       int capacity, const int32_t* seq_lens, int max_seq_len, float scale,
                                       float k_scale, float v_scale, float* out, void* workspace,
                                       size_t workspace_bytes, int32_t* status, void* stream) {
  // [batch, h_kv, capacity, d] is the pool layout with one page of `capacity` positions per sequence
  if (capacity < 1) return NBX_ERR_SHAPE;
  return decode_call(q, q_dtype, batch, rows, h_q, d, k_cache, v_cache, cache_dtype, batch < 1 ? 1 : batch, h_kv,
                     capacity, nullptr, 1, seq_lens, max_seq_len, scale, k_scale, v_scale, out, workspace,
                     workspace_bytes, status, static_cast<cudaStream_t>(stream), true, nullptr, 0);
}

NBX_API int nbx_paged_decode_step(const void* q, int q_dtype, int batch, int rows, int h_q, int d, const void* new_k,
                                  const void* new_v, int new_dtype, void* k_pool, void* v_pool, int pool_dtype,
                                  int num_pages, int h_kv, int page_tokens, const int32_t* block_table, int max_pages,
                                  int32_t* lens, int max_seq_len, float scale, float k_scale, float v_scale,
                                  float* out, void* workspace, size_t workspace_bytes, int32_t* status,
                                  void* stream) {
  // every check of the decode first, so an invalid call launches nothing
  if (!decode_shape_ok(batch, rows, h_q, h_kv, d, max_seq_len)) return NBX_ERR_SHAPE;
  if (new_dtype != NBX_F32 && new_dtype != NBX_BF16) return NBX_ERR_DTYPE;
  if (num_pages < 1 || page_tokens < 1 || max_pages < 1) return NBX_ERR_SHAPE;
  if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_pages) * page_tokens) return NBX_ERR_SHAPE;
  if ((page_tokens % NBX_TILE_POSITIONS) != 0) return NBX_ERR_PAGE_ALIGN;
  if (q_dtype != NBX_F32 && q_dtype != NBX_BF16) return NBX_ERR_DTYPE;
  if (pool_dtype != NBX_F32 && pool_dtype != NBX_BF16 && pool_dtype != NBX_E4M3) return NBX_ERR_DTYPE;
  if (!finite(scale) || !finite(k_scale) || !finite(v_scale) || !(k_scale > 0.f) || !(v_scale > 0.f))
    return NBX_ERR_VALUE;
  if (batch == 0) return NBX_OK;
  if (!q || !new_k || !new_v || !k_pool || !v_pool || !block_table || !lens || !out || !workspace) return NBX_ERR_NULL;
  if (!aligned16(new_k) || !aligned16(new_v) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) ||
      !aligned16(out))
    return NBX_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return NBX_ERR_ALIGN;
  WorkspaceLayout w;
  if (!workspace_layout(batch, rows, h_q, h_kv, d, max_seq_len, &w)) return NBX_ERR_SHAPE;
  if (workspace_bytes < w.total) return NBX_ERR_WORKSPACE;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the step's rows new positions per sequence, written at lens[b] .. lens[b] + rows - 1
  AppendParams a = {};
  a.new_k = new_k;
  a.new_v = new_v;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.status = status;
  a.n_tok = batch * rows;
  a.h_kv = h_kv;
  a.d = d;
  a.num_pages = num_pages;
  a.page_tokens = page_tokens;
  a.k_inv = 1.0f / k_scale;
  a.v_inv = 1.0f / v_scale;
  a.lens = lens;
  a.block_table = block_table;
  a.max_pages = max_pages;
  a.rows = rows;
  a.max_pos = max_seq_len;
  cudaError_t e = append_dispatch(a, new_dtype, pool_dtype, st);
  if (e != cudaSuccess) return NBX_ERR_CUDA;
  // then the decode with the advanced lengths; its plan kernel writes them back to lens
  return decode_call(q, q_dtype, batch, rows, h_q, d, k_pool, v_pool, pool_dtype, num_pages, h_kv, page_tokens,
                     block_table, max_pages, lens, max_seq_len, scale, k_scale, v_scale, out, workspace,
                     workspace_bytes, status, st, false, lens, rows);
}

NBX_API int nbx_paged_decode_merge(const float* acc_part, const float* m_part, const float* l_part, int n_rows,
                                   int splits, int d, float* out, void* stream) {
  if (n_rows < 0 || splits < 1 || splits > 4096 || d < 1 || d > 1024) return NBX_ERR_SHAPE;
  if (n_rows == 0) return NBX_OK;
  if (!acc_part || !m_part || !l_part || !out) return NBX_ERR_NULL;
  MergeParams p;
  p.acc_part = acc_part;
  p.m_part = m_part;
  p.l_part = l_part;
  p.out = out;
  p.n_rows = n_rows;
  p.splits = splits;
  p.d = d;
  const cudaError_t e = merge_dispatch(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? NBX_OK : NBX_ERR_CUDA;
}

}  // extern "C"
