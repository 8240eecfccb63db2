// Host-side internals of libnbx: launch parameter blocks, the workspace layout and the
// per-device launch facts. Not part of the C ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "nbx.h"

namespace nbx {

constexpr float kLog2eHost = 1.4426950408889634f;

struct DeviceInfo {
  int device;
  int sm_count;
  int max_smem_optin;
};

// Facts of the current device, queried once per device.
const DeviceInfo& device_info();

struct AppendParams {
  const void* new_k;
  const void* new_v;
  void* k_pool;
  void* v_pool;
  const int32_t* slot_mapping;
  int32_t* status;
  int n_tok, h_kv, d, num_pages, page_tokens;
  float k_inv, v_inv;
  // decode-step mode (lens != null): token t = b * rows + r goes to position lens[b] + r of
  // sequence b, its page read from the block table; positions at or past max_pos are refused
  const int32_t* lens;
  const int32_t* block_table;
  int max_pages, rows, max_pos;
};

cudaError_t append_dispatch(const AppendParams& p, int new_dtype, int pool_dtype, cudaStream_t stream);

// ---------------------------------------------------------------- decode
constexpr int kTileN = NBX_TILE_POSITIONS;  // positions per staged tile
constexpr int kQB = 4;                      // query vectors (rows x heads of one KV head) per work unit
constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;

// One sequence of the split plan.
struct SeqPlan {
  int32_t len;       // positions read (0 if the length was out of bounds)
  int32_t seg;       // positions per split (a whole number of pages)
  int32_t n_splits;  // non-empty splits: ceil(len / seg)
  int32_t pad;
};

// One (sequence, split) of the work list; a work unit is (entry, KV head, row block). The
// sequence's length and split count ride along, so a unit is described by one 32-byte load.
struct Entry {
  int32_t b, s, start, end;
  int32_t len, n_splits, pad0, pad1;
};
static_assert(sizeof(Entry) == 32, "Entry is one 32-byte load");

// Byte offsets of the workspace sections (each 256-byte aligned).
struct WorkspaceLayout {
  size_t header;    // int32[64]: [0] entries in the list, [1] work counter
  size_t ident_bt;  // int32[batch]: the identity block table of a contiguous cache (row b = page b)
  size_t plan;      // SeqPlan[batch]
  size_t entries;   // Entry[batch * max_splits]
  size_t m_part;    // f32[batch * rows * h_q * max_splits]   (log2 units)
  size_t l_part;    // f32[batch * rows * h_q * max_splits]
  size_t acc_part;  // f32[batch * rows * h_q * max_splits * d]
  size_t total;
  int max_splits;
  int row_blocks;
};

// Returns false if the sizes overflow.
bool workspace_layout(int batch, int rows, int h_q, int h_kv, int d, int max_seq_len, WorkspaceLayout* out);

int splits_for(int length);

struct DecodeParams {
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const int32_t* block_table;
  const int32_t* seq_lens;
  float* out;
  int32_t* status;
  // workspace sections
  int32_t* header;
  SeqPlan* plan;
  Entry* entries;
  float* m_part;
  float* l_part;
  float* acc_part;
  int batch, rows, h_q, h_kv, group, d, num_pages, page_tokens, max_pages, max_seq_len;
  int max_splits, row_blocks;
  float qk_scale_log2;  // scale * k_scale * log2(e): scores in log2 units
  float v_scale;
  // the plan kernel writes ident_bt[b] = b (a contiguous cache read as one page per sequence;
  // block_table then points at it), and, for a decode step, attends with seq_lens[b] + len_add
  // and writes that length to lens_out[b] (null: neither)
  int32_t* ident_bt;
  int32_t* lens_out;
  int len_add;
  // fraction of the split partials' lines written with an L2 evict-last policy: about 64 MB of them
  // stay resident for the merge (1 when they all fit)
  float keep_frac;
  // the SIMT partial kernel's wait bound, and a delay before its producer warp starts (0 in normal
  // use); set only through nbx_set_decode_wait_test, to make a bounded wait run out on purpose
  uint64_t wait_limit_ns;
  uint64_t producer_delay_ns;
  // fixed-shift softmax on the tensor-core kernel (null: the online max everywhere): per query vector
  // |q| [batch * rows * h_q], per (sequence, KV head) {max |k| * k_scale, max |v| * v_scale}, and
  // scale * log2(e)
  const float* fs_q_norm;
  const float* fs_kv_max;
  float fs_scale_log2;
  float k_scale_host;   // the pool's k scale (the bounds kernel reports |k| dequantised)
  // split partials as f16 acc / l (the partial normalised by its own sum) instead of fp32 acc: set
  // for fp8 pools on tensor cores, where acc / l is a convex combination of E4M3 codes (|code|
  // <= 448, the v scale is applied by the merge), so f16 neither overflows nor loses more than
  // 2^-11 relative; each (row, split) slot holds d halves in the first half of its d floats
  int part_f16;
  // split plan for a tensor-core window (0: the pages' rule, ceil(len / 256) splits of at most 64):
  // about tc_units work units in all, each of the tc_pairs (KV head, M tile) pairs of a sequence
  // taking floor(tc_units * len / (tc_pairs * sum of lens)) splits, clamped to [1, min(max_splits,
  // len / 64)]
  int tc_units;
  int tc_pairs;
};

cudaError_t bounds_dispatch(const DecodeParams& p, int q_dtype, int pool_dtype, float* q_norm, float* kv_max,
                            cudaStream_t stream);

cudaError_t decode_dispatch(const DecodeParams& p, int q_dtype, int pool_dtype, int grid_limit, cudaStream_t stream);

// The tensor-core partial kernel: used when the query vectors of one KV head fill an MMA tile
// (rows x group >= 64), q is bf16, the pools bf16 (kind::f16) or E4M3 (kind::f8f6f4 on the codes),
// d is 128 or 256 and pages hold a multiple of 64 positions.
bool mma_path_applies(const DecodeParams& p, int q_dtype, int pool_dtype);
constexpr int kMmaRowsPerTile = 128;   // query vectors of one M tile of the tensor-core kernel
cudaError_t decode_dispatch_mma(const DecodeParams& p, int pool_dtype, int grid_limit, cudaStream_t stream);

// Launch with programmatic dependent launch: the grid may start while the previous kernel in the
// stream finishes; the kernel orders itself after it with griddepcontrol.wait.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

struct MergeParams {
  const float* acc_part;
  const float* m_part;
  const float* l_part;
  float* out;
  int n_rows, splits, d;
};

cudaError_t merge_dispatch(const MergeParams& p, cudaStream_t stream);

}  // namespace nbx
