/*
 * libnbx: paged KV-cache append and split-KV ("flash-decoding") decode attention
 * for one NVIDIA GB300 GPU (sm_103a).
 *
 * C ABI. Every buffer argument is a plain pointer to memory the caller owns; the
 * library allocates and frees nothing and never synchronises the stream. Device
 * pointers are marked [device], host values are passed by value. Streams are
 * passed as `void*` holding a cudaStream_t (NULL = the legacy default stream).
 *
 * Layouts are row-major with the last dimension contiguous:
 *   pool         [num_pages, h_kv, page_tokens, d]   one pool per K and per V
 *   new_k/new_v  [n_tok, h_kv, d]
 *   slot_mapping [n_tok]            int32, slot = page * page_tokens + position in page
 *   q            [batch, rows, h_q, d]
 *   block_table  [batch, max_pages] int32 page ids, -1 past each sequence
 *   seq_lens     [batch]            int32 positions each sequence holds
 *   out          [batch, rows, h_q, d] fp32
 *
 * Sources (pages the method is described on):
 *   nbxtensor 0.0.1 wheel, nbxtensor/ops/attention_wrappers.py: paged_kv_append,
 *     paged_decode_attention, decode_reduce (the boundary and its checks);
 *   nbxtensor 0.0.1 wheel, nbxtensor/ops/paged_decode_attn.py: module docstring (pool
 *     layout, slot mapping, block table), paged_kv_append_kernel, paged_decode_splits,
 *     paged_decode_attn_split_kernel (the split partial);
 *   TensorFold PR #1219: the rows-first grid (all rows of a split share its K/V from
 *     L2), the fp8 cache, the merge's skip rule.
 *
 * Errors. Host-detectable problems return a negative nbx_status before anything is
 * launched. Problems only the device can see (a slot or a page id outside the pool,
 * a length outside its bounds, a wait that ran out of time) set bits in the optional
 * [device] int32 status word with an atomic OR and skip the offending work; kernels
 * never trap. The caller reads the word after synchronising; it is never cleared by
 * the library.
 */
#ifndef NBX_H
#define NBX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NBX_API __attribute__((visibility("default")))

typedef enum {
    NBX_F32 = 0,   /* IEEE binary32 */
    NBX_BF16 = 1,  /* bfloat16 */
    NBX_E4M3 = 2   /* OCP FP8 E4M3 (FN: no infinities, max 448), with one fp32 scale per pool */
} nbx_dtype;

typedef enum {
    NBX_OK = 0,
    NBX_ERR_NULL = -1,        /* a required pointer is NULL */
    NBX_ERR_SHAPE = -2,       /* sizes that do not fit together, or outside the supported set */
    NBX_ERR_DTYPE = -3,       /* a dtype code this call does not take */
    NBX_ERR_PAGE_ALIGN = -4,  /* page_tokens is not a multiple of NBX_TILE_POSITIONS */
    NBX_ERR_WORKSPACE = -5,   /* workspace smaller than nbx_paged_decode_workspace_bytes() */
    NBX_ERR_CUDA = -6,        /* a CUDA runtime call or launch failed */
    NBX_ERR_ALIGN = -7,       /* a buffer is not 16-byte aligned */
    NBX_ERR_VALUE = -8        /* a scalar argument is not finite or a scale is not positive */
} nbx_status;

/* Bits of the device status word. */
#define NBX_DEV_BAD_SLOT 0x1   /* an append slot outside [0, num_pages * page_tokens): token skipped */
#define NBX_DEV_BAD_PAGE 0x2   /* a block-table entry inside a sequence is -1 or >= num_pages: tile skipped */
#define NBX_DEV_BAD_LEN 0x4    /* seq_lens[b] < 0, > max_seq_len or > max_pages * page_tokens: sequence read as empty */
#define NBX_DEV_TIMEOUT 0x8    /* a bounded wait inside a kernel gave up: the output is incomplete */

/* Positions per staged tile: every page must hold a whole number of tiles, so no
 * tile straddles two pages (paged_decode_attention's "ZERO FALLBACK" check). */
#define NBX_TILE_POSITIONS 16
/* The pages' split rule (nbxtensor/ops/paged_decode_attn.py, paged_decode_splits): it bounds the
 * splits a workspace holds; the decode itself cuts splits of two of these (see nbx_paged_decode_attn). */
#define NBX_SPLIT_POSITIONS 256
#define NBX_MAX_SPLITS 64

/*
 * nbx_paged_kv_append -- write new positions into the pools through the slot mapping.
 * (nbxtensor/ops/attention_wrappers.py, paged_kv_append; nbxtensor/ops/paged_decode_attn.py,
 * paged_kv_append_kernel.)
 *
 * For token t and KV head h: page = slot_mapping[t] / page_tokens, pos = slot_mapping[t] %
 * page_tokens, k_pool[page, h, pos, :] = cast(new_k[t, h, :] * (1 / k_scale)), the same for V.
 * The reciprocal is taken once in fp32 on the host; the cast rounds to nearest even (bf16,
 * E4M3 with saturation to +-448) or copies (fp32).
 *
 *   new_k, new_v  [device] [n_tok, h_kv, d] in new_dtype (NBX_F32 or NBX_BF16)
 *   n_tok         tokens to write; 0 returns NBX_OK without a launch
 *   k_pool, v_pool [device] [num_pages, h_kv, page_tokens, d] in pool_dtype (any nbx_dtype)
 *   slot_mapping  [device] int32 [n_tok]; entries must be distinct. A slot outside
 *                 [0, num_pages*page_tokens) sets NBX_DEV_BAD_SLOT and the token is skipped.
 *   k_scale, v_scale  dequantisation scales of the pools (finite, > 0; use 1 unless E4M3)
 *   status        [device] int32 or NULL
 *   stream        cudaStream_t
 * Requirements: d a multiple of 16 and <= 1024; all buffers 16-byte aligned.
 */
NBX_API int nbx_paged_kv_append(const void* new_k, const void* new_v, int new_dtype, int n_tok, int h_kv, int d,
                                void* k_pool, void* v_pool, int pool_dtype, int num_pages, int page_tokens,
                                const int32_t* slot_mapping, float k_scale, float v_scale, int32_t* status,
                                void* stream);

/*
 * nbx_paged_decode_workspace_bytes -- bytes of workspace nbx_paged_decode_attn needs for
 * these sizes (the split plan, the work list and the fp32 split partials).
 * Returns 0 if the sizes are invalid. max_seq_len is the host-known bound on seq_lens.
 */
NBX_API size_t nbx_paged_decode_workspace_bytes(int batch, int rows, int h_q, int h_kv, int d, int max_seq_len);

/*
 * nbx_paged_decode_workspace_bytes_for -- the workspace for these sizes and formats. Every format
 * and page size needs the same today (the tensor-core kernel reads an fp8 pool's codes as they are
 * stored), so it equals nbx_paged_decode_workspace_bytes; the formats are taken so that a caller
 * sizing per call keeps working if that changes. Returns 0 if the sizes are invalid.
 */
NBX_API size_t nbx_paged_decode_workspace_bytes_for(int q_dtype, int pool_dtype, int batch, int rows, int h_q,
                                                    int h_kv, int d, int max_seq_len, int page_tokens);

/*
 * nbx_paged_decode_attn -- split-KV decode attention read through the block table.
 * (nbxtensor/ops/attention_wrappers.py, paged_decode_attention; nbxtensor/ops/paged_decode_attn.py,
 * paged_decode_splits and paged_decode_attn_split_kernel; TensorFold PR #1219, rows-first grid.)
 *
 * For sequence b, query row r and query head h: the row sits at position
 * p = seq_lens[b] - rows + r and attends keys 0..p of KV head h / (h_q / h_kv):
 *   s_j = scale * k_scale * (q . k_j),  out = v_scale * sum_j e^(s_j - max s) v_j / sum_j e^(s_j - max s).
 * A row with no visible key (p < 0, or seq_lens[b] == 0) gets 0. Each sequence is cut into
 * min(ceil(len/512), 64) splits of whole pages, two of the pages' 256-position splits each (a window
 * on tensor cores, see nbx_paged_decode_partial_kernel: about one work unit per SM in all, splits in
 * proportion to the lengths, at most min(ceil(max_seq_len/256), 64)); each split's unnormalised
 * partial (m, l, acc) is computed with an fp32 online softmax and the partials are merged in
 * ascending split order (a split with m = -inf is skipped, so NaN inputs reach the output). The
 * result does not depend on the physical page ids or on the order the work runs in.
 *
 *   q            [device] [batch, rows, h_q, d], q_dtype NBX_F32 or NBX_BF16
 *   k_pool, v_pool [device] [num_pages, h_kv, page_tokens, d] in pool_dtype
 *   block_table  [device] int32 [batch, max_pages]
 *   seq_lens     [device] int32 [batch]
 *   max_seq_len  host bound on seq_lens (sizes the splits and the workspace);
 *                must be <= max_pages * page_tokens
 *   scale        softmax scale (finite); k_scale, v_scale: pool scales (finite, > 0)
 *   out          [device] fp32 [batch, rows, h_q, d]
 *   workspace    [device] at least nbx_paged_decode_workspace_bytes(...) bytes, 256-byte aligned;
 *                its contents need no initialisation and are overwritten
 *   status       [device] int32 or NULL
 *   stream       cudaStream_t
 * Requirements: h_q % h_kv == 0; d in {64, 128, 256}; page_tokens a multiple of
 * NBX_TILE_POSITIONS; q, pools and out 16-byte aligned. batch == 0 returns NBX_OK without a launch.
 * Calls on one workspace must not overlap on the GPU.
 */
NBX_API int nbx_paged_decode_attn(const void* q, int q_dtype, int batch, int rows, int h_q, int d,
                                  const void* k_pool, const void* v_pool, int pool_dtype, int num_pages, int h_kv,
                                  int page_tokens, const int32_t* block_table, int max_pages,
                                  const int32_t* seq_lens, int max_seq_len, float scale, float k_scale,
                                  float v_scale, float* out, void* workspace, size_t workspace_bytes,
                                  int32_t* status, void* stream);

/*
 * nbx_paged_decode_step -- one decode step with no host-side positions: append, then attend.
 * (nbxtensor/ops/paged_decode_attn.py, paged_kv_append_step_kernel and paged_lens_advance_kernel:
 * the step writes at the layer's device length and the length then advances, so a recorded launch
 * replays unchanged; nbxtensor/ops/attention_wrappers.py, paged_decode_attention for the decode.)
 *
 * For each sequence b, with n = lens[b] on entry: the step's new keys and values are written at
 * positions n .. n + rows - 1 (page block_table[b, pos / page_tokens], slot pos % page_tokens,
 * cast on store exactly as nbx_paged_kv_append does), then the rows attend exactly as
 * nbx_paged_decode_attn with seq_lens[b] = n + rows, and lens[b] becomes n + rows. Everything
 * happens on the stream in that order; the call's arguments are the same at every step, so it
 * can be captured once in a CUDA graph and replayed.
 *
 *   new_k, new_v [device] [batch, rows, h_kv, d] in new_dtype (NBX_F32 or NBX_BF16): row r of
 *                sequence b is the key/value of query row r (position n + r)
 *   lens         [device] int32 [batch], read and then advanced by rows (in stream order)
 *   max_seq_len  host bound on every lens[b] + rows (sizes the splits and the workspace)
 *   every other argument as for nbx_paged_decode_attn; the workspace is sized by
 *   nbx_paged_decode_workspace_bytes(_for) with the same sizes.
 * Device-detected problems set status bits: a position at or past max_seq_len (NBX_DEV_BAD_LEN,
 * not written), a page id outside the pool (NBX_DEV_BAD_PAGE, not written). The host checks are
 * those of nbx_paged_decode_attn plus new_dtype; on any failure nothing is launched.
 * This library addition fuses what the pages run as separate launches.
 */
NBX_API int nbx_paged_decode_step(const void* q, int q_dtype, int batch, int rows, int h_q, int d, const void* new_k,
                                  const void* new_v, int new_dtype, void* k_pool, void* v_pool, int pool_dtype,
                                  int num_pages, int h_kv, int page_tokens, const int32_t* block_table, int max_pages,
                                  int32_t* lens, int max_seq_len, float scale, float k_scale, float v_scale,
                                  float* out, void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/*
 * nbx_decode_attn_contiguous -- split-KV decode over a contiguous (non-paged) cache.
 * (nbxtensor/ops/attention_wrappers.py, _decode_attn_vec: the same split read and fixed-order
 * merge without a page table.)
 *
 * The caches k_cache, v_cache [device] [batch, h_kv, capacity, d] in cache_dtype hold sequence b's
 * positions 0 .. capacity - 1. That is the pool layout with one page of capacity positions per
 * sequence, so the call is nbx_paged_decode_attn with num_pages = batch, page_tokens = capacity,
 * max_pages = 1 and the identity block table (page b for sequence b), which the library writes
 * into the workspace itself. Same results, rules and errors as nbx_paged_decode_attn;
 * capacity must be a multiple of NBX_TILE_POSITIONS and >= max_seq_len; the workspace is sized by
 * nbx_paged_decode_workspace_bytes_for(..., page_tokens = capacity).
 */
NBX_API int nbx_decode_attn_contiguous(const void* q, int q_dtype, int batch, int rows, int h_q, int d,
                                       const void* k_cache, const void* v_cache, int cache_dtype, int h_kv,
                                       int capacity, const int32_t* seq_lens, int max_seq_len, float scale,
                                       float k_scale, float v_scale, float* out, void* workspace,
                                       size_t workspace_bytes, int32_t* status, void* stream);

/*
 * nbx_paged_decode_merge -- the fixed-order merge of split partials on its own.
 * (nbxtensor/ops/attention_wrappers.py, decode_reduce; TensorFold PR #1219, the merge's skip rule.)
 *
 * For each row i: M = max_s m[i,s], L = sum_s l[i,s] e^(m[i,s]-M),
 * out[i,:] = sum_s acc[i,s,:] e^(m[i,s]-M) / L, s ascending, skipping splits with m = -inf.
 * A row with no live split gets 0. m is in natural-log units (the running max of the scores).
 *
 *   acc_part [device] fp32 [n_rows, splits, d];  m_part, l_part [device] fp32 [n_rows, splits]
 *   out      [device] fp32 [n_rows, d]
 * Requirements: 1 <= splits <= 4096, 1 <= d <= 1024. n_rows == 0 returns NBX_OK without a launch.
 */
NBX_API int nbx_paged_decode_merge(const float* acc_part, const float* m_part, const float* l_part, int n_rows,
                                   int splits, int d, float* out, void* stream);

/*
 * nbx_paged_decode_bounds -- the score bounds the fixed-shift softmax gates on.
 * (maxdiffusion PR #477, "fixed-m": the per-head metadata computed before the kernel, here per query
 * vector and per (sequence, KV head).)
 *
 * q_norm [device] fp32 [batch, rows, h_q]: |q| of every query vector.
 * kv_max [device] fp32 [batch, h_kv, 2]: {max_j |k_j| * k_scale, max_{j,d} |v_jd| * v_scale} over the
 * positions 0 .. seq_lens[b] - 1 of the sequence, read through the block table. A NaN input gives a
 * NaN bound (which no gate passes). One pass over the sequences' K and V. Other arguments, rules and
 * status bits as for nbx_paged_decode_attn (no workspace).
 */
NBX_API int nbx_paged_decode_bounds(const void* q, int q_dtype, int batch, int rows, int h_q, int d, const void* k_pool,
                                    const void* v_pool, int pool_dtype, int num_pages, int h_kv, int page_tokens,
                                    const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                                    int max_seq_len, float k_scale, float v_scale, float* q_norm, float* kv_max,
                                    int32_t* status, void* stream);

/*
 * nbx_paged_decode_attn_fixed_shift -- nbx_paged_decode_attn with the fixed-shift softmax of
 * maxdiffusion PR #477 ("fixed-m") on the tensor-core kernel, as an ablation of the online max.
 *
 * For a query row of a split of n keys, U = |q| * max|k| * scale * log2(e) bounds every score in
 * log2 units (Cauchy-Schwarz). With C(n) = 127 - ceil(log2 n) - ceil(log2 256) and the gate
 * floor((C(n) + 125) / 2): a row with U <= gate and max |v| <= 256 takes its weights as 2^(z - m),
 * m = ceil(U) - C(n), fixed before the split is read (no running max, no rescale; no weight above 2^C
 * or below 2^-125). A row that fails the gate, and every row of a window whose P enters the product
 * as E4M3 terms (an fp8 pool on tensor cores: E4M3 cannot hold 2^C), keeps the online max. Calls that
 * run the SIMT kernel are the same as nbx_paged_decode_attn. Results are within the decode's tolerance
 * of nbx_paged_decode_attn's.
 *
 *   q_norm, kv_max  [device] the bounds, as nbx_paged_decode_bounds writes them
 *   every other argument as for nbx_paged_decode_attn.
 */
NBX_API int nbx_paged_decode_attn_fixed_shift(const void* q, int q_dtype, int batch, int rows, int h_q, int d,
                                              const void* k_pool, const void* v_pool, int pool_dtype, int num_pages,
                                              int h_kv, int page_tokens, const int32_t* block_table, int max_pages,
                                              const int32_t* seq_lens, int max_seq_len, float scale, float k_scale,
                                              float v_scale, float* out, void* workspace, size_t workspace_bytes,
                                              const float* q_norm, const float* kv_max, int32_t* status,
                                              void* stream);

/*
 * nbx_decode_fixed_shift_gate -- the fixed-shift constants for n_keys keys and a value bound
 * (maxdiffusion PR #477, get_fixed_m_constants): C = 127 - ceil(log2 n_keys) - ceil(log2 v_max_bound)
 * and gate = floor((C + 125) / 2). Host-only. NBX_ERR_VALUE for n_keys < 1 or v_max_bound < 1.
 */
NBX_API int nbx_decode_fixed_shift_gate(int n_keys, double v_max_bound, int* c_out, int* gate_out);

/* Bytes of device scratch that libnbx keeps for nbx_paged_decode_attn_noalloc (32 MiB). */
#define NBX_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * nbx_paged_decode_attn_noalloc -- nbx_paged_decode_attn without a caller workspace.
 * The pages have no counterpart of this call: it exists for callers that cannot allocate device
 * memory (code running where cudaMalloc is not allowed, such as an allocator's own callbacks, a
 * process whose memory budget is fixed before the library loads, or a plug-in without access to
 * the host application's allocator).
 *
 * Same arguments, layouts and results as nbx_paged_decode_attn, minus workspace and
 * workspace_bytes. The scratch is a fixed array of NBX_NOALLOC_SCRATCH_BYTES in the library's
 * own device memory, held by every GPU that loads the library until the process exits. Sizes
 * whose workspace (nbx_paged_decode_workspace_bytes) exceeds it return NBX_ERR_WORKSPACE without
 * a launch. Nothing is allocated or freed.
 * The first call on a device looks up the array's device address with that device current; make
 * that first call before any stream capture. All calls share the one array and it keeps the last
 * call's contents (every call rewrites what it reads), so calls that overlap on the GPU race.
 */
NBX_API int nbx_paged_decode_attn_noalloc(const void* q, int q_dtype, int batch, int rows, int h_q, int d,
                                          const void* k_pool, const void* v_pool, int pool_dtype, int num_pages,
                                          int h_kv, int page_tokens, const int32_t* block_table, int max_pages,
                                          const int32_t* seq_lens, int max_seq_len, float scale, float k_scale,
                                          float v_scale, float* out, int32_t* status, void* stream);

/* The split-partial kernel a decode call runs (see nbx_paged_decode_partial_kernel). */
typedef enum {
    NBX_PARTIAL_SIMT = 0,            /* CUDA cores: work units of 4 query vectors, any supported shape */
    NBX_PARTIAL_TCGEN05 = 1,         /* tensor cores (tcgen05.mma): work units of 128 query vectors */
    NBX_PARTIAL_TCGEN05_FP8 = 2      /* fp8 (E4M3) pool: the tensor-core kernel on the codes as stored
                                        (tcgen05.mma kind::f8f6f4), Q and P as two E4M3 terms each */
} nbx_partial_kernel;

/*
 * nbx_paged_decode_partial_kernel -- which split-partial kernel nbx_paged_decode_attn (and
 * nbx_paged_decode_attn_noalloc) runs for these sizes and formats. Host-only; launches nothing.
 * (TensorFold PR #1219: the rows of one KV head read each K/V tile once; when rows x group
 * reaches a dense tile the QK^T and PV products become matrix products.)
 *
 * Returns NBX_PARTIAL_TCGEN05 when rows * (h_q / h_kv) >= 64, h_q / h_kv <= 128, q_dtype and
 * pool_dtype are both NBX_BF16, d is 128 or 256, page_tokens is a multiple of 64 and the pool has
 * fewer than 2^31 - 64 rows of d elements per K or V (the call itself also needs scale > 0; a
 * decode with scale <= 0 runs the SIMT kernel); NBX_PARTIAL_TCGEN05_FP8 under the same conditions
 * with an NBX_E4M3 pool; NBX_PARTIAL_SIMT for every other supported case; a negative nbx_status for
 * arguments nbx_paged_decode_attn rejects (shape, page alignment, dtype). The kernels compute the
 * same partials to within the decode's tolerance; none depends on page ids or on the grid size.
 */
NBX_API int nbx_paged_decode_partial_kernel(int q_dtype, int pool_dtype, int rows, int h_q, int h_kv, int d,
                                            int num_pages, int page_tokens);

/*
 * nbx_set_decode_grid_limit -- cap the number of CTAs nbx_paged_decode_attn launches for its split
 * partial (0 = each kernel's default: two or three CTAs per SM for the SIMT kernel, one per SM for
 * the tensor-core kernel). Process-wide; the output is bit-identical for every value.
 */
NBX_API void nbx_set_decode_grid_limit(int max_ctas);

/*
 * nbx_set_decode_wait_test -- for tests of the timeout path only; the pages have no counterpart.
 * Every wait inside the split-partial kernels is bounded (2 s by default): a wait that runs out
 * sets NBX_DEV_TIMEOUT, the kernel lets its copies in flight land (and, on tensor cores, its MMAs
 * complete and its TMEM go back) and returns, and the output of the call is incomplete. This sets
 * that bound (wait_limit_ns; 0 restores 2 s) and holds each CTA's producer warps back for
 * producer_delay_ns before they start (0 = no delay; capped at 50 ms), so a test can make the other
 * warps' waits run out without any invalid input. Process-wide; applies to calls launched after it.
 */
NBX_API void nbx_set_decode_wait_test(unsigned long long wait_limit_ns, unsigned long long producer_delay_ns);

/* A static, human-readable name for an nbx_status value. */
NBX_API const char* nbx_status_string(int status);

/* ABI version of this header (major * 100 + minor). */
NBX_API int nbx_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* NBX_H */
