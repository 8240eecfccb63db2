// The split plan kernel, the standalone merge kernel, the workspace layout and the
// decode launch sequence (plan, then the persistent partial kernel).
#include <cuda_fp16.h>

#include "decode_kernels.cuh"

namespace nbx {

constexpr int kPlanThreads = 256;
constexpr int kSortMax = 2048;   // batches up to this size are planned in shared memory, longest split first

// Dynamic shared memory of the plan kernel: five int arrays of the batch (4 (5B + 1) bytes), none
// above kSortMax. Sized to the batch, so that the CTA leaves room on its SM for a CTA of the
// partial kernel that follows it (launched while the plan runs): a fixed 40 KB took that room from
// one tensor-core CTA, whose late start lengthened a one-wave grid by the plan's own time.
inline size_t plan_smem_bytes(int batch) {
  return batch <= kSortMax ? static_cast<size_t>(5 * batch + 1) * sizeof(int) : 0;
}

// Positions per split of the SIMT partial kernel: two of the pages' splits (NBX_SPLIT_POSITIONS).
// Each work unit of the persistent kernel pays about 2.4 us at its boundaries (the cross-warp merge
// and the partial's stores, the next unit's query staging and first stage); at 512 positions a unit
// single_row's decode call took 109.4 against 115.5 us at 256 (ragged 754.1 against 755.9 us).
constexpr int kSimtSplitPositions = 2 * NBX_SPLIT_POSITIONS;

int splits_for(int length) {
  const int l = length < 1 ? 1 : length;
  int s = (l + NBX_SPLIT_POSITIONS - 1) / NBX_SPLIT_POSITIONS;
  return s < 1 ? 1 : (s > NBX_MAX_SPLITS ? NBX_MAX_SPLITS : s);
}

bool workspace_layout(int batch, int rows, int h_q, int h_kv, int d, int max_seq_len, WorkspaceLayout* w) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t S = static_cast<size_t>(splits_for(max_seq_len));
  const size_t rb = (static_cast<size_t>(rows) * (h_q / h_kv) + kQB - 1) / kQB;
  const size_t prow = static_cast<size_t>(batch) * rows * h_q * S;   // partial rows
  if (prow > (static_cast<size_t>(1) << 40) / static_cast<size_t>(d)) return false;
  size_t off = 0;
  w->header = off;
  off += up(64 * 4);
  w->ident_bt = off;
  off += up(static_cast<size_t>(batch) * 4);
  w->plan = off;
  off += up(static_cast<size_t>(batch) * sizeof(SeqPlan));
  w->entries = off;
  off += up(static_cast<size_t>(batch) * S * sizeof(Entry));
  w->m_part = off;
  off += up(prow * 4);
  w->l_part = off;
  off += up(prow * 4);
  w->acc_part = off;
  off += up(prow * static_cast<size_t>(d) * 4);
  w->total = off;
  w->max_splits = static_cast<int>(S);
  w->row_blocks = static_cast<int>(rb);
  return true;
}

// The plan kernel may run while the kernel before it (a decode step's append, which reads the
// lengths) still runs: it waits for that grid before the step's length advance, and before it
// completes, so the kernels after it see the append's positions.
__device__ __forceinline__ void plan_finish(const DecodeParams& p) {
  pdl_wait();
  if (p.lens_out)   // the step's length advance; nothing later reads seq_lens
    for (int b = threadIdx.x; b < p.batch; b += blockDim.x) p.lens_out[b] = p.seq_lens[b] + p.len_add;
}

// Reads the device lengths, writes every sequence's plan (len, positions per split, non-empty
// splits), zeroes the work counter, writes 0 to the output rows of empty sequences, and writes
// the work list of (sequence, split) entries: every sequence's last split first, then the other
// splits, sequences with the longest splits first (stable), splits ascending. Batches above kSortMax
// keep their own order and take a slower serial path.
// TC: a tensor-core window, whose splits are sized by the call's total work (DecodeParams::tc_units);
// otherwise splits of kSimtSplitPositions. Two instantiations keep each rule's code free of the other.
template <bool TC>
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(DecodeParams p) {
  extern __shared__ int plan_sm[];   // plan_smem_bytes(batch)
  int* const s_len = plan_sm;
  int* const s_seg = s_len + p.batch;
  int* const s_n = s_seg + p.batch;
  int* const s_order = s_n + p.batch;
  int* const s_base = s_order + p.batch;   // [batch + 1]
  __shared__ int s_warp[kPlanThreads / 32];
  __shared__ int s_empty;
  __shared__ int s_nb;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int B = p.batch;
  const int64_t cap = static_cast<int64_t>(p.max_pages) * p.page_tokens;
  const bool small = B <= kSortMax;
  pdl_launch_dependents();   // the partial kernel may start its prologue now; it waits for this grid
  __shared__ long long s_total;
  if (tid == 0) {
    s_empty = 0;
    s_nb = 0;
    if constexpr (TC) s_total = 0;
    p.header[1] = 0;
  }
  __syncthreads();
  // a tensor-core window sizes its splits by the whole call's work: the sum of the lengths
  long long len_sum = 0;
  if constexpr (TC) {
    long long part = 0;
    for (int b = tid; b < B; b += kPlanThreads) {
      const int L = p.seq_lens[b] + p.len_add;
      if (L > 0 && L <= p.max_seq_len && static_cast<int64_t>(L) <= cap) part += L;
    }
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0 && part) atomicAdd(reinterpret_cast<unsigned long long*>(&s_total), static_cast<unsigned long long>(part));
    __syncthreads();
    len_sum = s_total;
  }
  for (int b = tid; b < B; b += kPlanThreads) {
    int L = p.seq_lens[b] + p.len_add;   // a decode step attends to its own new positions
    if (p.ident_bt) p.ident_bt[b] = b;
    if (L < 0 || L > p.max_seq_len || static_cast<int64_t>(L) > cap) {
      raise_status(p.status, NBX_DEV_BAD_LEN);
      L = 0;
    }
    int S;
    if (TC && len_sum > 0) {
      // about tc_units units in all, shared in proportion to the lengths (the grid's one wave); a
      // split keeps at least 64 positions (the tensor-core tile), and a sequence has at most the
      // workspace's partial slots (max_splits, the pages' rule at the longest length)
      const long long want = static_cast<long long>(p.tc_units) * L / (static_cast<long long>(p.tc_pairs) * len_sum);
      const int cap_s = min(p.max_splits, max(1, L / 64));
      S = static_cast<int>(want < 1 ? 1 : (want > cap_s ? cap_s : want));
    } else {
      // two of the pages' 256-position splits a split: half the unit boundaries, at most 64 splits
      S = (max(L, 1) + kSimtSplitPositions - 1) / kSimtSplitPositions;
      S = S > NBX_MAX_SPLITS ? NBX_MAX_SPLITS : S;
    }
    int seg = (L + S - 1) / S;
    // splits start on whole pages, or on 256-position boundaries when a page is longer (a
    // contiguous cache read as one page per sequence): tile starts either way
    const int align = p.page_tokens <= NBX_SPLIT_POSITIONS ? p.page_tokens : NBX_SPLIT_POSITIONS;
    seg = ((seg + align - 1) / align) * align;
    const int n = L > 0 ? (L + seg - 1) / seg : 0;
    // kept in L2 for the merge, which reads the split counts after the K/V stream
    st_global_hint(reinterpret_cast<int4*>(p.plan + b), make_int4(L, seg, n, 0), l2_evict_last_policy());
    if (n == 0) s_empty = 1;
    else if (small) atomicAdd(&s_nb, 1);
    if (small) {
      s_len[b] = L;
      s_seg[b] = seg;
      s_n[b] = n;
    }
  }
  __syncthreads();
  // a sequence with no position to read gets no work unit: its rows are written here (0)
  if (s_empty) {
    const int64_t row_vec4 = static_cast<int64_t>(p.rows) * p.h_q * p.d / 4;
    for (int b = 0; b < B; ++b) {
      if ((small ? s_n[b] : p.plan[b].n_splits) != 0) continue;
      float4* o = reinterpret_cast<float4*>(p.out) + b * row_vec4;
      for (int64_t x = tid; x < row_vec4; x += kPlanThreads) o[x] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  if (!small) {
    // large batch: batch order, one thread writes the whole list
    if (tid == 0) {
      int base = 0;
      for (int b = 0; b < B; ++b) {
        const SeqPlan sp = p.plan[b];
        for (int s = 0; s < sp.n_splits; ++s) {
          Entry e;
          e.b = b;
          e.s = s;
          e.start = s * sp.seg;
          e.end = min((s + 1) * sp.seg, sp.len);
          e.len = sp.len;
          e.n_splits = sp.n_splits;
          e.pad0 = e.pad1 = 0;
          p.entries[base + s] = e;
        }
        base += sp.n_splits;
      }
      p.header[0] = base;
    }
    plan_finish(p);
    return;
  }
  // stable rank by split length, longest first (empty sequences last). The list then holds every
  // sequence's last split first (in that order), then the other splits: the last splits are of
  // uneven length, so the persistent grid's first wave of units ends at scattered times instead of
  // every CTA reaching a unit boundary at once; the rest follow longest first.
  for (int b = tid; b < B; b += kPlanThreads) {
    const int k = s_n[b] > 0 ? s_seg[b] : -1;
    int rank = 0;
    for (int c = 0; c < B; ++c) {
      const int kc = s_n[c] > 0 ? s_seg[c] : -1;
      rank += (kc > k) || (kc == k && c < b);
    }
    s_order[rank] = b;
  }
  __syncthreads();
  // exclusive scan of the split counts in list order (a contiguous run per thread, then a block scan)
  const int per = (B + kPlanThreads - 1) / kPlanThreads;
  const int lo = min(B, tid * per), hi = min(B, lo + per);
  int run = 0;
  for (int i = lo; i < hi; ++i) run += max(s_n[s_order[i]] - 1, 0);
  int x = run;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kPlanThreads / 32 ? s_warp[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kPlanThreads / 32) s_warp[lane] = w;
  }
  __syncthreads();
  int base = x - run + (warp > 0 ? s_warp[warp - 1] : 0);
  for (int i = lo; i < hi; ++i) {
    s_base[i] = base;
    base += max(s_n[s_order[i]] - 1, 0);
  }
  if (tid == kPlanThreads - 1) s_base[B] = x + (warp > 0 ? s_warp[warp - 1] : 0);
  __syncthreads();
  // the entries, in parallel: entry e belongs to the list position i with s_base[i] <= e < s_base[i+1]
  const int nb = s_nb;
  const int total = s_base[B] + nb;
  for (int e = tid; e < total; e += kPlanThreads) {
    int b, s;
    if (e < nb) {
      b = s_order[e];
      s = s_n[b] - 1;
    } else {
      const int e2 = e - nb;
      int l = 0, r = B - 1;
      while (l < r) {
        const int m = (l + r + 1) >> 1;
        if (s_base[m] <= e2) l = m; else r = m - 1;
      }
      b = s_order[l];
      s = e2 - s_base[l];
    }
    Entry en;
    en.b = b;
    en.s = s;
    en.start = s * s_seg[b];
    en.end = min((s + 1) * s_seg[b], s_len[b]);
    en.len = s_len[b];
    en.n_splits = s_n[b];
    en.pad0 = en.pad1 = 0;
    p.entries[e] = en;
  }
  if (tid == 0) p.header[0] = total;
  plan_finish(p);
}

// ------------------------------------------------------------------------------------ standalone merge
constexpr int kMergeThreads = 128;

// One CTA per row: M = max_s m_s, weights e^(m_s - M) (splits with m = -inf are skipped),
// L = sum_s l_s w_s, out = sum_s w_s acc_s / L, s ascending.
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(MergeParams p) {
  extern __shared__ float msm[];
  float* w = msm;
  int* live = reinterpret_cast<int*>(msm + p.splits);
  __shared__ float s_inv;
  __shared__ int s_dead;
  const int64_t row = blockIdx.x;
  const float* m = p.m_part + row * p.splits;
  const float* l = p.l_part + row * p.splits;
  if (threadIdx.x == 0) {
    float M = -INFINITY;
    for (int s = 0; s < p.splits; ++s) M = max_nan(M, m[s]);
    float L = 0.f;
    for (int s = 0; s < p.splits; ++s) {
      const float ms = m[s];
      const int lv = ms != -INFINITY;
      const float ws = lv ? fast_exp2((ms - M) * kLog2e) : 0.f;
      if (lv) L += ws * l[s];
      w[s] = ws;
      live[s] = lv;
    }
    s_dead = (M == -INFINITY);
    s_inv = 1.f / L;
  }
  __syncthreads();
  for (int d = threadIdx.x; d < p.d; d += kMergeThreads) {
    float A = 0.f;
    for (int s = 0; s < p.splits; ++s)
      if (live[s]) A += w[s] * p.acc_part[(row * p.splits + s) * p.d + d];
    p.out[row * p.d + d] = s_dead ? 0.f : A * s_inv;
  }
}

cudaError_t merge_dispatch(const MergeParams& p, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(p.splits) * 8;
  merge_kernel<<<static_cast<unsigned>(p.n_rows), kMergeThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------ decode merge
constexpr int kDecodeMergeThreads = 32;   // one warp per CTA

// Merges the split partials of every query vector of a (sequence, KV head) with more than one
// split: M = max_s m_s, w_s = 2^(m_s - M) (m in log2 units; splits with m = -inf skipped),
// out = v_scale * sum_s w_s acc_s / sum_s w_s l_s, s ascending. One-split sequences were written
// by the partial kernel.
// One warp per query vector and 128 output columns, each its own CTA so the work spreads evenly
// over the SMs: lane k holds m and l of splits k and k + 32 (max and sums are butterfly
// reductions, a fixed order), the weights reach every lane by shuffles, and each lane owns one
// float4 of the output, with every split's accumulator load in flight and the sum in ascending
// split order.
// F16: the partials are f16 acc / l (DecodeParams::part_f16); a split then weighs 2^(m - M) * l.
template <bool F16>
__global__ void __launch_bounds__(kDecodeMergeThreads) decode_merge_kernel(DecodeParams p) {
  const int lane = threadIdx.x;
  const int RG = p.rows * p.group;
  const int per_seq = p.h_kv * p.row_blocks;
  const int d4 = p.d / 4;
  const int n_col = (d4 + 31) / 32;   // 128-column pieces of a vector
  const int64_t n_items = static_cast<int64_t>(p.batch) * per_seq * kQB * n_col;
  // The plan kernel had completed before any CTA of the partial kernel passed its own wait, and this
  // grid is launched only after they did, so the first item's split count can be read (from L2)
  // before this grid waits for the partials.
  int s_first = 0;
  if (blockIdx.x < n_items)
    s_first = __ldcg(&p.plan[blockIdx.x / (static_cast<int64_t>(per_seq) * kQB * n_col)].n_splits);
  pdl_wait();   // every partial of the decode is written and visible from here on
  for (int64_t it = blockIdx.x; it < n_items; it += gridDim.x) {
    const int64_t vi = it / n_col;
    const int j = static_cast<int>(it - vi * n_col) * 32 + lane;   // this lane's float4 column
    const int64_t gi = vi / kQB;
    const int i = static_cast<int>(vi - gi * kQB);
    const int b = static_cast<int>(gi / per_seq);
    const int rem = static_cast<int>(gi - static_cast<int64_t>(b) * per_seq);
    const int h = rem / p.row_blocks;
    const int rb = rem - h * p.row_blocks;
    const int qi = rb * kQB + i;
    if (qi >= RG) continue;
    const int S = it == blockIdx.x ? s_first : p.plan[b].n_splits;
    if (S <= 1) continue;
    const int r = qi / p.group;
    const int g = qi - r * p.group;
    const int64_t orow = (static_cast<int64_t>(b) * p.rows + r) * p.h_q + static_cast<int64_t>(h) * p.group + g;
    const float* m = p.m_part + orow * p.max_splits;
    const float* l = p.l_part + orow * p.max_splits;
    const float4* acc = reinterpret_cast<const float4*>(p.acc_part + orow * p.max_splits * p.d);
    // f16 partials: the d halves at the start of each split's d-float slot, 4 per lane (8 bytes)
    const uint2* acc_h = reinterpret_cast<const uint2*>(p.acc_part + orow * p.max_splits * p.d);
    auto load_batch = [&](int j, int s0, float4 (&a)[32]) {
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const bool in = j < d4 && s0 + k < S;
        if constexpr (F16) {
          const uint2 hv = in ? acc_h[static_cast<int64_t>(s0 + k) * (2 * d4) + j] : make_uint2(0u, 0u);
          const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&hv.x));
          const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&hv.y));
          a[k] = make_float4(lo.x, lo.y, hi.x, hi.y);
        } else {
          a[k] = in ? acc[static_cast<int64_t>(s0 + k) * d4 + j] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    };
    float4 a[32];
    load_batch(j, 0, a);   // in flight together with the m / l loads
    float mv[2], lv[2];
    bool live[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int sp = lane + 32 * k;
      mv[k] = sp < S ? m[sp] : -INFINITY;
      lv[k] = sp < S ? l[sp] : 0.f;
      live[k] = mv[k] != -INFINITY;
    }
    float M = max_nan(mv[0], mv[1]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = max_nan(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    float wv[2];   // weight of split lane + 32k, -1 for a split with no visible key
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float w = live[k] ? fast_exp2(mv[k] - M) : 0.f;
      if (live[k]) L += w * lv[k];
      // an f16 partial is acc / l: its weight carries l
      wv[k] = live[k] ? (F16 ? w * lv[k] : w) : -1.f;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    const bool dead = M == -INFINITY;
    const float sc = p.v_scale / L;
    // every lane runs every step (the shuffles need the whole warp); lanes past the row store nothing
    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < S; s0 += 32) {
      if (s0 > 0) load_batch(j, s0, a);
      const float wsrc = s0 == 0 ? wv[0] : wv[1];
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        if (s0 + k >= S) break;
        const float w = __shfl_sync(0xffffffffu, wsrc, k);
        if (w != -1.f) {
          A.x += w * a[k].x;
          A.y += w * a[k].y;
          A.z += w * a[k].z;
          A.w += w * a[k].w;
        }
      }
    }
    if (j < d4)
      reinterpret_cast<float4*>(p.out + orow * p.d)[j] =
          dead ? make_float4(0.f, 0.f, 0.f, 0.f) : make_float4(A.x * sc, A.y * sc, A.z * sc, A.w * sc);
  }
}

// ------------------------------------------------------------------------------------ score bounds
constexpr int kBoundsThreads = 256;
constexpr int kBoundsChunk = 512;   // positions per CTA

// Score bounds for the fixed-shift softmax (maxdiffusion PR #477: the metadata computed before the
// kernel, here per query vector and per (sequence, KV head)): |q| of every query vector, and
// max_j |k_j| * k_scale and max_{j,d} |v_jd| * v_scale over the positions a sequence holds, read
// through the block table. A NaN input gives a NaN bound, which no gate passes; a length out of
// bounds is read as empty (NBX_DEV_BAD_LEN) and a page id outside the pool is skipped
// (NBX_DEV_BAD_PAGE). One CTA per (sequence, KV head, chunk of 512 positions), a warp per position;
// the chunks combine with an atomic max on the bit patterns (the bounds are >= 0, and a NaN's bits
// order above every finite value's), so kv_max must hold zeros first. The chunk-0 CTAs of KV head 0
// write the sequence's query norms.
template <class PT, class QT>
__global__ void __launch_bounds__(kBoundsThreads) bounds_kernel(DecodeParams p, float* q_norm, float* kv_max,
                                                                 int n_chunks) {
  __shared__ float s_k[kBoundsThreads / 32], s_v[kBoundsThreads / 32];
  const int chunk = static_cast<int>(blockIdx.x % static_cast<unsigned>(n_chunks));
  const int bh = static_cast<int>(blockIdx.x / static_cast<unsigned>(n_chunks));   // b * h_kv + h
  const int b = bh / p.h_kv;
  const int h = bh - b * p.h_kv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kWarps = kBoundsThreads / 32;
  int L = p.seq_lens[b];
  if (L < 0 || L > p.max_seq_len || static_cast<int64_t>(L) > static_cast<int64_t>(p.max_pages) * p.page_tokens) {
    if (h == 0 && chunk == 0 && threadIdx.x == 0) raise_status(p.status, NBX_DEV_BAD_LEN);
    L = 0;
  }
  const int j0 = chunk * kBoundsChunk, j1 = min(L, j0 + kBoundsChunk);
  float k2 = 0.f, va = 0.f;   // max |k|^2 and max |v| (pool units) over this warp's positions
  for (int j = j0 + warp; j < j1; j += kWarps) {
    const int page = p.block_table[static_cast<int64_t>(b) * p.max_pages + j / p.page_tokens];
    if (page < 0 || page >= p.num_pages) {
      if (lane == 0) raise_status(p.status, NBX_DEV_BAD_PAGE);
      continue;
    }
    const int64_t row = ((static_cast<int64_t>(page) * p.h_kv + h) * p.page_tokens + j % p.page_tokens) * p.d;
    const char* kr = static_cast<const char*>(p.k_pool) + row * PT::kBytes;
    const char* vr = static_cast<const char*>(p.v_pool) + row * PT::kBytes;
    float ks = 0.f, vm = 0.f;
    for (int e = 2 * lane; e < p.d; e += 64) {
      const float2 kk = load_pair<PT>(kr + e * PT::kBytes);
      const float2 vv = load_pair<PT>(vr + e * PT::kBytes);
      ks = fmaf(kk.x, kk.x, fmaf(kk.y, kk.y, ks));
      vm = max_nan(vm, max_nan(fabsf(vv.x), fabsf(vv.y)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ks += __shfl_xor_sync(0xffffffffu, ks, o);
      vm = max_nan(vm, __shfl_xor_sync(0xffffffffu, vm, o));
    }
    k2 = max_nan(k2, ks);
    va = max_nan(va, vm);
  }
  if (lane == 0) {
    s_k[warp] = k2;
    s_v[warp] = va;
  }
  __syncthreads();
  if (threadIdx.x == 0 && j0 < L) {
    float kt = 0.f, vt = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      kt = max_nan(kt, s_k[w]);
      vt = max_nan(vt, s_v[w]);
    }
    atomicMax(reinterpret_cast<int*>(kv_max) + 2 * bh, __float_as_int(sqrtf(kt) * p.k_scale_host));
    atomicMax(reinterpret_cast<int*>(kv_max) + 2 * bh + 1, __float_as_int(vt * p.v_scale));
  }
  if (h != 0 || chunk != 0) return;
  const int nq = p.rows * p.h_q;   // this sequence's query vectors
  for (int v = warp; v < nq; v += kWarps) {
    const char* qr = static_cast<const char*>(p.q) + (static_cast<int64_t>(b) * nq + v) * p.d * QT::kBytes;
    float qs = 0.f;
    for (int e = 2 * lane; e < p.d; e += 64) {
      const float2 qq = load_pair<QT>(qr + e * QT::kBytes);
      qs = fmaf(qq.x, qq.x, fmaf(qq.y, qq.y, qs));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) qs += __shfl_xor_sync(0xffffffffu, qs, o);
    if (lane == 0) q_norm[static_cast<int64_t>(b) * nq + v] = sqrtf(qs);
  }
}

cudaError_t bounds_dispatch(const DecodeParams& p, int q_dtype, int pool_dtype, float* q_norm, float* kv_max,
                            cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(kv_max, 0, static_cast<size_t>(p.batch) * p.h_kv * 2 * sizeof(float), stream);
  if (e != cudaSuccess) return e;
  const int n_chunks = p.max_seq_len > 0 ? (p.max_seq_len + kBoundsChunk - 1) / kBoundsChunk : 1;
  const unsigned grid = static_cast<unsigned>(static_cast<int64_t>(p.batch) * p.h_kv * n_chunks);
#define NBX_BOUNDS(PT, QT) bounds_kernel<PT, QT><<<grid, kBoundsThreads, 0, stream>>>(p, q_norm, kv_max, n_chunks)
  if (q_dtype == NBX_F32) {
    if (pool_dtype == NBX_F32) NBX_BOUNDS(F32, F32);
    else if (pool_dtype == NBX_BF16) NBX_BOUNDS(BF16, F32);
    else NBX_BOUNDS(E4M3, F32);
  } else {
    if (pool_dtype == NBX_F32) NBX_BOUNDS(F32, BF16);
    else if (pool_dtype == NBX_BF16) NBX_BOUNDS(BF16, BF16);
    else NBX_BOUNDS(E4M3, BF16);
  }
#undef NBX_BOUNDS
  return cudaGetLastError();
}

cudaError_t decode_dispatch(const DecodeParams& p, int q_dtype, int pool_dtype, int grid_limit,
                            cudaStream_t stream) {
  DecodeParams q = p;
  const bool mma = mma_path_applies(p, q_dtype, pool_dtype);
  q.part_f16 = mma && pool_dtype == NBX_E4M3 ? 1 : 0;   // fp8 pools on tensor cores: f16 partials
  if (mma) {
    // a tensor-core window: splits sized for one wave of work units over the GPU's SMs (the grid
    // limit does not enter, so the partition, and the result, is the same at any grid size)
    q.tc_units = device_info().sm_count;
    q.tc_pairs = p.h_kv * ((p.rows * p.group + kMmaRowsPerTile - 1) / kMmaRowsPerTile);
  }
  const size_t plan_smem = plan_smem_bytes(q.batch);
  cudaError_t e = q.tc_units > 0 ? launch_pdl(plan_kernel<true>, 1u, kPlanThreads, plan_smem, stream, q)
                                 : launch_pdl(plan_kernel<false>, 1u, kPlanThreads, plan_smem, stream, q);
  if (e != cudaSuccess) return e;
  if (mma) e = decode_dispatch_mma(q, pool_dtype, grid_limit, stream);
  else if (pool_dtype == NBX_F32) e = decode_dispatch_F32(q, q_dtype, grid_limit, stream);
  else if (pool_dtype == NBX_BF16) e = decode_dispatch_BF16(q, q_dtype, grid_limit, stream);
  else e = decode_dispatch_E4M3(q, q_dtype, grid_limit, stream);
  if (e != cudaSuccess) return e;
  if (q.max_splits <= 1) return cudaSuccess;   // every sequence has one split: the partials are the output
  const int64_t items = static_cast<int64_t>(q.batch) * q.h_kv * q.row_blocks * kQB * ((q.d / 4 + 31) / 32);
  int64_t grid = static_cast<int64_t>(device_info().sm_count) * 24;
  if (grid > items) grid = items;
  if (q.part_f16)
    return launch_pdl(decode_merge_kernel<true>, static_cast<unsigned>(grid), kDecodeMergeThreads, 0, stream, q);
  return launch_pdl(decode_merge_kernel<false>, static_cast<unsigned>(grid), kDecodeMergeThreads, 0, stream, q);
}

}  // namespace nbx
