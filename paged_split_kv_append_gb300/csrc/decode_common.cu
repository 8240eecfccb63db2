// The split plan kernel, the standalone merge kernel, the workspace layout and the
// decode launch sequence (plan, then the persistent partial kernel).
#include "decode_kernels.cuh"

namespace nbx {

constexpr int kPlanThreads = 1024;
constexpr int kSortMax = 2048;   // batches up to this size are ordered longest split first

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

// Reads the device lengths, writes every sequence's plan (len, positions per split, non-empty
// splits), zeroes the work counter, writes 0 to the output rows of empty sequences, and writes
// the work list of (sequence, split) entries: sequences with the longest splits first, splits
// ascending.
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(DecodeParams p) {
  __shared__ int s_key[kSortMax];
  __shared__ int s_order[kSortMax];
  __shared__ int s_cnt[kSortMax];
  __shared__ int s_seg[kSortMax];
  __shared__ int s_len[kSortMax];
  __shared__ int s_warp[kPlanThreads / 32];
  __shared__ int s_total;
  const int tid = threadIdx.x;
  const int B = p.batch;
  const int64_t cap = static_cast<int64_t>(p.max_pages) * p.page_tokens;
  const bool sorted = B <= kSortMax;
  pdl_launch_dependents();   // the partial kernel may start its prologue now; it waits for this grid
  for (int b = tid; b < B; b += kPlanThreads) {
    int L = p.seq_lens[b];
    if (L < 0 || L > p.max_seq_len || static_cast<int64_t>(L) > cap) {
      raise_status(p.status, NBX_DEV_BAD_LEN);
      L = 0;
    }
    int S = (max(L, 1) + NBX_SPLIT_POSITIONS - 1) / NBX_SPLIT_POSITIONS;
    S = S > NBX_MAX_SPLITS ? NBX_MAX_SPLITS : S;
    int seg = (L + S - 1) / S;
    seg = ((seg + p.page_tokens - 1) / p.page_tokens) * p.page_tokens;
    const int n = L > 0 ? (L + seg - 1) / seg : 0;
    SeqPlan sp;
    sp.len = L;
    sp.seg = seg;
    sp.n_splits = n;
    sp.pad = 0;
    p.plan[b] = sp;
    if (sorted) {
      s_key[b] = n > 0 ? seg : -1;
      s_cnt[b] = n;
      s_seg[b] = seg;
      s_len[b] = L;
    }
  }
  if (tid == 0) p.header[1] = 0;
  __syncthreads();
  // a sequence with no position to read gets no work unit: its rows are written here (0)
  const int64_t row_vec4 = static_cast<int64_t>(p.rows) * p.h_q * p.d / 4;
  for (int b = 0; b < B; ++b) {
    if ((sorted ? s_cnt[b] : p.plan[b].n_splits) != 0) continue;
    float4* o = reinterpret_cast<float4*>(p.out) + b * row_vec4;
    for (int64_t x = tid; x < row_vec4; x += kPlanThreads) o[x] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (sorted) {
    for (int b = tid; b < B; b += kPlanThreads) {
      const int k = s_key[b];
      int rank = 0;
      for (int c = 0; c < B; ++c) {
        const int kc = s_key[c];
        rank += (kc > k) || (kc == k && c < b);
      }
      s_order[rank] = b;
    }
    __syncthreads();
    for (int i = tid; i < B; i += kPlanThreads) s_key[i] = s_cnt[s_order[i]];   // counts in list order
    __syncthreads();
  }
  // exclusive scan of the split counts in list order: each thread a contiguous run, then a block scan
  const int per = (B + kPlanThreads - 1) / kPlanThreads;
  const int lo = min(B, tid * per), hi = min(B, lo + per);
  int run = 0;
  for (int i = lo; i < hi; ++i) run += sorted ? s_key[i] : p.plan[i].n_splits;
  const int lane = tid & 31, warp = tid >> 5;
  int x = run;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;
    if (lane == 31) s_total = w;
  }
  __syncthreads();
  int base = x - run + (warp > 0 ? s_warp[warp - 1] : 0);
  for (int i = lo; i < hi; ++i) {
    const int b = sorted ? s_order[i] : i;
    int n, seg, len;
    if (sorted) {
      n = s_cnt[b];
      seg = s_seg[b];
      len = s_len[b];
    } else {
      const SeqPlan sp = p.plan[b];
      n = sp.n_splits;
      seg = sp.seg;
      len = sp.len;
    }
    for (int s = 0; s < n; ++s) {
      Entry e;
      e.b = b;
      e.s = s;
      e.start = s * seg;
      e.end = min((s + 1) * seg, len);
      p.entries[base + s] = e;
    }
    base += n;
  }
  if (tid == 0) p.header[0] = s_total;
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
constexpr int kDecodeMergeThreads = 128;

// Merges the split partials of every (sequence, KV head, row block) with more than one split:
// M = max_s m_s, w_s = 2^(m_s - M) (m in log2 units; splits with m = -inf skipped),
// out = v_scale * sum_s w_s acc_s / sum_s w_s l_s, s ascending. One-split sequences were written
// by the partial kernel.
__global__ void __launch_bounds__(kDecodeMergeThreads) decode_merge_kernel(DecodeParams p) {
  __shared__ float s_m[kQB][NBX_MAX_SPLITS];
  __shared__ float s_l[kQB][NBX_MAX_SPLITS];
  __shared__ float s_scale[kQB];
  __shared__ int s_dead[kQB];
  __shared__ long long s_orow[kQB];
  pdl_wait();   // every partial of the decode is written and visible from here on
  const int tid = threadIdx.x;
  const int RG = p.rows * p.group;
  const int per_seq = p.h_kv * p.row_blocks;
  const int n_groups = p.batch * per_seq;
  for (int gi = blockIdx.x; gi < n_groups; gi += gridDim.x) {
    const int b = gi / per_seq;
    const int rem = gi - b * per_seq;
    const int h = rem / p.row_blocks;
    const int rb = rem - h * p.row_blocks;
    const int S = p.plan[b].n_splits;
    if (S <= 1) continue;
    const int q0 = rb * kQB;
    const int nvec = min(kQB, RG - q0);
    if (tid < nvec) {
      const int qi = q0 + tid;
      const int r = qi / p.group;
      const int g = qi - r * p.group;
      s_orow[tid] = (static_cast<long long>(b) * p.rows + r) * p.h_q + static_cast<long long>(h) * p.group + g;
    }
    __syncthreads();
    // every (vector, split) pair's m and l, one load each
    for (int x = tid; x < nvec * S; x += kDecodeMergeThreads) {
      const int i = x / S;
      const int sp = x - i * S;
      const long long row = s_orow[i] * p.max_splits + sp;
      s_m[i][sp] = p.m_part[row];
      s_l[i][sp] = p.l_part[row];
    }
    __syncthreads();
    if (tid < nvec) {
      float M = -INFINITY;
      for (int sp = 0; sp < S; ++sp) M = max_nan(M, s_m[tid][sp]);
      float L = 0.f;
      for (int sp = 0; sp < S; ++sp) {
        const float ms = s_m[tid][sp];
        const bool lv = ms != -INFINITY;
        const float w = lv ? fast_exp2(ms - M) : 0.f;
        if (lv) L += w * s_l[tid][sp];
        s_m[tid][sp] = lv ? w : -1.f;   // -1 marks a split with no visible key
      }
      s_dead[tid] = (M == -INFINITY) ? 1 : 0;
      s_scale[tid] = p.v_scale / L;
    }
    __syncthreads();
    // each thread a float4 of one vector's output; 16 splits' loads in flight per batch, summed in
    // ascending split order
    const int d4 = p.d / 4;
    for (int o = tid; o < nvec * d4; o += kDecodeMergeThreads) {
      const int i = o / d4;
      const int dd = (o - i * d4) * 4;
      const long long orow = s_orow[i];
      const float4* acc = reinterpret_cast<const float4*>(p.acc_part + orow * p.max_splits * p.d + dd);
      const int stride4 = p.d / 4;
      float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s0 = 0; s0 < S; s0 += 16) {
        float4 a[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
          a[k] = (s0 + k < S) ? acc[static_cast<long long>(s0 + k) * stride4] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          if (s0 + k >= S) break;
          const float w = s_m[i][s0 + k];
          if (w != -1.f) {
            A.x += w * a[k].x;
            A.y += w * a[k].y;
            A.z += w * a[k].z;
            A.w += w * a[k].w;
          }
        }
      }
      const float sc = s_scale[i];
      float4 r = s_dead[i] ? make_float4(0.f, 0.f, 0.f, 0.f) : make_float4(A.x * sc, A.y * sc, A.z * sc, A.w * sc);
      *reinterpret_cast<float4*>(p.out + orow * p.d + dd) = r;
    }
    __syncthreads();
  }
}

cudaError_t decode_dispatch(const DecodeParams& p, int q_dtype, int pool_dtype, int grid_limit,
                            cudaStream_t stream) {
  plan_kernel<<<1, kPlanThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (pool_dtype == NBX_F32) e = decode_dispatch_F32(p, q_dtype, grid_limit, stream);
  else if (pool_dtype == NBX_BF16) e = decode_dispatch_BF16(p, q_dtype, grid_limit, stream);
  else e = decode_dispatch_E4M3(p, q_dtype, grid_limit, stream);
  if (e != cudaSuccess) return e;
  if (p.max_splits <= 1) return cudaSuccess;   // every sequence has one split: the partials are the output
  const int64_t groups = static_cast<int64_t>(p.batch) * p.h_kv * p.row_blocks;
  int64_t grid = static_cast<int64_t>(device_info().sm_count) * 4;
  if (grid > groups) grid = groups;
  return launch_pdl(decode_merge_kernel, static_cast<unsigned>(grid), kDecodeMergeThreads, 0, stream, p);
}

}  // namespace nbx
