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
  w->tickets = off;
  off += up(static_cast<size_t>(batch) * h_kv * rb * 4);
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
// splits), zeroes the merge tickets and the work counter, and writes the work list of
// (sequence, split) entries: sequences with the longest splits first, splits ascending.
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(DecodeParams p) {
  __shared__ int s_key[kSortMax];
  __shared__ int s_order[kSortMax];
  __shared__ int s_cnt[kSortMax];
  __shared__ int s_warp[kPlanThreads / 32];
  __shared__ int s_total;
  const int tid = threadIdx.x;
  const int B = p.batch;
  const int64_t cap = static_cast<int64_t>(p.max_pages) * p.page_tokens;
  const bool sorted = B <= kSortMax;
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
    }
  }
  const int64_t n_tickets = static_cast<int64_t>(B) * p.h_kv * p.row_blocks;
  for (int64_t x = tid; x < n_tickets; x += kPlanThreads) p.tickets[x] = 0;
  if (tid == 0) p.header[1] = 0;
  __syncthreads();
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
    const SeqPlan sp = p.plan[b];
    for (int s = 0; s < sp.n_splits; ++s) {
      Entry e;
      e.b = b;
      e.s = s;
      e.start = s * sp.seg;
      e.end = min((s + 1) * sp.seg, sp.len);
      p.entries[base + s] = e;
    }
    base += sp.n_splits;
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
    for (int s = 0; s < p.splits; ++s) M = fmaxf(M, m[s]);
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

cudaError_t decode_dispatch(const DecodeParams& p, int q_dtype, int pool_dtype, int grid_limit,
                            cudaStream_t stream) {
  plan_kernel<<<1, kPlanThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (pool_dtype == NBX_F32) return decode_dispatch_F32(p, q_dtype, grid_limit, stream);
  if (pool_dtype == NBX_BF16) return decode_dispatch_BF16(p, q_dtype, grid_limit, stream);
  return decode_dispatch_E4M3(p, q_dtype, grid_limit, stream);
}

}  // namespace nbx
