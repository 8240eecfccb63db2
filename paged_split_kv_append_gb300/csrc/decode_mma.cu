// Kernel 2, tensor-core variant: the split partial on tcgen05 when the query rows of one KV
// head fill an MMA tile (rows x GQA group >= 64: verify windows, prefill chunks).
//
// Same maths as decode_partial_kernel (nbxtensor/ops/paged_decode_attn.py,
// paged_decode_attn_split_kernel: per split an online softmax over the split's keys, an
// unnormalised partial (m, l, acc)); the split plan and the fixed-order merge are shared. The
// query rows of one KV head become the M dimension, as in the grouped view of
// nbxtensor/ops/attention_wrappers.py, _math_attention, and as TensorFold PR #1219 ("Gotchas")
// describes for its attn_rows kernel: each K/V tile is read once for all rows of a stream.
//
// GB300 design (one CTA per SM, 6 warps):
//  * Work unit = (split entry, KV head, M tile), M tile fastest. An M tile holds Rt whole query
//    rows x the G query heads of the KV head (Rt = min(rows, 128 / G)), so its Q block, its output
//    block and its partial block are boxes of 4-D / 5-D tensor maps. Static round-robin over the
//    plan's longest-first list.
//  * warp 4 (producer, one thread): an event loop over three TMA streams -- the unit's Q box, K
//    tiles and V tiles of 64 positions (a page, or a 64-aligned part of one) into separate rings,
//    128-byte swizzle -- issuing whichever has a free slot. A page id outside the pool loads rows
//    before the tensor, which read as zeros, and its positions are masked.
//  * warp 5 (MMA): holds the TMEM; an event loop issues, as soon as their inputs are ready,
//      S[x % 2] = Q K(x)^T                    M=128, N=64, K=d; A, B from shared memory
//      O       += P_hi(y) V(y) + P_lo(y) V(y)  M=128, N=d, K=64; P from TMEM, V MN-major
//    (kind::f16, bf16 x bf16 -> fp32 in TMEM) and signals completions with tcgen05.commit. P
//    enters the product as two bf16 terms, P_hi = bf16(p) and P_lo = bf16(p - P_hi), so the
//    weights keep about 16 bits. The warp zeroes V rows past a split's end before their PV
//    (0 x NaN would otherwise leak) and skips 16-position steps that hold none.
//  * warps 0-3 (softmax, one query vector per thread = one TMEM lane): read S from TMEM, mask
//    (split end, causal row position, missing pages), run the online softmax in log2 units with
//    the lazy rescale (O is rescaled in TMEM only when a row's max grows by more than 2^8), and
//    write P_hi / P_lo over the S columns they came from. At the end of a unit they move O from
//    TMEM through 128-byte-swizzled shared memory to TMA tensor stores: the partial, or the
//    normalised output when the sequence has one split. Rows past the sequence's last row are
//    outside the tensor's row dimension, so the stores leave them alone.
//  * Every wait is bounded. On timeout the kernel records NBX_DEV_TIMEOUT, waits (bounded) for
//    its copies and MMAs in flight, releases its TMEM and returns.
#include <atomic>
#include <cuda.h>
#include <cudaTypedefs.h>

#include "nbx_device.cuh"
#include "nbx_internal.h"

namespace nbx {
namespace {

constexpr int kMmaM = 128;       // TMEM lanes / rows of an M tile
constexpr int kMmaN = 64;        // positions per K/V tile
constexpr int kMmaThreads = 192;
constexpr int kSoftmaxThreads = 128;
constexpr float kMmaTau = 8.0f;  // lazy-rescale threshold, log2 units
constexpr int kChunk = 32;       // output columns per epilogue store

template <int D>
struct MmaCfg {
  static constexpr int kStages = D <= 128 ? 4 : 2;    // K slots, and as many V slots
  static constexpr int kQBytes = kMmaM * D * 2;
  static constexpr int kTileBytes = kMmaN * D * 2;     // one K or V tile, bf16
  static constexpr int kStgBytes = kMmaM * kChunk * 4;  // one epilogue staging buffer
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kStgOff = kVOff + kStages * kTileBytes;
  static constexpr int kBarOff = kStgOff + 2 * kStgBytes;
  static constexpr int kSmem = kBarOff + 512 + 1024;   // barriers + slack for 1024-byte alignment
  static constexpr uint32_t kTmemCols = D <= 128 ? 256 : 512;
  static constexpr uint32_t kOCol = 128;               // S/P buffers at columns 0 and 64, O from 128
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

struct MmaMaps {
  CUtensorMap k, v;   // 2-D pool views [num_pages * h_kv * page_tokens][d], box 64 x 64
  CUtensorMap q;      // 4-D [batch][rows][h_q][d] bf16, box {64, G, Rt, 1}
  CUtensorMap out;    // 4-D [batch][rows][h_q][d] fp32, box {32, G, Rt, 1}
  CUtensorMap part;   // 5-D [batch][rows][h_q][max_splits][d] fp32, box {32, 1, G, Rt, 1}
};

// ---- tcgen05 / TMA wrappers (inline PTX)
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Arrives on `bar` once every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// D(tmem) = A(smem) * B(smem) (+ D if acc), kind::f16
__device__ __forceinline__ void tc_mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          bool acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc ? 1u : 0u)
      : "memory");
}

// D(tmem) = A(tmem) * B(smem) (+ D if acc), kind::f16; A row m in lane m, two 16-bit elements of
// K per 32-bit column (the lower K index in the low half)
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          bool acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc ? 1u : 0u)
      : "memory");
}

// 16 consecutive 32-bit TMEM columns of this thread's lane
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, const void* src, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}
__device__ __forceinline__ void tma_store_5d(const CUtensorMap* map, const void* src, int c0, int c1, int c2, int c3,
                                             int c4) {
  asm volatile("cp.async.bulk.tensor.5d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5, %6}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// every bulk store group but the newest `N` has finished reading shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// every bulk store group has completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Shared-memory matrix descriptor: start >> 4 in bits [0,14), leading byte offset >> 4 in [16,30),
// stride byte offset >> 4 in [32,46), descriptor version 1 in [46,48), base offset 0 (operand
// blocks are 1024-byte aligned), layout 2 = 128-byte swizzle in [61,64).
//   K-major, 128-byte swizzle: rows of 128 bytes (64 bf16 of K), 8-row groups 1024 bytes apart
//     (stride offset); a K step of 16 elements advances the start by 32 bytes.
//   MN-major, 128-byte swizzle: rows of 128 bytes (64 bf16 of N) per K index, 8-K groups 1024
//     bytes apart (stride offset), 64-wide N blocks `lbo` bytes apart (leading offset).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFF) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), bf16 A and B (bits 7-9,
// 10-12 = 1), A K-major (bit 15 = 0), B K-major or MN-major (bit 16), N >> 3 in bits 17-22,
// M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t mma_idesc(int m, int n, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// Bounded wait that also gives up when another role of the CTA has given up.
__device__ __forceinline__ bool bwait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if ((i & 3u) == 0u && global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// The same, with one answer for the whole warp (the tcgen05 .sync.aligned forms that follow need
// every lane).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return __all_sync(0xffffffffu, bwait(bar, parity, abort_flag));
}

struct MmaUnit {
  int b, s, h, mt, start, end, len, n_splits, tiles;
};

__device__ __forceinline__ MmaUnit mma_unit(const DecodeParams& p, int u, int m_tiles) {
  MmaUnit m;
  const int span = p.h_kv * m_tiles;
  const int e = u / span;
  const int rem = u - e * span;
  m.h = rem / m_tiles;
  m.mt = rem - m.h * m_tiles;
  const Entry en = p.entries[e];
  m.b = en.b;
  m.s = en.s;
  m.start = en.start;
  m.end = en.end;
  const SeqPlan sp = p.plan[en.b];
  m.len = sp.len;
  m.n_splits = sp.n_splits;
  m.tiles = (en.end - en.start + kMmaN - 1) / kMmaN;
  return m;
}

// Walks this CTA's tiles in order: units blockIdx.x, blockIdx.x + gridDim.x, ..., tiles of each.
struct TileIter {
  int u;        // unit index
  uint32_t k;   // unit ordinal within this CTA
  int t;        // tile within the unit
  uint32_t x;   // tile ordinal within this CTA
  bool done;
  MmaUnit mu;
  __device__ __forceinline__ void begin(const DecodeParams& p, int m_tiles, int n_units) {
    u = blockIdx.x;
    k = 0;
    t = 0;
    x = 0;
    done = u >= n_units;
    if (!done) mu = mma_unit(p, u, m_tiles);
  }
  __device__ __forceinline__ void next_unit(const DecodeParams& p, int m_tiles, int n_units) {
    t = 0;
    ++k;
    u += gridDim.x;
    done = u >= n_units;
    if (!done) mu = mma_unit(p, u, m_tiles);
  }
  __device__ __forceinline__ void next_tile(const DecodeParams& p, int m_tiles, int n_units) {
    ++x;
    if (++t >= mu.tiles) next_unit(p, m_tiles, n_units);
  }
};

// First pool row of the tile starting at position n0 of the unit's sequence, or -kMmaN (rows
// before the tensor, read as zeros) if its page id is outside the pool.
__device__ __forceinline__ int tile_row(const DecodeParams& p, const MmaUnit& mu, int n0) {
  const int page = p.block_table[static_cast<int64_t>(mu.b) * p.max_pages + n0 / p.page_tokens];
  if (page < 0 || page >= p.num_pages) {
    raise_status(p.status, NBX_DEV_BAD_PAGE);
    return -kMmaN;
  }
  return (page * p.h_kv + mu.h) * p.page_tokens + (n0 % p.page_tokens);
}

template <int D>
__global__ void __launch_bounds__(kMmaThreads, 1)
    decode_partial_mma_kernel(DecodeParams p, const __grid_constant__ MmaMaps maps) {
  using C = MmaCfg<D>;
  constexpr int NS = C::kStages;
  extern __shared__ __align__(1024) char smem_raw[];
  char* smem = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  char* q_s = smem + C::kQOff;
  char* k_s = smem + C::kKOff;
  char* v_s = smem + C::kVOff;
  char* stg_s = smem + C::kStgOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* k_full = bars;             // [NS]  K tile landed (TMA bytes)
  uint64_t* k_empty = bars + NS;       // [NS]  QK^T of the slot's tile done
  uint64_t* v_full = bars + 2 * NS;    // [NS]  V tile landed
  uint64_t* v_empty = bars + 3 * NS;   // [NS]  PV of the slot's tile done
  uint64_t* s_full = bars + 4 * NS;    // [2]   S of the buffer's tile in TMEM
  uint64_t* p_full = s_full + 2;       // [2]   P of the buffer's tile in TMEM (128 arrivals)
  uint64_t* sp_free = s_full + 4;      // [2]   PV of the buffer's tile done: S/P buffer reusable, O
                                       //       holds every PV up to that tile
  uint64_t* stg_full = s_full + 6;     // [2]   staging buffer written (128 arrivals)
  uint64_t* stg_free = s_full + 8;     // [2]   staging buffer read by its store
  uint64_t* q_full = s_full + 10;      //       the unit's Q box landed
  uint64_t* q_empty = s_full + 11;     //       every QK^T of the unit done
  uint64_t* o_free = s_full + 12;      //       O read out by the epilogue (128 arrivals)
  uint64_t* done_bar = s_full + 13;    //       every MMA of the CTA done
  volatile int* abort_flag = reinterpret_cast<int*>(s_full + 14);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_full + 15);
  // Phase discipline: a thread waits on phase j of a barrier only once it knows phase j - 1 has
  // completed and while phase j + 1 cannot have (a parity wait cannot tell them apart). The
  // softmax threads therefore track PV completion through sp_free[y % 2]: once S(g) has landed,
  // PV(g - 2) is known complete (QK(g) waited for it), so PV(g - 1) is exactly one phase ahead.

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], kSoftmaxThreads);
      mbar_init(&sp_free[i], 1);
      mbar_init(&stg_full[i], kSoftmaxThreads);
      mbar_init(&stg_free[i], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(o_free, kSoftmaxThreads);
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();   // the plan kernel's work list and the append's positions are visible from here on
  pdl_launch_dependents();

  const int G = p.group;
  const int Rt = min(p.rows, kMmaM / G);                 // query rows per M tile
  const int m_tiles = (p.rows + Rt - 1) / Rt;
  const int n_units = p.header[0] * p.h_kv * m_tiles;

  if (warp == 4) {
    // ======================================================== TMA producer (one thread)
    if (lane == 0) {
      TileIter qi, ki, vi;
      qi.begin(p, m_tiles, n_units);
      ki.begin(p, m_tiles, n_units);
      vi.begin(p, m_tiles, n_units);
      bool ok = true;
      uint64_t idle_since = 0;
      while (!vi.done) {
        bool moved = false;
        // the unit's Q box, once every QK^T of the previous unit is done
        if (!qi.done && (qi.k == 0 || mbar_test(q_empty, (qi.k - 1) & 1u))) {
          mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(D / 64) * 64u * G * Rt * 2u);
#pragma unroll
          for (int a = 0; a < D / 64; ++a)
            tma_load_4d(q_s + a * (kMmaM * 128), &maps.q, a * 64, qi.mu.h * G, qi.mu.mt * Rt, qi.mu.b, q_full);
          qi.next_unit(p, m_tiles, n_units);
          moved = true;
        }
        // K tile x into slot x % NS once the QK^T of tile x - NS is done
        if (!ki.done && (ki.x < static_cast<uint32_t>(NS) || mbar_test(&k_empty[ki.x % NS], (ki.x / NS - 1) & 1u))) {
          const int row0 = tile_row(p, ki.mu, ki.mu.start + ki.t * kMmaN);
          uint64_t* bar = &k_full[ki.x % NS];
          char* dst = k_s + (ki.x % NS) * C::kTileBytes;
          mbar_arrive_expect_tx(bar, C::kTileBytes);
#pragma unroll
          for (int a = 0; a < D / 64; ++a) tma_load_2d(dst + a * (kMmaN * 128), &maps.k, a * 64, row0, bar);
          ki.next_tile(p, m_tiles, n_units);
          moved = true;
        }
        // V tile y into slot y % NS once the PV of tile y - NS is done
        if (!vi.done && vi.x < ki.x &&
            (vi.x < static_cast<uint32_t>(NS) || mbar_test(&v_empty[vi.x % NS], (vi.x / NS - 1) & 1u))) {
          const int row0 = tile_row(p, vi.mu, vi.mu.start + vi.t * kMmaN);
          uint64_t* bar = &v_full[vi.x % NS];
          char* dst = v_s + (vi.x % NS) * C::kTileBytes;
          mbar_arrive_expect_tx(bar, C::kTileBytes);
#pragma unroll
          for (int a = 0; a < D / 64; ++a) tma_load_2d(dst + a * (kMmaN * 128), &maps.v, a * 64, row0, bar);
          vi.next_tile(p, m_tiles, n_units);
          moved = true;
        }
        if (moved) {
          idle_since = 0;
        } else {
          const uint64_t now = global_timer_ns();
          if (idle_since == 0) idle_since = now;
          if (*abort_flag || now - idle_since > kWaitLimitNs) {
            ok = false;
            break;
          }
          __nanosleep(64);
        }
      }
      if (!ok) {
        *abort_flag = 1;
        raise_status(p.status, NBX_DEV_TIMEOUT);
      }
      // the copies issued last have landed before the CTA can exit
      for (uint32_t j = ki.x > static_cast<uint32_t>(NS) ? ki.x - NS : 0; j < ki.x; ++j)
        mbar_wait(&k_full[j % NS], (j / NS) & 1u, 100000000ull);
      for (uint32_t j = vi.x > static_cast<uint32_t>(NS) ? vi.x - NS : 0; j < vi.x; ++j)
        mbar_wait(&v_full[j % NS], (j / NS) & 1u, 100000000ull);
      if (qi.k > 0) mbar_wait(q_full, (qi.k - 1) & 1u, 100000000ull);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ======================================================== MMA issuer (lane 0 decides and issues)
    constexpr uint32_t kIdescS = mma_idesc(kMmaM, kMmaN, false);
    constexpr uint32_t kIdescO = mma_idesc(kMmaM, D, true);
    const uint32_t q_addr = smem_u32(q_s);
    TileIter qk, pv;
    qk.begin(p, m_tiles, n_units);
    pv.begin(p, m_tiles, n_units);
    bool ok = true;
    uint64_t idle_since = 0;
    while (!pv.done) {
      bool moved = false;
      // ---- S(x) = Q K(x)^T: K landed, the S/P buffer's previous PV done, the unit's Q landed
      int go = 0;
      if (lane == 0 && !qk.done) {
        const uint32_t x = qk.x;
        go = mbar_test(&k_full[x % NS], (x / NS) & 1u) && (x < 2 || mbar_test(&sp_free[x & 1u], ((x >> 1) - 1) & 1u)) &&
             (qk.t > 0 || mbar_test(q_full, qk.k & 1u));
      }
      if (__shfl_sync(0xffffffffu, go, 0)) {
        tc_fence_after();
        if (lane == 0) {
          const uint32_t x = qk.x;
          const uint32_t kb = smem_u32(k_s + (x % NS) * C::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t a = kk >> 2, sub = kk & 3;
            const uint64_t ad = smem_desc(q_addr + a * (kMmaM * 128) + sub * 32, 16, 1024);
            const uint64_t bd = smem_desc(kb + a * (kMmaN * 128) + sub * 32, 16, 1024);
            tc_mma_ss(tmem + (x & 1u) * kMmaN, ad, bd, kIdescS, kk > 0);
          }
          tc_commit(&s_full[x & 1u]);
          tc_commit(&k_empty[x % NS]);
          if (qk.t == qk.mu.tiles - 1) tc_commit(q_empty);
        }
        __syncwarp();
        qk.next_tile(p, m_tiles, n_units);
        moved = true;
      }
      // ---- O += P(y) V(y): P written, V landed, O read out by the previous unit's epilogue
      go = 0;
      if (lane == 0 && pv.x < qk.x) {
        const uint32_t y = pv.x;
        go = mbar_test(&p_full[y & 1u], (y >> 1) & 1u) && mbar_test(&v_full[y % NS], (y / NS) & 1u) &&
             (pv.t > 0 || pv.k == 0 || mbar_test(o_free, (pv.k - 1) & 1u));
      }
      if (__shfl_sync(0xffffffffu, go, 0)) {
        const uint32_t y = pv.x;
        char* vd = v_s + (y % NS) * C::kTileBytes;
        const int valid = min(kMmaN, pv.mu.end - (pv.mu.start + pv.t * kMmaN));
        const int ksteps = (valid + 15) >> 4;
        if (valid & 15) {   // rows past the split's end inside the last 16-position step
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
          const int r0 = valid, nr = (ksteps << 4) - valid;
          for (int a = 0; a < D / 64; ++a)
            for (int i = lane; i < nr * 8; i += 32)
              *reinterpret_cast<uint4*>(vd + a * (kMmaN * 128) + (r0 + (i >> 3)) * 128 + (i & 7) * 16) = z;
          fence_proxy_async();
        }
        __syncwarp();
        tc_fence_after();
        if (lane == 0) {
          const uint32_t vb = smem_u32(vd);
          const uint32_t pcol = tmem + (y & 1u) * kMmaN;
#pragma unroll
          for (int part = 0; part < 2; ++part) {
#pragma unroll
            for (int kk = 0; kk < kMmaN / 16; ++kk) {
              if (kk < ksteps) {
                const uint64_t bd = smem_desc(vb + kk * (16 * 128), kMmaN * 128, 1024);
                tc_mma_ts(tmem + C::kOCol, pcol + part * (kMmaN / 2) + kk * 8, bd, kIdescO,
                          !(pv.t == 0 && part == 0 && kk == 0));
              }
            }
          }
          tc_commit(&v_empty[y % NS]);
          tc_commit(&sp_free[y & 1u]);
        }
        __syncwarp();
        pv.next_tile(p, m_tiles, n_units);
        moved = true;
      }
      if (moved) {
        idle_since = 0;
      } else {
        const uint64_t now = global_timer_ns();
        if (idle_since == 0) idle_since = now;
        const int give_up = *abort_flag || now - idle_since > kWaitLimitNs;
        if (__shfl_sync(0xffffffffu, give_up, 0)) {
          ok = false;
          break;
        }
        __nanosleep(32);
      }
    }
    if (!ok) {
      *abort_flag = 1;
      if (lane == 0) raise_status(p.status, NBX_DEV_TIMEOUT);
    }
    // every MMA of this CTA has completed before the TMEM is released
    if (lane == 0) tc_commit(done_bar);
    __syncwarp();
    mbar_wait(done_bar, 0, 100000000ull);
  } else {
    // ======================================================== softmax warps (row = threadIdx.x)
    const int row = threadIdx.x;
    const int rt = row / G;                       // query row within the M tile
    const int gq = row - rt * G;                  // query head within the KV head's group
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    bool ok = true;
    uint32_t g = 0, e = 0;
    TileIter it;
    it.begin(p, m_tiles, n_units);
    while (!it.done) {
      const MmaUnit mu = it.mu;
      const int r = mu.mt * Rt + rt;
      const bool row_ok = rt < Rt && r < p.rows;
      const int pos = mu.len - p.rows + r;   // last position this row sees
      float m_run = -INFINITY, l_run = 0.f;
      for (int t = 0; t < mu.tiles; ++t, ++g) {
        const int n0 = mu.start + t * kMmaN;
        const int page = p.block_table[static_cast<int64_t>(mu.b) * p.max_pages + n0 / p.page_tokens];
        const bool tile_ok = page >= 0 && page < p.num_pages;
        const uint32_t sbuf = tmem + (g & 1u) * kMmaN;
        if (!warp_wait(&s_full[g & 1u], (g >> 1) & 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[kMmaN];
#pragma unroll
        for (int c = 0; c < kMmaN / 16; ++c) tmem_ld16(lane_base + (sbuf - tmem) + c * 16, sr + c * 16);
        tmem_wait_ld();
        // ---- mask and row max (log2 units; NaN propagates through the max)
        const int lim = (row_ok && tile_ok) ? min(mu.end - 1, pos) - n0 : -1;   // last visible column
        float sv[kMmaN];
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < kMmaN; ++j) {
          sv[j] = j <= lim ? __uint_as_float(sr[j]) * p.qk_scale_log2 : -INFINITY;
          mx = max_nan(mx, sv[j]);
        }
        const bool grow = !(mx <= m_run + kMmaTau);
        const float m_new = grow ? mx : m_run;
        const float f = (m_new == m_run) ? 1.f : fast_exp2(m_run - m_new);
        if (t > 0 && __any_sync(0xffffffffu, f != 1.f)) {
          // O holds the PVs of tiles g-t .. g-1: wait for the last, then rescale it in TMEM
          if (!warp_wait(&sp_free[(g - 1) & 1u], ((g - 1) >> 1) & 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 16; ++c) {
            uint32_t ov[16];
            tmem_ld16(lane_base + C::kOCol + c * 16, ov);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * f);
            tmem_st16(lane_base + C::kOCol + c * 16, ov);
          }
        }
        m_run = m_new;
        l_run *= f;
        const float m_use = (m_run == -INFINITY) ? 0.f : m_run;   // all scores -inf: p = 0
        // ---- P = 2^(s - m) as bf16 P_hi + P_lo over the S columns: hi in [0, 32), lo in [32, 64)
        float lsum = 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t wh[16], wl[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float p0 = fast_exp2(sv[half * 32 + 2 * i] - m_use);
            const float p1 = fast_exp2(sv[half * 32 + 2 * i + 1] - m_use);
            lsum += p0;
            lsum += p1;
            const __nv_bfloat162 hi = __floats2bfloat162_rn(p0, p1);
            const float2 hf = __bfloat1622float2(hi);
            const __nv_bfloat162 lo = __floats2bfloat162_rn(p0 - hf.x, p1 - hf.y);
            wh[i] = *reinterpret_cast<const uint32_t*>(&hi);
            wl[i] = *reinterpret_cast<const uint32_t*>(&lo);
          }
          tmem_st16(lane_base + (sbuf - tmem) + half * 16, wh);
          tmem_st16(lane_base + (sbuf - tmem) + kMmaN / 2 + half * 16, wl);
        }
        l_run += lsum;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_full[g & 1u]);
      }
      if (!ok) break;
      // ---- epilogue: O from TMEM once the unit's last PV is done
      if (!warp_wait(&sp_free[(g - 1) & 1u], ((g - 1) >> 1) & 1u, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool single = mu.n_splits <= 1;
      const float sc = single ? ((m_run == -INFINITY) ? 0.f : p.v_scale / l_run) : 1.f;
      if (row_ok && !single) {
        const int64_t orow = (static_cast<int64_t>(mu.b) * p.rows + r) * p.h_q + static_cast<int64_t>(mu.h) * G + gq;
        p.m_part[orow * p.max_splits + mu.s] = m_run;
        p.l_part[orow * p.max_splits + mu.s] = l_run;
      }
      for (int ch = 0; ch < D / kChunk; ++ch, ++e) {
        uint32_t ov[kChunk];
        tmem_ld16(lane_base + C::kOCol + ch * kChunk, ov);
        tmem_ld16(lane_base + C::kOCol + ch * kChunk + 16, ov + 16);
        tmem_wait_ld();
        if (ch == D / kChunk - 1) {   // O is free for the next unit's first PV
          tc_fence_before();
          mbar_arrive(o_free);
        }
        // staging buffer e % 2 is free once the store of chunk e - 2 has read it
        if (e >= 2) {
          if (row == 0) {
            bulk_wait_read<1>();
            mbar_arrive(&stg_free[e & 1u]);
          }
          if (!warp_wait(&stg_free[e & 1u], ((e >> 1) - 1) & 1u, abort_flag)) {
            ok = false;
            break;
          }
        }
        char* buf = stg_s + (e & 1u) * C::kStgBytes;
#pragma unroll
        for (int c4 = 0; c4 < kChunk / 4; ++c4)
          *reinterpret_cast<float4*>(buf + row * (kChunk * 4) + ((c4 ^ (row & 7)) << 4)) =
              make_float4(__uint_as_float(ov[4 * c4]) * sc, __uint_as_float(ov[4 * c4 + 1]) * sc,
                          __uint_as_float(ov[4 * c4 + 2]) * sc, __uint_as_float(ov[4 * c4 + 3]) * sc);
        fence_proxy_async();
        mbar_arrive(&stg_full[e & 1u]);
        if (row == 0) {
          if (!mbar_wait(&stg_full[e & 1u], (e >> 1) & 1u)) {
            *abort_flag = 1;
          } else if (single) {
            tma_store_4d(&maps.out, buf, ch * kChunk, mu.h * G, mu.mt * Rt, mu.b);
          } else {
            tma_store_5d(&maps.part, buf, ch * kChunk, mu.s, mu.h * G, mu.mt * Rt, mu.b);
          }
          bulk_commit();
        }
      }
      if (!ok) break;
      it.next_unit(p, m_tiles, n_units);
    }
    if (!ok) {
      *abort_flag = 1;
      if (threadIdx.x == 0) raise_status(p.status, NBX_DEV_TIMEOUT);
    }
    if (row == 0) bulk_wait_all();   // the stores have completed before the grid does
  }

  // every role is done and the MMA warp has seen its last MMA complete: release the TMEM
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, C::kTmemCols);
}

// ---- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// A tiled map with 128-byte swizzle; dims and box innermost first, strides in bytes for dims 1...
bool encode(CUtensorMap* map, CUtensorMapDataType type, int rank, const void* base, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box) {
  const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(map, type, static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_maps(MmaMaps* m, const DecodeParams& p) {
  const cuuint64_t D = static_cast<cuuint64_t>(p.d);
  const cuuint32_t G = static_cast<cuuint32_t>(p.group);
  const cuuint32_t Rt = static_cast<cuuint32_t>(p.rows < kMmaM / p.group ? p.rows : kMmaM / p.group);
  const cuuint64_t R = static_cast<cuuint64_t>(p.rows), B = static_cast<cuuint64_t>(p.batch);
  const cuuint64_t HQ = static_cast<cuuint64_t>(p.h_q), S = static_cast<cuuint64_t>(p.max_splits);
  // pools: rows (page * h_kv + h) * page_tokens + position, columns d
  const cuuint64_t pool_dims[2] = {D, static_cast<cuuint64_t>(p.num_pages) * p.h_kv * p.page_tokens};
  const cuuint64_t pool_str[1] = {D * 2};
  const cuuint32_t pool_box[2] = {64, static_cast<cuuint32_t>(kMmaN)};
  // q [B][R][h_q][d] bf16
  const cuuint64_t q_dims[4] = {D, HQ, R, B};
  const cuuint64_t q_str[3] = {D * 2, HQ * D * 2, R * HQ * D * 2};
  const cuuint32_t q_box[4] = {64, G, Rt, 1};
  // out [B][R][h_q][d] fp32
  const cuuint64_t o_dims[4] = {D, HQ, R, B};
  const cuuint64_t o_str[3] = {D * 4, HQ * D * 4, R * HQ * D * 4};
  const cuuint32_t o_box[4] = {static_cast<cuuint32_t>(kChunk), G, Rt, 1};
  // partials [B][R][h_q][S][d] fp32
  const cuuint64_t a_dims[5] = {D, S, HQ, R, B};
  const cuuint64_t a_str[4] = {D * 4, S * D * 4, HQ * S * D * 4, R * HQ * S * D * 4};
  const cuuint32_t a_box[5] = {static_cast<cuuint32_t>(kChunk), 1, G, Rt, 1};
  return encode(&m->k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.k_pool, pool_dims, pool_str, pool_box) &&
         encode(&m->v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.v_pool, pool_dims, pool_str, pool_box) &&
         encode(&m->q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p.q, q_dims, q_str, q_box) &&
         encode(&m->out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.out, o_dims, o_str, o_box) &&
         encode(&m->part, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, p.acc_part, a_dims, a_str, a_box);
}

template <int D>
cudaError_t launch_mma(const DecodeParams& p, int grid_limit, cudaStream_t stream) {
  using C = MmaCfg<D>;
  static std::atomic<uint64_t> configured{0};   // devices whose shared-memory limit is raised
  MmaMaps maps;
  if (!make_maps(&maps, p)) return cudaErrorInvalidValue;
  const DeviceInfo& di = device_info();
  const uint64_t bit = 1ull << (di.device & 63);
  if ((configured.load() & bit) == 0) {
    const cudaError_t e =
        cudaFuncSetAttribute(decode_partial_mma_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  const int Rt = p.rows < kMmaM / p.group ? p.rows : kMmaM / p.group;
  const int m_tiles = (p.rows + Rt - 1) / Rt;
  const int64_t upper = static_cast<int64_t>(p.batch) * p.max_splits * p.h_kv * m_tiles;
  int64_t grid = di.sm_count;
  if (grid_limit > 0 && grid > grid_limit) grid = grid_limit;
  if (grid > upper) grid = upper;
  if (grid < 1) grid = 1;
  return launch_pdl(decode_partial_mma_kernel<D>, static_cast<unsigned>(grid), kMmaThreads, C::kSmem, stream, p,
                    maps);
}

}  // namespace

bool mma_path_applies(const DecodeParams& p, int q_dtype, int pool_dtype) {
  const int64_t pool_rows = static_cast<int64_t>(p.num_pages) * p.h_kv * p.page_tokens;
  return q_dtype == NBX_BF16 && pool_dtype == NBX_BF16 && (p.d == 128 || p.d == 256) &&
         (p.page_tokens % kMmaN) == 0 && p.group <= kMmaM && p.rows * p.group >= 64 &&
         pool_rows < (int64_t{1} << 31) - kMmaN;
}

cudaError_t decode_dispatch_mma(const DecodeParams& p, int grid_limit, cudaStream_t stream) {
  if (p.d == 128) return launch_mma<128>(p, grid_limit, stream);
  return launch_mma<256>(p, grid_limit, stream);
}

}  // namespace nbx
