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
//  * Work unit = (split entry, KV head, M tile of 128 query vectors), M tile fastest, so the M
//    tiles of one split run side by side and share its K/V through L2. Static round-robin over
//    the plan's longest-first list.
//  * warp 4 (producer): TMA (cp.async.bulk.tensor, 128-byte swizzle) brings 64-position tiles of
//    K and V (one page or a 64-aligned part of one) into a ring of stages. A page id outside the
//    pool loads rows outside the tensor, which read as zeros, and its positions are masked.
//  * warp 5 (MMA): holds the TMEM; one thread issues
//      S[g % 2] = Q K^T           (M=128, N=64, K=D; kind::f16, bf16 x bf16 -> fp32 in TMEM)
//      O       += P_hi V + P_lo V (M=128, N=D, K=64; V read as an MN-major operand)
//    with the QK^T of the next tile issued before the PV of this one, so the tensor core works
//    while the softmax warps run. Completion is signalled with tcgen05.commit on mbarriers. The
//    warp zeroes V rows past the split's end before their PV (0 x NaN would otherwise leak).
//    P is split into two bf16 terms (P_hi = bf16(p), P_lo = bf16(p - P_hi)), so the weights
//    enter the PV product with about 16 bits of precision instead of 8.
//  * warps 0-3 (softmax, one query vector per thread = one TMEM lane): stage the unit's Q tile
//    in the swizzled K-major layout, read each S tile from TMEM (tcgen05.ld), mask (split end,
//    causal row position, missing pages), run the online softmax in log2 units with the lazy
//    rescale (O is rescaled in TMEM only when a row's max grows by more than 2^8), write P into
//    shared memory in the swizzled K-major layout, and at the end move O from TMEM through
//    shared memory to coalesced global stores: the partial, or the normalised output when the
//    sequence has one split.
//  * Every wait is bounded. On timeout the kernel records NBX_DEV_TIMEOUT, waits (bounded) for
//    its MMAs and copies in flight, releases its TMEM and returns.
#include <atomic>
#include <cuda.h>
#include <cudaTypedefs.h>

#include "nbx_device.cuh"
#include "nbx_internal.h"

namespace nbx {
namespace {

constexpr int kMmaM = 128;       // query vectors per M tile (TMEM lanes)
constexpr int kMmaN = 64;        // positions per K/V tile
constexpr int kMmaThreads = 192;
constexpr int kSoftmaxThreads = 128;
constexpr float kMmaTau = 8.0f;  // lazy-rescale threshold, log2 units

template <int D>
struct MmaCfg {
  static constexpr int kStages = D <= 128 ? 4 : 2;
  static constexpr int kQBytes = kMmaM * D * 2;
  static constexpr int kTileBytes = kMmaN * D * 2;   // one K (or V) tile, bf16
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kPBytes = kMmaM * kMmaN * 2;  // one bf16 P term; the region holds P_hi, P_lo
  static constexpr int kQOff = 0;
  static constexpr int kStageOff = kQBytes;
  static constexpr int kPOff = kStageOff + kStages * kStageBytes;
  static constexpr int kBarOff = kPOff + 2 * kPBytes;
  static constexpr int kSmem = kBarOff + 256 + 1024;   // barriers + slack for 1024-byte alignment
  static constexpr uint32_t kTmemCols = D <= 128 ? 256 : 512;
  static constexpr uint32_t kOCol = 128;               // S buffers at columns 0 and 64, O from 128
  static_assert(kSmem <= 227 * 1024, "shared memory");
  static_assert(2 * kPBytes >= 2 * kMmaM * 32 * 4, "epilogue staging fits the P region");
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
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc ? 1u : 0u)
      : "memory");
}

// 16 consecutive 32-bit TMEM columns of this thread's lane
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
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

// Byte offset of (row, 16-byte chunk) in a 128-byte-swizzled operand block whose rows are 128
// bytes: 8-row groups of 1024 bytes, chunk index XOR (row mod 8).
__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t chunk) {
  return (row >> 3) * 1024u + (row & 7u) * 128u + ((chunk ^ (row & 7u)) << 4);
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

// Output row of query vector qi = r * group + g of KV head h, sequence b.
__device__ __forceinline__ int64_t out_row(const DecodeParams& p, int b, int h, int qi) {
  const int r = qi / p.group;
  const int g = qi - r * p.group;
  return (static_cast<int64_t>(b) * p.rows + r) * p.h_q + static_cast<int64_t>(h) * p.group + g;
}

template <int D>
__global__ void __launch_bounds__(kMmaThreads, 1)
    decode_partial_mma_kernel(DecodeParams p, const __grid_constant__ CUtensorMap k_map,
                              const __grid_constant__ CUtensorMap v_map) {
  using C = MmaCfg<D>;
  constexpr int NS = C::kStages;
  extern __shared__ __align__(1024) char smem_raw[];
  char* smem = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  char* q_s = smem + C::kQOff;
  char* stage_s = smem + C::kStageOff;
  char* p_s = smem + C::kPOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* kv_full = bars;              // [NS]  TMA bytes landed
  uint64_t* kv_empty = bars + NS;        // [NS]  PV of the stage done
  uint64_t* s_full = bars + 2 * NS;      // [2]   QK^T done
  uint64_t* s_empty = s_full + 2;        // [2]   S read by all softmax threads
  uint64_t* p_full = s_full + 4;         //       P written (and O rescaled)
  uint64_t* p_empty = s_full + 5;        //       PV done
  uint64_t* q_full = s_full + 6;         //       Q tile written
  uint64_t* q_empty = s_full + 7;        //       every MMA of the unit done
  uint64_t* done_bar = s_full + 8;       //       every MMA of the CTA done
  uint64_t* epi_bar = s_full + 9;        //       epilogue staging exchange
  volatile int* abort_flag = reinterpret_cast<int*>(s_full + 10);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_full + 11);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], kSoftmaxThreads);
    }
    mbar_init(p_full, kSoftmaxThreads);
    mbar_init(p_empty, 1);
    mbar_init(q_full, kSoftmaxThreads);
    mbar_init(q_empty, 1);
    mbar_init(done_bar, 1);
    mbar_init(epi_bar, kSoftmaxThreads);
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

  const int RG = p.rows * p.group;
  const int m_tiles = (RG + kMmaM - 1) / kMmaM;
  const int n_units = p.header[0] * p.h_kv * m_tiles;

  if (warp == 4) {
    // ======================================================== TMA producer (one thread)
    if (lane == 0) {
      bool ok = true;
      uint32_t g = 0;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const MmaUnit mu = mma_unit(p, u, m_tiles);
        const int32_t* bt = p.block_table + static_cast<int64_t>(mu.b) * p.max_pages;
        for (int t = 0; t < mu.tiles; ++t, ++g) {
          const int n0 = mu.start + t * kMmaN;
          const int page = bt[n0 / p.page_tokens];
          int row0 = -kMmaN;   // a missing page reads rows before the tensor: zeros
          if (page >= 0 && page < p.num_pages) {
            row0 = (page * p.h_kv + mu.h) * p.page_tokens + (n0 % p.page_tokens);
          } else {
            raise_status(p.status, NBX_DEV_BAD_PAGE);
          }
          const uint32_t st = g % NS;
          if (g >= static_cast<uint32_t>(NS) && !bwait(&kv_empty[st], ((g / NS) - 1) & 1u, abort_flag)) {
            ok = false;
            break;
          }
          char* kd = stage_s + st * C::kStageBytes;
          char* vd = kd + C::kTileBytes;
          mbar_arrive_expect_tx(&kv_full[st], C::kStageBytes);
#pragma unroll
          for (int a = 0; a < D / 64; ++a) {
            tma_load_2d(kd + a * (kMmaN * 128), &k_map, a * 64, row0, &kv_full[st]);
            tma_load_2d(vd + a * (kMmaN * 128), &v_map, a * 64, row0, &kv_full[st]);
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        raise_status(p.status, NBX_DEV_TIMEOUT);
      }
      // the copies issued last have landed before the CTA can exit
      for (uint32_t j = g > static_cast<uint32_t>(NS) ? g - NS : 0; j < g; ++j)
        mbar_wait(&kv_full[j % NS], (j / NS) & 1u, 100000000ull);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ======================================================== MMA issuer (one thread issues)
    constexpr uint32_t kIdescS = mma_idesc(kMmaM, kMmaN, false);
    constexpr uint32_t kIdescO = mma_idesc(kMmaM, D, true);
    const uint32_t q_addr = smem_u32(q_s);
    const uint32_t p_addr = smem_u32(p_s);
    bool ok = true;
    uint32_t g = 0, k = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++k) {
      const MmaUnit mu = mma_unit(p, u, m_tiles);
      if (!warp_wait(q_full, k & 1u, abort_flag)) {
        ok = false;
        break;
      }
      for (int t = -1; t < mu.tiles; ++t) {
        // S(g + t + 1) = Q K(g + t + 1)^T, one tile ahead of the PV
        if (t + 1 < mu.tiles) {
          const uint32_t gq = g + t + 1;
          const uint32_t st = gq % NS;
          if (!warp_wait(&kv_full[st], (gq / NS) & 1u, abort_flag) ||
              (gq >= 2 && !warp_wait(&s_empty[gq & 1u], ((gq >> 1) - 1) & 1u, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (lane == 0) {
            const uint32_t kb = smem_u32(stage_s + st * C::kStageBytes);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t a = kk >> 2, sub = kk & 3;
              const uint64_t ad = smem_desc(q_addr + a * (kMmaM * 128) + sub * 32, 16, 1024);
              const uint64_t bd = smem_desc(kb + a * (kMmaN * 128) + sub * 32, 16, 1024);
              tc_mma(tmem + (gq & 1u) * kMmaN, ad, bd, kIdescS, kk > 0);
            }
            tc_commit(&s_full[gq & 1u]);
          }
          __syncwarp();
        }
        if (t < 0) continue;
        // O += P(g + t) V(g + t)
        const uint32_t gp = g + t;
        const uint32_t st = gp % NS;
        if (!warp_wait(p_full, gp & 1u, abort_flag)) {
          ok = false;
          break;
        }
        char* vd = stage_s + st * C::kStageBytes + C::kTileBytes;
        const int valid = min(kMmaN, mu.end - (mu.start + t * kMmaN));
        if (valid < kMmaN) {
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
          for (int a = 0; a < D / 64; ++a)
            for (int i = lane; i < (kMmaN - valid) * 8; i += 32)
              *reinterpret_cast<uint4*>(vd + a * (kMmaN * 128) + (valid + (i >> 3)) * 128 + (i & 7) * 16) = z;
          fence_proxy_async();
        }
        __syncwarp();
        tc_fence_after();
        if (lane == 0) {
          const uint32_t vb = smem_u32(vd);
#pragma unroll
          for (int part = 0; part < 2; ++part) {
#pragma unroll
            for (int kk = 0; kk < kMmaN / 16; ++kk) {
              const uint64_t ad = smem_desc(p_addr + part * C::kPBytes + kk * 32, 16, 1024);
              const uint64_t bd = smem_desc(vb + kk * (16 * 128), kMmaN * 128, 1024);
              tc_mma(tmem + C::kOCol, ad, bd, kIdescO, !(t == 0 && part == 0 && kk == 0));
            }
          }
          tc_commit(p_empty);
          tc_commit(&kv_empty[st]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) tc_commit(q_empty);
      __syncwarp();
      g += mu.tiles;
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
    constexpr int kLanesPerRow = D / 8;            // 16-byte chunks per Q row
    constexpr int kRowsPerPass = 32 / kLanesPerRow;
    const int row = threadIdx.x;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    bool ok = true;
    uint32_t g = 0, k = 0, e = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++k) {
      const MmaUnit mu = mma_unit(p, u, m_tiles);
      const int q0 = mu.mt * kMmaM;
      const int qi = q0 + row;
      const bool row_ok = qi < RG;
      const int r = row_ok ? qi / p.group : 0;
      const int pos = mu.len - p.rows + r;   // last position this row sees
      // ---- Q tile: coalesced loads, swizzled K-major stores; rows past the last vector are zero
      if (k >= 1 && !warp_wait(q_empty, (k - 1) & 1u, abort_flag)) {
        ok = false;
        break;
      }
#pragma unroll 4
      for (int i = 0; i < 32 / kRowsPerPass; ++i) {
        const int rr = warp * 32 + i * kRowsPerPass + lane / kLanesPerRow;
        const int c = lane % kLanesPerRow;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (q0 + rr < RG)
          v = *reinterpret_cast<const uint4*>(static_cast<const char*>(p.q) + out_row(p, mu.b, mu.h, q0 + rr) * D * 2 +
                                              c * 16);
        *reinterpret_cast<uint4*>(q_s + (c >> 3) * (kMmaM * 128) + swz(rr, c & 7)) = v;
      }
      fence_proxy_async();
      mbar_arrive(q_full);

      const int32_t* bt = p.block_table + static_cast<int64_t>(mu.b) * p.max_pages;
      float m_run = -INFINITY, l_run = 0.f;
      for (int t = 0; t < mu.tiles; ++t, ++g) {
        const int n0 = mu.start + t * kMmaN;
        const int page = bt[n0 / p.page_tokens];
        const bool tile_ok = page >= 0 && page < p.num_pages;
        if (!warp_wait(&s_full[g & 1u], (g >> 1) & 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float sv[kMmaN];
#pragma unroll
        for (int c = 0; c < kMmaN / 16; ++c) tmem_ld16(lane_base + (g & 1u) * kMmaN + c * 16, sv + c * 16);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&s_empty[g & 1u]);
        // ---- mask and row max (log2 units; NaN propagates through the max)
        const int lim = min(mu.end - 1, pos) - n0;   // last visible column of this tile
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < kMmaN; ++j) {
          const bool valid = row_ok && tile_ok && j <= lim;
          sv[j] = valid ? sv[j] * p.qk_scale_log2 : -INFINITY;
          mx = max_nan(mx, sv[j]);
        }
        const bool grow = !(mx <= m_run + kMmaTau);
        const float m_new = grow ? mx : m_run;
        const float f = (m_new == m_run) ? 1.f : fast_exp2(m_run - m_new);
        // the previous PV has finished: P is free and O is stable
        if (g >= 1 && !warp_wait(p_empty, (g - 1) & 1u, abort_flag)) {
          ok = false;
          break;
        }
        if (t > 0 && __any_sync(0xffffffffu, f != 1.f)) {
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 16; ++c) {
            float ov[16];
            tmem_ld16(lane_base + C::kOCol + c * 16, ov);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) ov[i] *= f;
            tmem_st16(lane_base + C::kOCol + c * 16, ov);
          }
          tmem_wait_st();
        }
        m_run = m_new;
        l_run *= f;
        const float m_use = (m_run == -INFINITY) ? 0.f : m_run;   // all scores -inf: p = 0
        // ---- P = 2^(s - m) as bf16 P_hi + P_lo, rows of the swizzled K-major layout
        float lsum = 0.f;
#pragma unroll
        for (int c = 0; c < kMmaN / 8; ++c) {
          uint32_t wh[4], wl[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float p0 = fast_exp2(sv[c * 8 + 2 * i] - m_use);
            const float p1 = fast_exp2(sv[c * 8 + 2 * i + 1] - m_use);
            lsum += p0;
            lsum += p1;
            const __nv_bfloat162 hi = __floats2bfloat162_rn(p0, p1);
            const float2 hf = __bfloat1622float2(hi);
            const __nv_bfloat162 lo = __floats2bfloat162_rn(p0 - hf.x, p1 - hf.y);
            wh[i] = *reinterpret_cast<const uint32_t*>(&hi);
            wl[i] = *reinterpret_cast<const uint32_t*>(&lo);
          }
          *reinterpret_cast<uint4*>(p_s + swz(row, c)) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
          *reinterpret_cast<uint4*>(p_s + C::kPBytes + swz(row, c)) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
        }
        l_run += lsum;
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive(p_full);
      }
      if (!ok) break;
      // ---- epilogue: O from TMEM once the unit's last PV is done
      if (!warp_wait(p_empty, (g - 1) & 1u, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool single = mu.n_splits <= 1;
      const float sc = single ? ((m_run == -INFINITY) ? 0.f : p.v_scale / l_run) : 1.f;
      if (row_ok && !single) {
        const int64_t orow = out_row(p, mu.b, mu.h, qi);
        p.m_part[orow * p.max_splits + mu.s] = m_run;
        p.l_part[orow * p.max_splits + mu.s] = l_run;
      }
      // destination rows of the coalesced stores: this lane writes rows warp*32 + i*4 + lane/8
      float* dst[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int rr = q0 + warp * 32 + i * 4 + (lane >> 3);
        dst[i] = nullptr;
        if (rr < RG) {
          const int64_t orow = out_row(p, mu.b, mu.h, rr);
          dst[i] = single ? p.out + orow * D : p.acc_part + (orow * p.max_splits + mu.s) * D;
        }
      }
      // 32 columns at a time: TMEM -> registers -> staging [128][32] fp32 (16-byte chunks XOR row)
      // -> 128-byte row segments; two staging buffers in the P region
      for (int ch = 0; ch < D / 32; ++ch) {
        float ov[32];
        tmem_ld16(lane_base + C::kOCol + ch * 32, ov);
        tmem_ld16(lane_base + C::kOCol + ch * 32 + 16, ov + 16);
        tmem_wait_ld();
        float* buf = reinterpret_cast<float*>(p_s) + (ch & 1) * (kMmaM * 32);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4)
          *reinterpret_cast<float4*>(buf + row * 32 + ((c4 ^ (row & 7)) << 2)) =
              make_float4(ov[4 * c4] * sc, ov[4 * c4 + 1] * sc, ov[4 * c4 + 2] * sc, ov[4 * c4 + 3] * sc);
        mbar_arrive(epi_bar);
        if (!warp_wait(epi_bar, e & 1u, abort_flag)) {
          ok = false;
          break;
        }
        ++e;
        const int c4 = lane & 7;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int rr = warp * 32 + i * 4 + (lane >> 3);
          if (dst[i] != nullptr)
            *reinterpret_cast<float4*>(dst[i] + ch * 32 + c4 * 4) =
                *reinterpret_cast<const float4*>(buf + rr * 32 + ((c4 ^ (rr & 7)) << 2));
        }
      }
      if (!ok) break;
      tc_fence_before();
    }
    if (!ok) {
      *abort_flag = 1;
      if (threadIdx.x == 0) raise_status(p.status, NBX_DEV_TIMEOUT);
    }
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

// 2-D view of a bf16 pool: row (page * h_kv + h) * page_tokens + position, column d; boxes of
// 64 columns x 64 rows with 128-byte swizzle; reads outside the tensor return zeros.
bool make_pool_map(CUtensorMap* map, const void* pool, const DecodeParams& p) {
  const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.d),
                              static_cast<cuuint64_t>(p.num_pages) * p.h_kv * p.page_tokens};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.d) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kMmaN)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_mma(const DecodeParams& p, int grid_limit, cudaStream_t stream) {
  using C = MmaCfg<D>;
  static std::atomic<uint64_t> configured{0};   // devices whose shared-memory limit is raised
  CUtensorMap km, vm;
  if (!make_pool_map(&km, p.k_pool, p) || !make_pool_map(&vm, p.v_pool, p)) return cudaErrorInvalidValue;
  const DeviceInfo& di = device_info();
  const uint64_t bit = 1ull << (di.device & 63);
  if ((configured.load() & bit) == 0) {
    const cudaError_t e =
        cudaFuncSetAttribute(decode_partial_mma_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  const int m_tiles = (p.rows * p.group + kMmaM - 1) / kMmaM;
  const int64_t upper = static_cast<int64_t>(p.batch) * p.max_splits * p.h_kv * m_tiles;
  int64_t grid = di.sm_count;
  if (grid_limit > 0 && grid > grid_limit) grid = grid_limit;
  if (grid > upper) grid = upper;
  if (grid < 1) grid = 1;
  return launch_pdl(decode_partial_mma_kernel<D>, static_cast<unsigned>(grid), kMmaThreads, C::kSmem, stream, p, km,
                    vm);
}

}  // namespace

bool mma_path_applies(const DecodeParams& p, int q_dtype, int pool_dtype) {
  const int64_t pool_rows = static_cast<int64_t>(p.num_pages) * p.h_kv * p.page_tokens;
  return q_dtype == NBX_BF16 && pool_dtype == NBX_BF16 && (p.d == 128 || p.d == 256) &&
         (p.page_tokens % kMmaN) == 0 && p.rows * p.group >= 64 && pool_rows < (int64_t{1} << 31) - kMmaN;
}

cudaError_t decode_dispatch_mma(const DecodeParams& p, int grid_limit, cudaStream_t stream) {
  if (p.d == 128) return launch_mma<128>(p, grid_limit, stream);
  return launch_mma<256>(p, grid_limit, stream);
}

}  // namespace nbx
