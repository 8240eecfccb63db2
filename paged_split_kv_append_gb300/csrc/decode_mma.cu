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
// GB300 design (one CTA per SM, 8 warps):
//  * Work unit = (split entry, KV head, M tile), M tile fastest. The query vectors of one KV head,
//    v = row * G + head, are cut into M tiles of 128 (a tile may split one row's heads), so no tile
//    row is padding but in the last tile. Static round-robin over the plan's longest-first list.
//  * Shared memory: the unit's Q tile (128-byte-swizzled K-major atoms of 128 bytes a row), a K ring
//    and a V ring of 16 KB slots (64 positions x 128 bf16 columns: half of a d=256 tile, a whole
//    d=128 tile; or 64 positions x d E4M3 codes, a whole tile; a tile is one page or a 64-aligned
//    part of one). Every slot has a full barrier (TMA bytes) and an empty barrier (its consumer).
//  * warps 4 and 6 (producers) fill the K ring and the V ring with TMA (cp.async.bulk.tensor),
//    one thread issuing while the warp's lanes fetch block-table ids a chunk ahead. A page id
//    outside the pool loads rows before the tensor, which read as zeros; its positions are
//    masked. K halves free their slots at QK^T and V halves at PV, so the K stream runs ahead.
//  * TMEM (512 columns): three S/P buffers [0, 192), O [192, 192 + d). Three buffers let QK^T run
//    two tiles ahead of PV.
//  * Two issuing threads share the tensor pipe, each a plain sequence of bounded waits and MMAs
//    (fp32 accumulators in TMEM, completions signalled with tcgen05.commit):
//      warp 5:  S[x % 3] = Q K(x)^T   M=128, N=64, K=d; Q and K from shared memory; with a bf16
//               pool (kind::f16) its lanes 1-31 copy each unit's Q tile (a tensor box, or 16-byte
//               cp.async into the swizzled atoms, zeros past the last vector) once the previous
//               unit's last QK^T has completed
//      warp 7:  O += P_hi(y) V(y) + P_lo(y) V(y)   M=128, N=d (all V columns in one MMA), K=64;
//               P from TMEM. It zeroes V rows past a split's end before their PV (0 x NaN would
//               otherwise leak) and skips K steps that hold none.
//    Split between two threads, the per-tile control work of one overlaps the other's MMAs. With
//    a bf16 pool P enters the product as two bf16 terms, P_hi = p truncated to bf16 and
//    P_lo = (p - P_hi) truncated, so the weights keep 15 bits or more.
//  * An fp8 (E4M3) pool is read as it is stored: kind::f8f6f4 MMAs on the codes, K=32 a step. Q
//    enters as two E4M3 terms, Q_hi + Q_lo, of the query vector times a power of two 2^e that puts
//    its largest element in [128, 256): Q_hi holds 4 significant bits (rounded to nearest by a
//    Veltkamp split), Q_lo the rest, so a bf16 element of at least 2^-9 of the vector's largest
//    is exact and the others are off by at most 2^-16 of it; the softmax threads write them (one
//    query vector each) and fold 2^-e into their row's scale. P enters as P_hi + P_lo, the same
//    split of p: each p is off by at most 2^-9 p, plus 2^-9 when p < 2^-1 (E4M3 holds nothing
//    below 2^-9). The running max m moves up, to 5 below a tile's max, when that passes m + 8.75
//    (p stays below 448). A budget keeps the absolute parts within 2^-8 of the weight gathered:
//    a tile that could pass it has its small weights counted, and if they do pass it, m moves
//    down to 5 below the tile's max -- only while the weight gathered stays below 2^40 (past that
//    the tile, below 2^15, adds less than 2^-25 of the total). O and l are rescaled in TMEM
//    whenever m moves.
//  * warps 0-3 (softmax, one query vector per thread = one TMEM lane): read S from TMEM, mask
//    (split end, causal row position, missing pages), run the online softmax in log2 units with
//    the lazy rescale (O is rescaled in TMEM only when a row's max grows by more than 2^8; with an
//    fp8 pool as above), and write P_hi / P_lo over the S columns they came from, then, when m
//    moved, wait for the last PV into O and rescale it. After the unit's last PV each thread
//    stores its own row of O, 32 columns at a time, from registers with 32-byte stores -- the
//    partial, or the normalised output when the sequence has one split.
//  * Every wait is bounded. On timeout the kernel records NBX_DEV_TIMEOUT, waits (bounded) for
//    its copies and MMAs in flight, releases its TMEM and returns.
#include <atomic>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "nbx_device.cuh"
#include "nbx_internal.h"
#include "nbx_tcgen05.cuh"

namespace nbx {
namespace {

constexpr int kMmaM = 128;       // TMEM lanes / rows of an M tile
static_assert(kMmaM == kMmaRowsPerTile, "the plan's M tiles");
constexpr int kMmaN = 64;        // positions per K/V tile
constexpr int kMmaThreads = 256;
constexpr int kSoftmaxThreads = 128;
constexpr float kMmaTau = 8.0f;  // lazy-rescale threshold, log2 units
constexpr int kChunk = 32;       // output columns per epilogue step
constexpr int kSBufs = 3;        // S/P buffers in TMEM
constexpr int kSlotBytes = 16384;  // ring slot: 64 positions x 128 columns bf16, or x d E4M3 codes
constexpr int kAtomBytes = kMmaN * 128;   // one 128-byte-wide swizzle column of a 64-position tile
// fp8 pools: the running max sits kF8Mid below a tile's max after a move; it moves up when a
// tile's max passes m + kF8Hi (p <= 2^8.75 = 430, below 448, the largest E4M3), down only while
// the gathered weight stays <= 2^40
constexpr float kF8Hi = 8.75f, kF8Mid = 5.f, kF8MaxWeight = 1099511627776.f;

template <int D, bool F8>
struct MmaCfg {
  static constexpr int kHalves = F8 ? 1 : D / 128;         // ring slots per K (or V) tile
  static constexpr int kKSlots = D <= 128 ? 5 : 4;         // K ring
  static constexpr int kVSlots = kKSlots;                  // V ring
  static constexpr int kQBytes = kMmaM * D * 2;            // Q tile (bf16, or E4M3 Q_hi and Q_lo): atoms of 16 KB
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQBytes;
  static constexpr int kVOff = kKOff + kKSlots * kSlotBytes;
  static constexpr int kBarOff = kVOff + kVSlots * kSlotBytes;
  static constexpr int kSmem = kBarOff + 512 + 1024;   // barriers + slack for 1024-byte alignment
  // TMEM columns: S/P buffers [0, 192), O [192, 192 + D)
  static constexpr uint32_t kOCol = kSBufs * kMmaN;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kOCol + D <= kTmemCols, "TMEM");
  static_assert(kSmem <= 227 * 1024, "shared memory");
  static_assert((2 * (kKSlots + kVSlots) + 3 * kSBufs + 7) * 8 <= 512, "barrier area");
  // one PV MMA spans both V halves of a tile: their slots must be adjacent (even ordinals)
  static_assert(kHalves == 1 || (kVSlots % kHalves) == 0, "V ring length");
};

// Query rows per M tile when every tile holds whole rows (one tile, or a group dividing 128: the Q
// tile is then one tensor box of the rows), else 0 (tiles split a row's heads; Q is copied by lanes).
__host__ __device__ inline int whole_row_tile_rows(int rows, int group) {
  if (rows * group <= kMmaM) return rows;
  return (kMmaM % group) == 0 ? kMmaM / group : 0;
}

struct MmaMaps {
  CUtensorMap k, v;   // 2-D pool views [num_pages * h_kv * page_tokens][d], box 64 x 64
  CUtensorMap q;      // 4-D [batch][rows][h_q][d] bf16, box {64, G, rows per tile, 1} (whole-row tiles)
};

// Bounded wait that also gives up when another role of the CTA has given up.
// limit_ns: kWaitLimitNs (2 s), or DecodeParams::wait_limit_ns in the instantiation a test of the
// timeout path runs (a bound read at run time cost the fp8 window 8 us a call, so the kernels of
// normal calls keep the constant).
__device__ __forceinline__ bool bwait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if ((i & 3u) == 0u && global_timer_ns() - t0 > limit_ns) return false;
  }
}

// The same, with one answer for the whole warp (the tcgen05 .sync.aligned forms that follow need
// every lane).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t limit_ns) {
  return __all_sync(0xffffffffu, bwait(bar, parity, abort_flag, limit_ns));
}

struct MmaUnit {
  int b, s, h, mt, start, end, len, n_splits, tiles;
};

__device__ __forceinline__ MmaUnit unit_from(const Entry& en, int u, int span, int m_tiles) {
  MmaUnit m;
  const int rem = u - (u / span) * span;
  m.h = rem / m_tiles;
  m.mt = rem - m.h * m_tiles;
  m.b = en.b;
  m.s = en.s;
  m.start = en.start;
  m.end = en.end;
  m.len = en.len;
  m.n_splits = en.n_splits;
  m.tiles = (en.end - en.start + kMmaN - 1) / kMmaN;
  return m;
}

// Walks this CTA's tiles in order: units blockIdx.x, blockIdx.x + gridDim.x, ..., tiles of each.
// Ring ordinals: tile tt of the current unit fills slots kbase + tt * hh .. + hh - 1 of the K ring
// (and the same ordinals of the V ring). The next unit's work-list entry is loaded one unit ahead.
struct TileIter {
  int u;             // unit index
  uint32_t k;        // unit ordinal within this CTA
  int t;             // tile within the unit
  uint32_t x;        // tile ordinal within this CTA
  bool done;
  bool has_next;     // another unit follows in this CTA
  int span;          // units per work-list entry
  int m_tiles, n_units, hh;
  uint32_t kbase;
  MmaUnit mu;
  Entry nx;
  __device__ __forceinline__ void prefetch(const DecodeParams& p) {
    const int u2 = u + static_cast<int>(gridDim.x);
    has_next = u2 < n_units;
    if (has_next) nx = p.entries[u2 / span];
  }
  __device__ __forceinline__ void begin(const DecodeParams& p, int m_tiles_, int n_units_, int hh_) {
    m_tiles = m_tiles_;
    n_units = n_units_;
    hh = hh_;
    span = p.h_kv * m_tiles;
    u = blockIdx.x;
    k = 0;
    t = 0;
    x = 0;
    kbase = 0;
    has_next = false;
    done = u >= n_units;
    if (!done) {
      mu = unit_from(p.entries[u / span], u, span, m_tiles);
      prefetch(p);
    }
  }
  __device__ __forceinline__ uint32_t item(int tt) const { return kbase + tt * hh; }
  __device__ __forceinline__ MmaUnit next_mu() const {
    return unit_from(nx, u + static_cast<int>(gridDim.x), span, m_tiles);
  }
  __device__ __forceinline__ void next_unit(const DecodeParams& p) {
    kbase += mu.tiles * hh;
    t = 0;
    ++k;
    u += gridDim.x;
    done = u >= n_units;
    if (!done) {
      mu = unit_from(nx, u, span, m_tiles);
      prefetch(p);
    }
  }
  __device__ __forceinline__ void next_tile(const DecodeParams& p) {
    ++x;
    if (++t >= mu.tiles) next_unit(p);
  }
};

// Page id of tile 32 * chunk + lane of a unit (0 past the unit's last tile): one warp fetches the
// block table 32 tiles at a time.
__device__ __forceinline__ int chunk_pages(const DecodeParams& p, const MmaUnit& mu, int chunk, int lane) {
  const int t = chunk * 32 + lane;
  return t < mu.tiles ? p.block_table[static_cast<int64_t>(mu.b) * p.max_pages + (mu.start + t * kMmaN) / p.page_tokens]
                      : 0;
}

// First pool row of the tile at position n0 in page `page`, or -kMmaN (rows before the tensor,
// read as zeros) if the page id is outside the pool.
__device__ __forceinline__ int tile_row(const DecodeParams& p, const MmaUnit& mu, int n0, int page, bool report) {
  if (page < 0 || page >= p.num_pages) {
    if (report) raise_status(p.status, NBX_DEV_BAD_PAGE);
    return -kMmaN;
  }
  return (page * p.h_kv + mu.h) * p.page_tokens + (n0 % p.page_tokens);
}

// Block-table ids of one warp's tile stream: lane l holds the page of tile 32c + l of the current
// chunk, and the following chunk is loaded one chunk ahead (of this unit, or the next unit's
// first), so no page-id load sits between two copies.
struct PageStream {
  int cur, nxt;
  __device__ __forceinline__ static int following(const DecodeParams& p, const TileIter& it, int c, int lane) {
    if ((c + 1) * 32 < it.mu.tiles) return chunk_pages(p, it.mu, c + 1, lane);
    return it.has_next ? chunk_pages(p, it.next_mu(), 0, lane) : 0;
  }
  __device__ __forceinline__ void start(const DecodeParams& p, const TileIter& it, int lane) {
    cur = chunk_pages(p, it.mu, 0, lane);
    nxt = following(p, it, 0, lane);
  }
  // the iterator has just moved onto a tile t with t % 32 == 0 (a new unit's first tile included)
  __device__ __forceinline__ void advance(const DecodeParams& p, const TileIter& it, int lane) {
    cur = nxt;
    nxt = following(p, it, it.t >> 5, lane);
  }
  __device__ __forceinline__ int page(int t) const { return __shfl_sync(0xffffffffu, cur, t & 31); }
};

// Two floats to two E4M3 codes, rounded to nearest (saturating; NaN stays NaN), a in the low byte.
__device__ __forceinline__ uint32_t e4m3x2_rn(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

// x = hi + lo exactly, hi = x rounded to nearest with 4 significant bits (Veltkamp's splitting with
// the factor 2^20 + 1 on 24-bit significands; no operation may be fused or reordered, hence the _rn
// intrinsics). x of an E4M3 term: |x| <= 2^8, far from overflow.
__device__ __forceinline__ void split4(float x, float& hi, float& lo) {
  const float c = __fmul_rn(x, 1048577.0f);
  hi = __fsub_rn(c, __fsub_rn(c, x));
  lo = __fsub_rn(x, hi);
}

// Four weights (positions 4i .. 4i + 3 of a tile) as the E4M3 terms P_hi and P_lo, four codes a word.
__device__ __forceinline__ void p_terms4(const float* pv, uint32_t& wh, uint32_t& wl) {
  float h[4], l[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) split4(pv[q], h[q], l[q]);
  wh = e4m3x2_rn(h[0], h[1]) | (e4m3x2_rn(h[2], h[3]) << 16);
  wl = e4m3x2_rn(l[0], l[1]) | (e4m3x2_rn(l[2], l[3]) << 16);
}

// fp8 pools: this thread's query vector of unit `mu` as the terms Q_hi and Q_lo (E4M3) of the
// vector times 2^e, its largest |element| brought into [128, 256), written into row `row` of the
// Q tile's 128-byte-swizzled K-major atoms: Q_hi atoms first, then Q_lo. Rows past the last vector
// are zero; a vector holding NaN or infinity gets NaN codes. Returns 2^-e, which the row's scores
// take back.
template <int D>
__device__ __forceinline__ float q_to_e4m3_terms(const DecodeParams& p, const MmaUnit& mu, int row, char* q_s) {
  const int G = p.group;
  const int vq = mu.mt * kMmaM + row;
  const bool ok = vq < p.rows * G;
  const int r = ok ? vq / G : 0, gq = ok ? vq - r * G : 0;
  const uint4* src = reinterpret_cast<const uint4*>(
      static_cast<const char*>(p.q) +
      (((static_cast<int64_t>(mu.b) * p.rows + r) * p.h_q) + static_cast<int64_t>(mu.h) * G + gq) * (D * 2));
  float amax = 0.f;
  if (ok) {
#pragma unroll 4
    for (int c = 0; c < D / 8; ++c) {
      const uint4 v = __ldg(src + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = bf16x2_to_float2(w[i]);
        amax = max_nan(amax, max_nan(fabsf(f.x), fabsf(f.y)));
      }
    }
  }
  const bool bad = !(amax <= 3.402823466e38f);   // NaN or infinity in the vector
  int e = 0;
  if (!bad && amax > 0.f) {
    const int ex = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 127;   // floor(log2 amax), normal amax
    e = min(120, max(-120, 7 - ex));
  }
  const float sc = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);   // 2^e
  char* row_hi = q_s + row * 128;
  char* row_lo = q_s + (D / 128) * (kMmaM * 128) + row * 128;
#pragma unroll 2
  for (int c = 0; c < D / 16; ++c) {   // 16 elements: one 16-byte chunk of each term
    uint4 ph = make_uint4(0u, 0u, 0u, 0u), pl = ph;
    if (ok) {
      const uint4 v0 = __ldg(src + 2 * c), v1 = __ldg(src + 2 * c + 1);
      const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 a = bf16x2_to_float2(w[2 * i]), b = bf16x2_to_float2(w[2 * i + 1]);
        const float x[4] = {__fmul_rn(a.x, sc), __fmul_rn(a.y, sc), __fmul_rn(b.x, sc), __fmul_rn(b.y, sc)};
        p_terms4(x, hw[i], lw[i]);
      }
      ph = bad ? make_uint4(0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu) : make_uint4(hw[0], hw[1], hw[2], hw[3]);
      pl = bad ? make_uint4(0u, 0u, 0u, 0u) : make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
    const int a = c >> 3, cc = c & 7;   // 128-byte atom and its 16-byte chunk
    const int off = a * (kMmaM * 128) + ((cc ^ (row & 7)) << 4);
    *reinterpret_cast<uint4*>(row_hi + off) = ph;
    *reinterpret_cast<uint4*>(row_lo + off) = pl;
  }
  return __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
}

// F8: the pools hold E4M3 codes, read as they are by kind::f8f6f4 MMAs (Q and P as two E4M3 terms
// each); otherwise bf16 pools and kind::f16 MMAs (P as two bf16 terms). TW: a test of the timeout
// path (nbx_set_decode_wait_test): the waits take DecodeParams::wait_limit_ns and the producers
// start after DecodeParams::producer_delay_ns.
template <int D, bool F8, bool TW>
__global__ void __launch_bounds__(kMmaThreads, 1)
    decode_partial_mma_kernel(DecodeParams p, const __grid_constant__ MmaMaps maps) {
  using C = MmaCfg<D, F8>;
  constexpr int NK = C::kKSlots;
  constexpr int NV = C::kVSlots;
  constexpr int HI = C::kHalves;
  extern __shared__ __align__(1024) char smem_raw[];
  char* smem = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  char* q_s = smem + C::kQOff;
  char* kring = smem + C::kKOff;
  char* vring = smem + C::kVOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* kfull = bars;              // [NK]  the K slot's half landed (TMA bytes)
  uint64_t* kempty = kfull + NK;       // [NK]  the K slot's half consumed (its QK^T done)
  uint64_t* vfull = kempty + NK;       // [NV]  the V slot's half landed
  uint64_t* vempty = vfull + NV;       // [NV]  the V slot's half consumed (its PV done)
  uint64_t* s_full = vempty + NV;      // [3]   S of the buffer's tile in TMEM
  uint64_t* p_full = s_full + kSBufs;  // [3]   P of the buffer's tile in TMEM (128 arrivals)
  uint64_t* sp_free = p_full + kSBufs; // [3]   PV of the buffer's tile done: buffer reusable, O
                                       //       holds every PV up to that tile
  uint64_t* q_full = sp_free + kSBufs; //       the unit's Q tile landed (the QK warp's lanes 1-31)
  uint64_t* q_empty = q_full + 1;      //       every QK^T of the unit done
  uint64_t* o_free = q_full + 2;       //       O read out by the epilogue (128 arrivals)
  uint64_t* done_bar = q_full + 3;     //       every PV of the CTA done
  uint64_t* done_qk = q_full + 4;      //       every QK^T of the CTA done
  volatile int* abort_flag = reinterpret_cast<int*>(q_full + 5);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_full + 6);
  // Phase discipline: a thread waits on phase j of a barrier only once it knows phase j - 1 has
  // completed and while phase j + 1 cannot have (a parity wait cannot tell them apart). Each
  // issuer consumes its ring slots in order, so it tests a slot's half only after the half a ring
  // length earlier was consumed by itself. With three S/P buffers, QK(x) waits for PV(x - 3),
  // whose successor on that buffer, PV(x), needs QK(x) first; PV(y) waits for P(y), whose
  // successor P(y + 3) needs QK(y + 3) and so PV(y). The softmax threads track PV completion
  // through sp_free[y % 3]: once S(g) has landed, PV(g - 3) is known complete, so PV(g - 1) is
  // exactly one phase ahead on its buffer.

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NK; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&kempty[i], 1);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(&vfull[i], 1);
      mbar_init(&vempty[i], 1);
    }
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], kSoftmaxThreads);
      mbar_init(&sp_free[i], 1);
    }
    // the E4M3 terms of the 128 softmax threads, a tensor box (one arrival with the byte count), or
    // the cp.async completions of lanes 1-31
    mbar_init(q_full, F8 ? kSoftmaxThreads : (whole_row_tile_rows(p.rows, p.group) > 0 ? 1 : 31));
    mbar_init(q_empty, 1);
    mbar_init(o_free, kSoftmaxThreads);
    mbar_init(done_bar, 1);
    mbar_init(done_qk, 1);
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
  const uint64_t wlim = TW ? p.wait_limit_ns : kWaitLimitNs;
  pdl_wait();   // the plan kernel's work list and the append's positions are visible from here on
  pdl_launch_dependents();

  const int G = p.group;
  const int RG = p.rows * G;                             // query vectors of one KV head
  const int m_tiles = (RG + kMmaM - 1) / kMmaM;          // M tiles of 128 of them
  const int n_units = p.header[0] * p.h_kv * m_tiles;

  if (warp == 4 || warp == 6) {
    // ======================================================== TMA producers, one warp per ring:
    // warp 4 fills the K ring, warp 6 the V ring, each in tile order. Lane 0 waits and issues;
    // the warp's lanes fetch the block table a chunk ahead.
    const bool is_k = warp == 4;
    const int NR = is_k ? NK : NV;
    char* rbase = is_k ? kring : vring;
    uint64_t* rfull = is_k ? kfull : vfull;
    uint64_t* rempty = is_k ? kempty : vempty;
    const CUtensorMap* map = is_k ? &maps.k : &maps.v;
    if (TW && p.producer_delay_ns) {   // a test holds the producers back so that the other roles' waits run out
      const uint64_t t0 = global_timer_ns();
      while (global_timer_ns() - t0 < p.producer_delay_ns) __nanosleep(10000);
    }
    bool ok = true;
    uint32_t i = 0;   // ring ordinal
    TileIter it;
    it.begin(p, m_tiles, n_units, HI);
    PageStream ps;
    if (!it.done) ps.start(p, it, lane);
    while (!it.done && ok) {
      const int t = it.t;
      const int row0 = tile_row(p, it.mu, it.mu.start + t * kMmaN, ps.page(t), lane == 0 && is_k);
      for (int j = 0; j < HI; ++j, ++i) {
        int r = 1;
        if (lane == 0 && i >= static_cast<uint32_t>(NR)) r = bwait(&rempty[i % NR], (i / NR - 1) & 1u, abort_flag, wlim);
        if (!__shfl_sync(0xffffffffu, r, 0)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          char* dst = rbase + (i % NR) * kSlotBytes;
          if constexpr (F8) {   // the tile's D codes a position, 128 a box
            mbar_arrive_expect_tx(&rfull[i % NR], kMmaN * D);
#pragma unroll
            for (int a = 0; a < D / 128; ++a) tma_load_2d(dst + a * kAtomBytes, map, a * 128, row0, &rfull[i % NR]);
          } else {              // 128 bf16 columns of the tile, 64 a box
            mbar_arrive_expect_tx(&rfull[i % NR], kSlotBytes);
            tma_load_2d(dst, map, (2 * j) * 64, row0, &rfull[i % NR]);
            tma_load_2d(dst + kAtomBytes, map, (2 * j + 1) * 64, row0, &rfull[i % NR]);
          }
        }
      }
      if (!ok) break;
      it.next_tile(p);
      if (!it.done && (it.t & 31) == 0) ps.advance(p, it, lane);
    }
    if (lane == 0) {
      if (!ok) {
        *abort_flag = 1;
        raise_status(p.status, NBX_DEV_TIMEOUT);
      }
      // the copies issued last have landed before the CTA can exit
      for (uint32_t j = i > static_cast<uint32_t>(NR) ? i - NR : 0; j < i; ++j)
        mbar_wait(&rfull[j % NR], (j / NR) & 1u, 100000000ull);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ======================================================== QK^T issuer (lane 0), Q loader (lanes 1-31)
    const uint32_t q_addr = smem_u32(q_s);
    TileIter it;
    it.begin(p, m_tiles, n_units, HI);
    if (lane == 0) {
      constexpr uint32_t kIdescS = mma_idesc(kMmaM, kMmaN, false, F8);   // bf16, or E4M3 (format 0)
      bool ok = true;
      uint32_t sx = 0, sxp = 0;   // S/P buffer (x % 3) and its phase count (x / 3)
      while (!it.done) {
        // S(x) = Q K(x)^T once the buffer's previous PV is done, K(x) has landed and the unit's Q has
        const uint32_t ki = it.item(it.t);
        if (it.x >= static_cast<uint32_t>(kSBufs)) ok = bwait(&sp_free[sx], (sxp - 1) & 1u, abort_flag, wlim);
        for (int j = 0; j < HI && ok; ++j) ok = bwait(&kfull[(ki + j) % NK], ((ki + j) / NK) & 1u, abort_flag, wlim);
        if (ok && it.t == 0) ok = bwait(q_full, it.k & 1u, abort_flag, wlim);
        if (!ok) break;
        tc_fence_after();
        if (it.t == 0) fence_proxy_async();   // Q was written by cp.async or st.shared (generic proxy)
        if constexpr (F8) {
          // S = Q_hi K^T + Q_lo K^T, 32 codes of d a step: 128-byte atoms of Q and of the K slot
          const uint32_t kb = smem_u32(kring + (ki % NK) * kSlotBytes);
#pragma unroll
          for (int term = 0; term < 2; ++term)
#pragma unroll
            for (int kk = 0; kk < D / 32; ++kk) {
              const uint32_t a = kk >> 2, sub = kk & 3;
              const uint64_t ad = smem_desc(q_addr + (term * (D / 128) + a) * (kMmaM * 128) + sub * 32, 16, 1024);
              const uint64_t bd = smem_desc(kb + a * kAtomBytes + sub * 32, 16, 1024);
              tc_mma_ss_f8(tmem + sx * kMmaN, ad, bd, kIdescS, term > 0 || kk > 0);
            }
        } else {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t a = kk >> 2, sub = kk & 3;   // 64-column atom, 16-column step in it
            const uint64_t ad = smem_desc(q_addr + a * (kMmaM * 128) + sub * 32, 16, 1024);
            const uint32_t kb = smem_u32(kring + ((ki + (a >> 1)) % NK) * kSlotBytes) + (a & 1) * kAtomBytes;
            const uint64_t bd = smem_desc(kb + sub * 32, 16, 1024);
            tc_mma_ss(tmem + sx * kMmaN, ad, bd, kIdescS, kk > 0);
          }
        }
        tc_commit(&s_full[sx]);
        for (int j = 0; j < HI; ++j) tc_commit(&kempty[(ki + j) % NK]);
        if (it.t == it.mu.tiles - 1) tc_commit(q_empty);
        if (++sx == kSBufs) {
          sx = 0;
          ++sxp;
        }
        it.next_tile(p);
      }
      if (!ok) {
        *abort_flag = 1;
        raise_status(p.status, NBX_DEV_TIMEOUT);
      }
      // every QK^T of this CTA has completed before the TMEM is released
      tc_commit(done_qk);
      mbar_wait(done_qk, 0, 100000000ull);
    } else if constexpr (!F8) {   // (with an fp8 pool the softmax threads write Q)
      // Each unit's Q tile, once every QK^T of the previous unit has completed: vector i of the tile
      // (v = 128 mt + i, row v / G, head v % G of the KV head) into row i of the 128-byte-swizzled
      // K-major atoms, 16 bytes a copy; rows past the last vector are zero. These 31 lanes run apart
      // from lane 0's MMA loop, meeting it only through the barriers.
      constexpr unsigned kLoaders = 0xfffffffeu;
      constexpr int kRowChunks = D / 8;   // 16-byte chunks per query vector
      const int rt_box = whole_row_tile_rows(p.rows, G);   // > 0: the tile is one tensor box
      bool ok = true;
      for (uint32_t k = 0; !it.done; ++k) {
        int r = 1;
        if (lane == 1 && k > 0) r = bwait(q_empty, (k - 1) & 1u, abort_flag, wlim);
        if (!__shfl_sync(kLoaders, r, 1)) {
          ok = false;
          break;
        }
        if (rt_box > 0) {   // whole rows: lane 1 loads the tile's rows as one box per 64-column atom
          if (lane == 1) {
            mbar_arrive_expect_tx(q_full, static_cast<uint32_t>((D / 64) * 64 * G * rt_box * 2));
#pragma unroll
            for (int a = 0; a < D / 64; ++a)
              tma_load_4d(q_s + a * (kMmaM * 128), &maps.q, a * 64, it.mu.h * G, it.mu.mt * rt_box, it.mu.b, q_full);
          }
          it.next_unit(p);
          continue;
        }
        // lane l copies chunks l - 1, l + 30, ... of the tile: (vector i, chunk cc) and the vector's
        // row and head, stepped without divisions
        const int v0 = it.mu.mt * kMmaM;
        int i = (lane - 1) / kRowChunks, cc = (lane - 1) % kRowChunks;
        int v = v0 + i;
        int rr = v / G, gg = v - rr * G;
        const char* qb = static_cast<const char*>(p.q) +
                         (static_cast<int64_t>(it.mu.b) * p.rows * p.h_q + static_cast<int64_t>(it.mu.h) * G) * (D * 2);
        const int64_t row_stride = static_cast<int64_t>(p.h_q) * (D * 2);
        while (i < kMmaM) {
          const bool vq = v < RG;
          const char* src = qb + rr * row_stride + gg * (D * 2) + cc * 16;
          cp_async16_zfill(q_addr + (cc >> 3) * (kMmaM * 128) + i * 128 + (((cc & 7) ^ (i & 7)) << 4), vq ? src : qb, vq);
          cc += 31;
          while (cc >= kRowChunks) {
            cc -= kRowChunks;
            ++i;
            ++v;
            if (++gg == G) {
              gg = 0;
              ++rr;
            }
          }
        }
        cp_async_arrive_noinc(q_full);
        it.next_unit(p);
      }
      cp_async_wait_all();   // this lane's Q copies have landed before the CTA exits
      if (!ok && lane == 1) *abort_flag = 1;
    }
    __syncwarp();
  } else if (warp == 7) {
    // ======================================================== PV issuer (lane 0)
    if (lane == 0) {
      // one MMA covers every output column: the two V halves of a d = 256 tile sit in adjacent
      // ring slots (even ring ordinals, an even ring length), so their four 64-column atoms are
      // 8 KB apart throughout
      constexpr uint32_t kIdescO = mma_idesc(kMmaM, D, true, F8);   // bf16, or E4M3 (format 0)
      constexpr int kStep = F8 ? 32 : 16;                           // positions of one MMA's K
      TileIter it;
      it.begin(p, m_tiles, n_units, HI);
      bool ok = true;
      uint32_t sy = 0, syp = 0;   // S/P buffer (y % 3) and its phase count (y / 3)
      while (!it.done) {
        // O += P(y) V(y): P written, V landed, O read out by the previous unit's epilogue
        const uint32_t vi = it.item(it.t);
        ok = bwait(&p_full[sy], syp & 1u, abort_flag, wlim);
        if (ok && it.t == 0 && it.k > 0) ok = bwait(o_free, (it.k - 1) & 1u, abort_flag, wlim);
        for (int j = 0; j < HI && ok; ++j) ok = bwait(&vfull[(vi + j) % NV], ((vi + j) / NV) & 1u, abort_flag, wlim);
        if (!ok) break;
        const int valid = min(kMmaN, it.mu.end - (it.mu.start + it.t * kMmaN));
        const int ksteps = (valid + kStep - 1) / kStep;
        char* vd = vring + (vi % NV) * kSlotBytes;
        if (valid % kStep) {   // V rows past the split's end inside the last K step: zeros
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
          for (int at = 0; at < (F8 ? D / 128 : 2 * HI); ++at)
            for (int rr = valid; rr < ksteps * kStep; ++rr)
              for (int e = 0; e < 8; ++e) *reinterpret_cast<uint4*>(vd + at * kAtomBytes + rr * 128 + e * 16) = z;
          fence_proxy_async();
        }
        tc_fence_after();
        const uint32_t pcol = tmem + sy * kMmaN;
        const uint32_t vb = smem_u32(vd);
        // P_hi, then P_lo: K steps of kStep positions, 8 TMEM columns each (two bf16 or four E4M3
        // codes a column); the V atoms of one tile are kAtomBytes apart throughout
#pragma unroll
        for (int part = 0; part < 2; ++part) {
#pragma unroll
          for (int kk = 0; kk < kMmaN / kStep; ++kk) {
            if (kk < ksteps) {
              const uint32_t acol = pcol + part * (F8 ? kMmaN / 4 : kMmaN / 2) + kk * 8;
              const uint64_t bd = smem_desc(vb + kk * (kStep * 128), kAtomBytes, 1024);
              const bool acc = !(it.t == 0 && part == 0 && kk == 0);
              if constexpr (F8) tc_mma_ts_f8(tmem + C::kOCol, acol, bd, kIdescO, acc);
              else tc_mma_ts(tmem + C::kOCol, acol, bd, kIdescO, acc);
            }
          }
        }
        for (int j = 0; j < HI; ++j) tc_commit(&vempty[(vi + j) % NV]);
        tc_commit(&sp_free[sy]);
        if (++sy == kSBufs) {
          sy = 0;
          ++syp;
        }
        it.next_tile(p);
      }
      if (!ok) {
        *abort_flag = 1;
        raise_status(p.status, NBX_DEV_TIMEOUT);
      }
      // every PV of this CTA has completed before the TMEM is released
      tc_commit(done_bar);
      mbar_wait(done_bar, 0, 100000000ull);
    }
    __syncwarp();
  } else {
    // ======================================================== softmax warps (row = threadIdx.x)
    const int row = threadIdx.x;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    // the split partials stay in L2 for the merge
    const uint64_t keep = l2_keep_policy(p.keep_frac);
    bool ok = true;
    uint32_t g = 0;              // tile ordinal
    uint32_t gb = 0, gp = 0;     // S/P buffer (g % 3) and its phase count (g / 3)
    TileIter it;
    it.begin(p, m_tiles, n_units, HI);
    int pg_cur = it.done ? 0 : chunk_pages(p, it.mu, 0, lane), pg_nxt = 0;   // lane l: page of tile 32c + l
    float q_inv = 1.f;   // fp8 pools: 2^-e of this thread's query vector in the unit's Q terms
    if constexpr (F8) {
      if (!it.done) {
        q_inv = q_to_e4m3_terms<D>(p, it.mu, row, q_s);
        fence_proxy_async();   // the terms are read by the tensor pipe (async proxy)
        mbar_arrive(q_full);
      }
    }
    while (!it.done && ok) {
      const MmaUnit mu = it.mu;
      const int vq = mu.mt * kMmaM + row;            // this thread's query vector of the KV head
      const bool row_ok = vq < RG;
      const int r = row_ok ? vq / G : 0;             // its query row
      const int gq = row_ok ? vq - r * G : 0;        // its query head within the KV head's group
      const int pos = mu.len - p.rows + r;   // last position this row sees
      // Fixed shift (maxdiffusion PR #477, "fixed-m"), when the caller passes score bounds: a row
      // whose bound U >= |z| (log2 units, Cauchy-Schwarz: |q| max|k| scale log2 e) passes the gate
      // floor((C + 125) / 2), C = 127 - ceil(log2 n) - ceil(log2 256) for the split's n keys, with
      // every |v| <= 256, takes its weights as 2^(z - m) with m = ceil(U) - C fixed before the split is
      // read: no running max, no rescale, and no term overflows or falls below 2^-125. Other rows keep
      // the online max. P in E4M3 (an fp8 pool) cannot hold 2^C: that path is never fixed.
      bool fixed = false;
      float m_fix = 0.f;
      if (!F8 && p.fs_kv_max != nullptr && row_ok) {
        const int64_t orow = (static_cast<int64_t>(mu.b) * p.rows + r) * p.h_q + static_cast<int64_t>(mu.h) * G + gq;
        const float2 kv = *reinterpret_cast<const float2*>(p.fs_kv_max + 2 * (static_cast<int64_t>(mu.b) * p.h_kv + mu.h));
        const float U = p.fs_q_norm[orow] * kv.x * p.fs_scale_log2;
        const int n_keys = max(mu.end - mu.start, 1);
        const int Cn = 127 - (32 - __clz(n_keys - 1)) - 8;   // ceil(log2 n), ceil(log2 256) = 8
        fixed = U <= static_cast<float>((Cn + 125) / 2) && kv.y <= 256.f;   // false for NaN bounds
        m_fix = ceilf(U) - static_cast<float>(Cn);
      }
      float m_run = fixed ? m_fix : -INFINITY, l_run = 0.f;
      float e_run = 0.f;   // fp8 pools: bound on the terms' absolute floor errors so far (same scale as l)
      uint32_t pb = 0, pp = 0;   // buffer and phase count of the previous tile (g - 1)
      for (int t = 0; t < mu.tiles; ++t) {
        const int n0 = mu.start + t * kMmaN;
        if ((t & 31) == 0 && t + 32 < mu.tiles) pg_nxt = chunk_pages(p, mu, (t >> 5) + 1, lane);
        const int page = __shfl_sync(0xffffffffu, pg_cur, t & 31);
        if ((t & 31) == 31) pg_cur = pg_nxt;
        const bool tile_ok = page >= 0 && page < p.num_pages;
        const uint32_t sbuf = tmem + gb * kMmaN;
        if (!warp_wait(&s_full[gb], gp & 1u, abort_flag, wlim)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[kMmaN];
#pragma unroll
        for (int c = 0; c < kMmaN / 16; ++c) tmem_ld16(lane_base + (sbuf - tmem) + c * 16, sr + c * 16);
        tmem_wait_ld();
        // ---- mask, row max of the raw scores (the scale is positive, so it is the max of the
        // scaled ones; NaN propagates through the max), 8 independent chains
        const int lim = (row_ok && tile_ok) ? min(mu.end - 1, pos) - n0 : -1;   // last visible column
        if (!__all_sync(0xffffffffu, lim >= kMmaN - 1)) {
#pragma unroll
          for (int j = 0; j < kMmaN; ++j) sr[j] = j <= lim ? sr[j] : 0xff800000u;   // -inf
        }
        const float c = F8 ? p.qk_scale_log2 * q_inv : p.qk_scale_log2;   // 2^-e: exact
        float mx = -INFINITY;
        if (!fixed) {
          float mxa[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mxa[i] = __uint_as_float(sr[i]);
#pragma unroll
          for (int j = 8; j < kMmaN; ++j) mxa[j & 7] = max_nan(mxa[j & 7], __uint_as_float(sr[j]));
#pragma unroll
          for (int w = 4; w > 0; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i) mxa[i] = max_nan(mxa[i], mxa[i + w]);
          mx = mxa[0] * c;
        }
        // a NaN running max stays NaN (a later tile the row cannot see, max -inf, must not replace it)
        const bool grow = !fixed && !(mx <= m_run + (F8 ? kF8Hi : kMmaTau)) && m_run == m_run;
        float m_new = grow ? (F8 ? mx - kF8Mid : mx) : m_run;
        float f = grow ? fast_exp2(m_run - m_new) : 1.f;
        float ls[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) ls[i] = 0.f;
        float pv[F8 ? kMmaN : 1];   // fp8 pools: the tile's weights, kept until m is settled
        float e_tile = 0.f;
        if constexpr (F8) {
          const float nm0 = (m_new == -INFINITY) ? 0.f : -m_new;
#pragma unroll
          for (int j = 0; j < kMmaN; ++j) {
            pv[j] = fast_exp2(fmaf(__uint_as_float(sr[j]), c, nm0));
            ls[j & 7] += pv[j];
          }
          // The terms hold each p to 2^-9 p, plus an absolute floor of 2^-9 when p < 2^-1 (E4M3
          // holds nothing below 2^-9). The floors are kept within 2^-8 of the weight gathered,
          // l: e_run bounds their sum. A tile adds at most 2^-9 per visible position; only when
          // that could pass the budget are its weights below 2^-1 counted (branch-free: the sign
          // of bits(p) - bits(1/2), less the masked columns, exact zeros), and if they still pass
          // it, m moves down to put the tile's largest weight at 2^kF8Mid = 32, which leaves the
          // tile's floors (at most 64 * 2^-9) within 2^-8 of its weight and the budget kept -- unless
          // the weight gathered would pass 2^40 (f = inf included), when the tile adds less than
          // 2^-25 of the total.
          const int masked = lim >= kMmaN - 1 ? 0 : kMmaN - 1 - lim;
          e_tile = 0.001953125f * static_cast<float>(kMmaN - masked);
          float w_t = 0.f;
#pragma unroll
          for (int i = 0; i < 8; ++i) w_t += ls[i];
          const float budget = 0.00390625f * (l_run * f + w_t);
          if (e_run * f + e_tile > budget && mx > -INFINITY) {
            uint32_t n = 0;
#pragma unroll
            for (int j = 0; j < kMmaN; ++j) n += (__float_as_uint(pv[j]) - 0x3F000000u) >> 31;
            e_tile = 0.001953125f * static_cast<float>(static_cast<int>(n) - masked);
            const float fd = fast_exp2(m_new - (mx - kF8Mid));
            if (e_run * f + e_tile > budget && fd > 1.f && l_run * f * fd <= kF8MaxWeight) {
              m_new = mx - kF8Mid;
              f *= fd;
#pragma unroll
              for (int i = 0; i < 8; ++i) ls[i] *= fd;
#pragma unroll
              for (int j = 0; j < kMmaN; ++j) pv[j] *= fd;
              e_tile = 0.001953125f * static_cast<float>(kMmaN - masked);   // <= 2^-8 * 2^kF8Mid
            }
          }
        }
        const float nm = (m_new == -INFINITY) ? 0.f : -m_new;   // all scores -inf: p = 0
        // ---- p = 2^(s c - m) as two terms written over the S columns they came from (before any
        // rescale of O: the product of the previous tile may still run meanwhile)
        if constexpr (F8) {
          // E4M3 terms (split4), four codes a column: P_hi over S columns [0, 16), P_lo over [16, 32)
          uint32_t wh[16], wl[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) p_terms4(pv + 4 * i, wh[i], wl[i]);
          tmem_st16(lane_base + (sbuf - tmem), wh);
          tmem_st16(lane_base + (sbuf - tmem) + kMmaN / 4, wl);
        } else {
          // bf16 terms: P_hi = p with the low 16 bits cleared, P_lo = (p - P_hi) likewise, both exact
          // bf16 values, p - P_hi - P_lo < 2^-14 p; pairs packed with a byte permute (upper halves),
          // hi over S columns [0, 32), lo over [32, 64)
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t wh[16], wl[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int j = half * 32 + 2 * i;
              const float p0 = fast_exp2(fmaf(__uint_as_float(sr[j]), c, nm));
              const float p1 = fast_exp2(fmaf(__uint_as_float(sr[j + 1]), c, nm));
              ls[j & 7] += p0;
              ls[(j + 1) & 7] += p1;
              const uint32_t u0 = __float_as_uint(p0), u1 = __float_as_uint(p1);
              wh[i] = __byte_perm(u0, u1, 0x7632);
              const float l0 = p0 - __uint_as_float(u0 & 0xffff0000u);
              const float l1 = p1 - __uint_as_float(u1 & 0xffff0000u);
              wl[i] = __byte_perm(__float_as_uint(l0), __float_as_uint(l1), 0x7632);
            }
            tmem_st16(lane_base + (sbuf - tmem) + half * 16, wh);
            tmem_st16(lane_base + (sbuf - tmem) + kMmaN / 2 + half * 16, wl);
          }
        }
#pragma unroll
        for (int w = 4; w > 0; w >>= 1)
#pragma unroll
          for (int i = 0; i < w; ++i) ls[i] += ls[i + w];
        if (t > 0 && __any_sync(0xffffffffu, f != 1.f)) {
          // O holds the PVs of tiles g-t .. g-1: wait for the last, then rescale it in TMEM, 64
          // columns a round with the loads in flight together
          if (!warp_wait(&sp_free[pb], pp & 1u, abort_flag, wlim)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < D / 64; ++cc) {
            uint32_t ov[64];
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_ld16(lane_base + C::kOCol + cc * 64 + q * 16, ov + q * 16);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 64; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * f);
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_st16(lane_base + C::kOCol + cc * 64 + q * 16, ov + q * 16);
          }
        }
        m_run = m_new;
        l_run = l_run * f + ls[0];
        if constexpr (F8) e_run = e_run * f + e_tile;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_full[gb]);
        pb = gb;
        pp = gp;
        ++g;
        if (++gb == kSBufs) {
          gb = 0;
          ++gp;
        }
      }
      if (!ok) break;
      if (fixed && l_run == 0.f) m_run = -INFINITY;   // no visible key: an empty partial, as online
      float q_inv_next = 1.f;
      if constexpr (F8) {
        // the next unit's Q terms: every QK^T of this unit has completed (its last S was read)
        if (it.has_next) {
          q_inv_next = q_to_e4m3_terms<D>(p, it.next_mu(), row, q_s);
          fence_proxy_async();
          mbar_arrive(q_full);
        }
      }
      // ---- the unit's last PV is done: O is complete
      if (!warp_wait(&sp_free[pb], pp & 1u, abort_flag, wlim)) {
        ok = false;
        break;
      }
      it.next_unit(p);
      q_inv = q_inv_next;
      if (!it.done) pg_cur = chunk_pages(p, it.mu, 0, lane);
      // ---- epilogue: O from TMEM. Each thread stores its own row, 32 columns at a time, straight
      // from registers with 32-byte stores: every store fills whole 32-byte sectors, and nothing
      // waits on the copy engine, which is busy with the K/V stream.
      tc_fence_after();
      const bool single = mu.n_splits <= 1;
      const float sc = single ? ((m_run == -INFINITY) ? 0.f : p.v_scale / l_run) : 1.f;
      // f16 partials (fp8 pools): acc / l, which stays within the E4M3 codes' range
      const bool half_part = F8 && p.part_f16 && !single;
      const float il = (m_run == -INFINITY) ? 0.f : 1.f / l_run;
      float* dst = nullptr;
      if (row_ok) {
        const int64_t orow = (static_cast<int64_t>(mu.b) * p.rows + r) * p.h_q + static_cast<int64_t>(mu.h) * G + gq;
        dst = single ? p.out + orow * D : p.acc_part + (orow * p.max_splits + mu.s) * D;
        if (!single) {
          st_global_hint(p.m_part + orow * p.max_splits + mu.s, m_run, keep);
          st_global_hint(p.l_part + orow * p.max_splits + mu.s, l_run, keep);
        }
      }
#pragma unroll 1
      for (int ch = 0; ch < D / kChunk; ++ch) {
        uint32_t ov[kChunk];
        tmem_ld16(lane_base + C::kOCol + ch * kChunk, ov);
        tmem_ld16(lane_base + C::kOCol + ch * kChunk + 16, ov + 16);
        tmem_wait_ld();
        if (ch == D / kChunk - 1) {   // O is free for the next unit's first PV
          tc_fence_before();
          mbar_arrive(o_free);
        }
        if (dst != nullptr && half_part) {
          // 32 halves: two 32-byte stores into the first half of the split's slot
#pragma unroll
          for (int c16 = 0; c16 < kChunk / 16; ++c16) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const __half2 h = __floats2half2_rn(__uint_as_float(ov[16 * c16 + 2 * e]) * il,
                                                  __uint_as_float(ov[16 * c16 + 2 * e + 1]) * il);
              v[e] = __uint_as_float(*reinterpret_cast<const uint32_t*>(&h));
            }
            st_global_v8_hint(dst + (ch * kChunk) / 2 + c16 * 8, v, keep);   // kept in L2 for the merge
          }
        } else if (dst != nullptr) {
#pragma unroll
          for (int c8 = 0; c8 < kChunk / 8; ++c8) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(ov[8 * c8 + e]) * sc;
            if (single) st_global_v8(dst + ch * kChunk + c8 * 8, v);
            else st_global_v8_hint(dst + ch * kChunk + c8 * 8, v, keep);   // kept in L2 for the merge
          }
        }
      }
      if (!ok) break;
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

bool make_maps(MmaMaps* m, const DecodeParams& p, bool f8) {
  const cuuint64_t D = static_cast<cuuint64_t>(p.d);
  // pools: rows (page * h_kv + h) * page_tokens + position, columns d; a box is 64 positions of
  // 128 bytes (64 bf16 or 128 E4M3 codes)
  const cuuint64_t pool_dims[2] = {D, static_cast<cuuint64_t>(p.num_pages) * p.h_kv * p.page_tokens};
  const cuuint64_t pool_str[1] = {D * (f8 ? 1 : 2)};
  const cuuint32_t pool_box[2] = {f8 ? 128u : 64u, static_cast<cuuint32_t>(kMmaN)};
  const CUtensorMapDataType pool_type = f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!encode(&m->k, pool_type, 2, p.k_pool, pool_dims, pool_str, pool_box) ||
      !encode(&m->v, pool_type, 2, p.v_pool, pool_dims, pool_str, pool_box))
    return false;
  const int rt = whole_row_tile_rows(p.rows, p.group);
  if (f8 || rt == 0) return true;   // Q is written by threads
  // q [B][R][h_q][d] bf16
  const cuuint64_t HQ = static_cast<cuuint64_t>(p.h_q), R = static_cast<cuuint64_t>(p.rows);
  const cuuint64_t q_dims[4] = {D, HQ, R, static_cast<cuuint64_t>(p.batch)};
  const cuuint64_t q_str[3] = {D * 2, HQ * D * 2, R * HQ * D * 2};
  const cuuint32_t q_box[4] = {64, static_cast<cuuint32_t>(p.group), static_cast<cuuint32_t>(rt), 1};
  return encode(&m->q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p.q, q_dims, q_str, q_box);
}

// The tensor maps of the last few calls made from this host thread, keyed by everything they
// encode (so a hit is the map make_maps would write): three encodes cost an eagerly launched call
// a few microseconds of host time, which a caller stepping the same buffers would pay every step.
struct MapKey {
  const void *k, *v, *q;
  int num_pages, h_kv, page_tokens, d, batch, rows, h_q, group, device;
  bool f8;
  bool operator==(const MapKey& o) const {
    return k == o.k && v == o.v && q == o.q && num_pages == o.num_pages && h_kv == o.h_kv &&
           page_tokens == o.page_tokens && d == o.d && batch == o.batch && rows == o.rows && h_q == o.h_q &&
           group == o.group && device == o.device && f8 == o.f8;
  }
};

const MmaMaps* cached_maps(const DecodeParams& p, bool f8, int device) {
  constexpr int kSlots = 4;
  thread_local MapKey keys[kSlots];
  thread_local MmaMaps maps[kSlots];
  thread_local int used = 0, next = 0;
  const MapKey key{p.k_pool, p.v_pool, p.q, p.num_pages, p.h_kv, p.page_tokens, p.d, p.batch,
                   p.rows, p.h_q, p.group, device, f8};
  for (int i = 0; i < used; ++i)
    if (keys[i] == key) return &maps[i];
  const int slot = next;
  next = (next + 1) % kSlots;
  if (used < kSlots) ++used;
  keys[slot] = MapKey{};   // not valid until encoded
  if (!make_maps(&maps[slot], p, f8)) return nullptr;
  keys[slot] = key;
  return &maps[slot];
}

template <int D, bool F8>
cudaError_t launch_mma(const DecodeParams& p, int grid_limit, cudaStream_t stream) {
  using C = MmaCfg<D, F8>;
  static std::atomic<uint64_t> configured{0};   // devices whose shared-memory limit is raised
  const DeviceInfo& di = device_info();
  const MmaMaps* maps = cached_maps(p, F8, di.device);
  if (maps == nullptr) return cudaErrorInvalidValue;
  const uint64_t bit = 1ull << (di.device & 63);
  if ((configured.load() & bit) == 0) {
    cudaError_t e = cudaFuncSetAttribute(decode_partial_mma_kernel<D, F8, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_partial_mma_kernel<D, F8, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               C::kSmem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  const int m_tiles = (p.rows * p.group + kMmaM - 1) / kMmaM;
  const int64_t upper = static_cast<int64_t>(p.batch) * p.max_splits * p.h_kv * m_tiles;
  int64_t grid = di.sm_count;
  if (grid_limit > 0 && grid > grid_limit) grid = grid_limit;
  if (grid > upper) grid = upper;
  if (grid < 1) grid = 1;
  if (p.wait_limit_ns != kWaitLimitNs || p.producer_delay_ns != 0)   // a test of the timeout path
    return launch_pdl(decode_partial_mma_kernel<D, F8, true>, static_cast<unsigned>(grid), kMmaThreads, C::kSmem,
                      stream, p, *maps);
  return launch_pdl(decode_partial_mma_kernel<D, F8, false>, static_cast<unsigned>(grid), kMmaThreads, C::kSmem,
                    stream, p, *maps);
}

}  // namespace

bool mma_path_applies(const DecodeParams& p, int q_dtype, int pool_dtype) {
  const int64_t pool_rows = static_cast<int64_t>(p.num_pages) * p.h_kv * p.page_tokens;
  return q_dtype == NBX_BF16 && (pool_dtype == NBX_BF16 || pool_dtype == NBX_E4M3) && (p.d == 128 || p.d == 256) &&
         (p.page_tokens % kMmaN) == 0 && p.group <= kMmaM && p.rows * p.group >= 64 &&
         pool_rows < (int64_t{1} << 31) - kMmaN && p.qk_scale_log2 > 0.f;
}

cudaError_t decode_dispatch_mma(const DecodeParams& p, int pool_dtype, int grid_limit, cudaStream_t stream) {
  if (pool_dtype == NBX_E4M3) {
    if (p.d == 128) return launch_mma<128, true>(p, grid_limit, stream);
    return launch_mma<256, true>(p, grid_limit, stream);
  }
  if (p.d == 128) return launch_mma<128, false>(p, grid_limit, stream);
  return launch_mma<256, false>(p, grid_limit, stream);
}

}  // namespace nbx
