// Kernels 2 and 3: the per-(split, KV head, row block) partial and the fixed-order merge of
// split-KV decode attention read through a block table.
//
// Method (nbxtensor/ops/paged_decode_attn.py, paged_decode_splits and
// paged_decode_attn_split_kernel; nbxtensor/ops/attention_wrappers.py, decode_reduce):
// every sequence is cut into splits of whole pages (the pages' 256 positions; here two of those a
// split, and a tensor-core window's sized for about one work unit per SM); each split runs an
// online softmax over its keys and stores an unnormalised partial (m, l, acc); the partials of
// a query row are merged in ascending split order.
//
// GB300 design of decode_partial_kernel:
//  * Persistent: kMinBlocks CTAs per SM pull work units u = (entry, KV head, row block) from
//    an atomic counter, in the plan kernel's order (longest split first). Row blocks are the
//    fastest index, so all query rows of one split run side by side and share its K/V from L2
//    (TensorFold PR #1219, the rows-first grid). A unit covers kQB = 4 query vectors (rows x
//    GQA heads of one KV head): each K/V tile is read once for the whole GQA group.
//  * One producer warp streams 16-position page tiles of one KV head (one contiguous block of
//    the pool each, two per stage) into a ring of shared-memory stages: tiles of 4 KB or less
//    with 16-byte cp.async copies by its 32 lanes (each lane's completion arrives on the stage's
//    mbarrier), larger ones with one cp.async.bulk each (completing on the transaction count).
//    It also stages every unit's query vectors and metadata and runs ahead across unit
//    boundaries. A tile never straddles a page: split starts are page aligned and 16 divides the
//    page.
//  * Every consumer warp takes a fixed quarter of every stage (so every partial sum has a
//    fixed order, and the stages are consumed in ring order by all warps). Scores: LPT lanes
//    share one position and each
//    holds 16 elements of the 4 query vectors as packed fp32 pairs (fma.rn.f32x2); a lane group
//    scores TPG positions per pass and a transposing shuffle reduction leaves each lane with one
//    (position, vector) score. Online softmax in log2 units with a lazy rescale: the running max
//    moves only when a pass's max exceeds it by more than kTau, so the rescale branch is rare
//    and the weights stay below 2^kTau (exact enough in fp32). P*V: each lane owns D/32 output
//    elements of the 4 vectors.
//  * Epilogue: the four warps' states are merged in fixed warp order through shared memory: the
//    unit's last stage, held back from the producer until the merge has read it (this frees the
//    room of a fourth stage), or a double-buffered scratch for E4M3 stages, which are too small;
//    bounded barriers order the writes and reads. A one-split sequence writes its normalised
//    output; otherwise the unit stores its partial, with an L2 evict-last policy so that it is
//    still in L2 when decode_merge_kernel (launched after it) merges the splits in ascending
//    order. No atomics on values and fixed reduction orders:
//    the output is bit-identical under any schedule and any physical page placement.
//  * Every wait is bounded; on timeout the kernel records NBX_DEV_TIMEOUT, lets its copies in
//    flight land and returns.
#pragma once

#include "nbx_device.cuh"
#include "nbx_internal.h"

namespace nbx {

constexpr float kTau = 8.0f;                 // lazy-rescale threshold, log2 units
constexpr int kSmemPerSm = 228 * 1024;       // shared memory of one SM (1 KB of it reserved per CTA)

struct UnitMeta {
  int32_t b, s, h, start, end, n_splits, nvec, pad;
  int32_t pos[kQB];    // last key each vector sees (causal row position); -1 for a missing vector
  int64_t orow[kQB];   // output row (b * rows + r) * h_q + h * group + g
};

template <class PT, class QT, int D>
struct DecodeCfg {
  static constexpr int kLPT = D / 16;                  // lanes per position in the score layout
  static constexpr int kTPG = kLPT >= 8 ? 2 : 1;       // positions each lane group scores per pass
  static constexpr int kTG = 32 / kLPT;                // lane groups per warp
  static constexpr int kPassTok = kTG * kTPG;          // positions per warp pass
  static constexpr int kStageTok = 2 * kTileN;         // positions per stage: two 16-position page tiles
  static constexpr int kWarpTok = kStageTok / kConsumerWarps;   // positions of a stage each warp takes
  static constexpr int kWarpPasses = kWarpTok / kPassTok;
  static constexpr int kNV = 16 / PT::kEPV;            // 16-byte K vectors per lane
  static constexpr int kVPL = D / 32;                  // output elements per lane in the P*V layout
  static constexpr int kTileBytes = kTileN * D * PT::kBytes;     // one 16-position tile of K (or V)
  static constexpr int kHalfBytes = kStageTok * D * PT::kBytes;  // the K (or V) part of a stage
  static constexpr int kStageBytes = 2 * kHalfBytes;
  static constexpr int kQBytes = kQB * D * QT::kBytes;
  static constexpr int kRedFloats = kConsumerWarps * (kQB * D + 2 * kQB);   // one slot
  static constexpr int kPBufBytes = kConsumerWarps * kPassTok * kQB * 8;      // (p, p) pairs
  // the epilogue's cross-warp scratch lives in the unit's last stage when each warp's own K rows of
  // it hold the warp's accumulators (pool elements of 2 bytes or more), which leaves room for one
  // more stage; a warp reads only its own positions' rows, so it may write over them at once
  static constexpr bool kRedInStage = kWarpTok * D * PT::kBytes >= kQB * D * 4;
  // small page tiles (4 KB or less) are moved by the producer warp's 32 lanes with 16-byte cp.async
  // copies: the copy engine's fixed cost per bulk request would cap the stream below HBM speed
  static constexpr bool kWarpCopy = kTileBytes <= 4096;
  static constexpr int kFixed = 2 * kQBytes + (kRedInStage ? 0 : 2 * kRedFloats * 4) + kPBufBytes +
                                2 * (int)sizeof(UnitMeta) + 2048;
  // resident CTAs per SM: 3 (2 at head dim 256, where the registers allow no more), fewer when
  // shared memory cannot hold two stages for each of them
  static constexpr int kBlocksBySmem = kSmemPerSm / (kFixed + 2 * kStageBytes + 1024);
  static constexpr int kMinBlocks = (D <= 128 ? 3 : 2) < kBlocksBySmem ? (D <= 128 ? 3 : 2)
                                                                        : (kBlocksBySmem < 1 ? 1 : kBlocksBySmem);
  static constexpr int kSmemPerCta = kSmemPerSm / kMinBlocks - 1024;
  static constexpr int kStagesRaw = (kSmemPerCta - kFixed) / kStageBytes;
  static constexpr int kStages = kStagesRaw > 8 ? 8 : (kStagesRaw < 2 ? 2 : kStagesRaw);
  static_assert(kWarpTok % kPassTok == 0, "a warp's share of a stage holds whole passes");
  static_assert(!kRedInStage || kWarpTok * D * PT::kBytes >= 2 * kQB * 4, "a warp's V rows hold its m and l");
  static_assert(kLPT >= 4 && kLPT <= 16, "head dim 64..256");
};

struct SmemLayout {
  char* stages;
  char* qbuf;        // [2][kQBytes]
  float* red;        // [2][warps][kQB*D acc | kQB m | kQB l], or null when it lives in a stage
  f32x2* pbuf;       // [warps][kPassTok][kQB] (p, p) pairs
  UnitMeta* meta;    // [2]
  int* stage_ok;     // [stages] bit h: tile h of the stage was copied
  int* flags;        // [0] abort, [2] tiles issued
  uint64_t* full;    // [stages]
  uint64_t* empty;   // [stages]
  uint64_t* qfull;   // [2]
  uint64_t* qempty;  // [2]
  uint64_t* cbar;    // consumer-warp barrier
};

template <class C>
struct Carver {
  static constexpr int r(int b) { return ((b + 127) / 128) * 128; }
  static constexpr int bytes() {
    return r(C::kStages * C::kStageBytes) + r(2 * C::kQBytes) + r(C::kRedInStage ? 0 : 2 * C::kRedFloats * 4) + r(C::kPBufBytes) +
           r(2 * (int)sizeof(UnitMeta)) + r(C::kStages * 4) + r(16) + 2 * r(C::kStages * 8) + 2 * r(16) + r(8);
  }
  __device__ static SmemLayout carve(char* base) {
    SmemLayout s;
    char* p = base;
    auto take = [&](int b) {
      char* q = p;
      p += r(b);
      return q;
    };
    s.stages = take(C::kStages * C::kStageBytes);
    s.qbuf = take(2 * C::kQBytes);
    s.red = C::kRedInStage ? nullptr : reinterpret_cast<float*>(take(2 * C::kRedFloats * 4));
    s.pbuf = reinterpret_cast<f32x2*>(take(C::kPBufBytes));
    s.meta = reinterpret_cast<UnitMeta*>(take(2 * sizeof(UnitMeta)));
    s.stage_ok = reinterpret_cast<int*>(take(C::kStages * 4));
    s.flags = reinterpret_cast<int*>(take(16));
    s.full = reinterpret_cast<uint64_t*>(take(C::kStages * 8));
    s.empty = reinterpret_cast<uint64_t*>(take(C::kStages * 8));
    s.qfull = reinterpret_cast<uint64_t*>(take(16));
    s.qempty = reinterpret_cast<uint64_t*>(take(16));
    s.cbar = reinterpret_cast<uint64_t*>(take(8));
    return s;
  }
};

// Bounded wait (limit_ns of wall time) that also gives up as soon as another warp of the CTA has
// aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if ((i & 3u) == 0u && global_timer_ns() - t0 > limit_ns) return false;
  }
}

// VPL consecutive elements of format PT at shared address a (aligned to VPL elements), as packed pairs.
template <class PT, int VPL>
__device__ __forceinline__ void lds_row_x2(uint32_t a, f32x2* out) {
  constexpr int kBytes = VPL * PT::kBytes;
  if constexpr (kBytes >= 16) {
#pragma unroll
    for (int c = 0; c < kBytes / 16; ++c) unpack16x2<PT>(lds128(a + 16 * c), out + c * (PT::kEPV / 2));
  } else if constexpr (kBytes == 8) {
    const uint2 v = lds64(a);
    if constexpr (PT::kCode == NBX_F32) {
      out[0] = (static_cast<f32x2>(v.y) << 32) | v.x;
    } else if constexpr (PT::kCode == NBX_BF16) {
      out[0] = bf16x2_to_f32x2(v.x);
      out[1] = bf16x2_to_f32x2(v.y);
    } else {
      out[0] = e4m3x2_to_f32x2(v.x & 0xffffu);
      out[1] = e4m3x2_to_f32x2(v.x >> 16);
      out[2] = e4m3x2_to_f32x2(v.y & 0xffffu);
      out[3] = e4m3x2_to_f32x2(v.y >> 16);
    }
  } else if constexpr (kBytes == 4) {
    const uint32_t v = lds32(a);
    if constexpr (PT::kCode == NBX_BF16) {
      out[0] = bf16x2_to_f32x2(v);
    } else {
      out[0] = e4m3x2_to_f32x2(v & 0xffffu);
      out[1] = e4m3x2_to_f32x2(v >> 16);
    }
  } else {
    out[0] = e4m3x2_to_f32x2(lds16(a));
  }
}

// One position of P*V: acc_i += (p_i, p_i) * v for the 4 vectors, p pairs at pb, the lane's V
// elements at va (shared addresses).
template <class PT, int VPL>
__device__ __forceinline__ void pv_step(uint32_t pb, uint32_t va, f32x2 (&acc2)[kQB][VPL / 2]) {
  f32x2 p0, p1, p2, p3;
  lds2x64(pb, p0, p1);
  lds2x64(pb + 16, p2, p3);
  f32x2 vf[VPL / 2];
  lds_row_x2<PT, VPL>(va, vf);
#pragma unroll
  for (int k = 0; k < VPL / 2; ++k) {
    acc2[0][k] = fma2(p0, vf[k], acc2[0][k]);
    acc2[1][k] = fma2(p1, vf[k], acc2[1][k]);
    acc2[2][k] = fma2(p2, vf[k], acc2[2][k]);
    acc2[3][k] = fma2(p3, vf[k], acc2[3][k]);
  }
}

// The same, updating only the vectors whose bit is set in `mask` (the others do not see the
// position): a masked vector's accumulator is left as it is, not multiplied by a zero weight, so a
// NaN in a value row past its causal limit cannot reach it.
template <class PT, int VPL>
__device__ __forceinline__ void pv_step_masked(uint32_t pb, uint32_t va, f32x2 (&acc2)[kQB][VPL / 2], int mask) {
  f32x2 p0, p1, p2, p3;
  lds2x64(pb, p0, p1);
  lds2x64(pb + 16, p2, p3);
  f32x2 vf[VPL / 2];
  lds_row_x2<PT, VPL>(va, vf);
#pragma unroll
  for (int k = 0; k < VPL / 2; ++k) {
    if (mask & 1) acc2[0][k] = fma2(p0, vf[k], acc2[0][k]);
    if (mask & 2) acc2[1][k] = fma2(p1, vf[k], acc2[1][k]);
    if (mask & 4) acc2[2][k] = fma2(p2, vf[k], acc2[2][k]);
    if (mask & 8) acc2[3][k] = fma2(p3, vf[k], acc2[3][k]);
  }
}

// ------------------------------------------------------------------------------------ partial
template <class PT, class QT, int D>
__global__ void __launch_bounds__(kDecodeThreads, DecodeCfg<PT, QT, D>::kMinBlocks)
    decode_partial_kernel(DecodeParams p) {
  using C = DecodeCfg<PT, QT, D>;
  constexpr int NS = C::kStages;
  constexpr int LPT = C::kLPT;
  constexpr int TPG = C::kTPG;
  constexpr int NV = C::kNV;
  constexpr int EPV = PT::kEPV;
  constexpr int VPL = C::kVPL;
  constexpr int NW = kConsumerWarps;

  extern __shared__ __align__(1024) char smem_raw[];
  SmemLayout sm = Carver<C>::carve(smem_raw);
  volatile int* abort_flag = sm.flags;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      // bulk copies: lane 0's arrive with the byte count; warp copies: each lane's cp.async
      // completion plus lane 0's arrive after it published the stage's tile bits
      mbar_init(&sm.full[i], C::kWarpCopy ? 33 : 1);
      mbar_init(&sm.empty[i], NW);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.qfull[i], 1);
      mbar_init(&sm.qempty[i], NW);
    }
    mbar_init(sm.cbar, NW * 32);
    sm.flags[0] = 0;
    sm.flags[1] = 0;
    sm.flags[2] = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();              // the plan kernel's work list and the append's positions are visible from here on
  pdl_launch_dependents(); // the merge kernel may be scheduled as CTAs of this grid retire

  const int n_units = p.header[0] * p.h_kv * p.row_blocks;
  const int unit_span = p.h_kv * p.row_blocks;
  const int RG = p.rows * p.group;

  if (warp == NW) {
    // ================================================================ producer warp
    if (p.producer_delay_ns) {   // a test holds the producer back so that the consumers' waits run out
      const uint64_t t0 = global_timer_ns();
      while (global_timer_ns() - t0 < p.producer_delay_ns) __nanosleep(10000);
    }
    uint32_t tile_seq = 0, unit_seq = 0;
    int u = 0;
    if (lane == 0) u = atomicAdd(&p.header[1], 1);
    u = __shfl_sync(0xffffffffu, u, 0);
    bool ok = true;
    while (ok) {
      const uint32_t slot = unit_seq & 1u;
      if (lane == 0 && unit_seq >= 2)
        ok = wait_or_abort(&sm.qempty[slot], ((unit_seq >> 1) - 1) & 1u, abort_flag, p.wait_limit_ns);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      if (u >= n_units) {
        if (lane == 0) {
          sm.meta[slot].b = -1;
          mbar_arrive(&sm.qfull[slot]);
        }
        break;
      }
      const int e_idx = u / unit_span;
      const int rem = u - e_idx * unit_span;
      const int h = p.row_blocks == 1 ? rem : rem / p.row_blocks;
      const int rb = rem - h * p.row_blocks;
      const Entry en = p.entries[e_idx];   // carries its sequence's length and split count
      int u_next = 0;
      if (lane == 0) u_next = atomicAdd(&p.header[1], 1);
      if (lane == 0) {
        UnitMeta mt;
        mt.b = en.b;
        mt.s = en.s;
        mt.h = h;
        mt.start = en.start;
        mt.end = en.end;
        mt.n_splits = en.n_splits;
        const int q0 = rb * kQB;
        const int nvalid = min(kQB, RG - q0);
        mt.nvec = nvalid;
        mt.pad = 0;
        int r = p.rows == 1 ? 0 : q0 / p.group;   // query row and head of vector q0 + i, stepped
        int g = q0 - r * p.group;
#pragma unroll
        for (int i = 0; i < kQB; ++i) {
          const bool vq = i < nvalid;
          mt.pos[i] = vq ? en.len - p.rows + r : -1;
          mt.orow[i] = vq ? (static_cast<int64_t>(en.b) * p.rows + r) * p.h_q + static_cast<int64_t>(h) * p.group + g
                          : 0;
          if (++g == p.group) {
            g = 0;
            ++r;
          }
        }
        sm.meta[slot] = mt;
        mbar_arrive_expect_tx(&sm.qfull[slot], static_cast<uint32_t>(nvalid * D * QT::kBytes));
        for (int i = 0; i < nvalid; ++i)
          bulk_g2s(sm.qbuf + slot * C::kQBytes + i * D * QT::kBytes,
                   static_cast<const char*>(p.q) + mt.orow[i] * D * QT::kBytes, D * QT::kBytes, &sm.qfull[slot]);
      }
      // stages of two 16-position tiles; page ids fetched 32 at a time by the whole warp
      const int P = p.page_tokens;
      const int32_t* bt_row = p.block_table + static_cast<int64_t>(en.b) * p.max_pages;
      const int last_page = (en.end - 1) / P;
      int pc = en.start / P;
      int my_page = (pc + lane <= last_page) ? bt_row[pc + lane] : -1;
      // page index and position in the page of the next tile, advanced tile by tile (no division)
      int t_pi = pc, t_po = en.start - pc * P;
      for (int n0 = en.start; n0 < en.end; n0 += C::kStageTok) {
        int pages[2], pofs[2];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int nh = n0 + hf * kTileN;
          const int pi = t_pi;
          pofs[hf] = t_po;
          t_po += kTileN;
          if (t_po == P) {
            t_po = 0;
            ++t_pi;
          }
          if (nh < en.end && pi >= pc + 32) {   // warp-uniform: next chunk of page ids
            pc = pi;
            my_page = (pc + lane <= last_page) ? bt_row[pc + lane] : -1;
          }
          pages[hf] = __shfl_sync(0xffffffffu, my_page, (pi - pc) & 31);
        }
        const uint32_t stage = tile_seq % NS;
        int okbits = 0;
        if (lane == 0) {
          if (tile_seq >= static_cast<uint32_t>(NS))
            ok = wait_or_abort(&sm.empty[stage], ((tile_seq / NS) - 1) & 1u, abort_flag, p.wait_limit_ns);
          if (ok) {
            uint32_t bytes = 0;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const int nh = n0 + hf * kTileN;
              if (nh >= en.end) continue;
              if (pages[hf] >= 0 && pages[hf] < p.num_pages) {
                okbits |= 1 << hf;
                bytes += 2 * C::kTileBytes;
              } else {
                raise_status(p.status, NBX_DEV_BAD_PAGE);
              }
            }
            sm.stage_ok[stage] = okbits;
            char* dst = sm.stages + stage * C::kStageBytes;
            if (C::kWarpCopy) {
              mbar_arrive(&sm.full[stage]);   // releases the tile bits; the lanes' copies follow
            } else if (bytes) {
              mbar_arrive_expect_tx(&sm.full[stage], bytes);
#pragma unroll
              for (int hf = 0; hf < 2; ++hf) {
                if (!((okbits >> hf) & 1)) continue;
                const int64_t off = ((static_cast<int64_t>(pages[hf]) * p.h_kv + h) * P + pofs[hf]) * D * PT::kBytes;
                bulk_g2s(dst + hf * C::kTileBytes, static_cast<const char*>(p.k_pool) + off, C::kTileBytes,
                         &sm.full[stage]);
                bulk_g2s(dst + C::kHalfBytes + hf * C::kTileBytes, static_cast<const char*>(p.v_pool) + off,
                         C::kTileBytes, &sm.full[stage]);
              }
            } else {
              mbar_arrive(&sm.full[stage]);
            }
            sm.flags[2] = static_cast<int>(tile_seq + 1);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        if constexpr (C::kWarpCopy) {
          // the stage's tiles in 16-byte pieces, 512 contiguous bytes per warp instruction
          okbits = __shfl_sync(0xffffffffu, okbits, 0);
          const uint32_t dst = smem_u32(sm.stages + stage * C::kStageBytes);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            if (!((okbits >> hf) & 1)) continue;
            const int64_t off = ((static_cast<int64_t>(pages[hf]) * p.h_kv + h) * P + pofs[hf]) * D * PT::kBytes;
            const char* ks = static_cast<const char*>(p.k_pool) + off;
            const char* vs = static_cast<const char*>(p.v_pool) + off;
#pragma unroll
            for (int c = lane; c < C::kTileBytes / 16; c += 32) {
              cp_async16(dst + hf * C::kTileBytes + c * 16, ks + c * 16);
              cp_async16(dst + C::kHalfBytes + hf * C::kTileBytes + c * 16, vs + c * 16);
            }
          }
          cp_async_arrive_noinc(&sm.full[stage]);
        }
        ++tile_seq;
      }
      ++unit_seq;
      u = __shfl_sync(0xffffffffu, u_next, 0);
    }
    if constexpr (C::kWarpCopy) cp_async_wait_all();   // this lane's copies have landed
    if (!ok && lane == 0) {
      // gave up: record it, then let the copies already issued land before the CTA exits
      raise_status(p.status, NBX_DEV_TIMEOUT);
      *abort_flag = 1;
      const uint32_t issued = tile_seq;
      for (uint32_t i = issued > static_cast<uint32_t>(NS) ? issued - NS : 0; i < issued; ++i)
        mbar_wait(&sm.full[i % NS], (i / NS) & 1u, 100000000ull);
      for (uint32_t i = unit_seq > 2 ? unit_seq - 2 : 0; i < unit_seq; ++i)
        mbar_wait(&sm.qfull[i & 1u], (i >> 1) & 1u, 100000000ull);
    }
    return;
  }

  // ================================================================== consumer warps
  const int j = lane % LPT;   // lane within its position group
  const int tg = lane / LPT;  // position group within the warp
  // after the transposing reduction this lane holds the score of (position tsel, vector vsel)
  const int tsel = (TPG == 2) ? (j & 1) : 0;
  const int vsel = (TPG == 2) ? ((((j >> 1) & 1) << 1) | ((j >> 2) & 1)) : (((j & 1) << 1) | ((j >> 1) & 1));
  const bool p_writer = (LPT <= 8) || j < 8;   // one lane per distinct (position, vector)
  const int ct = threadIdx.x;    // 0 .. 127
  uint32_t tile_seq = 0, unit_seq = 0, cphase = 0;
  bool ok = true;
  // bounded barrier over the consumer threads (an mbarrier: a warp that gave up cannot hang the others)
  auto csync = [&]() -> bool {
    mbar_arrive(sm.cbar);
    const bool r = wait_or_abort(sm.cbar, cphase & 1u, abort_flag, p.wait_limit_ns);
    ++cphase;
    return r;
  };
  // 32-bit shared addresses; per-lane offsets inside a stage are fixed for the whole kernel
  const uint32_t stages_base = smem_u32(sm.stages);
  const uint32_t k_lane_off = static_cast<uint32_t>(tg * TPG * D * PT::kBytes + j * 16);
  const uint32_t v_lane_off = static_cast<uint32_t>(C::kHalfBytes + lane * VPL * PT::kBytes);
  const uint32_t pb_addr = smem_u32(sm.pbuf + warp * C::kPassTok * kQB);
  const uint32_t p_store = pb_addr + static_cast<uint32_t>(((tg * TPG + tsel) * kQB + vsel) * 8);

  for (;;) {
    const uint32_t slot = unit_seq & 1u;
    if (!wait_or_abort(&sm.qfull[slot], (unit_seq >> 1) & 1u, abort_flag, p.wait_limit_ns)) {
      ok = false;
      break;
    }
    // the unit's metadata stays in its shared slot until this unit's epilogue is done
    const UnitMeta* mtp = &sm.meta[slot];
    const int u_b = mtp->b;
    if (u_b < 0) break;
    const int u_start = mtp->start, u_end = mtp->end, u_nvec = mtp->nvec;

    // ---- query vectors: this lane's 16 elements of each, scaled into log2 units
    f32x2 q2[kQB][8];
    {
      // the lane's elements of a vector come in runs of EPV, one wide shared load each
      const uint32_t qs = smem_u32(sm.qbuf + slot * C::kQBytes);
      const f32x2 sc2 = pack2(p.qk_scale_log2, p.qk_scale_log2);
#pragma unroll
      for (int i = 0; i < kQB; ++i) {
        const bool vq = i < u_nvec;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          f32x2 x[EPV / 2];
          lds_row_x2<QT, EPV>(qs + static_cast<uint32_t>((i * D + (j + v * LPT) * EPV) * QT::kBytes), x);
#pragma unroll
          for (int e2 = 0; e2 < EPV / 2; ++e2) q2[i][v * (EPV / 2) + e2] = vq ? mul2(x[e2], sc2) : 0ull;
        }
      }
    }
    const int pos_sel = mtp->pos[vsel];   // last visible key of vector vsel

    float m_run = -INFINITY;
    float l_run = 0.f;
    f32x2 acc2[kQB][VPL / 2];
#pragma unroll
    for (int i = 0; i < kQB; ++i)
#pragma unroll
      for (int k = 0; k < VPL / 2; ++k) acc2[i][k] = 0ull;

    const int n_stages = (u_end - u_start + C::kStageTok - 1) / C::kStageTok;
    uint32_t last_stage = 0;   // the unit's last stage: held for the epilogue's scratch
    for (int t = 0; t < n_stages; ++t, ++tile_seq) {
      const uint32_t stage = tile_seq % NS;
      if (!wait_or_abort(&sm.full[stage], (tile_seq / NS) & 1u, abort_flag, p.wait_limit_ns)) {
        ok = false;
        break;
      }
      const int okbits = sm.stage_ok[stage];
      if (okbits) {
        const int n0 = u_start + t * C::kStageTok;
        // every position of the stage copied, inside the split, and seen by every vector of the unit
        // (vector 0 has the unit's smallest causal limit)
        const bool full_stage = (okbits == 3) && (n0 + C::kStageTok <= u_end) && (n0 + C::kStageTok - 1 <= mtp->pos[0]);
        const uint32_t st_base = stages_base + stage * C::kStageBytes;
#pragma unroll 1
        for (int pass = 0; pass < C::kWarpPasses; ++pass) {
          const int pbase = warp * C::kWarpTok + pass * C::kPassTok;   // first position of this pass in the stage
          // ---- scores s[tk][i] = q_i . k for this lane group's TPG positions, partial over 16 elements
          f32x2 s2[TPG][kQB];
#pragma unroll
          for (int tk = 0; tk < TPG; ++tk)
#pragma unroll
            for (int i = 0; i < kQB; ++i) s2[tk][i] = 0ull;
#pragma unroll
          for (int tk = 0; tk < TPG; ++tk) {
#pragma unroll
            for (int v = 0; v < NV; ++v) {
              const uint4 kv = lds128(st_base + (pbase + tk) * D * PT::kBytes + k_lane_off + v * LPT * 16);
              f32x2 kf[EPV / 2];
              unpack16x2<PT>(kv, kf);
#pragma unroll
              for (int e2 = 0; e2 < EPV / 2; ++e2)
#pragma unroll
                for (int i = 0; i < kQB; ++i) s2[tk][i] = fma2(q2[i][v * (EPV / 2) + e2], kf[e2], s2[tk][i]);
            }
          }
          float sv[TPG][kQB];
#pragma unroll
          for (int tk = 0; tk < TPG; ++tk)
#pragma unroll
            for (int i = 0; i < kQB; ++i) {
              const float2 t2 = unpack2(s2[tk][i]);
              sv[tk][i] = t2.x + t2.y;
            }
          // ---- transposing reduction over the LPT lanes of a position group
          float mine;
          if constexpr (TPG == 2) {
            const bool b0 = j & 1;   // keep position b0, send the other
            float a[kQB];
#pragma unroll
            for (int i = 0; i < kQB; ++i)
              a[i] = (b0 ? sv[1][i] : sv[0][i]) + __shfl_xor_sync(0xffffffffu, b0 ? sv[0][i] : sv[1][i], 1);
            const bool b1 = (j >> 1) & 1;   // keep vectors 2*b1, 2*b1+1
            const float c0 = (b1 ? a[2] : a[0]) + __shfl_xor_sync(0xffffffffu, b1 ? a[0] : a[2], 2);
            const float c1 = (b1 ? a[3] : a[1]) + __shfl_xor_sync(0xffffffffu, b1 ? a[1] : a[3], 2);
            const bool b2 = (j >> 2) & 1;   // keep vector 2*b1 + b2
            mine = (b2 ? c1 : c0) + __shfl_xor_sync(0xffffffffu, b2 ? c0 : c1, 4);
            if constexpr (LPT == 16) mine += __shfl_xor_sync(0xffffffffu, mine, 8);
          } else {
            const bool b0 = j & 1;   // keep vectors 2*b0, 2*b0+1
            const float k0 = (b0 ? sv[0][2] : sv[0][0]) + __shfl_xor_sync(0xffffffffu, b0 ? sv[0][0] : sv[0][2], 1);
            const float k1 = (b0 ? sv[0][3] : sv[0][1]) + __shfl_xor_sync(0xffffffffu, b0 ? sv[0][1] : sv[0][3], 1);
            const bool b1 = (j >> 1) & 1;   // keep vector 2*b0 + b1
            mine = (b1 ? k1 : k0) + __shfl_xor_sync(0xffffffffu, b1 ? k0 : k1, 2);
          }
          const int rs = pbase + tg * TPG + tsel;   // this lane's position inside the stage
          const int n = n0 + rs;
          const bool valid = ((okbits >> (rs / kTileN)) & 1) && (n < u_end) && (n <= pos_sel);
          const float s = valid ? mine : -INFINITY;
          // ---- online softmax, lazy rescale; the max runs over the lanes holding the same vector
          // (NaN-propagating max: a NaN score makes the running max NaN, so it reaches the output)
          float mx = s;
          if constexpr (TPG == 2) mx = max_nan(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
#pragma unroll
          for (int off = LPT; off < 32; off <<= 1) mx = max_nan(mx, __shfl_xor_sync(0xffffffffu, mx, off));
          // a NaN running max stays NaN: a later pass whose positions are all masked (max -inf) must
          // not replace it, or the warp's state would read as empty and the NaN would be dropped
          const bool need = !(mx <= m_run + kTau) && m_run == m_run;
          if (__any_sync(0xffffffffu, need)) {
            const float m_new = need ? mx : m_run;
            const float f = need ? fast_exp2(m_run - m_new) : 1.f;
            m_run = m_new;
            l_run *= f;
#pragma unroll
            for (int i = 0; i < kQB; ++i) {
              const int src = (TPG == 2) ? (((i >> 1) << 1) | ((i & 1) << 2)) : (((i & 1) << 1) | (i >> 1));
              const float fi = __shfl_sync(0xffffffffu, f, src);
              const f32x2 fi2 = pack2(fi, fi);
#pragma unroll
              for (int k = 0; k < VPL / 2; ++k) acc2[i][k] = mul2(acc2[i][k], fi2);
            }
          }
          const float pw = valid ? fast_exp2(s - m_run) : 0.f;
          l_run += pw;
          if (p_writer) sts64(p_store, pack2(pw, pw));
          __syncwarp();
          // ---- acc_i += p_i,n * v_n over this pass's positions (no per-position test in full stages)
          if (full_stage) {
#pragma unroll
            for (int pt = 0; pt < C::kPassTok; ++pt)
              pv_step<PT, VPL>(pb_addr + pt * kQB * 8, st_base + v_lane_off + (pbase + pt) * D * PT::kBytes, acc2);
          } else {
            // a position updates only the vectors whose causal limit it is within
#pragma unroll
            for (int pt = 0; pt < C::kPassTok; ++pt) {
              const int n = n0 + pbase + pt;
              if (((okbits >> ((pbase + pt) / kTileN)) & 1) && n < u_end) {
                const int mask = (n <= mtp->pos[0] ? 1 : 0) | (n <= mtp->pos[1] ? 2 : 0) | (n <= mtp->pos[2] ? 4 : 0) |
                                 (n <= mtp->pos[3] ? 8 : 0);
                pv_step_masked<PT, VPL>(pb_addr + pt * kQB * 8, st_base + v_lane_off + (pbase + pt) * D * PT::kBytes,
                                        acc2, mask);
              }
            }
          }
          __syncwarp();
        }
      }
      __syncwarp();
      if (!C::kRedInStage || t + 1 < n_stages) {
        if (lane == 0) mbar_arrive(&sm.empty[stage]);
      } else {
        last_stage = stage;
      }
    }
    if (!ok) break;

    // ---- epilogue: merge the four warps' states in warp order. Warp w's state (acc [kQB][D], then
    // m [kQB] and l [kQB]) sits over its own K rows and V rows of the unit's last stage, which only
    // it reads, or in a double-buffered scratch.
    char* const red_base = C::kRedInStage ? sm.stages + last_stage * C::kStageBytes
                                          : reinterpret_cast<char*>(sm.red + slot * C::kRedFloats);
    auto acc_of = [&](int w) -> float* {
      return C::kRedInStage ? reinterpret_cast<float*>(red_base + w * C::kWarpTok * D * PT::kBytes)
                            : reinterpret_cast<float*>(red_base) + w * (kQB * D + 2 * kQB);
    };
    auto ml_of = [&](int w) -> float* {
      return C::kRedInStage ? reinterpret_cast<float*>(red_base + C::kHalfBytes + w * C::kWarpTok * D * PT::kBytes)
                            : reinterpret_cast<float*>(red_base) + w * (kQB * D + 2 * kQB) + kQB * D;
    };
    {
      float l_tot = l_run;
      if constexpr (TPG == 2) l_tot += __shfl_xor_sync(0xffffffffu, l_tot, 1);
#pragma unroll
      for (int off = LPT; off < 32; off <<= 1) l_tot += __shfl_xor_sync(0xffffffffu, l_tot, off);
      __syncwarp();   // every lane of this warp is done with its rows of the last stage
      float* rw = acc_of(warp);
      float* rm = ml_of(warp);
      if (lane < 8 && tsel == 0) {   // one lane per vector
        rm[vsel] = m_run;
        rm[kQB + vsel] = l_tot;
      }
#pragma unroll
      for (int i = 0; i < kQB; ++i)
#pragma unroll
        for (int k = 0; k < VPL / 2; ++k) *reinterpret_cast<f32x2*>(rw + i * D + lane * VPL + 2 * k) = acc2[i][k];
    }
    if (!csync()) {
      ok = false;
      break;
    }
    const bool multi = mtp->n_splits > 1;
    const int u_split = mtp->s;
    // the merged values go to registers first: the last stage and the metadata slot are handed back
    // before the global stores, so neither the proxy fence nor the arrives wait behind them
    constexpr int kOut = kQB * D / (NW * 32);
    float r_a[kOut], r_m[kOut], r_l[kOut];
    int64_t r_row[kOut];
#pragma unroll
    for (int x = 0; x < kOut; ++x) {
      const int o = ct + x * NW * 32;
      const int i = o / D;
      const int dd = o - i * D;
      r_row[x] = i < u_nvec ? mtp->orow[i] : -1;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = max_nan(M, ml_of(w)[i]);
      float L = 0.f, A = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          const float mw = ml_of(w)[i];
          if (mw != -INFINITY) {
            const float f = fast_exp2(mw - M);
            L += f * ml_of(w)[kQB + i];
            A += f * acc_of(w)[i * D + dd];
          }
        }
      }
      r_a[x] = A;
      r_m[x] = M;
      r_l[x] = L;
    }
    if constexpr (C::kRedInStage) {
      // the stage goes back to the producer. Its next fill is a bulk copy (async proxy) unless the
      // tiles are warp copies: cp.async is a generic-proxy write, ordered by the barrier alone.
      if constexpr (!C::kWarpCopy) fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[last_stage]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.qempty[slot]);   // the slot's queries and metadata are free again
#pragma unroll
    for (int x = 0; x < kOut; ++x) {
      if (r_row[x] < 0) continue;
      const int dd = (ct + x * NW * 32) % D;
      if (!multi) {
        p.out[r_row[x] * D + dd] = (r_m[x] == -INFINITY) ? 0.f : r_a[x] * (p.v_scale / r_l[x]);
      } else {
        // the partial stays in L2 for the merge
        const uint64_t keep = l2_keep_policy(p.keep_frac);
        const int64_t prow = r_row[x] * p.max_splits + u_split;
        st_global_hint(p.acc_part + prow * D + dd, r_a[x], keep);
        if (dd == 0) {
          st_global_hint(p.m_part + prow, r_m[x], keep);
          st_global_hint(p.l_part + prow, r_l[x], keep);
        }
      }
    }
    ++unit_seq;
  }

  if (!ok) {
    *abort_flag = 1;
    if (threadIdx.x == 0) {
      raise_status(p.status, NBX_DEV_TIMEOUT);
      // let the copies already issued land before the CTA exits
      const uint32_t issued = static_cast<uint32_t>(sm.flags[2]);
      for (uint32_t i = issued > static_cast<uint32_t>(NS) ? issued - NS : 0; i < issued; ++i)
        mbar_wait(&sm.full[i % NS], (i / NS) & 1u, 100000000ull);
      for (uint32_t i = unit_seq; i < unit_seq + 3; ++i) mbar_wait(&sm.qfull[i & 1u], (i >> 1) & 1u, 100000000ull);
    }
  }
}

// ------------------------------------------------------------------------------------ launch
template <class PT, class QT, int D>
cudaError_t launch_decode(const DecodeParams& p, int grid_limit, cudaStream_t stream) {
  using C = DecodeCfg<PT, QT, D>;
  constexpr int smem = Carver<C>::bytes();
  static_assert(smem <= C::kSmemPerCta, "shared memory per CTA");
  const DeviceInfo& di = device_info();
  static int configured_for = -1;
  if (configured_for != di.device) {
    cudaError_t e = cudaFuncSetAttribute(decode_partial_kernel<PT, QT, D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured_for = di.device;
  }
  const int64_t upper = static_cast<int64_t>(p.batch) * p.max_splits * p.h_kv * p.row_blocks;
  int64_t grid = static_cast<int64_t>(di.sm_count) * C::kMinBlocks;
  if (grid_limit > 0 && grid > grid_limit) grid = grid_limit;
  if (grid > upper) grid = upper;
  if (grid < 1) grid = 1;
  return launch_pdl(decode_partial_kernel<PT, QT, D>, static_cast<unsigned>(grid), kDecodeThreads, smem, stream, p);
}

#define NBX_DECODE_FOR_POOL(PT)                                                                                   \
  cudaError_t decode_dispatch_##PT(const DecodeParams& p, int q_dtype, int grid_limit, cudaStream_t stream) {     \
    if (q_dtype == NBX_F32) {                                                                                      \
      if (p.d == 64) return launch_decode<PT, F32, 64>(p, grid_limit, stream);                                     \
      if (p.d == 128) return launch_decode<PT, F32, 128>(p, grid_limit, stream);                                   \
      return launch_decode<PT, F32, 256>(p, grid_limit, stream);                                                   \
    }                                                                                                              \
    if (p.d == 64) return launch_decode<PT, BF16, 64>(p, grid_limit, stream);                                      \
    if (p.d == 128) return launch_decode<PT, BF16, 128>(p, grid_limit, stream);                                    \
    return launch_decode<PT, BF16, 256>(p, grid_limit, stream);                                                    \
  }

cudaError_t decode_dispatch_F32(const DecodeParams& p, int q_dtype, int grid_limit, cudaStream_t stream);
cudaError_t decode_dispatch_BF16(const DecodeParams& p, int q_dtype, int grid_limit, cudaStream_t stream);
cudaError_t decode_dispatch_E4M3(const DecodeParams& p, int q_dtype, int grid_limit, cudaStream_t stream);

}  // namespace nbx
