// Kernels 2 and 3: the split plan, the per-(split, KV head, row block) partial and the
// fixed-order merge of split-KV decode attention read through a block table.
//
// Method (nbxtensor/ops/paged_decode_attn.py, paged_decode_splits and
// paged_decode_attn_split_kernel; nbxtensor/ops/attention_wrappers.py, decode_reduce):
// every sequence is cut into min(ceil(len/256), 64) splits of whole pages; each split
// runs an online softmax over its keys and stores an unnormalised partial (m, l, acc);
// the partials of a query row are merged in ascending split order.
//
// GB300 design:
//  * plan_kernel (one CTA) reads the device lengths, computes every sequence's split
//    plan and writes a work list of (sequence, split) entries ordered longest split
//    first, so the persistent partial kernel balances a ragged batch.
//  * decode_partial_kernel is persistent: 2 CTAs per SM pull work units
//    u = (entry, KV head, row block) from an atomic counter. Row blocks are the fastest
//    index, so all query rows of one split run side by side and share its K/V from L2
//    (TensorFold PR #1219, the rows-first grid). A unit covers kQB = 4 query vectors
//    (rows x GQA heads of one KV head), so each K/V tile is read once for the whole
//    GQA group instead of once per query head.
//  * One producer warp streams page tiles (16 positions of one KV head, one contiguous
//    block of the pool) into a ring of shared-memory stages with cp.async.bulk and
//    mbarrier transaction counts, running ahead across unit boundaries; it also stages
//    each unit's query vectors. A tile never straddles a page: split starts are page
//    aligned and 16 divides the page.
//  * Four consumer warps compute. Scores: 8 (or 4, 16) lanes share one position, each
//    holding 16 elements of the 4 query vectors in registers; packed fp32 FMAs
//    (fma.rn.f32x2) form partial dots and a transposing shuffle reduction leaves each
//    lane with one (position, vector) score. The online softmax works in log2 units and
//    rescales lazily: the running max moves only when a score exceeds it by more than
//    kTau (the accumulated weights stay below 2^kTau times the tile count, exact in
//    fp32), so the rescale branch is almost never taken. P*V: every lane owns D/32
//    output elements of all 4 vectors and accumulates all positions of its warp.
//  * Epilogue: the four warps' states are merged in fixed warp order through shared
//    memory. A one-split sequence writes the normalised output directly; otherwise the
//    unit stores its partial, and the CTA that takes the last ticket of its
//    (sequence, KV head, row block) merges all splits in ascending order. No inter-CTA
//    waits, no atomics on values: the output is bit-identical under any schedule and
//    any physical page placement.
//  * Every wait is bounded; on timeout the kernel records NBX_DEV_TIMEOUT, drains its
//    copies in flight and returns.
#pragma once

#include "nbx_device.cuh"
#include "nbx_internal.h"

namespace nbx {

constexpr float kTau = 8.0f;                 // lazy-rescale threshold, log2 units
constexpr int kSmemPerCta = 112 * 1024;      // two CTAs per SM

struct UnitMeta {
  int32_t b, s, h, rb, start, end, n_splits, len;
};

template <class PT, class QT, int D>
struct DecodeCfg {
  static constexpr int kLPT = D / 16;                 // lanes per position in the score layout
  static constexpr int kTG = 32 / kLPT;               // positions per warp pass
  static constexpr int kNV = 16 / PT::kEPV;           // 16-byte K vectors per lane
  static constexpr int kVPL = D / 32;                 // output elements per lane in the P*V layout
  static constexpr int kGroups = kTileN / kTG;        // warp passes per tile
  static constexpr int kTileBytes = kTileN * D * PT::kBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kQBytes = kQB * D * QT::kBytes;
  // shared memory carve-up (bytes, each section 128-byte aligned)
  static constexpr int kRedAccBytes = kConsumerWarps * kQB * D * 4;
  static constexpr int kRedMLBytes = kConsumerWarps * kQB * 4 * 2;
  static constexpr int kPBufBytes = kConsumerWarps * kTG * kQB * 4;
  static constexpr int kMergeBytes = kQB * NBX_MAX_SPLITS * 4 * 2 + kQB * 4 * 4;
  static constexpr int kFixed = ((2 * kQBytes + 127) / 128) * 128 + kRedAccBytes + 128 + kPBufBytes + 128 +
                                kMergeBytes + 128 + 2 * (int)sizeof(UnitMeta) + 1024;
  static constexpr int kStagesRaw = (kSmemPerCta - kFixed) / kStageBytes;
  static constexpr int kStages = kStagesRaw > 16 ? 16 : (kStagesRaw < 2 ? 2 : kStagesRaw);
  static_assert(kTileN % kTG == 0, "a tile holds whole warp passes");
  static_assert(kLPT >= 4 && kLPT <= 16, "head dim 64..256");
};

struct SmemLayout {
  char* stages;
  char* qbuf;        // [2][kQBytes]
  float* red_acc;    // [warps][kQB][D]
  float* red_m;      // [warps][kQB]
  float* red_l;      // [warps][kQB]
  float* pbuf;       // [warps][kTG][kQB]
  float* mg_m;       // [kQB][max splits]
  float* mg_w;       // [kQB][max splits]
  float* mg_scale;   // [kQB]
  int* mg_dead;      // [kQB]
  UnitMeta* meta;    // [2]
  int* stage_ok;     // [stages]
  int* flags;        // [0] abort, [1] last-ticket, [2] tiles issued
  uint64_t* full;    // [stages]
  uint64_t* empty;   // [stages]
  uint64_t* qfull;   // [2]
  uint64_t* qempty;  // [2]
  uint64_t* cbar;    // consumer-warp barrier (count: consumer threads)
};

template <class C, int D>
__device__ __forceinline__ SmemLayout carve(char* base) {
  SmemLayout s;
  char* p = base;
  auto take = [&](int bytes) {
    char* r = p;
    p += ((bytes + 127) / 128) * 128;
    return r;
  };
  s.stages = take(C::kStages * C::kStageBytes);
  s.qbuf = take(2 * C::kQBytes);
  s.red_acc = reinterpret_cast<float*>(take(C::kRedAccBytes));
  s.red_m = reinterpret_cast<float*>(take(kConsumerWarps * kQB * 4));
  s.red_l = reinterpret_cast<float*>(take(kConsumerWarps * kQB * 4));
  s.pbuf = reinterpret_cast<float*>(take(C::kPBufBytes));
  s.mg_m = reinterpret_cast<float*>(take(kQB * NBX_MAX_SPLITS * 4));
  s.mg_w = reinterpret_cast<float*>(take(kQB * NBX_MAX_SPLITS * 4));
  s.mg_scale = reinterpret_cast<float*>(take(kQB * 4));
  s.mg_dead = reinterpret_cast<int*>(take(kQB * 4));
  s.meta = reinterpret_cast<UnitMeta*>(take(2 * sizeof(UnitMeta)));
  s.stage_ok = reinterpret_cast<int*>(take(C::kStages * 4));
  s.flags = reinterpret_cast<int*>(take(4 * 4));
  s.full = reinterpret_cast<uint64_t*>(take(C::kStages * 8));
  s.empty = reinterpret_cast<uint64_t*>(take(C::kStages * 8));
  s.qfull = reinterpret_cast<uint64_t*>(take(2 * 8));
  s.qempty = reinterpret_cast<uint64_t*>(take(2 * 8));
  s.cbar = reinterpret_cast<uint64_t*>(take(8));
  return s;
}

template <class C, int D>
constexpr int smem_bytes() {
  int n = 0;
  auto r = [](int b) { return ((b + 127) / 128) * 128; };
  n += r(C::kStages * C::kStageBytes) + r(2 * C::kQBytes) + r(C::kRedAccBytes) + 2 * r(kConsumerWarps * kQB * 4) +
       r(C::kPBufBytes) + 2 * r(kQB * NBX_MAX_SPLITS * 4) + 2 * r(kQB * 4) + r(2 * sizeof(UnitMeta)) +
       r(C::kStages * 4) + r(16) + 2 * r(C::kStages * 8) + 2 * r(16) + r(8);
  return n;
}

// Bounded wait that also gives up as soon as another warp of the CTA has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0u) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}

// ------------------------------------------------------------------------------------ partial
// VPL consecutive elements of format PT at p (aligned to VPL elements), as float pairs.
template <class PT, int VPL>
__device__ __forceinline__ void load_row_pairs(const char* p, float2* out) {
  constexpr int kBytes = VPL * PT::kBytes;
  if constexpr (kBytes >= 16) {
#pragma unroll
    for (int c = 0; c < kBytes / 16; ++c) {
      const uint4 v = *reinterpret_cast<const uint4*>(p + 16 * c);
      unpack16<PT>(v, out + c * (PT::kEPV / 2));
    }
  } else if constexpr (kBytes == 8) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    if constexpr (PT::kCode == NBX_F32) {
      out[0] = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
    } else if constexpr (PT::kCode == NBX_BF16) {
      out[0] = bf16x2_to_float2(v.x);
      out[1] = bf16x2_to_float2(v.y);
    } else {
      out[0] = e4m3x2_to_float2(v.x & 0xffffu);
      out[1] = e4m3x2_to_float2(v.x >> 16);
      out[2] = e4m3x2_to_float2(v.y & 0xffffu);
      out[3] = e4m3x2_to_float2(v.y >> 16);
    }
  } else if constexpr (kBytes == 4) {
    const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
    if constexpr (PT::kCode == NBX_BF16) {
      out[0] = bf16x2_to_float2(v);
    } else {
      out[0] = e4m3x2_to_float2(v & 0xffffu);
      out[1] = e4m3x2_to_float2(v >> 16);
    }
  } else {
    out[0] = e4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(p));
  }
}

template <class PT, class QT, int D>
__global__ void __launch_bounds__(kDecodeThreads, 2) decode_partial_kernel(DecodeParams p) {
  using C = DecodeCfg<PT, QT, D>;
  constexpr int NS = C::kStages;
  constexpr int LPT = C::kLPT;
  constexpr int TG = C::kTG;
  constexpr int NV = C::kNV;
  constexpr int EPV = PT::kEPV;
  constexpr int VPL = C::kVPL;
  constexpr int NW = kConsumerWarps;

  extern __shared__ __align__(1024) char smem_raw[];
  SmemLayout sm = carve<C, D>(smem_raw);
  volatile int* abort_flag = sm.flags;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&sm.full[i], 1);
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

  const int n_units = p.header[0] * p.h_kv * p.row_blocks;
  const int unit_span = p.h_kv * p.row_blocks;
  const int RG = p.rows * p.group;

  if (warp == NW) {
    // ================================================================ producer warp
    uint32_t tile_seq = 0, unit_seq = 0;
    int u = 0;
    if (lane == 0) u = atomicAdd(&p.header[1], 1);
    u = __shfl_sync(0xffffffffu, u, 0);
    bool ok = true;
    while (ok) {
      const uint32_t slot = unit_seq & 1u;
      if (lane == 0 && unit_seq >= 2) ok = wait_or_abort(&sm.qempty[slot], ((unit_seq >> 1) - 1) & 1u, abort_flag);
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
      const int h = rem / p.row_blocks;
      const int rb = rem - h * p.row_blocks;
      const Entry en = p.entries[e_idx];
      const SeqPlan sp = p.plan[en.b];
      int u_next = 0;
      if (lane == 0) u_next = atomicAdd(&p.header[1], 1);
      if (lane == 0) {
        UnitMeta mt;
        mt.b = en.b;
        mt.s = en.s;
        mt.h = h;
        mt.rb = rb;
        mt.start = en.start;
        mt.end = en.end;
        mt.n_splits = sp.n_splits;
        mt.len = sp.len;
        sm.meta[slot] = mt;
        const int q0 = rb * kQB;
        const int nvalid = min(kQB, RG - q0);
        mbar_arrive_expect_tx(&sm.qfull[slot], static_cast<uint32_t>(nvalid * D * QT::kBytes));
        for (int i = 0; i < nvalid; ++i) {
          const int qi = q0 + i;
          const int r = qi / p.group;
          const int g = qi - r * p.group;
          const int64_t row = (static_cast<int64_t>(en.b) * p.rows + r) * p.h_q + static_cast<int64_t>(h) * p.group + g;
          bulk_g2s(sm.qbuf + slot * C::kQBytes + i * D * QT::kBytes,
                   static_cast<const char*>(p.q) + row * D * QT::kBytes, D * QT::kBytes, &sm.qfull[slot]);
        }
      }
      // tiles of the split, page ids fetched 32 at a time by the whole warp
      const int P = p.page_tokens;
      const int first_page = en.start / P;
      const int last_page = (en.end - 1) / P;
      const int32_t* bt_row = p.block_table + static_cast<int64_t>(en.b) * p.max_pages;
      for (int pc = first_page; pc <= last_page && ok; pc += 32) {
        const int my_page = (pc + lane <= last_page) ? bt_row[pc + lane] : -1;
        const int n_lo = max(en.start, pc * P);
        const int n_hi = min(en.end, (pc + 32) * P);
        for (int n0 = n_lo; n0 < n_hi; n0 += kTileN) {
          const int page = __shfl_sync(0xffffffffu, my_page, n0 / P - pc);
          if (lane == 0) {
            const uint32_t stage = tile_seq % NS;
            if (tile_seq >= static_cast<uint32_t>(NS))
              ok = wait_or_abort(&sm.empty[stage], ((tile_seq / NS) - 1) & 1u, abort_flag);
            if (ok) {
              const bool valid = page >= 0 && page < p.num_pages;
              sm.stage_ok[stage] = valid ? 1 : 0;
              if (valid) {
                const int64_t off = ((static_cast<int64_t>(page) * p.h_kv + h) * P + (n0 - (n0 / P) * P)) * D;
                char* dst = sm.stages + stage * C::kStageBytes;
                mbar_arrive_expect_tx(&sm.full[stage], C::kStageBytes);
                bulk_g2s(dst, static_cast<const char*>(p.k_pool) + off * PT::kBytes, C::kTileBytes, &sm.full[stage]);
                bulk_g2s(dst + C::kTileBytes, static_cast<const char*>(p.v_pool) + off * PT::kBytes, C::kTileBytes,
                         &sm.full[stage]);
              } else {
                raise_status(p.status, NBX_DEV_BAD_PAGE);
                mbar_arrive(&sm.full[stage]);
              }
              sm.flags[2] = static_cast<int>(tile_seq + 1);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) break;
          ++tile_seq;
        }
      }
      ++unit_seq;
      u = __shfl_sync(0xffffffffu, u_next, 0);
    }
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
  const int j = lane % LPT;                                  // lane within its position
  const int tg = lane / LPT;                                 // position within the warp pass
  const int gsel = ((j & 1) << 1) | ((j >> 1) & 1);          // vector this lane's score belongs to
  const int ct = threadIdx.x;                                // 0 .. 127
  uint32_t tile_seq = 0, unit_seq = 0, cphase = 0;
  bool ok = true;
  // bounded barrier over the consumer threads (an mbarrier, so a warp that gave up cannot hang the others)
  auto csync = [&]() -> bool {
    mbar_arrive(sm.cbar);
    const bool r = wait_or_abort(sm.cbar, cphase & 1u, abort_flag);
    ++cphase;
    return r;
  };
  float* pb = sm.pbuf + warp * TG * kQB;

  for (;;) {
    const uint32_t slot = unit_seq & 1u;
    if (!wait_or_abort(&sm.qfull[slot], (unit_seq >> 1) & 1u, abort_flag)) { ok = false; break; }
    const UnitMeta mt = sm.meta[slot];
    if (mt.b < 0) break;
    const int q0 = mt.rb * kQB;

    // ---- query vectors: this lane's 16 elements of each, scaled into log2 units
    float2 q2[kQB][8];
    {
      const char* qs = sm.qbuf + slot * C::kQBytes;
#pragma unroll
      for (int i = 0; i < kQB; ++i) {
        const bool vq = q0 + i < RG;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
#pragma unroll
          for (int e2 = 0; e2 < EPV / 2; ++e2) {
            const int el = (j + v * LPT) * EPV + 2 * e2;
            float2 x = load_pair<QT>(qs + (i * D + el) * QT::kBytes);
            x.x = vq ? x.x * p.qk_scale_log2 : 0.f;
            x.y = vq ? x.y * p.qk_scale_log2 : 0.f;
            q2[i][v * (EPV / 2) + e2] = x;
          }
        }
      }
    }
    int pos_sel = -1;   // last visible key of vector gsel (causal window of multi-row units)
    {
      const int qi = q0 + gsel;
      if (qi < RG) pos_sel = mt.len - p.rows + qi / p.group;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.qempty[slot]);

    float m_run = -INFINITY;
    float l_run = 0.f;
    float2 acc2[kQB][VPL / 2];
#pragma unroll
    for (int i = 0; i < kQB; ++i)
#pragma unroll
      for (int k = 0; k < VPL / 2; ++k) acc2[i][k] = make_float2(0.f, 0.f);

    for (int n0 = mt.start; n0 < mt.end; n0 += kTileN) {
      const uint32_t stage = tile_seq % NS;
      if (!wait_or_abort(&sm.full[stage], (tile_seq / NS) & 1u, abort_flag)) { ok = false; break; }
      if (sm.stage_ok[stage]) {
        const char* kt = sm.stages + stage * C::kStageBytes;
        const char* vt = kt + C::kTileBytes;
#pragma unroll 1
        for (int grp = warp; grp < C::kGroups; grp += NW) {
          const int t = grp * TG + tg;
          const int n = n0 + t;
          // ---- scores s_i = q_i . k_n for the 4 vectors, partial over this lane's elements
          float2 s2[kQB];
#pragma unroll
          for (int i = 0; i < kQB; ++i) s2[i] = make_float2(0.f, 0.f);
#pragma unroll
          for (int v = 0; v < NV; ++v) {
            const uint4 kv = *reinterpret_cast<const uint4*>(kt + t * D * PT::kBytes + (j + v * LPT) * 16);
            float2 kf[EPV / 2];
            unpack16<PT>(kv, kf);
#pragma unroll
            for (int e2 = 0; e2 < EPV / 2; ++e2)
#pragma unroll
              for (int i = 0; i < kQB; ++i) s2[i] = ffma2(q2[i][v * (EPV / 2) + e2], kf[e2], s2[i]);
          }
          const float s0 = s2[0].x + s2[0].y, s1 = s2[1].x + s2[1].y;
          const float s2v = s2[2].x + s2[2].y, s3 = s2[3].x + s2[3].y;
          // ---- transposing reduction over the LPT lanes of this position
          const bool b0 = j & 1;
          float k0 = b0 ? s2v : s0, k1 = b0 ? s3 : s1;
          k0 += __shfl_xor_sync(0xffffffffu, b0 ? s0 : s2v, 1);
          k1 += __shfl_xor_sync(0xffffffffu, b0 ? s1 : s3, 1);
          const bool b1 = (j >> 1) & 1;
          float mine = b1 ? k1 : k0;
          mine += __shfl_xor_sync(0xffffffffu, b1 ? k0 : k1, 2);
#pragma unroll
          for (int off = 4; off < LPT; off <<= 1) mine += __shfl_xor_sync(0xffffffffu, mine, off);
          const bool valid = (n < mt.end) && (n <= pos_sel);
          const float s = valid ? mine : -INFINITY;
          // ---- online softmax, lazy rescale
          float mx = s;
#pragma unroll
          for (int off = LPT; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
          const bool need = mx > m_run + kTau;
          if (__any_sync(0xffffffffu, need)) {
            const float m_new = need ? mx : m_run;
            const float f = (m_new == m_run) ? 1.f : fast_exp2(m_run - m_new);
            m_run = m_new;
            l_run *= f;
#pragma unroll
            for (int i = 0; i < kQB; ++i) {
              const float fi = __shfl_sync(0xffffffffu, f, ((i & 1) << 1) | (i >> 1));
#pragma unroll
              for (int k = 0; k < VPL / 2; ++k) acc2[i][k] = fmul2(acc2[i][k], make_float2(fi, fi));
            }
          }
          const float pw = valid ? fast_exp2(s - m_run) : 0.f;
          l_run += pw;
          if (j < 4) pb[tg * kQB + gsel] = pw;
          __syncwarp();
          // ---- acc_i += p_i,n * v_n over this pass's positions
#pragma unroll
          for (int tt = 0; tt < TG; ++tt) {
            const int trow = grp * TG + tt;
            if (n0 + trow < mt.end) {
              const float4 pv = *reinterpret_cast<const float4*>(pb + tt * kQB);
              float2 vf[VPL / 2];
              load_row_pairs<PT, VPL>(vt + (trow * D + lane * VPL) * PT::kBytes, vf);
#pragma unroll
              for (int k = 0; k < VPL / 2; ++k) {
                acc2[0][k] = ffma2(make_float2(pv.x, pv.x), vf[k], acc2[0][k]);
                acc2[1][k] = ffma2(make_float2(pv.y, pv.y), vf[k], acc2[1][k]);
                acc2[2][k] = ffma2(make_float2(pv.z, pv.z), vf[k], acc2[2][k]);
                acc2[3][k] = ffma2(make_float2(pv.w, pv.w), vf[k], acc2[3][k]);
              }
            }
          }
          __syncwarp();
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[stage]);
      ++tile_seq;
    }
    if (!ok) break;

    // ---- epilogue: merge the four warps' states in warp order
    {
      float l_tot = l_run;
#pragma unroll
      for (int off = LPT; off < 32; off <<= 1) l_tot += __shfl_xor_sync(0xffffffffu, l_tot, off);
      if (lane < 4) {
        sm.red_m[warp * kQB + gsel] = m_run;
        sm.red_l[warp * kQB + gsel] = l_tot;
      }
      float* ra = sm.red_acc + warp * kQB * D;
#pragma unroll
      for (int i = 0; i < kQB; ++i)
#pragma unroll
        for (int k = 0; k < VPL / 2; ++k)
          *reinterpret_cast<float2*>(ra + i * D + lane * VPL + 2 * k) = acc2[i][k];
    }
    if (!csync()) { ok = false; break; }
    const bool multi = mt.n_splits > 1;
    for (int o = ct; o < kQB * D; o += NW * 32) {
      const int i = o / D;
      const int dd = o - i * D;
      const int qi = q0 + i;
      if (qi >= RG) continue;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, sm.red_m[w * kQB + i]);
      float L = 0.f, A = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          const float mw = sm.red_m[w * kQB + i];
          if (mw != -INFINITY) {
            const float f = fast_exp2(mw - M);
            L += f * sm.red_l[w * kQB + i];
            A += f * sm.red_acc[(w * kQB + i) * D + dd];
          }
        }
      }
      const int r = qi / p.group;
      const int g = qi - r * p.group;
      const int64_t orow = (static_cast<int64_t>(mt.b) * p.rows + r) * p.h_q + static_cast<int64_t>(mt.h) * p.group + g;
      if (!multi) {
        p.out[orow * D + dd] = (M == -INFINITY) ? 0.f : A * (p.v_scale / L);
      } else {
        const int64_t prow = orow * p.max_splits + mt.s;
        p.acc_part[prow * D + dd] = A;
        if (dd == 0) {
          p.m_part[prow] = M;
          p.l_part[prow] = L;
        }
      }
    }
    if (multi) {
      __threadfence();
      if (!csync()) { ok = false; break; }
      if (ct == 0) {
        const int64_t tk = (static_cast<int64_t>(mt.b) * p.h_kv + mt.h) * p.row_blocks + mt.rb;
        const int old = atomicAdd(&p.tickets[tk], 1);
        sm.flags[1] = (old == mt.n_splits - 1) ? 1 : 0;
      }
      if (!csync()) { ok = false; break; }
      if (sm.flags[1]) {
        // ---- last split of this (sequence, KV head, row block) to finish: merge in split order
        __threadfence();
        const int S = mt.n_splits;
        for (int x = ct; x < kQB * S; x += NW * 32) {
          const int i = x / S;
          const int s = x - i * S;
          const int qi = q0 + i;
          float mv = -INFINITY, lv = 0.f;
          if (qi < RG) {
            const int r = qi / p.group;
            const int g = qi - r * p.group;
            const int64_t orow =
                (static_cast<int64_t>(mt.b) * p.rows + r) * p.h_q + static_cast<int64_t>(mt.h) * p.group + g;
            mv = ld_cg_f32(p.m_part + orow * p.max_splits + s);
            lv = ld_cg_f32(p.l_part + orow * p.max_splits + s);
          }
          sm.mg_m[i * NBX_MAX_SPLITS + s] = mv;
          sm.mg_w[i * NBX_MAX_SPLITS + s] = lv;
        }
        if (!csync()) { ok = false; break; }
        if (ct < kQB) {
          const int i = ct;
          float M = -INFINITY;
          for (int s = 0; s < S; ++s) M = fmaxf(M, sm.mg_m[i * NBX_MAX_SPLITS + s]);
          float L = 0.f;
          for (int s = 0; s < S; ++s) {
            const float mv = sm.mg_m[i * NBX_MAX_SPLITS + s];
            const float w = (mv == -INFINITY) ? 0.f : fast_exp2(mv - M);
            L += w * sm.mg_w[i * NBX_MAX_SPLITS + s];
            sm.mg_w[i * NBX_MAX_SPLITS + s] = w;
          }
          sm.mg_dead[i] = (M == -INFINITY) ? 1 : 0;
          sm.mg_scale[i] = p.v_scale / L;
        }
        if (!csync()) { ok = false; break; }
        for (int o = ct; o < kQB * D; o += NW * 32) {
          const int i = o / D;
          const int dd = o - i * D;
          const int qi = q0 + i;
          if (qi >= RG) continue;
          const int r = qi / p.group;
          const int g = qi - r * p.group;
          const int64_t orow =
              (static_cast<int64_t>(mt.b) * p.rows + r) * p.h_q + static_cast<int64_t>(mt.h) * p.group + g;
          float A = 0.f;
          for (int s = 0; s < S; ++s) {
            if (sm.mg_m[i * NBX_MAX_SPLITS + s] == -INFINITY) continue;
            A += sm.mg_w[i * NBX_MAX_SPLITS + s] * ld_cg_f32(p.acc_part + (orow * p.max_splits + s) * D + dd);
          }
          p.out[orow * D + dd] = sm.mg_dead[i] ? 0.f : A * sm.mg_scale[i];
        }
      }
    }
    if (!csync()) { ok = false; break; }   // shared scratch is reused by the next unit
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
  constexpr int smem = smem_bytes<C, D>();
  static_assert(smem <= 227 * 1024, "shared memory per CTA");
  const DeviceInfo& di = device_info();
  static int configured_for = -1;
  if (configured_for != di.device) {
    cudaError_t e = cudaFuncSetAttribute(decode_partial_kernel<PT, QT, D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured_for = di.device;
  }
  const int64_t upper = static_cast<int64_t>(p.batch) * p.max_splits * p.h_kv * p.row_blocks;
  int64_t grid = static_cast<int64_t>(di.sm_count) * 2;
  if (grid_limit > 0 && grid > grid_limit) grid = grid_limit;
  if (grid > upper) grid = upper;
  if (grid < 1) grid = 1;
  decode_partial_kernel<PT, QT, D><<<static_cast<unsigned>(grid), kDecodeThreads, smem, stream>>>(p);
  return cudaGetLastError();
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
