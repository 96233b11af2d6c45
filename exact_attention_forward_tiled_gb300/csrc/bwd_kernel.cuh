// Exact attention backward for sm_103a (GB300): dQ, dK, dV of
// O = softmax(scale * Q K^T [+ causal mask]) V for an upstream gradient dO.
//
// The pages give the forward only ("Flash Attention 3 principles (guijiagi)"
// section 1.2 with the section 2.2 softmax; the "FlashAttention-3 (lukebest
// wiki)" table reports backward speed without the algorithm). The gradient
// is the plain derivative of that forward:
//
//   P = exp(scale * S - LSE)     (recomputed tile by tile from the forward's LSE)
//   dV = P^T dO,   dP = dO V^T,   dS = P * (dP - Delta),   Delta = rowsum(dO * O)
//   dQ = scale * dS K,   dK = scale * dS^T Q
//
// Two persistent kernels share this template (deterministic, no atomics):
//
//   dK/dV kernel: a CTA keeps one 128-key block of K and V in shared memory
//     and streams the 128-row blocks of Q and dO that can see it:
//       S^T = K Q^T, dP^T = V dO^T          (tcgen05, both operands in SMEM)
//       P^T, dS^T -> 16-bit, back into tensor memory over S^T, dP^T
//       dV += P^T dO, dK += dS^T Q          (tcgen05, A from tensor memory)
//   dQ kernel: a CTA keeps one 128-row block of Q and dO and streams K, V:
//       S = Q K^T, dP = dO V^T;  P, dS -> tensor memory;  dQ += dS K
//
// The dQ kernel recomputes S and dP (7 instead of 5 matrix products in all)
// so that every output row is written by exactly one CTA.
//
// D = 256: the accumulators of dK and dV (256 tensor-memory columns each) and
// the two 128-column score buffers do not fit the 512 columns together, nor do
// two resident and two streamed tiles of 64 KB fit shared memory. The
// gradient then takes three kernels -- dQ, dK, dV -- and the streamed tiles
// arrive as two 128-column halves (32 KB ring slots); the streamed operand
// that the accumulating product needs again (K for dQ, Q for dK) is loaded a
// second time from L2 rather than held. dK recomputes S^T and dP^T, dV
// recomputes S^T: 8 products run where 5 are algorithmic.
//
// Roles: eight "softmax" warps (two warpgroups, each owning half of the 128
// streamed columns of every resident row: thread = resident row), one MMA
// warp (one thread issues), one load warp (TMA). The softmax warps hand a
// block back in two phases -- P as soon as S is read, dS once dP is -- and
// the MMA warp fills the gaps with the next block's S and dP products, so the
// tensor core keeps working while P and dS are made. Every mbarrier wait is
// bounded (see pipeline.cuh).
#pragma once

#include <cstdint>
#include <math_constants.h>

#include "fa_internal.h"
#include "pipeline.cuh"
#include "ptx.cuh"

namespace fa {

// What one backward kernel computes: dQ (resident Q, dO), dK and dV together
// (resident K, V; D <= 128), or, at D = 256, dK alone or dV alone.
enum BwdMode : int { kBwdDQ = 0, kBwdDKDV = 1, kBwdDK = 2, kBwdDV = 3 };

template <int D_, int STAGES_, int KIND_, int MODE_>
struct BwdCfg {
  static constexpr int D = D_;
  static constexpr int STAGES = STAGES_;
  static constexpr int KIND = KIND_;
  static constexpr int MODE = MODE_;
  static constexpr bool DQ = MODE == kBwdDQ;   // resident Q, dO; streamed K, V
  // D = 256: streamed tiles in two 128-column halves, one ring slot each
  static constexpr bool kSplit = D == 256;
  static constexpr bool kNeedY = MODE != kBwdDV;    // dP (dP^T) and dS (dS^T) are made
  static constexpr bool kStoreP = MODE == kBwdDKDV || MODE == kBwdDV;   // P^T kept for dV += P^T dO
  static constexpr int kResident = MODE == kBwdDV ? 1 : 2;              // R1 (and R2) held
  static constexpr int kBoxCols = 64;               // 16-bit elements per 128-byte box row
  static constexpr int kBoxes = D / kBoxCols;
  static constexpr int kBoxBytes = 128 * 128;
  static constexpr int kTileBytes = kBoxes * kBoxBytes;   // one 128-row tile
  static constexpr int kTBytes = kSplit ? 2 * kBoxBytes : kTileBytes;   // one streamed ring slot
  static constexpr int kKSteps = D / 16;                 // MMA K steps over D
  static constexpr int kSoftmaxWarps = 8;
  static constexpr int kMmaWarp = 8, kLoadWarp = 9;
  static constexpr int kThreads = 320;
  static constexpr int kTmemCols = 512;
  // tensor memory: accumulators at 0 (dQ, or dV) and D (dK); X (S or S^T)
  // at 256 and Y (dP or dP^T) at 384; the 16-bit P / dS go over X / Y
  static constexpr uint32_t kColAcc1 = MODE == kBwdDKDV ? (uint32_t)D : 0u;   // dQ or dK
  static constexpr uint32_t kColAcc2 = 0u;                      // dV
  static constexpr uint32_t kColX = 256u, kColY = 384u;
  // shared memory
  static constexpr int kOffR = 0;                                // R1, R2
  static constexpr int kOffT = kResident * kTileBytes;           // ring of T tiles (halves at D = 256)
  static constexpr int kOffVec = kOffT + STAGES * kTBytes;       // per-warp column constants
  static constexpr int kVecBytes = DQ ? 0 : 2 * 64 * 4;
  static constexpr int kOffBar = kOffVec + kSoftmaxWarps * kVecBytes;
  static constexpr int kTileRing = 4;
  // barriers: r_full, r_empty, t_full[S], t_empty[S]; x_full, y_full (MMA ->
  // softmax: S or dP of the block is in tensor memory); p_full, ds_full
  // (softmax -> MMA: P, then dS, of the block handed back); acc_full,
  // mma_done, tile_full[R], tile_empty[R]
  static constexpr int kBarRFull = 0, kBarREmpty = 1, kBarTFull = 2, kBarTEmpty = 2 + STAGES,
                       kBarXFull = 2 + 2 * STAGES, kBarYFull = kBarXFull + 1, kBarPFull = kBarYFull + 1,
                       kBarDSFull = kBarPFull + 1, kBarAccFull = kBarDSFull + 1, kBarMmaDone = kBarAccFull + 1,
                       kBarTileFull = kBarMmaDone + 1, kBarTileEmpty = kBarTileFull + kTileRing,
                       kNumBars = kBarTileEmpty + kTileRing;
  static constexpr int kTileConsumers = 1 + kSoftmaxWarps;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 4 * kTileRing + 1024;

  static_assert(D == 64 || D == 128 || D == 256, "head dimension");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kSplit ? MODE != kBwdDKDV : (MODE == kBwdDQ || MODE == kBwdDKDV), "modes per head size");
  static_assert((MODE == kBwdDKDV ? 2 * D : D) <= 256, "accumulators below the score columns");
};

// Work tile: one 128-row block of the resident side of one (sequence, head).
struct BwdTile {
  int b, h;
  int r0;          // first resident row within its sequence
  int Lq, Lk;
  int rtok, ttok;  // token of row 0 of the sequence on the resident / streamed side
  int t_first;     // first streamed 128-row block
  int n_t;         // streamed blocks to visit
  bool live;       // false: the block starts beyond its sequence
};

template <bool DQ, bool CAUSAL>
__device__ __forceinline__ BwdTile bwd_tile(const BwdParams& p, int w) {
  BwdTile t;
  int bh, j;
  tile_order(w, p.n_rblk, p.B * p.H, p.head_group, bh, j);
  // causal: heavy tiles first (dQ: the last query blocks see the most keys;
  // dK/dV: the first key blocks are seen by the most queries)
  const int rblk = (DQ && CAUSAL) ? p.n_rblk - 1 - j : j;
  t.b = bh / p.H;
  t.h = bh - t.b * p.H;
  int qs, ks;
  if (p.cu_q != nullptr) {
    qs = __ldg(p.cu_q + t.b);
    const int qe = __ldg(p.cu_q + t.b + 1);
    ks = __ldg(p.cu_k + t.b);
    const int ke = __ldg(p.cu_k + t.b + 1);
    t.Lq = qe - qs;
    t.Lk = ke - ks;
    if (qs < 0 || qe < qs || qe > p.total_q || ks < 0 || ke < ks || ke > p.total_k || t.Lq > p.Sq ||
        t.Lk > p.Sk) {
      t.Lq = 0;
      t.Lk = 0;
      if (rblk == 0) atomicOr(p.status, kDevBadSeqlens);
    }
  } else {
    qs = t.b * p.Sq;
    ks = t.b * p.Sk;
    t.Lq = p.Sq;
    t.Lk = p.Sk;
  }
  t.r0 = rblk * 128;
  const int shift = t.Lk - t.Lq;   // causal: query i sees keys j <= i + shift
  t.t_first = 0;
  t.n_t = 0;
  if (DQ) {
    t.rtok = qs;
    t.ttok = ks;
    t.live = t.r0 < t.Lq;
    if (t.live) {
      const int last = min(t.r0 + 128, t.Lq) - 1;
      const int lim = CAUSAL ? min(t.Lk, last + shift + 1) : t.Lk;
      t.n_t = lim > 0 ? (lim + 127) / 128 : 0;
    }
  } else {
    t.rtok = ks;
    t.ttok = qs;
    t.live = t.r0 < t.Lk;
    if (t.live) {
      const int q_lo = CAUSAL ? max(0, t.r0 - shift) : 0;   // first query that sees key r0
      if (q_lo < t.Lq) {
        t.t_first = q_lo / 128;
        t.n_t = (t.Lq + 127) / 128 - t.t_first;
      }
    }
  }
  return t;
}

__device__ __forceinline__ int bwd_fetch_tile(const BwdParams& p, int j) {
  const int w = j == 0 ? (int)blockIdx.x : (int)gridDim.x + (int)atomicAdd(p.sched, 1u);
  return w < p.ntiles ? w : -1;
}

// ------------------------------------------------------------------ load warp (lane 0)
template <class C, bool CAUSAL>
__device__ void bwd_load_role(const CUtensorMap* tr1, const CUtensorMap* tr2, const CUtensorMap* tt1,
                              const CUtensorMap* tt2, const BwdParams& p, uint32_t sbase, const Waiter& wt,
                              const TileRing& ring) {
  const uint32_t bars = sbase + C::kOffBar;
  auto bar = [&](int i) { return bars + 8u * i; };
  uint32_t tc = 0, rcount = 0;
  bool ok = true;
  auto load_tile = [&](const CUtensorMap* m, int h, int row, uint32_t dst, uint32_t b) {
#pragma unroll
    for (int bx = 0; bx < C::kBoxes; ++bx)
      ptx::tma_load_2d(dst + bx * C::kBoxBytes, m, h * C::D + bx * C::kBoxCols, row, b);
  };
  // one streamed ring slot: a whole tile, or (D = 256) its 128-column half
  auto load_t = [&](const CUtensorMap* m, int h, int row, int half) -> bool {
    const int s = tc % C::STAGES;
    const uint32_t ph = (tc / C::STAGES) & 1u;
    if (!wt.wait(bar(C::kBarTEmpty + s), ph ^ 1u, 22)) return false;
    ptx::mbar_arrive_expect_tx(bar(C::kBarTFull + s), C::kTBytes);
    const uint32_t dst = sbase + C::kOffT + s * C::kTBytes;
    if (C::kSplit) {
#pragma unroll
      for (int bx = 0; bx < 2; ++bx)
        ptx::tma_load_2d(dst + bx * C::kBoxBytes, m, h * C::D + 128 * half + bx * C::kBoxCols, row,
                         bar(C::kBarTFull + s));
    } else {
      load_tile(m, h, row, dst, bar(C::kBarTFull + s));
    }
    ++tc;
    return true;
  };
  // a streamed block: one slot, or (D = 256) two consecutive half slots
  auto load_block = [&](const CUtensorMap* m, int h, int row) -> bool {
    if (!load_t(m, h, row, 0)) return false;
    return !C::kSplit || load_t(m, h, row, 1);
  };

  for (int j = 0; ok; ++j) {
    const int rs = j % C::kTileRing;
    if (!wt.wait(ring.empty(rs), ((j / C::kTileRing) & 1u) ^ 1u, 20)) break;
    const int w = bwd_fetch_tile(p, j);
    ring.slots[rs] = w;
    ptx::mbar_arrive(ring.full(rs));
    if (w < 0) break;
    const BwdTile ti = bwd_tile<C::DQ, CAUSAL>(p, w);
    if (!ti.live || ti.n_t == 0) continue;
    if (!wt.wait(bar(C::kBarREmpty), (rcount & 1u) ^ 1u, 21)) break;
    ptx::mbar_arrive_expect_tx(bar(C::kBarRFull), C::kResident * C::kTileBytes);
    load_tile(tr1, ti.h, ti.rtok + ti.r0, sbase + C::kOffR, bar(C::kBarRFull));
    if (C::kResident == 2) load_tile(tr2, ti.h, ti.rtok + ti.r0, sbase + C::kOffR + C::kTileBytes, bar(C::kBarRFull));
    ++rcount;
    const int n = ti.n_t;
    auto trow = [&](int i) { return ti.ttok + 128 * (ti.t_first + i); };
    if (!C::kSplit) {
      // T1, T2 of each block, in the order the MMA thread consumes them
      for (int i = 0; ok && i < n; ++i) ok = load_block(tt1, ti.h, trow(i)) && load_block(tt2, ti.h, trow(i));
    } else if (C::kNeedY) {
      // dQ, dK at D = 256: T1_0, T2_0, then per block i: T1_{i+1}, T1_i again
      // (for the accumulating product), T2_{i+1}
      ok = load_block(tt1, ti.h, trow(0)) && load_block(tt2, ti.h, trow(0));
      for (int i = 0; ok && i < n; ++i) {
        if (i + 1 < n) ok = load_block(tt1, ti.h, trow(i + 1));
        ok = ok && load_block(tt1, ti.h, trow(i));
        if (ok && i + 1 < n) ok = load_block(tt2, ti.h, trow(i + 1));
      }
    } else {
      // dV at D = 256: T1_0, then per block i: T2_i, T1_{i+1}
      ok = load_block(tt1, ti.h, trow(0));
      for (int i = 0; ok && i < n; ++i) {
        ok = load_block(tt2, ti.h, trow(i));
        if (ok && i + 1 < n) ok = load_block(tt1, ti.h, trow(i + 1));
      }
    }
  }
  if (*wt.abort_flag) {
    const uint32_t first = tc > (uint32_t)C::STAGES ? tc - C::STAGES : 0u;
    for (uint32_t c = first; c < tc; ++c)
      wt.drain(bar(C::kBarTFull + (int)(c % C::STAGES)), (c / C::STAGES) & 1u);
    if (rcount > 0) wt.drain(bar(C::kBarRFull), (rcount - 1) & 1u);
  }
}

// ------------------------------------------------------------------ MMA warp (one thread)
template <class C, bool CAUSAL>
__device__ void bwd_mma_role(const BwdParams& p, uint32_t sbase, uint32_t tmem, const Waiter& wt,
                             const TileRing& ring) {
  const uint32_t bars = sbase + C::kOffBar;
  auto bar = [&](int i) { return bars + 8u * i; };
  constexpr uint32_t fmt = C::KIND == kBF16 ? 1u : 0u;
  constexpr uint32_t idesc_s = ptx::make_idesc(fmt, false, 128, 128);   // X, Y: 128 x 128
  constexpr uint32_t idesc_acc = ptx::make_idesc(fmt, true, 128, C::D); // acc += Z T (T MN-major)
  const uint32_t r1 = sbase + C::kOffR, r2 = r1 + C::kTileBytes;
  auto slot_addr = [&](uint32_t c) { return sbase + C::kOffT + (c % C::STAGES) * C::kTBytes; };

  // X or Y = R T^T over the head dimension (both K-major), committed to `b`
  auto mm_s = [&](uint32_t col, uint32_t r_addr, uint32_t t_addr, int b) {
#pragma unroll
    for (int kk = 0; kk < C::kKSteps; ++kk) {
      const uint32_t off = (kk >> 2) * C::kBoxBytes + (kk & 3) * 32;
      ptx::mma_f16_ss(tmem + col, ptx::smem_desc_sw128(r_addr + off, 16, 1024),
                      ptx::smem_desc_sw128(t_addr + off, 16, 1024), idesc_s, kk > 0);
    }
    ptx::mma_commit(bar(b));
  };
  // acc (+)= Z T: Z (16-bit, in tensor memory over X or Y; warpgroup g's 64
  // streamed rows packed at columns 64 g .. 64 g + 31) times the T tile
  // (MN-major B: 16 streamed rows per step)
  auto mm_acc = [&](uint32_t acc_col, uint32_t z_col, uint32_t t_addr, bool acc) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t zc = z_col + 64u * (kk >> 2) + 8u * (kk & 3);
      const uint64_t b = ptx::smem_desc_sw128(t_addr + kk * 16 * 128, C::kBoxBytes, 1024);
      ptx::mma_f16_ts(tmem + acc_col, tmem + zc, b, idesc_acc, (acc || kk > 0) ? 1u : 0u);
    }
  };
  auto t_ready = [&](uint32_t c) {
    const bool r = wt.wait(bar(C::kBarTFull + (int)(c % C::STAGES)), (c / C::STAGES) & 1u, 23);
    ptx::tc_fence_after();
    return r;
  };
  // D = 256, T in two half slots c, c + 1:
  // X or Y = R T^T over the 256 columns (steps 0-7 from half 0, 8-15 from half 1)
  auto mm_s_split = [&](uint32_t col, uint32_t r_addr, uint32_t c, int b) {
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const uint32_t r_off = (kk >> 2) * C::kBoxBytes + (kk & 3) * 32;
      const uint32_t t_off = ((kk >> 2) & 1) * C::kBoxBytes + (kk & 3) * 32;
      ptx::mma_f16_ss(tmem + col, ptx::smem_desc_sw128(r_addr + r_off, 16, 1024),
                      ptx::smem_desc_sw128(slot_addr(c + (kk >> 3)) + t_off, 16, 1024), idesc_s, kk > 0);
    }
    ptx::mma_commit(bar(b));
  };
  // acc (+)= Z T over 256 columns: accumulator half h from T's half slot c + h
  constexpr uint32_t idesc_half = ptx::make_idesc(fmt, true, 128, 128);
  auto mm_acc_split = [&](uint32_t acc_col, uint32_t z_col, uint32_t c, bool acc) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t zc = z_col + 64u * (kk >> 2) + 8u * (kk & 3);
        const uint64_t b = ptx::smem_desc_sw128(slot_addr(c + half) + kk * 16 * 128, C::kBoxBytes, 1024);
        ptx::mma_f16_ts(tmem + acc_col + 128u * half, tmem + zc, b, idesc_half, (acc || kk > 0) ? 1u : 0u);
      }
    }
  };
  auto halves_ready = [&](uint32_t c) { return t_ready(c) && t_ready(c + 1); };
  auto release_halves = [&](uint32_t c) {
    ptx::mma_commit(bar(C::kBarTEmpty + (int)(c % C::STAGES)));
    ptx::mma_commit(bar(C::kBarTEmpty + (int)((c + 1) % C::STAGES)));
  };

  // Issue order per block i (T tiles of block i in slots c, c + 1):
  //   [P_i handed back]  dV += P_i^T dO_i (dK/dV kernel),  X_{i+1}
  //   [dS_i handed back] acc1 += dS_i T1_i,                Y_{i+1}
  // so the tensor core computes the next block's scores while the softmax
  // warps turn this block's dP into dS, and the next block's dP while they
  // make the next P. X_{i+1} overwrites P_i and Y_{i+1} overwrites dS_i only
  // after the products that read them (tcgen05 MMAs run in issue order).
  uint32_t tc = 0, it = 0, rcount = 0;
  bool ok = true;
  int w = 0;
  for (int j = 0; ok && next_tile(ring, wt, j, C::kTileRing, false, true, w); ++j) {
    const BwdTile ti = bwd_tile<C::DQ, CAUSAL>(p, w);
    if (!ti.live || ti.n_t == 0) continue;
    if (!(ok = wt.wait(bar(C::kBarRFull), rcount & 1u, 24))) break;
    ++rcount;
    ptx::tc_fence_after();
    const int n = ti.n_t;
    if (C::kSplit) {
      // D = 256: the same overlap of the next block's scores with this
      // block's softmax work, T in half slots; each pair of half slots is
      // released as soon as its products have read it
      uint32_t c = tc;
      if (!(ok = halves_ready(c))) break;
      mm_s_split(C::kColX, r1, c, C::kBarXFull);
      release_halves(c);
      c += 2;
      if (C::kNeedY) {
        if (!(ok = halves_ready(c))) break;
        mm_s_split(C::kColY, r2, c, C::kBarYFull);
        release_halves(c);
        c += 2;
      }
      if (n == 1) ptx::mma_commit(bar(C::kBarREmpty));   // last use of R1, R2
      for (int i = 0; i < n; ++i, ++it) {
        const bool more = i + 1 < n;
        if (!(ok = wt.wait(bar(C::kBarPFull), it & 1u, 25))) break;
        ptx::tc_fence_after();
        if (!C::kNeedY) {
          // dV: dV += P^T dO, then the next block's S^T over P^T
          if (!(ok = halves_ready(c))) break;
          mm_acc_split(C::kColAcc2, C::kColX, c, i > 0);
          release_halves(c);
          c += 2;
          if (more) {
            if (!(ok = halves_ready(c))) break;
            mm_s_split(C::kColX, r1, c, C::kBarXFull);
            release_halves(c);
            c += 2;
            if (i + 2 == n) ptx::mma_commit(bar(C::kBarREmpty));
          }
          continue;
        }
        if (more) {
          if (!(ok = halves_ready(c))) break;
          mm_s_split(C::kColX, r1, c, C::kBarXFull);
          release_halves(c);
          c += 2;
        }
        if (!(ok = wt.wait(bar(C::kBarDSFull), it & 1u, 26))) break;
        ptx::tc_fence_after();
        if (!(ok = halves_ready(c))) break;
        mm_acc_split(C::kColAcc1, C::kColY, c, i > 0);   // dQ += dS K  or  dK += dS^T Q
        release_halves(c);
        c += 2;
        if (more) {
          if (!(ok = halves_ready(c))) break;
          mm_s_split(C::kColY, r2, c, C::kBarYFull);
          release_halves(c);
          c += 2;
          if (i + 2 == n) ptx::mma_commit(bar(C::kBarREmpty));
        }
      }
      if (!ok) break;
      tc = c;
      ptx::mma_commit(bar(C::kBarAccFull));
      continue;
    }
    if (!(ok = t_ready(tc))) break;
    mm_s(C::kColX, r1, slot_addr(tc), C::kBarXFull);
    if (!(ok = t_ready(tc + 1))) break;
    mm_s(C::kColY, r2, slot_addr(tc + 1), C::kBarYFull);
    if (n == 1) ptx::mma_commit(bar(C::kBarREmpty));   // last use of R1, R2
    for (int i = 0; i < n; ++i, ++it) {
      const uint32_t c = tc + 2 * i;
      const bool more = i + 1 < n;
      if (!(ok = wt.wait(bar(C::kBarPFull), it & 1u, 25))) break;
      ptx::tc_fence_after();
      if (!C::DQ) mm_acc(C::kColAcc2, C::kColX, slot_addr(c + 1), i > 0);   // dV += P^T dO
      if (more) {
        if (!(ok = t_ready(c + 2))) break;
        mm_s(C::kColX, r1, slot_addr(c + 2), C::kBarXFull);
      }
      if (!(ok = wt.wait(bar(C::kBarDSFull), it & 1u, 26))) break;
      ptx::tc_fence_after();
      mm_acc(C::kColAcc1, C::kColY, slot_addr(c), i > 0);   // dQ += dS K  or  dK += dS^T Q
      ptx::mma_commit(bar(C::kBarTEmpty + (int)(c % C::STAGES)));
      ptx::mma_commit(bar(C::kBarTEmpty + (int)((c + 1) % C::STAGES)));
      if (more) {
        if (!(ok = t_ready(c + 3))) break;
        mm_s(C::kColY, r2, slot_addr(c + 3), C::kBarYFull);
        if (i + 2 == n) ptx::mma_commit(bar(C::kBarREmpty));
      }
    }
    if (!ok) break;
    tc += 2 * n;
    ptx::mma_commit(bar(C::kBarAccFull));
  }
  ptx::mma_commit(bar(C::kBarMmaDone));
  wt.drain(bar(C::kBarMmaDone), 0);
}

// ------------------------------------------------------------------ softmax warps
template <int KIND>
__device__ __forceinline__ uint32_t pack16(float lo, float hi) {
  return KIND == kF16 ? ptx::pack_f16(lo, hi) : ptx::pack_bf16(lo, hi);
}

// Write one output row (D values, times `mul`) from tensor-memory columns
// [col, col + n) into out[0 .. n) as 16-bit.
template <int KIND>
__device__ __forceinline__ void store_acc_row(uint32_t taddr, int n, float mul, uint16_t* out, bool write) {
#pragma unroll 1
  for (int ch = 0; ch < n / 32; ++ch) {
    uint32_t v[32];
    ptx::tmem_ld32(taddr + 32 * ch, v);
    ptx::tmem_wait_ld();
    ptx::reg_fence(v);
    uint32_t pk[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      pk[j] = pack16<KIND>(__uint_as_float(v[2 * j]) * mul, __uint_as_float(v[2 * j + 1]) * mul);
    if (write) {
      uint4* dst = reinterpret_cast<uint4*>(out + 32 * ch);
#pragma unroll
      for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    }
  }
}

template <int KIND>
__device__ __forceinline__ void zero_row(uint16_t* out, int n, bool write) {
  if (!write) return;
  for (int d = 0; d < n; d += 8) *reinterpret_cast<uint4*>(out + d) = make_uint4(0, 0, 0, 0);
}

template <class C, bool CAUSAL>
__device__ void bwd_softmax_role(const BwdParams& p, uint32_t sbase, uint8_t* smem, uint32_t tmem,
                                 const Waiter& wt, const TileRing& ring, int warp) {
  const uint32_t bars = sbase + C::kOffBar;
  auto bar = [&](int i) { return bars + 8u * i; };
  const int lane = threadIdx.x & 31;
  const int quarter = warp & 3, g = warp >> 2;
  const int r = quarter * 32 + lane;                            // resident row within the block
  const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);  // this warp's lane quarter
  float* vec = reinterpret_cast<float*>(smem + C::kOffVec + warp * C::kVecBytes);   // -lse2[64], -delta[64]
  const float c = p.c;
  const uint64_t c2 = ptx::f2pack(c, c);

  uint32_t it = 0, acount = 0;
  int w = 0;
  for (int jt = 0; next_tile(ring, wt, jt, C::kTileRing, true, lane == 0, w); ++jt) {
    const BwdTile ti = bwd_tile<C::DQ, CAUSAL>(p, w);
    if (!ti.live) continue;
    const int row = ti.r0 + r;                         // resident row within the sequence
    const bool row_ok = row < (C::DQ ? ti.Lq : ti.Lk);
    const int64_t tok = (int64_t)ti.rtok + row;
    // dr1: dQ or dK (every mode but dV alone); dr2: dV (dK/dV and dV alone)
    uint16_t* out1 = C::MODE != kBwdDV ? reinterpret_cast<uint16_t*>(p.dr1) + (tok * p.H + ti.h) * C::D : nullptr;
    uint16_t* out2 = C::kStoreP ? reinterpret_cast<uint16_t*>(p.dr2) + (tok * p.H + ti.h) * C::D : nullptr;
    if (ti.n_t == 0) {
      // no pair of this block is visible: zero gradient rows
      if (C::MODE == kBwdDKDV) {
        zero_row<C::KIND>(g == 0 ? out1 : out2, C::D, row_ok);
      } else {
        zero_row<C::KIND>((C::MODE == kBwdDV ? out2 : out1) + g * (C::D / 2), C::D / 2, row_ok);
      }
      continue;
    }
    const int shift = ti.Lk - ti.Lq;
    // dQ kernel: this row's constants; visible keys [0, k_hi)
    float nl_row = 0.f, nd_row = 0.f;
    int k_hi = 0;
    // dK/dV kernel: this key's visible queries [q_lo, Lq)
    int q_lo = 0;
    if (C::DQ) {
      if (row_ok) {
        const int64_t qi = (int64_t)ti.h * p.total_q + tok;
        nl_row = -__ldg(p.lse2 + qi);
        nd_row = -__ldg(p.delta + qi);
      }
      k_hi = row_ok ? (CAUSAL ? min(ti.Lk, row + shift + 1) : ti.Lk) : 0;
    } else {
      q_lo = CAUSAL ? row - shift : 0;
    }
    bool ok = true;
    for (int i = 0; i < ti.n_t; ++i, ++it) {
      const int tb = ti.t_first + i;             // streamed block within the sequence
      const int col0 = 128 * tb + 64 * g;        // first streamed row of this warpgroup's half
      if (!C::DQ) {
        // this warpgroup's 64 query columns: -lse2 and -delta (0 beyond the sequence)
        const float* l2 = p.lse2 + (int64_t)ti.h * p.total_q + ti.ttok;
        const float* dl = p.delta + (int64_t)ti.h * p.total_q + ti.ttok;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int qq = col0 + lane + 32 * k;
          const bool in = qq < ti.Lq;
          vec[lane + 32 * k] = in ? -__ldg(l2 + qq) : 0.f;
          vec[64 + lane + 32 * k] = in ? -__ldg(dl + qq) : 0.f;
        }
        __syncwarp();
      }
      // visible columns of this thread: [lo, hi) relative to col0
      int lo, hi;
      if (C::DQ) {
        lo = 0;
        hi = k_hi - col0;
      } else {
        lo = q_lo - col0;
        hi = row_ok ? ti.Lq - col0 : 0;
      }
      // phase 1: P = exp2(S c - lse2) of this warpgroup's 64 columns, kept in
      // registers; the dK/dV kernel also stores it (16-bit, columns 64 g ..
      // 64 g + 31, already read) for dV += P^T dO. The hand-off also tells
      // the MMA warp that S has been read.
      if (!(ok = wt.wait_warp(bar(C::kBarXFull), it & 1u, 27))) break;
      ptx::tc_fence_after();
      float pv[64];
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t xv[32];
        ptx::tmem_ld32(tl + C::kColX + 64 * g + 32 * ch, xv);
        ptx::tmem_wait_ld();
        ptx::reg_fence(xv);
        const int clo = lo - 32 * ch, chi = hi - 32 * ch;
        const bool masked = clo > 0 || chi < 32;
        float4 nl4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          uint64_t nl2;
          if (C::DQ) {
            nl2 = ptx::f2pack(nl_row, nl_row);
          } else {
            // one 16-byte broadcast load serves two column pairs
            if ((j & 3) == 0) nl4 = *reinterpret_cast<const float4*>(vec + 32 * ch + j);
            nl2 = (j & 3) == 0 ? ptx::f2pack(nl4.x, nl4.y) : ptx::f2pack(nl4.z, nl4.w);
          }
          float e0, e1;
          ptx::f2unpack(ptx::fma2(ptx::f2pack(__uint_as_float(xv[j]), __uint_as_float(xv[j + 1])), c2, nl2),
                        e0, e1);
          float p0 = ptx::ex2(e0), p1 = ptx::ex2(e1);
          if (masked) {
            p0 = (j >= clo && j < chi) ? p0 : 0.f;
            p1 = (j + 1 >= clo && j + 1 < chi) ? p1 : 0.f;
          }
          pv[32 * ch + j] = p0;
          pv[32 * ch + j + 1] = p1;
        }
        if (C::kStoreP) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) pk[j] = pack16<C::KIND>(pv[32 * ch + 2 * j], pv[32 * ch + 2 * j + 1]);
          ptx::tmem_st16(tl + C::kColX + 64 * g + 16 * ch, pk);
        }
      }
      if (C::kStoreP) ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(C::kBarPFull));
      if (!C::kNeedY) continue;   // dV alone: no dP, no dS
      // phase 2: dS = P (dP - Delta), 16-bit, over dP (columns 64 g .. 64 g + 31)
      if (!(ok = wt.wait_warp(bar(C::kBarYFull), it & 1u, 28))) break;
      ptx::tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t yv[32];
        ptx::tmem_ld32(tl + C::kColY + 64 * g + 32 * ch, yv);
        ptx::tmem_wait_ld();
        ptx::reg_fence(yv);
        uint32_t pk[16];
        float4 nd4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          uint64_t nd2;
          if (C::DQ) {
            nd2 = ptx::f2pack(nd_row, nd_row);
          } else {
            if ((j & 3) == 0) nd4 = *reinterpret_cast<const float4*>(vec + 64 + 32 * ch + j);
            nd2 = (j & 3) == 0 ? ptx::f2pack(nd4.x, nd4.y) : ptx::f2pack(nd4.z, nd4.w);
          }
          const uint64_t t = ptx::add2(ptx::f2pack(__uint_as_float(yv[j]), __uint_as_float(yv[j + 1])), nd2);
          float d0, d1;
          ptx::f2unpack(ptx::mul2(ptx::f2pack(pv[32 * ch + j], pv[32 * ch + j + 1]), t), d0, d1);
          pk[j >> 1] = pack16<C::KIND>(d0, d1);
        }
        ptx::tmem_st16(tl + C::kColY + 64 * g + 16 * ch, pk);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(C::kBarDSFull));
    }
    if (!ok) return;
    if (!wt.wait_warp(bar(C::kBarAccFull), acount & 1u, 29)) return;
    ++acount;
    ptx::tc_fence_after();
    if (C::MODE == kBwdDKDV) {
      if (g == 0)
        store_acc_row<C::KIND>(tl + C::kColAcc1, C::D, p.scale, out1, row_ok);   // dK
      else
        store_acc_row<C::KIND>(tl + C::kColAcc2, C::D, 1.f, out2, row_ok);       // dV
    } else if (C::MODE == kBwdDV) {
      // each warpgroup writes half of the row
      store_acc_row<C::KIND>(tl + C::kColAcc2 + g * (C::D / 2), C::D / 2, 1.f, out2 + g * (C::D / 2), row_ok);
    } else {
      store_acc_row<C::KIND>(tl + C::kColAcc1 + g * (C::D / 2), C::D / 2, p.scale, out1 + g * (C::D / 2), row_ok);
    }
    // the next tile's first accumulating MMAs overwrite these columns only
    // after this warp's next P and dS hand-offs
    ptx::tc_fence_before();
  }
}

// ------------------------------------------------------------------ kernel
template <int D, int STAGES, int KIND, int MODE, bool CAUSAL>
__global__ void __launch_bounds__(320, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tr1, const __grid_constant__ CUtensorMap tr2,
                  const __grid_constant__ CUtensorMap tt1, const __grid_constant__ CUtensorMap tt2,
                  const BwdParams p) {
  using C = BwdCfg<D, STAGES, KIND, MODE>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  if (threadIdx.x == 0) {
    const uint32_t bars = sbase + C::kOffBar;
    for (int i = 0; i < C::kNumBars; ++i) {
      uint32_t count = 1;
      if (i == C::kBarPFull || i == C::kBarDSFull) count = C::kSoftmaxWarps;
      if (i >= C::kBarTileEmpty) count = C::kTileConsumers;
      ptx::mbar_init(bars + 8u * i, count);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == C::kLoadWarp && lane == 0) {
    ptx::prefetch_tmap(&tr1);
    ptx::prefetch_tmap(&tr2);
    ptx::prefetch_tmap(&tt1);
    ptx::prefetch_tmap(&tt2);
  }
  if (warp == C::kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_holder), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const Waiter wt{abort_flag, p.status};
  const TileRing ring{sbase + C::kOffBar + 8u * C::kBarTileFull, sbase + C::kOffBar + 8u * C::kBarTileEmpty,
                      reinterpret_cast<volatile int*>(smem + C::kOffMisc + 16)};
  if (warp == C::kLoadWarp) {
    if (lane == 0) bwd_load_role<C, CAUSAL>(&tr1, &tr2, &tt1, &tt2, p, sbase, wt, ring);
  } else if (warp == C::kMmaWarp) {
    if (lane == 0) bwd_mma_role<C, CAUSAL>(p, sbase, tmem, wt, ring);
  } else {
    bwd_softmax_role<C, CAUSAL>(p, sbase, smem, tmem, wt, ring, warp);
  }
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
      atomicExch(p.sched, 0u);
      atomicExch(p.sched + 1, 0u);
    }
  }
}

template <int D, int STAGES, int KIND, int MODE>
cudaError_t launch_bwd_dir(const BwdLaunch& L) {
  using C = BwdCfg<D, STAGES, KIND, MODE>;
  auto kern = L.causal ? fa_bwd_kernel<D, STAGES, KIND, MODE, true> : fa_bwd_kernel<D, STAGES, KIND, MODE, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = L.p.ntiles < L.num_sms ? L.p.ntiles : L.num_sms;
  if (grid <= 0) return cudaSuccess;
  kern<<<grid, C::kThreads, C::kSmemBytes, L.stream>>>(L.tr1, L.tr2, L.tt1, L.tt2, L.p);
  return cudaGetLastError();
}

template <int D, int STAGES_KV, int STAGES_Q>
cudaError_t launch_bwd_impl(const BwdLaunch& L) {
  if (L.kind == kF16)
    return L.dq ? launch_bwd_dir<D, STAGES_Q, kF16, kBwdDQ>(L) : launch_bwd_dir<D, STAGES_KV, kF16, kBwdDKDV>(L);
  return L.dq ? launch_bwd_dir<D, STAGES_Q, kBF16, kBwdDQ>(L) : launch_bwd_dir<D, STAGES_KV, kBF16, kBwdDKDV>(L);
}

}  // namespace fa
