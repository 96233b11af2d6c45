// Exact tiled attention forward for sm_103a (GB300).
//
// O = softmax(scale * Q K^T [+ causal mask]) V and LSE = ln sum exp(scale * Q K^T),
// computed tile by tile with the online-softmax running max / sum recurrence
// ("Flash Attention 3 principles (guijiagi)", sections 2.1-2.2 and 3.1: Q is
// split into 128-row tiles that each CTA owns end to end, K/V stream through
// on-chip memory in 128-row tiles, only O and LSE are written back).
//
// One persistent CTA per SM runs a sequence of work tiles. Each work tile is
// QT query tiles of 128 rows of one (sequence, head) -- QT = 2 for D <= 128,
// 1 for D = 256 -- and the CTA's warps have fixed roles:
//
//   softmax warpgroups (4 warps per query tile, thread r owns row r)
//       tcgen05.ld the fp32 score row from tensor memory, mask, row max,
//       lazy rescale of O (only when the row max grows by more than kTau in
//       log2 units), P = exp2(S * scale * log2 e - m), row sum, P -> 16-bit
//       (or e4m3), tcgen05.st P back into tensor memory over its scores; at
//       the end of the work tile O / l and LSE are written to global memory.
//   MMA warp (one thread)
//       tcgen05.mma: S_t = Q_t K_j^T (both operands in shared memory) and
//       O_t += P_t V_j (P from tensor memory, V from shared memory),
//       accumulators in tensor memory; tcgen05.commit signals mbarriers. For
//       QT = 2 the issue order QK0_j, PV1_{j-1}, QK1_j, PV0_j keeps the tensor
//       core busy while the two softmax warpgroups take turns (the ping-pong
//       of the FlashAttention-3 wiki, technique 1, done with two tensor-memory
//       score buffers instead of two register files).
//   load warp (one thread; a whole warp, plus a V-load warp, for paged K/V)
//       TMA loads of the Q tiles and of K_j, V_j into a ring of shared-memory
//       slots guarded by full / empty mbarriers (producer / consumer of the
//       wiki's technique 1; multi-stage K/V pipeline of technique 2). Paged
//       K/V: two whole warps, one for Q and K, one for V (a block of small
//       pages is many small copies, and one warp issues them one at a time).
//
// Input kinds: fp16 or bf16 (tcgen05 kind::f16, 16 keys per MMA step), or
// e4m3 with per-128-row-block scales (kind::f8f6f4, 32 keys per step; the
// FlashAttention-3 wiki, technique 3). For e4m3 the block scales are folded
// into the per-tile softmax constant (q_s * k_s) and into P (v_s relative to
// the head's largest V scale) so the MMAs run on raw codes.
//
// Every wait on an mbarrier is bounded: after kWaitLimitNs the waiting role
// records a timeout in the device status word, raises an abort flag that the
// other roles see, and all roles leave; tensor memory is freed on the way out.
#pragma once

#include <cstdint>
#include <math_constants.h>

#include "fa_internal.h"
#include "pipeline.cuh"
#include "ptx.cuh"

namespace fa {

template <int D_, int QT_, int STAGES_, int KIND_>
struct FwdCfg {
  static constexpr int D = D_;
  static constexpr int QT = QT_;
  static constexpr int STAGES = STAGES_;
  static constexpr int KIND = KIND_;
  static constexpr bool kFp8 = KIND == kE4M3;
  static constexpr int EB = kFp8 ? 1 : 2;          // bytes per input element
  static constexpr int kRows = 128 * QT;            // query rows per work tile
  // a tile is D / kBoxCols TMA boxes of 128 rows; a box row is 128 bytes in
  // the 128-byte swizzle, or 64 bytes in the 64-byte swizzle when a whole row
  // is 64 bytes (e4m3 at D = 64)
  static constexpr int kRowBytes = D * EB < 128 ? D * EB : 128;   // bytes per box row
  static constexpr int kBoxCols = kRowBytes / EB;   // elements per box row
  static constexpr int kBoxes = D / kBoxCols;       // boxes per 128-row tile
  static constexpr int kBoxBytes = 128 * kRowBytes; // one box: 128 rows
  static constexpr int kTileBytes = kBoxes * kBoxBytes;
  static constexpr int kQkSteps = D * EB / 32;      // MMA K steps (32 bytes each) over D
  static constexpr int kKeysPerStep = 32 / EB;      // keys per PV MMA step
  static constexpr int kPvSteps = 128 / kKeysPerStep;
  // lazy-rescale threshold (log2 units) and, for e4m3, the power of two P is
  // scaled by before it is rounded (P * 2^kappa <= 2^(tau + kappa) = 256 < 448)
  static constexpr float kTau = kFp8 ? 4.0f : 8.0f;
  // P goes to the MMA warp in one piece. Handing e4m3 P over in two halves of
  // 64 keys, so that the first half's products start while the second is
  // made, bought nothing measurable (same box, c5 attention 1659 with halves
  // against 1652 in one piece; c2 1494 against 1506 TFLOP/s)
  static constexpr float kKappaScale = kFp8 ? 16.0f : 1.0f;
  static constexpr float kLog2Kappa = kFp8 ? 4.0f : 0.0f;
  static constexpr int kSoftmaxWarps = 4 * QT;
  static constexpr int kMmaWarp = kSoftmaxWarps;
  static constexpr int kLoadWarp = kSoftmaxWarps + 1;
  static constexpr int kVLoadWarp = kSoftmaxWarps + 2;   // paged K/V only: the V loads
  // QT = 2: a third warpgroup (MMA warp, load warp, V-load warp, one idle
  // warp) gives its registers to the two softmax warpgroups: 384 threads
  // launch at 168 registers each (64512); 128 x 64 + 256 x 216 = 63488 <= 64512.
  static constexpr bool kRebalance = QT == 2;
  // QT = 2, 16-bit: softmax warpgroup 1 frees the K/V ring slots when it sees
  // S1 (K of the block and V of the one before have been read by then), which
  // takes two commits per block off the MMA thread (a commit costs it about
  // as much as a product): c2 1456 -> 1491 TFLOP/s, same box. The e4m3
  // kernel, whose softmax is the critical path, keeps the commits (1650
  // against 1632 with the softmax release).
  static constexpr bool kSoftmaxFreesKV = QT == 2 && !kFp8;
  static constexpr int kRegsLow = 64, kRegsHigh = 216;
  static constexpr int kThreads = kRebalance ? 384 : 32 * (kSoftmaxWarps + 3);
  static_assert(!kRebalance || kThreads * 168 >= 128 * kRegsLow + 256 * kRegsHigh, "register split");
  static constexpr int kTmemCols = 512;
  // tensor-memory columns: score buffers S0, S1; accumulators O0 (, O1)
  __host__ __device__ static constexpr uint32_t col_s(uint32_t b) { return b ? 128u : 0u; }
  __host__ __device__ static constexpr uint32_t col_o(uint32_t t) { return 256u + t * D; }
  // shared memory (offsets from a 1024-byte aligned base)
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = QT * kTileBytes;
  // O leaves through shared memory and TMA stores (a 128-row x 64-column
  // 16-bit box per softmax warpgroup, 128-byte swizzle) when the query tile
  // is whole. Kept out of: the one-tile configurations of short query
  // sequences (decode), whose tiles are almost never whole and whose K/V ring
  // fills shared memory, and the e4m3 kernel, whose per-thread epilogue with
  // four chunk loads under one wait measured faster (same box, c5 attention
  // 1660 against 1638 TFLOP/s; 16-bit c2 1433 -> 1451, c4 1244 -> 1263)
  static constexpr bool kTmaStore = !kFp8 && (QT == 2 || D == 256);
  static constexpr int kEpiBytes = 128 * 128;
  static constexpr int kOffEpi = kOffKV + STAGES * kTileBytes;
  static constexpr int kOffBar = kOffEpi + (kTmaStore ? QT * kEpiBytes : 0);
  // barriers: q_full[2], q_empty[2] (per query tile, so the next work tile's
  // first Q tile loads while this one's last MMAs run), kv_full[S], kv_empty[S], s_full[2],
  // p_full[2] (per score buffer),
  // o_full[2], pv_done, mma_done, tile_full[R], tile_empty[R]
  static constexpr int kTileRing = 4;   // work tiles fetched ahead by the load warp
  static constexpr int kBarQFull = 0, kBarQEmpty = 2, kBarKVFull = 4, kBarKVEmpty = 4 + STAGES,
                       kBarSFull = 4 + 2 * STAGES, kBarPFull = kBarSFull + 2,
                       kBarOFull = kBarPFull + 2, kBarPVDone = kBarOFull + 2,
                       kBarMmaDone = kBarPVDone + 1, kBarTileFull = kBarMmaDone + 1,
                       kBarTileEmpty = kBarTileFull + kTileRing, kNumBars = kBarTileEmpty + kTileRing;
  // MMA thread + one lane per softmax warp (+ the V-load warp with paged K/V)
  static constexpr int kTileConsumers = 1 + kSoftmaxWarps;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;   // tmem address, abort flag, tile ring
  static constexpr int kSmemBytes = kOffMisc + 16 + 4 * kTileRing + 1024;

  static_assert(D == 64 || D == 128 || D == 256, "head dimension");
  static_assert(kRowBytes == 128 || kRowBytes == 64, "box rows of 128 or 64 bytes");
  static_assert(D % kBoxCols == 0, "a 128-row tile must be whole boxes");
  static_assert(QT == 1 || 2 * 128 + QT * D <= kTmemCols, "tensor memory budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Work tile: CTA query block of one (sequence, head).
struct TileInfo {
  int b, h;
  int split;       // key range (split-KV) of this tile, 0 without split
  int kb0;         // first 128-key block of the range
  int qblk;        // CTA query block index within the sequence
  int q0;          // first query row of the block within its sequence
  int Lq, Lk;      // sequence lengths
  int qtok, ktok;  // token index of row 0 of the sequence in Q/O and in K/V
  int n_kv;        // key blocks of 128 to visit
  bool live;       // false: the block starts beyond the sequence
};

// Heads are the outer loop (in groups of p.head_group, tile_order) so that
// the CTAs running at the same time share their K/V through L2; under the
// causal mask the blocks of a head are ranked from the most expensive (last
// rows) to the cheapest.
template <int ROWS, bool CAUSAL>
__device__ __forceinline__ TileInfo tile_info(const FwdParams& p, int w) {
  TileInfo t;
  const int per_head = p.n_qblk * p.n_split;
  int bh, jj;
  tile_order(w, per_head, p.B * p.H, p.head_group, bh, jj);
  const int j = jj / p.n_split;
  t.split = jj - j * p.n_split;
  const int qblk = CAUSAL ? (p.n_qblk - 1 - j) : j;
  t.qblk = qblk;
  t.b = bh / p.H;
  t.h = bh - t.b * p.H;
  if (p.block_table != nullptr) {
    // paged K/V: keys from seqlens_k through the block table; queries of a
    // fixed length, or packed by cu_q
    int qs = t.b * p.Sq, qe = qs + p.Sq;
    if (p.cu_q != nullptr) {
      qs = __ldg(p.cu_q + t.b);
      qe = __ldg(p.cu_q + t.b + 1);
    }
    t.qtok = qs;
    t.ktok = 0;
    t.Lq = qe - qs;
    t.Lk = __ldg(p.seqlens_k + t.b);
    if (qs < 0 || qe < qs || qe > p.total_q || t.Lq > p.Sq || t.Lk < 0 || t.Lk > p.Sk) {
      t.Lq = 0;
      t.Lk = 0;
      if (qblk == 0) atomicOr(p.status, kDevBadSeqlens);
    }
  } else if (p.cu_q != nullptr) {
    const int qs = __ldg(p.cu_q + t.b), qe = __ldg(p.cu_q + t.b + 1);
    const int ks = __ldg(p.cu_k + t.b), ke = __ldg(p.cu_k + t.b + 1);
    t.qtok = qs;
    t.ktok = ks;
    t.Lq = qe - qs;
    t.Lk = ke - ks;
    // a sequence that breaks the declared bounds is skipped (and reported)
    bool bad = qs < 0 || qe < qs || qe > p.total_q || ks < 0 || ke < ks || ke > p.total_k ||
               t.Lq > p.Sq || t.Lk > p.Sk;
    if (!bad && p.cu_blocks_q != nullptr) {
      // e4m3 block-scale offsets: this sequence's entries must span exactly its
      // blocks and stay inside the first total / 128 + B rows of the
      // [n_blocks, H] scale arrays
      const int bq0 = __ldg(p.cu_blocks_q + t.b), bq1 = __ldg(p.cu_blocks_q + t.b + 1);
      const int bk0 = __ldg(p.cu_blocks_k + t.b), bk1 = __ldg(p.cu_blocks_k + t.b + 1);
      const int bqn = __ldg(p.cu_blocks_q + p.B), bkn = __ldg(p.cu_blocks_k + p.B);
      bad = bq0 < 0 || bq1 - bq0 != (t.Lq + 127) / 128 || bq1 > bqn || bqn > p.total_q / 128 + p.B ||
            bk0 < 0 || bk1 - bk0 != (t.Lk + 127) / 128 || bk1 > bkn || bkn > p.total_k / 128 + p.B;
    }
    if (bad) {
      t.Lq = 0;
      t.Lk = 0;
      if (qblk == 0) atomicOr(p.status, kDevBadSeqlens);
    }
  } else {
    t.qtok = t.b * p.Sq;
    t.ktok = t.b * p.Sk;
    t.Lq = p.Sq;
    t.Lk = p.Sk;
  }
  t.q0 = qblk * ROWS;
  t.live = t.q0 < t.Lq;
  t.kb0 = t.split * p.split_blocks;
  int n = 0;
  if (t.live) {
    const int last = min(t.q0 + ROWS, t.Lq) - 1;
    int lim = t.Lk;
    if (CAUSAL) lim = min(lim, last + t.Lk - t.Lq + 1);
    const int kb1 = min(lim > 0 ? (lim + 127) / 128 : 0, t.kb0 + p.split_blocks);
    n = max(kb1 - t.kb0, 0);
  }
  t.n_kv = n;
  return t;
}

template <int R>
__device__ __forceinline__ int fetch_tile(const FwdParams& p, int j) {
  const int w = j == 0 ? (int)blockIdx.x : (int)gridDim.x + (int)atomicAdd(p.sched, 1u);
  return w < p.ntiles ? w : -1;
}

// ------------------------------------------------------------------ load warp
// MODE 0, contiguous K/V: lane 0 of the load warp alone runs this role (the
// idle lanes would cost the contiguous one-tile configuration issue slots,
// measured 6 % at D = 256). Paged K/V: two whole warps, MODE 1 (the load
// warp: work tiles into the ring, Q, K) and MODE 2 (the V-load warp: takes
// the work tiles from the ring like the other consumers, loads V). In each,
// lane 0 does the waits and every lane s < 128 / page_rows looks up, and
// loads, box s of a tile itself, so a tile's block-table reads and copies are
// issued in parallel. Each warp issues its copies one after another (about 55
// cycles each, measured), so at 16-row pages one warp for both K and V was the
// limit. Both paged warps walk the same ring-slot sequence (K0, V0, K1, ... or
// K0, K1, V0, K2, ...) and act on their own tensor's slots only; every fill
// of a slot waits for the consumption of the one before it.
template <class C, bool CAUSAL, int MODE>
__device__ void load_role(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                          const FwdParams& p, uint32_t sbase, const Waiter& wt, const TileRing& ring) {
  const uint32_t bars = sbase + C::kOffBar;
  auto bar = [&](int i) { return bars + 8u * i; };
  const int lane = threadIdx.x & 31;
  const bool lead = lane == 0;
  constexpr bool paged = MODE != 0;
  constexpr bool do_k = MODE != 2, do_v = MODE != 1;
  const unsigned lanes = paged ? 0xffffffffu : 1u;   // the lanes running this role
  uint32_t kvc = 0, tcount = 0;
  uint32_t acted = 0;   // bit i: this warp filled slot kvc - 1 - i
  bool ok = true;
  // lane 0 waits; every participating lane learns the outcome
  auto wait0 = [&](uint32_t b, uint32_t parity, int where) -> bool {
    bool r = true;
    if (lead) r = wt.wait(b, parity, where);
    return __shfl_sync(lanes, r ? 1 : 0, 0) != 0;
  };

  auto load_tile = [&](const CUtensorMap* m, int h, int row, uint32_t dst, uint32_t b) {
#pragma unroll
    for (int bx = 0; bx < C::kBoxes; ++bx)
      ptx::tma_load_2d(dst + bx * C::kBoxBytes, m, h * C::D + bx * C::kBoxCols, row, b);
  };
  // paged K/V: lane s's row for box s of a 128-key block, looked up once per
  // block (K and V share it). The one-query-tile configuration caches two
  // blocks (entries A and B), since its order K0, K1, V0, K2, V1, ...
  // alternates between two; the two-tile one needs entry A only. page_fetch
  // issues the lane's block-table read before lane 0 waits for a free slot,
  // page_rows turns it into a row after the wait, so the read's latency hides
  // behind the wait. Page sizes that are powers of two divide by shifting.
  const int nsub = paged ? 128 / p.page_rows : 0;
  const bool my_box = lane < nsub;
  int tag_a = -1, tag_b = -1;       // pack_tag of the cached blocks
  int row_a = 0, row_b = 0;
  bool raw_a = false, raw_b = false, next_a = true, use_a = true;
  auto pack_tag = [&](const TileInfo& ti, int kb) { return ti.b * p.n_kblk_tag + kb; };
  auto page_fetch = [&](const TileInfo& ti, int kb) {
    const int tag = pack_tag(ti, kb);
    if (tag == tag_a) { use_a = true; return; }
    if (C::QT == 1 && tag == tag_b) { use_a = false; return; }
    // two query tiles load K_i, V_i in pairs: one entry is enough
    use_a = C::QT == 2 ? true : next_a;
    next_a = !next_a;
    const int key = 128 * kb + lane * p.page_rows;
    int pg = -2;   // -2: a box past the sequence
    if (my_box && key < ti.Lk) {
      const int pi = p.page_shift >= 0 ? key >> p.page_shift : key / p.page_size;
      pg = __ldg(p.block_table + (int64_t)ti.b * p.max_pages + pi);
    }
    if (use_a) { row_a = pg; tag_a = tag; raw_a = true; } else { row_b = pg; tag_b = tag; raw_b = true; }
  };
  auto page_rows = [&](int kb) -> int {
    int& row = use_a ? row_a : row_b;
    bool& raw = use_a ? raw_a : raw_b;
    if (raw) {
      const int key = 128 * kb + lane * p.page_rows;
      const int in_page = p.page_shift >= 0 ? key & (p.page_size - 1) : key % p.page_size;
      const int pg = row;
      row = p.num_pages * p.page_size;   // past the cache: TMA fills zeros
      if (pg >= 0 && pg < p.num_pages)
        row = pg * p.page_size + in_page;
      else if (pg != -2)
        atomicOr(p.status, kDevBadSeqlens);
      raw = false;
    }
    return row;
  };
  // K or V tile of 128-key block kb (absolute within the sequence); a tile
  // of the other paged warp's tensor only takes its place in the slot order
  bool first_tile = true;   // this CTA's first work tile (the test build's withheld tile)
  auto load_kv = [&](const CUtensorMap* m, const TileInfo& ti, int kb, bool act) -> bool {
#ifdef FA_TEST_WITHHOLD_KV
    // test build only: CTA 0 never loads the K tile of key block
    // p.test_withhold_kb of its first work tile -- no expected bytes, no copy,
    // so nothing can land later -- and the MMA thread's bounded wait for it
    // runs out; the release build has no such path
    if (act && m == tk && blockIdx.x == 0 && first_tile && kb == p.test_withhold_kb) act = false;
#endif
    acted = (acted << 1) | (act ? 1u : 0u);
    if (!act) {
      ++kvc;
      return true;
    }
    const int s = kvc % C::STAGES;
    const uint32_t ph = (kvc / C::STAGES) & 1u;
    if (paged) page_fetch(ti, kb);
    if (!wait0(bar(C::kBarKVEmpty + s), ph ^ 1u, 2)) return false;
    const uint32_t dst = sbase + C::kOffKV + s * C::kTileBytes, b = bar(C::kBarKVFull + s);
    if (lead) ptx::mbar_arrive_expect_tx(b, C::kTileBytes);
    if (!paged) {
      if (lead) load_tile(m, ti.h, ti.ktok + 128 * kb, dst, b);
    } else {
      // paged: page_rows-row boxes, each from its page; rows past the
      // sequence (or a bad page entry) point past the cache, where TMA fills
      // zeros. page_rows is a multiple of 16, so every box starts on a
      // 2 KB boundary of the swizzled tile. The expected byte count is set
      // before any lane's copy is issued.
      const int row = page_rows(kb);
      __syncwarp(lanes);
      if (my_box) {
#pragma unroll
        for (int bx = 0; bx < C::kBoxes; ++bx)
          ptx::tma_load_2d(dst + bx * C::kBoxBytes + lane * p.page_rows * C::kRowBytes, m, ti.h * C::D + bx * C::kBoxCols,
                           row, b);
      }
    }
    ++kvc;
    return true;
  };

  for (int j = 0; ok; ++j) {
    int w = 0;
    if (MODE == 2) {
      // the V-load warp takes the work tiles from the ring
      if (!next_tile(ring, wt, j, C::kTileRing, true, lead, w)) break;
    } else {
      const int rs = j % C::kTileRing;
      if (!wait0(ring.empty(rs), ((j / C::kTileRing) & 1u) ^ 1u, 9)) break;
      if (lead) {
        w = fetch_tile<C::kTileRing>(p, j);
        ring.slots[rs] = w;
        ptx::mbar_arrive(ring.full(rs));
      }
      w = __shfl_sync(lanes, w, 0);
      if (w < 0) break;
    }
    const TileInfo ti = tile_info<C::kRows, CAUSAL>(p, w);
    first_tile = j == 0;
    if (ti.n_kv == 0) continue;
    if (MODE != 2) {
#pragma unroll
      for (int t = 0; t < C::QT; ++t) {
        if (!wait0(bar(C::kBarQEmpty + t), (tcount & 1u) ^ 1u, 1)) { ok = false; break; }
        if (lead) {
          ptx::mbar_arrive_expect_tx(bar(C::kBarQFull + t), C::kTileBytes);
          load_tile(tq, ti.h, ti.qtok + ti.q0 + 128 * t, sbase + C::kOffQ + t * C::kTileBytes,
                    bar(C::kBarQFull + t));
        }
      }
      if (!ok) break;
      ++tcount;
    }
    const int n = ti.n_kv;
    const int kb0 = ti.kb0;   // first key block of the tile's range
    if (C::QT == 2) {
      // consumption order of the MMA warp: K0, V0, K1, V1, ...
      for (int i = 0; ok && i < n; ++i) {
        ok = load_kv(tk, ti, kb0 + i, do_k) && load_kv(tv, ti, kb0 + i, do_v);
      }
    } else {
      // consumption order: K0, K1, V0, K2, V1, ..., V_{n-1}
      ok = load_kv(tk, ti, kb0, do_k);
      for (int i = 0; ok && i < n; ++i) {
        if (i + 1 < n) ok = load_kv(tk, ti, kb0 + i + 1, do_k);
        if (ok) ok = load_kv(tv, ti, kb0 + i, do_v);
      }
    }
  }
  if (lead && *wt.abort_flag) {
    // let the copies still in flight land before the CTA's memory goes away
    // (each paged warp drains the slots it filled itself)
    const uint32_t first = kvc > (uint32_t)C::STAGES ? kvc - C::STAGES : 0u;
    for (uint32_t c = first; c < kvc; ++c)
      if ((acted >> (kvc - 1u - c)) & 1u) wt.drain(bar(C::kBarKVFull + (int)(c % C::STAGES)), (c / C::STAGES) & 1u);
    if (MODE != 2)
      for (int t = 0; t < C::QT && tcount > 0; ++t) wt.drain(bar(C::kBarQFull + t), (tcount - 1) & 1u);
  }
}

// ------------------------------------------------------------------ MMA warp
template <class C, bool CAUSAL>
__device__ void mma_role(const FwdParams& p, uint32_t sbase, uint32_t tmem, const Waiter& wt,
                         const TileRing& ring) {
  const uint32_t bars = sbase + C::kOffBar;
  auto bar = [&](int i) { return bars + 8u * i; };
  // operand format field: kind::f16 0 = f16, 1 = bf16; kind::f8f6f4 0 = e4m3
  constexpr uint32_t fmt = C::KIND == kBF16 ? 1u : 0u;
  constexpr uint32_t idesc_qk = ptx::make_idesc(fmt, false, 128, 128);
  constexpr uint32_t idesc_pv = ptx::make_idesc(fmt, true, 128, C::D);
  const uint32_t sq = sbase + C::kOffQ;
  auto slot_addr = [&](uint32_t c) { return sbase + C::kOffKV + (c % C::STAGES) * C::kTileBytes; };
  auto slot = [&](uint32_t c) { return (int)(c % C::STAGES); };

  // S[s_col] = Q_t K^T : steps of 32 bytes of the head dimension (16 f16 or 32 e4m3)
  auto qk = [&](uint32_t s_col, uint32_t q_addr, uint32_t k_addr) {
#pragma unroll
    for (int kk = 0; kk < C::kQkSteps; ++kk) {
      constexpr int kStepsPerBox = C::kRowBytes / 32;
      const uint32_t off = (kk / kStepsPerBox) * C::kBoxBytes + (kk % kStepsPerBox) * 32;
      const uint64_t a = ptx::smem_desc_sw<C::kRowBytes>(q_addr + off, 16, 8 * C::kRowBytes);
      const uint64_t b = ptx::smem_desc_sw<C::kRowBytes>(k_addr + off, 16, 8 * C::kRowBytes);
      if (C::kFp8)
        ptx::mma_f8_ss(tmem + s_col, a, b, idesc_qk, kk > 0);
      else
        ptx::mma_f16_ss(tmem + s_col, a, b, idesc_qk, kk > 0);
    }
  };
  // O[o_col] (+)= P[p_col] V : steps of kKeysPerStep keys; 8 P columns per
  // step, once P of score buffer pbuf is in tensor memory
  auto pv = [&](uint32_t o_col, uint32_t p_col, uint32_t v_addr, bool acc, int pbuf, uint32_t parity) -> bool {
    if (!wt.wait(bar(C::kBarPFull + pbuf), parity, 5)) return false;
    ptx::tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < C::kPvSteps; ++kk) {
      const uint64_t b = ptx::smem_desc_sw<C::kRowBytes>(v_addr + kk * C::kKeysPerStep * C::kRowBytes,
                                                         C::kBoxBytes, 8 * C::kRowBytes);
      const uint32_t en = (acc || kk > 0) ? 1u : 0u;
      if (C::kFp8)
        ptx::mma_f8_ts(tmem + o_col, tmem + p_col + kk * 8, b, idesc_pv, en);
      else
        ptx::mma_f16_ts(tmem + o_col, tmem + p_col + kk * 8, b, idesc_pv, en);
    }
    return true;
  };
  auto kv_ready = [&](uint32_t c) {
    const bool r = wt.wait(bar(C::kBarKVFull + slot(c)), (c / C::STAGES) & 1u, 4);
    ptx::tc_fence_after();
    return r;
  };

  uint32_t kvc = 0, it = 0, tcount = 0;
  bool ok = true;
  int w = 0;
  for (int j = 0; ok && next_tile(ring, wt, j, C::kTileRing, false, true, w); ++j) {
    const TileInfo ti = tile_info<C::kRows, CAUSAL>(p, w);
    if (ti.n_kv == 0) continue;
    const uint32_t qpar = tcount & 1u;
    if (!wt.wait(bar(C::kBarQFull), qpar, 3)) { ok = false; break; }
    ++tcount;
    ptx::tc_fence_after();
    const int n = ti.n_kv;
    if (C::QT == 2) {
      if (!(ok = kv_ready(kvc))) break;
      qk(C::col_s(0), sq, slot_addr(kvc));
      ptx::mma_commit(bar(C::kBarSFull + 0));
      if (n == 1) ptx::mma_commit(bar(C::kBarQEmpty + 0));   // last use of Q0
      if (!(ok = wt.wait(bar(C::kBarQFull + 1), qpar, 3))) break;
      ptx::tc_fence_after();
      for (int i = 0; i < n; ++i) {
        const uint32_t ck = kvc + 2 * i, cv = ck + 1;
        if (i > 0) {
          if (!(ok = pv(C::col_o(1), C::col_s(1), slot_addr(cv - 2), i - 1 > 0, 1, (it + i - 1) & 1u))) break;
          if (!C::kSoftmaxFreesKV) ptx::mma_commit(bar(C::kBarKVEmpty + slot(cv - 2)));
        }
        qk(C::col_s(1), sq + C::kTileBytes, slot_addr(ck));
        ptx::mma_commit(bar(C::kBarSFull + 1));
        if (!C::kSoftmaxFreesKV) ptx::mma_commit(bar(C::kBarKVEmpty + slot(ck)));
        if (i == n - 1) ptx::mma_commit(bar(C::kBarQEmpty + 1));   // last use of Q1
        if (!(ok = kv_ready(cv))) break;
        if (!(ok = pv(C::col_o(0), C::col_s(0), slot_addr(cv), i > 0, 0, (it + i) & 1u))) break;
        if (i == n - 1) ptx::mma_commit(bar(C::kBarOFull + 0));
        if (i + 1 < n) {
          if (!(ok = kv_ready(ck + 2))) break;
          qk(C::col_s(0), sq, slot_addr(ck + 2));
          ptx::mma_commit(bar(C::kBarSFull + 0));
          if (i + 2 == n) ptx::mma_commit(bar(C::kBarQEmpty + 0));   // last use of Q0
        }
      }
      if (!ok) break;
      const uint32_t cl = kvc + 2 * n - 1;
      if (!(ok = pv(C::col_o(1), C::col_s(1), slot_addr(cl), n - 1 > 0, 1, (it + n - 1) & 1u))) break;
      if (!C::kSoftmaxFreesKV) ptx::mma_commit(bar(C::kBarKVEmpty + slot(cl)));
      ptx::mma_commit(bar(C::kBarOFull + 1));
      kvc += 2 * n;
      it += n;
    } else {
      if (!(ok = kv_ready(kvc))) break;
      qk(C::col_s(it & 1u), sq, slot_addr(kvc));
      ptx::mma_commit(bar(C::kBarSFull + (int)(it & 1u)));
      ptx::mma_commit(bar(C::kBarKVEmpty + slot(kvc)));
      ++kvc;
      if (n == 1) ptx::mma_commit(bar(C::kBarQEmpty));
      for (int i = 0; i < n; ++i) {
        const uint32_t iti = it + i;
        if (i + 1 < n) {
          if (!(ok = kv_ready(kvc))) break;
          qk(C::col_s((iti + 1) & 1u), sq, slot_addr(kvc));
          ptx::mma_commit(bar(C::kBarSFull + (int)((iti + 1) & 1u)));
          ptx::mma_commit(bar(C::kBarKVEmpty + slot(kvc)));
          ++kvc;
          if (i + 1 == n - 1) ptx::mma_commit(bar(C::kBarQEmpty));
        }
        if (!(ok = kv_ready(kvc))) break;
        if (!(ok = pv(C::col_o(0), C::col_s(iti & 1u), slot_addr(kvc), i > 0, (int)(iti & 1u), (iti >> 1) & 1u)))
          break;
        ptx::mma_commit(bar(C::kBarKVEmpty + slot(kvc)));
        ptx::mma_commit(bar(C::kBarPVDone));
        ++kvc;
        if (i == n - 1) ptx::mma_commit(bar(C::kBarOFull + 0));
      }
      it += n;
    }
  }
  // all issued MMAs complete before tensor memory can be released
  ptx::mma_commit(bar(C::kBarMmaDone));
  wt.drain(bar(C::kBarMmaDone), 0);
}

// ------------------------------------------------------------------ softmax warpgroups
template <int KIND>
__device__ __forceinline__ uint32_t pack_out(float lo, float hi) {
  // output element pair: fp16 for fp16 inputs, bf16 otherwise (e4m3 -> bf16 O)
  return KIND == kF16 ? ptx::pack_f16(lo, hi) : ptx::pack_bf16(lo, hi);
}

template <int KIND>
__device__ __forceinline__ uint32_t pack_p16(float lo, float hi) {
  return KIND == kF16 ? ptx::pack_f16(lo, hi) : ptx::pack_bf16(lo, hi);
}

// one warpgroup's named barrier (ids 1, 2; 0 is __syncthreads)
__device__ __forceinline__ void wg_sync(int t) {
  asm volatile("bar.sync %0, 128;" ::"r"(1 + t) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

template <class C, bool CAUSAL>
__device__ void softmax_role(const FwdParams& p, const CUtensorMap* to, uint32_t sbase, uint32_t tmem,
                             const Waiter& wt, const TileRing& ring, int t, int quarter) {
  const uint32_t bars = sbase + C::kOffBar;
  auto bar = [&](int i) { return bars + 8u * i; };
  const int lane = threadIdx.x & 31;
  const int r = quarter * 32 + lane;                            // row within the 128-row tile
  const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);  // this warp's lane quarter
  const float NEG_INF = -CUDART_INF_F;

  uint32_t it = 0, tcount = 0;
  int w = 0;
  for (int jt = 0; next_tile(ring, wt, jt, C::kTileRing, true, lane == 0, w); ++jt) {
    const TileInfo ti = tile_info<C::kRows, CAUSAL>(p, w);
    if (!ti.live) continue;
    const int row = ti.q0 + 128 * t + r;
    const bool row_ok = row < ti.Lq;
    const bool split = p.o_part != nullptr;
    // this row's outputs (formed where they are written, so that they are not
    // held in registers across the key loop)
    auto out_ptrs = [&](uint16_t*& orow, float*& oprow, float*& lse_ptr) {
      const int64_t tok = (int64_t)ti.qtok + row;
      orow = reinterpret_cast<uint16_t*>(p.o) + (tok * p.H + ti.h) * C::D;
      oprow = split ? p.o_part + (((int64_t)ti.split * p.total_q + tok) * p.H + ti.h) * C::D : nullptr;
      lse_ptr = split ? p.lse_part + (((int64_t)ti.split * p.B + ti.b) * p.H + ti.h) * p.Sq + row
                : p.cu_q != nullptr ? p.lse + (int64_t)ti.h * p.total_q + tok
                                    : p.lse + ((int64_t)ti.b * p.H + ti.h) * p.Sq + row;
    };
    if (ti.n_kv == 0) {
      uint16_t* orow;
      float* oprow;
      float* lse_ptr;
      out_ptrs(orow, oprow, lse_ptr);
      // no visible key for any row of this block (or of this key range):
      // O = 0, LSE = -inf
      if (row_ok) {
        if (split) {
          for (int d = 0; d < C::D; d += 4) *reinterpret_cast<float4*>(oprow + d) = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
          for (int d = 0; d < C::D; d += 8) *reinterpret_cast<uint4*>(orow + d) = make_uint4(0, 0, 0, 0);
        }
        *lse_ptr = NEG_INF;
      }
      continue;
    }
    // e4m3: per-tile score constant c * q_s * k_s(j); P weight v_s(j) / v_ref
    float c_q = p.c, v_ref = 1.f;
    const float* ks_row = nullptr;
    const float* vs_row = nullptr;
    int sstride = 1;   // between the scales of consecutive blocks
    if (C::kFp8) {
      // block scales: [B, H, nblk] (fixed length) or [n_blocks, H] (varlen,
      // block g = cu_blocks[b] + blk counted per sequence, heads fastest)
      const int nq = (ti.Lq + 127) / 128, nk = (ti.Lk + 127) / 128;
      const float* qs_row;
      if (p.cu_blocks_q != nullptr) {
        sstride = p.H;
        qs_row = p.q_scale + (int64_t)__ldg(p.cu_blocks_q + ti.b) * p.H + ti.h;
        ks_row = p.k_scale + (int64_t)__ldg(p.cu_blocks_k + ti.b) * p.H + ti.h;
        vs_row = p.v_scale + (int64_t)__ldg(p.cu_blocks_k + ti.b) * p.H + ti.h;
      } else {
        const int64_t hb = (int64_t)ti.b * p.H + ti.h;
        qs_row = p.q_scale + hb * p.nblk_q;
        ks_row = p.k_scale + hb * p.nblk_k;
        vs_row = p.v_scale + hb * p.nblk_k;
      }
      c_q = p.c * __ldg(qs_row + (int64_t)min(ti.qblk * C::QT + t, nq - 1) * sstride);
      // v_ref = the head's largest V block scale: the lanes of the warp take
      // every 32nd block, then a butterfly max
      float vmax = 0.f;
      for (int j = lane; j < nk; j += 32) vmax = fmaxf(vmax, __ldg(vs_row + (int64_t)j * sstride));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
      v_ref = vmax > 0.f ? vmax : 1.f;
    }
    const float inv_vref = 1.f / v_ref;
    const int key_lim = CAUSAL ? min(ti.Lk, row + ti.Lk - ti.Lq + 1) : ti.Lk;
    float m_ref = NEG_INF, l = 0.f;
    bool ok = true;
    // e4m3: the K and V scales of the next block are loaded one block ahead,
    // so their latency is hidden behind this block's softmax
    float ks_next = 0.f, vs_next = 0.f;
    if (C::kFp8) {
      ks_next = __ldg(ks_row + (int64_t)ti.kb0 * sstride);
      vs_next = __ldg(vs_row + (int64_t)ti.kb0 * sstride);
    }
    for (int i = 0; i < ti.n_kv; ++i, ++it) {
      const int kb = ti.kb0 + i;   // absolute 128-key block
      const float ks_cur = ks_next, vs_cur = vs_next;
      if (C::kFp8 && i + 1 < ti.n_kv) {
        ks_next = __ldg(ks_row + (int64_t)(kb + 1) * sstride);
        vs_next = __ldg(vs_row + (int64_t)(kb + 1) * sstride);
      }
      const float c = C::kFp8 ? c_q * ks_cur : c_q;
      // log2 of the factor the stored P carries: 2^kappa * v_s(j) / v_ref (e4m3 only)
      const float lg_pw = C::kFp8 ? ptx::lg2(vs_cur * inv_vref) + C::kLog2Kappa : 0.f;
      const int buf = C::QT == 2 ? t : (int)(it & 1u);
      const uint32_t par = C::QT == 2 ? (it & 1u) : ((it >> 1) & 1u);
      if (!(ok = wt.wait_warp(bar(C::kBarSFull + buf), par, 6))) break;
      ptx::tc_fence_after();
      if (C::kSoftmaxFreesKV && t == 1 && quarter == 0 && lane == 0) {
        // S1 of block `it` proves QK0, QK1 of the block and the PV1 before
        // them done (one thread's products complete in order): K of this
        // block and V of the previous one (it - 1, possibly of the previous
        // work tile) have been read; their ring slots are free
        ptx::mbar_arrive(bar(C::kBarKVEmpty + (int)((2u * it) % C::STAGES)));
        if (it > 0) ptx::mbar_arrive(bar(C::kBarKVEmpty + (int)((2u * it - 1u) % C::STAGES)));
      }
      const uint32_t s_addr = tl + C::col_s(buf);
      uint32_t sv[128];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
        ptx::tmem_ld32(s_addr + 32 * ch, *reinterpret_cast<uint32_t(*)[32]>(sv + 32 * ch));
      ptx::tmem_wait_ld();
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) ptx::reg_fence(*reinterpret_cast<uint32_t(*)[32]>(sv + 32 * ch));
      float s[128];
#pragma unroll
      for (int j = 0; j < 128; ++j) s[j] = __uint_as_float(sv[j]);
      const int lim_local = key_lim - 128 * kb;
      const bool masked = lim_local < 128;  // keys j >= lim_local are not visible
      if (masked) {
#pragma unroll
        for (int j = 0; j < 128; ++j) s[j] = j < lim_local ? s[j] : NEG_INF;
      }
      // row max as a tree of three-input maxima, 128 -> 43 -> 15 -> 5 -> 2 -> 1:
      // the same 65 instructions as four running maxima, five deep instead
      // of sixteen (same box, c5 attention 1652 -> 1658 TFLOP/s, the 16-bit
      // rows unchanged)
      float mx1[43], mx2[15], mx3[5];
#pragma unroll
      for (int q = 0; q < 42; ++q) mx1[q] = ptx::max3(s[3 * q], s[3 * q + 1], s[3 * q + 2]);
      mx1[42] = fmaxf(s[126], s[127]);
#pragma unroll
      for (int q = 0; q < 14; ++q) mx2[q] = ptx::max3(mx1[3 * q], mx1[3 * q + 1], mx1[3 * q + 2]);
      mx2[14] = mx1[42];
#pragma unroll
      for (int q = 0; q < 5; ++q) mx3[q] = ptx::max3(mx2[3 * q], mx2[3 * q + 1], mx2[3 * q + 2]);
      const float mt = fmaxf(ptx::max3(mx3[0], mx3[1], mx3[2]), fmaxf(mx3[3], mx3[4]));
      const float m_tile = mt == NEG_INF ? NEG_INF : mt * c;  // scaled log2 units (c >= 0)
      if (i == 0) {
        m_ref = m_tile;
      } else {
        const bool need = m_tile > m_ref + C::kTau;
        if (__any_sync(0xffffffffu, need)) {
          if (C::QT == 1) {
            // the previous PV must have landed in O before it is rescaled
            if (!(ok = wt.wait_warp(bar(C::kBarPVDone), (it - 1) & 1u, 8))) break;
            ptx::tc_fence_after();
          }
          const float alpha = need ? ptx::ex2(m_ref - m_tile) : 1.f;
          if (need) {
            m_ref = m_tile;
            l *= alpha;
          }
          const uint64_t a2 = ptx::f2pack(alpha, alpha);
          const uint32_t o_addr = tl + C::col_o(t);
#pragma unroll 1
          for (int ch = 0; ch < C::D / 32; ++ch) {
            uint32_t v[32];
            ptx::tmem_ld32(o_addr + 32 * ch, v);
            ptx::tmem_wait_ld();
            ptx::reg_fence(v);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              float lo, hi;
              ptx::f2unpack(ptx::mul2(ptx::f2pack(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), a2),
                            lo, hi);
              v[j] = __float_as_uint(lo);
              v[j + 1] = __float_as_uint(hi);
            }
            ptx::tmem_st32(o_addr + 32 * ch, v);
          }
          ptx::tmem_wait_st();
        }
      }
      // exponent argument s * c - m (+ log2 of the e4m3 P weight), two lanes
      // at a time, in two halves of 64 keys; P goes to the MMA warp once both
      // sit in tensor memory; the row sum comes after
      const float mu = (m_ref == NEG_INF ? 0.f : m_ref) - lg_pw;
      const uint64_t c2 = ptx::f2pack(c, c), nm2 = ptx::f2pack(-mu, -mu);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
        for (int j = 64 * hf; j < 64 * hf + 64; j += 2) {
          float lo, hi;
          ptx::f2unpack(ptx::fma2(ptx::f2pack(s[j], s[j + 1]), c2, nm2), lo, hi);
          s[j] = ptx::ex2(lo);
          s[j + 1] = ptx::ex2(hi);
        }
        if (masked) {
          // zero the invisible keys after the exponent: with c = 0 their
          // -inf * c would be NaN
#pragma unroll
          for (int j = 64 * hf; j < 64 * hf + 64; ++j) s[j] = j < lim_local ? s[j] : 0.f;
        }
        if (C::kFp8) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int e = 64 * hf + 4 * j;
            pk[j] = ptx::pack_e4m3x4(s[e], s[e + 1], s[e + 2], s[e + 3]);
          }
          ptx::tmem_st16(s_addr + 16 * hf, pk);
        } else {
          uint32_t pk[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) pk[j] = pack_p16<C::KIND>(s[64 * hf + 2 * j], s[64 * hf + 2 * j + 1]);
          ptx::tmem_st32(s_addr + 32 * hf, pk);
        }
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(C::kBarPFull + buf));
      // the row sum on packed pairs as a tree: 32 sums of two pairs, then
      // halving to one pair. 63 packed adds, six deep; four running sums of
      // sixteen pairs each were as many adds, sixteen deep, and the softmax
      // warpgroup's tail after P is handed over paces the next block (same
      // box: c2 1494 -> 1521, c4 1295 -> 1312 TFLOP/s, c5 unchanged)
      uint64_t ps[32];
#pragma unroll
      for (int q = 0; q < 32; ++q)
        ps[q] = ptx::add2(ptx::f2pack(s[4 * q], s[4 * q + 1]), ptx::f2pack(s[4 * q + 2], s[4 * q + 3]));
#pragma unroll
      for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
        for (int q = 0; q < w; ++q) ps[q] = ptx::add2(ps[q], ps[q + w]);
      float a0, a1;
      ptx::f2unpack(ps[0], a0, a1);
      const float tile_sum = a0 + a1;
      {
        // e4m3: the stored P carries the weight 2^lg_pw; l sums unweighted P
        l += C::kFp8 ? tile_sum * ptx::ex2(-lg_pw) : tile_sum;
      }
    }
    if (!ok) return;
    // epilogue: O / l (e4m3: O * v_ref * 2^-kappa / l), LSE
    if (!wt.wait_warp(bar(C::kBarOFull + (C::QT == 2 ? t : 0)), tcount & 1u, 7)) return;
    ++tcount;
    ptx::tc_fence_after();
    const float inv_l = l > 0.f ? (C::kFp8 ? v_ref / (C::kKappaScale * l) : 1.f / l) : 0.f;
    const uint32_t o_addr = tl + C::col_o(C::QT == 2 ? t : 0);
    uint16_t* orow;
    float* oprow;
    float* lse_ptr;
    out_ptrs(orow, oprow, lse_ptr);
    if (C::kTmaStore && !split && ti.q0 + 128 * t + 128 <= ti.Lq) {
      // a whole query tile: O / l in 16 bits, 64 columns at a time, written
      // row by row into this warpgroup's staging box in the 128-byte swizzle
      // (16-byte chunk c of row r at chunk c ^ (r & 7)), then one TMA store;
      // thread 0 of the warpgroup issues the stores and, before the box is
      // reused, waits until the previous store has read it
      const uint32_t stage = sbase + C::kOffEpi + (uint32_t)t * C::kEpiBytes;
      const bool lead = quarter == 0 && lane == 0;
#pragma unroll 1
      for (int hb = 0; hb < C::D / 64; ++hb) {
        if (lead) ptx::bulk_wait_read_all();
        wg_sync(t);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t v[32];
          ptx::tmem_ld32(o_addr + 64 * hb + 32 * half, v);
          ptx::tmem_wait_ld();
          ptx::reg_fence(v);
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            pk[j] = pack_out<C::KIND>(__uint_as_float(v[2 * j]) * inv_l, __uint_as_float(v[2 * j + 1]) * inv_l);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            st_shared_v4(stage + (uint32_t)r * 128u + ((uint32_t)((4 * half + c) ^ (r & 7)) << 4), pk[4 * c],
                         pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
        ptx::fence_proxy_async_smem();
        wg_sync(t);
        if (lead) {
          ptx::tma_store_2d(to, stage, ti.h * C::D + 64 * hb, ti.qtok + ti.q0 + 128 * t);
          ptx::bulk_commit();
        }
      }
    } else {
      // O leaves tensor memory in 32-column chunks. e4m3: batches of up to four
      // chunks whose loads are issued back to back under one wait (the next
      // work tile's first P of this warpgroup waits for this epilogue; measured
      // on one box, c5 attention 1637 -> 1661 TFLOP/s); 16-bit: one chunk per
      // wait (batching cost c2 1435 -> 1392 there)
      constexpr int kBatch = !C::kFp8 ? 1 : (C::D / 32 < 4 ? C::D / 32 : 4);
#pragma unroll 1
      for (int cb = 0; cb < C::D / 32; cb += kBatch) {
        uint32_t v[kBatch][32];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) ptx::tmem_ld32(o_addr + 32 * (cb + q), v[q]);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
          ptx::reg_fence(v[q]);
          const int ch = cb + q;
          if (split) {
            // partial O of this key range, fp32, normalised by its own l
            if (row_ok) {
              float4* dst = reinterpret_cast<float4*>(oprow + 32 * ch);
#pragma unroll
              for (int k4 = 0; k4 < 8; ++k4)
                dst[k4] = make_float4(__uint_as_float(v[q][4 * k4]) * inv_l, __uint_as_float(v[q][4 * k4 + 1]) * inv_l,
                                      __uint_as_float(v[q][4 * k4 + 2]) * inv_l,
                                      __uint_as_float(v[q][4 * k4 + 3]) * inv_l);
            }
            continue;
          }
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            pk[j] = pack_out<C::KIND>(__uint_as_float(v[q][2 * j]) * inv_l, __uint_as_float(v[q][2 * j + 1]) * inv_l);
          if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(orow + 32 * ch);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4)
              dst[k4] = make_uint4(pk[4 * k4], pk[4 * k4 + 1], pk[4 * k4 + 2], pk[4 * k4 + 3]);
          }
        }
      }
    }
    if (row_ok) *lse_ptr = l > 0.f ? (m_ref + ptx::lg2(l)) * kLn2 : NEG_INF;
    // the next work tile's PV may overwrite O only after these reads
    ptx::tc_fence_before();
  }
}

// ------------------------------------------------------------------ kernel
template <int D, int QT, int STAGES, int KIND, bool CAUSAL>
__global__ void __launch_bounds__(FwdCfg<D, QT, STAGES, KIND>::kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                  const FwdParams p) {
  using C = FwdCfg<D, QT, STAGES, KIND>;
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
      if (i >= C::kBarPFull && i < C::kBarPFull + 2) count = 4;
      if (i >= C::kBarTileEmpty) count = C::kTileConsumers + (p.block_table != nullptr ? 1 : 0);
      ptx::mbar_init(bars + 8u * i, count);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == C::kLoadWarp && lane == 0) {
    ptx::prefetch_tmap(&tq);
    ptx::prefetch_tmap(&tk);
    ptx::prefetch_tmap(&tv);
    if (C::kTmaStore) ptx::prefetch_tmap(&to);
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
  // each role runs inside the branch that set its register budget, so the
  // register allocator sees one budget per role
  if (warp >= C::kSoftmaxWarps) {
    if constexpr (C::kRebalance) ptx::setmaxnreg_dec<C::kRegsLow>();
    if (warp == C::kLoadWarp) {
      if (p.block_table != nullptr)
        load_role<C, CAUSAL, 1>(&tq, &tk, &tv, p, sbase, wt, ring);
      else if (lane == 0)
        load_role<C, CAUSAL, 0>(&tq, &tk, &tv, p, sbase, wt, ring);
    } else if (warp == C::kVLoadWarp) {
      if (p.block_table != nullptr) load_role<C, CAUSAL, 2>(&tq, &tk, &tv, p, sbase, wt, ring);
    } else if (warp == C::kMmaWarp) {
      if (lane == 0) mma_role<C, CAUSAL>(p, sbase, tmem, wt, ring);
    }
  } else {
    if constexpr (C::kRebalance) ptx::setmaxnreg_inc<C::kRegsHigh>();
    softmax_role<C, CAUSAL>(p, &to, sbase, tmem, wt, ring, warp >> 2, warp & 3);
    // every O store this warpgroup issued has completed before the CTA ends
    if (C::kTmaStore && (threadIdx.x & 127) == 0) ptx::bulk_wait_all();
  }
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0) {
    // every fetch of this CTA is done; the last CTA out re-arms the counter
    __threadfence();
    if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
      atomicExch(p.sched, 0u);
      atomicExch(p.sched + 1, 0u);
    }
  }
}

template <int D, int QT, int STAGES, int KIND>
cudaError_t launch_fwd_kind(const FwdLaunch& L) {
  using C = FwdCfg<D, QT, STAGES, KIND>;
  auto kern = L.causal ? fa_fwd_kernel<D, QT, STAGES, KIND, true> : fa_fwd_kernel<D, QT, STAGES, KIND, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  int grid = L.p.ntiles < L.num_sms ? L.p.ntiles : L.num_sms;
  if (grid <= 0) return cudaSuccess;
  kern<<<grid, C::kThreads, C::kSmemBytes, L.stream>>>(L.tq, L.tk, L.tv, L.to, L.p);
  return cudaGetLastError();
}

// 16-bit inputs: fp16 or bf16
template <int D, int QT, int STAGES>
cudaError_t launch_fwd_impl(const FwdLaunch& L) {
  return L.kind == kF16 ? launch_fwd_kind<D, QT, STAGES, kF16>(L) : launch_fwd_kind<D, QT, STAGES, kBF16>(L);
}

}  // namespace fa
