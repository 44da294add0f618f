// prefill_kernel.cuh -- fused attention forward for dense and varlen
// (group-mode) problems on sm_103a, compiled once per head dimension
// (prefill_d64.cu, prefill_d128.cu define ATTN_PREFILL_D and include this): TMA loads into 128B-swizzled shared memory behind
// mbarrier rings, S = Q K^T and O += P V on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in tensor memory), online softmax in registers.
//
// Prior art on the pages: the DefTruth flash_attn_mma_share_kv_F32F16F16F32.cu
// kernel (FlashAttention-2 with mma.sync: Q tile kept on chip, K/V tiles
// streamed, online max/sum with the exp(m_old - m_new) rescale, final 1/l),
// the FlashAttention-3 hopper/epilogue_fwd.hpp epilogue (one LSE writer per
// row, predicated stores for varlen, store_zero for empty work) and the
// Composable Kernel fmha_fwd_pagedkv_kernel.hpp prologue (group-mode offsets,
// GQA kv head = h / ratio, heaviest causal tiles first, the scale*log2(e)
// fold).  The Blackwell design here differs from all three:
//
//  * persistent: one CTA per SM walks a list of work items (a query block of
//    two 128-row tiles of one batch and one head group; with PackGQA a tile
//    holds 128 / g queries of each of the g query heads of a kv head, which
//    then share every K/V tile in shared memory): dense masked problems run the per-CTA
//    lists the host packed for the shape (longest processing time first),
//    other dense problems a snake order across CTAs; in group mode and over
//    a paged cache every CTA first sorts the (query block, sequence) pairs
//    by cost.  The next item's Q load and its first S = Q K^T overlap the
//    current item's last P.V and epilogue.
//  * each item is two 128-row query tiles sharing every 128-key K/V tile;
//    warps 0-3 run the softmax of tile 0, warps 4-7 that of tile 1, warp 8
//    issues TMA, warp 9 issues tcgen05.mma (the whole warp runs the loop, one
//    elected lane issues).  While one warpgroup computes
//    exponentials the tensor core works on the other tile (ping-pong).
//  * S lives in tensor memory (fp32, 128 columns per tile).  The softmax
//    writes P (bf16/fp16) back over the first 64 columns of its S and the
//    P.V MMA reads its A operand straight from tensor memory; P goes out in
//    two halves of 64 keys, so the first half's P.V MMAs run while the
//    second half is computed.
//  * O accumulates in tensor memory.  The running max used as the exp2
//    subtrahend is only raised when the row max grows by more than 8 (log2
//    units); otherwise O is not rescaled.  This is exact: the final O/l and
//    LSE use the same subtrahend.
//  * the epilogue stages each warp's rows in shared memory (128 or 64 bytes
//    of each row per round, swizzled like the TMA store) and stores them with
//    TMA for dense problems, row by row with predicates in group mode and
//    over a paged cache.
//  * every mbarrier wait is bounded (Waiter): a CTA that gives up records a
//    bit in the device error word, drains its own copies and MMAs, frees its
//    tensor memory and returns.
#pragma once
#include "ptx.cuh"
#include "common.cuh"
#include "launch.h"

#include <cstdio>
#include <cstring>
#include <type_traits>

// L2 eviction priorities: Q tiles and O rows are touched once per launch
// (evict first); K/V tiles are re-read by every query block of their head
// (evict last), so the streaming Q and O do not push them out of L2.
#ifndef ATTN_L2_HINTS
#define ATTN_L2_HINTS 1
#endif

// P handed to the MMA warp in two halves of 64 keys: the P.V MMAs of the
// first half start while the softmax computes the second.
// Row maxima taken by the tensor-memory load (tcgen05.ld.red.max, sm_103a)
// where no key of the tile is masked, instead of a 3-input max tree.
#ifndef ATTN_HW_ROW_MAX
#define ATTN_HW_ROW_MAX 1
#endif
#ifndef ATTN_P_HALVES
#define ATTN_P_HALVES 1
#endif

namespace attn {

template <int D_, int DT_ = kDtBF16>
struct PrefillCfg {
  static constexpr int D = D_;
  static constexpr bool FP8 = DT_ == kDtE4M3;
  static constexpr int EB = FP8 ? 1 : 2;         // bytes per input element
  static constexpr int ATOM = 128 / EB;          // elements per 128-byte swizzle atom row
  static constexpr int BM = 128;                 // rows per query tile
  static constexpr int BN = 128;                 // keys per K/V tile
  static constexpr int NCHUNK = D / ATOM;        // swizzle atoms along d
  static constexpr int TILE_BYTES = BN * D * EB;  // one Q, K or V tile as loaded
  static constexpr int CHUNK_BYTES = BN * 128;   // one swizzle-atom column of a tile
  static constexpr int NS = (D == 128 && !FP8) ? 2 : 3;  // K/V ring depth
  // FP8: V widened to fp16 (two 64-column atoms per tile), double-buffered.
  static constexpr int NVC = FP8 ? 2 : 1;
  static constexpr int VC_BYTES = FP8 ? BN * D * 2 : 16;
  static constexpr int SOFT_WARPS = 8;            // softmax warps (two query tiles of 4)
  static constexpr int WARP_TMA = SOFT_WARPS;     // then the producer, the MMA issuer
  static constexpr int WARP_MMA = SOFT_WARPS + 1;  // and two more warps (FP8: V widening)
  // The third warpgroup (the producer, MMA and two spare warps) gives
  // registers to the two softmax warpgroups with setmaxnreg (launch: 384 x
  // 168 = 64512 registers; after: 256 x 192 + 128 x 120 = 64512).  The MMA
  // warp's issue rate limits the step time, so it keeps enough registers not
  // to spill (measured: 192/120 beats 200/96, 184/136 and 176/152 on the
  // dense causal workloads).  The host checks the launch count before the
  // first launch (launch_prefill_t): a split above the launch total would
  // leave setmaxnreg.inc waiting.
  static constexpr int THREADS = 32 * (SOFT_WARPS + 4);
  static constexpr int LAUNCH_REGS = 168;
  static constexpr int SOFT_REGS = 192;
  static constexpr int OTHER_REGS = 120;
  static_assert(SOFT_WARPS * 32 * SOFT_REGS + 128 * OTHER_REGS <= THREADS * LAUNCH_REGS,
                "register split exceeds the launch total");
  static constexpr uint32_t TM_COLS = 512;
  // Tensor-memory columns: S/P of tile t at 128*t, O of tile t at 256 + D*t.
  __device__ static constexpr uint32_t tm_s(int t) { return 128u * t; }
  __device__ static constexpr uint32_t tm_o(int t) { return 256u + D * t; }
};

// Group mode / paged cache: most (query block, sequence) slots the per-CTA
// work-order sort handles (more: the plain order).
constexpr int kMaxSlots = 2048;

// FP8 only: V widened to fp16 and its barriers.  An empty base for the
// 16-bit kernels, so their shared-memory layout carries nothing for it.
template <class C, bool FP8 = C::FP8>
struct PrefillSmemFp8 {};
template <class C>
struct PrefillSmemFp8<C, true> {
  alignas(1024) uint8_t vc[C::NVC][C::VC_BYTES];
  uint64_t vc_full[C::NVC], vc_empty[C::NVC];
};

// Group-mode / paged work order (order_items): slots heaviest first, each
// slot's cost while sorting, per-cost bucket cursors, slots in use.  Dense
// kernels take their order from the host and carry none of it.
template <bool ORD>
struct PrefillSmemOrder {};
template <>
struct PrefillSmemOrder<true> {
  uint16_t slot_order[kMaxSlots];
  uint8_t slot_cost[kMaxSlots];
  int cost_cursor[256];
  int n_slots;
};

// Bytes of each output row staged per epilogue round: dense problems store
// whole rounds by TMA; group mode and paged caches write row pieces from a
// smaller stage.
template <class C, bool ORD>
constexpr int kStageRowBytes = ORD ? 64 : prefill_o_round_bytes(C::FP8, 1);

template <class C, bool ORD>
struct PrefillSmem : PrefillSmemFp8<C>, PrefillSmemOrder<ORD> {
  alignas(1024) uint8_t q[2][C::TILE_BYTES];
  alignas(1024) uint8_t k[C::NS][C::TILE_BYTES];
  alignas(1024) uint8_t v[C::NS][C::TILE_BYTES];
  uint64_t q_full[2], q_empty[2];  // per query tile
  uint64_t k_full[C::NS], k_empty[C::NS], v_full[C::NS], v_empty[C::NS];
  uint64_t s_full[2], p_half[2], p_full[2], o_final[2], o_free[2];
  uint64_t teardown;
  uint32_t tmem_base;
  int abort_flag;
  // Epilogue staging, one 32-row block per softmax warp (kStageRowBytes per
  // row): rows go in from the thread that owns them and out by TMA or as
  // row pieces.  (1024-byte aligned: the TMA store reads it with the 64- or
  // 128-byte swizzle, whose pattern repeats every 512 or 1024 bytes.)
  alignas(1024) uint4 ostage[C::SOFT_WARPS][32 * kStageRowBytes<C, ORD> / 16];
  alignas(16) float lstage[C::SOFT_WARPS][32];  // LSE of the warp's rows (TMA store)
};

// Maximum of N values: a tree of 3-input max instructions (N = 128: 64
// instructions, depth 5).
template <int N>
__device__ __forceinline__ float max_n(const float* v) {
  if constexpr (N == 1) {
    return v[0];
  } else if constexpr (N == 2) {
    return fmaxf(v[0], v[1]);
  } else if constexpr (N == 3) {
    return fmax3(v[0], v[1], v[2]);
  } else {
    constexpr int M = (N + 2) / 3;
    float m[M];
#pragma unroll
    for (int i = 0; i < M; ++i)
      m[i] = 3 * i + 2 < N ? fmax3(v[3 * i], v[3 * i + 1], v[3 * i + 2])
                           : (3 * i + 1 < N ? fmaxf(v[3 * i], v[3 * i + 1]) : v[3 * i]);
    return max_n<M>(m);
  }
}

// P for one row: p_c = 2^(s_c * a - b) for c < 2 NP (a = scale*log2e, or
// cap*log2e when s holds tanh values), the FMA done two lanes at a time,
// packed to bf16/fp16 pairs, with 4 packed partial sums (8 lanes).  A masked
// score is -inf and gives p = 0 exactly.
template <bool BF16, int NP, int I = 0>
__device__ __forceinline__ void exp_pack_row(const float* s, uint64_t a2, uint64_t nb2,
                                             uint32_t* pk, uint64_t* acc2) {
  if constexpr (I < NP) {
    float x0, x1;
    f2_unpack(f2_fma(f2_pack(s[2 * I], s[2 * I + 1]), a2, nb2), x0, x1);
    const float p0 = ex2_approx(x0);
    const float p1 = ex2_approx(x1);
    acc2[I & 3] = f2_add(acc2[I & 3], f2_pack(p0, p1));
    pk[I] = BF16 ? pack_bf16(p0, p1) : pack_f16(p0, p1);
    exp_pack_row<BF16, NP, I + 1>(s, a2, nb2, pk, acc2);
  }
}

// Soft-cap in the form the softmax consumes: s <- r = 1 / (2^(2 y log2 e) + 1)
// with y = in_scale * s, so that tanh(y) = 1 - 2 r and the capped score in
// log2 units is c (1 - 2 r), c = cap * log2 e.  The exponent's FMA then takes
// r directly (r * (-2c) + (c - m)) and the row maximum is c (1 - 2 min r):
// the tanh's own final FMA disappears from the chain.
template <int N>
__device__ __forceinline__ void softcap_r_n(float* s, float in_scale) {
  const uint64_t k2 = f2_pack(in_scale * 2.0f * kLog2e, in_scale * 2.0f * kLog2e);
  const uint64_t one2 = f2_pack(1.0f, 1.0f);
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {
    float e0, e1;
    f2_unpack(f2_mul(f2_pack(s[2 * i], s[2 * i + 1]), k2), e0, e1);
    e0 = ex2_approx(e0);
    e1 = ex2_approx(e1);
    float d0, d1;
    f2_unpack(f2_add(f2_pack(e0, e1), one2), d0, d1);
    s[2 * i] = rcp_approx(d0);
    s[2 * i + 1] = rcp_approx(d1);
  }
}

// Minimum of N values (a tree of 3-input min instructions).
template <int N>
__device__ __forceinline__ float min_n(const float* v) {
  if constexpr (N == 1) {
    return v[0];
  } else if constexpr (N == 2) {
    return fminf(v[0], v[1]);
  } else if constexpr (N == 3) {
    return fmin3(v[0], v[1], v[2]);
  } else {
    constexpr int M = (N + 2) / 3;
    float m[M];
#pragma unroll
    for (int i = 0; i < M; ++i)
      m[i] = 3 * i + 2 < N ? fmin3(v[3 * i], v[3 * i + 1], v[3 * i + 2])
                           : (3 * i + 1 < N ? fminf(v[3 * i], v[3 * i + 1]) : v[3 * i]);
    return min_n<M>(m);
  }
}

// FP8: one 128-key V tile, e4m3 rows of 128 bytes (128B-swizzled as TMA
// wrote them) -> fp16 in the MN-major layout the P.V MMA reads (two 64-column
// 128B-swizzled atoms).  64 threads, 16 of the 1024 (row, 16-byte piece)
// pairs each; e4m3 -> fp16 is exact.
template <class C>
__device__ __forceinline__ void widen_v_tile(const uint8_t* raw, uint8_t* out, int ct) {
#pragma unroll 4
  for (int k = 0; k < 16; ++k) {
    const int i = ct + 64 * k;
    const int r = i >> 3, u = i & 7;  // key row, 16-byte piece (columns 16u .. 16u+15)
    const uint4 x = *reinterpret_cast<const uint4*>(raw + r * 128 + ((u ^ (r & 7)) << 4));
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t h[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      h[2 * j] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[j] & 0xffffu));
      h[2 * j + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[j] >> 16));
    }
    uint8_t* atom = out + (u >> 2) * C::CHUNK_BYTES + r * 128;
    const int p0 = 2 * (u & 3);  // 16-byte unit of columns 16u .. 16u+7 within the atom
    *reinterpret_cast<uint4*>(atom + ((p0 ^ (r & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(atom + (((p0 + 1) ^ (r & 7)) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

// Elementwise bias (Composable Kernel bias kargs).  One row's segment for a
// K/V tile (8 NC keys: the thread's score columns) is loaded into registers
// a step ahead, raw: 16-byte loads where all 8 keys are valid, element loads
// at the tail (keys past the end read as 0; they are masked later).
template <int NC>
__device__ __forceinline__ void load_bias_regs(uint4 (&bn)[NC], const void* src, int nvalid) {
  const uint16_t* b = reinterpret_cast<const uint16_t*>(src);
#pragma unroll
  for (int c8 = 0; c8 < NC; ++c8) {
    if (8 * c8 + 8 <= nvalid) {
      bn[c8] = __ldg(reinterpret_cast<const uint4*>(b + 8 * c8));
    } else {
      uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (8 * c8 + i < nvalid) w[i >> 1] |= static_cast<uint32_t>(__ldg(b + 8 * c8 + i)) << (16 * (i & 1));
      bn[c8] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// Adds 32 bias values (natural-log units, so divided by the scale folded in
// later) to 32 raw scores.
template <bool BF16>
__device__ __forceinline__ void add_bias_quarter(float* s, const uint4* bn, float inv_scale) {
#pragma unroll
  for (int c8 = 0; c8 < 4; ++c8) {
    const uint32_t w[4] = {bn[c8].x, bn[c8].y, bn[c8].z, bn[c8].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float lo, hi;
      if constexpr (BF16) {
        lo = __uint_as_float(w[i] << 16);
        hi = __uint_as_float(w[i] & 0xffff0000u);
      } else {
        const __half2 h2 = *reinterpret_cast<const __half2*>(&w[i]);
        lo = __low2float(h2);
        hi = __high2float(h2);
      }
      s[8 * c8 + 2 * i] = fmaf(lo, inv_scale, s[8 * c8 + 2 * i]);
      s[8 * c8 + 2 * i + 1] = fmaf(hi, inv_scale, s[8 * c8 + 2 * i + 1]);
    }
  }
}

// Wait for a barrier phase ignoring the abort flag (teardown only).
__device__ __forceinline__ bool wait_raw(uint64_t* bar, uint32_t parity, uint64_t deadline) {
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() > deadline) return false;
  }
  return true;
}

// One unit of work: a query block of two 128-row tiles against all of its
// keys.  Without packing a tile is 128 queries of query head h; with PackGQA
// (FlashAttention-3 epilogue, PackGQA row <-> (head, query) mapping) it is
// 128 / g queries of each of the g query heads h .. h + g - 1 of kv head hk.
struct PrefillItem {
  int b, h, hk, rq0, rk0, bcoord, Lq, Lk, m0;
  int jb;     // first K/V tile of the item
  int cnt;    // K/V tiles streamed for the item (0: nothing to compute)
  int ub[2];  // query tile t takes part in steps [ub[t], ue[t]) of the item
  int ue[2];
};

// One 128-key K or V tile of sequence it.b gathered from a paged pool
// (Composable Kernel page block navigator: key j is row j mod page of
// physical page block_table[b][j / page]).  The map is 3-D (d, Hkv, pool
// rows); one box of min(page, 128) rows per page piece and 64-column chunk.
// Pieces past the sequence end, or behind a block-table entry outside
// [0, num_pages) (an error: device error word bit), load from one row past
// the pool, which the copy engine fills with zeros, so every tile delivers
// its full byte count.
template <class C>
__device__ __forceinline__ void load_paged_tile(const PrefillParams& p, const PrefillItem& it,
                                                int key0, const CUtensorMap* map, uint8_t* dst,
                                                uint64_t* bar, uint64_t pol) {
  const int P = p.page_size;
  const int BR = P < C::BN ? P : C::BN;  // rows per box
  const int32_t* bt = p.block_table + static_cast<int64_t>(it.b) * p.max_pages;
  const int oob_row = p.num_pages * P;
  for (int r0 = 0; r0 < C::BN; r0 += BR) {
    const int key = key0 + r0;
    int row = oob_row;
    if (key < it.Lk) {
      const int lp = key / P;
      const int phys = lp < p.max_pages ? bt[lp] : -1;
      if (phys >= 0 && phys < p.num_pages)
        row = phys * P + (key - lp * P);
      else if (p.err)
        atomicOr(p.err, 1u << kErrPrefillBadPage);
    }
#pragma unroll
    for (int c = 0; c < C::NCHUNK; ++c) {
      if constexpr (ATTN_L2_HINTS)
        tma_load_3d_hint(dst + c * C::CHUNK_BYTES + r0 * 128, map, bar, c * C::ATOM, it.hk, row, pol);
      else
        tma_load_3d(dst + c * C::CHUNK_BYTES + r0 * 128, map, bar, c * C::ATOM, it.hk, row);
    }
  }
}

// Item index -> coordinates.  Masked problems list the heaviest query blocks
// first (Composable Kernel GetTileIndex reverses the m-tile order when
// masking).  Returns false when the block starts past the sequence end.
// Key bounds per query row i (bottom-right aligned, Composable Kernel mask
// from the left/right window): i + (Lk - Lq) - win_left <= j <= i + (Lk - Lq)
// + win_right, a negative bound meaning unbounded; causal is win_right = 0.
template <int BM, int BN, bool MASK>
__device__ __forceinline__ bool decode_pair(const PrefillParams& p, int b, int mb, int unit,
                                            PrefillItem& it) {
  it.h = unit * p.pack;  // first query head of the item
  it.b = b;
  it.hk = it.h / (p.Hq / p.Hkv);
  it.Lq = p.Lq;
  it.Lk = p.Lk;
  it.rq0 = 0;
  it.rk0 = 0;
  it.bcoord = it.b;
  if (p.cu_q != nullptr) {  // group mode (Composable Kernel seqstart_q/k)
    it.rq0 = p.cu_q[it.b];
    it.Lq = p.cu_q[it.b + 1] - it.rq0;
    it.rk0 = p.cu_k[it.b];
    it.Lk = p.cu_k[it.b + 1] - it.rk0;
    it.bcoord = 0;
    // Sequences never reach past the packed tensors, whatever cu_seqlens holds.
    if (it.rq0 < 0 || it.rq0 > p.total_q) it.Lq = 0;
    it.Lq = min(it.Lq, p.total_q - it.rq0);
    if (it.rk0 < 0 || it.rk0 > p.total_k) it.Lk = 0;
    it.Lk = max(0, min(it.Lk, p.total_k - it.rk0));
  } else if (p.seqlens_k != nullptr) {  // paged KV cache: per-sequence key count
    it.Lk = max(0, min(p.seqlens_k[it.b], p.max_pages * p.page_size));
  }
  const int qpt = 1 << p.qpt_log2;  // queries per tile (BM without packing)
  it.m0 = mb * 2 * qpt;
  if (it.m0 >= it.Lq) return false;
  const int diag = p.top_left ? 0 : it.Lk - it.Lq;  // key on row 0's diagonal
  int tb[2], te[2];  // K/V tile range [tb, te) of each query tile
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int mt = it.m0 + t * qpt;
    tb[t] = te[t] = 0;
    if (mt < it.Lq) {
      const int last = min(mt + qpt - 1, it.Lq - 1);
      int kend = it.Lk, kbeg = 0;  // keys [kbeg, kend) some row of the tile keeps
      if (MASK && p.win_right >= 0) kend = min(it.Lk, last + diag + p.win_right + 1);
      if (MASK && p.win_left >= 0) kbeg = max(0, mt + diag - p.win_left);
      if (kend > kbeg) {
        tb[t] = kbeg / BN;
        te[t] = (kend + BN - 1) / BN;
      }
    }
  }
  const bool has0 = te[0] > tb[0], has1 = te[1] > tb[1];
  it.jb = has0 ? (has1 ? min(tb[0], tb[1]) : tb[0]) : tb[1];
  const int je = max(has0 ? te[0] : 0, has1 ? te[1] : 0);
  it.cnt = (has0 || has1) ? je - it.jb : 0;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const bool has = te[t] > tb[t];
    it.ub[t] = has ? tb[t] - it.jb : 0;
    it.ue[t] = has ? te[t] - it.jb : 0;
  }
  return true;
}

// Work-item order.  Dense problems keep the plain order: query block (the
// heaviest causal blocks first), then (batch, head).  In group mode and over a
// paged cache the sequences differ in length, so that order leaves holes
// (blocks past a short sequence's end) and mixes costs; there every CTA sorts
// the (query block, sequence) slots by their K/V step count, heaviest first,
// and items become (slot, head group) in that order.
struct ItemOrder {
  const uint16_t* slot;  // slot = query block * B + sequence, heaviest first
  int n;                 // slots in use; -1: plain order
};

template <int BM, int BN, bool MASK, bool ORD>
__device__ __forceinline__ bool decode_item(const PrefillParams& p, const ItemOrder& ord, int item,
                                            PrefillItem& it) {
  if constexpr (ORD) {
    if (ord.n >= 0) {
      const int pos = item / p.units;
      if (pos >= ord.n) return false;
      const int slot = ord.slot[pos];
      const int mb = slot / p.B;
      return decode_pair<BM, BN, MASK>(p, slot - mb * p.B, mb, item - pos * p.units, it);
    }
  }
  const int nbh = p.B * p.units;
  const int mb_i = item / nbh;
  const int bh = item - mb_i * nbh;
  const int mb = MASK ? (p.num_m_blocks - 1 - mb_i) : mb_i;
  return decode_pair<BM, BN, MASK>(p, bh / p.units, mb, bh % p.units, it);
}

// Builds the group-mode / paged work order in shared memory; every thread of
// the CTA calls it (it synchronises the block).  Costs are K/V steps + 1
// (a slot with rows but no key still writes its output), 0 for a slot past
// its sequence's end; a histogram gives each cost's first position, heaviest
// first, and one warp places the slots in slot order within a cost, so that
// every CTA builds the same list.
template <int BM, int BN, bool MASK, class C>
__device__ void order_items(const PrefillParams& p, PrefillSmem<C, true>& sm) {
  const int nslots = p.num_m_blocks * p.B;
  if ((p.cu_q == nullptr && p.seqlens_k == nullptr) || nslots > kMaxSlots) {
    if (threadIdx.x == 0) sm.n_slots = -1;
    __syncthreads();
    return;
  }
  for (int i = threadIdx.x; i < 256; i += blockDim.x) sm.cost_cursor[i] = 0;
  __syncthreads();
  for (int s = threadIdx.x; s < nslots; s += blockDim.x) {
    PrefillItem it;
    const int mb = s / p.B;
    int c = 0;
    if (decode_pair<BM, BN, MASK>(p, s - mb * p.B, mb, 0, it)) c = min(it.cnt, 254) + 1;
    sm.slot_cost[s] = static_cast<uint8_t>(c);
    if (c > 0) atomicAdd(&sm.cost_cursor[c], 1);
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    // First position of each cost, heaviest first (costs 255 .. 1, 32 at a time).
    int run = 0;
    for (int c0 = 255; c0 > 0; c0 -= 32) {
      const int c = c0 - lane;
      const int v = c > 0 ? sm.cost_cursor[c] : 0;
      int x = v;  // inclusive prefix over the lanes
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (c > 0) sm.cost_cursor[c] = run + x - v;
      run += __shfl_sync(0xffffffffu, x, 31);
    }
    __syncwarp();
    // Place the slots 32 at a time; equal costs keep slot order.
    for (int s0 = 0; s0 < nslots; s0 += 32) {
      const int s = s0 + lane;
      const int c = s < nslots ? sm.slot_cost[s] : 0;
      const unsigned same = __match_any_sync(0xffffffffu, c);
      const int rank = __popc(same & ((1u << lane) - 1u));
      if (c > 0) sm.slot_order[sm.cost_cursor[c] + rank] = static_cast<uint16_t>(s);
      __syncwarp();
      if (c > 0 && rank == __popc(same) - 1) sm.cost_cursor[c] += __popc(same);
      __syncwarp();
    }
    if (lane == 0) sm.n_slots = run;
  }
  __syncthreads();
}

// The r-th item of this CTA: rounds of gridDim.x items, alternating direction
// (snake), so the heavy head of the list is spread evenly across CTAs.
// With a host-packed schedule, the r-th item of this CTA's list instead
// (past its end: num_items, which ends every role's loop).
__device__ __forceinline__ int item_of_round(const PrefillParams& p, int r) {
  const int G = gridDim.x, c = blockIdx.x;
  if (p.sched_n > 0) {
    const int pos = p.sched_off[c] + r;
    return pos < p.sched_off[c + 1] ? static_cast<int>(p.sched_item[pos]) : p.num_items;
  }
  return r * G + ((r & 1) ? (G - 1 - c) : c);
}

// XF: score transform before masking (ScoreXf): none, soft-cap, ALiBi or an
// elementwise bias (the last two are mutually exclusive with the soft-cap).
// ORD: group mode or paged cache, work items in the sorted order (order_items).
template <int D, int DT, bool MASK, int XF, bool ORD>
__global__ void __launch_bounds__(PrefillCfg<D, DT>::THREADS, 1)
    attn_prefill_kernel(const __grid_constant__ PrefillParams p) {
  using C = PrefillCfg<D, DT>;
  constexpr bool FP8 = C::FP8;
  constexpr bool BF16 = DT == kDtBF16;  // P / V type of the P.V MMA (FP8: fp16)
  // P in two halves where the score transform leaves the registers for it
  // (ALiBi and the elementwise bias would spill).
  constexpr bool HALVES = ATTN_P_HALVES && (XF == kXfNone || XF == kXfSoftcap);
  // Row maxima from the tensor-memory load itself (sm_103a tcgen05.ld.red) on
  // tiles without masked keys, for untransformed scores (with the soft-cap,
  // measured slower: the scalar tanh of the maximum then sits on the chain
  // and the kernel spills).
  constexpr bool HW_MAX = ATTN_HW_ROW_MAX && XF == kXfNone;
  extern __shared__ uint8_t smem_raw[];
  PrefillSmem<C, ORD>& sm = *reinterpret_cast<PrefillSmem<C, ORD>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm.q_full[t], 1);
      mbar_init(&sm.q_empty[t], 1);
    }
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v_empty[s], FP8 ? 64 : 1);  // FP8: released by the 64 widening threads
    }
    if constexpr (FP8) {
      for (int c = 0; c < C::NVC; ++c) {
        mbar_init(&sm.vc_full[c], 64);
        mbar_init(&sm.vc_empty[c], 1);
      }
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm.s_full[t], 1);
      mbar_init(&sm.p_half[t], 128);  // every softmax thread of the tile
      mbar_init(&sm.p_full[t], 128);
      mbar_init(&sm.o_final[t], 1);
      mbar_init(&sm.o_free[t], 128);
    }
    mbar_init(&sm.teardown, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::WARP_MMA) {
    tmem_alloc(&sm.tmem_base, C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  ItemOrder ord{nullptr, -1};
  if constexpr (ORD) {
    order_items<C::BM, C::BN, MASK>(p, sm);
    ord = ItemOrder{sm.slot_order, sm.n_slots};
  }
  const uint32_t tmem = sm.tmem_base;
  const Waiter w{globaltimer_ns() + p.timeout_ns, &sm.abort_flag, p.err};

  if (warp >= C::SOFT_WARPS) {
    setmaxnreg_dec<C::OTHER_REGS>();
    if (warp == C::WARP_TMA && lane == 0) {
      // ===================== TMA producer =====================================
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      const uint64_t pol_once = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      int g = 0, qn = 0, k_armed = 0, v_armed = 0;
      int qa[2] = {0, 0};  // arms of each tile's q_full
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int item = item_of_round(p, r);
        if (item >= p.num_items) break;
        PrefillItem it;
        if (!decode_item<C::BM, C::BN, MASK, ORD>(p, ord, item, it) || it.cnt == 0) continue;
        // Each tile's Q buffer is reloaded once the previous item's last S
        // MMA of that tile is done (tile 0 usually a step before tile 1).
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (qn > 0 && !(ok = w.wait(&sm.q_empty[t], (qn - 1) & 1, kErrPrefillQ))) break;
          mbar_arrive_expect_tx(&sm.q_full[t], C::TILE_BYTES);
          ++qa[t];
#pragma unroll
          for (int c = 0; c < C::NCHUNK; ++c) {  // box {ATOM, qpt queries, pack heads}
            if constexpr (ATTN_L2_HINTS)
              tma_load_4d_hint(sm.q[t] + c * C::CHUNK_BYTES, &p.tm_q, &sm.q_full[t], c * C::ATOM,
                               it.rq0 + it.m0 + (t << p.qpt_log2), it.h, it.bcoord, pol_once);
            else
              tma_load_4d(sm.q[t] + c * C::CHUNK_BYTES, &p.tm_q, &sm.q_full[t], c * C::ATOM,
                          it.rq0 + it.m0 + (t << p.qpt_log2), it.h, it.bcoord);
          }
        }
        if (!ok) break;
        ++qn;
        for (int j = 0; j < it.cnt; ++j, ++g) {
          const int s = g % C::NS;
          const uint32_t ph = (g / C::NS) & 1;
          if (!(ok = w.wait(&sm.k_empty[s], ph ^ 1, kErrPrefillKEmpty))) break;
          mbar_arrive_expect_tx(&sm.k_full[s], C::TILE_BYTES);
          if (p.block_table != nullptr) {
            load_paged_tile<C>(p, it, (it.jb + j) * C::BN, &p.tm_k, sm.k[s], &sm.k_full[s],
                               pol_kv);
          } else {
#pragma unroll
            for (int c = 0; c < C::NCHUNK; ++c) {
              if constexpr (ATTN_L2_HINTS)
                tma_load_4d_hint(sm.k[s] + c * C::CHUNK_BYTES, &p.tm_k, &sm.k_full[s],
                                 c * C::ATOM, it.rk0 + (it.jb + j) * C::BN, it.hk, it.bcoord,
                                 pol_kv);
              else
                tma_load_4d(sm.k[s] + c * C::CHUNK_BYTES, &p.tm_k, &sm.k_full[s],
                            c * C::ATOM, it.rk0 + (it.jb + j) * C::BN, it.hk, it.bcoord);
            }
          }
          ++k_armed;
          if (!(ok = w.wait(&sm.v_empty[s], ph ^ 1, kErrPrefillVEmpty))) break;
          mbar_arrive_expect_tx(&sm.v_full[s], C::TILE_BYTES);
          if (p.block_table != nullptr) {
            load_paged_tile<C>(p, it, (it.jb + j) * C::BN, &p.tm_v, sm.v[s], &sm.v_full[s],
                               pol_kv);
          } else {
#pragma unroll
            for (int c = 0; c < C::NCHUNK; ++c) {
              if constexpr (ATTN_L2_HINTS)
                tma_load_4d_hint(sm.v[s] + c * C::CHUNK_BYTES, &p.tm_v, &sm.v_full[s],
                                 c * C::ATOM, it.rk0 + (it.jb + j) * C::BN, it.hk, it.bcoord,
                                 pol_kv);
              else
                tma_load_4d(sm.v[s] + c * C::CHUNK_BYTES, &p.tm_v, &sm.v_full[s],
                            c * C::ATOM, it.rk0 + (it.jb + j) * C::BN, it.hk, it.bcoord);
            }
          }
          ++v_armed;
        }
      }
      if (w.aborted()) {
        // Drain: every copy this CTA started must land before shared memory
        // is released.  The last armed phase of each full barrier completes
        // when its bytes arrive.
        const uint64_t dl = globaltimer_ns() + 50000000ull;
        for (int t = 0; t < 2; ++t)
          if (qa[t] > 0) wait_raw(&sm.q_full[t], (qa[t] - 1) & 1, dl);
        for (int jj = max(0, k_armed - C::NS); jj < k_armed; ++jj)
          wait_raw(&sm.k_full[jj % C::NS], (jj / C::NS) & 1, dl);
        for (int jj = max(0, v_armed - C::NS); jj < v_armed; ++jj)
          wait_raw(&sm.v_full[jj % C::NS], (jj / C::NS) & 1, dl);
      }
    } else if (warp == C::WARP_MMA) {
      // ===================== MMA issuer (whole warp) ==========================
      // Every lane runs the loop (so its operand arithmetic stays warp-uniform)
      // and waits on the barriers itself; only the elected lane issues MMAs and
      // commits, so lanes need no vote: nothing here is warp-synchronous.
      const uint32_t lead = elect_one() ? 1u : 0u;
      constexpr uint32_t idesc_s =
          FP8 ? idesc_e4m3_f32(128, C::BN) : idesc_f16_f32(BF16, 128, C::BN, false, false);
      constexpr uint32_t idesc_o = idesc_f16_f32(BF16, 128, D, false, true);
      // Descriptors of the operand buffers, built once; an MMA's operand
      // start is the buffer's plus a constant (no carry leaves the 14-bit
      // start-address field: shared memory is below 256 KB).
      const uint64_t qdesc0 = sdesc_sw128(smem_u32(sm.q[0]), 16, 1024);
      const uint64_t qdesc1 = sdesc_sw128(smem_u32(sm.q[1]), 16, 1024);
      const uint64_t kdesc0 = sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);
      const uint64_t vdesc0 = sdesc_sw128(smem_u32(sm.v[0]), C::CHUNK_BYTES, 1024);
      constexpr uint32_t kTileDesc = C::TILE_BYTES >> 4;  // ring slot stride in descriptor units
      auto issue_s = [&](int t, int g) {  // S_t = Q_t K_g^T
        const uint64_t qd = t ? qdesc1 : qdesc0;
        const uint64_t kd = kdesc0 + static_cast<uint64_t>((g % C::NS) * kTileDesc);
        // 32 bytes of d per MMA (16 fp16 / bf16 or 32 e4m3 elements).
#pragma unroll
        for (int k = 0; k < D * C::EB / 32; ++k) {
          const uint32_t off = ((k >> 2) * C::CHUNK_BYTES + (k & 3) * 32) >> 4;
          if constexpr (FP8)
            umma_ss_f8_warp(tmem + C::tm_s(t), qd + off, kd + off, idesc_s, k > 0 ? 1u : 0u, lead);
          else
            umma_ss_warp(tmem + C::tm_s(t), qd + off, kd + off, idesc_s, k > 0 ? 1u : 0u, lead);
        }
        umma_commit_warp(&sm.s_full[t], lead);
      };
      // O_t (+)= P_t V_g over keys [16 k0, 16 k1) of the tile.
      auto issue_pv = [&](int t, int g, bool acc, int k0, int k1) {
        uint64_t vd;
        if constexpr (FP8) vd = sdesc_sw128(smem_u32(sm.vc[g % C::NVC]), C::CHUNK_BYTES, 1024);
        else vd = vdesc0 + static_cast<uint64_t>((g % C::NS) * kTileDesc);
#pragma unroll
        for (int k = k0; k < k1; ++k) {  // 16 keys per MMA
          umma_ts_warp(tmem + C::tm_o(t), tmem + C::tm_s(t) + k * 8, vd + ((k * 16 * 128) >> 4),
                       idesc_o, (acc || k > 0) ? 1u : 0u, lead);
        }
      };
      int g = 0, qn = 0;
      int pc[2] = {0, 0};  // participations of each tile so far (p_full phases)
      int oc[2] = {0, 0};  // items finished by each tile so far (o_free phases)
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int item = item_of_round(p, r);
        if (item >= p.num_items) break;
        PrefillItem it;
        if (!decode_item<C::BM, C::BN, MASK, ORD>(p, ord, item, it) || it.cnt == 0) continue;
        ok = w.wait(&sm.k_full[g % C::NS], (g / C::NS) & 1, kErrPrefillKFull);
        // Each tile's first S as soon as its Q is in; a tile's Q buffer is
        // free for the next item once its last S MMA completes: commit right
        // after that issue so the next Q load overlaps the tail.
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!ok || !(ok = w.wait(&sm.q_full[t], qn & 1, kErrPrefillQ))) break;
          tc_fence_after();
          if (it.ub[t] == 0 && it.ue[t] > 0) issue_s(t, g);
          if (it.ue[t] <= 1) umma_commit_warp(&sm.q_empty[t], lead);  // no later S for tile t
        }
        ++qn;
        if (!ok) break;
        umma_commit_warp(&sm.k_empty[g % C::NS], lead);
        // Every streamed K/V tile is waited for and released at its step, used
        // or not (a narrow window can leave a tile to neither query tile).
        for (int u = 0; ok && u < it.cnt; ++u) {
          const int gu = g + u;
          const int s = gu % C::NS;
          if constexpr (FP8)
            ok = w.wait(&sm.vc_full[gu % C::NVC], (gu / C::NVC) & 1, kErrPrefillVFull);
          else
            ok = w.wait(&sm.v_full[s], (gu / C::NS) & 1, kErrPrefillVFull);
          if (!ok) break;
          const bool next = u + 1 < it.cnt;
          if (next && !(ok = w.wait(&sm.k_full[(gu + 1) % C::NS], ((gu + 1) / C::NS) & 1,
                                    kErrPrefillKFull)))
            break;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (it.ub[t] <= u && u < it.ue[t]) {
              if (!(ok = w.wait(HALVES ? &sm.p_half[t] : &sm.p_full[t], pc[t] & 1,
                                kErrPrefillPFull)))
                break;
              // O_t is free once the previous item's epilogue has read it.
              if (u == it.ub[t] && oc[t] > 0 &&
                  !(ok = w.wait(&sm.o_free[t], (oc[t] - 1) & 1, kErrPrefillOFinal)))
                break;
              tc_fence_after();
              if constexpr (HALVES) {
                issue_pv(t, gu, u > it.ub[t], 0, C::BN / 32);
                if (!(ok = w.wait(&sm.p_full[t], pc[t] & 1, kErrPrefillPFull))) break;
                tc_fence_after();
                issue_pv(t, gu, true, C::BN / 32, C::BN / 16);
              } else {
                issue_pv(t, gu, u > it.ub[t], 0, C::BN / 16);
              }
              ++pc[t];
              if (u + 1 == it.ue[t]) umma_commit_warp(&sm.o_final[t], lead);
            }
            // No fence of its own: S_t(u+1) is ordered after this tile's
            // p_full wait by the fence above (or, for a tile that starts at
            // u+1, touches no column the softmax still reads), and its K tile
            // by the k_full wait (copy engine to tensor core).
            if (next && it.ub[t] <= u + 1 && u + 1 < it.ue[t]) {
              issue_s(t, gu + 1);
              if (u + 2 == it.ue[t]) umma_commit_warp(&sm.q_empty[t], lead);  // tile t's last S
            }
          }
          if constexpr (FP8) umma_commit_warp(&sm.vc_empty[gu % C::NVC], lead);
          else umma_commit_warp(&sm.v_empty[s], lead);
          if (next) umma_commit_warp(&sm.k_empty[(gu + 1) % C::NS], lead);
        }
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (it.ue[t] > it.ub[t]) ++oc[t];
        g += it.cnt;
      }
      // All MMAs this warp issued must finish before tensor memory is freed.
      umma_commit_warp(&sm.teardown, lead);
      if (!wait_raw(&sm.teardown, 0, globaltimer_ns() + 50000000ull) && p.err)
        atomicOr(p.err, 1u << kErrPrefillTeardown);
    } else if (warp == C::WARP_MMA + 1 || warp == C::WARP_MMA + 2) {
      if constexpr (FP8) {
      // ============== FP8: widen each V tile from e4m3 to fp16 ================
      // (the P.V MMA runs on the fp16 tensor path: its operands must share
      // one type, and P keeps more precision than e4m3 that way).
      const int ct = threadIdx.x - 32 * (C::WARP_MMA + 1);  // 0..63
      int g = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int item = item_of_round(p, r);
        if (item >= p.num_items) break;
        PrefillItem it;
        if (!decode_item<C::BM, C::BN, MASK, ORD>(p, ord, item, it) || it.cnt == 0) continue;
        for (int j = 0; j < it.cnt; ++j, ++g) {
          const int s = g % C::NS, c = g % C::NVC;
          ok = __all_sync(0xffffffffu, w.wait(&sm.v_full[s], (g / C::NS) & 1, kErrPrefillVFull)) &&
               __all_sync(0xffffffffu,
                          w.wait(&sm.vc_empty[c], ((g / C::NVC) & 1) ^ 1, kErrPrefillVEmpty));
          if (!ok) break;
          widen_v_tile<C>(sm.v[s], sm.vc[c], ct);
          fence_proxy_async_smem();  // the tensor core reads what these threads wrote
          mbar_arrive(&sm.vc_full[c]);
          mbar_arrive(&sm.v_empty[s]);
        }
      }
      }
    }
    // the other lanes: no role
  } else {
    setmaxnreg_inc<C::SOFT_REGS>();
    // ======================= softmax warpgroups =============================
    // Warps 4t .. 4t+3 run query tile t, thread = row = TMEM lane (warp & 3
    // picks the lane quarter).
    using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    constexpr int W = C::BN;                          // score columns per thread per step
    const int t = warp >> 2;                          // query tile of this warp
    const int r = (warp & 3) * 32 + lane;             // row within the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + C::tm_s(t) + lane_base;
    const uint32_t tO = tmem + C::tm_o(t) + lane_base;
    int pc = 0, oc = 0;
    bool ok = true;
    for (int rr = 0; ok; ++rr) {
      const int item = item_of_round(p, rr);
      if (item >= p.num_items) break;
      PrefillItem it;
      if (!decode_item<C::BM, C::BN, MASK, ORD>(p, ord, item, it)) continue;
      const int qmask = (1 << p.qpt_log2) - 1;
      const int mt = it.m0 + (t << p.qpt_log2);  // first query of this tile
      if (mt >= it.Lq) continue;                  // this tile has no row
      const int qi = mt + (r & qmask);            // this row's query index within the sequence
      const int hr = it.h + (r >> p.qpt_log2);    // and its query head
      const int nt = it.ue[t] - it.ub[t];  // K/V steps of this tile
      const int diag = p.top_left ? 0 : it.Lk - it.Lq;  // key on row 0's diagonal
      const int last = min(mt + qmask, it.Lq - 1);      // last query of this tile
      float alibi_raw = 0.0f;      // ALiBi slope / scale (raw-score units)
      const T* bias_row = nullptr;  // this row's bias, key 0
      if constexpr (XF == kXfAlibi) alibi_raw = p.alibi[it.b * p.alibi_stride + hr] * p.inv_scale;
      if constexpr (XF == kXfBias)
        bias_row = reinterpret_cast<const T*>(p.bias) + it.b * p.bias_batch + hr * p.bias_head +
                   static_cast<int64_t>(qi) * p.bias_row;

      float m_use = -INFINITY;  // exp2 subtrahend currently in use (log2 units)
      float l = 0.0f;           // running denominator w.r.t. m_use
      // Bias: this row's segment for the coming K/V tile, loaded right after
      // the previous step's P is handed over, so that the loads run while the
      // tensor core computes the next S; the L2 is warmed one step further
      // ahead (the valid bytes only).
      uint4 bn[W / 8];
      auto fetch_bias = [&](int jj) {  // registers for step jj, L2 for step jj + 1
        const int k0 = (it.jb + it.ub[t] + jj) * C::BN;
        load_bias_regs<W / 8>(bn, bias_row + k0, it.Lk - k0);
        if (jj + 1 < nt) {
          const char* nb = reinterpret_cast<const char*>(bias_row + k0 + C::BN);
          const int bytes = min(it.Lk - (k0 + C::BN), W) * static_cast<int>(sizeof(T));
          if (bytes > 0) {
            prefetch_l2(nb);
            if (bytes > 128) prefetch_l2(nb + 128);
            prefetch_l2(nb + bytes - 1);
          }
        }
      };
      if constexpr (XF == kXfBias)
        if (qi < it.Lq && nt > 0) fetch_bias(0);
      for (int j = 0; j < nt; ++j) {
        ok = __all_sync(0xffffffffu, w.wait(&sm.s_full[t], pc & 1, kErrPrefillSFull));
        if (!ok) break;
        ++pc;
        tc_fence_after();
        uint32_t sr[W];
        const int j0 = (it.jb + it.ub[t] + j) * C::BN;  // first key of this K/V tile
        // Whether some key of this tile is masked for some row of the tile
        // (the tail past Lk, the causal / window band): the same for every
        // thread of the warpgroup.
        const bool masked = (j0 + W > it.Lk) ||
                            (MASK && p.win_right >= 0 && j0 + W - 1 > mt + diag + p.win_right) ||
                            (MASK && p.win_left >= 0 && j0 < last + diag - p.win_left);
        float raw_max = -INFINITY;  // (HW_MAX) the row maximum of the raw scores
        if constexpr (XF == kXfBias) {
          // A quarter of 32 scores at a time, each taking its bias from
          // registers as it lands, so that the prefetched segment and the
          // scores are never all live at once.
#pragma unroll
          for (int qq = 0; qq < W / 32; ++qq) {
            uint32_t (&aq)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * qq]);
            tmem_ld32(tS + 32 * qq, aq);
            tmem_ld_wait();
            reg_fence(aq);
            if (qi < it.Lq)
              add_bias_quarter<BF16>(reinterpret_cast<float*>(&sr[32 * qq]), &bn[4 * qq], p.inv_scale);
          }
        } else if (HW_MAX) {
          // The row maximum of the raw scores comes with the load (used where
          // no key of the tile is masked and the transform keeps the order).
          uint32_t m4[W / 32];
#pragma unroll
          for (int qq = 0; qq < W / 32; ++qq)
            tmem_ld32_max(tS + 32 * qq, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * qq]),
                          *reinterpret_cast<float*>(&m4[qq]));
          tmem_ld_wait();
          reg_fence(sr);
          reg_fence(m4);
          static_assert(W == 128, "four partial maxima");
          raw_max = fmaxf(fmax3(__uint_as_float(m4[0]), __uint_as_float(m4[1]),
                                __uint_as_float(m4[2])), __uint_as_float(m4[3]));
        } else {
#pragma unroll
          for (int qq = 0; qq < W / 32; ++qq)
            tmem_ld32(tS + 32 * qq, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * qq]));
          tmem_ld_wait();
          reg_fence(sr);
        }
        // Raw scores in place; the soft-cap variant turns them into r (see
        // softcap_r_n: log2-unit score c (1 - 2 r), masked keys +inf), the
        // others keep them, with scale*log2(e) folded into the exponent's FMA
        // (CK MakeKargs FAST_EXP2 fold).
        float* s = reinterpret_cast<float*>(sr);
        if constexpr (XF == kXfSoftcap) {
          softcap_r_n<W>(s, p.scale * p.softcap_inv);
        } else if constexpr (XF == kXfAlibi) {
          // CK ALiBi position encoding (slope per (batch, head), aligned like
          // the mask): natural-log score - slope*|diag - j|, in raw-score
          // units (divided by the scale folded in later).
          // The distance |diag - j| in float from one conversion per row:
          // the column offsets are constants and every value is an integer
          // below 2^24, so the subtraction is exact.
          const int dq = qi + diag - j0;  // this row's diagonal, as a column
          const float fdq = static_cast<float>(dq);
          if (dq >= W - 1 || dq <= 0) {
            // All columns on one side of the diagonal: -slope*|dq - c| is
            // +-slope*(c - dq), two packed operations per pair of scores
            // (an exact subtraction, then the same single-rounding FMA).
            const float k = dq > 0 ? alibi_raw : -alibi_raw;
            const uint64_t k2 = f2_pack(k, k), nq2 = f2_pack(-fdq, -fdq);
#pragma unroll
            for (int i = 0; i < W / 2; ++i) {
              const uint64_t d2 = f2_add(f2_pack(static_cast<float>(2 * i), static_cast<float>(2 * i + 1)), nq2);
              f2_unpack(f2_fma(k2, d2, f2_pack(s[2 * i], s[2 * i + 1])), s[2 * i], s[2 * i + 1]);
            }
          } else {
#pragma unroll
            for (int c = 0; c < W; ++c)
              s[c] = fmaf(-alibi_raw, fabsf(fdq - static_cast<float>(c)), s[c]);
          }
        }
        // (The elementwise bias was added above, as the scores left tensor
        // memory.)
        // Row maximum in log2 units, and the exponent p = 2^(s a + b - msub).
        float a_coef, b_coef, m_cand;
        if constexpr (XF == kXfSoftcap) {
          a_coef = -2.0f * p.softcap * kLog2e;
          b_coef = p.softcap * kLog2e;
        } else {
          a_coef = p.scale_log2;
          b_coef = 0.0f;
        }
        if (HW_MAX && !masked) {
          if constexpr (XF == kXfSoftcap) {
            // min r is r of the largest raw score (r decreases with the
            // score), computed as softcap_r_n does for every score.
            const float r_min =
                rcp_approx(ex2_approx(raw_max * (p.scale * p.softcap_inv * 2.0f * kLog2e)) + 1.0f);
            m_cand = fmaf(r_min, a_coef, b_coef);  // c (1 - 2 min r)
          } else {
            m_cand = raw_max * a_coef;  // a_coef > 0: order kept
          }
        } else {
          if (masked) {
            int hi = it.Lk - 1 - j0, lo = 0;  // kept columns [lo, hi] of this row
            if (MASK && p.win_right >= 0) hi = min(hi, qi + diag + p.win_right - j0);
            if (MASK && p.win_left >= 0) lo = qi + diag - p.win_left - j0;
            constexpr float kDrop = XF == kXfSoftcap ? INFINITY : -INFINITY;  // a masked key
            if (lo <= 0) {  // no left bound inside the columns (plain causal or the tail)
#pragma unroll
              for (int c = 0; c < W; ++c) s[c] = c <= hi ? s[c] : kDrop;
            } else {
#pragma unroll
              for (int c = 0; c < W; ++c) s[c] = (c <= hi && c >= lo) ? s[c] : kDrop;
            }
          }
          if constexpr (XF == kXfSoftcap)
            m_cand = fmaf(min_n<W>(s), a_coef, b_coef);  // c (1 - 2 min r); -inf if all masked
          else
            m_cand = max_n<W>(s) * a_coef;  // a_coef > 0: order kept
        }
        const float m_new = fmaxf(m_use, m_cand);
        float alpha = 1.0f;
        if (m_new - m_use > 8.0f) {  // false when both are -inf (NaN compare)
          alpha = ex2_approx(m_use - m_new);
          m_use = m_new;
        }
        const float msub = (m_use == -INFINITY) ? 0.0f : m_use;
        // The P.V MMA of the previous K/V tile finished before this S was
        // produced (its commit covers every earlier MMA), so O can be
        // rescaled now; with P in halves, before the first half goes out.
        auto rescale_o = [&]() {
          if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll
            for (int c = 0; c < D; c += 32) {
              uint32_t ov[32];
              tmem_ld32(tO + c, ov);
              tmem_ld_wait();
              reg_fence(ov);
#pragma unroll
              for (int i = 0; i < 32; ++i)
                ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
              tmem_st32(tO + c, ov);
            }
          }
        };
        uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};  // +0.0f in both lanes
        uint32_t pk[W / 2];
        const uint64_t a2 = f2_pack(a_coef, a_coef), b2 = f2_pack(b_coef - msub, b_coef - msub);
        if constexpr (HALVES) {
          static_assert(W == 128, "P halves of one 32-column store each");
          exp_pack_row<BF16, W / 4>(s, a2, b2, pk, acc2);
          tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
          rescale_o();  // (here, with half of the scores consumed: fewer live registers)
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&sm.p_half[t]);
          exp_pack_row<BF16, W / 4>(s + W / 2, a2, b2, pk + W / 4, acc2);
          tmem_st32(tS + W / 4, *reinterpret_cast<uint32_t(*)[32]>(&pk[W / 4]));
        } else {
          exp_pack_row<BF16, W / 2>(s, a2, b2, pk, acc2);
          // P over the first W/2 columns of S.
#pragma unroll
          for (int qq = 0; qq < W / 64; ++qq)
            tmem_st32(tS + 32 * qq, *reinterpret_cast<uint32_t(*)[32]>(&pk[32 * qq]));
        }
        float r0, r1;
        f2_unpack(f2_add(f2_add(acc2[0], acc2[1]), f2_add(acc2[2], acc2[3])), r0, r1);
        l = l * alpha + (r0 + r1);
        if constexpr (!HALVES) rescale_o();
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sm.p_full[t]);
        if constexpr (XF == kXfBias)
          if (qi < it.Lq && j + 1 < nt) fetch_bias(j + 1);
      }
      if (!ok) break;

      // ---- epilogue: O = O / l, LSE = ln(l) + m (FA2 final rescale; FA3 store)
      bool have_o = false;
      if (nt > 0) {
        have_o = __all_sync(0xffffffffu, w.wait(&sm.o_final[t], oc & 1, kErrPrefillOFinal));
        ++oc;
        if (!have_o) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      const float msub = (m_use == -INFINITY) ? 0.0f : m_use;
      const bool row_ok = qi < it.Lq;
      float oscale;  // 1 / denominator (with the sink's share)
      float mfin = msub, ltot = l;
      if (p.sink != nullptr) {
        const float sl = p.sink[hr] * kLog2e;
        if (l > 0.0f) {
          mfin = fmaxf(msub, sl);
          const float a = ex2_approx(msub - mfin);
          ltot = l * a + ex2_approx(sl - mfin);
          oscale = a / ltot;
        } else {
          mfin = sl;
          ltot = 1.0f;
          oscale = 0.0f;
        }
      } else {
        oscale = (l > 0.0f) ? 1.0f / l : 0.0f;
      }
      const float lse_out = (ltot > 0.0f) ? (mfin + __log2f(ltot)) * kLn2 : -INFINITY;  // natural log
      // The warp's 32 rows are 32 consecutive queries of one head when the
      // stores go by TMA (host: at most 4 heads per tile): its first one and
      // its head are the box's coordinates.
      const int wq0 = mt + (((warp & 3) * 32) & qmask);
      const int wh = it.h + (((warp & 3) * 32) >> p.qpt_log2);
      // The previous item's stores have read the stages (they had this
      // item's K/V steps to do it, so this rarely waits).
      if (p.o_tma || p.lse_tma) {
        if (lane == 0) bulk_wait_read();
        __syncwarp();
      }
      if (p.lse_tma) {
        // Rows past Lq fall outside the map: whatever they hold is not written.
        sm.lstage[warp][lane] = lse_out;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && wq0 < it.Lq) {  // (a warp with no row inside issues nothing)
          if constexpr (ATTN_L2_HINTS)
            tma_store_3d_hint(&p.tm_lse, sm.lstage[warp], wq0, wh, it.b, l2_policy_evict_first());
          else
            tma_store_3d(&p.tm_lse, sm.lstage[warp], wq0, wh, it.b);
          bulk_commit();
        }
      } else if (row_ok && p.lse != nullptr) {
        p.lse[it.b * p.lse_batch + hr * p.lse_head + it.rq0 + qi] = lse_out;
      }
      constexpr int OB = FP8 ? 1 : 2;  // bytes per output element
      // Output row of tile row R (its head and query; valid while the query
      // is inside the sequence).
      auto orow = [&](int R, bool& valid) -> uint8_t* {
        const int q = mt + (R & qmask);
        valid = q < it.Lq;
        return reinterpret_cast<uint8_t*>(p.o) +
               (it.b * p.o_batch + static_cast<int64_t>(it.h + (R >> p.qpt_log2)) * p.o_head +
                static_cast<int64_t>(it.rq0 + q) * p.o_row) * OB;
      };
      if (have_o) {
        // O is read from tensor memory first (one wait) and goes back to the
        // MMA warp before any packing or store; then RB bytes of each row per
        // round: each thread packs its row into the stage (16-byte pieces,
        // XOR-swizzled like the TMA store's 64- or 128-byte swizzle, so 8
        // consecutive rows hit distinct banks).  Dense problems then store the
        // stage with one TMA store per round (the FlashAttention-3 epilogue's
        // non-varlen path); the others write 32 / (RB / 16) rows x RB bytes
        // per instruction, row by row predicated (a box cannot stop at a
        // packed sequence's end).  Rounds of 128 bytes where the host asks
        // for them (problems without PackGQA: measured faster there, slower
        // with packed heads), else 64.
        const uint64_t pol_o = l2_policy_evict_first();
        (void)pol_o;
        if constexpr (FP8) oscale *= p.o_scale;  // FP8 static quantisation: scale_p * scale_o
        uint32_t ov[D];
#pragma unroll
        for (int c = 0; c < D; c += 32) tmem_ld32(tO + c, *reinterpret_cast<uint32_t(*)[32]>(&ov[c]));
        tmem_ld_wait();
        reg_fence(ov);
        tc_fence_before();
        mbar_arrive(&sm.o_free[t]);
        const bool tma = p.o_tma != 0;
        uint4* stage = sm.ostage[warp];
        auto rounds = [&](auto rb_c) {
          constexpr int RB = decltype(rb_c)::value;  // bytes of each row per round
          constexpr int RC = RB / OB;                // columns per round
          constexpr int LPR = RB / 16;               // 16-byte pieces of a row per round
          static_assert(RB == 64 || RB == 128, "64- or 128-byte rounds");
          const int lr = lane;
          auto sw = [](int R) { return ((R * RB) >> 7) & (LPR - 1); };  // piece q of row R at q ^ sw(R)
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += RC) {
            if (tma && c0 > 0) {  // the previous round's store has read the stage
              if (lane == 0) bulk_wait_read();
              __syncwarp();
            }
            if constexpr (FP8) {
#pragma unroll
              for (int q = 0; q < LPR; ++q) {  // 16 e4m3 columns per 16-byte piece
                uint32_t w4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const uint32_t* x = &ov[c0 + 16 * q + 4 * i];
                  w4[i] = pack_e4m3x4(__uint_as_float(x[0]) * oscale, __uint_as_float(x[1]) * oscale,
                                      __uint_as_float(x[2]) * oscale, __uint_as_float(x[3]) * oscale);
                }
                stage[lr * LPR + (q ^ sw(lr))] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
              }
            } else {
#pragma unroll
              for (int q = 0; q < LPR; ++q) {  // 8 fp16/bf16 columns per 16-byte piece
                uint32_t w4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const float a = __uint_as_float(ov[c0 + 8 * q + 2 * i]) * oscale;
                  const float bb = __uint_as_float(ov[c0 + 8 * q + 2 * i + 1]) * oscale;
                  w4[i] = BF16 ? pack_bf16(a, bb) : pack_f16(a, bb);
                }
                stage[lr * LPR + (q ^ sw(lr))] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
              }
            }
            if (tma) {
              fence_proxy_async_smem();  // the stage, written here, is read by the async proxy
              __syncwarp();
              if (lane == 0) {
                if constexpr (ATTN_L2_HINTS) tma_store_4d_hint(&p.tm_o, stage, c0, wq0, wh, it.b, pol_o);
                else tma_store_4d(&p.tm_o, stage, c0, wq0, wh, it.b);
                bulk_commit();
              }
              continue;
            }
            __syncwarp();
#pragma unroll
            for (int k = 0; k < LPR; ++k) {  // 32 / LPR rows per instruction
              const int rw = (32 / LPR) * k + lr / LPR, q = lr % LPR;
              const uint4 v4 = stage[rw * LPR + (q ^ sw(rw))];
              bool valid;
              uint8_t* dst = orow((warp & 3) * 32 + rw, valid);
              if (valid) {
                if constexpr (ATTN_L2_HINTS) st_global_v4_hint(dst + c0 * OB + 16 * q, v4, pol_o);
                else *reinterpret_cast<uint4*>(dst + c0 * OB + 16 * q) = v4;
              }
            }
            __syncwarp();
          }
        };
        if constexpr (kStageRowBytes<C, ORD> == 128) {
          if (p.o_tma == 64) rounds(std::integral_constant<int, 64>{});
          else rounds(std::integral_constant<int, 128>{});
        } else {
          rounds(std::integral_constant<int, 64>{});
        }
      } else if (row_ok) {
        bool valid;  // == row_ok
        uint4* dst = reinterpret_cast<uint4*>(orow(r, valid));
        (void)valid;
#pragma unroll
        for (int i = 0; i < D * OB / 16; ++i) dst[i] = make_uint4(0, 0, 0, 0);
      }
    }
    // Every tensor store this warp issued has completed before the CTA ends.
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

template <int D, int DT, bool MASK, int XF, bool ORD = false>
static cudaError_t launch_prefill_t(const PrefillParams& p, int grid, cudaStream_t stream) {
  using C = PrefillCfg<D, DT>;
  auto kern = attn_prefill_kernel<D, DT, MASK, XF, ORD>;
  const int smem = static_cast<int>(sizeof(PrefillSmem<C, ORD>)) + 1024;
  static_assert(sizeof(PrefillSmem<C, ORD>) + 1024 <= 227 * 1024, "shared memory per block");
  static bool configured = false;  // per instantiation; attribute set is idempotent
  if (!configured) {
    // The softmax warpgroups raise their register budget with setmaxnreg,
    // drawing on what the block was launched with: the kernel must have been
    // built with exactly the launch count the split assumes, else that
    // instruction would wait forever.  Refuse to launch otherwise.
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != C::LAUNCH_REGS) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  kern<<<grid, C::THREADS, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int DT, bool MASK>
static cudaError_t launch_prefill_x(const PrefillParams& p, int grid, int xf,
                                   cudaStream_t stream) {
  // Group mode and paged caches take the sorted work order (no bias there).
  if (p.cu_q != nullptr || p.seqlens_k != nullptr) {
    switch (xf) {
      case kXfNone: return launch_prefill_t<ATTN_PREFILL_D, DT, MASK, kXfNone, true>(p, grid, stream);
      case kXfSoftcap:
        return launch_prefill_t<ATTN_PREFILL_D, DT, MASK, kXfSoftcap, true>(p, grid, stream);
      case kXfAlibi: return launch_prefill_t<ATTN_PREFILL_D, DT, MASK, kXfAlibi, true>(p, grid, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (xf) {
    case kXfNone: return launch_prefill_t<ATTN_PREFILL_D, DT, MASK, kXfNone>(p, grid, stream);
    case kXfSoftcap: return launch_prefill_t<ATTN_PREFILL_D, DT, MASK, kXfSoftcap>(p, grid, stream);
    case kXfAlibi: return launch_prefill_t<ATTN_PREFILL_D, DT, MASK, kXfAlibi>(p, grid, stream);
    case kXfBias: return launch_prefill_t<ATTN_PREFILL_D, DT, MASK, kXfBias>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <>
cudaError_t launch_prefill_d<ATTN_PREFILL_D>(const PrefillParams& p, int grid, int dt,
                                             bool masked, int xf, cudaStream_t stream) {
  if (dt == kDtBF16) return masked ? launch_prefill_x<kDtBF16, true>(p, grid, xf, stream)
                                   : launch_prefill_x<kDtBF16, false>(p, grid, xf, stream);
  if (dt == kDtF16) return masked ? launch_prefill_x<kDtF16, true>(p, grid, xf, stream)
                                  : launch_prefill_x<kDtF16, false>(p, grid, xf, stream);
#if ATTN_PREFILL_D == 128
  // FP8 static quantisation: head dimension 128, no score transform.
  if (dt == kDtE4M3 && xf == kXfNone) {
    if (p.cu_q != nullptr)
      return masked ? launch_prefill_t<128, kDtE4M3, true, kXfNone, true>(p, grid, stream)
                    : launch_prefill_t<128, kDtE4M3, false, kXfNone, true>(p, grid, stream);
    return masked ? launch_prefill_t<128, kDtE4M3, true, kXfNone>(p, grid, stream)
                  : launch_prefill_t<128, kDtE4M3, false, kXfNone>(p, grid, stream);
  }
#endif
  return cudaErrorInvalidValue;
}

}  // namespace attn
