// decode_kernel.cuh -- paged-KV split-KV attention forward (decode and short query
// chunks) on sm_103a, compiled once per head dimension (decode_d64.cu,
// decode_d128.cu define ATTN_DECODE_D and include this).
//
// Prior art on the pages: the Composable Kernel fmha_fwd_pagedkv_kernel.hpp
// page block navigator (physical page = block_table[b][logical page], page
// stride, kv-head offset, partial last page) and the FlashAttention-3
// hopper/epilogue_fwd.hpp split layout (partial O and LSE per split, O = 0 /
// LSE = -inf for an empty split).  The design here is Blackwell-first:
//
//  * one CTA per (split, kv head, batch).  The R = Lq * (Hq/Hkv) query rows
//    that share the kv head (PackGQA-style packing, row = query * g + head
//    in group) are padded to N = 16 and the scores are computed transposed,
//    S^T[128 keys x 16] = K_blk . Q^T, with tcgen05.mma (M = 128 keys), so
//    each K/V byte is read from HBM once for all g heads.
//  * O^T[d x 16] += V_blk^T . P^T accumulates in tensor memory (A = V read
//    MN-major straight from the TMA tile, B = P^T written to shared memory
//    by the softmax threads).
//  * a TMA producer warp gathers pages through the block table into ONE ring
//    in consumption order K0, K1, V0, K2, V1, ..., so HBM streams
//    continuously; the ring holds 3 x 32 KB (d = 128), two CTAs per SM.
//  * softmax: thread = key lane.  Per block the row maxima are all-reduced
//    (warp butterfly + 4-way shared-memory exchange); row sums stay
//    per-thread until the end of the split.  O is rescaled only when a row
//    max grows by more than 8 (log2 units), as in the prefill kernel.
#pragma once
#include "ptx.cuh"
#include "common.cuh"
#include "launch.h"

#include <cstdio>
#include <type_traits>

namespace attn {

template <int D_>
struct DecodeCfg {
  static constexpr int D = D_;
  static constexpr int BK = 128;                       // keys per block
  static constexpr int NR = 16;                        // padded query rows (MMA N)
  static constexpr int NCHUNK = D / 64;
  static constexpr int BLK_BYTES = BK * D * 2;         // one K or V block
  static constexpr int CHUNK_BYTES = BK * 128;         // one 64-wide column of a block
  static constexpr int NSLOT = (D == 128) ? 3 : 6;     // ring depth (items)
  static constexpr int THREADS = 192;
  static constexpr uint32_t TM_COLS = 64;
  __device__ static constexpr uint32_t tm_s(int i) { return 16u * (i & 1); }
  static constexpr uint32_t TM_O = 32;
};

template <class C>
struct DecodeSmem {
  alignas(1024) uint8_t ring[C::NSLOT][C::BLK_BYTES];
  alignas(1024) uint8_t q[C::NCHUNK][C::NR * 128];      // Q rows, K-major SW128
  alignas(1024) uint8_t pt[2][2][C::NR * 128];          // P^T [buf][key chunk] SW128
  float red[2][4][C::NR];                               // per-warp row maxima
  float lred[4][C::NR];                                 // per-warp row sums
  uint64_t full[C::NSLOT], empty[C::NSLOT];
  uint64_t q_ready, s_full[2], p_full[2], o_done, teardown;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ float tanh_via_exp2_d(float y) {
  const float e = ex2_approx(y * (2.0f * kLog2e));
  return 1.0f - 2.0f * rcp_approx(e + 1.0f);
}

__device__ __forceinline__ bool wait_raw_d(uint64_t* bar, uint32_t parity, uint64_t deadline) {
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() > deadline) return false;
  }
  return true;
}

// Max over the 32 lanes of each of 16 values.  On return lane l holds the
// result for row  8*b4 + 4*b3 + 2*b2 + b1  (b_k = bit k of l); lanes l and
// l^1 hold the same row.
template <bool MAX>
__device__ __forceinline__ float butterfly16(const float (&a)[16]) {
  const int lane = threadIdx.x & 31;
  float b[8], c[4], d2[2];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool hi = lane & 16;
    const float send = hi ? a[i] : a[i + 8];
    const float keep = hi ? a[i + 8] : a[i];
    const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
    b[i] = MAX ? fmaxf(keep, recv) : keep + recv;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool hi = lane & 8;
    const float send = hi ? b[i] : b[i + 4];
    const float keep = hi ? b[i + 4] : b[i];
    const float recv = __shfl_xor_sync(0xffffffffu, send, 8);
    c[i] = MAX ? fmaxf(keep, recv) : keep + recv;
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool hi = lane & 4;
    const float send = hi ? c[i] : c[i + 2];
    const float keep = hi ? c[i + 2] : c[i];
    const float recv = __shfl_xor_sync(0xffffffffu, send, 4);
    d2[i] = MAX ? fmaxf(keep, recv) : keep + recv;
  }
  float e;
  {
    const bool hi = lane & 2;
    const float send = hi ? d2[0] : d2[1];
    const float keep = hi ? d2[1] : d2[0];
    const float recv = __shfl_xor_sync(0xffffffffu, send, 2);
    e = MAX ? fmaxf(keep, recv) : keep + recv;
  }
  const float recv = __shfl_xor_sync(0xffffffffu, e, 1);
  return MAX ? fmaxf(e, recv) : e + recv;
}
__device__ __forceinline__ int butterfly16_row(int lane) {
  return ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 +
         ((lane >> 1) & 1);
}

// FEAT: 0 = no mask and no ALiBi (the decode fast path), 1 = causal / window
// masks (either alignment), 2 = masks and ALiBi.  Only the instantiations a
// call needs pay for the per-key checks.
template <int D, bool BF16, bool SOFTCAP, int FEAT>
__global__ void __launch_bounds__(192, 2)
    attn_decode_kernel(const __grid_constant__ DecodeParams p) {
  using C = DecodeCfg<D>;
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  extern __shared__ uint8_t smem_raw[];
  DecodeSmem<C>& sm = *reinterpret_cast<DecodeSmem<C>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int split = blockIdx.x;
  const int hk = blockIdx.y;
  const int b = blockIdx.z;
  const int g = p.Hq / p.Hkv;
  const int R = p.Lq * g;  // real query rows (<= 16)
  const int L = p.seqlens_k[b];
  const int P = p.page_size;
  const int pages_b = (L + P - 1) / P;
  // With a left window the splits tile only the pages holding kept keys:
  // every row's right bound reaches the last key, the first row's left bound
  // is the lowest.
  const int diag0 = p.top_left ? 0 : L - p.Lq;  // key on query row 0's diagonal
  const int k_lo = (FEAT > 0 && p.win_left >= 0) ? max(0, diag0 - p.win_left) : 0;
  const int pg0 = k_lo / P + split * p.chunk_pages;
  const int pg1 = min(pg0 + p.chunk_pages, pages_b);
  const int k0 = pg0 * P;
  const int k1 = min(pg1 * P, L);
  const int nblk = (k1 > k0) ? (k1 - k0 + C::BK - 1) / C::BK : 0;
  const bool partial_out = p.num_splits > 1;
  const int64_t rows_total = static_cast<int64_t>(p.B) * p.Hq * p.Lq;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Row rho = qi * g + hg  <->  query head h = hk * g + hg, query qi.
  auto out_row = [&](int rho, int& h, int& qi) {
    qi = rho / g;
    h = hk * g + (rho - qi * g);
  };

  if (nblk == 0) {
    // Empty split (FlashAttention-3 store_zero): O = 0, LSE = -inf; without
    // splits the final row is written directly (sink-only rows keep LSE = sink).
    for (int idx = threadIdx.x; idx < R * D; idx += blockDim.x) {
      const int rho = idx / D, c = idx - rho * D;
      int h, qi;
      out_row(rho, h, qi);
      if (partial_out) {
        p.o_part[((static_cast<int64_t>(split) * rows_total) +
                  (static_cast<int64_t>(b) * p.Hq + h) * p.Lq + qi) * D + c] = 0.0f;
      } else {
        reinterpret_cast<T*>(p.o)[((static_cast<int64_t>(b) * p.Lq + qi) * p.Hq + h) * D + c] =
            T(0.0f);
      }
    }
    for (int rho = threadIdx.x; rho < R; rho += blockDim.x) {
      int h, qi;
      out_row(rho, h, qi);
      const int64_t r = (static_cast<int64_t>(b) * p.Hq + h) * p.Lq + qi;
      if (partial_out) {
        p.lse_part[split * rows_total + r] = -INFINITY;
      } else if (p.lse != nullptr) {
        p.lse[r] = p.sink != nullptr ? p.sink[h] : -INFINITY;
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    mbar_init(&sm.q_ready, 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.p_full[i], 128);
    }
    mbar_init(&sm.o_done, 1);
    mbar_init(&sm.teardown, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&sm.tmem_base, C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const Waiter w{globaltimer_ns() + p.timeout_ns, &sm.abort_flag, p.err};

  // Item order in the ring: K0, K1, V0, K2, V1, ..., K_{n-1}, V_{n-2}, V_{n-1}.
  // Item index of K_i is (i == 0 ? 0 : 2i - 1); of V_i is 2i + 2 (i < n-1),
  // and V_{n-1} is the last item 2n - 1.
  auto k_item = [](int i) { return i == 0 ? 0 : 2 * i - 1; };
  auto v_item = [nblk](int i) { return i == nblk - 1 ? 2 * nblk - 1 : 2 * i + 2; };
  const int n_items = 2 * nblk;

  if (warp == 4) {
    // ======================= TMA producer (page gather) ======================
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      const int BR = min(P, C::BK);  // rows per box
      const int32_t* bt = p.block_table + static_cast<int64_t>(b) * p.max_pages;
      const int oob_row = p.num_pages * P;  // past the pool: TMA fills zeros
      int armed = 0;
      for (int it = 0; it < n_items; ++it) {
        // item -> (is_v, block)
        int blk;
        bool is_v;
        if (it == 0) { blk = 0; is_v = false; }
        else if (it == n_items - 1) { blk = nblk - 1; is_v = true; }
        else if (it & 1) { blk = (it + 1) / 2; is_v = false; }   // K_{(it+1)/2}
        else { blk = it / 2 - 1; is_v = true; }                    // V_{it/2 - 1}
        const int s = it % C::NSLOT;
        if (!w.wait(&sm.empty[s], ((it / C::NSLOT) & 1) ^ 1, kErrDecodeEmpty)) break;
        mbar_arrive_expect_tx(&sm.full[s], C::BLK_BYTES);
        const CUtensorMap* map = is_v ? &p.tm_v : &p.tm_k;
        const int kb = k0 + blk * C::BK;
        for (int r0 = 0; r0 < C::BK; r0 += BR) {
          const int key = kb + r0;
          int row = oob_row;
          if (key < k1) {
            const int lp = key / P;
            const int phys = lp < p.max_pages ? bt[lp] : -1;
            if (phys >= 0 && phys < p.num_pages) {
              row = phys * P + (key - lp * P);
            } else if (p.err) {
              atomicOr(p.err, 1u << kErrDecodeBadPage);
            }
          }
#pragma unroll
          for (int c = 0; c < C::NCHUNK; ++c)
            tma_load_3d(sm.ring[s] + c * C::CHUNK_BYTES + r0 * 128, map, &sm.full[s], c * 64,
                        hk, row);
        }
        ++armed;
      }
      if (w.aborted()) {
        const uint64_t dl = globaltimer_ns() + 50000000ull;
        for (int it = max(0, armed - C::NSLOT); it < armed; ++it)
          wait_raw_d(&sm.full[it % C::NSLOT], (it / C::NSLOT) & 1, dl);
      }
    }
  } else if (warp == 5) {
    // ======================= MMA issuer ======================================
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16_f32(BF16, 128, C::NR, false, false);
      constexpr uint32_t idesc_o = idesc_f16_f32(BF16, 128, C::NR, true, false);
      const uint32_t qa = smem_u32(sm.q[0]);
      auto issue_s = [&](int i) {
        const int it = k_item(i), s = it % C::NSLOT;
        const uint32_t ka = smem_u32(sm.ring[s]);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t c = k >> 2, kin = (k & 3) * 32;
          umma_ss(tmem + C::tm_s(i), sdesc_sw128(ka + c * C::CHUNK_BYTES + kin, 16, 1024),
                  sdesc_sw128(qa + c * (C::NR * 128) + kin, 16, 1024), idesc_s,
                  k > 0 ? 1u : 0u);
        }
        umma_commit(&sm.s_full[i & 1]);
        umma_commit(&sm.empty[s]);
      };
      auto issue_pv = [&](int i) {
        const int it = v_item(i);
        const int s = it % C::NSLOT;
        const uint32_t va = smem_u32(sm.ring[s]);
        const uint32_t pa = smem_u32(sm.pt[i & 1][0]);
        // d = 64: the second 64-row half of M re-reads the same column (LBO 0)
        // and the duplicate lanes 64..127 of O^T are ignored.
        const uint32_t lbo = (C::NCHUNK > 1) ? C::CHUNK_BYTES : 0;
#pragma unroll
        for (int k = 0; k < C::BK / 16; ++k) {
          const uint32_t c = k >> 2, kin = (k & 3) * 32;
          umma_ss(tmem + C::TM_O, sdesc_sw128(va + k * 16 * 128, lbo, 1024),
                  sdesc_sw128(pa + c * (C::NR * 128) + kin, 16, 1024), idesc_o,
                  (i > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(&sm.o_done);
        umma_commit(&sm.empty[s]);
      };
      auto item_wait = [&](int it, uint32_t site) {
        return w.wait(&sm.full[it % C::NSLOT], (it / C::NSLOT) & 1, site);
      };
      bool ok = w.wait(&sm.q_ready, 0, kErrDecodeFull);
      for (int i = 0; ok && i < nblk; ++i) {
        ok = item_wait(k_item(i), kErrDecodeFull);
        if (!ok) break;
        tc_fence_after();
        issue_s(i);
        if (i >= 1) {
          const int pi = i - 1;
          ok = item_wait(v_item(pi), kErrDecodeFull) &&
               w.wait(&sm.p_full[pi & 1], (pi >> 1) & 1, kErrDecodeFull);
          if (!ok) break;
          tc_fence_after();
          issue_pv(pi);
        }
      }
      if (ok) {
        const int pi = nblk - 1;
        ok = item_wait(v_item(pi), kErrDecodeFull) &&
             w.wait(&sm.p_full[pi & 1], (pi >> 1) & 1, kErrDecodeFull);
        if (ok) {
          tc_fence_after();
          issue_pv(pi);
        }
      }
      umma_commit(&sm.teardown);
      if (!wait_raw_d(&sm.teardown, 0, globaltimer_ns() + 50000000ull) && p.err)
        atomicOr(p.err, 1u << kErrDecodeTeardown);
    }
  } else {
    // ======================= softmax / epilogue (128 threads) ================
    const int tid = threadIdx.x;  // 0..127 == TMEM lane == key in block / d index
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    // Q rows into shared memory (K-major, 128-byte swizzle), zero padding.
    {
      const T* qb = reinterpret_cast<const T*>(p.q);
      for (int idx = tid; idx < C::NR * (D / 8); idx += 128) {
        const int rho = idx / (D / 8), ch = idx - rho * (D / 8);  // 16-byte chunk
        uint4 val = make_uint4(0, 0, 0, 0);
        if (rho < R) {
          int h, qi;
          out_row(rho, h, qi);
          val = *reinterpret_cast<const uint4*>(
              qb + ((static_cast<int64_t>(b) * p.Lq + qi) * p.Hq + h) * D + ch * 8);
        }
        const int c = ch >> 3, cc = ch & 7;
        *reinterpret_cast<uint4*>(sm.q[c] + rho * 128 + ((cc ^ (rho & 7)) << 4)) = val;
      }
      fence_proxy_async_smem();
      mbar_arrive(&sm.q_ready);
    }
    float m_use[C::NR];   // exp2 subtrahend per row (log2 units), identical in all threads
    float lpart[C::NR];   // this thread's share of each row sum
#pragma unroll
    for (int r = 0; r < C::NR; ++r) {
      m_use[r] = -INFINITY;
      lpart[r] = 0.0f;
    }
    const int diag = diag0;  // key on query row 0's diagonal (bottom-right unless top-left)
    // ALiBi slope of each row's query head, in log2 units (CK position
    // encoding: -slope * |diag(i) - j| on the natural-log score).
    float al[C::NR];
#pragma unroll
    for (int r = 0; r < C::NR; ++r) {
      const int h = hk * g + (r % g);
      al[r] = (FEAT == 2 && r < R) ? p.alibi[b * p.alibi_stride + h] * kLog2e : 0.0f;
    }
    // Every thread runs every iteration and every named barrier even after a
    // timeout (waits then return at once), so the four warps never part ways
    // at a barrier.
    bool ok = true;
    for (int i = 0; i < nblk; ++i) {
      const bool got_s =
          __all_sync(0xffffffffu, w.wait(&sm.s_full[i & 1], (i >> 1) & 1, kErrDecodeFull));
      ok = ok && got_s;
      uint32_t sr[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) sr[r] = 0u;
      if (got_s) {
        tc_fence_after();
        tmem_ld16(tmem + C::tm_s(i) + lane_base, sr);
        tmem_ld_wait();
        reg_fence(sr);
      }
      const int key = k0 + i * C::BK + tid;
      float x[C::NR];
#pragma unroll
      for (int r = 0; r < C::NR; ++r) {
        float s = __uint_as_float(sr[r]);
        if constexpr (SOFTCAP) {
          s = p.softcap * kLog2e * tanh_via_exp2_d(s * p.scale * p.softcap_inv);
        } else {
          s *= p.scale_log2;
        }
        if constexpr (FEAT == 2)
          s = fmaf(-al[r], fabsf(static_cast<float>((r / g) + diag - key)), s);
        bool valid = (key < k1) && (r < R);
        if constexpr (FEAT > 0) {
          if (p.win_right >= 0) valid = valid && (key <= (r / g) + diag + p.win_right);
          if (p.win_left >= 0) valid = valid && (key >= (r / g) + diag - p.win_left);
        }
        x[r] = valid ? s : -INFINITY;
      }
      const float wmax = butterfly16<true>(x);
      if ((lane & 1) == 0) sm.red[i & 1][warp][butterfly16_row(lane)] = wmax;
      named_bar_sync(1, 128);
      float alpha[C::NR];
      bool any_rescale = false;
#pragma unroll
      for (int r = 0; r < C::NR; ++r) {
        const float mb = fmaxf(fmaxf(sm.red[i & 1][0][r], sm.red[i & 1][1][r]),
                               fmaxf(sm.red[i & 1][2][r], sm.red[i & 1][3][r]));
        const float m_new = fmaxf(m_use[r], mb);
        alpha[r] = 1.0f;
        if (m_new - m_use[r] > 8.0f) {
          alpha[r] = ex2_approx(m_use[r] - m_new);
          m_use[r] = m_new;
          any_rescale = true;
        }
      }
      // P^T[r][key] in bf16/fp16 into the K-major swizzled B tile.
      uint8_t* pt = sm.pt[i & 1][tid >> 6];
      const int kk = tid & 63;
#pragma unroll
      for (int r = 0; r < C::NR; ++r) {
        const float msub = (m_use[r] == -INFINITY) ? 0.0f : m_use[r];
        const float pv = ex2_approx(x[r] - msub);
        lpart[r] = lpart[r] * alpha[r] + pv;
        const T pe = T(pv);
        *reinterpret_cast<T*>(pt + r * 128 + (((kk >> 3) ^ (r & 7)) << 4) + (kk & 7) * 2) = pe;
      }
      // The last block: zero V rows past the split end so stale cache
      // contents can never reach the MMA (0 * NaN would).
      if (i == nblk - 1 && key >= k1) {
        const int it = (nblk == 1) ? 1 : 2 * nblk - 1;
        if (wait_raw_d(&sm.full[it % C::NSLOT], (it / C::NSLOT) & 1, w.deadline)) {
          uint8_t* vb = sm.ring[it % C::NSLOT];
#pragma unroll
          for (int c = 0; c < C::NCHUNK; ++c)
#pragma unroll
            for (int q16 = 0; q16 < 8; ++q16)
              *reinterpret_cast<uint4*>(vb + c * C::CHUNK_BYTES + tid * 128 + q16 * 16) =
                  make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      // Wait for P.V(i-1) at every step (phase i-1 of o_done; P.V(i-2) is
      // done, the S commit seen above covers it, so the parity is exact):
      // an O rescale needs it, and waiting for each phase in turn keeps the
      // final wait of the epilogue exact as well (o_done completes once per
      // P.V; a parity wait cannot tell phases two apart).
      if (ok && i > 0) {
        const bool got = __all_sync(0xffffffffu, w.wait(&sm.o_done, (i - 1) & 1, kErrDecodeFull));
        if (!got) {
          ok = false;
        } else if (any_rescale) {
          tc_fence_after();
          uint32_t ov[16];
          tmem_ld16(tmem + C::TM_O + lane_base, ov);
          tmem_ld_wait();
          reg_fence(ov);
#pragma unroll
          for (int r = 0; r < C::NR; ++r)
            ov[r] = __float_as_uint(__uint_as_float(ov[r]) * alpha[r]);
          tmem_st16(tmem + C::TM_O + lane_base, ov);
          tmem_st_wait();
        }
      }
      tc_fence_before();
      mbar_arrive(&sm.p_full[i & 1]);
    }
    // ---- end of split: row sums, then O^T / l and LSE ------------------------
    const float wsum = butterfly16<false>(lpart);
    if ((lane & 1) == 0) sm.lred[warp][butterfly16_row(lane)] = wsum;
    named_bar_sync(1, 128);
    float l[C::NR];
#pragma unroll
    for (int r = 0; r < C::NR; ++r)
      l[r] = (sm.lred[0][r] + sm.lred[1][r]) + (sm.lred[2][r] + sm.lred[3][r]);
    // Every step i >= 1 waited for P.V(i-1) (phase i-1 of o_done), so the
    // barrier is now in phase nblk-1 or nblk and this parity wait is exact.
    const bool have_o =
        __all_sync(0xffffffffu, ok && w.wait(&sm.o_done, (nblk - 1) & 1, kErrDecodeFull));
    if (have_o) {
      tc_fence_after();
      uint32_t ov[16];
      tmem_ld16(tmem + C::TM_O + lane_base, ov);
      tmem_ld_wait();
      reg_fence(ov);
      if (tid < D) {
        for (int r = 0; r < R; ++r) {
          int h, qi;
          out_row(r, h, qi);
          const int64_t row = (static_cast<int64_t>(b) * p.Hq + h) * p.Lq + qi;
          const float msub = (m_use[r] == -INFINITY) ? 0.0f : m_use[r];
          float oscale, lse;
          if (partial_out) {
            oscale = l[r] > 0.0f ? 1.0f / l[r] : 0.0f;
            lse = l[r] > 0.0f ? (msub + __log2f(l[r])) * kLn2 : -INFINITY;
            p.o_part[(split * rows_total + row) * D + tid] = __uint_as_float(ov[r]) * oscale;
            if (tid == 0) p.lse_part[split * rows_total + row] = lse;
          } else {
            float mfin = msub, ltot = l[r];
            if (p.sink != nullptr) {
              const float sl = p.sink[h] * kLog2e;
              if (l[r] > 0.0f) {
                mfin = fmaxf(msub, sl);
                const float a = ex2_approx(msub - mfin);
                ltot = l[r] * a + ex2_approx(sl - mfin);
                oscale = a / ltot;
              } else {
                mfin = sl;
                ltot = 1.0f;
                oscale = 0.0f;
              }
            } else {
              oscale = l[r] > 0.0f ? 1.0f / l[r] : 0.0f;
            }
            lse = ltot > 0.0f ? (mfin + __log2f(ltot)) * kLn2 : -INFINITY;
            reinterpret_cast<T*>(p.o)[((static_cast<int64_t>(b) * p.Lq + qi) * p.Hq + h) * D +
                                      tid] = T(__uint_as_float(ov[r]) * oscale);
            if (tid == 0 && p.lse != nullptr) p.lse[row] = lse;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

template <int D, bool BF16, bool SOFTCAP, int FEAT>
static cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t stream) {
  using C = DecodeCfg<D>;
  auto kern = attn_decode_kernel<D, BF16, SOFTCAP, FEAT>;
  const int smem = static_cast<int>(sizeof(DecodeSmem<C>)) + 1024;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(p.num_splits, p.Hkv, p.B);
  kern<<<grid, C::THREADS, smem, stream>>>(p);
  return cudaGetLastError();
}

template <bool BF16>
static cudaError_t launch_decode_f(const DecodeParams& p, bool softcap, int feat,
                                   cudaStream_t stream) {
  if (softcap) {  // ALiBi with the soft-cap is rejected before launch
    if (feat == 0) return launch_decode_t<ATTN_DECODE_D, BF16, true, 0>(p, stream);
    if (feat == 1) return launch_decode_t<ATTN_DECODE_D, BF16, true, 1>(p, stream);
    return cudaErrorInvalidValue;
  }
  if (feat == 0) return launch_decode_t<ATTN_DECODE_D, BF16, false, 0>(p, stream);
  if (feat == 1) return launch_decode_t<ATTN_DECODE_D, BF16, false, 1>(p, stream);
  if (feat == 2) return launch_decode_t<ATTN_DECODE_D, BF16, false, 2>(p, stream);
  return cudaErrorInvalidValue;
}

template <>
cudaError_t launch_decode_d<ATTN_DECODE_D>(const DecodeParams& p, bool bf16, bool softcap,
                                           int feat, cudaStream_t stream) {
  return bf16 ? launch_decode_f<true>(p, softcap, feat, stream)
              : launch_decode_f<false>(p, softcap, feat, stream);
}

}  // namespace attn
