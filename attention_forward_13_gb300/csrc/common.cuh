// common.cuh -- parameter blocks and small device helpers shared by the
// attention kernels of this library (prefill, paged decode, combine).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

// Bytes of each output row the dense prefill epilogue stages and stores per
// round (one TMA store per softmax warp and round): 128 without PackGQA, 64
// with packed heads (measured) and for FP8 (whose widened V buffers take the
// shared memory a 128-byte stage would need).
#ifndef ATTN_O_ROUND_BYTES
#define ATTN_O_ROUND_BYTES 128
#endif

namespace attn {

constexpr int prefill_o_round_bytes(bool fp8, int pack) {
  return (fp8 || pack > 1) ? 64 : ATTN_O_ROUND_BYTES;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Device error word bits (one per wait site / check).
enum ErrBits : uint32_t {
  kErrPrefillQ = 0,
  kErrPrefillKFull = 1,
  kErrPrefillVFull = 2,
  kErrPrefillKEmpty = 3,
  kErrPrefillVEmpty = 4,
  kErrPrefillSFull = 5,
  kErrPrefillPFull = 6,
  kErrPrefillOFinal = 7,
  kErrPrefillTeardown = 8,
  kErrPrefillBadPage = 9,
  kErrDecodeFull = 12,
  kErrDecodeEmpty = 13,
  kErrDecodeBadPage = 14,
  kErrDecodeTeardown = 15,
  kErrSelftest = 20,
};

// Element types of a prefill instantiation: fp16 / bf16 end to end, or e4m3
// Q/K/V/O (FP8 static quantisation: S on the kind::f8f6f4 tensor path, V
// widened to fp16 on chip for P.V, O scaled and saturated to e4m3).
enum PrefillDt : int { kDtF16 = 0, kDtBF16 = 1, kDtE4M3 = 2 };

// Score transform of a prefill instantiation (applied to the raw score
// before masking).
enum ScoreXf : int { kXfNone = 0, kXfSoftcap = 1, kXfAlibi = 2, kXfBias = 3 };

// Bounds of the host-packed static schedule carried in PrefillParams, chosen
// so that the launch parameters stay within 4 KB.
constexpr int kSchedMaxCtas = 160;
constexpr int kSchedMaxItems = 1408;

// Prefill (dense / varlen) launch parameters.  Tensor maps are 4-D
// (d, rows, heads, batch); varlen problems use one batch slot and a row base.
struct PrefillParams {
  CUtensorMap tm_q;
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  // Dense problems whose softmax warps each own 32 consecutive queries of one
  // head (no packing, or at most 4 heads per tile): the epilogue stores O and
  // LSE by TMA through these maps (o_tma / lse_tma nonzero).  O: 4-D
  // (d, Lq, Hq, B), box {o_tma bytes of d (64 or 128), 32 rows, 1, 1},
  // swizzle of the same width; LSE: 3-D (Lq, Hq, B) fp32, box {32, 1, 1}.
  // Rows past Lq fall outside the maps and are not written.
  CUtensorMap tm_o;
  CUtensorMap tm_lse;
  int o_tma, lse_tma;  // o_tma: bytes of each row per store (0: no map)
  void* o;
  float* lse;
  int64_t o_row, o_head, o_batch;  // element strides of O
  int64_t lse_head, lse_batch;     // element strides of LSE (row stride 1)
  const int32_t* cu_q;             // varlen: [B+1] (nullptr in batch mode)
  const int32_t* cu_k;
  const float* sink;               // [Hq] or nullptr
  int B, Hq, Hkv, Lq, Lk;          // batch-mode lengths (ignored for varlen)
  int total_q, total_k;            // varlen: packed extents (sequences are clamped to them)
  // Query heads per work item (PackGQA): 1, or g = Hq / Hkv when the g query
  // heads of a kv head share every tile.  A 128-row tile then holds
  // qpt = 128 / pack queries of each of the pack heads, head-major (row
  // r <-> head h0 + (r >> qpt_log2), query m0 + (r & (qpt - 1))), as one
  // TMA box {d, qpt queries, pack heads} lands them.
  int pack;
  int qpt_log2;                    // log2(queries per 128-row tile)
  int units;                       // Hq / pack: head groups per batch
  int num_m_blocks;                // query blocks (two tiles) per (b, head group)
  int num_items;                   // num_m_blocks * B * units work items
  float scale_log2;                // scale * log2(e)
  float scale;                     // plain scale (soft-cap path)
  float softcap;                   // cap (> 0 when the soft-cap variant runs)
  float softcap_inv;               // 1 / cap
  // Key bounds of query row i (bottom-right aligned): i + Lk - Lq - win_left
  // <= j <= i + Lk - Lq + win_right; a negative bound is unbounded.  Causal
  // masking is win_right = 0.  Only read by the masked instantiations.
  int win_left, win_right;
  int top_left;                    // masks and ALiBi aligned top-left (row i on key i)
  float o_scale;                   // FP8 static quantisation: scale_p * scale_o on O
  float inv_scale;                 // 1 / scale (bias and ALiBi go to raw-score units)
  const float* alibi;              // ALiBi slopes, (b, h) at b * alibi_stride + h
  int alibi_stride;
  const void* bias;                // elementwise bias (input dtype), batch mode only
  int64_t bias_row, bias_head, bias_batch;  // its element strides (key stride 1)
  // Paged KV cache (chunked prefill): tm_k / tm_v are then 3-D maps
  // (d, Hkv, num_pages * page_size) over the pools, and sequence b has
  // seqlens_k[b] keys; nullptr otherwise.
  const int32_t* block_table;
  const int32_t* seqlens_k;
  int page_size, max_pages, num_pages;
  unsigned int* err;
  uint64_t timeout_ns;
  // Dense masked problems: a static assignment of the work items to CTAs,
  // packed on the host (sched_n > 0).  CTA c takes items
  // sched_item[sched_off[c]] .. sched_item[sched_off[c + 1] - 1] in order;
  // sched_n == 0: the snake order over the plain item list.
  int sched_n;
  uint16_t sched_off[kSchedMaxCtas + 1];
  uint16_t sched_item[kSchedMaxItems];
};
static_assert(sizeof(PrefillParams) <= 4096, "prefill launch parameters exceed 4 KB");

// Paged split-KV decode parameters.
struct DecodeParams {
  CUtensorMap tm_k;  // 3-D (d, Hkv, num_pages * page_size)
  CUtensorMap tm_v;
  const void* q;     // [B][Lq][Hq][d]
  const int32_t* block_table;
  const int32_t* seqlens_k;
  void* o;           // final O [B][Lq][Hq][d] (num_splits == 1)
  float* lse;        // final LSE [B][Hq][Lq] or nullptr (num_splits == 1)
  float* o_part;     // [S][B][Hq][Lq][d] (num_splits > 1)
  float* lse_part;   // [S][B][Hq][Lq]
  const float* sink; // [Hq] or nullptr (used only when num_splits == 1)
  int B, Lq, Hq, Hkv, page_size, num_pages, max_pages, num_splits, chunk_pages;
  float scale_log2, scale, softcap, softcap_inv;
  int win_left, win_right;  // as in PrefillParams (causal is win_right = 0)
  int top_left;
  const float* alibi;       // ALiBi slopes as in PrefillParams, or nullptr
  int alibi_stride;
  unsigned int* err;
  uint64_t timeout_ns;
};

struct CombineParams {
  const float* o_part;
  const float* lse_part;
  const float* sink;
  void* o;
  float* lse;
  int num_splits, B, Hq, Lq, d;
};

}  // namespace attn
