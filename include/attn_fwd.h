/*
 * attn_fwd.h -- C ABI of the GB300 (sm_103a) fused attention forward library.
 *
 * What the library computes, per batch b, query head h, kv head
 * hk = h / (Hq / Hkv) and query row i:
 *
 *   s_ij = scale * q_i . k_j                      (Composable Kernel
 *          fmha_fwd_pagedkv_kernel.hpp, header comment: S = Q K^T, S' = S*scale)
 *   s_ij <- softcap * tanh(s_ij / softcap)        if softcap > 0 (Composable Kernel
 *          fmha_fwd_pagedkv_kernel.hpp, FmhaFwdLogitsSoftCapKargs; tanh form)
 *   keys kept: j < Lk, and if causal  j <= i + (Lk - Lq)  (bottom-right
 *          alignment, the Composable Kernel mask default)
 *   z_i   = sum_kept exp(s_ij) [+ exp(sink[h])]   (Composable Kernel operator():
 *          one sink logit per query head; it adds to the denominator only)
 *   LSE_i = ln z_i,  O_i = sum_kept exp(s_ij - LSE_i) v_j   (P = softmax(S), O = P V)
 *   rows with nothing kept: O_i = 0, LSE_i = -inf, or LSE_i = sink[h] with a sink
 *          (FlashAttention-3 hopper/epilogue_fwd.hpp, CollectiveEpilogueFwd::store_zero)
 *
 * computed tile by tile with an online softmax (DefTruth
 * flash_attn_mma_share_kv_F32F16F16F32.cu, rescale by exp(m_old - m_new)), so
 * S and P never reach global memory.  Accumulation is fp32; O is written in
 * the input type; LSE is fp32, natural log.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *    never allocates or frees device memory; split-KV scratch is passed in.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and runs asynchronously.  A returned ATTN_OK means the launch was
 *    enqueued, not that it finished.
 *  - Arguments are validated before anything is launched; an invalid call
 *    launches nothing and returns ATTN_ERR_INVALID or ATTN_ERR_UNSUPPORTED.
 *  - No entry point throws, aborts or prints (unless ATTN_LOG=1 is set in the
 *    environment, which logs each launch to stderr).
 *  - Every wait inside a kernel is bounded.  A kernel that gives up records a
 *    bit in a device error word and returns; attn_device_error() reports it
 *    as ATTN_ERR_TIMEOUT after the caller has synchronised.
 *  - Element strides: the innermost (head-dim) stride is always 1; row, head
 *    and batch strides are in elements and must be multiples of 8 (16 bytes);
 *    base pointers must be 16-byte aligned.
 *  - Supported: d in {64, 128}; fp16 or bf16 Q/K/V/O; Hq % Hkv == 0.
 */
#ifndef ATTN_FWD_H
#define ATTN_FWD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID = 1,     /* bad pointer, size, stride or alignment */
  ATTN_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. d = 96) */
  ATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
  ATTN_ERR_TIMEOUT = 4      /* a kernel gave up on a bounded wait */
} attn_status;

/* ATTN_E4M3: OCP FP8 e4m3 ("fn": no infinities, max 448) for Q, K, V and O,
 * attn_fwd and attn_fwd_varlen with d = 128 only (FP8 static quantisation,
 * see scale_p / scale_o). */
typedef enum { ATTN_F16 = 0, ATTN_BF16 = 1, ATTN_E4M3 = 2 } attn_dtype;

/* Element strides of a 4-D [batch][head][row][d] (or packed [row][head][d])
 * tensor.  d-stride is 1. */
typedef struct {
  int64_t batch;
  int64_t head;
  int64_t row;
} attn_strides;

/*
 * Options.  A zero-initialised struct is plain softmax attention with the
 * default scale.  Masks (Composable Kernel mask from window_size_left /
 * window_size_right, generic attention mask) are bottom-right aligned: query
 * row i of a sequence with Lq queries and Lk keys sits on key diagonal
 * i + Lk - Lq.  Causal keeps keys j <= i + Lk - Lq.  A window keeps
 * i + Lk - Lq - window_left <= j <= i + Lk - Lq + window_right, a negative
 * bound meaning unbounded on that side; with causal also set both apply.
 * A row that keeps no key (and has no sink) gives O = 0, LSE = -inf.
 */
typedef struct {
  float scale;       /* softmax scale; <= 0 selects 1/sqrt(d) (DefTruth FA2 kernel prologue) */
  int causal;        /* nonzero: bottom-right aligned causal mask */
  float softcap;     /* > 0: s <- softcap * tanh(s / softcap); <= 0: off */
  const float* sink; /* device fp32 [Hq] sink logits (natural-log units), or NULL */
  int use_window;    /* nonzero: apply window_left / window_right */
  int window_left;   /* keys kept left of the diagonal (< 0: all) */
  int window_right;  /* keys kept right of the diagonal (< 0: all) */
  int top_left;      /* nonzero: row i's diagonal is key i (CK MASK_FROM_TOP_LEFT) for the
                        causal, window and ALiBi terms, instead of key i + Lk - Lq */
  /* ALiBi (CK position encoding): device fp32 slopes, the slope of (batch b,
   * query head h) at alibi_slopes[b * alibi_stride + h] (alibi_stride 0: one
   * [Hq] vector for every batch, else >= Hq).  Adds -slope * |diag(i) - j| to
   * the scaled score (natural-log units).  NULL: off. */
  const float* alibi_slopes;
  int alibi_stride;
  /* Elementwise bias (CK bias kargs), attn_fwd only: device, the input dtype,
   * element (b, h, i, j) at bias + b*batch + h*head + i*row + j (strides in
   * elements, multiples of 8, 0 broadcasts; 16-byte aligned base), added to
   * the scaled score (natural-log units).  NULL: off. */
  const void* bias;
  attn_strides bias_strides;
  /* FP8 static quantisation (CK FmhaFwdFp8StaticQuantKargs), ATTN_E4M3 only:
   * O = saturate_e4m3(scale_o * scale_p * softmax(S) V), each <= 0 meaning 1.
   * The caller folds the Q and K dequantisation factors into scale and V's
   * into scale_o.  P is kept in fp16 on chip (its storage type is not fixed
   * by the pages), so scale_p changes no rounding.  No soft-cap, ALiBi or
   * bias with ATTN_E4M3. */
  float scale_p;
  float scale_o;
} attn_opts;
/* Combinations not built: soft-cap with ALiBi or bias (the pages do not fix
 * the order), ALiBi with bias, bias outside attn_fwd: ATTN_ERR_UNSUPPORTED. */

/*
 * attn_fwd -- dense batch mode.
 *   q [B][Hq][Lq][d], k/v [B][Hkv][Lk][d], o [B][Hq][Lq][d] with the given
 *   strides (the default contiguous layout is batch = H*L*d, head = L*d,
 *   row = d); lse: fp32 [B][Hq][Lq] contiguous, or NULL to skip it.
 *   B, Lq, Lk >= 0 (zero-sized problems are a no-op; Lk = 0 gives empty rows).
 */
attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int Hq, int Hkv, int Lq, int Lk, int d, attn_dtype dtype, attn_strides sq,
                     attn_strides sk, attn_strides sv, attn_strides so, const attn_opts* opts,
                     void* stream);

/*
 * attn_fwd_varlen -- group mode (Composable Kernel operator(), group mode:
 * sequence b owns packed rows cu_seqlens[b] .. cu_seqlens[b+1]-1).
 *   q [total_q][Hq][d], k/v [total_k][Hkv][d], o [total_q][Hq][d]; only the
 *   head and row fields of the strides are used.
 *   cu_seqlens_q/k: device int32 [B+1], non-decreasing, cu[0] = 0,
 *   cu[B] = total.  max_seqlen_q >= every query length (it sizes the grid;
 *   tiles past a sequence's end exit at once).
 *   lse: fp32 [Hq][total_q] contiguous, or NULL.
 */
attn_status attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int B,
                            int total_q, int total_k, int max_seqlen_q, int Hq, int Hkv, int d,
                            attn_dtype dtype, attn_strides sq, attn_strides sk, attn_strides sv,
                            attn_strides so, const attn_opts* opts, void* stream);

/*
 * attn_fwd_paged -- paged KV cache with split-KV (Composable Kernel
 * operator(), page block navigator; FlashAttention-3 epilogue num_splits).
 *   q [B][Lq][Hq][d] contiguous; k_pool/v_pool [num_pages][page_size][Hkv][d]
 *   contiguous; block_table device int32 [B][max_pages_per_seq]: logical page
 *   p of sequence b lives in physical page block_table[b][p]; seqlens_k
 *   device int32 [B] (0 <= L_b <= max_pages_per_seq * page_size); entries past
 *   ceil(L_b / page_size) are not read.  Every entry read must lie in
 *   [0, num_pages): the kernel checks it and treats a bad entry as an error
 *   (device error word bit, that page's keys skipped).
 *   o [B][Lq][Hq][d] contiguous (input dtype); lse fp32 [B][Hq][Lq] or NULL.
 *   Causal masking, if set, is bottom-right within each sequence.
 *   page_size one of 16, 32, 64, 128, 256.
 *   Lq * (Hq / Hkv) <= 16 (decode, short chunks) runs the split-KV decode
 *   kernel described below.  Longer chunks (chunked prefill: the chunk's
 *   own keys already written to the cache, L_b counting them) run the
 *   prefill kernel with its K/V tiles gathered page by page; there
 *   num_splits, o_partial and lse_partial are ignored and nothing else
 *   changes.
 *   num_splits: 0 = choose automatically (attn_paged_auto_splits), else
 *   1..64.  Split s of sequence b covers logical pages
 *   [f_b + s*c, min(f_b + (s+1)*c, e_b)), c = ceil(W / num_splits); a split
 *   with no page is empty (O = 0, LSE = -inf).  Without a window f_b = 0,
 *   e_b = ceil(L_b/page_size) and W = max_pages_per_seq.  With a window the
 *   pages are those holding a key some query row keeps: f_b = floor(k_lo /
 *   page_size), e_b = ceil(k_hi / page_size) for the kept key range
 *   [k_lo, k_hi) of the sequence, and W = attn_paged_window_pages().
 *   When num_splits > 1, o_partial (fp32 [num_splits][B][Hq][Lq][d]) and
 *   lse_partial (fp32 [num_splits][B][Hq][Lq]) are caller-owned scratch of
 *   attn_paged_workspace_bytes() bytes in total, and attn_splitkv_combine is
 *   enqueued automatically; when it is 1 they may be NULL.
 */
attn_status attn_fwd_paged(const void* q, const void* k_pool, const void* v_pool,
                           const int32_t* block_table, const int32_t* seqlens_k, void* o,
                           float* lse, int B, int Lq, int Hq, int Hkv, int d, attn_dtype dtype,
                           int page_size, int num_pages, int max_pages_per_seq, int num_splits,
                           float* o_partial, float* lse_partial, const attn_opts* opts,
                           void* stream);

/*
 * attn_fwd_paged_noalloc -- attn_fwd_paged without caller-provided scratch.
 * The pages have no counterpart of this entry point; it exists for callers
 * that cannot allocate device memory when they call: a plugin inside a host
 * engine that owns every allocation and gives plugins no allocator, a
 * serving loop that must not call cudaMalloc (it can synchronise the device
 * and take milliseconds), a runtime that reserved its memory budget up front.
 *   Same arguments and results as attn_fwd_paged, minus o_partial and
 *   lse_partial: the split scratch comes from a fixed array of
 *   ATTN_NOALLOC_SCRATCH_BYTES inside this library, reserved on each GPU
 *   that loads the library and held until the process exits.
 *   For decode (Lq * (Hq / Hkv) <= 16) an explicit num_splits whose scratch
 *   (attn_paged_workspace_bytes) would exceed that size is rejected with
 *   ATTN_ERR_INVALID, and num_splits = 0 picks the automatic count, lowered
 *   until it fits.  Longer chunks run the prefill kernel, which uses no
 *   scratch: there num_splits is ignored, as in attn_fwd_paged.  The call allocates and
 *   frees no device memory.  The first call on each device looks up the
 *   array's address with that device current; make it before any stream
 *   capture.  All calls on a device share the array: calls whose kernels
 *   overlap on the GPU (unordered streams) race on it; calls ordered on one
 *   stream are safe.  Nothing in the array needs to start at zero.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
attn_status attn_fwd_paged_noalloc(const void* q, const void* k_pool, const void* v_pool,
                                   const int32_t* block_table, const int32_t* seqlens_k, void* o,
                                   float* lse, int B, int Lq, int Hq, int Hkv, int d,
                                   attn_dtype dtype, int page_size, int num_pages,
                                   int max_pages_per_seq, int num_splits, const attn_opts* opts,
                                   void* stream);

/*
 * attn_splitkv_combine -- LSE-weighted merge of split partials (derived from
 * the definition of LSE; FlashAttention-3 epilogue num_splits layout):
 *   M = max_s LSE_s,  w_s = exp(LSE_s - M),
 *   LSE = M + ln(sum_s w_s + exp(sink[h] - M)),  O = sum_s exp(LSE_s - LSE) O_s.
 *   Splits with LSE_s = -inf contribute nothing; if none contributes and
 *   there is no sink, O = 0 and LSE = -inf.
 *   o_partial fp32 [num_splits][B][Hq][Lq][d]; lse_partial fp32
 *   [num_splits][B][Hq][Lq]; sink fp32 [Hq] or NULL (added once, here);
 *   o [B][Lq][Hq][d] in dtype; lse fp32 [B][Hq][Lq] or NULL.
 */
attn_status attn_splitkv_combine(const float* o_partial, const float* lse_partial,
                                 int num_splits, int B, int Hq, int Lq, int d,
                                 const float* sink, void* o, attn_dtype dtype, float* lse,
                                 void* stream);

/* Bytes of split-KV scratch attn_fwd_paged needs (o_partial then lse_partial). */
size_t attn_paged_workspace_bytes(int B, int Lq, int Hq, int d, int num_splits);

/* The split count attn_fwd_paged uses for num_splits = 0 on the current device
 * (pass W of attn_paged_window_pages as max_pages_per_seq). */
int attn_paged_auto_splits(int B, int Hkv, int max_pages_per_seq);

/* W of the paged split layout: the most logical pages of one sequence that
 * hold a key some query row keeps.  max_pages_per_seq without a left window,
 * else min(max_pages_per_seq, ceil((Lq + window_left) / page_size) + 1)
 * (the kept keys of a sequence of length L are [max(0, L - Lq - window_left),
 * L), as every row's right bound reaches the last key or beyond).
 * opts may be NULL. */
int attn_paged_window_pages(int Lq, int page_size, int max_pages_per_seq, const attn_opts* opts);

/* The static work schedule attn_fwd runs for a dense problem with a causal
 * or window mask on a grid of `grid` CTAs (a load-balancing order of this
 * implementation; the pages fix none).  A work item is a query block of two
 * 128-row tiles of one batch and one head group: with g = Hq / Hkv a power
 * of two from 2 to 16 the g query heads of a kv head share every tile
 * (PackGQA, FlashAttention-3 epilogue: 128 / g queries of each of the g
 * heads), else a head group is one query head and a tile holds 128 queries.
 * With U = Hq / (heads per group) groups and Q = 256 / (heads per group)
 * queries per block, work item i is query block ceil(Lq / Q) - 1 - i / (B*U)
 * of batch (i % (B*U)) / U and head group i % U; CTA c runs items
 * item[off[c]] .. item[off[c+1] - 1] in that order.  The items are packed
 * longest processing time first (cost: the block's K/V tiles of 128 keys
 * plus 4), then moved and swapped off the most loaded CTA while that lowers
 * its load; each CTA's list runs lightest first.  attn_fwd launches
 * min(SM count, items) CTAs and uses this schedule exactly when this call
 * returns ATTN_OK for that grid.
 *   off: host int32 [grid + 1]; item: host int32 [B * U * ceil(Lq / Q)].
 *   Returns ATTN_ERR_UNSUPPORTED when the problem keeps the plain snake
 *   order (no mask, more than 1408 items or 160 CTAs, or no more items than
 *   CTAs), ATTN_ERR_INVALID for non-positive sizes, Hq % Hkv != 0 or NULL
 *   buffers.  Host only: needs no device.  opts as for attn_fwd (only the
 *   mask fields are read); may be NULL. */
attn_status attn_dense_schedule(int B, int Hq, int Hkv, int Lq, int Lk, const attn_opts* opts,
                                int grid, int32_t* off, int32_t* item);

/* Human-readable name of a status. */
const char* attn_status_string(attn_status status);

/* Trait string of the kernel the last call on this thread launched (empty if
 * none); for a split-KV attn_fwd_paged call, the decode kernel's and the
 * combine kernel's joined by '+'. */
const char* attn_last_kernel_name(void);

/* Reads and clears the current device's error word.  Returns ATTN_OK if no
 * kernel gave up, ATTN_ERR_TIMEOUT (with *bits set to the word) if one did,
 * ATTN_ERR_CUDA if the read failed.  Synchronises the device. */
attn_status attn_device_error(unsigned int* bits);

/* Launches a one-block kernel whose mbarrier wait can never complete, with the
 * given wait limit in nanoseconds; the kernel must give up, record the timeout
 * and return.  Used to test the timeout path without faulting the GPU. */
attn_status attn_selftest_timeout(uint64_t timeout_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_FWD_H */
