/*
 * attn_oracle.c -- plain fp64 CPU oracle for the fused attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this file; only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes (written out from the definitions on the pages, no tiling,
 * no online softmax, no fusion):
 *
 *   Composable Kernel, fmha_fwd_pagedkv_kernel.hpp, header comment:
 *     S   = Q . K^T                       (per head, fp64 here)
 *     S'  = S * scale
 *     S'' = S' + Bias                  (elementwise bias, [Lq][Lk] per head)
 *     P   = softmax(S'')   row by row
 *     O   = P . V
 *   DefTruth flash_attn_mma_share_kv_F32F16F16F32.cu, kernel prologue:
 *     default scale = 1/sqrt(d) (the caller passes the scale explicitly).
 *   Composable Kernel, FmhaFwdLogitsSoftCapKargs::init_logits_soft_cap:
 *     a cap c > 0 enables the logit soft-cap, c <= 0 disables it.  The form is
 *     not printed on the page; the reading used is  s <- c * tanh(s / c),
 *     applied to the scaled score, before masking and before the sink.
 *   Composable Kernel, operator() (sink_value) and the kHasSink trait:
 *     one sink logit per query head.  Reading used: the sink adds exp(sigma_h)
 *     to the softmax denominator and contributes no row of V; the returned LSE
 *     is the log of that full denominator.
 *   Composable Kernel, operator() (mask from the left/right window,
 *     MASK_FROM_TOP_LEFT vs. the default bottom-right alignment):
 *     causal bottom-right keeps key j for query i iff j <= i + (Lk - Lq).
 *     The window mask (window_size_left / window_size_right of the same
 *     kargs, same bottom-right alignment) keeps j iff
 *       i + (Lk - Lq) - left <= j <= i + (Lk - Lq) + right,
 *     a negative size meaning unbounded on that side; causal is right = 0.
 *     MASK_FROM_TOP_LEFT instead puts query i on key diagonal i (no Lk - Lq
 *     shift), for both the causal and the window bounds.
 *   Composable Kernel, operator() (position encoding, ALiBi): one slope per
 *     (batch, query head) (alibi_slope_ptr + i_batch * stride + i_nhead), the
 *     bias aligned like the mask (bottom-right unless MASK_FROM_TOP_LEFT).  The
 *     position term itself is not printed on the page; the reading used is the
 *     ALiBi definition  S'' = S' - slope * |diag(i) - j|,  diag(i) the key on
 *     query i's diagonal, added to the scaled (natural-log) score.
 *   Composable Kernel, FmhaFwdCommonBiasKargs (bias_ptr with row, head and
 *     batch strides): the elementwise bias is added to the scaled score.  With
 *     the soft-cap the order is not on the pages; those combinations are not
 *     evaluated (the library rejects them).
 *   Composable Kernel, FmhaFwdFp8StaticQuantKargs and the pipeline's element
 *     functions (P scaled by scale_p, the O accumulator scaled by scale_o and
 *     saturated to fp8): for fp8 inputs the oracle takes the e4m3 values
 *     exactly and returns O * o_scale with o_scale = scale_p * scale_o; the
 *     caller rounds to e4m3.  P itself is not quantized here: its on-chip
 *     storage type is not fixed by the page (reading stated with the kernel).
 *   FlashAttention-3 hopper/epilogue_fwd.hpp, CollectiveEpilogueFwd::store_zero:
 *     a row with no key to attend to gets O = 0 and LSE = -inf (with a sink:
 *     O = 0 and LSE = sigma).
 *   Composable Kernel, operator() (i_nhead / nhead_ratio_qk):
 *     GQA: query head h reads kv head h / (Hq / Hkv).
 *   Composable Kernel, operator() (page block navigator):
 *     paged KV: key j of sequence b is row (j mod page) of physical page
 *     block_table[b][j / page]; the last page may be partial.
 *   Composable Kernel, operator() (group mode, seqstart_q/k):
 *     varlen: sequence b owns rows cu[b] .. cu[b+1]-1 of the packed tensors.
 *   Split-KV (FlashAttention-3 epilogue, num_splits dimension of O/LSE):
 *     a split is the same softmax restricted to a key range; the merge of
 *     splits follows from the definition of LSE:
 *       LSE = log sum_s exp(LSE_s),  O = sum_s exp(LSE_s - LSE) O_s.
 *
 * The softmax of a row is evaluated with the row maximum subtracted before
 * exp (max-shift), in fp64; this changes no value beyond rounding.
 *
 * Layouts (all row-major, contiguous, fp64 unless stated):
 *   dense   q [B][Hq][Lq][d]   k,v [B][Hkv][Lk][d]   o [B][Hq][Lq][d]
 *           lse [B][Hq][Lq]
 *   varlen  q [total_q][Hq][d] k,v [total_k][Hkv][d] o [total_q][Hq][d]
 *           lse [Hq][total_q]  cu_q, cu_k int32 [B+1]
 *   paged   q [B][Lq][Hq][d]   pools [num_pages][page][Hkv][d]
 *           block_table int32 [B][max_pages]  seqlens_k int32 [B]
 *           o [B][Lq][Hq][d]   lse [B][Hq][Lq]
 *
 * Mutation switch: compiling with -DORACLE_MUTANT=n plants one deliberate
 * mistake (see the MUTANT() sites).  The pin tests build each mutant and check
 * that at least one pin fails; the normal build has ORACLE_MUTANT undefined.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif
#define MUTANT(n) (ORACLE_MUTANT == (n))

/* One query row against Lk keys of one head.
 *   q: [d], k: rows kbase + j*kstride (j < Lk), v likewise.
 *   diag: index (into these Lk keys) of the key on this row's diagonal; the
 *     causal, window and ALiBi terms are measured from it.
 *   bias_row: [Lk] additive bias of this row, or NULL.
 *   alibi: ALiBi slope of this row's (batch, head) (0: none).
 *   s_row/p_row: scratch of length Lk (also returned to the caller when asked).
 *   keep: scratch of length Lk.
 *   o: [d] output row; *lse: output.
 * Returns nothing; empty rows follow the store_zero convention. */
static void row_forward(const double* q, const double* k, const double* v, long kvstride,
                        int Lk, long diag, int d, double scale, int causal, int wl, int wr,
                        double softcap, const double* bias_row, double alibi,
                        int has_sink, double sink,
                        double* s_row, double* p_row, unsigned char* keep,
                        double* o, double* lse)
{
    /* S'_ij = scale * sum_t q_it k_jt */
    for (int j = 0; j < Lk; ++j) {
        const double* kj = k + (long)j * kvstride;
        double acc = 0.0;
        for (int t = 0; t < d; ++t) {
            if (MUTANT(1)) acc += q[t] * kj[(t + 1) % d]; /* wrong index */
            else acc += q[t] * kj[t];
        }
        double s = MUTANT(2) ? acc : acc * scale; /* dropped scale */
        if (softcap > 0.0) {
            if (MUTANT(3)) s = tanh(s / softcap);          /* dropped outer cap */
            else s = softcap * tanh(s / softcap);
        }
        if (bias_row) s += bias_row[j];
        if (alibi != 0.0) {
            const double dist = fabs((double)(diag - (long)j));
            s += MUTANT(10) ? alibi * dist : -alibi * dist; /* MUTANT 10: sign flipped */
        }
        s_row[j] = s;
        int kept = !causal || (long)j <= diag;
        if (wr >= 0 && (long)j > diag + wr) kept = 0;
        if (wl >= 0 && (long)j < diag - wl + (MUTANT(9) ? 1 : 0)) kept = 0; /* MUTANT 9: off by one */
        keep[j] = (unsigned char)kept;
    }

    int any = 0;
    double m = -INFINITY;
    for (int j = 0; j < Lk; ++j)
        if (keep[j]) { any = 1; if (s_row[j] > m) m = s_row[j]; }
    if (has_sink && sink > m) m = sink;

    if (!any && !has_sink) {
        /* store_zero: O = 0, LSE = -inf */
        for (int j = 0; j < Lk; ++j) p_row[j] = 0.0;
        for (int t = 0; t < d; ++t) o[t] = 0.0;
        *lse = -INFINITY;
        return;
    }

    double z = 0.0;
    for (int j = 0; j < Lk; ++j)
        if (keep[j]) z += exp(s_row[j] - m);
    if (has_sink && !MUTANT(5)) z += exp(sink - m);       /* MUTANT 5: sink dropped */
    double L = m + log(z);
    if (MUTANT(6)) L = log(z);                             /* dropped max term */
    *lse = L;

    for (int j = 0; j < Lk; ++j)
        p_row[j] = keep[j] ? exp(s_row[j] - L) : 0.0;

    for (int t = 0; t < d; ++t) o[t] = 0.0;
    for (int j = 0; j < Lk; ++j) {
        if (p_row[j] == 0.0) continue;
        const double* vj = v + (long)j * kvstride;
        for (int t = 0; t < d; ++t) {
            if (MUTANT(7)) o[t] += p_row[j] * vj[d - 1 - t]; /* transposed operand */
            else o[t] += p_row[j] * vj[t];
        }
    }
}

/* Key on query i's diagonal: bottom-right (i + Lk - Lq) unless top-left. */
static long row_diag(int i, int Lq, int Lk, int top_left)
{
    if (top_left || MUTANT(4)) return i;  /* MUTANT 4: top-left instead of bottom-right */
    return (long)i + (long)(Lk - Lq);
}

static int kv_head_of(int h, int Hq, int Hkv)
{
    int g = Hq / Hkv;
    if (MUTANT(8)) return h % Hkv; /* interleaved GQA grouping */
    return h / g;
}

/* Dense [B,H,L,d].  s_out/p_out: optional [B][Hq][Lq][Lk].
 * alibi: optional slopes [B][Hq]; bias: optional [B][Hq][Lq][Lk]. */
int oracle_attn_dense(const double* q, const double* k, const double* v,
                      double* o, double* lse,
                      int B, int Hq, int Hkv, int Lq, int Lk, int d,
                      double scale, int causal, int wl, int wr, double softcap,
                      const double* sink, double* s_out, double* p_out,
                      int top_left, const double* alibi, const double* bias, double o_scale)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || Lq < 0 || Lk < 0 || d <= 0) return 1;
    long nbh = (long)B * Hq;
#pragma omp parallel for schedule(dynamic)
    for (long bh = 0; bh < nbh; ++bh) {
        int b = (int)(bh / Hq), h = (int)(bh % Hq);
        int hk = kv_head_of(h, Hq, Hkv);
        const double* qh = q + ((long)b * Hq + h) * Lq * d;
        const double* kh = k + ((long)b * Hkv + hk) * Lk * d;
        const double* vh = v + ((long)b * Hkv + hk) * Lk * d;
        double* s_row = (double*)malloc(sizeof(double) * (Lk > 0 ? Lk : 1));
        double* p_row = (double*)malloc(sizeof(double) * (Lk > 0 ? Lk : 1));
        unsigned char* keep = (unsigned char*)malloc(Lk > 0 ? Lk : 1);
        for (int i = 0; i < Lq; ++i) {
            const double* brow = NULL;
            if (bias) {
                int bi = MUTANT(11) ? (i + 1) % Lq : i;  /* MUTANT 11: bias row shifted */
                brow = bias + (((long)b * Hq + h) * Lq + bi) * Lk;
            }
            row_forward(qh + (long)i * d, kh, vh, d, Lk, row_diag(i, Lq, Lk, top_left), d, scale,
                        causal, wl, wr, softcap, brow, alibi ? alibi[(long)b * Hq + h] : 0.0,
                        sink != NULL, sink ? sink[h] : 0.0, s_row, p_row, keep,
                        o + (((long)b * Hq + h) * Lq + i) * d,
                        lse + ((long)b * Hq + h) * Lq + i);
            if (o_scale != 1.0) {
                for (int t = 0; t < d; ++t) o[(((long)b * Hq + h) * Lq + i) * d + t] *= o_scale;
                if (MUTANT(12)) lse[((long)b * Hq + h) * Lq + i] *= o_scale; /* scale on LSE too */
            }
            if (s_out) memcpy(s_out + (((long)b * Hq + h) * Lq + i) * Lk, s_row, sizeof(double) * Lk);
            if (p_out) memcpy(p_out + (((long)b * Hq + h) * Lq + i) * Lk, p_row, sizeof(double) * Lk);
        }
        free(s_row); free(p_row); free(keep);
    }
    return 0;
}

/* Varlen (group mode): packed [total, H, d]; lse [Hq][total_q]. */
int oracle_attn_varlen(const double* q, const double* k, const double* v,
                       double* o, double* lse,
                       const int32_t* cu_q, const int32_t* cu_k,
                       int B, int Hq, int Hkv, int d,
                       double scale, int causal, int wl, int wr, double softcap,
                       const double* sink, int top_left, const double* alibi, double o_scale)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0) return 1;
    int total_q = cu_q[B];
    long nbh = (long)B * Hq;
#pragma omp parallel for schedule(dynamic)
    for (long bh = 0; bh < nbh; ++bh) {
        int b = (int)(bh / Hq), h = (int)(bh % Hq);
        int hk = kv_head_of(h, Hq, Hkv);
        int q0 = cu_q[b], Lq = cu_q[b + 1] - cu_q[b];
        int k0 = cu_k[b], Lk = cu_k[b + 1] - cu_k[b];
        double* s_row = (double*)malloc(sizeof(double) * (Lk > 0 ? Lk : 1));
        double* p_row = (double*)malloc(sizeof(double) * (Lk > 0 ? Lk : 1));
        unsigned char* keep = (unsigned char*)malloc(Lk > 0 ? Lk : 1);
        long kvstride = (long)Hkv * d;
        const double* kh = k + (long)k0 * kvstride + (long)hk * d;
        const double* vh = v + (long)k0 * kvstride + (long)hk * d;
        for (int i = 0; i < Lq; ++i) {
            long row = q0 + i;
            row_forward(q + (row * Hq + h) * d, kh, vh, kvstride, Lk, row_diag(i, Lq, Lk, top_left),
                        d, scale, causal, wl, wr, softcap, NULL,
                        alibi ? alibi[(long)b * Hq + h] : 0.0,
                        sink != NULL, sink ? sink[h] : 0.0, s_row, p_row, keep,
                        o + (row * Hq + h) * d, lse + (long)h * total_q + row);
            if (o_scale != 1.0 && !MUTANT(13))                   /* MUTANT 13: scale dropped */
                for (int t = 0; t < d; ++t) o[(row * Hq + h) * d + t] *= o_scale;
        }
        free(s_row); free(p_row); free(keep);
    }
    return 0;
}

/* Gather the logical K or V rows [0, L) of (b, hk) out of a paged pool into
 * dst [L][d] (page navigator: physical page = block_table[b][j / page]). */
static void gather_pages(const double* pool, const int32_t* bt_row, int page, int Hkv, int hk,
                         int d, int L, double* dst)
{
    for (int j = 0; j < L; ++j) {
        long pg = bt_row[j / page];
        int r = j % page;
        memcpy(dst + (long)j * d, pool + ((pg * page + r) * (long)Hkv + hk) * d, sizeof(double) * d);
    }
}

/* Paged KV: q [B][Lq][Hq][d]; o [B][Lq][Hq][d]; lse [B][Hq][Lq]. */
int oracle_attn_paged(const double* q, const double* k_pool, const double* v_pool,
                      const int32_t* block_table, const int32_t* seqlens_k,
                      double* o, double* lse,
                      int B, int Lq, int Hq, int Hkv, int d, int page, int max_pages,
                      double scale, int causal, int wl, int wr, double softcap,
                      const double* sink, int top_left, const double* alibi)
{
    if (B < 0 || Lq < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0 || page <= 0) return 1;
    long nbh = (long)B * Hq;
#pragma omp parallel for schedule(dynamic)
    for (long bh = 0; bh < nbh; ++bh) {
        int b = (int)(bh / Hq), h = (int)(bh % Hq);
        int hk = kv_head_of(h, Hq, Hkv);
        int Lk = seqlens_k[b];
        double* kg = (double*)malloc(sizeof(double) * ((long)(Lk > 0 ? Lk : 1) * d));
        double* vg = (double*)malloc(sizeof(double) * ((long)(Lk > 0 ? Lk : 1) * d));
        gather_pages(k_pool, block_table + (long)b * max_pages, page, Hkv, hk, d, Lk, kg);
        gather_pages(v_pool, block_table + (long)b * max_pages, page, Hkv, hk, d, Lk, vg);
        double* s_row = (double*)malloc(sizeof(double) * (Lk > 0 ? Lk : 1));
        double* p_row = (double*)malloc(sizeof(double) * (Lk > 0 ? Lk : 1));
        unsigned char* keep = (unsigned char*)malloc(Lk > 0 ? Lk : 1);
        for (int i = 0; i < Lq; ++i) {
            row_forward(q + (((long)b * Lq + i) * Hq + h) * d, kg, vg, d, Lk,
                        row_diag(i, Lq, Lk, top_left), d, scale, causal, wl, wr, softcap, NULL,
                        alibi ? alibi[(long)b * Hq + h] : 0.0,
                        sink != NULL, sink ? sink[h] : 0.0, s_row, p_row, keep,
                        o + (((long)b * Lq + i) * Hq + h) * d, lse + ((long)b * Hq + h) * Lq + i);
        }
        free(kg); free(vg); free(s_row); free(p_row); free(keep);
    }
    return 0;
}

/* Split-KV partials of the paged problem.  Split s of sequence b covers the
 * key pages [f + s*chunk_pages, min(f + (s+1)*chunk_pages, pages_b)), pages_b =
 * ceil(seqlens_k[b] / page); a split with no key page is empty (O = 0,
 * LSE = -inf).  No sink in a split (the merge adds it once).  f = 0 without a
 * left window; with one, f is the page of the first key any query row keeps,
 * max(0, L - Lq - wl) (every row's right bound is at or past the last key),
 * so the splits tile only the pages the window reaches. 
 * o_part [S][B][Hq][Lq][d], lse_part [S][B][Hq][Lq]. */
int oracle_attn_paged_partials(const double* q, const double* k_pool, const double* v_pool,
                               const int32_t* block_table, const int32_t* seqlens_k,
                               double* o_part, double* lse_part,
                               int B, int Lq, int Hq, int Hkv, int d, int page, int max_pages,
                               int num_splits, int chunk_pages,
                               double scale, int causal, int wl, int wr, double softcap,
                               int top_left, const double* alibi)
{
    if (B < 0 || Lq < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0 || page <= 0 ||
        num_splits <= 0 || chunk_pages <= 0) return 1;
    long nbh = (long)B * Hq;
    long rows = (long)B * Hq * Lq;
#pragma omp parallel for schedule(dynamic)
    for (long bh = 0; bh < nbh; ++bh) {
        int b = (int)(bh / Hq), h = (int)(bh % Hq);
        int hk = kv_head_of(h, Hq, Hkv);
        int Lk = seqlens_k[b];
        double* kg = (double*)malloc(sizeof(double) * ((long)(Lk > 0 ? Lk : 1) * d));
        double* vg = (double*)malloc(sizeof(double) * ((long)(Lk > 0 ? Lk : 1) * d));
        gather_pages(k_pool, block_table + (long)b * max_pages, page, Hkv, hk, d, Lk, kg);
        gather_pages(v_pool, block_table + (long)b * max_pages, page, Hkv, hk, d, Lk, vg);
        double* s_row = (double*)malloc(sizeof(double) * (Lk > 0 ? Lk : 1));
        double* p_row = (double*)malloc(sizeof(double) * (Lk > 0 ? Lk : 1));
        unsigned char* keep = (unsigned char*)malloc(Lk > 0 ? Lk : 1);
        long first = 0;
        /* first key any row keeps: the left bound of row 0 */
        if (wl >= 0 && row_diag(0, Lq, Lk, top_left) - wl > 0)
            first = (row_diag(0, Lq, Lk, top_left) - wl) / page;
        for (int s = 0; s < num_splits; ++s) {
            long j0 = (first + (long)s * chunk_pages) * page;
            long j1 = (first + (long)(s + 1) * chunk_pages) * page;
            if (j1 > Lk) j1 = Lk;
            for (int i = 0; i < Lq; ++i) {
                long ridx = ((long)b * Hq + h) * Lq + i;
                double* orow = o_part + ((long)s * rows + ridx) * d;
                double* lrow = lse_part + (long)s * rows + ridx;
                if (j0 >= j1) {
                    for (int t = 0; t < d; ++t) orow[t] = 0.0;
                    *lrow = -INFINITY;
                    continue;
                }
                /* Scores over the split's keys only: the diagonal is measured
                 * in the split's own key indices (absolute key = j0 + j). */
                int Lks = (int)(j1 - j0);
                row_forward(q + (((long)b * Lq + i) * Hq + h) * d, kg + j0 * d, vg + j0 * d, d,
                            Lks, row_diag(i, Lq, Lk, top_left) - j0, d, scale, causal, wl, wr,
                            softcap, NULL, alibi ? alibi[(long)b * Hq + h] : 0.0, 0, 0.0,
                            s_row, p_row, keep, orow, lrow);
            }
        }
        free(kg); free(vg); free(s_row); free(p_row); free(keep);
    }
    return 0;
}

/* LSE-weighted merge of split partials.
 *   o_part [S][rows][d], lse_part [S][rows]; sink: optional per-row logit.
 *   LSE = log( sum_s exp(LSE_s) + exp(sink) ),  O = sum_s exp(LSE_s - LSE) O_s.
 * All splits empty and no sink: O = 0, LSE = -inf. */
int oracle_combine(const double* o_part, const double* lse_part, int num_splits, long rows, int d,
                   const double* sink_rows, double* o, double* lse)
{
    if (num_splits <= 0 || rows < 0 || d <= 0) return 1;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) {
        double m = -INFINITY;
        for (int s = 0; s < num_splits; ++s) {
            double l = lse_part[(long)s * rows + r];
            if (l > m) m = l;
        }
        if (sink_rows && sink_rows[r] > m) m = sink_rows[r];
        double* orow = o + r * d;
        for (int t = 0; t < d; ++t) orow[t] = 0.0;
        if (m == -INFINITY) { lse[r] = -INFINITY; continue; }
        double z = 0.0;
        for (int s = 0; s < num_splits; ++s) {
            double l = lse_part[(long)s * rows + r];
            if (l == -INFINITY) continue;
            z += exp(l - m);
        }
        if (sink_rows) z += exp(sink_rows[r] - m);
        double L = m + log(z);
        lse[r] = L;
        for (int s = 0; s < num_splits; ++s) {
            double l = lse_part[(long)s * rows + r];
            if (l == -INFINITY) continue;
            double w = exp(l - L);
            const double* os = o_part + ((long)s * rows + r) * d;
            for (int t = 0; t < d; ++t) orow[t] += w * os[t];
        }
    }
    return 0;
}

int oracle_mutant_id(void) { return ORACLE_MUTANT; }
