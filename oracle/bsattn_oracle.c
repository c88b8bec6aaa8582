/*
 * bsattn_oracle.c -- plain fp64 CPU oracle for block-sparse attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only the tests, the package smoke check and the CPU
 * baseline leg of the benchmark load it.  It shares no code with the CUDA path.
 *
 * What it computes is the plain definition the block-sparse kernels reach up to
 * rounding: softmax(Q K^T / sqrt(d)) V restricted, row by row, to the keys the
 * block mask (or the decode block list) makes visible.  Sources:
 *
 *  - TileLang block-sparse Flash-Attention guide, section 5 (the reference
 *    check): expand the block mask to token level (kron with a BLOCKxBLOCK block
 *    of ones), crop to the sequence, AND with the causal lower triangle, then
 *    evaluate an ordinary masked softmax attention.
 *  - same guide, sections 6.1-6.2 (GQA varlen sparse decode): query head h uses
 *    kv head h / (Hq/Hkv); block t of the list covers tokens [t*BLOCK,
 *    (t+1)*BLOCK) clipped to cache_seqlens[b]; -1 slots are skipped.
 *  - same guide, section 7 (paged KV): logical block -> (page, tile) -> physical
 *    page through block_table.
 *  - TileLang FlashAttention guide, BHSD variant: with seq_kv > seq_q the causal
 *    rule is aligned bottom-right, key j visible to query i iff
 *    j <= i + (seq_kv - seq_q).
 *
 * Conventions the pages leave open, fixed here:
 *  - a query row with no visible key outputs exactly 0;
 *  - block indices are a set: order and repeats do not matter; slots < 0 are
 *    empty; blocks at or past the sequence end contribute no tokens.
 *
 * Every computation is fp64: inputs stored as fp16 / bf16 are widened exactly.
 * Parallelism: OpenMP over independent output rows only; each row is computed
 * by one thread in a fixed order, so results do not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1, ORACLE_F64 = 2 };

/* ---- exact widening of the storage formats ---------------------------------- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -24);               /* subnormal: f * 2^-14 * 2^-10 */
    else if (e == 31)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + f), e - 25);   /* (1 + f/1024) * 2^(e-15) */
    return sign ? -mag : mag;
}

/* bfloat16 is the upper half of an IEEE binary32. */
double oracle_bf16_to_f64(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static double load(const void *base, int64_t i, int dtype)
{
    if (dtype == ORACLE_F64)
        return ((const double *)base)[i];
    uint16_t raw = ((const uint16_t *)base)[i];
    return dtype == ORACLE_F16 ? oracle_f16_to_f64(raw) : oracle_bf16_to_f64(raw);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- one softmax-attention row over an explicit list of visible keys -------- */

/*
 * out[0..d) = sum_j softmax_j(s) v_j over the keys in `keys` (n of them), where
 * s_j = (q . k_j) / sqrt(d).  k_row(j) / v_row(j) are element offsets of the key
 * and value rows.  n == 0 gives exactly 0.  `s` is scratch of length >= n.
 */
static void attend_row(const void *q, int64_t q_off, const void *k, const void *v,
                       const int64_t *k_off, const int64_t *v_off, int64_t n, int d,
                       int dtype, double *s, double *out)
{
    for (int c = 0; c < d; ++c)
        out[c] = 0.0;
    if (n == 0)
        return;
    const double inv_sqrt_d = 1.0 / sqrt((double)d);
    double m = -INFINITY;
    for (int64_t t = 0; t < n; ++t) {
        double dot = 0.0;
        for (int c = 0; c < d; ++c)
            dot += load(q, q_off + c, dtype) * load(k, k_off[t] + c, dtype);
        s[t] = dot * inv_sqrt_d;
        if (s[t] > m)
            m = s[t];
    }
    double l = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        double w = exp(s[t] - m);
        l += w;
        for (int c = 0; c < d; ++c)
            out[c] += w * load(v, v_off[t] + c, dtype);
    }
    for (int c = 0; c < d; ++c)
        out[c] /= l;
}

/* ---- prefill ------------------------------------------------------------------ */

/*
 * Rows of one (batch, head): q [Sq, d], k and v [Sk, d] (row-major), mask
 * [ceil(Sq/block), ceil(Sk/block)] (nonzero = visit).  Query i sees key j iff
 *   mask[i / block][j / block] != 0  and  j < Sk  and
 *   (not causal  or  j <= i + (Sk - Sq)).
 * rows[0..nrows) are query positions in [0, Sq); out is [nrows, d].
 * Returns 0, or -1 on a bad argument / allocation failure.
 */
int oracle_prefill_rows(const void *q, const void *k, const void *v, int dtype,
                        const uint8_t *mask, int causal, int Sq, int Sk, int d, int block,
                        const int32_t *rows, int nrows, double *out)
{
    if (Sq < 0 || Sk < 0 || d <= 0 || block <= 0 || nrows < 0)
        return -1;
    const int nk = (Sk + block - 1) / block;
    int bad = 0;
#pragma omp parallel
    {
        int64_t *koff = (int64_t *)malloc(sizeof(int64_t) * (size_t)(Sk > 0 ? Sk : 1));
        double *s = (double *)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
        if (!koff || !s) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int r = 0; r < nrows; ++r) {
            int i = rows[r];
            if (!koff || !s || i < 0 || i >= Sq) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            const uint8_t *mrow = mask + (int64_t)(i / block) * nk;
            int64_t n = 0;
            for (int j = 0; j < Sk; ++j) {
                if (!mrow[j / block])
                    continue;
                if (causal && (int64_t)j > (int64_t)i + (Sk - Sq))
                    continue;
                koff[n++] = (int64_t)j * d;
            }
            attend_row(q, (int64_t)i * d, k, v, koff, koff, n, d, dtype, s,
                       out + (int64_t)r * d);
        }
        free(koff);
        free(s);
    }
    return bad ? -1 : 0;
}

/*
 * Whole prefill: q [B,H,Sq,d], k/v [B,H,Sk,d], mask [B,H,nq,nk], out [B,H,Sq,d].
 */
int oracle_prefill(const void *q, const void *k, const void *v, int dtype, const uint8_t *mask,
                   int causal, int B, int H, int Sq, int Sk, int d, int block, double *out)
{
    if (B < 0 || H < 0 || Sq < 0 || Sk < 0 || d <= 0 || block <= 0)
        return -1;
    const int nq = (Sq + block - 1) / block, nk = (Sk + block - 1) / block;
    const size_t esz = dtype == ORACLE_F64 ? 8 : 2;
    int32_t *rows = (int32_t *)malloc(sizeof(int32_t) * (size_t)(Sq > 0 ? Sq : 1));
    if (!rows)
        return -1;
    for (int i = 0; i < Sq; ++i)
        rows[i] = i;
    int rc = 0;
    for (int b = 0; b < B && rc == 0; ++b)
        for (int h = 0; h < H && rc == 0; ++h) {
            int64_t bh = (int64_t)b * H + h;
            rc = oracle_prefill_rows((const char *)q + bh * Sq * d * esz,
                                     (const char *)k + bh * Sk * d * esz,
                                     (const char *)v + bh * Sk * d * esz, dtype,
                                     mask + bh * nq * nk, causal, Sq, Sk, d, block, rows, Sq,
                                     out + bh * Sq * d);
        }
    free(rows);
    return rc;
}

/* ---- GQA varlen sparse decode ---------------------------------------------------- */

/*
 * Token set of sequence b for kv head g: the union over the slots t of
 * block_indices[b, g, :] with t >= 0 of tokens [t*block, (t+1)*block), clipped
 * to [0, seqlen).  `sel` (length >= seqlen) is scratch; returns the count and
 * fills tok[] with the selected token positions in ascending order.
 */
static int64_t decode_token_set(const int32_t *slots, int max_sel, int seqlen, int block,
                                uint8_t *sel, int64_t *tok)
{
    memset(sel, 0, (size_t)seqlen);
    for (int t = 0; t < max_sel; ++t) {
        int blk = slots[t];
        if (blk < 0)
            continue;
        for (int64_t p = (int64_t)blk * block; p < (int64_t)blk * block + block && p < seqlen; ++p)
            sel[p] = 1;
    }
    int64_t n = 0;
    for (int p = 0; p < seqlen; ++p)
        if (sel[p])
            tok[n++] = p;
    return n;
}

/*
 * q [B,Hq,d]; k, v [B,Smax,Hkv,d] (BSHD); cache_seqlens [B] (each in [0, Smax]);
 * block_indices [B,Hkv,max_sel]; out [B,Hq,d].  Query head h reads kv head
 * h / (Hq / Hkv).
 */
int oracle_decode(const void *q, const void *k, const void *v, int dtype,
                  const int32_t *cache_seqlens, const int32_t *block_indices, int B, int Hq,
                  int Hkv, int Smax, int d, int max_sel, int block, double *out)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || Smax < 0 || d <= 0 || max_sel < 0 ||
        block <= 0)
        return -1;
    for (int b = 0; b < B; ++b)
        if (cache_seqlens[b] < 0 || cache_seqlens[b] > Smax)
            return -1;
    const int group = Hq / Hkv;
    int bad = 0;
#pragma omp parallel
    {
        uint8_t *sel = (uint8_t *)malloc((size_t)(Smax > 0 ? Smax : 1));
        int64_t *tok = (int64_t *)malloc(sizeof(int64_t) * (size_t)(Smax > 0 ? Smax : 1));
        double *s = (double *)malloc(sizeof(double) * (size_t)(Smax > 0 ? Smax : 1));
        if (!sel || !tok || !s) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int bh = 0; bh < B * Hq; ++bh) {
            if (!sel || !tok || !s)
                continue;
            int b = bh / Hq, h = bh % Hq, g = h / group;
            const int32_t *slots = block_indices + ((int64_t)b * Hkv + g) * max_sel;
            int64_t n = decode_token_set(slots, max_sel, cache_seqlens[b], block, sel, tok);
            for (int64_t t = 0; t < n; ++t)
                tok[t] = (((int64_t)b * Smax + tok[t]) * Hkv + g) * d;
            attend_row(q, (int64_t)bh * d, k, v, tok, tok, n, d, dtype, s,
                       out + (int64_t)bh * d);
        }
        free(sel);
        free(tok);
        free(s);
    }
    return bad ? -1 : 0;
}

/*
 * Paged variant: k, v [num_pages, page_size, Hkv, d]; block_table
 * [B, max_pages_per_seq] maps logical page p of sequence b to a physical page.
 * Logical token position P lives at page block_table[b][P / page_size], row
 * P % page_size.  Everything else is as in oracle_decode.
 */
int oracle_decode_paged(const void *q, const void *k, const void *v, int dtype,
                        const int32_t *cache_seqlens, const int32_t *block_indices,
                        const int32_t *block_table, int B, int Hq, int Hkv, int num_pages,
                        int page_size, int max_pages_per_seq, int d, int max_sel, int block,
                        double *out)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || num_pages <= 0 || page_size <= 0 ||
        max_pages_per_seq <= 0 || d <= 0 || max_sel < 0 || block <= 0)
        return -1;
    const int64_t cap = (int64_t)page_size * max_pages_per_seq;
    for (int b = 0; b < B; ++b)
        if (cache_seqlens[b] < 0 || cache_seqlens[b] > cap)
            return -1;
    const int group = Hq / Hkv;
    int bad = 0;
#pragma omp parallel
    {
        uint8_t *sel = (uint8_t *)malloc((size_t)cap);
        int64_t *tok = (int64_t *)malloc(sizeof(int64_t) * (size_t)cap);
        double *s = (double *)malloc(sizeof(double) * (size_t)cap);
        if (!sel || !tok || !s) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int bh = 0; bh < B * Hq; ++bh) {
            if (!sel || !tok || !s)
                continue;
            int b = bh / Hq, h = bh % Hq, g = h / group;
            const int32_t *slots = block_indices + ((int64_t)b * Hkv + g) * max_sel;
            int64_t n = decode_token_set(slots, max_sel, cache_seqlens[b], block, sel, tok);
            for (int64_t t = 0; t < n; ++t) {
                int64_t P = tok[t];
                int64_t page = block_table[(int64_t)b * max_pages_per_seq + P / page_size];
                if (page < 0 || page >= num_pages) {
#pragma omp atomic write
                    bad = 1;
                    page = 0;
                }
                tok[t] = ((page * page_size + P % page_size) * Hkv + g) * d;
            }
            attend_row(q, (int64_t)bh * d, k, v, tok, tok, n, d, dtype, s,
                       out + (int64_t)bh * d);
        }
        free(sel);
        free(tok);
        free(s);
    }
    return bad ? -1 : 0;
}
