/*
 * dsa_oracle.c -- plain, slow, single-threaded CPU oracle for the DSA indexer
 * decode path (paged MQA logits, fused coarse histogram, histogram-driven
 * top-k, and the two-level candidate path).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this file: only the test suite, the smoke check and the bench's CPU
 * baseline leg load it.  It shares no code, header, table or constant with
 * the CUDA library; every number it needs it derives here from the formats'
 * definitions.
 *
 * Sources (the three pull-request pages this library follows):
 *   [DG94]  DeepGEMM PR #94, "[SM100] Paged MQA logits: fused coarse score
 *           histogram for LiteTopK decode" -- sections "Motivation", "What this
 *           adds", "Producer cost", commit 2d3b1c1 and the cross-referenced
 *           SGLang commit 7e252c5 (select.cuh / coarse_bins.cuh).
 *   [SG38944] SGLang PR #38944, "[DSV4.1] Enable the two-level candidate
 *           indexer on DeepGEMM's paged sparse MQA logits" -- squashed commit
 *           texts (amax8_varlen, sort_candidate_blocks, candidate_row_lens,
 *           row pairing) and the PR body ("What this enables", "Tests").
 *   [VL52696] vLLM PR #52696, "[Performance][MLA] Use FP16 logits for sparse
 *           indexer" -- "Summary" and "Why" sections.
 *
 * Readings where the pages leave a step open (each one is also listed in the
 * design notes of the repository):
 *   R1  Row r = b*next_n + j of a request with context length C sees
 *       n_r = C - (next_n - 1 - j) keys ([DG94] "Producer cost": token j of a
 *       request sees L + j keys, so C = L + next_n - 1).
 *   R2  ReLU is applied to q.k * kscale, as the logits formula is written.
 *   R3  Unit bins use floor(|x|) for both signs: a negative unit bin holds the
 *       magnitudes [n, n+1), i.e. x in (-n-1, -n] ([DG94] "What this adds":
 *       16 <= |x| < 223 unit-width bins, |x| >= 223 saturating).
 *   R4  +0 falls in bin 511 and -0 in bin 512 (the sign bit decides).
 *   R5  FP16 rounding is round-to-nearest-even and happens before the
 *       low 6 bits of the half are dropped.
 *   R6  Top-k orders by value, ties go to the lower column, NaN is never
 *       selected, short rows are padded with -1.
 *   R7  amax8: the block maximum follows the same value order as the top-k
 *       (-0 below +0), NaN is ignored inside a block, an all-NaN block stays
 *       NaN; the newest block (index ceil(n/8)-1) is +inf.
 *   R8  Block-table padding (ids and physical blocks) is INT32_MAX; the live
 *       length of a sparse row counts the live tokens of the chosen blocks.
 *   R9  Sparse positions that are padding or past the row's live length are
 *       -inf in the output.
 *   R14 The BF16 sibling of the FP16 select (the next step the pages point
 *       to, [VL52696] "Why" for FP16): bfloat16 rounding is round-to-nearest-
 *       even, NaN never selected, the same order and tie rule as FP16.
 *   R16 MXFP4 index keys: 128 E2M1 codes two per byte (even dimension in
 *       the low nibble) plus 4 UE8M0 block exponents per token (68 bytes).
 *   R15 Row pairing of the sparse pass: rows 2m and 2m+1 of a request form
 *       one unit (an odd last row is alone) whose pass walks the ascending
 *       union of the two tables; each row's scores keep its own positions.
 *   (R10-R13 concern the CUDA path's contracts, not this file's arithmetic.)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define O_INT32_MAX 2147483647

/* ------------------------------------------------------------------------ */
/* O1: FP8 E4M3 decode, from the format definition (1 sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits, subnormals when the exponent field is 0,
 * no infinities, S.1111.111 is NaN, largest finite value 448).              */
double o_e4m3_to_double(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double mag;
    if (e == 15 && m == 7) {
        return NAN;
    }
    if (e == 0) {
        mag = ldexp((double)m / 8.0, 1 - 7);          /* subnormal */
    } else {
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);    /* normal    */
    }
    return sign ? -mag : mag;
}

void o_e4m3_table(double *out256)
{
    for (int c = 0; c < 256; ++c) out256[c] = o_e4m3_to_double((uint8_t)c);
}

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary32 -> binary16, round to nearest, ties to even, written from
 * the definition with exact double arithmetic.  Returns the 16-bit pattern.  */
static double o_round_half_even(double q)
{
    double fl = floor(q);
    double diff = q - fl;            /* exact: q has at most 53 bits        */
    if (diff > 0.5) return fl + 1.0;
    if (diff < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

uint16_t o_fp16_rn_bits(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    if (isnan(x)) return (uint16_t)(sign | 0x7E00u);
    double a = fabs((double)x);
    if (isinf(x)) return (uint16_t)(sign | 0x7C00u);
    /* Largest finite half is 65504 = (2 - 2^-10) * 2^15; the midpoint to the
     * next (unrepresentable) step 65536 is 65520, which ties to the even
     * neighbour 65536, i.e. overflows.                                       */
    if (a >= 65520.0) return (uint16_t)(sign | 0x7C00u);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: quantum 2^-24 */
        double q = o_round_half_even(a * ldexp(1.0, 24));
        return (uint16_t)(sign | (uint16_t)q);  /* q == 1024 is the smallest normal */
    }
    int E;
    (void)frexp(a, &E);          /* a = f * 2^E, f in [0.5, 1) */
    int e = E - 1;               /* a in [2^e, 2^(e+1))        */
    double q = o_round_half_even(a * ldexp(1.0, 10 - e));   /* in [1024, 2048] */
    if (q >= 2048.0) {
        q = 1024.0;
        e += 1;
    }
    if (e + 15 >= 31) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)(((e + 15) << 10) | ((int)q - 1024)));
}

/* bfloat16 (1 sign, 8 exponent bits with bias 127, 7 mantissa bits; the top
 * half of a binary32), round-to-nearest-even from the value, as the FP16
 * conversion above (the BF16 sibling of the FP16 select, NEXT-3).          */
uint16_t o_bf16_rn_bits(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    if (isnan(x)) return (uint16_t)(sign | 0x7FC0u);
    if (isinf(x)) return (uint16_t)(sign | 0x7F80u);
    double a = fabs((double)x);
    if (a < ldexp(1.0, -126)) {
        /* subnormal range: quantum 2^-133 */
        double q = o_round_half_even(a * ldexp(1.0, 133));
        return (uint16_t)(sign | (uint16_t)q);  /* q == 128 is the smallest normal */
    }
    int E;
    (void)frexp(a, &E);          /* a = f * 2^E, f in [0.5, 1) */
    int e = E - 1;               /* a in [2^e, 2^(e+1))        */
    double q = o_round_half_even(a * ldexp(1.0, 7 - e));    /* in [128, 256] */
    if (q >= 256.0) {
        q = 128.0;
        e += 1;
    }
    if (e + 127 >= 255) return (uint16_t)(sign | 0x7F80u);
    return (uint16_t)(sign | (uint16_t)(((e + 127) << 7) | ((int)q - 128)));
}

/* bfloat16 pattern -> double, from the definition. */
double o_bf16_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 255;
    int m = h & 127;
    double mag;
    if (e == 255) mag = (m == 0) ? INFINITY : NAN;
    else if (e == 0) mag = ldexp((double)m, -133);
    else mag = ldexp(1.0 + (double)m / 128.0, e - 127);
    return sign ? -mag : mag;
}

/* binary16 pattern -> double, from the definition (used by the FP16 select). */
double o_fp16_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double mag;
    if (e == 31) mag = (m == 0) ? INFINITY : NAN;
    else if (e == 0) mag = ldexp((double)m, -24);
    else mag = ldexp(1.0 + (double)m / 1024.0, e - 15);
    return sign ? -mag : mag;
}

/* ------------------------------------------------------------------------ */
/* O3: the 1024-bin coarse score bin ([DG94] "What this adds").  Bins descend,
 * so bin 0 holds the largest scores.  Magnitude code m:
 *   |x| >= 223 (incl. inf)  -> 511                       (saturating end bin)
 *   16 <= |x| < 223         -> 304 + floor(|x|) - 16      (unit-width bins)
 *   |x| < 16                -> FP16-RN(|x|) >> 6          (exponent + 4 mantissa bits)
 * and bin = 511 - m for a clear sign bit, 512 + m for a set one.
 * Returns -1 for NaN (never counted).                                       */
int32_t o_coarse_bin(float x)
{
    if (isnan(x)) return -1;
    double a = fabs((double)x);
    int m;
    if (a >= 223.0) {
        m = 511;
    } else if (a >= 16.0) {
        m = 304 + (int)floor(a) - 16;
    } else {
        m = o_fp16_rn_bits((float)a) >> 6;
    }
    return signbit(x) ? 512 + m : 511 - m;
}

/* ------------------------------------------------------------------------ */
/* O2: paged MQA logits ([DG94] "What this adds"; the logits formula)
 *   logits[r, t] = sum_h w[r, h] * ReLU( (sum_d q[r, h, d] * k[t, d]) * kscale[t] )
 * for t < n_r (R1).  K token t of request b lives in physical slot
 * page_table[b][t / page_size] * page_size + t % page_size.  The per-head dot
 * is exact in double (products of E4M3 values have at most 8 significant
 * bits and 128-term sums stay well inside 53 bits); the head sum is done in
 * double and rounded once to float.                                         */
static double o_logit_one(const uint8_t *q_row /* [H][D] */, const uint8_t *k_tok /* [D] */,
                          double kscale, const float *w_row /* [H] */, int H, int D,
                          const double *tab)
{
    double acc = 0.0;
    for (int h = 0; h < H; ++h) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += tab[q_row[h * D + d]] * tab[k_tok[d]];
        double v = dot * kscale;
        if (!(v > 0.0)) v = 0.0;                     /* ReLU (R2) */
        acc += (double)w_row[h] * v;
    }
    return acc;
}

static int64_t o_slot_of(const int32_t *page_table, int64_t pt_stride, int b, int64_t t, int ps)
{
    int32_t page = page_table[(int64_t)b * pt_stride + t / ps];
    return (int64_t)page * ps + t % ps;
}

/* Rows with n_r <= 0 have no live columns.  Only live columns are written. */
void o_paged_mqa_logits(const uint8_t *q, const uint8_t *kv, const float *kscale,
                        const float *weights, const int32_t *page_table, int64_t pt_stride,
                        const int32_t *context_lens, int B, int next_n, int H, int D,
                        int page_size, float *logits, int64_t logits_stride)
{
    double tab[256];
    o_e4m3_table(tab);
    for (int b = 0; b < B; ++b) {
        for (int j = 0; j < next_n; ++j) {
            int64_t r = (int64_t)b * next_n + j;
            int64_t n_r = (int64_t)context_lens[b] - (next_n - 1 - j);
            for (int64_t t = 0; t < n_r; ++t) {
                int64_t slot = o_slot_of(page_table, pt_stride, b, t, page_size);
                double v = o_logit_one(q + r * H * D, kv + slot * D, (double)kscale[slot],
                                       weights + r * H, H, D, tab);
                logits[r * logits_stride + t] = (float)v;
            }
        }
    }
}

/* Logits at an explicit list of (row, column) pairs, for sampled checks of
 * full-size runs.  Row r belongs to request r / next_n.                     */
void o_logits_at(const uint8_t *q, const uint8_t *kv, const float *kscale,
                 const float *weights, const int32_t *page_table, int64_t pt_stride,
                 int next_n, int H, int D, int page_size, const int64_t *rows,
                 const int64_t *cols, int64_t count, float *out)
{
    double tab[256];
    o_e4m3_table(tab);
    for (int64_t i = 0; i < count; ++i) {
        int64_t r = rows[i];
        int b = (int)(r / next_n);
        int64_t slot = o_slot_of(page_table, pt_stride, b, cols[i], page_size);
        out[i] = (float)o_logit_one(q + r * H * D, kv + slot * D, (double)kscale[slot],
                                    weights + r * H, H, D, tab);
    }
}

/* ------------------------------------------------------------------------ */
/* O3 continued: histogram of live, non-NaN scores, ADDED to the incoming
 * counts ([DG94]: counts accumulate across calls; the consumer resets).     */
void o_histogram_accumulate(const float *logits, int64_t stride, const int64_t *row_lens,
                            int R, int32_t *hist /* [R][1024] */)
{
    for (int r = 0; r < R; ++r) {
        for (int64_t t = 0; t < row_lens[r]; ++t) {
            int bin = o_coarse_bin(logits[(int64_t)r * stride + t]);
            if (bin >= 0) hist[(int64_t)r * 1024 + bin] += 1;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* O4: exact top-k by full sort (the textbook definition).  The FP32 order key
 * maps the IEEE bit pattern to an unsigned integer that sorts like the value
 * (-inf lowest, -0 below +0).  Ties on equal key go to the lower column (R6). */
static uint32_t o_f32_order_key(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

typedef struct {
    uint32_t key;
    int64_t col;
} o_kc_t;

static int o_kc_cmp(const void *pa, const void *pb)
{
    const o_kc_t *a = (const o_kc_t *)pa, *b = (const o_kc_t *)pb;
    if (a->key != b->key) return (a->key > b->key) ? -1 : 1;   /* key descending */
    return (a->col < b->col) ? -1 : (a->col > b->col);         /* column ascending */
}

/* One row: out[0..k) = selected columns in (value desc, column asc) order,
 * padded with -1.  Returns the number selected.                             */
int64_t o_topk_row(const float *row, int64_t n, int64_t k, int32_t *out)
{
    o_kc_t *buf = (o_kc_t *)malloc(sizeof(o_kc_t) * (size_t)(n > 0 ? n : 1));
    int64_t cnt = 0;
    for (int64_t t = 0; t < n; ++t) {
        if (isnan(row[t])) continue;
        buf[cnt].key = o_f32_order_key(row[t]);
        buf[cnt].col = t;
        ++cnt;
    }
    qsort(buf, (size_t)cnt, sizeof(o_kc_t), o_kc_cmp);
    int64_t take = cnt < k ? cnt : k;
    for (int64_t i = 0; i < k; ++i) out[i] = (i < take) ? (int32_t)buf[i].col : -1;
    free(buf);
    return take;
}

void o_topk(const float *logits, int64_t stride, const int64_t *row_lens, int R, int64_t k,
            int32_t *out /* [R][k] */)
{
    for (int r = 0; r < R; ++r)
        o_topk_row(logits + (int64_t)r * stride, row_lens[r], k, out + (int64_t)r * k);
}

/* ------------------------------------------------------------------------ */
/* O5: block max over 8 consecutive scores ([SG38944] amax8_varlen): for the
 * first nb = ceil(n/8) blocks of a row, block i < nb-1 holds the max of its 8
 * scores (R7), block nb-1 (the newest) is +inf, nothing past nb is written.
 * Rows with nb <= skip_le are left untouched when skip_le > 0.              */
void o_block_amax8(const float *logits, int64_t stride, const int64_t *row_lens, int R,
                   int64_t skip_le, float *amax, int64_t amax_stride)
{
    for (int r = 0; r < R; ++r) {
        int64_t n = row_lens[r];
        if (n <= 0) continue;
        int64_t nb = (n + 7) / 8;
        if (skip_le > 0 && nb <= skip_le) continue;
        for (int64_t i = 0; i + 1 < nb; ++i) {
            float m = NAN;
            for (int e = 0; e < 8; ++e) {
                float v = logits[(int64_t)r * stride + 8 * i + e];
                if (isnan(v)) continue;
                if (isnan(m) || o_f32_order_key(v) > o_f32_order_key(m)) m = v;
            }
            amax[(int64_t)r * amax_stride + i] = m;
        }
        amax[(int64_t)r * amax_stride + nb - 1] = INFINITY;
    }
}

/* ------------------------------------------------------------------------ */
/* O6: candidate block table ([SG38944] amax_topk_blocks + sort_candidate_blocks):
 * the top-kb blocks of the amax row (O4 rules, ties to the lower block id),
 * sorted ascending, padded with INT32_MAX; rows with nb <= kb get the
 * identity table 0..nb-1.  Physical block = pool slot / 8 through the row's
 * page table; valid length = live tokens covered by the chosen blocks (R8).  */
void o_block_table(const float *amax, int64_t amax_stride, const int64_t *row_lens,
                   const int32_t *row_to_req, int R, int kb, const int32_t *page_table,
                   int64_t pt_stride, int page_size, int32_t *table /* [R][kb] */,
                   int32_t *phys /* [R][kb] */, int32_t *valid_len /* [R] */)
{
    int32_t *sel = (int32_t *)malloc(sizeof(int32_t) * (size_t)kb);
    for (int r = 0; r < R; ++r) {
        int64_t n = row_lens[r] > 0 ? row_lens[r] : 0;
        int64_t nb = (n + 7) / 8;
        int64_t nsel = 0;
        if (nb <= kb) {
            for (int64_t i = 0; i < nb; ++i) sel[nsel++] = (int32_t)i;
        } else {
            nsel = o_topk_row(amax + (int64_t)r * amax_stride, nb, kb, sel);
            /* ascending order of block id: simple insertion sort */
            for (int64_t i = 1; i < nsel; ++i) {
                int32_t v = sel[i];
                int64_t p = i - 1;
                while (p >= 0 && sel[p] > v) {
                    sel[p + 1] = sel[p];
                    --p;
                }
                sel[p + 1] = v;
            }
        }
        int64_t live = 0;
        int b = row_to_req[r];
        for (int64_t i = 0; i < kb; ++i) {
            if (i < nsel) {
                int64_t id = sel[i];
                int64_t tok = id * 8;
                int64_t slot = o_slot_of(page_table, pt_stride, b, tok, page_size);
                table[(int64_t)r * kb + i] = (int32_t)id;
                phys[(int64_t)r * kb + i] = (int32_t)(slot / 8);
                int64_t in_blk = n - tok;
                live += in_blk < 8 ? in_blk : 8;
            } else {
                table[(int64_t)r * kb + i] = O_INT32_MAX;
                phys[(int64_t)r * kb + i] = O_INT32_MAX;
            }
        }
        valid_len[r] = (int32_t)live;
    }
    free(sel);
}

/* ------------------------------------------------------------------------ */
/* O7: sparse logits over the chosen blocks ([SG38944] "What this enables":
 * only the published blocks are scored).  Position i of row r is token
 * t = table[r][i/8]*8 + i%8; it takes the O2 value, or -inf when the table
 * entry is padding or t >= n_r (R9).                                         */
void o_sparse_logits(const uint8_t *q, const uint8_t *kv, const float *kscale,
                     const float *weights, const int32_t *page_table, int64_t pt_stride,
                     const int64_t *row_lens, const int32_t *row_to_req, int R, int H, int D,
                     int page_size, const int32_t *table, int kb, float *out, int64_t out_stride)
{
    double tab[256];
    o_e4m3_table(tab);
    for (int r = 0; r < R; ++r) {
        int b = row_to_req[r];
        for (int64_t i = 0; i < (int64_t)kb * 8; ++i) {
            int32_t id = table[(int64_t)r * kb + i / 8];
            int64_t t = (int64_t)id * 8 + i % 8;
            float v = -INFINITY;
            if (id != O_INT32_MAX && id >= 0 && t < row_lens[r]) {
                int64_t slot = o_slot_of(page_table, pt_stride, b, t, page_size);
                v = (float)o_logit_one(q + (int64_t)r * H * D, kv + slot * D,
                                       (double)kscale[slot], weights + (int64_t)r * H, H, D, tab);
            }
            out[(int64_t)r * out_stride + i] = v;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* O9: row pairing of the sparse pass ([SG38944] commit text on DeepGEMM's
 * sparse schedule: two consecutive rows of one request share one KV pass,
 * each keeping its own block list and output layout, on a shared page-table
 * row).  Reading R15: within a request, rows 2m and 2m+1 form a unit and an
 * odd last row is a unit of its own; a unit's pass walks the ascending union
 * of its rows' tables.  Union entry e holds the physical block and, for each
 * row, its position in that row's table plus one (0: the row does not hold
 * the block).  The union is a plain two-pointer merge of the two ascending
 * tables (INT32_MAX ends a table).  Units: B * ceil(next_n / 2); each output
 * row has 2*kb slots, padded with INT32_MAX (phys) and 0 (positions).        */
void o_pair_union(const int32_t *table, const int32_t *phys, int R, int next_n, int kb,
                  int32_t *uphys, int32_t *upos, int32_t *ulen)
{
    int upr = (next_n + 1) / 2;
    int U = (R / next_n) * upr;
    for (int u = 0; u < U; ++u) {
        int b = u / upr, m = u % upr;
        int ra = b * next_n + 2 * m;
        int rb = (2 * m + 1 < next_n) ? ra + 1 : -1;
        const int32_t *ta = table + (int64_t)ra * kb, *pa = phys + (int64_t)ra * kb;
        const int32_t *tb = rb >= 0 ? table + (int64_t)rb * kb : NULL;
        const int32_t *pb = rb >= 0 ? phys + (int64_t)rb * kb : NULL;
        int na = 0, nb = 0;
        while (na < kb && ta[na] != O_INT32_MAX) ++na;
        while (tb && nb < kb && tb[nb] != O_INT32_MAX) ++nb;
        int i = 0, j = 0, e = 0;
        int32_t *up = uphys + (int64_t)u * 2 * kb, *uq = upos + (int64_t)u * 2 * kb;
        while (i < na || j < nb) {
            if (j >= nb || (i < na && ta[i] < tb[j])) {
                up[e] = pa[i];
                uq[e] = i + 1;
                ++i;
            } else if (i >= na || tb[j] < ta[i]) {
                up[e] = pb[j];
                uq[e] = (j + 1) << 16;
                ++j;
            } else {
                up[e] = pa[i];
                uq[e] = (i + 1) | ((j + 1) << 16);
                ++i;
                ++j;
            }
            ++e;
        }
        ulen[u] = e;
        for (; e < 2 * kb; ++e) {
            up[e] = O_INT32_MAX;
            uq[e] = 0;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* O10: MXFP4 index keys.  The pages point to a block-scaled E2M1 index-K
 * cache as the next format: [SG38944] (the Hopper prefill commit text:
 * decode block-scaled E2M1 index keys directly to E4M3), [VL52696] ("Why"
 * and the MXFP4 indexer-cache tests: the packed 68-byte cache layout), and
 * [DG94] "What this adds" (the fused histogram is specified for FP8 "non-MX"
 * only).  Reading R16: a token's key is 128 E2M1 codes packed two per byte
 * (dimension 2i in the low nibble of byte i, 2i+1 in the high nibble: 64
 * bytes) plus 4 UE8M0 block exponents (block b covers dimensions 32b ..
 * 32b+31: 4 bytes) -- 68 bytes; k[d] = E2M1(code[d]) * 2^(e[d / 32] - 127),
 * with no per-token kscale.  E2M1: sign bit 3, exponent bits 2..1 with bias 1,
 * mantissa bit 0, exponent field 0 subnormal (m * 0.5), no inf or NaN.
 * UE8M0: 2^(e - 127), e = 255 is NaN.  Queries stay FP8 E4M3.              */
double o_e2m1(uint8_t c)
{
    int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

double o_ue8m0(uint8_t e)
{
    return e == 255 ? NAN : ldexp(1.0, (int)e - 127);
}

/* one logit with an MXFP4 key (the O2 formula with kscale = 1); the per-head
 * dot is exact in double while a token's block exponents lie within about 40
 * binades of each other */
static double o_logit_one_mx(const uint8_t *q_row /* [H][D] */, const uint8_t *k_codes /* [D/2] */,
                             const uint8_t *k_exp /* [D/32] */, const float *w_row, int H, int D,
                             const double *tab)
{
    double acc = 0.0;
    for (int h = 0; h < H; ++h) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) {
            uint8_t byte = k_codes[d / 2];
            uint8_t code = (d % 2 == 0) ? (byte & 0xF) : (byte >> 4);
            double k = o_e2m1(code) * o_ue8m0(k_exp[d / 32]);
            dot += tab[q_row[h * D + d]] * k;
        }
        double v = dot;
        if (!(v > 0.0)) v = 0.0;                     /* ReLU (R2) */
        acc += (double)w_row[h] * v;
    }
    return acc;
}

/* dense logits over an MXFP4 paged cache: k_codes [slots][D/2], k_exp
 * [slots][D/32], slots = num_pages * page_size; same rows and gather as O2,
 * live columns written only */
void o_paged_mqa_logits_mx(const uint8_t *q, const uint8_t *k_codes, const uint8_t *k_exp,
                           const float *weights, const int32_t *page_table, int64_t pt_stride,
                           const int32_t *context_lens, int B, int next_n, int H, int D,
                           int page_size, float *out, int64_t out_stride)
{
    double tab[256];
    o_e4m3_table(tab);
    for (int b = 0; b < B; ++b) {
        for (int j = 0; j < next_n; ++j) {
            int r = b * next_n + j;
            int64_t n = (int64_t)context_lens[b] - (next_n - 1 - j);
            for (int64_t t = 0; t < n && t < out_stride; ++t) {
                int64_t slot = o_slot_of(page_table, pt_stride, b, t, page_size);
                out[(int64_t)r * out_stride + t] =
                    (float)o_logit_one_mx(q + (int64_t)r * H * D, k_codes + slot * (D / 2),
                                          k_exp + slot * (D / 32), weights + (int64_t)r * H, H,
                                          D, tab);
            }
        }
    }
}

/* MXFP4 logits at an explicit list of (row, column) pairs (full-size sampled
 * checks); row r belongs to request r / next_n. */
void o_logits_at_mx(const uint8_t *q, const uint8_t *k_codes, const uint8_t *k_exp,
                    const float *weights, const int32_t *page_table, int64_t pt_stride,
                    int next_n, int H, int D, int page_size, const int64_t *rows,
                    const int64_t *cols, int64_t n, float *out)
{
    double tab[256];
    o_e4m3_table(tab);
    for (int64_t i = 0; i < n; ++i) {
        int64_t r = rows[i];
        int b = (int)(r / next_n);
        int64_t slot = o_slot_of(page_table, pt_stride, b, cols[i], page_size);
        out[i] = (float)o_logit_one_mx(q + r * H * D, k_codes + slot * (D / 2),
                                       k_exp + slot * (D / 32), weights + r * H, H, D, tab);
    }
}

/* ------------------------------------------------------------------------ */
/* O8: top-k over FP16 scores ([VL52696] "Why": select on FP16 score bits).
 * Positions i < valid_len[r] take part unless NaN; order by the FP16 value,
 * ties to the lower position; the output is the logical column
 * table[r][i/8]*8 + i%8 when a table is given, else the position i.        */
static uint32_t o_f16_order_key(uint16_t h)
{
    /* sign-magnitude 16-bit formats (FP16 and BF16 alike) order by this key */
    return (h & 0x8000u) ? (uint32_t)(~h & 0xFFFFu) : (uint32_t)(h | 0x8000u);
}

static void o_topk_16(const uint16_t *scores, int64_t stride, const int32_t *valid_len, int R,
                      int64_t k, const int32_t *table, int kb, int32_t *out,
                      double (*decode)(uint16_t))
{
    for (int r = 0; r < R; ++r) {
        int64_t n = valid_len[r];
        o_kc_t *buf = (o_kc_t *)malloc(sizeof(o_kc_t) * (size_t)(n > 0 ? n : 1));
        int64_t cnt = 0;
        for (int64_t i = 0; i < n; ++i) {
            uint16_t h = scores[(int64_t)r * stride + i];
            if (isnan(decode(h))) continue;
            buf[cnt].key = o_f16_order_key(h);
            buf[cnt].col = i;
            ++cnt;
        }
        qsort(buf, (size_t)cnt, sizeof(o_kc_t), o_kc_cmp);
        int64_t take = cnt < k ? cnt : k;
        for (int64_t i = 0; i < k; ++i) {
            int32_t v = -1;
            if (i < take) {
                int64_t p = buf[i].col;
                v = table ? (int32_t)((int64_t)table[(int64_t)r * kb + p / 8] * 8 + p % 8)
                          : (int32_t)p;
            }
            out[(int64_t)r * k + i] = v;
        }
        free(buf);
    }
}

void o_topk_fp16(const uint16_t *scores, int64_t stride, const int32_t *valid_len, int R,
                 int64_t k, const int32_t *table, int kb, int32_t *out /* [R][k] */)
{
    o_topk_16(scores, stride, valid_len, R, k, table, kb, out, o_fp16_bits_to_double);
}

/* The same selection over BF16 scores. */
void o_topk_bf16(const uint16_t *scores, int64_t stride, const int32_t *valid_len, int R,
                 int64_t k, const int32_t *table, int kb, int32_t *out /* [R][k] */)
{
    o_topk_16(scores, stride, valid_len, R, k, table, kb, out, o_bf16_bits_to_double);
}

/* ------------------------------------------------------------------------ */
/* Sweep helpers for exhaustive pins: evaluate over a range of bit patterns. */
void o_fp16_rn_sweep(uint64_t start, uint64_t count, uint16_t *out)
{
    for (uint64_t i = 0; i < count; ++i) {
        uint32_t u = (uint32_t)(start + i);
        float x;
        memcpy(&x, &u, 4);
        out[i] = o_fp16_rn_bits(x);
    }
}

void o_coarse_bin_sweep(uint64_t start, uint64_t count, int16_t *out)
{
    for (uint64_t i = 0; i < count; ++i) {
        uint32_t u = (uint32_t)(start + i);
        float x;
        memcpy(&x, &u, 4);
        out[i] = (int16_t)o_coarse_bin(x);
    }
}

/* Element-wise helpers over arrays (same scalar functions as above). */
void o_coarse_bins(const float *x, int64_t n, int16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = (int16_t)o_coarse_bin(x[i]);
}

void o_fp16_rn_array(const float *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = o_fp16_rn_bits(x[i]);
}

void o_bf16_rn_array(const float *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = o_bf16_rn_bits(x[i]);
}

void o_bf16_rn_sweep(uint64_t start, uint64_t count, uint16_t *out)
{
    for (uint64_t i = 0; i < count; ++i) {
        uint32_t u = (uint32_t)(start + i);
        float x;
        memcpy(&x, &u, 4);
        out[i] = o_bf16_rn_bits(x);
    }
}
