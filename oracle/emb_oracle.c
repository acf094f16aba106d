/*
 * CPU oracle for the sparse embedding training step -- TEST INFRASTRUCTURE.
 *
 * Only the tests, the package smoke check and the benchmark's CPU-baseline leg
 * load this file.  It shares no code, header, table or helper with the CUDA
 * library: it is a plain, slow, single-threaded restatement of what the step
 * computes, with every sum accumulated in binary64 and rounded once at the end.
 *
 * Passages followed (page title, then section / slide):
 *  - "Merlin HugeCTR: GPU-accelerated recommender system training and
 *    inference" (GTC 2022 slides), slide "COMMON EMBEDDING PRIMITIVES":
 *    (1) table lookup, (2) pooling/reduction, (3) concatenation; slide
 *    "HUGECTR EMBEDDING LAYER" (lookup + reduction + concatenation as one op).
 *  - Merlin overview article, section "HugeCTR": the features of one slot are
 *    each turned into an embedding vector and then reduced to a single vector.
 *  - Same slides, slide "WEIGHT CONVERSION FOR MIXED PRECISION TRAINING": the
 *    optimizer computes in FP32 and the result is cast to the FP16 table.
 *  - "NVIDIA EMBark revoluciona la formacion en sistemas de recomendacion a
 *    escala", section "Integracion del cluster": reduction-based (RB) and
 *    unique-based (UB) handling only reorganise the backward; the update they
 *    produce is the same, so the oracle computes it once, by definition.
 *  - The optimizers are not on the pages.  SGD is W <- W - lr*G.  Adagrad is
 *    the per-element form of Duchi, Hazan & Singer (JMLR 2011) with eps outside
 *    the square root and the accumulator updated before the weight:
 *    A <- A + G*G ; W <- W - lr*G/(sqrt(A)+eps).  Row-wise Adagrad keeps one
 *    accumulator per row and adds the mean over the row's columns of G*G to
 *    it: A <- A + (1/dim) * sum_c G_c^2 ; W <- W - lr*G/(sqrt(A)+eps) (the
 *    form used by the open DLRM embedding libraries; the pages do not define it).
 *  - GTC 2022 HugeCTR slides, "WEIGHT CONVERSION FOR MIXED PRECISION
 *    TRAINING": the optimizer works on FP32 weights and the FP16 copy the
 *    forward reads is converted from them.  A table with an fp32 master copy
 *    updates the master in fp32 and stores the 16-bit weight as the master
 *    rounded to nearest-even.
 *  - Duplicate keys in one batch: their gradients are summed first and each
 *    touched row gets exactly one optimizer step per batch.
 *
 * Conventions: bag j = t*B + b (table-major), so table_ids[j] must equal j/B;
 * the pooled output is the concatenation out[b][doff[t] .. doff[t]+dim[t]).
 * A key outside [0, rows_t), or a bag whose table id is not j/B, contributes
 * nothing and is counted as an error.  Mean pooling divides by the bag length
 * L = offsets[j+1]-offsets[j]; an empty bag pools to 0.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Round-to-nearest-even from binary64 into the table storage formats.        */
/* ------------------------------------------------------------------------- */

/* Round |x| (finite, non-negative) to a binary format with `mbits` fraction
 * bits, minimum normal exponent `emin` and exponent bias `bias`; returns the
 * bit pattern without sign, or the infinity pattern on overflow. */
static uint32_t rne_bits(double ax, int mbits, int emin, int emax, int ebits)
{
    const uint32_t inf = ((1u << ebits) - 1u) << mbits;
    if (ax == 0.0) return 0;
    int e2;
    frexp(ax, &e2);                  /* ax = m * 2^e2, m in [0.5, 1) */
    int e = e2 - 1;                  /* ax in [2^e, 2^(e+1)) */
    if (e < emin) e = emin;          /* subnormal range shares the quantum of emin */
    double q = ldexp(1.0, e - mbits);
    double n = rint(ax / q);         /* exact scaling, ties to even */
    double v = n * q;                /* rounded magnitude */
    if (v == 0.0) return 0;
    if (v >= ldexp(1.0, emax + 1)) return inf;
    int ev;
    frexp(v, &ev);
    ev -= 1;
    if (ev < emin) {                 /* subnormal: bits are the multiple of 2^(emin-mbits) */
        return (uint32_t)ldexp(v, mbits - emin);
    }
    double frac = ldexp(v, -ev) - 1.0;                 /* in [0, 1) */
    uint32_t mant = (uint32_t)ldexp(frac, mbits);
    uint32_t bias = (1u << (ebits - 1)) - 1u;
    return ((uint32_t)(ev + (int)bias) << mbits) | mant;
}

uint16_t ora_round_f16(double x)
{
    if (isnan(x)) return 0x7E00;
    uint16_t s = signbit(x) ? 0x8000 : 0;
    return (uint16_t)(s | rne_bits(fabs(x), 10, -14, 15, 5));
}

uint16_t ora_round_bf16(double x)
{
    if (isnan(x)) return 0x7FC0;
    uint16_t s = signbit(x) ? 0x8000 : 0;
    return (uint16_t)(s | rne_bits(fabs(x), 7, -126, 127, 8));
}

static double decode_bits(uint32_t b, int mbits, int ebits, int sign_bit)
{
    int neg = (b >> sign_bit) & 1u;
    uint32_t ex = (b >> mbits) & ((1u << ebits) - 1u);
    uint32_t mant = b & ((1u << mbits) - 1u);
    int bias = (1 << (ebits - 1)) - 1;
    double v;
    if (ex == ((1u << ebits) - 1u)) v = mant ? NAN : INFINITY;
    else if (ex == 0) v = ldexp((double)mant, 1 - bias - mbits);
    else v = ldexp((double)(mant | (1u << mbits)), (int)ex - bias - mbits);
    return neg ? -v : v;
}

double ora_f16_to_f64(uint16_t h) { return decode_bits(h, 10, 5, 15); }
double ora_bf16_to_f64(uint16_t h) { return decode_bits(h, 7, 8, 15); }

void ora_round_f16_array(const double* x, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = ora_round_f16(x[i]);
}
void ora_round_bf16_array(const double* x, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = ora_round_bf16(x[i]);
}

/* ------------------------------------------------------------------------- */
/* Step a2: global row ids.                                                   */
/* ------------------------------------------------------------------------- */

/* gid_i = row_base[t] + key_i for every position i of bag j = t*B + b.
 * Positions whose key is outside [0, rows[t]) or whose bag has a wrong table
 * id get -1.  Returns the number of such positions (and bad bags). */
int64_t ora_global_ids(int32_t T, int32_t B, const int64_t* offsets, const int64_t* keys,
                       const int32_t* table_ids, const int64_t* rows, const int64_t* row_base,
                       int64_t* gids)
{
    int64_t bad = 0;
    for (int64_t j = 0; j < (int64_t)T * B; ++j) {
        int32_t t = (int32_t)(j / B);
        int table_ok = table_ids[j] == t;
        if (!table_ok) ++bad;
        for (int64_t i = offsets[j]; i < offsets[j + 1]; ++i) {
            int64_t k = keys[i];
            if (table_ok && k >= 0 && k < rows[t]) {
                gids[i] = row_base[t] + k;
            } else {
                gids[i] = -1;
                if (table_ok) ++bad;
            }
        }
    }
    return bad;
}

/* ------------------------------------------------------------------------- */
/* Step a3: unique keys, inverse index, counts, segment offsets.              */
/* ------------------------------------------------------------------------- */

static int cmp_i64(const void* a, const void* b)
{
    int64_t x = *(const int64_t*)a, y = *(const int64_t*)b;
    return (x > y) - (x < y);
}

static int64_t lower_bound_i64(const int64_t* a, int64_t n, int64_t v)
{
    int64_t lo = 0, hi = n;
    while (lo < hi) {
        int64_t mid = lo + (hi - lo) / 2;
        if (a[mid] < v) lo = mid + 1; else hi = mid;
    }
    return lo;
}

/* Sorted-ascending distinct values uniq[0..U) of keys[0..n), with
 * uniq[inverse[i]] == keys[i], counts[k] = #{i : keys[i] == uniq[k]} and
 * seg_off[k] = counts[0] + ... + counts[k-1] (seg_off[U] = n).
 * `skip_negative` != 0 leaves keys < 0 out (their inverse becomes U).
 * Returns U. */
int64_t ora_unique(const int64_t* keys, int64_t n, int skip_negative,
                   int64_t* uniq, int32_t* inverse, int32_t* counts, int32_t* seg_off)
{
    int64_t m = 0;
    int64_t* tmp = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    for (int64_t i = 0; i < n; ++i)
        if (!skip_negative || keys[i] >= 0) tmp[m++] = keys[i];
    qsort(tmp, (size_t)m, sizeof(int64_t), cmp_i64);
    int64_t U = 0;
    for (int64_t i = 0; i < m; ++i) {
        if (i == 0 || tmp[i] != tmp[i - 1]) {
            uniq[U] = tmp[i];
            if (seg_off) seg_off[U] = (int32_t)i;
            if (counts) counts[U] = 0;
            ++U;
        }
        if (counts) counts[U - 1] += 1;
    }
    if (seg_off) seg_off[U] = (int32_t)m;
    if (inverse) {
        for (int64_t i = 0; i < n; ++i) {
            if (skip_negative && keys[i] < 0) { inverse[i] = (int32_t)U; continue; }
            inverse[i] = (int32_t)lower_bound_i64(uniq, U, keys[i]);
        }
    }
    free(tmp);
    return U;
}

/* ------------------------------------------------------------------------- */
/* Step a1: lookup, pooling and concatenation.                               */
/* ------------------------------------------------------------------------- */

/* For every bag j = t*B + b in `bags` (all bags when bags == NULL):
 *   out[b*ld + doff[t] + c] = s_j * sum_{i in bag j} W_t[key_i][c]
 * with s_j = 1 (sum) or 1/L_j (mean), accumulated in binary64 in position
 * order and rounded once to fp32.  Row values come from the row store:
 * position i reads vals[row_start[inv[i]] + c]; inv[i] < 0 or >= U marks an
 * invalid position, which contributes nothing.  absacc (nullable) receives
 * s_j * sum |W| per element, the magnitude scale of the sum. */
void ora_forward(int32_t T, int32_t B, const int64_t* offsets, const int32_t* inv, int64_t U,
                 const int64_t* row_start, const double* vals,
                 const int32_t* dims, const int64_t* doff, const int32_t* pooling, int64_t ld,
                 const int64_t* bags, int64_t nbags, float* out, double* absacc)
{
    int64_t total = bags ? nbags : (int64_t)T * B;
    int32_t maxdim = 0;
    for (int32_t t = 0; t < T; ++t) if (dims[t] > maxdim) maxdim = dims[t];
    double* acc = (double*)malloc(sizeof(double) * (size_t)maxdim * 2);
    double* aab = acc + maxdim;
    for (int64_t q = 0; q < total; ++q) {
        int64_t j = bags ? bags[q] : q;
        int32_t t = (int32_t)(j / B);
        int64_t b = j % B;
        int32_t d = dims[t];
        for (int32_t c = 0; c < d; ++c) { acc[c] = 0.0; aab[c] = 0.0; }
        int64_t L = offsets[j + 1] - offsets[j];
        for (int64_t i = offsets[j]; i < offsets[j + 1]; ++i) {
            int64_t k = inv[i];
            if (k < 0 || k >= U) continue;
            const double* w = vals + row_start[k];
            for (int32_t c = 0; c < d; ++c) { acc[c] += w[c]; aab[c] += fabs(w[c]); }
        }
        int mean = pooling[t] == 1 && L > 0;
        for (int32_t c = 0; c < d; ++c) {
            double v = mean ? acc[c] / (double)L : acc[c];
            double a = mean ? aab[c] / (double)L : aab[c];
            out[b * ld + doff[t] + c] = (float)v;
            if (absacc) absacc[b * ld + doff[t] + c] = a;
        }
    }
    free(acc);
}

/* ------------------------------------------------------------------------- */
/* Step a4: per-unique-row gradient reduction.                               */
/* ------------------------------------------------------------------------- */

/* G[row_start[k] + c] = sum over positions i with inv[i] == k, ascending i, of
 *   s_bag(i) * grad_out[b(i)*ld + doff[t] + c]
 * in binary64 (s = 1 for sum pooling, 1/L for mean).  Gabs (nullable) gets
 * the sum of magnitudes of the same terms.  G and Gabs are zeroed here. */
void ora_reduce(int32_t T, int32_t B, const int64_t* offsets, const int32_t* inv, int64_t U,
                const int64_t* row_start, int64_t row_total,
                const int32_t* dims, const int64_t* doff, const int32_t* pooling, int64_t ld,
                const float* grad_out, double* G, double* Gabs)
{
    memset(G, 0, sizeof(double) * (size_t)row_total);
    if (Gabs) memset(Gabs, 0, sizeof(double) * (size_t)row_total);
    for (int64_t j = 0; j < (int64_t)T * B; ++j) {
        int32_t t = (int32_t)(j / B);
        int64_t b = j % B;
        int64_t L = offsets[j + 1] - offsets[j];
        const float* g = grad_out + b * ld + doff[t];
        for (int64_t i = offsets[j]; i < offsets[j + 1]; ++i) {
            int64_t k = inv[i];
            if (k < 0 || k >= U) continue;
            double* dst = G + row_start[k];
            for (int32_t c = 0; c < dims[t]; ++c) {
                double term = pooling[t] == 1 ? (double)g[c] / (double)L : (double)g[c];
                dst[c] += term;
                if (Gabs) Gabs[row_start[k] + c] += fabs(term);
            }
        }
    }
}

/* Same sums restricted to the sorted sample of global ids `sample[0..S)`:
 * G[q*maxdim + c] for sample q; positions are matched by their global id. */
void ora_reduce_sampled(int32_t T, int32_t B, const int64_t* offsets, const int64_t* gids,
                        const int64_t* sample, int64_t S, int32_t maxdim,
                        const int32_t* dims, const int64_t* doff, const int32_t* pooling, int64_t ld,
                        const float* grad_out, double* G, double* Gabs, int64_t* count)
{
    memset(G, 0, sizeof(double) * (size_t)(S * maxdim));
    if (Gabs) memset(Gabs, 0, sizeof(double) * (size_t)(S * maxdim));
    memset(count, 0, sizeof(int64_t) * (size_t)S);
    for (int64_t j = 0; j < (int64_t)T * B; ++j) {
        int32_t t = (int32_t)(j / B);
        int64_t b = j % B;
        int64_t L = offsets[j + 1] - offsets[j];
        const float* g = grad_out + b * ld + doff[t];
        for (int64_t i = offsets[j]; i < offsets[j + 1]; ++i) {
            if (gids[i] < 0) continue;
            int64_t q = lower_bound_i64(sample, S, gids[i]);
            if (q >= S || sample[q] != gids[i]) continue;
            count[q] += 1;
            for (int32_t c = 0; c < dims[t]; ++c) {
                double term = pooling[t] == 1 ? (double)g[c] / (double)L : (double)g[c];
                G[q * maxdim + c] += term;
                if (Gabs) Gabs[q * maxdim + c] += fabs(term);
            }
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Step a5: optimizer update of every touched row, one step per batch.       */
/* ------------------------------------------------------------------------- */

/* For each row k (table row_table[k], `dim` = dims[row_table[k]]):
 *   SGD:     W' = W - lr*G
 *   Adagrad: A' = A + G*G ;  W' = W - lr*G/(sqrt(A')+eps)
 *   row-wise Adagrad (opt 2): a' = a + (1/dim) sum_c G_c^2 for the row's one
 *     accumulator a, W' = W - lr*G/(sqrt(a')+eps); the row store holds a in
 *     every column of the row (all equal)
 * in binary64 from the stored values; W' is then rounded once to the table
 * storage type (0 fp32, 1 fp16, 2 bf16) and A' to fp32, and both are written
 * back as the binary64 value of the rounded result.  Wscale/Ascale
 * (nullable) receive the magnitude scales |W| + lr*Gabs/(sqrt(A')+eps) (SGD:
 * |W| + lr*Gabs) and A + Gabs^2 (row-wise: a + (1/dim) sum_c Gabs_c^2) used
 * to judge rounding error.
 * master (nullable): for tables with master[t] set (16-bit storage), W holds
 * the fp32 master values; W' is rounded to fp32 as the new master and the
 * stored 16-bit weight is that master rounded to the storage type.  W16
 * (nullable) receives the stored weight after the step for every row (the
 * same as W for tables without a master). */
void ora_update(int64_t U, const int32_t* row_table, const int64_t* row_start,
                const int32_t* dims, const int32_t* dtype, const int32_t* opt,
                const int32_t* master, const double* lr, const double* eps,
                const double* G, const double* Gabs, double* W, double* A,
                double* Wscale, double* Ascale, double* W16)
{
    for (int64_t k = 0; k < U; ++k) {
        int32_t t = row_table[k];
        int64_t base = row_start[k];
        double row_a = 0.0, row_den = 0.0, row_ascale = 0.0;
        if (opt[t] == 2) {
            double ssq = 0.0, ssq_abs = 0.0;
            for (int32_t c = 0; c < dims[t]; ++c) {
                ssq += G[base + c] * G[base + c];
                if (Gabs) ssq_abs += Gabs[base + c] * Gabs[base + c];
            }
            row_a = A[base] + ssq / (double)dims[t];
            row_den = sqrt(row_a) + eps[t];
            row_ascale = A[base] + ssq_abs / (double)dims[t];
        }
        for (int32_t c = 0; c < dims[t]; ++c) {
            double g = G[base + c];
            double w = W[base + c];
            double wn, step_scale;
            if (opt[t] == 2) {
                wn = w - lr[t] * g / row_den;
                step_scale = Gabs ? lr[t] * Gabs[base + c] / row_den : 0.0;
                if (Ascale) Ascale[base + c] = row_ascale;
                A[base + c] = (double)(float)row_a;
            } else if (opt[t] == 1) {
                double a = A[base + c] + g * g;
                double den = sqrt(a) + eps[t];
                wn = w - lr[t] * g / den;
                step_scale = Gabs ? lr[t] * Gabs[base + c] / den : 0.0;
                if (Ascale) Ascale[base + c] = A[base + c] + (Gabs ? Gabs[base + c] * Gabs[base + c] : 0.0);
                A[base + c] = (double)(float)a;
            } else {
                wn = w - lr[t] * g;
                step_scale = Gabs ? lr[t] * Gabs[base + c] : 0.0;
            }
            if (Wscale) Wscale[base + c] = fabs(w) + step_scale;
            if (master && master[t] && dtype[t] != 0) {
                wn = (double)(float)wn;   /* the new fp32 master */
                if (W16)
                    W16[base + c] = dtype[t] == 1 ? ora_f16_to_f64(ora_round_f16(wn))
                                                  : ora_bf16_to_f64(ora_round_bf16(wn));
            } else {
                if (dtype[t] == 1) wn = ora_f16_to_f64(ora_round_f16(wn));
                else if (dtype[t] == 2) wn = ora_bf16_to_f64(ora_round_bf16(wn));
                else wn = (double)(float)wn;
                if (W16) W16[base + c] = wn;
            }
            W[base + c] = wn;
        }
    }
}
