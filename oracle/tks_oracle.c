/*
 * CPU oracle for the DSA TopK selector.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the test-suite, the smoke check and the benchmark's CPU-baseline leg
 * load this file.  The selection library never calls, links or includes it,
 * and this file includes nothing from the library.
 *
 * What it computes ("Technical Deep Dive | ... Triton-TLE ... TopK Selector",
 * section "01. Why the TopK Selector Needs Optimization", and the collection
 * step of the radix_topk pseudocode in section "02. Traditional GPU Approach:
 * Radix Selection"): for one row of L logits v[0..L) and a count k, the set of
 * the k positions holding the largest values, indices only, no sorted output.
 * Where the k-th value is shared by several positions, the pseudocode first
 * takes every value strictly above it and then appends positions equal to it
 * while walking the row from the start, so ties go to the lowest indices.
 *
 * That is the first min(k, L) entries of the row ordered by the strict total
 * order "i before j" defined in rank_before() below, which this file realises
 * plainly: a stable merge sort of the positions 0..L-1, then the first k.
 *
 * Readings where the page is silent (each also listed with the design notes):
 *   - +0.0 ranks above -0.0 (the sign-flip key of the "Mapping" step orders
 *     them that way; plain float comparison would call them equal);
 *   - -inf is an ordinary, lowest value, selected only if fewer than k other
 *     values exist; validity of a position is given by the row length alone;
 *   - subnormals keep their exact order (no flush to zero): build without
 *     -ffast-math; tks_oracle_selftest() checks this at run time;
 *   - NaN in the valid prefix is outside the contract: the call fails;
 *   - if L < k the remaining k - L outputs are -1 (the flush of the
 *     selector's output buffer in section "5. Triton-TLE" pads with -1);
 *   - the returned set is sorted ascending, so that sets compare element-wise;
 *     the "ordered" entry points instead return the selected positions in
 *     the order above (largest value first, ties by lower position), the
 *     optional sorted output of the pseudocode's final step.
 *
 * Parity pins (brute force, rank counting, the page's base-10 digit
 * selection, closed forms, invariants) live in the test-suite.
 *
 * Plain C11, single thread, no SIMD, no library sort.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define TKS_ORACLE_OK 0
#define TKS_ORACLE_EINVAL 1
#define TKS_ORACLE_ENAN 2
#define TKS_ORACLE_ENOMEM 3

/* Test-only mutants: a test compiles this file with one of these defined to
 * check that the pins catch a plausible mistake.  Never defined otherwise. */
#ifndef TKS_ORACLE_MUTANT
#define TKS_ORACLE_MUTANT 0
#endif

/* Strict total order on positions of one row: i comes before j when its value
 * is larger; for equal values +0.0 comes before -0.0; for equal values of the
 * same sign the lower position comes first. */
static int rank_before(const float *v, int64_t i, int64_t j)
{
    float a = v[i], b = v[j];
#if TKS_ORACLE_MUTANT == 1 /* ascending instead of descending */
    if (a < b) return 1;
    if (a > b) return 0;
#else
    if (a > b) return 1;
    if (a < b) return 0;
#endif
    {
        int sa = signbit(a) ? 1 : 0, sb = signbit(b) ? 1 : 0;
#if TKS_ORACLE_MUTANT == 2 /* -0.0 above +0.0 */
        if (sa != sb) return sa > sb;
#elif TKS_ORACLE_MUTANT == 3 /* sign rule dropped */
        (void)sa; (void)sb;
#else
        if (sa != sb) return sa < sb;
#endif
    }
#if TKS_ORACLE_MUTANT == 4 /* ties to the highest index */
    return i > j;
#else
    return i < j;
#endif
}

/* Bottom-up stable merge sort of pos[0..n) under rank_before. */
static void merge_sort_positions(const float *v, int64_t *pos, int64_t *tmp, int64_t n)
{
    int64_t width, lo;
    for (width = 1; width < n; width *= 2) {
        for (lo = 0; lo < n; lo += 2 * width) {
            int64_t mid = lo + width < n ? lo + width : n;
            int64_t hi = lo + 2 * width < n ? lo + 2 * width : n;
            int64_t a = lo, b = mid, o = lo;
            while (a < mid && b < hi) {
                /* take from the right run only if it strictly comes first */
                if (rank_before(v, pos[b], pos[a])) tmp[o++] = pos[b++];
                else tmp[o++] = pos[a++];
            }
            while (a < mid) tmp[o++] = pos[a++];
            while (b < hi) tmp[o++] = pos[b++];
        }
        memcpy(pos, tmp, (size_t)n * sizeof(int64_t));
    }
}

/* Ascending insertion into out[0..m): plain sort for the final canonical set. */
static void sort_ascending_i64(int64_t *a, int64_t m)
{
    /* shell sort with the 3x+1 gaps: small code, O(m^1.5) */
    int64_t gap = 1, i, j;
    while (gap < m / 3) gap = 3 * gap + 1;
    for (; gap >= 1; gap /= 3) {
        for (i = gap; i < m; ++i) {
            int64_t x = a[i];
            for (j = i; j >= gap && a[j - gap] > x; j -= gap) a[j] = a[j - gap];
            a[j] = x;
        }
    }
}

/* Top-k of one float row.  out has room for k entries.  ordered = 0: the
 * set in ascending position order; ordered = 1: in rank order. */
int tks_oracle_topk_f32_order(const float *v, int64_t row_len, int64_t k, int32_t ordered,
                              int32_t *out)
{
    int64_t *pos, *tmp, i, take;
    if (row_len < 0 || k < 1 || (row_len > 0 && v == NULL) || out == NULL) return TKS_ORACLE_EINVAL;
    if (row_len > INT32_MAX) return TKS_ORACLE_EINVAL;
    for (i = 0; i < row_len; ++i)
        if (isnan(v[i])) return TKS_ORACLE_ENAN;
    take = row_len < k ? row_len : k;
#if TKS_ORACLE_MUTANT == 5 /* one element short */
    if (take > 0) take -= 1;
#endif
    pos = (int64_t *)malloc((size_t)(row_len > 0 ? row_len : 1) * sizeof(int64_t));
    tmp = (int64_t *)malloc((size_t)(row_len > 0 ? row_len : 1) * sizeof(int64_t));
    if (pos == NULL || tmp == NULL) {
        free(pos);
        free(tmp);
        return TKS_ORACLE_ENOMEM;
    }
    for (i = 0; i < row_len; ++i) pos[i] = i;
    merge_sort_positions(v, pos, tmp, row_len);
#if TKS_ORACLE_MUTANT == 7 /* rank order with ties reversed */
    if (ordered) {
        int64_t a = 0, b2;
        while (a < take) {
            b2 = a + 1;
            while (b2 < take && v[pos[b2]] == v[pos[a]] && signbit(v[pos[b2]]) == signbit(v[pos[a]])) ++b2;
            for (i = 0; i < (b2 - a) / 2; ++i) {
                int64_t t = pos[a + i];
                pos[a + i] = pos[b2 - 1 - i];
                pos[b2 - 1 - i] = t;
            }
            a = b2;
        }
    }
#endif
    if (!ordered) sort_ascending_i64(pos, take);
    for (i = 0; i < take; ++i) out[i] = (int32_t)pos[i];
    for (i = take; i < k; ++i) out[i] = -1;
    free(pos);
    free(tmp);
    return TKS_ORACLE_OK;
}

/* bfloat16 is the upper half of a float32: widening by a 16-bit shift is exact. */
static float widen_bf16(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
#if TKS_ORACLE_MUTANT == 6 /* wrong half */
    u = (uint32_t)b;
#endif
    memcpy(&f, &u, sizeof f);
    return f;
}

int tks_oracle_topk_f32(const float *v, int64_t row_len, int64_t k, int32_t *out)
{
    return tks_oracle_topk_f32_order(v, row_len, k, 0, out);
}

int tks_oracle_topk_bf16_order(const uint16_t *b, int64_t row_len, int64_t k, int32_t ordered,
                               int32_t *out)
{
    float *v;
    int64_t i;
    int rc;
    if (row_len < 0 || (row_len > 0 && b == NULL)) return TKS_ORACLE_EINVAL;
    v = (float *)malloc((size_t)(row_len > 0 ? row_len : 1) * sizeof(float));
    if (v == NULL) return TKS_ORACLE_ENOMEM;
    for (i = 0; i < row_len; ++i) v[i] = widen_bf16(b[i]);
    rc = tks_oracle_topk_f32_order(v, row_len, k, ordered, out);
    free(v);
    return rc;
}

int tks_oracle_topk_bf16(const uint16_t *b, int64_t row_len, int64_t k, int32_t *out)
{
    return tks_oracle_topk_bf16_order(b, row_len, k, 0, out);
}

/* A batch laid out as rows of row_stride elements; dtype 0 = float32, 1 = bf16.
 * row_len may be NULL (every row has row_stride valid elements).
 * out is [batch][k]. */
int tks_oracle_topk_batch_order(const void *values, int32_t dtype, int64_t batch, int64_t row_stride,
                                const int32_t *row_len, int64_t k, int32_t ordered, int32_t *out)
{
    int64_t r;
    if (batch < 0 || row_stride < 0 || k < 1 || (dtype != 0 && dtype != 1)) return TKS_ORACLE_EINVAL;
    for (r = 0; r < batch; ++r) {
        int64_t L = row_len ? (int64_t)row_len[r] : row_stride;
        int rc;
        if (L < 0 || L > row_stride) return TKS_ORACLE_EINVAL;
        if (dtype == 0)
            rc = tks_oracle_topk_f32_order((const float *)values + r * row_stride, L, k, ordered,
                                           out + r * k);
        else
            rc = tks_oracle_topk_bf16_order((const uint16_t *)values + r * row_stride, L, k, ordered,
                                            out + r * k);
        if (rc != TKS_ORACLE_OK) return rc;
    }
    return TKS_ORACLE_OK;
}

int tks_oracle_topk_batch(const void *values, int32_t dtype, int64_t batch, int64_t row_stride,
                          const int32_t *row_len, int64_t k, int32_t *out)
{
    return tks_oracle_topk_batch_order(values, dtype, batch, row_stride, row_len, k, 0, out);
}

/* 0 when the build keeps subnormals distinct from zero and keeps -0.0 signed. */
int tks_oracle_selftest(void)
{
    volatile float d = FLT_TRUE_MIN;
    volatile float z = 0.0f;
    volatile float nz = -0.0f;
    if (!(d > z)) return 1;
    if (!(-d < nz)) return 2;
    if (!signbit(nz) || signbit(z)) return 3;
    return 0;
}

int tks_oracle_mutant(void) { return TKS_ORACLE_MUTANT; }
