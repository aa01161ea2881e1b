/*
 * oracle.c -- CPU oracle for DeepSelect row-wise top-k.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or load this
 * file: only the tests, the smoke check and the CPU-baseline leg of the benchmark use
 * it.  It shares no code, header, table or constant generator with the CUDA library.
 *
 * What it computes, and where that is defined:
 *   - Element order.  Values are compared through an order-preserving integer key:
 *     IEEE bits with the sign bit set are inverted, otherwise the sign bit is set
 *     (the "distort" mapping of the DeepSelect TopK tutorial, section 4.6).  This is a
 *     total order: -NaN < -inf < ... < -0 < +0 < ... < +inf < +NaN.
 *   - oracle_topk_sort: the plain definition of the row top-k.  Each row is sorted by
 *     (key descending, column ascending) and the first k entries are returned.  This is
 *     the stable-sort reference of the TileKernels two-backends tutorial (section on
 *     the stable_topk reference), which breaks ties toward the smaller index.
 *   - oracle_topk_sample: top-k sampling from the top k of oracle_topk_sort (the
 *     sampler's use of top-k, DeepSelect TopK tutorial, section 1.1), in double
 *     precision; see the function.
 *   - oracle_deepselect: the DeepSelectTopk pseudocode of DeepSelect-deep-dive.md
 *     ("Algorithm"), step by step: threshold T = -inf, blocks of size B visited in a
 *     random order that does not depend on x, every element with key > T appended to
 *     the candidate buffer, and after a whole block, if the buffer holds at least k+B2
 *     entries, RadixSelectTopK back to k entries with T set to the smallest kept key.
 *     A final RadixSelectTopK returns the answer.  RadixSelectTopK is written as its
 *     plain definition (the k largest keys; among equal keys the earlier buffer
 *     position wins), since any exact selection returns that set.
 *     It is instrumented with the quantities of the deep-dive's "Expected Upper Bound"
 *     section: A (appended elements), R (in-loop compactions), W (total input size of
 *     all compactions, the final one included), max |C|, and checks of the invariants
 *     stated in its "Notes" (|C| <= k+B2+B at all times, each element read exactly
 *     once) and in the proof (|C| < k+B2 at the start of every block, T never
 *     decreases, R*B2 <= A, W = A + k*R).
 *   - Block order.  The pages ask only for a uniform random permutation independent of
 *     x.  Reading used here: for block b of row r draw
 *         u_b = Philox4x32-10(key = (seed_lo, seed_hi), counter = (b, r_lo, r_hi, 0))[0]
 *     and visit the blocks sorted by (u_b ascending, b ascending).  Philox4x32-10 is
 *     written from its published definition (Salmon, Moraes, Dror, Shaw, "Parallel
 *     Random Numbers: As Easy as 1, 2, 3", SC'11): 10 rounds of the 4x32 S-box with
 *     multipliers 0xD2511F53 / 0xCD9E8D57 and Weyl key increments 0x9E3779B9 /
 *     0xBB67AE85.
 *   - oracle_work_bound: E[W] <= (1 + k/B2) (k+B+B2) H_m with m = ceil(N/B)
 *     (DeepSelect-deep-dive.md, boxed bound).
 *
 * Every result here is pinned by tests against things other than this file: brute
 * force on tiny inputs, the block-order experiment table and the complexity tables of
 * the DeepSelect TopK tutorial (sections 2.3 and 3.7), a closed form for block-ordered
 * inputs, the harmonic-number bound, and published Philox known-answer vectors.
 */
#include <stdint.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_BF16 = 0, OR_FP32 = 1 };

/* statistics written per row by oracle_deepselect */
enum {
    OR_STAT_A = 0,      /* elements appended to the candidate buffer             */
    OR_STAT_R = 1,      /* in-loop RadixSelectTopK calls                           */
    OR_STAT_W = 2,      /* sum of the input sizes of all RadixSelectTopK calls     */
    OR_STAT_MAXC = 3,   /* largest candidate-buffer size reached                   */
    OR_STAT_M = 4,      /* number of blocks, ceil(N/B)                             */
    OR_STAT_FLAGS = 5,  /* invariant violations, OR of OR_F_* bits                 */
    OR_STAT_TUPD = 6,   /* number of times T was set                               */
    OR_NSTAT = 8
};

enum {
    OR_F_CAP = 1,          /* |C| exceeded k+B2+B                                  */
    OR_F_BLOCKSTART = 2,   /* |C| >= k+B2 at the start of a block                  */
    OR_F_TDECR = 4,        /* T decreased                                          */
    OR_F_READS = 8,        /* some element was not read exactly once               */
    OR_F_RB2 = 16,         /* R*B2 > A                                             */
    OR_F_WSUM = 32,        /* W != A + k*R                                         */
    OR_F_FINAL_SHORT = 64  /* fewer than k candidates at the final compaction      */
};

/* ---------------------------------------------------------------- keys ---------- */

static uint32_t or_key32(uint32_t b) { return (b & 0x80000000u) ? ~b : (b | 0x80000000u); }

static uint32_t or_key16(uint32_t b)
{
    b &= 0xFFFFu;
    return (b & 0x8000u) ? ((~b) & 0xFFFFu) : (b | 0x8000u);
}

static uint32_t or_key_at(const void* x, int dtype, int64_t off)
{
    if (dtype == OR_BF16) return or_key16(((const uint16_t*)x)[off]);
    return or_key32(((const uint32_t*)x)[off]);
}

/* raw bits of element off, as stored */
static uint32_t or_bits_at(const void* x, int dtype, int64_t off)
{
    if (dtype == OR_BF16) return ((const uint16_t*)x)[off];
    return ((const uint32_t*)x)[off];
}

static void or_store_bits(void* out, int dtype, int64_t off, uint32_t bits)
{
    if (dtype == OR_BF16) ((uint16_t*)out)[off] = (uint16_t)bits;
    else ((uint32_t*)out)[off] = bits;
}

/* exported so tests can check the mapping itself */
uint32_t oracle_key(uint32_t bits, int dtype) { return dtype == OR_BF16 ? or_key16(bits) : or_key32(bits); }

/* ---------------------------------------------------------------- Philox ------- */

static void or_mulhilo32(uint32_t a, uint32_t b, uint32_t* hi, uint32_t* lo)
{
    uint64_t p = (uint64_t)a * (uint64_t)b;
    *hi = (uint32_t)(p >> 32);
    *lo = (uint32_t)p;
}

/* Philox4x32 with 10 rounds: out = f(counter, key). */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint32_t hi0, lo0, hi1, lo1;
        or_mulhilo32(0xD2511F53u, c0, &hi0, &lo0);
        or_mulhilo32(0xCD9E8D57u, c2, &hi1, &lo1);
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* the draw u_b that orders block b of row `row` */
uint32_t oracle_block_draw(uint64_t seed, int64_t row, int64_t b)
{
    uint32_t ctr[4] = {(uint32_t)b, (uint32_t)row, (uint32_t)((uint64_t)row >> 32), 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    return out[0];
}

typedef struct { uint32_t u; int64_t b; } or_draw;

static int or_cmp_draw(const void* pa, const void* pb)
{
    const or_draw* a = (const or_draw*)pa;
    const or_draw* b = (const or_draw*)pb;
    if (a->u != b->u) return a->u < b->u ? -1 : 1;
    if (a->b != b->b) return a->b < b->b ? -1 : 1;
    return 0;
}

/* perm[0..m) = the visiting order of the m blocks of row `row` */
int oracle_block_permutation(uint64_t seed, int64_t row, int64_t m, int64_t* perm)
{
    or_draw* d = (or_draw*)malloc((size_t)(m > 0 ? m : 1) * sizeof(or_draw));
    if (!d) return -1;
    for (int64_t b = 0; b < m; ++b) {
        d[b].u = oracle_block_draw(seed, row, b);
        d[b].b = b;
    }
    qsort(d, (size_t)m, sizeof(or_draw), or_cmp_draw);
    for (int64_t i = 0; i < m; ++i) perm[i] = d[i].b;
    free(d);
    return 0;
}

/* ------------------------------------------------------- full stable sort -------- */

typedef struct { uint32_t key; int64_t pos; } or_item;

/* key descending, then position ascending: a stable descending sort */
static int or_cmp_item(const void* pa, const void* pb)
{
    const or_item* a = (const or_item*)pa;
    const or_item* b = (const or_item*)pb;
    if (a->key != b->key) return a->key > b->key ? -1 : 1;
    if (a->pos != b->pos) return a->pos < b->pos ? -1 : 1;
    return 0;
}

static int or_topk_sort_row(const void* xrow, int dtype, int64_t N, int32_t k,
                            void* vals_row, int32_t* idx_row)
{
    or_item* it = (or_item*)malloc((size_t)N * sizeof(or_item));
    if (!it) return -1;
    for (int64_t j = 0; j < N; ++j) {
        it[j].key = or_key_at(xrow, dtype, j);
        it[j].pos = j;
    }
    qsort(it, (size_t)N, sizeof(or_item), or_cmp_item);
    for (int32_t i = 0; i < k; ++i) {
        or_store_bits(vals_row, dtype, i, or_bits_at(xrow, dtype, it[i].pos));
        idx_row[i] = (int32_t)it[i].pos;
    }
    free(it);
    return 0;
}

static int64_t or_esize(int dtype) { return dtype == OR_BF16 ? 2 : 4; }

int oracle_topk_sort(const void* x, int dtype, int64_t rows, int64_t N, int64_t stride,
                     int32_t k, void* out_vals, int32_t* out_idx, int32_t nthreads)
{
    if (!x || !out_vals || !out_idx || rows < 0 || N < 1 || k < 1 || k > N || stride < N) return -2;
    const int64_t es = or_esize(dtype);
    int err = 0;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : err)
#endif
    for (int64_t r = 0; r < rows; ++r) {
        const char* xrow = (const char*)x + r * stride * es;
        char* vrow = (char*)out_vals + r * (int64_t)k * es;
        if (or_topk_sort_row(xrow, dtype, N, k, vrow, out_idx + r * (int64_t)k)) err |= 1;
    }
    (void)nthreads;
    return err ? -1 : 0;
}

/* ------------------------------------------------------- transcription ----------- */

/* RadixSelectTopK(C, k) by its plain definition: keep the k entries with the largest
 * keys, earlier buffer positions first among equal keys, and leave the kept entries in
 * their buffer order.  Returns the smallest kept key. */
static uint32_t or_select_topk(uint32_t* ckey, int64_t* cidx, int64_t n, int32_t k, or_item* scratch,
                               unsigned char* keep)
{
    for (int64_t i = 0; i < n; ++i) {
        scratch[i].key = ckey[i];
        scratch[i].pos = i;
        keep[i] = 0;
    }
    qsort(scratch, (size_t)n, sizeof(or_item), or_cmp_item);
    for (int32_t i = 0; i < k; ++i) keep[scratch[i].pos] = 1;
    uint32_t kth = scratch[k - 1].key;
    int64_t w = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (keep[i]) {
            ckey[w] = ckey[i];
            cidx[w] = cidx[i];
            ++w;
        }
    }
    return kth;
}

static int or_deepselect_row(const void* xrow, int dtype, int64_t row, int64_t N, int32_t k,
                             int32_t B, int32_t B2, uint64_t seed, const int64_t* given_perm,
                             void* vals_row, int32_t* idx_row, int64_t* st)
{
    const int64_t m = (N + B - 1) / B;
    const int64_t cap = (int64_t)k + B2 + B;
    int64_t* perm = (int64_t*)malloc((size_t)m * sizeof(int64_t));
    uint32_t* ckey = (uint32_t*)malloc((size_t)cap * sizeof(uint32_t));
    int64_t* cidx = (int64_t*)malloc((size_t)cap * sizeof(int64_t));
    or_item* scratch = (or_item*)malloc((size_t)cap * sizeof(or_item));
    unsigned char* keep = (unsigned char*)malloc((size_t)cap);
    unsigned char* reads = (unsigned char*)calloc((size_t)N, 1);
    if (!perm || !ckey || !cidx || !scratch || !keep || !reads) {
        free(perm); free(ckey); free(cidx); free(scratch); free(keep); free(reads);
        return -1;
    }
    if (given_perm) memcpy(perm, given_perm, (size_t)m * sizeof(int64_t));
    else oracle_block_permutation(seed, row, m, perm);

    int64_t A = 0, R = 0, W = 0, maxC = 0, tupd = 0, flags = 0;
    int64_t n = 0;           /* |C| */
    int have_T = 0;          /* T = -inf until the first compaction */
    uint32_t T = 0;

    for (int64_t i = 0; i < m; ++i) {
        const int64_t b = perm[i];
        const int64_t lo = b * (int64_t)B;
        const int64_t hi = lo + B < N ? lo + B : N;
        if (n >= (int64_t)k + B2) flags |= OR_F_BLOCKSTART;
        for (int64_t j = lo; j < hi; ++j) {
            if (reads[j] < 255) reads[j]++;
            const uint32_t kj = or_key_at(xrow, dtype, j);
            if (!have_T || kj > T) {
                if (n >= cap) { flags |= OR_F_CAP; continue; }
                ckey[n] = kj;
                cidx[n] = j;
                ++n;
                ++A;
            }
        }
        if (n > maxC) maxC = n;
        if (n > cap) flags |= OR_F_CAP;
        if (n >= (int64_t)k + B2) {
            W += n;
            const uint32_t newT = or_select_topk(ckey, cidx, n, k, scratch, keep);
            n = k;
            if (have_T && newT < T) flags |= OR_F_TDECR;
            T = newT;
            have_T = 1;
            ++R;
            ++tupd;
        }
    }
    W += n;
    if (n < k) {
        flags |= OR_F_FINAL_SHORT;
    } else {
        or_select_topk(ckey, cidx, n, k, scratch, keep);
        n = k;
    }
    for (int64_t j = 0; j < N; ++j)
        if (reads[j] != 1) { flags |= OR_F_READS; break; }
    if (R * (int64_t)B2 > A) flags |= OR_F_RB2;
    if (W != A + (int64_t)k * R) flags |= OR_F_WSUM;

    for (int64_t i = 0; i < n && i < k; ++i) {
        or_store_bits(vals_row, dtype, i, or_bits_at(xrow, dtype, cidx[i]));
        idx_row[i] = (int32_t)cidx[i];
    }
    if (st) {
        st[OR_STAT_A] = A;
        st[OR_STAT_R] = R;
        st[OR_STAT_W] = W;
        st[OR_STAT_MAXC] = maxC;
        st[OR_STAT_M] = m;
        st[OR_STAT_FLAGS] = flags;
        st[OR_STAT_TUPD] = tupd;
        st[7] = 0;
    }
    free(perm); free(ckey); free(cidx); free(scratch); free(keep); free(reads);
    return 0;
}

/*
 * DeepSelectTopk for `rows` rows of `N` values (row r starts at x + r*stride elements).
 * out_vals / out_idx: rows*k, in the order the final buffer holds them.
 * perm: optional explicit block order shared by every row (m = ceil(N/B) entries);
 * NULL draws the Philox order described above for each row.
 * stats: optional rows*OR_NSTAT int64.
 */
int oracle_deepselect(const void* x, int dtype, int64_t rows, int64_t N, int64_t stride,
                      int32_t k, int32_t B, int32_t B2, uint64_t seed, const int64_t* perm,
                      void* out_vals, int32_t* out_idx, int64_t* stats, int32_t nthreads)
{
    if (!x || !out_vals || !out_idx || rows < 0 || N < 1 || k < 1 || k > N || B < 1 || B2 < 1 ||
        stride < N)
        return -2;
    const int64_t es = or_esize(dtype);
    int err = 0;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : err)
#endif
    for (int64_t r = 0; r < rows; ++r) {
        const char* xrow = (const char*)x + r * stride * es;
        char* vrow = (char*)out_vals + r * (int64_t)k * es;
        if (or_deepselect_row(xrow, dtype, r, N, k, B, B2, seed, perm, vrow, out_idx + r * (int64_t)k,
                              stats ? stats + r * OR_NSTAT : NULL))
            err |= 1;
    }
    (void)nthreads;
    return err ? -1 : 0;
}

/* ------------------------------------------------------- bound -------------------- */

/* (1 + k/B2) * (k + B + B2) * H_m, m = ceil(N/B) */
/* ------------------------------------------------------- top-k sampling ---------- */

/* oracle_topk_sample: the sampler's use of top-k (DeepSelect TopK tutorial, section 1.1:
 * at sampling time top-k picks candidate tokens out of the vocabulary's logits), read
 * plainly as top-k sampling.  For each row: its top k in the order of oracle_topk_sort
 * (key descending, column ascending), values v_0 >= v_1 >= ...; weights
 * w_i = exp((v_i - v_0) / temperature); running sums s_i = w_0 + ... + w_i in that order;
 * the row's token is the column of the first i with s_i > u * s_{k-1} (u = uniforms[row]
 * in [0, 1)), or of the last candidate if none.  prob[row] = w_i / s_{k-1}; cdf (rows x k,
 * may be NULL) receives s_i / s_{k-1}.  All in double precision. */
int oracle_topk_sample(const void* x, int dtype, int64_t rows, int64_t N, int64_t stride, int32_t k,
                       double temperature, const double* uniforms, int32_t* token, double* prob, double* cdf,
                       int32_t nthreads)
{
    if (!x || !uniforms || !token || !prob || rows < 0 || N < 1 || k < 1 || k > N || stride < N) return -2;
    if (!(temperature > 0.0)) return -2;
    const int64_t es = or_esize(dtype);
    int err = 0;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : err)
#endif
    for (int64_t r = 0; r < rows; ++r) {
        const char* xrow = (const char*)x + r * stride * es;
        uint32_t* vb = (uint32_t*)malloc((size_t)k * sizeof(uint32_t));
        int32_t* ix = (int32_t*)malloc((size_t)k * sizeof(int32_t));
        double* s = (double*)malloc((size_t)k * sizeof(double));
        if (!vb || !ix || !s) {
            err |= 1;
        } else {
            /* the sorted top k, as 32-bit patterns of the values */
            uint16_t* v16 = (uint16_t*)vb;
            if (or_topk_sort_row(xrow, dtype, N, k, dtype == OR_BF16 ? (void*)v16 : (void*)vb, ix)) err |= 1;
            double v0 = 0.0;
            for (int32_t i = 0; i < k; ++i) {
                const uint32_t b = dtype == OR_BF16 ? ((uint32_t)v16[i] << 16) : vb[i];
                float f;
                memcpy(&f, &b, sizeof f);
                if (i == 0) v0 = (double)f;
                const double w = exp(((double)f - v0) / temperature);
                s[i] = (i ? s[i - 1] : 0.0) + w;
            }
            const double total = s[k - 1];
            const double target = uniforms[r] * total;
            int32_t pick = k - 1;
            for (int32_t i = 0; i < k; ++i) {
                if (s[i] > target) {
                    pick = i;
                    break;
                }
            }
            token[r] = ix[pick];
            prob[r] = (s[pick] - (pick ? s[pick - 1] : 0.0)) / total;
            if (cdf)
                for (int32_t i = 0; i < k; ++i) cdf[r * (int64_t)k + i] = s[i] / total;
        }
        free(vb);
        free(ix);
        free(s);
    }
    (void)nthreads;
    return err ? -1 : 0;
}

double oracle_work_bound(int64_t N, int32_t k, int32_t B, int32_t B2)
{
    const int64_t m = (N + B - 1) / B;
    double H = 0.0;
    for (int64_t i = m; i >= 1; --i) H += 1.0 / (double)i;
    return (1.0 + (double)k / (double)B2) * ((double)k + (double)B + (double)B2) * H;
}

int oracle_num_threads_max(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
