/*
 * rdot_oracle.c -- plain, slow, fp64 CPU oracle for ragged-dot / Group-GEMM.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load this library. The product path (the CUDA library) never calls it, includes it
 * or shares code with it.
 *
 * Every function below writes out a definition from the pages, with no blocking, fusion or
 * reordering of a reduction beyond what the definition states. All arithmetic is in double.
 *
 *   offsets      "Group-GEMM in XLA", Part 3 "Non-Contracting": exclusive prefix sum of
 *                group_sizes gives each group's start row, the inclusive one its end row.
 *   group_of_row same section (Table 2): a row belongs to the group whose [start, end)
 *                interval contains it.
 *   forward      Part 1 "The Ragged-Dot Operation" and Part 3 "Non-Contracting":
 *                out[i, :] = lhs[i, :] @ rhs[g(i)]; rows past sum(group_sizes) are zero
 *                (Part 2 "Autotuning" notes those rows are otherwise left unwritten; the AITER
 *                pull request #5831 item 1 zero-fills them).
 *   grad_weight  Part 3 "Contracting" and Part 4 Table 7 (wgrad_wi):
 *                dW[g] = lhs_g^T . dy_g, the contraction running over group g's rows only.
 *   grad_input   Part 4 Table 7 (dgrad_wi): dlhs[M,K] from dy[M,N] and rhs[E,K,N], contracting
 *                dy's dimension 1 with rhs's dimension 2 (the weight's output features):
 *                dlhs[i, :] = dy[i, :] @ rhs[g(i)]^T; rows past sum(group_sizes) are zero.
 *   mxfp8        AITER PR #5658: E4M3 operands with one E8M0 scale per 32 elements of K;
 *                the element value is decode(code) * 2^(scale - 127).
 *   tile_map     not on the pages: the enumeration order of the library's per-group tiles,
 *                written out by brute force so the device scheduler can be checked bit for bit.
 *
 * Readings where the pages are silent (stated again in the design notes):
 *   - a negative group size counts as 0, and each end offset is clamped to M; flag bit 1 is set
 *     when either happens;
 *   - rows at or past offsets[G] belong to no group and produce zero rows.
 *
 * dtype codes of this file (its own, unrelated to the CUDA library's):
 *   0 = f32, 1 = bf16 (raw 16-bit patterns), 3 = f64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_F32 0
#define ORC_BF16 1
#define ORC_F64 3

/* bf16 is the upper half of an IEEE binary32 pattern: widening is exact. */
static double orc_bf16_to_f64(uint16_t bits) {
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

static double orc_load(const void* base, int dtype, int64_t idx) {
    switch (dtype) {
        case ORC_F32: return (double)((const float*)base)[idx];
        case ORC_BF16: return orc_bf16_to_f64(((const uint16_t*)base)[idx]);
        case ORC_F64: return ((const double*)base)[idx];
        default: return NAN;
    }
}

/* OCP FP8 E4M3 ("e4m3fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits; no infinities;
 * exponent 1111 with mantissa 111 is NaN; exponent 0 encodes subnormals m/8 * 2^-6. */
double orc_e4m3_decode(uint8_t code) {
    int s = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* OCP E8M0 scale: an unsigned biased exponent (bias 127), 0xFF is NaN. */
double orc_e8m0_decode(uint8_t code) {
    if (code == 0xFF) return NAN;
    return ldexp(1.0, (int)code - 127);
}

/* offsets[0] = 0, offsets[g+1] = offsets[g] + group_sizes[g] (with the clamping reading).
 * Returns the flag word: bit 0 set when a size was negative or an offset was clamped to m. */
int orc_offsets(const int32_t* group_sizes, int g_count, int64_t m, int64_t* offsets) {
    int flags = 0;
    offsets[0] = 0;
    for (int g = 0; g < g_count; ++g) {
        int64_t s = group_sizes[g];
        if (s < 0) { s = 0; flags |= 1; }
        int64_t end = offsets[g] + s;
        if (end > m) { end = m; flags |= 1; }
        offsets[g + 1] = end;
    }
    return flags;
}

/* Group of a row: the unique g with offsets[g] <= row < offsets[g+1], or -1 for none. */
int orc_group_of_row(const int64_t* offsets, int g_count, int64_t row) {
    for (int g = 0; g < g_count; ++g)
        if (offsets[g] <= row && row < offsets[g + 1]) return g;
    return -1;
}

/* Forward (non-contracting ragged dimension) for a list of rows.
 * lhs [m, k], rhs [g, k, n], out [nrows, n] (row r of out is row rows[r] of the full output).
 * Each element is sum_{kk ascending} lhs[i, kk] * rhs[g(i), kk, j] in double. */
int orc_forward_rows(const void* lhs, int lhs_dtype, const void* rhs, int rhs_dtype,
                     const int32_t* group_sizes, int64_t m, int64_t k, int64_t n, int g_count,
                     const int64_t* rows, int64_t nrows, double* out) {
    int64_t* off = (int64_t*)malloc(sizeof(int64_t) * (size_t)(g_count + 1));
    if (!off) return -1;
    int flags = orc_offsets(group_sizes, g_count, m, off);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows[r];
        double* o = out + r * n;
        for (int64_t j = 0; j < n; ++j) o[j] = 0.0;
        int g = (i >= 0 && i < m) ? orc_group_of_row(off, g_count, i) : -1;
        if (g < 0) continue;
        for (int64_t kk = 0; kk < k; ++kk) {
            double a = orc_load(lhs, lhs_dtype, i * k + kk);
            int64_t b0 = ((int64_t)g * k + kk) * n;
            for (int64_t j = 0; j < n; ++j) o[j] += a * orc_load(rhs, rhs_dtype, b0 + j);
        }
    }
    free(off);
    return flags;
}

/* Weight gradient (contracting ragged dimension) for a list of (group, row-of-dW) pairs.
 * lhs [m, k], dy [m, n]; entry e of out [npairs, n] is dW[gsel[e], asel[e], :], where
 * dW[g, a, b] = sum_{i in [off[g], off[g+1]) ascending} lhs[i, a] * dy[i, b]. Empty group -> 0. */
int orc_grad_weight_rows(const void* lhs, int lhs_dtype, const void* dy, int dy_dtype,
                         const int32_t* group_sizes, int64_t m, int64_t k, int64_t n,
                         int g_count, const int32_t* gsel, const int64_t* asel, int64_t npairs,
                         double* out) {
    int64_t* off = (int64_t*)malloc(sizeof(int64_t) * (size_t)(g_count + 1));
    if (!off) return -1;
    int flags = orc_offsets(group_sizes, g_count, m, off);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t e = 0; e < npairs; ++e) {
        int g = gsel[e];
        int64_t a = asel[e];
        double* o = out + e * n;
        for (int64_t b = 0; b < n; ++b) o[b] = 0.0;
        if (g < 0 || g >= g_count || a < 0 || a >= k) continue;
        for (int64_t i = off[g]; i < off[g + 1]; ++i) {
            double x = orc_load(lhs, lhs_dtype, i * k + a);
            for (int64_t b = 0; b < n; ++b) o[b] += x * orc_load(dy, dy_dtype, i * n + b);
        }
    }
    free(off);
    return flags;
}

/* Data gradient (dgrad_wi: the weight's output-feature axis is contracted) for a list of rows.
 * dy [m, n], rhs [g, k, n], out [nrows, k] (row r of out is row rows[r] of the full dlhs).
 * Each element is sum_{j ascending} dy[i, j] * rhs[g(i), kk, j] in double. */
int orc_grad_input_rows(const void* dy, int dy_dtype, const void* rhs, int rhs_dtype,
                        const int32_t* group_sizes, int64_t m, int64_t k, int64_t n, int g_count,
                        const int64_t* rows, int64_t nrows, double* out) {
    int64_t* off = (int64_t*)malloc(sizeof(int64_t) * (size_t)(g_count + 1));
    if (!off) return -1;
    int flags = orc_offsets(group_sizes, g_count, m, off);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows[r];
        double* o = out + r * k;
        for (int64_t kk = 0; kk < k; ++kk) o[kk] = 0.0;
        int g = (i >= 0 && i < m) ? orc_group_of_row(off, g_count, i) : -1;
        if (g < 0) continue;
        for (int64_t kk = 0; kk < k; ++kk) {
            int64_t b0 = ((int64_t)g * k + kk) * n;
            double acc = 0.0;
            for (int64_t j = 0; j < n; ++j) acc += orc_load(dy, dy_dtype, i * n + j) * orc_load(rhs, rhs_dtype, b0 + j);
            o[kk] = acc;
        }
    }
    free(off);
    return flags;
}

/* MXFP8 forward for a list of rows. lhs_q [m, k] E4M3 codes, lhs_s [m, k/32] E8M0,
 * rhs_q [g, k, n] E4M3 codes, rhs_s [g, k/32, n] E8M0; both operands are dequantised
 * element by element (value = decode(code) * 2^(scale - 127)) and then the forward
 * definition applies. k must be a multiple of 32. */
int orc_forward_mxfp8_rows(const uint8_t* lhs_q, const uint8_t* lhs_s, const uint8_t* rhs_q,
                           const uint8_t* rhs_s, const int32_t* group_sizes, int64_t m,
                           int64_t k, int64_t n, int g_count, const int64_t* rows,
                           int64_t nrows, double* out) {
    if (k % 32) return -2;
    int64_t kb = k / 32;
    int64_t* off = (int64_t*)malloc(sizeof(int64_t) * (size_t)(g_count + 1));
    if (!off) return -1;
    int flags = orc_offsets(group_sizes, g_count, m, off);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows[r];
        double* o = out + r * n;
        for (int64_t j = 0; j < n; ++j) o[j] = 0.0;
        int g = (i >= 0 && i < m) ? orc_group_of_row(off, g_count, i) : -1;
        if (g < 0) continue;
        for (int64_t kk = 0; kk < k; ++kk) {
            double a = orc_e4m3_decode(lhs_q[i * k + kk]) * orc_e8m0_decode(lhs_s[i * kb + kk / 32]);
            const uint8_t* bq = rhs_q + ((int64_t)g * k + kk) * n;
            const uint8_t* bs = rhs_s + ((int64_t)g * kb + kk / 32) * n;
            for (int64_t j = 0; j < n; ++j)
                o[j] += a * (orc_e4m3_decode(bq[j]) * orc_e8m0_decode(bs[j]));
        }
    }
    free(off);
    return flags;
}

/* The library's tile map, enumerated by brute force.
 * Group g has ceil(m_g / bm) row tiles and ceil(n / bn) column tiles. Groups are visited in
 * index order; inside a group, m_inner = 1 visits row tiles fastest (column tile outer), and
 * m_inner = 0 visits column tiles fastest. tile_prefix[g] is the number of tiles before group g
 * in that plain order (tile_prefix[G] = total).
 * big_mt > 0 selects the interleaved order: the plain sequence is split into the tiles of groups
 * with at least big_mt row tiles ("big") and the rest ("small"), each keeping its order, and
 * the two are merged so that among the first w items exactly floor(w * nb / W) are big
 * (nb = number of big tiles, W = all tiles).
 * tiles [max_tiles, 3] receives (g, row tile, column tile) per work item. Returns the total
 * number of tiles (entries beyond max_tiles are not written). */
int64_t orc_tile_map(const int32_t* group_sizes, int g_count, int64_t m, int64_t n, int bm,
                     int bn, int m_inner, int big_mt, int32_t* tile_prefix, int32_t* tiles,
                     int64_t max_tiles) {
    int64_t* off = (int64_t*)malloc(sizeof(int64_t) * (size_t)(g_count + 1));
    if (!off) return -1;
    orc_offsets(group_sizes, g_count, m, off);
    int64_t nt = (n + bn - 1) / bn;
    int64_t total = 0;
    for (int g = 0; g < g_count; ++g) {
        tile_prefix[g] = (int32_t)total;
        total += ((off[g + 1] - off[g] + bm - 1) / bm) * nt;
    }
    tile_prefix[g_count] = (int32_t)total;
    /* the plain sequence, and for each entry whether its group is big */
    int32_t* seq = (int32_t*)malloc(sizeof(int32_t) * 3 * (size_t)(total > 0 ? total : 1));
    char* is_big = (char*)malloc((size_t)(total > 0 ? total : 1));
    if (!seq || !is_big) {
        free(off);
        free(seq);
        free(is_big);
        return -1;
    }
    int64_t w = 0, nb = 0;
    for (int g = 0; g < g_count; ++g) {
        int64_t mt = (off[g + 1] - off[g] + bm - 1) / bm;
        int big = big_mt > 0 && mt >= big_mt;
        for (int64_t outer = 0; outer < (m_inner ? nt : mt); ++outer)
            for (int64_t inner = 0; inner < (m_inner ? mt : nt); ++inner) {
                seq[3 * w + 0] = g;
                seq[3 * w + 1] = (int32_t)(m_inner ? inner : outer);
                seq[3 * w + 2] = (int32_t)(m_inner ? outer : inner);
                is_big[w] = (char)big;
                nb += big;
                ++w;
            }
    }
    /* merge: walk the big and the small entries of the plain sequence with two cursors */
    int64_t cb = 0, cs = 0, taken_big = 0;
    for (int64_t k = 0; k < total; ++k) {
        int pick_big = big_mt > 0 && (k + 1) * nb / total > taken_big;
        int64_t* cur = pick_big ? &cb : &cs;
        while (is_big[*cur] != (char)pick_big) ++*cur;
        if (k < max_tiles) {
            tiles[3 * k + 0] = seq[3 * *cur + 0];
            tiles[3 * k + 1] = seq[3 * *cur + 1];
            tiles[3 * k + 2] = seq[3 * *cur + 2];
        }
        ++*cur;
        taken_big += pick_big;
    }
    free(seq);
    free(is_big);
    free(off);
    return total;
}

int orc_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}
