/*
 * kvfix_oracle.c -- plain, slow CPU oracle for the reused-KV-chunk repair path.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load this library. The CUDA library never links, includes or
 * calls it, and it shares no source with the CUDA library.
 *
 * Every function is the plain definition written out: loops over the tensors in
 * index order, all arithmetic in double, library routines (pow, cos, sin, exp, log2,
 * fabs, sqrt, qsort, memcmp) as single steps.  bf16 inputs are decoded exactly; bf16 outputs are
 * rounded double -> float (round to nearest even, the C conversion) -> bf16 (round
 * to nearest even on the float bit pattern, from the IEEE-754 definition).
 *
 * Tensor layouts (all contiguous, bf16 stored as raw uint16 bit patterns):
 *   KV plane         [chunk][layer][token][head][dim]
 *   low-rank A       [chunk][layer][head][token][rank]
 *   low-rank B       [chunk][layer][head][rank][dim]
 *   draft queries    [chunk][layer][step][q_head][dim]
 *   anchor factors   A [segment][anchor][layer][token][r], Bt [segment][anchor][layer][feature][r]
 *   paged pool       [layer][slot][head][dim]
 *
 * Parity status per function (what pins it, other than itself, is listed in the
 * test files):
 *   bf16 rounding, rerope, scores, top-b, mean correction, low-rank apply, draft
 *   scores, top-k, diff encode/gather, diff restore, anchor gate / weights /
 *   correction, repair layouts, master selection, per-plane diffs: pinned.
 *   mean correction at the synthetic configs beyond the pinned invariants: the pages
 *   print no worked tensor, so those outputs rest on the definition alone.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define EXPORT __attribute__((visibility("default")))

/* ------------------------------------------------------------------ bf16 */

/* bf16 is the upper half of an IEEE-754 binary32 pattern: decoding is exact. */
static double bf16_decode(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a binary32 pattern to the nearest bf16, ties to even; NaN stays NaN. */
static uint16_t bf16_round_float(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

static uint16_t bf16_encode(double x)
{
    return bf16_round_float((float)x);
}

EXPORT void oracle_bf16_encode(const double* x, uint16_t* out, int64_t count)
{
    for (int64_t i = 0; i < count; ++i) out[i] = bf16_encode(x[i]);
}

EXPORT void oracle_bf16_decode(const uint16_t* x, double* out, int64_t count)
{
    for (int64_t i = 0; i < count; ++i) out[i] = bf16_decode(x[i]);
}

EXPORT int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

EXPORT void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------ RoPE */

/*
 * Rotary frequencies, rotate-half convention: theta_i = base^(-2i/D), i < D/2, and
 * dimension i is paired with dimension i + D/2.
 */
EXPORT void oracle_rope_theta(double base, int D, double* theta)
{
    for (int i = 0; i < D / 2; ++i) theta[i] = pow(base, -2.0 * (double)i / (double)D);
}

/*
 * Re-align one cached key row from its source position p to target p + delta:
 * with rotate-half RoPE, R(p + delta) = R(delta) R(p), so the re-alignment is one
 * more rotation by delta (KVCMAS, section 2.2: every compared method re-aligns the
 * cached keys to their target positions before reuse, and App. A.3: values are not
 * rotated; TokenDance section 4.4, Algorithm 1, the RoPERecover(P_old, P_new) step;
 * Budgeted Cache Repair, App. A: re-rotation is one scalar shift per segment).
 *   y_i       = x_i cos(delta theta_i) - x_{i+D/2} sin(delta theta_i)
 *   y_{i+D/2} = x_{i+D/2} cos(delta theta_i) + x_i sin(delta theta_i)
 */
static void rotate_row(const double* x, double* y, int D, double delta, const double* theta)
{
    int h = D / 2;
    if (delta == 0.0) { /* rotation by zero is the identity (also for signed zeros) */
        memcpy(y, x, sizeof(double) * (size_t)D);
        return;
    }
    for (int i = 0; i < h; ++i) {
        double a = delta * theta[i];
        double c = cos(a), s = sin(a);
        double x0 = x[i], x1 = x[i + h];
        y[i] = x0 * c - x1 * s;
        y[i + h] = x1 * c + x0 * s;
    }
}

/* Rotate rows given in double (no rounding); rows = count of D-vectors. */
EXPORT void oracle_rotate_f64(const double* x, double* y, int64_t rows, int D, double delta,
                              double base)
{
    double theta[1024];
    oracle_rope_theta(base, D, theta);
    for (int64_t r = 0; r < rows; ++r) rotate_row(x + r * D, y + r * D, D, delta, theta);
}

/*
 * kvfix_rerope: k_out[c] = bf16(rotate(k_in[c], delta[c])) for every layer, token and
 * head of chunk c.
 */
EXPORT void oracle_rerope(const uint16_t* k_in, uint16_t* k_out, int C, int L, int n, int H,
                          int D, const int32_t* delta, double base)
{
    double theta[1024];
    oracle_rope_theta(base, D, theta);
    int64_t rows_per_chunk = (int64_t)L * n * H;
#pragma omp parallel for schedule(static)
    for (int64_t cr = 0; cr < (int64_t)C * rows_per_chunk; ++cr) {
        int64_t c = cr / rows_per_chunk;
        double x[1024], y[1024];
        for (int e = 0; e < D; ++e) x[e] = bf16_decode(k_in[cr * D + e]);
        rotate_row(x, y, D, (double)delta[c], theta);
        for (int e = 0; e < D; ++e) k_out[cr * D + e] = bf16_encode(y[e]);
    }
}

/*
 * Synthetic-input composition used by the tests (not a step of the method):
 * fresh[a][r] = bf16(rotate(reuse[r], delta[a][r]) + mu[a][r][l][h][:] + xi[a][r][l][t][h][:])
 * with rotate the identity when rotate_keys == 0.  mu is [A*R][L][H][D] (one shared
 * offset vector per layer and head), xi is [A*R][L][n][H][D] (float32 draws).
 */
EXPORT void oracle_compose_fresh(const uint16_t* reuse, const float* mu, const float* xi,
                                 const int32_t* delta, int A, int R, int L, int n, int H, int D,
                                 double base, int rotate_keys, uint16_t* fresh)
{
    double theta[1024];
    oracle_rope_theta(base, D, theta);
    int64_t rows = (int64_t)L * n * H;
#pragma omp parallel for schedule(static)
    for (int64_t ar_row = 0; ar_row < (int64_t)A * R * rows; ++ar_row) {
        int64_t ar = ar_row / rows, row = ar_row % rows;
        int64_t r = ar % R;
        int64_t l = row / ((int64_t)n * H), h = row % H;
        double x[1024], y[1024];
        const uint16_t* src = reuse + (r * rows + row) * D;
        for (int e = 0; e < D; ++e) x[e] = bf16_decode(src[e]);
        if (rotate_keys) rotate_row(x, y, D, (double)delta[ar], theta);
        else memcpy(y, x, sizeof(double) * (size_t)D);
        const float* m = mu + ((ar * L + l) * H + h) * D;
        const float* z = xi + ar_row * D;
        for (int e = 0; e < D; ++e)
            fresh[ar_row * D + e] = bf16_encode(y[e] + (double)m[e] + (double)z[e]);
    }
}

/* ---------------------------------------------------- divergence scores */

/*
 * Check-layer divergence (AgentKVShift, "Core idea and method": the score of each
 * token and the displayed d_{K,j} = || K_fresh,j - K_reuse,j ||_2; TokenDance section 4.2: the rotated
 * keys are compared with the cached ones at one check layer):
 *   d[a][r][j] = sqrt( sum over heads h, dims e of (fresh[a][r][j][h][e] - rot(reuse[r][j][h])[e])^2 )
 * The norm runs over the whole token row (all KV heads), since probes are tokens.
 * reuse is [R][n][H][D] (one layer), fresh is [A*R][n][H][D].  rotate_keys selects
 * keys (rotated by delta[a*R+r]) or values (no rotation).
 */
EXPORT void oracle_scores(const uint16_t* reuse, const uint16_t* fresh, int A, int R, int n,
                          int H, int D, const int32_t* delta, double base, int rotate_keys,
                          double* d)
{
    double theta[1024];
    oracle_rope_theta(base, D, theta);
#pragma omp parallel for schedule(static)
    for (int64_t aj = 0; aj < (int64_t)A * R * n; ++aj) {
        int64_t ar = aj / n, j = aj % n;
        int64_t r = ar % R;
        double acc = 0.0;
        for (int h = 0; h < H; ++h) {
            double x[1024], y[1024];
            const uint16_t* src = reuse + ((r * n + j) * H + h) * D;
            const uint16_t* fr = fresh + ((ar * n + j) * H + h) * D;
            for (int e = 0; e < D; ++e) x[e] = bf16_decode(src[e]);
            if (rotate_keys) rotate_row(x, y, D, (double)delta[ar], theta);
            else memcpy(y, x, sizeof(double) * (size_t)D);
            for (int e = 0; e < D; ++e) {
                double diff = bf16_decode(fr[e]) - y[e];
                acc += diff * diff;
            }
        }
        d[aj] = sqrt(acc);
    }
}

/* ------------------------------------------------------------- top-b / top-k */

typedef struct {
    double key;
    int32_t idx;
} keyed;

static int by_key_desc_idx_asc(const void* pa, const void* pb)
{
    const keyed* a = (const keyed*)pa;
    const keyed* b = (const keyed*)pb;
    if (a->key > b->key) return -1;
    if (a->key < b->key) return 1;
    return (a->idx > b->idx) - (a->idx < b->idx);
}

static int int_asc(const void* pa, const void* pb)
{
    int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
    return (a > b) - (a < b);
}

/*
 * The b indices with the largest key, ties to the lower index, returned in
 * ascending index order (AgentKVShift, "Core idea and method": the b tokens with the largest score,
 * one set per score; Budgeted Cache Repair section 3: the best-scoring rows up to the
 * budget).  keys_as_float != 0 rounds each key to binary32 first, so that the
 * ranking decision is taken in the same precision as a float32 score.
 * Plain definition: sort all n (key, index) pairs and keep the first b.
 */
EXPORT void oracle_topk(const double* keys, int n, int b, int keys_as_float, int32_t* idx_out)
{
    keyed* v = (keyed*)malloc(sizeof(keyed) * (size_t)(n > 0 ? n : 1));
    for (int j = 0; j < n; ++j) {
        v[j].key = keys_as_float ? (double)(float)keys[j] : keys[j];
        v[j].idx = j;
    }
    qsort(v, (size_t)n, sizeof(keyed), by_key_desc_idx_asc);
    for (int i = 0; i < b; ++i) idx_out[i] = v[i].idx;
    qsort(idx_out, (size_t)b, sizeof(int32_t), int_asc);
    free(v);
}

/* ------------------------------------------------------- mean correction */

/*
 * Probe-mean correction of a reused chunk, every layer (AgentKVShift, "Core idea and
 * method", steps 3-4 and the displayed mu-hat and K_corr equations):
 *   mu[a][r][l][h][e] = (1/b) sum_{j in S} (fresh[a][r][l][j][h][e] - rot(reuse[r][l][j][h])[e])
 *   out[a][r][l][j]   = fresh[a][r][l][j]                         if j in S
 *                     = bf16(rot(reuse[r][l][j]) + w[a][r][j] mu)   otherwise
 * S = idx[a][r][0..b-1] (the same set in every layer), w[a][r][j] the clipped weight.
 * b == 0 gives mu = 0 and out = bf16(rot(reuse)).
 * reuse [R][L][n][H][D]; fresh, out [A*R][L][n][H][D]; mu [A*R][L][H][D] (double).
 */
EXPORT void oracle_mean_correct(const uint16_t* reuse, const uint16_t* fresh, int A, int R,
                                int L, int n, int H, int D, const int32_t* delta, double base,
                                int rotate_keys, const int32_t* idx, int b, const double* w,
                                uint16_t* out, double* mu)
{
    double theta[1024];
    oracle_rope_theta(base, D, theta);
#pragma omp parallel for schedule(dynamic)
    for (int64_t arl = 0; arl < (int64_t)A * R * L; ++arl) {
        int64_t ar = arl / L, l = arl % L;
        int64_t r = ar % R;
        const int32_t* S = idx + ar * b;
        const uint16_t* reuse_l = reuse + (r * L + l) * (int64_t)n * H * D;
        const uint16_t* fresh_l = fresh + (ar * L + l) * (int64_t)n * H * D;
        uint16_t* out_l = out + (ar * L + l) * (int64_t)n * H * D;
        double* m = mu + (ar * L + l) * (int64_t)H * D;
        double x[1024], y[1024];
        char* in_s = (char*)calloc((size_t)n, 1);
        for (int i = 0; i < b; ++i) in_s[S[i]] = 1;
        for (int64_t he = 0; he < (int64_t)H * D; ++he) m[he] = 0.0;
        for (int i = 0; i < b; ++i) {
            int64_t j = S[i];
            for (int h = 0; h < H; ++h) {
                const uint16_t* src = reuse_l + (j * H + h) * D;
                const uint16_t* fr = fresh_l + (j * H + h) * D;
                for (int e = 0; e < D; ++e) x[e] = bf16_decode(src[e]);
                if (rotate_keys) rotate_row(x, y, D, (double)delta[ar], theta);
                else memcpy(y, x, sizeof(double) * (size_t)D);
                for (int e = 0; e < D; ++e) m[h * D + e] += bf16_decode(fr[e]) - y[e];
            }
        }
        if (b > 0)
            for (int64_t he = 0; he < (int64_t)H * D; ++he) m[he] /= (double)b;
        for (int64_t j = 0; j < n; ++j) {
            for (int h = 0; h < H; ++h) {
                int64_t o = (j * H + h) * D;
                if (in_s[j]) {
                    memcpy(out_l + o, fresh_l + o, sizeof(uint16_t) * (size_t)D);
                    continue;
                }
                for (int e = 0; e < D; ++e) x[e] = bf16_decode(reuse_l[o + e]);
                if (rotate_keys) rotate_row(x, y, D, (double)delta[ar], theta);
                else memcpy(y, x, sizeof(double) * (size_t)D);
                double wj = w[ar * n + j];
                for (int e = 0; e < D; ++e) {
                    double v = (b > 0) ? y[e] + wj * m[h * D + e] : y[e];
                    out_l[o + e] = bf16_encode(v);
                }
            }
        }
        free(in_s);
    }
}

/*
 * The scalar form of the correction with given probe residuals and weights, for the
 * worked example (AgentKVShift, the single-coordinate numerical example and its table):
 *   mu = mean(probe_residuals); corrected[i] = reused[i] + weight[i] * mu.
 */
EXPORT double oracle_correct_with_weights(const double* probe_residuals, int b,
                                          const double* reused, const double* weight, int m,
                                          double* corrected)
{
    double mu = 0.0;
    for (int i = 0; i < b; ++i) mu += probe_residuals[i];
    mu = b > 0 ? mu / (double)b : 0.0;
    for (int i = 0; i < m; ++i) corrected[i] = reused[i] + weight[i] * mu;
    return mu;
}

/* --------------------------------------------------------- low-rank apply */

/*
 * Delta correction with a rank-r factorised delta (KVCMAS, Eq. 4 C_hat = C_ref +
 * Delta_hat; Eq. 7 Z ~ A_Z B_Z; Eq. 8 with one anchor of weight 1):
 *   out[c][l][j][h][e] = bf16( x[c][l][j][h][e] + sum_{k<r} A[c][l][h][j][k] B[c][l][h][k][e] )
 */
EXPORT void oracle_lowrank_apply(const uint16_t* x, const uint16_t* A, const uint16_t* B, int C,
                                 int L, int n, int H, int D, int r, uint16_t* out)
{
#pragma omp parallel for schedule(static)
    for (int64_t clj = 0; clj < (int64_t)C * L * n; ++clj) {
        int64_t cl = clj / n, j = clj % n;
        for (int h = 0; h < H; ++h) {
            const uint16_t* a = A + ((cl * H + h) * (int64_t)n + j) * r;
            const uint16_t* bm = B + (cl * H + h) * (int64_t)r * D;
            int64_t o = (clj * H + h) * D;
            for (int e = 0; e < D; ++e) {
                double acc = bf16_decode(x[o + e]);
                for (int k = 0; k < r; ++k) acc += bf16_decode(a[k]) * bf16_decode(bm[(int64_t)k * D + e]);
                out[o + e] = bf16_encode(acc);
            }
        }
    }
}

/* ------------------------------------------------------------ draft rank */

/*
 * Draft-attention row scores (Budgeted Cache Repair, section 3 "The repair": a_j is the
 * softmax(Q K~^T / sqrt(d_head)) mass the draft queries put on row j, over layers after
 * the first; App. B, Algorithm 2, grouped-query keys expanded to query heads):
 *   a[c][j] = sum_{l >= layer_begin} sum_{t < T} sum_{h < Hq}
 *               exp(z_j - max z) / sum_i exp(z_i - max z),
 *   z_i = q[c][l][t][h] . k[c][l][i][h / (Hq/Hkv)] / sqrt(D).
 * Summed rather than averaged over (t, h): the ranking is the same.
 */
EXPORT void oracle_draft_scores(const uint16_t* k, const uint16_t* q, int C, int L, int n,
                                int Hkv, int D, int T, int Hq, int layer_begin, double* scores)
{
    int group = Hq / Hkv;
    double inv_sqrt_d = 1.0 / sqrt((double)D);
    int nl = L - layer_begin;
    if (nl < 0) nl = 0;
    double* unit = (double*)calloc((size_t)C * (size_t)(nl > 0 ? nl : 1) * (size_t)n, sizeof(double));
#pragma omp parallel for schedule(dynamic)
    for (int64_t cl = 0; cl < (int64_t)C * nl; ++cl) {
        int64_t c = cl / nl, l = layer_begin + cl % nl;
        double* u = unit + cl * n;
        double* z = (double*)malloc(sizeof(double) * (size_t)n);
        double qv[1024];
        for (int t = 0; t < T; ++t) {
            for (int h = 0; h < Hq; ++h) {
                const uint16_t* qq = q + (((c * L + l) * T + t) * (int64_t)Hq + h) * D;
                for (int e = 0; e < D; ++e) qv[e] = bf16_decode(qq[e]);
                int kvh = h / group;
                double zmax = -INFINITY;
                for (int64_t i = 0; i < n; ++i) {
                    const uint16_t* kk = k + (((c * L + l) * (int64_t)n + i) * Hkv + kvh) * D;
                    double dot = 0.0;
                    for (int e = 0; e < D; ++e) dot += qv[e] * bf16_decode(kk[e]);
                    z[i] = dot * inv_sqrt_d;
                    if (z[i] > zmax) zmax = z[i];
                }
                double s = 0.0;
                for (int64_t i = 0; i < n; ++i) s += exp(z[i] - zmax);
                for (int64_t i = 0; i < n; ++i) u[i] += exp(z[i] - zmax) / s;
            }
        }
        free(z);
    }
    for (int64_t c = 0; c < C; ++c) {
        for (int64_t i = 0; i < n; ++i) {
            double a = 0.0;
            for (int64_t l = 0; l < nl; ++l) a += unit[(c * nl + l) * n + i];
            scores[c * n + i] = a;
        }
    }
    free(unit);
}

/*
 * Budgeted repair of the selected rows (Budgeted Cache Repair, App. B, Algorithm 1:
 * the selected rows' keys and values are overwritten with exact ones; KVCMAS
 * Eq. 3 selective recomputation): for every layer and head,
 *   kv[c][l][j] = fresh[c][l][j] for j in idx[c][0..k-1].
 */
EXPORT void oracle_row_overwrite(uint16_t* kv, const uint16_t* fresh, int C, int L, int n, int H,
                                 int D, const int32_t* idx, int k)
{
    int64_t row = (int64_t)H * D;
    for (int64_t c = 0; c < C; ++c)
        for (int64_t l = 0; l < L; ++l)
            for (int i = 0; i < k; ++i) {
                int64_t j = idx[c * k + i];
                int64_t o = ((c * L + l) * (int64_t)n + j) * row;
                memcpy(kv + o, fresh + o, sizeof(uint16_t) * (size_t)row);
            }
}

/* ------------------------------------------------------ diff encode / gather */

/*
 * Block-sparse sibling diff against one master (TokenDance section 4.3 master-mirror
 * layout and block-sparse K/V diff; section 5: a mirror keeps the indices of the blocks
 * it touches plus those blocks' K and V contents, with one index list shared by K and V
 * when both planes touch the same blocks):
 *   entry (s, l, blk) is dirty iff some bf16 word of K or V in tokens
 *   [bt*blk, bt*blk + bt) x all heads x all dims of layer l differs bitwise from master.
 *   mask bit i (i = (s*L + l)*nblk + blk; word i/32, bit i%32) = dirty.
 *   offsets[i] = number of dirty entries before i; offsets[S*L*nblk] = total.
 *   payload entry e = the sibling's K block then its V block (values, not deltas).
 * Returns the number of entries; writes the payload only if all of it fits the capacity.
 */
EXPORT int64_t oracle_diff_encode(const uint16_t* mk, const uint16_t* mv, const uint16_t* sk,
                                  const uint16_t* sv, int S, int L, int n, int H, int D, int bt,
                                  uint32_t* mask, int64_t* offsets, uint16_t* payload,
                                  int64_t capacity_entries)
{
    int nblk = n / bt;
    int64_t row = (int64_t)H * D;
    int64_t blk_elems = (int64_t)bt * row;
    int64_t plane = (int64_t)L * n * row;
    int64_t entries = (int64_t)S * L * nblk;
    char* dirty = (char*)calloc((size_t)(entries > 0 ? entries : 1), 1);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < entries; ++i) {
        int64_t s = i / ((int64_t)L * nblk), l = (i / nblk) % L, blk = i % nblk;
        int64_t mo = (l * n + blk * bt) * row;
        int64_t so = s * plane + mo;
        dirty[i] = memcmp(mk + mo, sk + so, sizeof(uint16_t) * (size_t)blk_elems) != 0 ||
                   memcmp(mv + mo, sv + so, sizeof(uint16_t) * (size_t)blk_elems) != 0;
    }
    memset(mask, 0, sizeof(uint32_t) * (size_t)((entries + 31) / 32));
    int64_t total = 0;
    for (int64_t i = 0; i < entries; ++i) {
        offsets[i] = total;
        if (dirty[i]) {
            mask[i / 32] |= 1u << (i % 32);
            ++total;
        }
    }
    offsets[entries] = total;
    if (total <= capacity_entries) {
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < entries; ++i) {
            if (!dirty[i]) continue;
            int64_t s = i / ((int64_t)L * nblk), l = (i / nblk) % L, blk = i % nblk;
            int64_t so = s * plane + (l * n + blk * bt) * row;
            uint16_t* e = payload + offsets[i] * 2 * blk_elems;
            memcpy(e, sk + so, sizeof(uint16_t) * (size_t)blk_elems);
            memcpy(e + blk_elems, sv + so, sizeof(uint16_t) * (size_t)blk_elems);
        }
    }
    free(dirty);
    return total;
}

/*
 * Mirror restore (TokenDance section 4.4, Algorithm 1: load the master block, then
 * overwrite it with the diff values at the diff's block indices): for every sibling,
 * layer and block, out = payload entry if the mask bit is set, else the master block.
 */
EXPORT void oracle_diff_gather(const uint16_t* mk, const uint16_t* mv, const uint32_t* mask,
                               const int64_t* offsets, const uint16_t* payload, int S, int L,
                               int n, int H, int D, int bt, uint16_t* ok, uint16_t* ov)
{
    int nblk = n / bt;
    int64_t row = (int64_t)H * D;
    int64_t blk_elems = (int64_t)bt * row;
    int64_t plane = (int64_t)L * n * row;
    int64_t entries = (int64_t)S * L * nblk;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < entries; ++i) {
        int64_t s = i / ((int64_t)L * nblk), l = (i / nblk) % L, blk = i % nblk;
        int64_t mo = (l * n + blk * bt) * row;
        int64_t so = s * plane + mo;
        if (mask[i / 32] >> (i % 32) & 1u) {
            const uint16_t* e = payload + offsets[i] * 2 * blk_elems;
            memcpy(ok + so, e, sizeof(uint16_t) * (size_t)blk_elems);
            memcpy(ov + so, e + blk_elems, sizeof(uint16_t) * (size_t)blk_elems);
        } else {
            memcpy(ok + so, mk + mo, sizeof(uint16_t) * (size_t)blk_elems);
            memcpy(ov + so, mv + mo, sizeof(uint16_t) * (size_t)blk_elems);
        }
    }
}

/*
 * Fused restore of mirrored caches into a paged KV pool (TokenDance, section 4.4,
 * Algorithm 1: per layer, the master block, overwritten where the mirror's block-sparse
 * diff touches it, keys re-aligned from the old to the new positions (RoPERecover), rows
 * written to the paged cache through the slot mapping).  Readings: re-aligning mirror s
 * is one rotation by delta[s] = P_new - P_old (one shift per mirror, as for a reused
 * chunk); values are not rotated; token t of mirror s goes to row slot_map[s][t] of the
 * pool in every layer, and a negative (or out-of-range) slot means the token is not
 * restored.  Pool planes are [L][slots][H][D]; rows not written keep their contents.
 */
EXPORT void oracle_diff_restore(const uint16_t* mk, const uint16_t* mv, const uint32_t* mask,
                                const int64_t* offsets, const uint16_t* payload, int S, int L,
                                int n, int H, int D, int bt, const int32_t* delta, double base,
                                const int32_t* slot_map, int64_t slots, uint16_t* pk, uint16_t* pv)
{
    double theta[1024];
    oracle_rope_theta(base, D, theta);
    int nblk = n / bt;
    int64_t row = (int64_t)H * D;
    int64_t blk_elems = (int64_t)bt * row;
#pragma omp parallel for schedule(static)
    for (int64_t st = 0; st < (int64_t)S * L * n; ++st) {
        int64_t s = st / ((int64_t)L * n), l = (st / n) % L, t = st % n;
        int32_t slot = slot_map[s * n + t];
        if (slot < 0 || slot >= slots) continue;
        int64_t i = (s * L + l) * nblk + t / bt;
        const uint16_t *kr, *vr;
        if (mask[i / 32] >> (i % 32) & 1u) {
            const uint16_t* e = payload + offsets[i] * 2 * blk_elems + (t % bt) * row;
            kr = e;
            vr = e + blk_elems;
        } else {
            kr = mk + (l * n + t) * row;
            vr = mv + (l * n + t) * row;
        }
        int64_t po = (l * slots + slot) * row;
        double x[1024], y[1024];
        for (int h = 0; h < H; ++h) {
            for (int e = 0; e < D; ++e) x[e] = bf16_decode(kr[h * D + e]);
            rotate_row(x, y, D, (double)delta[s], theta);
            for (int e = 0; e < D; ++e) pk[po + h * D + e] = bf16_encode(y[e]);
        }
        memcpy(pv + po, vr, sizeof(uint16_t) * (size_t)row);
    }
}

/* ------------------------------------------------------------ anchor-pool correction */

/*
 * One reconstructed row of an anchor's low-rank state (KVCMAS, section 3.3, Eq. 7: a
 * state Z of a segment is kept as factors A_Z [n x r] and B_Z [r x F]).  The second
 * factor is stored transposed, bt[f][c] = B_Z[c][f], so that each feature's r weights
 * are contiguous.  rec[f] = sum_c a[c] * bt[f][c].
 */
static void anchor_row(const uint16_t* a, const uint16_t* bt, int F, int r, double* rec)
{
    for (int f = 0; f < F; ++f) {
        double s = 0.0;
        for (int c = 0; c < r; ++c) s += bf16_decode(a[c]) * bf16_decode(bt[(int64_t)f * r + c]);
        rec[f] = s;
    }
}

/*
 * Reliability gate (KVCMAS, App. A.3 "Reliability Gate", Eq. 9-11): for each segment c,
 *   d_v = ( sum_l || V_src^(l)[:k] - V~^(v,l)[:k] ||_F^2 )^(1/2),
 *   g_v = exp(-d_v / T) / sum_u exp(-d_u / T),
 *   Hbar = -sum_v g_v log2 g_v / log2 V,  accepted iff V >= 2 and Hbar <= tau.
 * v_src [C][L][n][F] (the source value plane), ac [C][V][L][n][r], bct [C][V][L][F][r].
 * The softmax is evaluated with the smallest distance subtracted (the same ratios);
 * 0 log 0 = 0.  Writes d, g [C][V], hbar [C] (NaN when V < 2) and accept [C].
 */
EXPORT void oracle_anchor_gate(const uint16_t* v_src, const uint16_t* ac, const uint16_t* bct, int C,
                               int V, int L, int n, int F, int r, int k, double T, double tau,
                               double* d, double* g, double* hbar, int32_t* accept)
{
#pragma omp parallel for schedule(dynamic)
    for (int64_t cv = 0; cv < (int64_t)C * V; ++cv) {
        int64_t c = cv / V, v = cv % V;
        double* rec = (double*)malloc(sizeof(double) * (size_t)F);
        double s = 0.0;
        for (int l = 0; l < L; ++l)
            for (int t = 0; t < k; ++t) {
                const uint16_t* a = ac + (((c * V + v) * L + l) * (int64_t)n + t) * r;
                const uint16_t* bt = bct + ((c * V + v) * L + l) * (int64_t)F * r;
                const uint16_t* x = v_src + ((c * L + l) * (int64_t)n + t) * F;
                anchor_row(a, bt, F, r, rec);
                for (int f = 0; f < F; ++f) {
                    double e = bf16_decode(x[f]) - rec[f];
                    s += e * e;
                }
            }
        d[cv] = sqrt(s);
        free(rec);
    }
    for (int c = 0; c < C; ++c) {
        const double* dc = d + (int64_t)c * V;
        double* gc = g + (int64_t)c * V;
        double dmin = dc[0], z = 0.0, h = 0.0;
        for (int v = 1; v < V; ++v)
            if (dc[v] < dmin) dmin = dc[v];
        for (int v = 0; v < V; ++v) z += (gc[v] = exp(-(dc[v] - dmin) / T));
        for (int v = 0; v < V; ++v) {
            gc[v] /= z;
            if (gc[v] > 0.0) h -= gc[v] * log2(gc[v]);
        }
        hbar[c] = V >= 2 ? h / log2((double)V) : NAN;
        accept[c] = V >= 2 && hbar[c] <= tau;
    }
}

/*
 * Token-wise interpolation weights (KVCMAS, App. A.3 "Correction Weighting and Positional
 * Alignment"): for each segment c, layer l, token t of one plane (keys in their canonical
 * positions, as stored),
 *   m_v = (1/F) sum_f | x[f] - (A_C,v[t] B_C,v)[f] |,   w_v = exp(-m_v / T) / sum_u exp(-m_u / T).
 * x [C][L][n][F], ac [C][V][L][n][r], bct [C][V][L][F][r]; writes w [C][L][n][V].
 */
EXPORT void oracle_anchor_weights(const uint16_t* x, const uint16_t* ac, const uint16_t* bct, int C,
                                  int V, int L, int n, int F, int r, double T, double* w)
{
#pragma omp parallel for schedule(static)
    for (int64_t clt = 0; clt < (int64_t)C * L * n; ++clt) {
        int64_t c = clt / ((int64_t)L * n), l = (clt / n) % L, t = clt % n;
        double* rec = (double*)malloc(sizeof(double) * (size_t)F);
        double* m = w + clt * V;
        const uint16_t* xr = x + clt * F;
        double mmin = 0.0, z = 0.0;
        for (int v = 0; v < V; ++v) {
            anchor_row(ac + (((c * V + v) * L + l) * (int64_t)n + t) * r,
                       bct + ((c * V + v) * L + l) * (int64_t)F * r, F, r, rec);
            double s = 0.0;
            for (int f = 0; f < F; ++f) s += fabs(bf16_decode(xr[f]) - rec[f]);
            m[v] = s / F;
            if (v == 0 || m[v] < mmin) mmin = m[v];
        }
        for (int v = 0; v < V; ++v) z += (m[v] = exp(-(m[v] - mmin) / T));
        for (int v = 0; v < V; ++v) m[v] /= z;
        free(rec);
    }
}

/*
 * Anchor-weighted low-rank correction of the aligned source (KVCMAS Eq. 4 and Eq. 8 with
 * the token-wise weights of App. A.3; keys re-aligned to their target positions, values
 * not rotated):
 *   out[t] = bf16( Align(x[t]) + sum_v w[t][v] (A_D,v[t] B_D,v) ),
 * Align = rotate-half RoPE by delta[c] over each head (rotate != 0), else the identity.
 * x [C][L][n][H*D], ad [C][V][L][n][r], bdt [C][V][L][H*D][r], w [C][L][n][V].
 */
EXPORT void oracle_anchor_correct(const uint16_t* x, const uint16_t* ad, const uint16_t* bdt,
                                  const double* w, int C, int V, int L, int n, int H, int D, int r,
                                  const int32_t* delta, double base, int rotate, uint16_t* out)
{
    double theta[1024];
    oracle_rope_theta(base, D, theta);
    const int F = H * D;
#pragma omp parallel for schedule(static)
    for (int64_t clt = 0; clt < (int64_t)C * L * n; ++clt) {
        int64_t c = clt / ((int64_t)L * n), l = (clt / n) % L, t = clt % n;
        double* y = (double*)malloc(sizeof(double) * (size_t)F * 3);
        double* rec = y + F;
        double* xd = y + 2 * F;
        const uint16_t* xr = x + clt * F;
        for (int f = 0; f < F; ++f) xd[f] = bf16_decode(xr[f]);
        for (int h = 0; h < H; ++h) {
            if (rotate) rotate_row(xd + h * D, y + h * D, D, (double)delta[c], theta);
            else memcpy(y + h * D, xd + h * D, sizeof(double) * (size_t)D);
        }
        for (int v = 0; v < V; ++v) {
            double wv = w[clt * V + v];
            anchor_row(ad + (((c * V + v) * L + l) * (int64_t)n + t) * r,
                       bdt + ((c * V + v) * L + l) * (int64_t)F * r, F, r, rec);
            for (int f = 0; f < F; ++f) y[f] += wv * rec[f];
        }
        for (int f = 0; f < F; ++f) out[clt * F + f] = bf16_encode(y[f]);
        free(y);
    }
}

/* ------------------------------------------------------------ repair layouts */

/* p / q rounded to the nearest integer, halves to even (p, q >= 0, q > 0). */
static int64_t round_half_even(int64_t p, int64_t q)
{
    int64_t f = p / q, r = p - f * q;
    if (2 * r > q || (2 * r == q && (f & 1))) ++f;
    return f;
}

/*
 * Rows to repair from per-row draft scores, in the three layouts of Budgeted Cache
 * Repair (section 3 "The layouts"; App. A.2 "The policy" and Table 8; App. B,
 * Algorithms 1 and 2), for each unit u of scores [U][n]:
 *   layout 0 (single): the round(rho n) rows with the largest scores;
 *   layout 1 (chunk):  B-token chunks (the last one may be short), each scored by the mean
 *                      of its rows' scores; the max(1, round(rho n / B)) best chunks, all
 *                      their rows; with skip != 0, no rows when n < 2B or rho n < B;
 *   layout 2 (grow):   round(rho n) rows: the best unselected row seeds a span, which
 *                      takes the better of its two unselected neighbours while that one
 *                      scores at least tau times the seed, until neither qualifies or the
 *                      budget is spent; then the next seed.
 * Ties go to the lower index (rows, chunks, and left before right).  rho = num / den,
 * rounding halves to even.  Writes the rows ascending into idx [U][max_rows] (then -1)
 * and their number into counts [U]; returns the largest count.
 */
EXPORT int oracle_repair_layout(const double* scores, int U, int n, int layout, int B, int num, int den,
                                double tau, int skip, int32_t* idx, int max_rows, int32_t* counts)
{
    int most = 0;
    for (int u = 0; u < U; ++u) {
        const double* s = scores + (int64_t)u * n;
        unsigned char* sel = (unsigned char*)calloc((size_t)n + 1, 1);
        int chosen = 0;
        if (layout == 0 || layout == 2) {
            int k = (int)round_half_even((int64_t)num * n, den);
            if (k > n) k = n;
            keyed* order = (keyed*)malloc(sizeof(keyed) * (size_t)(n > 0 ? n : 1));
            for (int j = 0; j < n; ++j) order[j] = (keyed){s[j], j};
            qsort(order, (size_t)n, sizeof(keyed), by_key_desc_idx_asc);
            int p = 0;
            while (chosen < k) {
                while (sel[order[p].idx]) ++p;
                int seed = order[p].idx, lo = seed, hi = seed;
                sel[seed] = 1;
                ++chosen;
                if (layout == 0) continue;
                double thr = tau * s[seed];
                while (chosen < k) {
                    int l_ok = lo > 0 && !sel[lo - 1] && s[lo - 1] >= thr;
                    int r_ok = hi < n - 1 && !sel[hi + 1] && s[hi + 1] >= thr;
                    if (!l_ok && !r_ok) break;
                    if (l_ok && (!r_ok || s[lo - 1] >= s[hi + 1])) sel[--lo] = 1;
                    else sel[++hi] = 1;
                    ++chosen;
                }
            }
            free(order);
        } else {
            int nch = (n + B - 1) / B;
            int skipped = skip && (n < 2 * B || (int64_t)num * n < (int64_t)den * B);
            int c = (int)round_half_even((int64_t)num * n, (int64_t)den * B);
            if (c < 1) c = 1;
            if (c > nch) c = nch;
            if (!skipped && nch > 0) {
                keyed* order = (keyed*)malloc(sizeof(keyed) * (size_t)nch);
                for (int i = 0; i < nch; ++i) {
                    int a = i * B, b = a + B < n ? a + B : n;
                    double sum = 0.0;
                    for (int j = a; j < b; ++j) sum += s[j];
                    order[i] = (keyed){sum / (b - a), i};
                }
                qsort(order, (size_t)nch, sizeof(keyed), by_key_desc_idx_asc);
                for (int t = 0; t < c; ++t) {
                    int a = order[t].idx * B, b = a + B < n ? a + B : n;
                    for (int j = a; j < b; ++j) sel[j] = 1;
                    chosen += b - a;
                }
                free(order);
            }
        }
        int w = 0;
        for (int j = 0; j < n; ++j)
            if (sel[j] && w < max_rows) idx[(int64_t)u * max_rows + w++] = j;
        for (int t = w; t < max_rows; ++t) idx[(int64_t)u * max_rows + t] = -1;
        counts[u] = chosen;
        if (chosen > most) most = chosen;
        free(sel);
    }
    return most;
}

/* ------------------------------------------------------------ master selection, split diffs */

/*
 * Master of a round's cache family (TokenDance, section 4.2 "reuse plan output": the reuse
 * pass accumulates a deviation score per request, and the master is the request with the
 * lowest total deviation from the shared blocks): for agent a,
 *   total[a] = sum_{r < R} sum_{j < n} (d_k[a R + r][j] + d_v[a R + r][j]),
 * summed in that order in double; master = the agent with the smallest total (ties to the
 * lower index).  Either plane's scores may be NULL.
 */
EXPORT int oracle_master_select(const float* d_k, const float* d_v, int A, int R, int n, double* total)
{
    int best = 0;
    for (int a = 0; a < A; ++a) {
        double s = 0.0;
        for (int64_t r = 0; r < R; ++r)
            for (int64_t j = 0; j < n; ++j) {
                int64_t o = ((int64_t)a * R + r) * n + j;
                if (d_k) s += (double)d_k[o];
                if (d_v) s += (double)d_v[o];
            }
        total[a] = s;
        if (s < total[best]) best = a;
    }
    return best;
}

/*
 * Block-sparse diff with one index list per plane (TokenDance, section 5: the K and V
 * planes share one block list only when they touch the same blocks).  For plane P
 * (K = 0, V = 1), entry i = (s L + l) nblk + blk is dirty iff some bf16 word of plane P in
 * that block differs bitwise from the master's; offsets_P = exclusive counts (last =
 * total); payload_P [entries_P][bt][H][D] holds the sibling's plane-P block.  Returns the
 * totals in need[2]; payload entries beyond capacity[P] are not written.
 */
EXPORT void oracle_diff_encode_split(const uint16_t* mk, const uint16_t* mv, const uint16_t* sk,
                                     const uint16_t* sv, int S, int L, int n, int H, int D, int bt,
                                     uint32_t* mask_k, uint32_t* mask_v, int64_t* off_k,
                                     int64_t* off_v, uint16_t* pay_k, uint16_t* pay_v,
                                     const int64_t* capacity, int64_t* need)
{
    int nblk = n / bt;
    int64_t E = (int64_t)S * L * nblk;
    int64_t row = (int64_t)H * D, blk_elems = (int64_t)bt * row;
    for (int p = 0; p < 2; ++p) {
        const uint16_t* m = p ? mv : mk;
        const uint16_t* sb = p ? sv : sk;
        uint32_t* mask = p ? mask_v : mask_k;
        int64_t* off = p ? off_v : off_k;
        uint16_t* pay = p ? pay_v : pay_k;
        memset(mask, 0, sizeof(uint32_t) * (size_t)((E + 31) / 32));
        int64_t count = 0;
        for (int64_t i = 0; i < E; ++i) {
            int64_t s = i / ((int64_t)L * nblk), l = (i / nblk) % L, blk = i % nblk;
            const uint16_t* a = m + (l * n + blk * bt) * row;
            const uint16_t* b = sb + ((s * L + l) * n + blk * bt) * row;
            off[i] = count;
            if (memcmp(a, b, sizeof(uint16_t) * (size_t)blk_elems) != 0) {
                mask[i >> 5] |= 1u << (i & 31);
                if (count < capacity[p]) memcpy(pay + count * blk_elems, b, sizeof(uint16_t) * (size_t)blk_elems);
                ++count;
            }
        }
        off[E] = count;
        need[p] = count;
    }
}

/* Inverse of oracle_diff_encode_split: out_P[s] = the master's plane P, with each dirty
 * block replaced from payload_P. */
EXPORT void oracle_diff_gather_split(const uint16_t* mk, const uint16_t* mv, const uint32_t* mask_k,
                                     const uint32_t* mask_v, const int64_t* off_k,
                                     const int64_t* off_v, const uint16_t* pay_k,
                                     const uint16_t* pay_v, int S, int L, int n, int H, int D,
                                     int bt, uint16_t* ok, uint16_t* ov)
{
    int nblk = n / bt;
    int64_t E = (int64_t)S * L * nblk;
    int64_t row = (int64_t)H * D, blk_elems = (int64_t)bt * row;
    for (int p = 0; p < 2; ++p) {
        const uint16_t* m = p ? mv : mk;
        const uint32_t* mask = p ? mask_v : mask_k;
        const int64_t* off = p ? off_v : off_k;
        const uint16_t* pay = p ? pay_v : pay_k;
        uint16_t* out = p ? ov : ok;
        for (int64_t i = 0; i < E; ++i) {
            int64_t s = i / ((int64_t)L * nblk), l = (i / nblk) % L, blk = i % nblk;
            const uint16_t* src = (mask[i >> 5] >> (i & 31) & 1u) ? pay + off[i] * blk_elems
                                                                  : m + (l * n + blk * bt) * row;
            memcpy(out + ((s * L + l) * n + blk * bt) * row, src, sizeof(uint16_t) * (size_t)blk_elems);
        }
    }
}
