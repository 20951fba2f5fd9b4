/*
 * moe_oracle.c -- plain, slow, scalar CPU oracle for MoE layout, dispatch
 * and combine on logical ranks.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this file's library. The product
 * path (the CUDA library and its Python binding) never calls it, and the two
 * share no code, header, table or helper.
 *
 * Every function is the written-out definition of one step, in the order the
 * DeepEP V2 deep-dive page ("DeepEP V2 深度深潜") gives it:
 *   - routing: rank = expert / experts_per_rank, -1 = masked choice
 *     (section 2.2, the top-k load of the dispatch kernel);
 *   - counting: one count per expert per valid choice, one count per rank
 *     per token after de-duplication (section 3.3, notify warps), followed by
 *     exclusive prefix sums (section 3.5, "prefix sum -> psum_num_recv_tokens");
 *   - dispatch: one copy of the token row per distinct destination rank
 *     (section 1.3 factor 2: read once, written once per rank; section 3.3
 *     stage 2), with the receive regions of the ranks laid out one after the
 *     other (section 3.3 stage 3, the prefix walk of the copy epilogue);
 *   - combine: the per-rank partial rows of a token summed back into one row.
 * Readings where the page is silent (slot order, first-lane ownership, fp8
 * recipe, combine order) are listed in the design notes; the code below
 * states each one where it is used.
 *
 * Compiled with plain IEEE arithmetic: no -ffast-math, no FMA contraction.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Result flags (bit set; 0 = clean). */
#define ORACLE_BAD_TOPK   1  /* an entry outside [-1, E); treated as masked */
#define ORACLE_CAPACITY   2  /* a destination row beyond the receive capacity; not written */
#define ORACLE_BAD_ARG    4  /* shape arguments violate the contract */

/* ------------------------------------------------------------------ */
/* Number formats, written from their definitions.                     */
/* ------------------------------------------------------------------ */

static uint32_t float_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_float(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* bfloat16 is the upper half of an IEEE binary32. Widening is exact. */
float oracle_bf16_to_float(uint16_t h) { return bits_float(((uint32_t)h) << 16); }

/* binary32 -> bfloat16, round to nearest, ties to even (IEEE 754 default
 * rounding), keeping the 16 high bits. Overflow carries into the exponent
 * and yields infinity, as the definition implies. NaN stays a quiet NaN. */
uint16_t oracle_bf16_from_float(float f)
{
    uint32_t u = float_bits(f);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);        /* quiet NaN */
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xFFFFu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

/* Round a non-negative double to the nearest integer, ties to even. The
 * argument is always an exact scaled copy of a float, so this is exact. */
static double rne_nonneg(double v)
{
    double fl = floor(v);
    double frac = v - fl;
    if (frac > 0.5) return fl + 1.0;
    if (frac < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* binary32 -> OCP OFP8 E4M3 (sign, 4 exponent bits with bias 7, 3 mantissa
 * bits; no infinities; S.1111.111 is NaN; largest finite 448; subnormal step
 * 2^-9). Round to nearest even, saturating finite values above 448 to +-448.
 * The finite E4M3 magnitudes in code order are consecutive multiples of a
 * quantum that is 2^-9 below 2^-6 and 2^(e-3) within binade [2^e, 2^(e+1)),
 * so the code is the count of quanta below the rounded value. */
uint8_t oracle_e4m3_from_float(float f)
{
    uint32_t u = float_bits(f);
    uint8_t sign = (uint8_t)((u >> 24) & 0x80u);
    if (isnan(f)) return (uint8_t)(sign | 0x7F);
    double a = fabs((double)f);
    if (a > 448.0) return (uint8_t)(sign | 0x7E);          /* satfinite */
    int code;
    if (a < ldexp(1.0, -6)) {
        code = (int)rne_nonneg(a * ldexp(1.0, 9));           /* subnormals, 0..8 */
    } else {
        int ex;
        (void)frexp(a, &ex);                                  /* a = m * 2^ex, m in [0.5,1) */
        int e = ex - 1;                                       /* a in [2^e, 2^(e+1)) */
        int n = (int)rne_nonneg(a * ldexp(1.0, 3 - e));      /* 8..16 quanta of 2^(e-3) */
        code = (e + 6) * 8 + n;
    }
    if (code > 0x7E) code = 0x7E;
    return (uint8_t)(sign | code);
}

/* E4M3 -> value, straight from the format definition. */
float oracle_e4m3_to_float(uint8_t c)
{
    int s = c >> 7, E = (c >> 3) & 0xF, M = c & 7;
    if (E == 15 && M == 7) return NAN;
    double v = (E == 0) ? ldexp((double)M / 8.0, -6) : ldexp(1.0 + (double)M / 8.0, E - 7);
    return (float)(s ? -v : v);
}

/* ------------------------------------------------------------------ */
/* Layout: counts, in-rank positions, global receive rows.             */
/* ------------------------------------------------------------------ */

/* For token t and choice j: the destination rank, or -1 when the choice is
 * masked (-1) or invalid (outside [0, E), also flagged). */
static int rank_of(const int64_t *topk_idx, int k, int t, int j, int E, int m, int *flags)
{
    int64_t e = topk_idx[(int64_t)t * k + j];
    if (e == -1) return -1;
    if (e < 0 || e >= E) { *flags |= ORACLE_BAD_TOPK; return -1; }
    return (int)(e / m);
}

/* Is choice j the lowest-indexed valid choice of token t that lands on its
 * rank? (Reading: when several experts of one token live on the same rank,
 * the lowest lane owns the rank's receive slot.) */
static int is_first_lane(const int64_t *topk_idx, int k, int t, int j, int E, int m)
{
    int dummy = 0;
    int r = rank_of(topk_idx, k, t, j, E, m, &dummy);
    if (r < 0) return 0;
    for (int jj = 0; jj < j; ++jj)
        if (rank_of(topk_idx, k, t, jj, E, m, &dummy) == r) return 0;
    return 1;
}

int oracle_layout(const int64_t *topk_idx, int T, int k, int E, int R,
                  int32_t *num_tokens_per_rank,     /* [R]   */
                  int32_t *num_tokens_per_expert,   /* [E]   */
                  uint8_t *is_token_in_rank,        /* [T,R] */
                  int32_t *rank_prefix,             /* [R+1] */
                  int32_t *expert_prefix,           /* [E+1] */
                  int32_t *token_dst_row)           /* [T,k] */
{
    if (T < 0 || k < 1 || k > 32 || E < 1 || R < 1 || E % R != 0) return ORACLE_BAD_ARG;
    int flags = 0;
    int m = E / R;

    for (int r = 0; r < R; ++r) num_tokens_per_rank[r] = 0;
    for (int e = 0; e < E; ++e) num_tokens_per_expert[e] = 0;
    memset(is_token_in_rank, 0, (size_t)T * (size_t)R);

    /* Step 1: per-choice expert counts; per-token rank membership. */
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int r = rank_of(topk_idx, k, t, j, E, m, &flags);
            if (r < 0) continue;
            num_tokens_per_expert[topk_idx[(int64_t)t * k + j]] += 1;
            is_token_in_rank[(int64_t)t * R + r] = 1;
        }
    }
    /* Step 2: per-rank token counts (each token once per rank), exclusive prefixes. */
    for (int t = 0; t < T; ++t)
        for (int r = 0; r < R; ++r)
            num_tokens_per_rank[r] += is_token_in_rank[(int64_t)t * R + r];
    rank_prefix[0] = 0;
    for (int r = 0; r < R; ++r) rank_prefix[r + 1] = rank_prefix[r] + num_tokens_per_rank[r];
    expert_prefix[0] = 0;
    for (int e = 0; e < E; ++e) expert_prefix[e + 1] = expert_prefix[e] + num_tokens_per_expert[e];

    /* Step 3: rows of a rank are ordered by source token; the global row is
     * the rank's region start plus the token's position inside the region. */
    int32_t *next = (int32_t *)calloc((size_t)R, sizeof(int32_t));
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int64_t idx = (int64_t)t * k + j;
            token_dst_row[idx] = -1;
            if (!is_first_lane(topk_idx, k, t, j, E, m)) continue;
            int r = (int)(topk_idx[idx] / m);
            token_dst_row[idx] = rank_prefix[r] + next[r];
            next[r] += 1;
        }
    }
    free(next);
    return flags;
}

/* ------------------------------------------------------------------ */
/* Dispatch: one copy of the token per distinct destination rank.       */
/* ------------------------------------------------------------------ */

/* Metadata of receive row `row` holding token t on rank r: its source token,
 * its top-k choices localised to rank r (expert - r*m where the expert lives
 * on r, else -1) and the matching weights (0 where not local). */
static void write_metadata(const int64_t *topk_idx, const float *topk_weights, int k, int E, int m,
                           int t, int r, int64_t row,
                           int64_t *recv_topk_idx, float *recv_topk_weights, int32_t *recv_src_idx)
{
    recv_src_idx[row] = t;
    for (int j = 0; j < k; ++j) {
        int64_t e = topk_idx[(int64_t)t * k + j];
        int local = (e >= 0 && e < E && (int)(e / m) == r);
        recv_topk_idx[row * k + j] = local ? e - (int64_t)r * m : -1;
        if (recv_topk_weights)
            recv_topk_weights[row * k + j] = (local && topk_weights) ? topk_weights[(int64_t)t * k + j] : 0.0f;
    }
}

/* The bf16 dispatch of tokens t0 <= t < t1 (every token's rows and metadata
 * depend on that token alone). */
static int dispatch_bf16_tokens(const uint16_t *x, int H,
                                const int64_t *topk_idx, const float *topk_weights, int k, int E, int R,
                                const int32_t *token_dst_row, int recv_capacity,
                                uint16_t *recv_x, int64_t *recv_topk_idx, float *recv_topk_weights,
                                int32_t *recv_src_idx, int t0, int t1)
{
    int flags = 0, m = E / R;
    for (int t = t0; t < t1; ++t) {
        for (int j = 0; j < k; ++j) {
            int64_t row = token_dst_row[(int64_t)t * k + j];
            if (row < 0) continue;
            if (row >= recv_capacity) { flags |= ORACLE_CAPACITY; continue; }
            int r = (int)(topk_idx[(int64_t)t * k + j] / m);
            for (int h = 0; h < H; ++h) recv_x[row * H + h] = x[(int64_t)t * H + h];
            write_metadata(topk_idx, topk_weights, k, E, m, t, r, row,
                           recv_topk_idx, recv_topk_weights, recv_src_idx);
        }
    }
    return flags;
}

int oracle_dispatch_bf16(const uint16_t *x, int T, int H,
                         const int64_t *topk_idx, const float *topk_weights, int k, int E, int R,
                         const int32_t *token_dst_row, int recv_capacity,
                         uint16_t *recv_x, int64_t *recv_topk_idx, float *recv_topk_weights,
                         int32_t *recv_src_idx)
{
    if (T < 0 || H < 1 || k < 1 || k > 32 || E % R != 0) return ORACLE_BAD_ARG;
    return dispatch_bf16_tokens(x, H, topk_idx, topk_weights, k, E, R, token_dst_row, recv_capacity,
                                recv_x, recv_topk_idx, recv_topk_weights, recv_src_idx, 0, T);
}

/* Per-128-channel block quantisation of one token row: amax = max |x| over
 * the block, scale = amax / 448 (fp32, round to nearest), code = E4M3 of
 * x / scale (fp32 division, then round-to-nearest-even with saturation).
 * A block of zeros has scale 0 and all codes 0. */
static void quantize_row(const uint16_t *xrow, int H, uint8_t *q, float *scales)
{
    for (int b = 0; b < H / 128; ++b) {
        float amax = 0.0f;
        for (int i = 0; i < 128; ++i) {
            float v = fabsf(oracle_bf16_to_float(xrow[b * 128 + i]));
            if (v > amax) amax = v;
        }
        float s = amax / 448.0f;
        scales[b] = s;
        for (int i = 0; i < 128; ++i) {
            float v = oracle_bf16_to_float(xrow[b * 128 + i]);
            q[b * 128 + i] = (s == 0.0f) ? 0 : oracle_e4m3_from_float(v / s);
        }
    }
}

int oracle_dispatch_fp8(const uint16_t *x, int T, int H,
                        const int64_t *topk_idx, const float *topk_weights, int k, int E, int R,
                        const int32_t *token_dst_row, int recv_capacity,
                        uint8_t *recv_x, float *recv_x_scales, int64_t *recv_topk_idx,
                        float *recv_topk_weights, int32_t *recv_src_idx, float *x_scales_out)
{
    if (T < 0 || H < 128 || H % 128 != 0 || k < 1 || k > 32 || E % R != 0) return ORACLE_BAD_ARG;
    int flags = 0, m = E / R, nb = H / 128;
    uint8_t *q = (uint8_t *)malloc((size_t)H);
    float *s = (float *)malloc(sizeof(float) * (size_t)nb);
    for (int t = 0; t < T; ++t) {
        quantize_row(x + (int64_t)t * H, H, q, s);
        if (x_scales_out)
            for (int b = 0; b < nb; ++b) x_scales_out[(int64_t)t * nb + b] = s[b];
        for (int j = 0; j < k; ++j) {
            int64_t row = token_dst_row[(int64_t)t * k + j];
            if (row < 0) continue;
            if (row >= recv_capacity) { flags |= ORACLE_CAPACITY; continue; }
            int r = (int)(topk_idx[(int64_t)t * k + j] / m);
            for (int h = 0; h < H; ++h) recv_x[row * H + h] = q[h];
            for (int b = 0; b < nb; ++b) recv_x_scales[row * nb + b] = s[b];
            write_metadata(topk_idx, topk_weights, k, E, m, t, r, row,
                           recv_topk_idx, recv_topk_weights, recv_src_idx);
        }
    }
    free(q);
    free(s);
    return flags;
}

/* Dispatch of rows that are already E4M3 codes with their per-128 scales
 * (the scales travel next to the hidden bytes): codes and scales are copied
 * unchanged, once per distinct destination rank. */
int oracle_dispatch_fp8_input(const uint8_t *x, const float *x_scales, int T, int H,
                              const int64_t *topk_idx, const float *topk_weights, int k, int E, int R,
                              const int32_t *token_dst_row, int recv_capacity,
                              uint8_t *recv_x, float *recv_x_scales, int64_t *recv_topk_idx,
                              float *recv_topk_weights, int32_t *recv_src_idx)
{
    if (T < 0 || H < 128 || H % 128 != 0 || k < 1 || k > 32 || E % R != 0) return ORACLE_BAD_ARG;
    int flags = 0, m = E / R, nb = H / 128;
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int64_t row = token_dst_row[(int64_t)t * k + j];
            if (row < 0) continue;
            if (row >= recv_capacity) { flags |= ORACLE_CAPACITY; continue; }
            int r = (int)(topk_idx[(int64_t)t * k + j] / m);
            for (int h = 0; h < H; ++h) recv_x[row * H + h] = x[(int64_t)t * H + h];
            for (int b = 0; b < nb; ++b) recv_x_scales[row * nb + b] = x_scales[(int64_t)t * nb + b];
            write_metadata(topk_idx, topk_weights, k, E, m, t, r, row,
                           recv_topk_idx, recv_topk_weights, recv_src_idx);
        }
    }
    return flags;
}

/* ------------------------------------------------------------------ */
/* Combine: partial rows back into token order, fp32 sum, bf16 out.     */
/* ------------------------------------------------------------------ */

/* out[t] = bf16( sum over the receive rows of token t, taken in ascending
 * rank order, of float(partial[row]) ), accumulator starting at +0.0f.
 * Rank regions are laid out in ascending rank order, so ascending rank is
 * ascending row. A token with no rows gets +0. */
static int combine_tokens(const uint16_t *partial, int num_rows, int H, int k,
                          const int32_t *token_dst_row, uint16_t *out, int t0, int t1)
{
    int flags = 0;
    int32_t rows[32];
    for (int t = t0; t < t1; ++t) {
        int n = 0;
        for (int j = 0; j < k; ++j) {
            int32_t row = token_dst_row[(int64_t)t * k + j];
            if (row < 0) continue;
            if (row >= num_rows) { flags |= ORACLE_CAPACITY; continue; }
            rows[n++] = row;
        }
        for (int a = 1; a < n; ++a)                          /* insertion sort, ascending */
            for (int b = a; b > 0 && rows[b - 1] > rows[b]; --b) {
                int32_t tmp = rows[b]; rows[b] = rows[b - 1]; rows[b - 1] = tmp;
            }
        for (int h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int i = 0; i < n; ++i)
                acc += oracle_bf16_to_float(partial[(int64_t)rows[i] * H + h]);
            out[(int64_t)t * H + h] = oracle_bf16_from_float(acc);
        }
    }
    return flags;
}

int oracle_combine(const uint16_t *partial, int num_rows, int T, int H, int k,
                   const int32_t *token_dst_row, uint16_t *out)
{
    if (T < 0 || H < 1 || k < 1 || k > 32) return ORACLE_BAD_ARG;
    return combine_tokens(partial, num_rows, H, k, token_dst_row, out, 0, T);
}

/* ------------------------------------------------------------------ */
/* Thread-parallel forms, for timing the oracle on every host core.     */
/* ------------------------------------------------------------------ */

/* The dispatch and the combine above, run by `threads` POSIX threads over
 * contiguous token ranges: thread i takes tokens [T*i/n, T*(i+1)/n). Every
 * token's outputs are computed by exactly the code above, from that token's
 * inputs alone, into rows no other token writes, so the results are the
 * single-threaded ones byte for byte (the tests check this); only the wall
 * time changes. The result flags are OR-ed over the threads. */
typedef struct {
    int kind;                                   /* 0: bf16 dispatch, 1: combine */
    const uint16_t *src;                        /* x or partial */
    int num_rows, H, k, E, R, recv_capacity;
    const int64_t *topk_idx;
    const float *topk_weights;
    const int32_t *token_dst_row;
    uint16_t *dst;                              /* recv_x or out */
    int64_t *recv_topk_idx;
    float *recv_topk_weights;
    int32_t *recv_src_idx;
    int t0, t1, flags;
} token_job;

static void *run_token_job(void *arg)
{
    token_job *j = (token_job *)arg;
    if (j->kind == 0)
        j->flags = dispatch_bf16_tokens(j->src, j->H, j->topk_idx, j->topk_weights, j->k, j->E, j->R,
                                        j->token_dst_row, j->recv_capacity, j->dst, j->recv_topk_idx,
                                        j->recv_topk_weights, j->recv_src_idx, j->t0, j->t1);
    else
        j->flags = combine_tokens(j->src, j->num_rows, j->H, j->k, j->token_dst_row, j->dst, j->t0, j->t1);
    return NULL;
}

static int run_token_jobs(const token_job *proto, int T, int threads)
{
    if (threads < 1) threads = 1;
    if (threads > 1024) threads = 1024;
    token_job *jobs = (token_job *)malloc(sizeof(token_job) * (size_t)threads);
    pthread_t *tids = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)threads);
    int *started = (int *)calloc((size_t)threads, sizeof(int));
    for (int i = 0; i < threads; ++i) {
        jobs[i] = *proto;
        jobs[i].t0 = (int)((int64_t)T * i / threads);
        jobs[i].t1 = (int)((int64_t)T * (i + 1) / threads);
        jobs[i].flags = 0;
        started[i] = (i > 0 && pthread_create(&tids[i], NULL, run_token_job, &jobs[i]) == 0);
    }
    run_token_job(&jobs[0]);
    for (int i = 1; i < threads; ++i) {
        if (started[i]) pthread_join(tids[i], NULL);
        else run_token_job(&jobs[i]);            /* no thread could be started: run it here */
    }
    int flags = 0;
    for (int i = 0; i < threads; ++i) flags |= jobs[i].flags;
    free(jobs);
    free(tids);
    free(started);
    return flags;
}

int oracle_dispatch_bf16_mt(const uint16_t *x, int T, int H,
                            const int64_t *topk_idx, const float *topk_weights, int k, int E, int R,
                            const int32_t *token_dst_row, int recv_capacity,
                            uint16_t *recv_x, int64_t *recv_topk_idx, float *recv_topk_weights,
                            int32_t *recv_src_idx, int threads)
{
    if (T < 0 || H < 1 || k < 1 || k > 32 || E % R != 0) return ORACLE_BAD_ARG;
    token_job j;
    memset(&j, 0, sizeof j);
    j.kind = 0; j.src = x; j.H = H; j.k = k; j.E = E; j.R = R; j.recv_capacity = recv_capacity;
    j.topk_idx = topk_idx; j.topk_weights = topk_weights; j.token_dst_row = token_dst_row;
    j.dst = recv_x; j.recv_topk_idx = recv_topk_idx; j.recv_topk_weights = recv_topk_weights;
    j.recv_src_idx = recv_src_idx;
    return run_token_jobs(&j, T, threads);
}

int oracle_combine_mt(const uint16_t *partial, int num_rows, int T, int H, int k,
                      const int32_t *token_dst_row, uint16_t *out, int threads)
{
    if (T < 0 || H < 1 || k < 1 || k > 32) return ORACLE_BAD_ARG;
    token_job j;
    memset(&j, 0, sizeof j);
    j.kind = 1; j.src = partial; j.num_rows = num_rows; j.H = H; j.k = k;
    j.token_dst_row = token_dst_row; j.dst = out;
    return run_token_jobs(&j, T, threads);
}

/* ------------------------------------------------------------------ */
/* Array forms of the number-format conversions (for exhaustive pins). */
/* ------------------------------------------------------------------ */

void oracle_bf16_from_float_n(const float *v, uint16_t *h, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) h[i] = oracle_bf16_from_float(v[i]);
}

void oracle_e4m3_from_float_n(const float *v, uint8_t *q, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) q[i] = oracle_e4m3_from_float(v[i]);
}

/* Combine with per-row weights and the reduction of the received top-k
 * weights. For token t with receive rows in ascending rank order:
 *   out[t] = bf16( acc ), acc = +0.0f then acc = fma(w[row], partial[row], acc)
 *            (single-rounding fused multiply-add per term; w = 1 when
 *            row_weights is NULL, which is then the plain ascending sum);
 *   combined_topk_weights[t, j] = sum over the same rows, ascending, of
 *            recv_topk_weights[row, j] in fp32 from +0.0f. */
int oracle_combine_weighted(const uint16_t *partial, int num_rows, int T, int H, int k,
                            const int32_t *token_dst_row, const float *row_weights,
                            const float *recv_topk_weights, uint16_t *out, float *combined_topk_weights)
{
    if (T < 0 || H < 1 || k < 1 || k > 32) return ORACLE_BAD_ARG;
    int flags = 0;
    int32_t rows[32];
    for (int t = 0; t < T; ++t) {
        int n = 0;
        for (int j = 0; j < k; ++j) {
            int32_t row = token_dst_row[(int64_t)t * k + j];
            if (row < 0) continue;
            if (row >= num_rows) { flags |= ORACLE_CAPACITY; continue; }
            rows[n++] = row;
        }
        for (int a = 1; a < n; ++a)
            for (int b = a; b > 0 && rows[b - 1] > rows[b]; --b) {
                int32_t tmp = rows[b]; rows[b] = rows[b - 1]; rows[b - 1] = tmp;
            }
        for (int h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int i = 0; i < n; ++i) {
                float w = row_weights ? row_weights[rows[i]] : 1.0f;
                acc = fmaf(w, oracle_bf16_to_float(partial[(int64_t)rows[i] * H + h]), acc);
            }
            out[(int64_t)t * H + h] = oracle_bf16_from_float(acc);
        }
        if (combined_topk_weights && recv_topk_weights) {
            for (int j = 0; j < k; ++j) {
                float acc = 0.0f;
                for (int i = 0; i < n; ++i) acc += recv_topk_weights[(int64_t)rows[i] * k + j];
                combined_topk_weights[(int64_t)t * k + j] = acc;
            }
        }
    }
    return flags;
}

/* ------------------------------------------------------------------ */
/* Expand mode: one receive row per valid top-k entry, grouped by expert. */
/* ------------------------------------------------------------------ */

/* The copy epilogue of the DeepEP V2 deep-dive page (section 3.3 stage 3), in
 * expand mode, takes each received token's destination from a counter per
 * expert that starts at the exclusive prefix of the per-expert counts
 * (psum_num_recv_tokens_per_expert) and advances by one per placed token.
 * Readings: one row per valid top-k entry (the per-expert counts of the
 * notify stage count entries, so that is what fills each region exactly);
 * entries are placed in source order -- token ascending, then choice index
 * ascending -- instead of arrival order. Masked (-1) and invalid entries get
 * -1 (invalid ones are flagged). Writes expert_prefix [E+1] and
 * token_expert_row [T, k]. */
int oracle_expand_layout(const int64_t *topk_idx, int T, int k, int E,
                         int32_t *expert_prefix, int32_t *token_expert_row)
{
    if (T < 0 || k < 1 || k > 32 || E < 1) return ORACLE_BAD_ARG;
    int flags = 0;
    int32_t *count = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int64_t i = 0; i < (int64_t)T * k; ++i) {
        int64_t e = topk_idx[i];
        if (e == -1) continue;
        if (e < 0 || e >= E) { flags |= ORACLE_BAD_TOPK; continue; }
        count[e] += 1;
    }
    expert_prefix[0] = 0;
    for (int e = 0; e < E; ++e) expert_prefix[e + 1] = expert_prefix[e] + count[e];
    /* the counter of each expert starts at its region's first row */
    for (int e = 0; e < E; ++e) count[e] = expert_prefix[e];
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int64_t idx = (int64_t)t * k + j;
            int64_t e = topk_idx[idx];
            token_expert_row[idx] = -1;
            if (e < 0 || e >= E) continue;
            token_expert_row[idx] = count[e];
            count[e] += 1;
        }
    }
    free(count);
    return flags;
}

/* Dispatch in expand mode. The row of every valid entry (t, j) receives the
 * token, exactly as in the three dispatch forms above (mode 0: bf16 copy;
 * mode 1: fused per-128 E4M3 quantisation, with x_scales_out; mode 2: E4M3
 * codes and their given scales copied). Reading: a row of the expand layout
 * belongs to one (token, expert) entry, so its metadata keeps that entry only:
 *   recv_topk_idx[row, jj]     = e - rank(e)*m for jj == j, else -1
 *   recv_topk_weights[row, jj] = topk_weights[t, j] for jj == j, else 0
 *   recv_src_idx[row]          = t. */
int oracle_dispatch_expand(int mode, const void *x, const float *x_scales_in, int T, int H,
                           const int64_t *topk_idx, const float *topk_weights, int k, int E, int R,
                           const int32_t *token_expert_row, int recv_capacity,
                           void *recv_x, float *recv_x_scales, int64_t *recv_topk_idx,
                           float *recv_topk_weights, int32_t *recv_src_idx, float *x_scales_out)
{
    if (T < 0 || H < 1 || k < 1 || k > 32 || E % R != 0 || mode < 0 || mode > 2) return ORACLE_BAD_ARG;
    if (mode != 0 && (H < 128 || H % 128 != 0)) return ORACLE_BAD_ARG;
    int flags = 0, m = E / R, nb = H / 128;
    uint8_t *q = (uint8_t *)malloc((size_t)H);
    float *s = (float *)malloc(sizeof(float) * (size_t)(nb > 0 ? nb : 1));
    for (int t = 0; t < T; ++t) {
        if (mode == 1) {
            quantize_row((const uint16_t *)x + (int64_t)t * H, H, q, s);
            if (x_scales_out)
                for (int b = 0; b < nb; ++b) x_scales_out[(int64_t)t * nb + b] = s[b];
        }
        for (int j = 0; j < k; ++j) {
            int64_t row = token_expert_row[(int64_t)t * k + j];
            if (row < 0) continue;
            if (row >= recv_capacity) { flags |= ORACLE_CAPACITY; continue; }
            if (mode == 0) {
                const uint16_t *src = (const uint16_t *)x + (int64_t)t * H;
                uint16_t *dst = (uint16_t *)recv_x + row * H;
                for (int h = 0; h < H; ++h) dst[h] = src[h];
            } else if (mode == 1) {
                uint8_t *dst = (uint8_t *)recv_x + row * H;
                for (int h = 0; h < H; ++h) dst[h] = q[h];
                for (int b = 0; b < nb; ++b) recv_x_scales[row * nb + b] = s[b];
            } else {
                const uint8_t *src = (const uint8_t *)x + (int64_t)t * H;
                uint8_t *dst = (uint8_t *)recv_x + row * H;
                for (int h = 0; h < H; ++h) dst[h] = src[h];
                for (int b = 0; b < nb; ++b) recv_x_scales[row * nb + b] = x_scales_in[(int64_t)t * nb + b];
            }
            int64_t e = topk_idx[(int64_t)t * k + j];
            int r = (int)(e / m);
            recv_src_idx[row] = t;
            for (int jj = 0; jj < k; ++jj) {
                recv_topk_idx[row * k + jj] = (jj == j) ? e - (int64_t)r * m : -1;
                if (recv_topk_weights)
                    recv_topk_weights[row * k + jj] = (jj == j && topk_weights) ? topk_weights[(int64_t)t * k + j] : 0.0f;
            }
        }
    }
    free(q);
    free(s);
    return flags;
}

/* Combine of E4M3 partial rows (codes plus one fp32 scale per 128 channels,
 * the layout the FP8 dispatch produces). Reading: each element is first
 * dequantised on its own, v = RN(value(code) * scale) in fp32, and the
 * token's dequantised rows are then summed as in oracle_combine: ascending
 * receive row, fp32 from +0.0f, one round-to-nearest-even cast to bf16. */
int oracle_combine_fp8(const uint8_t *codes, const float *scales, int num_rows, int T, int H, int k,
                       const int32_t *token_dst_row, uint16_t *out)
{
    if (T < 0 || H < 128 || H % 128 != 0 || k < 1 || k > 32) return ORACLE_BAD_ARG;
    int flags = 0, nb = H / 128;
    int32_t rows[32];
    for (int t = 0; t < T; ++t) {
        int n = 0;
        for (int j = 0; j < k; ++j) {
            int32_t row = token_dst_row[(int64_t)t * k + j];
            if (row < 0) continue;
            if (row >= num_rows) { flags |= ORACLE_CAPACITY; continue; }
            rows[n++] = row;
        }
        for (int a = 1; a < n; ++a)
            for (int b = a; b > 0 && rows[b - 1] > rows[b]; --b) {
                int32_t tmp = rows[b]; rows[b] = rows[b - 1]; rows[b - 1] = tmp;
            }
        for (int h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int i = 0; i < n; ++i) {
                float s = scales[(int64_t)rows[i] * nb + h / 128];
                float v = oracle_e4m3_to_float(codes[(int64_t)rows[i] * H + h]) * s;
                acc = acc + v;
            }
            out[(int64_t)t * H + h] = oracle_bf16_from_float(acc);
        }
    }
    return flags;
}
