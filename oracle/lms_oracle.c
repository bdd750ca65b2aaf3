/*
 * CPU oracle for exact Gumbel-max token sampling fused with the LM-head projection.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's CPU-baseline /
 * reference leg may load this library.  The product path (the CUDA library) never calls it, and
 * the two share no code: no header, helper, table or constant generator.
 *
 * Everything is plain, slow and in fp64, written so that each step can be checked by eye
 * against the pages it follows:
 *
 *   [MLM]  "Megatron-LM pull request 8370: fp64_sampling_noise" -- sections "Problem" (the
 *          exponential race argmax(p/E), E = -log U; the tail-rate closed form) and
 *          "The change" (seeded noise keyed by (request seed, absolute position, vocabulary
 *          index); two Philox words forming the 52-bit midpoint uniform (k + 1/2)/2^52).
 *   [FS]   "FlashSampling: fast and memory-efficient exact sampling" (summary page of
 *          arXiv 2603.15854) -- "Gumbel-Max trick" (i* = argmax_i e_i + g_i), "core method"
 *          and "method step details" (Stage 1 steps 1-6 per vocab tile, Stage 2 argmax over
 *          tile maxima; g = -log(-log u)).
 *   [SDO]  "spec-decode-ops" kernels card -- "Randomness is counter-based Philox".
 *   [SK]   "Write Triton Sampling Kernel" -- reasoning steps 3-4 (greedy short-circuit at T == 0
 *          with smallest-index tie-break; bias added before division by T), "Kernel design
 *          rules" (out-of-range / masked entries are -inf).
 *   [P123] Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11:
 *          the Philox4x32 round function, its multipliers and the Weyl key schedule.
 *
 * Readings where the pages leave a step open (each is also listed with the design notes):
 *   - Philox variant: Philox4x32 with 10 rounds (the pages say "Philox" and "two words ... the
 *     other three", i.e. four 32-bit words per call).
 *   - Key and counter: seeded row  -> key = (seed lo, seed hi), counter = (n, pos lo, pos hi, 0);
 *                      unseeded row -> key = (base_seed lo, base_seed hi),
 *                                      counter = (n, offset lo, offset hi, 0x80000000 | b).
 *     One call gives four words and serves consecutive vocabulary entries: with fp32 noise the
 *     entry v uses word (v & 3) of the call n = v >> 2; with wide noise it uses words 2(v & 1)
 *     and 2(v & 1) + 1 of the call n = v >> 1.  The variate stays a function of (seed, position,
 *     v) alone, as the Megatron-LM PR requires, and no generated word is dropped.
 *   - fp32 noise: k = w >> 8 (the top 24 bits of the entry's word), u = (k + 1/2) / 2^24.
 *     wide noise: k = ((hi << 32) | lo) >> 12 (the top 52 bits of the entry's two words, lo the
 *     first), u = (k + 1/2) / 2^52.  Both u are exact in fp64.  E = -log(u), g = -log(E).
 *   - Transform: masked -> -inf; T == 0 -> greedy, s = y + bias (no noise); otherwise
 *     s = (y + bias) / T + g.  T < 0 or NaN -> the row is invalid (status 2, index -1).
 *     A NaN score counts as -inf.
 *   - Argmax: largest s; ties go to the smallest vocabulary index; -inf never wins; a row with
 *     no finite-or-+inf score gives index -1 and status 1.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------------------------ */
/* Philox4x32-10 [P123]                                                                        */
/* ------------------------------------------------------------------------------------------ */

/* Round multipliers and Weyl key increments as published in [P123] (Table / section 5:
 * M0, M1 for Philox4x32; W0 = golden ratio, W1 = sqrt(3) - 1, both scaled to 32 bits). */
#define ORC_PHILOX_M0 0xD2511F53u
#define ORC_PHILOX_M1 0xCD9E8D57u
#define ORC_PHILOX_W0 0x9E3779B9u
#define ORC_PHILOX_W1 0xBB67AE85u

/* One Philox4x32 round: two 32x32->64 products, the high halves mixed with the other words and
 * the round key, the low halves carried over (the S-box / permutation of [P123]). */
static void orc_philox_round(uint32_t x[4], const uint32_t k[2]) {
    uint64_t p0 = (uint64_t)ORC_PHILOX_M0 * (uint64_t)x[0];
    uint64_t p1 = (uint64_t)ORC_PHILOX_M1 * (uint64_t)x[2];
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t y0 = hi1 ^ x[1] ^ k[0];
    uint32_t y1 = lo1;
    uint32_t y2 = hi0 ^ x[3] ^ k[1];
    uint32_t y3 = lo0;
    x[0] = y0; x[1] = y1; x[2] = y2; x[3] = y3;
}

/* Philox4x32 with R rounds: the first round uses the key as given, each later round the key
 * bumped once more by (W0, W1). */
void orc_philox4x32(const uint32_t ctr[4], const uint32_t key[2], int rounds, uint32_t out[4]) {
    uint32_t x[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
    uint32_t k[2] = {key[0], key[1]};
    for (int r = 0; r < rounds; ++r) {
        if (r > 0) {
            k[0] += ORC_PHILOX_W0;
            k[1] += ORC_PHILOX_W1;
        }
        orc_philox_round(x, k);
    }
    out[0] = x[0]; out[1] = x[1]; out[2] = x[2]; out[3] = x[3];
}

/* Batched form for tests: n calls, ctr [n][4], key [n][2], out [n][4]. */
void orc_philox4x32_many(int64_t n, const uint32_t* ctr, const uint32_t* key, int rounds,
                         uint32_t* out) {
    for (int64_t i = 0; i < n; ++i) orc_philox4x32(ctr + 4 * i, key + 2 * i, rounds, out + 4 * i);
}

/* (request seed, absolute position, call index n) -> (key, counter) [MLM "The change"];
 * unseeded rows are keyed by (base_seed, offset, row) instead [SDO "Randomness"]. */
void orc_key_counter(int seeded, int64_t seed, int64_t pos, uint64_t base_seed, uint64_t offset,
                     int64_t row, uint32_t n, uint32_t ctr[4], uint32_t key[2]) {
    if (seeded) {
        uint64_t s = (uint64_t)seed, p = (uint64_t)pos;
        key[0] = (uint32_t)s; key[1] = (uint32_t)(s >> 32);
        ctr[0] = n; ctr[1] = (uint32_t)p; ctr[2] = (uint32_t)(p >> 32); ctr[3] = 0u;
    } else {
        key[0] = (uint32_t)base_seed; key[1] = (uint32_t)(base_seed >> 32);
        ctr[0] = n; ctr[1] = (uint32_t)offset; ctr[2] = (uint32_t)(offset >> 32);
        ctr[3] = 0x80000000u | (uint32_t)row;
    }
}

/* The Philox call that vocabulary entry v draws from, and the word(s) it uses:
 * fp32 noise -> call n = v >> 2, word (v & 3); wide noise -> call n = v >> 1, words 2(v & 1)
 * (low half) and 2(v & 1) + 1 (high half).  Writes the call's four words to `call` and the
 * entry's words to lo / hi (hi is unused for fp32 noise). */
void orc_entry_words(int seeded, int64_t seed, int64_t pos, uint64_t base_seed, uint64_t offset,
                     int64_t row, uint32_t v, int wide, uint32_t call[4], uint32_t* lo,
                     uint32_t* hi) {
    uint32_t ctr[4], key[2];
    uint32_t n = wide ? (v >> 1) : (v >> 2);
    orc_key_counter(seeded, seed, pos, base_seed, offset, row, n, ctr, key);
    orc_philox4x32(ctr, key, 10, call);
    if (wide) {
        *lo = call[2 * (v & 1u)];
        *hi = call[2 * (v & 1u) + 1];
    } else {
        *lo = call[v & 3u];
        *hi = 0u;
    }
}

/* ------------------------------------------------------------------------------------------ */
/* Uniform and noise [MLM "Problem", "The change"; FS step 3]                                  */
/* ------------------------------------------------------------------------------------------ */

/* The midpoint uniform u = (k + 1/2) / 2^m, exact in fp64, from the entry's word(s):
 * fp32 noise: k = lo >> 8 (m = 24); wide noise: k = ((hi << 32) | lo) >> 12 (m = 52). */
double orc_uniform(uint32_t lo, uint32_t hi, int wide) {
    if (wide) {
        uint64_t k = ((((uint64_t)hi) << 32) | (uint64_t)lo) >> 12;
        return ldexp((double)k + 0.5, -52);
    } else {
        uint32_t k = lo >> 8;
        return ldexp((double)k + 0.5, -24);
    }
}

/* Exponential variate E = -log U and Gumbel variate g = -log E = -log(-log U). */
double orc_exponential(double u) { return -log(u); }
double orc_gumbel(double u) { return -log(-log(u)); }

static int row_is_seeded(const int64_t* seeds, int64_t b) { return seeds != NULL && seeds[b] >= 0; }

/* Noise for a [B][V] grid, any of the outputs may be NULL:
 *   words [B][V][4] uint32 (the four words of the call entry v draws from), u, E, g [B][V]. */
void orc_noise_fill(int64_t B, int64_t V, const int64_t* seeds, const int64_t* positions,
                    uint64_t base_seed, uint64_t offset, int wide, uint32_t* words, double* u,
                    double* E, double* g) {
    for (int64_t b = 0; b < B; ++b) {
        int seeded = row_is_seeded(seeds, b);
        int64_t seed = seeded ? seeds[b] : 0, pos = seeded ? positions[b] : 0;
        for (int64_t v = 0; v < V; ++v) {
            uint32_t w[4], lo, hi;
            orc_entry_words(seeded, seed, pos, base_seed, offset, b, (uint32_t)v, wide, w, &lo, &hi);
            int64_t i = b * V + v;
            if (words) memcpy(words + 4 * i, w, sizeof w);
            double uu = orc_uniform(lo, hi, wide);
            if (u) u[i] = uu;
            if (E) E[i] = orc_exponential(uu);
            if (g) g[i] = orc_gumbel(uu);
        }
    }
}

/* Gumbel noise g[v] (v < V) of one row given its row index and absolute position explicitly
 * (speculative verification draws at positions pos + i of one batch row). */
void orc_noise_row(int seeded, int64_t seed, int64_t pos, uint64_t base_seed, uint64_t offset,
                   int64_t row, int64_t V, int wide, double* g) {
    for (int64_t v = 0; v < V; ++v) {
        uint32_t w[4], lo, hi;
        orc_entry_words(seeded, seed, pos, base_seed, offset, row, (uint32_t)v, wide, w, &lo, &hi);
        g[v] = orc_gumbel(orc_uniform(lo, hi, wide));
    }
}

/* The acceptance uniform of speculative verification [SDO "verify", "Randomness"]: the Philox
 * call with counter word 0 = 0xffffffff (a call index no vocabulary entry uses, V < 2^31), keyed
 * like the race's noise; its first word (fp32 noise) or first two words (wide noise) give the
 * midpoint uniform. */
double orc_accept_uniform(int seeded, int64_t seed, int64_t pos, uint64_t base_seed,
                          uint64_t offset, int64_t row, int wide) {
    uint32_t ctr[4], key[2], w[4];
    orc_key_counter(seeded, seed, pos, base_seed, offset, row, 0xffffffffu, ctr, key);
    orc_philox4x32(ctr, key, 10, w);
    return orc_uniform(w[0], w[1], wide);
}

/* ------------------------------------------------------------------------------------------ */
/* Per-row race: transform, perturb, argmax, per-tile maxima [FS steps 2-6, Stage 2; SK]        */
/* ------------------------------------------------------------------------------------------ */

typedef struct {
    /* logits: either y [B][ld_y] (fp64; ld_y == 0 broadcasts one row) or computed on the fly */
    const double* y; int64_t ld_y;
    int64_t B, V;
    const double* T;              /* [B] or NULL (all 1) */
    const int64_t* seeds;         /* [B] or NULL (all unseeded); seed < 0 -> unseeded row */
    const int64_t* positions;     /* [B] (read for seeded rows) */
    const double* bias; int64_t ld_bias;    /* [B][ld_bias] or NULL; ld_bias == 0 broadcasts */
    const uint32_t* mask; int64_t ld_mask;  /* [B][ld_mask] allow bits or NULL; 0 broadcasts */
    uint64_t base_seed, offset;
    int wide;
    int64_t tile_v;               /* > 0: also report per-tile maxima */
    /* outputs */
    int64_t* out; int32_t* status; double* top1; double* top2;
    double* tile_max; int64_t* tile_idx;   /* [B][n_tiles] when tile_v > 0 */
    double* scores;                /* optional [B][V] perturbed scores */
    const int64_t* rows;           /* optional: evaluate only these batch rows; output slot i and
                                      y row i belong to batch row rows[i] (n_rows of them) */
    int64_t n_rows;
} orc_rows_args;

/* Perturbed score s for row b, column v, given the (untransformed) logit y. */
static double orc_score(const orc_rows_args* a, int64_t b, int64_t v, double y) {
    if (a->mask) {
        uint32_t word = a->mask[b * a->ld_mask + (v >> 5)];
        if (((word >> (v & 31)) & 1u) == 0u) return -INFINITY;
    }
    double T = a->T ? a->T[b] : 1.0;
    double bias = a->bias ? a->bias[b * a->ld_bias + v] : 0.0;
    double t = y + bias;                       /* bias before temperature [SK step 4] */
    double s;
    if (T == 0.0) {
        s = t;                                 /* greedy: no noise [SK step 3] */
    } else {
        int seeded = row_is_seeded(a->seeds, b);
        uint32_t w[4], lo, hi;
        orc_entry_words(seeded, seeded ? a->seeds[b] : 0, seeded ? a->positions[b] : 0,
                        a->base_seed, a->offset, b, (uint32_t)v, a->wide, w, &lo, &hi);
        s = t / T + orc_gumbel(orc_uniform(lo, hi, a->wide));
    }
    if (isnan(s)) s = -INFINITY;
    return s;
}

/* Row b of the batch, its logits yrow, its outputs at slot o (o == b unless a subset of rows
 * is evaluated). */
static void orc_one_row(const orc_rows_args* a, int64_t b, int64_t o, const double* yrow) {
    int64_t V = a->V;
    double T = a->T ? a->T[b] : 1.0;
    int64_t nt = a->tile_v > 0 ? (V + a->tile_v - 1) / a->tile_v : 0;
    if (isnan(T) || T < 0.0) {                 /* invalid temperature: rejected per row */
        a->out[o] = -1; a->status[o] = 2;
        if (a->top1) a->top1[o] = -INFINITY;
        if (a->top2) a->top2[o] = -INFINITY;
        for (int64_t t = 0; t < nt; ++t) { a->tile_max[o * nt + t] = -INFINITY; a->tile_idx[o * nt + t] = -1; }
        if (a->scores) for (int64_t v = 0; v < V; ++v) a->scores[o * V + v] = -INFINITY;
        return;
    }
    double best = -INFINITY, second = -INFINITY;
    int64_t arg = -1;
    for (int64_t t = 0; t < nt; ++t) { a->tile_max[o * nt + t] = -INFINITY; a->tile_idx[o * nt + t] = -1; }
    for (int64_t v = 0; v < V; ++v) {
        double s = orc_score(a, b, v, yrow[v]);
        if (a->scores) a->scores[o * V + v] = s;
        if (s > -INFINITY) {
            if (arg < 0 || s > best) {         /* strict '>' keeps the smallest index on ties */
                second = best; best = s; arg = v;
            } else if (s > second) {
                second = s;
            }
            if (nt > 0) {
                int64_t t = v / a->tile_v;
                if (a->tile_idx[o * nt + t] < 0 || s > a->tile_max[o * nt + t]) {
                    a->tile_max[o * nt + t] = s; a->tile_idx[o * nt + t] = v;
                }
            }
        }
    }
    a->out[o] = arg;
    a->status[o] = arg < 0 ? 1 : 0;
    if (a->top1) a->top1[o] = best;
    if (a->top2) a->top2[o] = second;
}

typedef struct { const orc_rows_args* a; int64_t b0, b1; } orc_rows_job;

static void* orc_rows_worker(void* p) {
    const orc_rows_job* j = (const orc_rows_job*)p;
    for (int64_t i = j->b0; i < j->b1; ++i) {
        int64_t b = j->a->rows ? j->a->rows[i] : i;
        orc_one_row(j->a, b, i, j->a->y + i * j->a->ld_y);
    }
    return NULL;
}

static void orc_run_rows(const orc_rows_args* a, int nthreads) {
    int64_t n = a->rows ? a->n_rows : a->B;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n) nthreads = (int)(n > 0 ? n : 1);
    pthread_t th[256];
    orc_rows_job jobs[256];
    if (nthreads > 256) nthreads = 256;
    for (int i = 0; i < nthreads; ++i) {
        jobs[i].a = a;
        jobs[i].b0 = n * i / nthreads;
        jobs[i].b1 = n * (i + 1) / nthreads;
        pthread_create(&th[i], NULL, orc_rows_worker, &jobs[i]);
    }
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
}

/* Gumbel race over materialised logits (the second entry point): y [B][ld_y] in fp64. */
void orc_sample_from_logits(const double* y, int64_t ld_y, int64_t B, int64_t V, const double* T,
                            const int64_t* seeds, const int64_t* positions, const double* bias,
                            int64_t ld_bias, const uint32_t* mask, int64_t ld_mask,
                            uint64_t base_seed, uint64_t offset, int wide, int64_t tile_v,
                            int64_t* out, int32_t* status, double* top1, double* top2,
                            double* tile_max, int64_t* tile_idx, double* scores, int nthreads) {
    orc_rows_args a = {y, ld_y, B, V, T, seeds, positions, bias, ld_bias, mask, ld_mask,
                       base_seed, offset, wide, tile_v, out, status, top1, top2,
                       tile_max, tile_idx, scores, NULL, 0};
    orc_run_rows(&a, nthreads);
}

/* ------------------------------------------------------------------------------------------ */
/* LM-head logits Y = H W^T in fp64 from bf16 inputs [FS step 1]                              */
/* ------------------------------------------------------------------------------------------ */

/* bf16 -> fp64: the bf16 bits are the upper half of an fp32; the conversion is exact. */
static double orc_bf16(uint16_t h) {
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t* H; int64_t ldh; const uint16_t* W; int64_t ldw;
    int64_t B, D, V; double* y; int64_t v0, v1;
    const int64_t* rows;   /* NULL: all B rows; else y row i is H row rows[i] (B of them) */
} orc_gemm_job;

static void* orc_gemm_worker(void* p) {
    const orc_gemm_job* j = (const orc_gemm_job*)p;
    double* hrow = (double*)malloc(sizeof(double) * (size_t)j->D);
    double* wrow = (double*)malloc(sizeof(double) * (size_t)j->D);
    for (int64_t v = j->v0; v < j->v1; ++v) {
        for (int64_t d = 0; d < j->D; ++d) wrow[d] = orc_bf16(j->W[v * j->ldw + d]);
        for (int64_t i = 0; i < j->B; ++i) {
            int64_t b = j->rows ? j->rows[i] : i;
            double acc = 0.0;
            for (int64_t d = 0; d < j->D; ++d) acc += orc_bf16(j->H[b * j->ldh + d]) * wrow[d];
            j->y[i * j->V + v] = acc;
        }
    }
    free(hrow); free(wrow);
    return NULL;
}

static void orc_gemm(const uint16_t* H, int64_t ldh, const uint16_t* W, int64_t ldw, int64_t B,
                     int64_t D, int64_t V, double* y, const int64_t* rows, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    orc_gemm_job jobs[256];
    for (int i = 0; i < nthreads; ++i) {
        orc_gemm_job j = {H, ldh, W, ldw, B, D, V, y, V * i / nthreads, V * (i + 1) / nthreads, rows};
        jobs[i] = j;
        pthread_create(&th[i], NULL, orc_gemm_worker, &jobs[i]);
    }
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
}

/* y [B][V] = sum_d H[b][d] * W[v][d], accumulated in fp64 in increasing d. */
void orc_lmhead_logits(const uint16_t* H, int64_t ldh, const uint16_t* W, int64_t ldw, int64_t B,
                       int64_t D, int64_t V, double* y, int nthreads) {
    orc_gemm(H, ldh, W, ldw, B, D, V, y, NULL, nthreads);
}

/* The fused path's result: logits in fp64, then the same per-row race. */
int orc_lmhead_sample(const uint16_t* H, int64_t ldh, const uint16_t* W, int64_t ldw, int64_t B,
                      int64_t D, int64_t V, const double* T, const int64_t* seeds,
                      const int64_t* positions, const double* bias, int64_t ld_bias,
                      const uint32_t* mask, int64_t ld_mask, uint64_t base_seed, uint64_t offset,
                      int wide, int64_t tile_v, int64_t* out, int32_t* status, double* top1,
                      double* top2, double* tile_max, int64_t* tile_idx, double* scores,
                      int nthreads) {
    double* y = (double*)malloc(sizeof(double) * (size_t)(B * V));
    if (!y) return 1;
    orc_gemm(H, ldh, W, ldw, B, D, V, y, NULL, nthreads);
    orc_sample_from_logits(y, V, B, V, T, seeds, positions, bias, ld_bias, mask, ld_mask,
                           base_seed, offset, wide, tile_v, out, status, top1, top2, tile_max,
                           tile_idx, scores, nthreads);
    free(y);
    return 0;
}

/* Perturbed scores at n chosen (b, v) pairs of the fused path, each computed on its own:
 * one fp64 dot product, the transform and the noise.  Used where a full-size oracle pass is
 * too slow (sampled checks) and to score the index another implementation chose. */
void orc_lmhead_scores_at(const uint16_t* H, int64_t ldh, const uint16_t* W, int64_t ldw,
                          int64_t B, int64_t D, int64_t V, const double* T, const int64_t* seeds,
                          const int64_t* positions, const double* bias, int64_t ld_bias,
                          const uint32_t* mask, int64_t ld_mask, uint64_t base_seed,
                          uint64_t offset, int wide, int64_t n, const int64_t* bs,
                          const int64_t* vs, double* s_out) {
    orc_rows_args a = {NULL, 0, B, V, T, seeds, positions, bias, ld_bias, mask, ld_mask,
                       base_seed, offset, wide, 0, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                       NULL, 0};
    for (int64_t i = 0; i < n; ++i) {
        int64_t b = bs[i], v = vs[i];
        double Tb = T ? T[b] : 1.0;
        if (isnan(Tb) || Tb < 0.0) { s_out[i] = -INFINITY; continue; }
        double acc = 0.0;
        for (int64_t d = 0; d < D; ++d) acc += orc_bf16(H[b * ldh + d]) * orc_bf16(W[v * ldw + d]);
        s_out[i] = orc_score(&a, b, v, acc);
    }
}

/* The fused path's result for a subset of the batch: rows[i] (i < n_rows) are batch rows of the
 * full B-row problem (their own temperature, seed, position, bias and mask rows, and row index
 * for unseeded keys); outputs are [n_rows] / [n_rows][n_tiles], and the perturbed scores
 * [n_rows][V] when `scores` is not NULL. */
int orc_lmhead_sample_rows(const uint16_t* H, int64_t ldh, const uint16_t* W, int64_t ldw,
                           int64_t B, int64_t D, int64_t V, const int64_t* rows, int64_t n_rows,
                           const double* T, const int64_t* seeds, const int64_t* positions,
                           const double* bias, int64_t ld_bias, const uint32_t* mask,
                           int64_t ld_mask, uint64_t base_seed, uint64_t offset, int wide,
                           int64_t tile_v, int64_t* out, int32_t* status, double* top1,
                           double* top2, double* tile_max, int64_t* tile_idx, double* scores,
                           int nthreads) {
    double* y = (double*)malloc(sizeof(double) * (size_t)(n_rows * V));
    if (!y) return 1;
    orc_gemm(H, ldh, W, ldw, n_rows, D, V, y, rows, nthreads);
    orc_rows_args a = {y, V, B, V, T, seeds, positions, bias, ld_bias, mask, ld_mask,
                       base_seed, offset, wide, tile_v, out, status, top1, top2,
                       tile_max, tile_idx, scores, rows, n_rows};
    orc_run_rows(&a, nthreads);
    free(y);
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* Filtered race: top-k -> top-p -> min-p, then the Gumbel race over the kept tokens           */
/* [SDO "Semantics"; SK reasoning steps 6-8, "Correctness requirements"]                      */
/* ------------------------------------------------------------------------------------------ */
/* Readings (also listed with the design notes):
 *   - t = (y + bias) / T as in the race (masked -> -inf); T == 0 rows are greedy (filters cannot
 *     remove the top token, so the greedy token is the filtered one too).
 *   - Sorted order: t descending, then v ascending.  top-k keeps the first k of that order
 *     (1 <= top_k; values above k_max count as k_max; <= 0 or >= V = off).
 *   - top-p (0 < top_p < 1) keeps the shortest prefix of the top-k set (or, with top-k off, of
 *     the first k_max tokens) whose probability mass -- normalised over that set -- reaches
 *     top_p, the crossing token included.
 *   - min-p (0 < min_p <= 1) keeps p_i >= min_p * p_max, i.e. t_i - t_max >= log(min_p).
 *   - Every filter keeps the top token.  The race over the kept set samples the softmax
 *     renormalised to it (Gumbel-max over a subset). */

typedef struct { double t; int64_t v; } orc_tv;

static int orc_cmp_desc(const void* x, const void* y) {
    const orc_tv* a = (const orc_tv*)x; const orc_tv* b = (const orc_tv*)y;
    if (a->t > b->t) return -1;
    if (a->t < b->t) return 1;
    return (a->v < b->v) ? -1 : (a->v > b->v);
}

typedef struct {
    const double* y; int64_t ld_y; int64_t B, V;
    const double* T; const int64_t* seeds; const int64_t* positions;
    const double* bias; int64_t ld_bias; const uint32_t* mask; int64_t ld_mask;
    uint64_t base_seed, offset; int wide;
    const int32_t* top_k; const double* top_p; const double* min_p; int32_t k_max;
    double p_shift;      /* added to top_p (to probe the decision boundary) */
    double minp_scale;   /* multiplies min_p (same) */
    int64_t* out; int32_t* status; int32_t* kept;
    double* top1; double* top2;    /* optional: the two best perturbed scores of the kept set */
} orc_filt_args;

static void orc_filtered_row(const orc_filt_args* f, int64_t b) {
    int64_t V = f->V;
    double T = f->T ? f->T[b] : 1.0;
    if (f->top1) { f->top1[b] = -INFINITY; f->top2[b] = -INFINITY; }
    if (isnan(T) || T < 0.0) { f->out[b] = -1; f->status[b] = 2; if (f->kept) f->kept[b] = 0; return; }
    const double* yrow = f->y + b * f->ld_y;
    orc_rows_args a = {NULL, 0, f->B, V, f->T, f->seeds, f->positions, f->bias, f->ld_bias, f->mask,
                       f->ld_mask, f->base_seed, f->offset, f->wide, 0, NULL, NULL, NULL, NULL,
                       NULL, NULL, NULL, NULL, 0};
    /* transformed logits (no noise), -inf for masked / NaN */
    orc_tv* tv = (orc_tv*)malloc(sizeof(orc_tv) * (size_t)V);
    int64_t n_fin = 0;
    for (int64_t v = 0; v < V; ++v) {
        double t = -INFINITY;
        int ok = 1;
        if (f->mask) ok = (f->mask[b * f->ld_mask + (v >> 5)] >> (v & 31)) & 1u;
        if (ok) {
            double bias = f->bias ? f->bias[b * f->ld_bias + v] : 0.0;
            t = (T == 0.0) ? yrow[v] + bias : (yrow[v] + bias) / T;
            if (isnan(t)) t = -INFINITY;
        }
        tv[v].t = t; tv[v].v = v;
        if (t > -INFINITY) ++n_fin;
    }
    if (n_fin == 0) { f->out[b] = -1; f->status[b] = 1; if (f->kept) f->kept[b] = 0; free(tv); return; }
    qsort(tv, (size_t)V, sizeof(orc_tv), orc_cmp_desc);   /* -inf entries sort last */
    int32_t k = f->top_k ? f->top_k[b] : 0;
    int64_t kmax = f->k_max > 0 ? f->k_max : 1024;
    double p = f->top_p ? f->top_p[b] + f->p_shift : 1.0;
    double mp = f->min_p ? f->min_p[b] * f->minp_scale : 0.0;
    int topk_on = k >= 1 && k < V;
    int topp_on = f->top_p && f->top_p[b] > 0.0 && f->top_p[b] < 1.0;
    int64_t n = n_fin;                                    /* kept prefix length */
    if (topk_on) n = (k > kmax ? kmax : k) < n ? (k > kmax ? kmax : k) : n;
    else if (topp_on && n > kmax) n = kmax;
    if (topp_on) {
        double z = 0.0;
        for (int64_t i = 0; i < n; ++i) z += exp(tv[i].t - tv[0].t);
        double c = 0.0;
        int64_t m = n;
        for (int64_t i = 0; i < n; ++i) {
            c += exp(tv[i].t - tv[0].t) / z;
            if (c >= p) { m = i + 1; break; }
        }
        n = m;
    }
    if (f->min_p && f->min_p[b] > 0.0) {
        double thr = tv[0].t + log(mp);
        int64_t m = 1;
        while (m < n && tv[m].t >= thr) ++m;
        n = m;
    }
    if (n < 1) n = 1;
    /* race over the kept prefix */
    double best = -INFINITY, second = -INFINITY;
    int64_t arg = -1;
    for (int64_t i = 0; i < n; ++i) {
        int64_t v = tv[i].v;
        double s = orc_score(&a, b, v, yrow[v]);
        if (arg < 0 || s > best || (s == best && v < arg)) {
            if (arg >= 0) second = best > second ? best : second;
            best = s; arg = v;
        } else if (s > second) {
            second = s;
        }
    }
    if (f->top1) { f->top1[b] = best; f->top2[b] = second; }
    f->out[b] = arg;
    f->status[b] = 0;
    if (f->kept) f->kept[b] = (int32_t)n;
    free(tv);
}

typedef struct { const orc_filt_args* f; int64_t b0, b1; } orc_filt_job;

static void* orc_filt_worker(void* p) {
    const orc_filt_job* j = (const orc_filt_job*)p;
    for (int64_t b = j->b0; b < j->b1; ++b) orc_filtered_row(j->f, b);
    return NULL;
}

/* Filtered race over materialised logits y [B][ld_y] (ld_y == 0 broadcasts one row). */
void orc_sample_filtered(const double* y, int64_t ld_y, int64_t B, int64_t V, const double* T,
                         const int64_t* seeds, const int64_t* positions, const double* bias,
                         int64_t ld_bias, const uint32_t* mask, int64_t ld_mask,
                         uint64_t base_seed, uint64_t offset, int wide, const int32_t* top_k,
                         const double* top_p, const double* min_p, int32_t k_max, double p_shift,
                         double minp_scale, int64_t* out, int32_t* status, int32_t* kept,
                         double* top1, double* top2, int nthreads) {
    orc_filt_args f = {y, ld_y, B, V, T, seeds, positions, bias, ld_bias, mask, ld_mask,
                       base_seed, offset, wide, top_k, top_p, min_p, k_max, p_shift, minp_scale,
                       out, status, kept, top1, top2};
    if (nthreads < 1) nthreads = 1;
    if (nthreads > B) nthreads = (int)B;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    orc_filt_job jobs[256];
    for (int i = 0; i < nthreads; ++i) {
        jobs[i].f = &f; jobs[i].b0 = B * i / nthreads; jobs[i].b1 = B * (i + 1) / nthreads;
        pthread_create(&th[i], NULL, orc_filt_worker, &jobs[i]);
    }
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
}

/* ------------------------------------------------------------------------------------------ */
/* FP8 (E4M3) inputs: W8A8 with per-row scales [FS "Limitations": low-precision FP8 inputs]     */
/* ------------------------------------------------------------------------------------------ */
/* E4M3 ("fn" variant): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0
 * holds subnormals m/8 * 2^-6; no infinities; S.1111.111 is NaN; the largest finite value is
 * S.1111.110 = 1.75 * 2^8 = 448. */
double orc_e4m3_decode(uint8_t c) {
    int s = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round to the nearest finite E4M3 value (ties to the even code), saturating at +-448:
 * written as a search over every finite code, so it can be checked by eye. */
uint8_t orc_e4m3_encode(double x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = (x < 0.0 || (x == 0.0 && signbit(x))) ? 0x80 : 0x00;
    double a = fabs(x);
    uint8_t best = 0;
    double best_d = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {                       /* non-negative finite codes */
        double d = fabs(orc_e4m3_decode((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) { best_d = d; best = (uint8_t)c; }
    }
    return (uint8_t)(sign | best);
}

/* Per-row power-of-two quantisation of bf16 activations: e_b is the smallest integer with
 * max_d |h[b][d]| * 2^-e_b <= 448 (0 for an all-zero row); q = E4M3(h * 2^-e_b).  Scaling by a
 * power of two is exact, so the rounding to E4M3 is the only step. */
void orc_quantize_rows_e4m3(const uint16_t* H, int64_t ldh, int64_t B, int64_t D, uint8_t* q,
                            int64_t ldq, int32_t* e_out) {
    for (int64_t b = 0; b < B; ++b) {
        double amax = 0.0;
        for (int64_t d = 0; d < D; ++d) {
            double h = fabs(orc_bf16(H[b * ldh + d]));
            if (h > amax) amax = h;
        }
        int e = 0;
        if (amax > 0.0) {
            e = -160;
            while (ldexp(amax, -e) > 448.0) ++e;
        }
        e_out[b] = e;
        for (int64_t d = 0; d < D; ++d) q[b * ldq + d] = orc_e4m3_encode(ldexp(orc_bf16(H[b * ldh + d]), -e));
    }
}

typedef struct {
    const uint8_t* H8; int64_t ldh; const int32_t* e_h; const uint8_t* W8; int64_t ldw;
    const double* w_scale; int64_t B, D, V; double* y; int64_t v0, v1; const int64_t* rows;
} orc_gemm8_job;

static void* orc_gemm8_worker(void* p) {
    const orc_gemm8_job* j = (const orc_gemm8_job*)p;
    double* wrow = (double*)malloc(sizeof(double) * (size_t)j->D);
    for (int64_t v = j->v0; v < j->v1; ++v) {
        for (int64_t d = 0; d < j->D; ++d) wrow[d] = orc_e4m3_decode(j->W8[v * j->ldw + d]);
        for (int64_t i = 0; i < j->B; ++i) {
            int64_t b = j->rows ? j->rows[i] : i;
            double acc = 0.0;
            for (int64_t d = 0; d < j->D; ++d) acc += orc_e4m3_decode(j->H8[b * j->ldh + d]) * wrow[d];
            j->y[i * j->V + v] = acc * ldexp(1.0, j->e_h[b]) * j->w_scale[v];
        }
    }
    free(wrow);
    return NULL;
}

/* y[b][v] = 2^e_h[b] * w_scale[v] * sum_d E4M3(H8[b][d]) * E4M3(W8[v][d]), in fp64; rows as in
 * orc_lmhead_sample_rows (NULL = all B). */
void orc_lmhead_logits_fp8(const uint8_t* H8, int64_t ldh, const int32_t* e_h, const uint8_t* W8,
                           int64_t ldw, const double* w_scale, int64_t B, int64_t D, int64_t V,
                           const int64_t* rows, int64_t n_rows, double* y, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    orc_gemm8_job jobs[256];
    int64_t nb = rows ? n_rows : B;
    for (int i = 0; i < nthreads; ++i) {
        orc_gemm8_job j = {H8, ldh, e_h, W8, ldw, w_scale, nb, D, V, y, V * i / nthreads,
                           V * (i + 1) / nthreads, rows};
        jobs[i] = j;
        pthread_create(&th[i], NULL, orc_gemm8_worker, &jobs[i]);
    }
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
}

/* The fused FP8 path's result for rows (NULL = all): quantise H, fp64 logits from the FP8
 * operands and scales, then the same per-row race (tile maxima for tile_v). */
int orc_lmhead_sample_fp8(const uint16_t* H, int64_t ldh, const uint8_t* W8, int64_t ldw,
                          const double* w_scale, int64_t B, int64_t D, int64_t V,
                          const int64_t* rows, int64_t n_rows, const double* T,
                          const int64_t* seeds, const int64_t* positions, const double* bias,
                          int64_t ld_bias, const uint32_t* mask, int64_t ld_mask,
                          uint64_t base_seed, uint64_t offset, int wide, int64_t tile_v,
                          int64_t* out, int32_t* status, double* top1, double* top2,
                          double* tile_max, int64_t* tile_idx, int nthreads) {
    uint8_t* q = (uint8_t*)malloc((size_t)(B * D));
    int32_t* e = (int32_t*)malloc(sizeof(int32_t) * (size_t)B);
    int64_t nb = rows ? n_rows : B;
    double* y = (double*)malloc(sizeof(double) * (size_t)(nb * V));
    if (!q || !e || !y) { free(q); free(e); free(y); return 1; }
    orc_quantize_rows_e4m3(H, ldh, B, D, q, D, e);
    orc_lmhead_logits_fp8(q, D, e, W8, ldw, w_scale, B, D, V, rows, n_rows, y, nthreads);
    orc_rows_args a = {y, V, B, V, T, seeds, positions, bias, ld_bias, mask, ld_mask,
                       base_seed, offset, wide, tile_v, out, status, top1, top2,
                       tile_max, tile_idx, NULL, rows, rows ? n_rows : 0};
    orc_run_rows(&a, nthreads);
    free(q); free(e); free(y);
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* MXFP4 weights (W4A16) [FS "Limitations", "Future directions": low-precision inputs for the  */
/* memory-bound regime].  The format is the Open Compute Project's Microscaling MXFP4: E2M1     */
/* elements, one shared UE8M0 scale per block of 32 consecutive elements of a row.              */
/* ------------------------------------------------------------------------------------------ */
/* E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.  Exponent field 0 is the
 * subnormal 0.5 * m; otherwise (1 + m / 2) * 2^(e - 1).  Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6;
 * no infinities or NaN. */
double orc_e2m1_decode(uint8_t code) {
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double v = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, e - 1);
    return s ? -v : v;
}

/* UE8M0: an unsigned 8-bit exponent, 2^(s - 127); s = 255 is NaN. */
double orc_ue8m0_decode(uint8_t s) { return s == 255 ? NAN : ldexp(1.0, (int)s - 127); }

/* Nearest E2M1 code of x (ties to the code with mantissa bit 0), saturating at +-6: a search over
 * the eight magnitudes, so it can be checked by eye. */
uint8_t orc_e2m1_encode(double x) {
    uint8_t sign = (x < 0.0 || (x == 0.0 && signbit(x))) ? 8 : 0;
    double a = fabs(x);
    uint8_t best = 0;
    double best_d = INFINITY;
    for (int c = 0; c < 8; ++c) {
        double d = fabs(orc_e2m1_decode((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) { best_d = d; best = (uint8_t)c; }
    }
    return (uint8_t)(sign | best);
}

/* The weight W[v][d] of an MXFP4 matrix: element d of row v is the low (d even) or high (d odd)
 * nibble of byte W4[v][d / 2]; its scale is S[d / 32][v] (block-major scales, lds >= V). */
double orc_mxfp4_weight(const uint8_t* W4, int64_t ldw4, const uint8_t* S, int64_t lds, int64_t v,
                        int64_t d) {
    uint8_t byte = W4[v * ldw4 + d / 2];
    uint8_t code = (d % 2 == 0) ? (byte & 15) : (byte >> 4);
    return orc_e2m1_decode(code) * orc_ue8m0_decode(S[(d / 32) * lds + v]);
}

typedef struct {
    const uint16_t* H; int64_t ldh; const uint8_t* W4; int64_t ldw4; const uint8_t* S; int64_t lds;
    int64_t B, D, V; double* y; int64_t v0, v1; const int64_t* rows;
} orc_gemm4_job;

static void* orc_gemm4_worker(void* p) {
    const orc_gemm4_job* j = (const orc_gemm4_job*)p;
    double* wrow = (double*)malloc(sizeof(double) * (size_t)j->D);
    for (int64_t v = j->v0; v < j->v1; ++v) {
        for (int64_t d = 0; d < j->D; ++d) wrow[d] = orc_mxfp4_weight(j->W4, j->ldw4, j->S, j->lds, v, d);
        for (int64_t i = 0; i < j->B; ++i) {
            int64_t b = j->rows ? j->rows[i] : i;
            double acc = 0.0;
            for (int64_t d = 0; d < j->D; ++d) acc += orc_bf16(j->H[b * j->ldh + d]) * wrow[d];
            j->y[i * j->V + v] = acc;
        }
    }
    free(wrow);
    return NULL;
}

/* y[b][v] = sum_d bf16(H[b][d]) * E2M1(W4[v][d]) * 2^(S[d/32][v] - 127), in fp64 (each product
 * is exact), summed in increasing d; rows as in orc_lmhead_sample_rows (NULL = all B). */
void orc_lmhead_logits_mxfp4(const uint16_t* H, int64_t ldh, const uint8_t* W4, int64_t ldw4,
                             const uint8_t* S, int64_t lds, int64_t B, int64_t D, int64_t V,
                             const int64_t* rows, int64_t n_rows, double* y, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    orc_gemm4_job jobs[256];
    int64_t nb = rows ? n_rows : B;
    for (int i = 0; i < nthreads; ++i) {
        orc_gemm4_job j = {H, ldh, W4, ldw4, S, lds, nb, D, V, y, V * i / nthreads,
                           V * (i + 1) / nthreads, rows};
        jobs[i] = j;
        pthread_create(&th[i], NULL, orc_gemm4_worker, &jobs[i]);
    }
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
}

/* The fused MXFP4 path's result for rows (NULL = all): fp64 logits from bf16 H and the decoded
 * MXFP4 weights, then the same per-row race (tile maxima for tile_v). */
int orc_lmhead_sample_mxfp4(const uint16_t* H, int64_t ldh, const uint8_t* W4, int64_t ldw4,
                            const uint8_t* S, int64_t lds, int64_t B, int64_t D, int64_t V,
                            const int64_t* rows, int64_t n_rows, const double* T,
                            const int64_t* seeds, const int64_t* positions, const double* bias,
                            int64_t ld_bias, const uint32_t* mask, int64_t ld_mask,
                            uint64_t base_seed, uint64_t offset, int wide, int64_t tile_v,
                            int64_t* out, int32_t* status, double* top1, double* top2,
                            double* tile_max, int64_t* tile_idx, int nthreads) {
    int64_t nb = rows ? n_rows : B;
    double* y = (double*)malloc(sizeof(double) * (size_t)(nb * V));
    if (!y) return 1;
    orc_lmhead_logits_mxfp4(H, ldh, W4, ldw4, S, lds, B, D, V, rows, n_rows, y, nthreads);
    orc_rows_args a = {y, V, B, V, T, seeds, positions, bias, ld_bias, mask, ld_mask,
                       base_seed, offset, wide, tile_v, out, status, top1, top2,
                       tile_max, tile_idx, NULL, rows, rows ? n_rows : 0};
    orc_run_rows(&a, nthreads);
    free(y);
    return 0;
}
