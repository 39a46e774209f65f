/*
 * kvevict_oracle.c -- plain, slow CPU oracle for one decode step of attention
 * over a budget-bounded KV cache with eviction.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may load this code. The product path never
 * calls it, and it shares no code, header, table or helper with the CUDA
 * library.
 *
 * Arithmetic is fp64 throughout. Inputs are kept exactly as given (fp32
 * values, or bf16 values held in fp32) and widened to fp64 when used.
 * Everything is per unit: one (sequence, layer, KV head) cache, independent
 * of every other unit.
 *
 * Sources (page title, then section):
 *  - "KV Cache 驱逐策略：从 LRU 到 H2O" (wiblog.cn), "注意力分数" and the
 *    eviction flowchart: each generated token attends over the cache, every
 *    cached token's cumulative attention score is updated, and eviction only
 *    happens once the pool is full.
 *  - "h2o: heavy-hitter oracle ..." summary (fmread.com), the Algorithm 1
 *    paragraph: budget K; at step i the candidate set is S_{i-1} plus {i};
 *    if it exceeds K, remove the element v whose removal leaves the remaining
 *    set with the highest cumulative score.
 *  - "Attention Sinks 与 KV Cache 淘汰策略" (10100.com), section 4.1
 *    (StreamingLLM: first 4 tokens locked as sinks, ring buffer for the most
 *    recent W) and section 4.2 (H2O: sink + heavy hitters + recent window;
 *    per-step loop attend -> accumulate -> select -> evict).
 *  - "Random Attention" summary (ai-feeds.com), "方法": keep every prompt
 *    token; for generated tokens over budget K, evict uniformly at random,
 *    independently per attention head, with a periodic budget K and buffer r.
 *  - Philox4x64-10: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
 *    Easy as 1, 2, 3", SC'11.
 *
 * Readings where the pages leave a step open (each one also listed with the
 * design notes):
 *  - the new token attends over the retained set plus itself; eviction comes
 *    after attention and accumulation, and the new token takes the victim's
 *    slot;
 *  - the H2O recent window is a position window that includes the new token:
 *    a token is a candidate iff n_sink <= pos <= p - n_recent;
 *  - f_score is additive, so the remaining set's score after removing v is
 *    F(T) - s(v); ties go to the lower score, then the older position;
 *  - one decision per unit; with GQA the unit's score is the mean of its G
 *    query heads' probabilities;
 *  - prompt tokens enter with score 0 through the same admission rule (the
 *    API gives prefill no queries);
 *  - softmax scale 1/sqrt(d), no position encoding;
 *  - Random: a cut happens when the generated count reaches K + r and removes
 *    the r generated tokens with the smallest 64-bit Philox key (ties: older
 *    position), counter (pos, step, layer * 2^16 + head, seq), key
 *    (seed, 0x5EED0001).
 *  - two-pool H2O (the H2OCache class of "KV Cache 驱逐策略：从 LRU 到 H2O",
 *    section "实现要点"): the new token joins the recent pool; when that pool
 *    holds more than n_recent tokens its lowest (score, position) member
 *    leaves, the new token included; it enters the heavy-hitter pool iff its
 *    score is strictly above hh_threshold, else it is dropped; a heavy-hitter
 *    pool above n_heavy drops its lowest member, the one just promoted
 *    included. Ties go to the older position in both pools.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORC_H2O = 0, ORC_SINK_WINDOW = 1, ORC_RANDOM = 2, ORC_H2O_BLOCK = 3, ORC_H2O_POOLS = 4 };
enum { ORC_OK = 0, ORC_EINVAL = -1, ORC_ECAPACITY = -2, ORC_ESTATE = -3 };

#define ORC_RANDOM_KEY_TAG 0x5EED0001ull

typedef struct orc_unit {
    int policy, n_sink, n_heavy, n_recent, budget, r, max_prompt, cap, G, d;
    uint64_t seed;
    int seq, layer, head;
    int prompt_len;      /* prompt tokens appended so far */
    int t;               /* decode steps committed */
    int n_gen;           /* generated tokens currently held (Random) */
    int n_cuts;
    int32_t *pos;        /* [cap] position held by each slot, -1 = empty */
    float *k, *v;        /* [cap][d] */
    double *score;       /* [cap] cumulative attention score (H2O) */
    double evicted_mass; /* sum of the scores of evicted tokens (H2O) */
    /* the token of the step in progress */
    int have_new;
    int is_prompt;
    int32_t new_pos;
    float *k_new, *v_new;
    double score_new;
    int32_t last_victim_pos; /* position removed by the last commit, -1 if none */
    int greedy_disagreements; /* argmax F(T\{v}) != argmin (score, pos): must stay 0 */
    int last_block;      /* H2O_BLOCK: block released for the token of the last step, -1 if none */
    double forget;       /* score storage: s <- (1 - forget) s + a each step (0: exact accumulation) */
    int half;            /* score storage: every stored score rounded to IEEE binary16 */
    int int8;            /* score storage: unsigned 8-bit codes times one scale per unit (absmax) */
    double qscale;       /* INT8: the unit's scale, its largest score / 255 (0 before any step) */
    double qmax;         /* INT8: that largest score M */
    double *qx;          /* INT8: [cap] each slot's s * 255 / M before rounding, at the last update */
    double qx_new;       /* INT8: the same for the new token */
    /* two-pool H2O */
    signed char *pool;   /* [cap] 0: recent pool, 1: heavy-hitter pool (slots with pos >= 0) */
    double hh_threshold; /* promotion needs a score strictly above this */
    int dec_slot;        /* decision of the last orc_choose: slot for the new token (cap: dropped), */
    int dec_pool;        /* the pool it joins, */
    int dec_promote;     /* the slot of a held token moved to the heavy-hitter pool (-1: none), */
    double dec_margin;   /* and the smallest relative gap among the comparisons that decided it */
    int last_promote;    /* the promotion of the last commit: slot, -2 the new token itself, -1 none */
} orc_unit;

/* ------------------------------------------------------------------------ */
/* Philox4x64-10 (SC'11).                                                    */
/* ------------------------------------------------------------------------ */

static void mulhilo64(uint64_t a, uint64_t b, uint64_t *hi, uint64_t *lo)
{
    unsigned __int128 p = (unsigned __int128)a * (unsigned __int128)b;
    *hi = (uint64_t)(p >> 64);
    *lo = (uint64_t)p;
}

void orc_philox4x64_10(const uint64_t ctr_in[4], const uint64_t key_in[2], uint64_t out[4])
{
    /* Round multipliers and Weyl key increments from the SC'11 paper. */
    const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
    const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
    uint64_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint64_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { k0 += W0; k1 += W1; }
        uint64_t hi0, lo0, hi1, lo1;
        mulhilo64(M0, c0, &hi0, &lo0);
        mulhilo64(M1, c2, &hi1, &lo1);
        uint64_t n0 = hi1 ^ c1 ^ k0;
        uint64_t n1 = lo1;
        uint64_t n2 = hi0 ^ c3 ^ k1;
        uint64_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The eviction key Random Attention draws for one generated token at one cut. */
uint64_t orc_random_key(uint64_t seed, int seq, int layer, int head, int step, int pos)
{
    uint64_t ctr[4] = {(uint64_t)(uint32_t)pos, (uint64_t)(uint32_t)step,
                       ((uint64_t)(uint32_t)layer << 16) + (uint64_t)(uint32_t)head,
                       (uint64_t)(uint32_t)seq};
    uint64_t key[2] = {seed, ORC_RANDOM_KEY_TAG};
    uint64_t out[4];
    orc_philox4x64_10(ctr, key, out);
    return out[0];
}

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 rounding (round to nearest, ties to even).               */
/* ------------------------------------------------------------------------ */

/* The binary16 value nearest to x (x >= 0, finite): 11 significant bits for
 * normal values (x >= 2^-14), a fixed spacing of 2^-24 below, +inf from
 * 65520 on (the halfway point past the largest finite value, 65504). */
double orc_round_half(double x)
{
    if (!(x > 0.0)) return x == 0.0 ? 0.0 : x;
    if (x >= 65520.0) return INFINITY;
    int e;
    frexp(x, &e);                       /* x = f 2^e, f in [0.5, 1): 2^(e-1) <= x < 2^e */
    int q = e - 1 - 10;                 /* the spacing 2^q of 11-bit significands at x */
    if (q < -24) q = -24;               /* subnormal range */
    const double ulp = ldexp(1.0, q);
    return nearbyint(x / ulp) * ulp;    /* default rounding mode: ties to even */
}

/* ------------------------------------------------------------------------ */
/* Unit lifetime.                                                            */
/* ------------------------------------------------------------------------ */

orc_unit *orc_new(int policy, int n_sink, int n_heavy, int n_recent, int budget, int r, int max_prompt,
                  int G, int d, uint64_t seed, int seq, int layer, int head)
{
    if (G < 1 || d < 1 || budget < 1) return NULL;
    if (policy == ORC_H2O) {
        if (n_sink < 0 || n_heavy < 0 || n_recent < 1 || n_sink + n_heavy + n_recent != budget) return NULL;
    } else if (policy == ORC_SINK_WINDOW) {
        if (n_sink < 0 || n_heavy != 0 || n_recent < 1 || n_sink + n_recent != budget) return NULL;
    } else if (policy == ORC_RANDOM) {
        if (r < 1 || max_prompt < 0) return NULL;
    } else if (policy == ORC_H2O_POOLS) {
        /* no sinks: the class keeps a recent pool and a heavy-hitter pool only */
        if (n_sink != 0 || n_heavy < 0 || n_recent < 1 || n_heavy + n_recent != budget) return NULL;
    } else if (policy == ORC_H2O_BLOCK) {
        /* r is the block size; the budget is whole blocks, and besides the
         * blocks holding sinks at least one block lies outside the recent
         * window, so a full cache always has a block to release */
        if (n_sink < 0 || n_heavy < 0 || n_recent < 1 || n_sink + n_heavy + n_recent != budget) return NULL;
        if (r < 1 || budget % r != 0) return NULL;
        const int nb = budget / r, nsb = (n_sink + r - 1) / r;
        if ((long long)(nb - nsb - 1) * r < n_recent) return NULL;
    } else {
        return NULL;
    }
    orc_unit *u = (orc_unit *)calloc(1, sizeof(orc_unit));
    if (!u) return NULL;
    u->policy = policy; u->n_sink = n_sink; u->n_heavy = n_heavy; u->n_recent = n_recent;
    u->budget = budget; u->r = r; u->max_prompt = max_prompt; u->G = G; u->d = d;
    u->seed = seed; u->seq = seq; u->layer = layer; u->head = head;
    u->cap = (policy == ORC_RANDOM) ? max_prompt + budget + r : budget;
    u->pos = (int32_t *)malloc(sizeof(int32_t) * (size_t)u->cap);
    u->k = (float *)calloc((size_t)u->cap * (size_t)d, sizeof(float));
    u->v = (float *)calloc((size_t)u->cap * (size_t)d, sizeof(float));
    u->score = (double *)calloc((size_t)u->cap, sizeof(double));
    u->k_new = (float *)calloc((size_t)d, sizeof(float));
    u->v_new = (float *)calloc((size_t)d, sizeof(float));
    u->pool = (signed char *)calloc((size_t)u->cap, 1);
    u->qx = (double *)calloc((size_t)u->cap, sizeof(double));
    if (!u->pos || !u->k || !u->v || !u->score || !u->k_new || !u->v_new || !u->pool || !u->qx) {
        free(u->pos); free(u->k); free(u->v); free(u->score); free(u->k_new); free(u->v_new); free(u->pool);
        free(u->qx);
        free(u);
        return NULL;
    }
    for (int s = 0; s < u->cap; ++s) u->pos[s] = -1;
    u->last_victim_pos = -1;
    u->last_block = -1;
    u->dec_slot = -1;
    u->dec_promote = -1;
    u->last_promote = -1;
    return u;
}

/* The promotion threshold of two-pool H2O (the class leaves it open): a
 * token leaving the recent pool enters the heavy-hitter pool iff its score is
 * strictly above theta. Any value but NaN; -INFINITY promotes every token. On
 * an empty unit. */
int orc_set_hh_threshold(orc_unit *u, double theta)
{
    if (u->policy != ORC_H2O_POOLS || isnan(theta)) return ORC_EINVAL;
    if (u->prompt_len != 0 || u->t != 0 || u->have_new) return ORC_ESTATE;
    u->hh_threshold = theta;
    return ORC_OK;
}

/* Score-storage variants ("Attention Sinks 与 KV Cache 淘汰策略" section 6.2: the
 * cumulative scores are stored in FP16, or a moving average replaces the exact
 * accumulation): every step s <- (1 - forget) s + a for each retained token,
 * with 0 <= forget < 1 (0 is the exact cumulative score), and with half != 0
 * every stored score (the new token's too) is rounded to binary16 right after
 * its update. The score-keeping policies only (half: not block H2O), on an
 * empty unit. */
int orc_set_score_storage(orc_unit *u, double forget, int half)
{
    if (u->policy != ORC_H2O && u->policy != ORC_H2O_BLOCK && u->policy != ORC_H2O_POOLS) return ORC_EINVAL;
    if (half && u->policy == ORC_H2O_BLOCK) return ORC_EINVAL;
    if (half && u->int8) return ORC_EINVAL;
    if (!(forget >= 0.0 && forget < 1.0)) return ORC_EINVAL;
    if (u->prompt_len != 0 || u->t != 0 || u->have_new) return ORC_ESTATE;
    u->forget = forget;
    u->half = half != 0;
    return ORC_OK;
}

/* INT8 score storage (the same section names "INT8 quantisation" of the
 * scores and gives no scale or zero point; the reading here is symmetric
 * absmax quantisation per unit, zero point 0 as scores are >= 0): after each
 * step's update, with M the largest score of the unit's retained tokens and
 * the new token, every score s becomes the code c = round(s * 255 / M)
 * (nearest, ties to even; 0..255) and is stored as c * M / 255. Written from
 * that definition, in fp64 like the rest of the oracle. Plain H2O only; not
 * with binary16; on an empty unit. */
int orc_set_score_int8(orc_unit *u, int on)
{
    if (u->policy != ORC_H2O || (on && u->half)) return ORC_EINVAL;
    if (u->prompt_len != 0 || u->t != 0 || u->have_new) return ORC_ESTATE;
    u->int8 = on != 0;
    return ORC_OK;
}

/* The code of score s under absmax M: round(s * 255 / M), ties to even (the
 * default rounding mode), within 0..255; *x receives s * 255 / M unrounded. */
static double int8_code(double s, double M, double *x)
{
    *x = M > 0.0 ? s * 255.0 / M : 0.0;
    double c = nearbyint(*x);
    if (c > 255.0) c = 255.0;
    if (!(c >= 0.0)) c = 0.0;
    return c;
}

/* Requantises every retained score and the new token's after an update. */
static void quantise_int8(orc_unit *u)
{
    double M = u->score_new;
    for (int s = 0; s < u->cap; ++s)
        if (u->pos[s] >= 0 && u->score[s] > M) M = u->score[s];
    for (int s = 0; s < u->cap; ++s) {
        u->qx[s] = 0.0;
        if (u->pos[s] >= 0) u->score[s] = int8_code(u->score[s], M, &u->qx[s]) * M / 255.0;
    }
    u->score_new = int8_code(u->score_new, M, &u->qx_new) * M / 255.0;
    u->qmax = M;
    u->qscale = M / 255.0;
}

double orc_score_scale(const orc_unit *u) { return u->qscale; }

/* The INT8 codes of the unit's slots (0 for empty slots and before any step). */
void orc_score_codes(const orc_unit *u, uint8_t *dst)
{
    for (int s = 0; s < u->cap; ++s)
        dst[s] = (u->pos[s] >= 0 && u->qmax > 0.0) ? (uint8_t)nearbyint(u->score[s] * 255.0 / u->qmax) : 0;
}

/* INT8: each slot's s * 255 / M before the last rounding (0 for empty slots),
 * and the pending new token's (test use: how close a code was to a midpoint). */
void orc_int8_unrounded(const orc_unit *u, double *dst, double *new_x)
{
    for (int s = 0; s < u->cap; ++s) dst[s] = u->pos[s] >= 0 ? u->qx[s] : 0.0;
    *new_x = u->qx_new;
}

/* Test hook: replaces the code of the token in `slot` (slot == cap: the
 * pending new token) by `code`, one code away from its own, so that a caller
 * checking another implementation can continue from that implementation's
 * value where the two rounded a midpoint apart. Nothing else changes. */
int orc_adopt_int8_code(orc_unit *u, int slot, int code)
{
    if (!u->int8 || !(u->qmax > 0.0) || code < 0 || code > 255 || slot < 0 || slot > u->cap) return ORC_EINVAL;
    if (slot == u->cap && !u->have_new) return ORC_ESTATE;
    if (slot < u->cap && u->pos[slot] < 0) return ORC_EINVAL;
    double *v = slot == u->cap ? &u->score_new : &u->score[slot];
    const double own = nearbyint(*v * 255.0 / u->qmax);
    if (fabs(own - (double)code) > 1.0) return ORC_EINVAL;
    *v = (double)code * u->qmax / 255.0;
    return ORC_OK;
}

/* Test hook: replaces the stored cumulative scores of the retained tokens
 * (scores[slot]; empty slots ignored) and of the pending new token, for
 * checking another selector on the same values: the choice that follows is
 * made by the steps of this file, on these values. */
int orc_set_scores(orc_unit *u, const double *scores, double score_new)
{
    if (!u->have_new) return ORC_ESTATE;
    for (int s = 0; s < u->cap; ++s)
        if (u->pos[s] >= 0) u->score[s] = scores[s];
    u->score_new = score_new;
    return ORC_OK;
}

void orc_free(orc_unit *u)
{
    if (!u) return;
    free(u->pos); free(u->k); free(u->v); free(u->score); free(u->k_new); free(u->v_new); free(u->pool);
    free(u->qx);
    free(u);
}

int orc_capacity(const orc_unit *u) { return u->cap; }
int orc_steps(const orc_unit *u) { return u->t; }
int orc_prompt_len(const orc_unit *u) { return u->prompt_len; }
int orc_cuts(const orc_unit *u) { return u->n_cuts; }
int orc_greedy_disagreements(const orc_unit *u) { return u->greedy_disagreements; }
double orc_evicted_mass(const orc_unit *u) { return u->evicted_mass; }
int32_t orc_last_victim_pos(const orc_unit *u) { return u->last_victim_pos; }
int orc_last_block(const orc_unit *u) { return u->last_block; }
double orc_new_score(const orc_unit *u) { return u->score_new; }

void orc_positions(const orc_unit *u, int32_t *dst) { memcpy(dst, u->pos, sizeof(int32_t) * (size_t)u->cap); }
void orc_pools(const orc_unit *u, signed char *dst) { memcpy(dst, u->pool, (size_t)u->cap); }
int orc_last_promote(const orc_unit *u) { return u->last_promote; }
double orc_decision_margin(const orc_unit *u) { return u->dec_margin; }
void orc_decision(const orc_unit *u, int *out3)
{
    out3[0] = u->dec_slot;
    out3[1] = u->dec_pool;
    out3[2] = u->dec_promote;
}
void orc_scores(const orc_unit *u, double *dst) { memcpy(dst, u->score, sizeof(double) * (size_t)u->cap); }

/* Copy out the stored K/V of one slot (test use). */
void orc_slot_kv(const orc_unit *u, int slot, float *k, float *v)
{
    memcpy(k, u->k + (size_t)slot * u->d, sizeof(float) * (size_t)u->d);
    memcpy(v, u->v + (size_t)slot * u->d, sizeof(float) * (size_t)u->d);
}

int32_t orc_pos_at(const orc_unit *u, int slot)
{
    return (slot >= 0 && slot < u->cap) ? u->pos[slot] : -2;
}

int orc_count(const orc_unit *u)
{
    int n = 0;
    for (int s = 0; s < u->cap; ++s) n += (u->pos[s] >= 0);
    return n;
}

static int first_free_slot(const orc_unit *u)
{
    for (int s = 0; s < u->cap; ++s)
        if (u->pos[s] < 0) return s;
    return -1;
}

/* ------------------------------------------------------------------------ */
/* Step (i)+(ii): attention of the new token's G queries over the retained   */
/* tokens plus the new token itself, and the cumulative-score update.        */
/* ------------------------------------------------------------------------ */

/* Block-granular H2O ("Attention Sinks 与 KV Cache 淘汰策略" section 5: a paged
 * cache releases whole blocks, and the block that matters least goes first).
 * The slots form blocks of r consecutive slots. When a token needs a slot and
 * the cache is full, one block is released before that token attends: among
 * the blocks whose tokens all lie outside the sinks and the recent window
 * (n_sink <= pos <= p - n_recent, p the incoming token's position), the block
 * B that leaves the remaining set with the highest cumulative score F(T \ B)
 * = F(T) - sum of B's scores; ties go to the lower sum, then to the block
 * holding the oldest token. Its slots become free; the incoming token and the
 * next ones take them lowest first. */
static int release_block(orc_unit *u, int32_t p)
{
    const int bs = u->r, nb = u->cap / bs;
    double total = 0.0;
    for (int s = 0; s < u->cap; ++s)
        if (u->pos[s] >= 0) total += u->score[s];
    int best = -1, am = -1;
    double best_F = -INFINITY, best_sum = 0.0, am_sum = 0.0;
    int32_t best_min = 0, am_min = 0;
    for (int b = 0; b < nb; ++b) {
        double sum = 0.0;
        int32_t mn = INT32_MAX, mx = -1;
        int full = 1;
        for (int s = b * bs; s < (b + 1) * bs; ++s) {
            if (u->pos[s] < 0) { full = 0; break; }
            sum += u->score[s];
            if (u->pos[s] < mn) mn = u->pos[s];
            if (u->pos[s] > mx) mx = u->pos[s];
        }
        if (!full || mn < u->n_sink || mx > p - u->n_recent) continue;
        const double F = total - sum;
        if (best < 0 || F > best_F || (F == best_F && (sum < best_sum || (sum == best_sum && mn < best_min)))) {
            best = b; best_F = F; best_sum = sum; best_min = mn;
        }
        if (am < 0 || sum < am_sum || (sum == am_sum && mn < am_min)) { am = b; am_sum = sum; am_min = mn; }
    }
    if (best < 0) return ORC_ECAPACITY;
    if (am != best) u->greedy_disagreements++;
    for (int s = best * bs; s < (best + 1) * bs; ++s) {
        u->evicted_mass += u->score[s];
        u->pos[s] = -1;
        u->score[s] = 0.0;
    }
    u->last_block = best;
    return ORC_OK;
}

int orc_attend(orc_unit *u, const float *q, const float *k_new, const float *v_new, double *out)
{
    if (u->have_new) return ORC_ESTATE;
    u->last_block = -1;
    if (u->policy == ORC_H2O_BLOCK && orc_count(u) == u->cap) {
        int rc = release_block(u, u->prompt_len + u->t);
        if (rc) return rc;
    }
    const int G = u->G, d = u->d, cap = u->cap;
    const double scale = 1.0 / sqrt((double)d);
    memcpy(u->k_new, k_new, sizeof(float) * (size_t)d);
    memcpy(u->v_new, v_new, sizeof(float) * (size_t)d);
    u->new_pos = u->prompt_len + u->t;
    u->is_prompt = 0;

    double *z = (double *)malloc(sizeof(double) * (size_t)(cap + 1));
    double *mass = (double *)calloc((size_t)(cap + 1), sizeof(double)); /* sum over heads of p */
    if (!z || !mass) { free(z); free(mass); return ORC_ECAPACITY; }

    for (int g = 0; g < G; ++g) {
        const float *qg = q + (size_t)g * d;
        /* logits of every retained token, in slot order, then the new token */
        double m = -INFINITY;
        for (int s = 0; s <= cap; ++s) {
            const float *ks;
            if (s < cap) {
                if (u->pos[s] < 0) continue;
                ks = u->k + (size_t)s * d;
            } else {
                ks = u->k_new;
            }
            double dot = 0.0;
            for (int i = 0; i < d; ++i) dot += (double)qg[i] * (double)ks[i];
            z[s] = dot * scale;
            if (z[s] > m) m = z[s];
        }
        double l = 0.0;
        for (int s = 0; s <= cap; ++s) {
            if (s < cap && u->pos[s] < 0) continue;
            l += exp(z[s] - m);
        }
        double *og = out + (size_t)g * d;
        for (int i = 0; i < d; ++i) og[i] = 0.0;
        for (int s = 0; s <= cap; ++s) {
            if (s < cap && u->pos[s] < 0) continue;
            double p = exp(z[s] - m) / l;
            const float *vs = (s < cap) ? u->v + (size_t)s * d : u->v_new;
            for (int i = 0; i < d; ++i) og[i] += p * (double)vs[i];
            mass[s] += p;
        }
    }
    /* H2O: every retained token's cumulative score grows by this step's
     * probability (mean over the unit's G query heads); the new token starts
     * with its own. Sink-window and Random keep no scores. */
    if (u->policy == ORC_H2O || u->policy == ORC_H2O_BLOCK || u->policy == ORC_H2O_POOLS) {
        for (int s = 0; s < cap; ++s) {
            if (u->pos[s] < 0) continue;
            u->score[s] = (1.0 - u->forget) * u->score[s] + mass[s] / (double)G;
            if (u->half) u->score[s] = orc_round_half(u->score[s]);
        }
        u->score_new = mass[cap] / (double)G;
        if (u->half) u->score_new = orc_round_half(u->score_new);
        if (u->int8) quantise_int8(u);
    } else {
        u->score_new = 0.0;
    }
    free(z);
    free(mass);
    u->have_new = 1;
    return ORC_OK;
}

/* Stages a decode token without computing attention. Only for the
 * policies whose retained set never depends on attention (StreamingLLM,
 * Random): their slot tables can then be replayed cheaply over long traces,
 * with orc_attend used only at the steps whose outputs are compared. */
int orc_stage(orc_unit *u, const float *k_new, const float *v_new)
{
    if (u->have_new) return ORC_ESTATE;
    if (u->policy == ORC_H2O || u->policy == ORC_H2O_BLOCK || u->policy == ORC_H2O_POOLS) return ORC_EINVAL;
    memcpy(u->k_new, k_new, sizeof(float) * (size_t)u->d);
    memcpy(u->v_new, v_new, sizeof(float) * (size_t)u->d);
    u->new_pos = u->prompt_len + u->t;
    u->is_prompt = 0;
    u->score_new = 0.0;
    u->have_new = 1;
    return ORC_OK;
}

/* A prompt token is admitted like a decode token, with score 0 and no
 * attention. */
static int stage_prompt_token(orc_unit *u, const float *k, const float *v)
{
    if (u->have_new) return ORC_ESTATE;
    if (u->t > 0) return ORC_ESTATE;
    if (u->policy == ORC_RANDOM && u->prompt_len >= u->max_prompt) return ORC_ECAPACITY;
    u->last_block = -1;
    if (u->policy == ORC_H2O_BLOCK && orc_count(u) == u->cap) {
        int rc = release_block(u, u->prompt_len);
        if (rc) return rc;
    }
    memcpy(u->k_new, k, sizeof(float) * (size_t)u->d);
    memcpy(u->v_new, v, sizeof(float) * (size_t)u->d);
    u->new_pos = u->prompt_len;
    u->is_prompt = 1;
    u->score_new = 0.0;
    u->have_new = 1;
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Step (iii): where the new token goes.                                     */
/* ------------------------------------------------------------------------ */

/* H2O, Algorithm 1: T = S u {new}; if |T| > K remove the eligible v that
 * maximises F(T \ {v}). Returns the slot the new token takes. */
static int choose_h2o(orc_unit *u)
{
    int count = orc_count(u);
    if (count + 1 <= u->budget) return first_free_slot(u);

    const int32_t p = u->new_pos;
    double total = u->score_new; /* F(T) */
    for (int s = 0; s < u->cap; ++s)
        if (u->pos[s] >= 0) total += u->score[s];

    int best = -1;
    double best_F = -INFINITY, best_s = 0.0;
    int32_t best_pos = 0;
    for (int s = 0; s < u->cap; ++s) {
        int32_t ps = u->pos[s];
        if (ps < 0) continue;
        if (!(ps >= u->n_sink && ps <= p - u->n_recent)) continue; /* sink or recent: protected */
        double F = total - u->score[s]; /* the remaining set's cumulative score */
        int better = 0;
        if (best < 0 || F > best_F) better = 1;
        else if (F == best_F && (u->score[s] < best_s || (u->score[s] == best_s && ps < best_pos))) better = 1;
        if (better) { best = s; best_F = F; best_s = u->score[s]; best_pos = ps; }
    }
    /* The new token is never a candidate: it sits inside the recent window. */

    /* Cross-check against the plain argmin of (score, position). */
    int am = -1;
    for (int s = 0; s < u->cap; ++s) {
        int32_t ps = u->pos[s];
        if (ps < 0 || !(ps >= u->n_sink && ps <= p - u->n_recent)) continue;
        if (am < 0 || u->score[s] < u->score[am] || (u->score[s] == u->score[am] && ps < u->pos[am])) am = s;
    }
    if (am != best) u->greedy_disagreements++;
    return best;
}

/* StreamingLLM, written as the ring it is: the first n_sink positions are
 * locked; the window holds the newest n_recent tokens and a new token
 * overwrites the oldest window entry. */
static int choose_sink_window(orc_unit *u)
{
    if (u->new_pos < u->n_sink) return first_free_slot(u);
    int in_window = 0, oldest = -1;
    for (int s = 0; s < u->cap; ++s) {
        if (u->pos[s] < u->n_sink) continue; /* empty or sink */
        in_window++;
        if (oldest < 0 || u->pos[s] < u->pos[oldest]) oldest = s;
    }
    if (in_window < u->n_recent) return first_free_slot(u);
    return oldest;
}

/* (score a, position pa) below (score b, position pb): the lower score, then
 * the older position. */
static int key_less(double a, int32_t pa, double b, int32_t pb) { return a < b || (a == b && pa < pb); }

static double rel_gap(double a, double b)
{
    const double m = fmax(fabs(a), fabs(b));
    if (isinf(a) || isinf(b)) return a == b ? 0.0 : INFINITY;
    return m > 0.0 ? fabs(a - b) / m : 0.0;
}

/* Two-pool H2O, the H2OCache class's add step ("KV Cache 驱逐策略：从 LRU 到
 * H2O", section "实现要点"), after the scores were updated by orc_attend:
 *   1. the new token joins the recent pool;
 *   2. if the recent pool now holds more than n_recent tokens, its lowest
 *      (score, position) member v leaves it (the new token is a member);
 *   3. if score(v) > hh_threshold, v joins the heavy-hitter pool, and if that
 *      pool now holds more than n_heavy tokens its lowest member leaves the
 *      cache (v included); otherwise v leaves the cache.
 * The new token, unless it is the one leaving, takes the slot of the token
 * that left, else the lowest empty slot. Records the decision in dec_* and
 * returns the slot, or cap when the new token itself left. */
static int choose_pools(orc_unit *u)
{
    const int32_t pn = u->new_pos;
    const double sn = u->score_new;
    int n_rec = 0, n_hh = 0, v = -1, w = -1;
    for (int s = 0; s < u->cap; ++s) {
        if (u->pos[s] < 0) continue;
        if (u->pool[s] == 0) {
            n_rec++;
            if (v < 0 || key_less(u->score[s], u->pos[s], u->score[v], u->pos[v])) v = s;
        } else {
            n_hh++;
            if (w < 0 || key_less(u->score[s], u->pos[s], u->score[w], u->pos[w])) w = s;
        }
    }
    u->dec_pool = 0;
    u->dec_promote = -1;
    u->dec_margin = INFINITY;
    if (n_rec + 1 <= u->n_recent) { /* 1: room in the recent pool */
        u->dec_slot = first_free_slot(u);
        return u->dec_slot;
    }
    /* 2: v leaves the recent pool -- its lowest member, the new token included */
    const int v_new = v < 0 || key_less(sn, pn, u->score[v], u->pos[v]);
    const double sv = v_new ? sn : u->score[v];
    const int32_t pv = v_new ? pn : u->pos[v];
    if (!(sv > u->hh_threshold)) { /* 3: v leaves the cache */
        u->dec_slot = v_new ? u->cap : v;
    } else if (n_hh + 1 <= u->n_heavy) { /* 3: v promoted, room in the heavy-hitter pool */
        u->dec_slot = first_free_slot(u);
        if (v_new) u->dec_pool = 1; else u->dec_promote = v;
    } else if (w >= 0 && key_less(u->score[w], u->pos[w], sv, pv)) { /* 3: v promoted, w leaves */
        u->dec_slot = w;
        if (v_new) u->dec_pool = 1; else u->dec_promote = v;
    } else { /* 3: v promoted and, the pool's lowest, leaves at once */
        u->dec_slot = v_new ? u->cap : v;
    }

    /* Diagnostic: the smallest relative gap of the comparisons that decided
     * -- the two lowest of the recent pool plus the new token, score(v)
     * against the threshold, the two lowest of the heavy-hitter pool plus v
     * when it overflowed. */
    double gap = rel_gap(sv, u->hh_threshold);
    for (int s = 0; s <= u->cap; ++s) { /* s == cap: the new token */
        const int held = s < u->cap && u->pos[s] >= 0;
        if (s < u->cap && !held) continue;
        const double x = s < u->cap ? u->score[s] : sn;
        const int in_rec = s == u->cap || u->pool[s] == 0;
        const int is_v = v_new ? s == u->cap : s == v;
        if (in_rec && !is_v) gap = fmin(gap, rel_gap(x, sv));
        if (sv > u->hh_threshold && n_hh + 1 > u->n_heavy && s < u->cap && !in_rec) {
            /* the heavy-hitter pool plus v: its lowest against every other member */
            if (key_less(u->score[w], u->pos[w], sv, pv)) gap = fmin(gap, rel_gap(s == w ? sv : x, u->score[w]));
            else gap = fmin(gap, rel_gap(x, sv));
        }
    }
    u->dec_margin = gap;
    return u->dec_slot;
}

int orc_choose(orc_unit *u)
{
    if (!u->have_new) return ORC_ESTATE;
    switch (u->policy) {
    case ORC_H2O: return choose_h2o(u);
    case ORC_SINK_WINDOW: return choose_sink_window(u);
    case ORC_H2O_POOLS: return choose_pools(u);
    default: return first_free_slot(u); /* Random, H2O_BLOCK: the lowest free slot */
    }
}

/* ------------------------------------------------------------------------ */
/* Step (iv): admit the new token into `slot`, evicting what it held.        */
/* ------------------------------------------------------------------------ */

typedef struct { uint64_t key; int32_t pos; int slot; } orc_draw;

static int cmp_draw(const void *a, const void *b)
{
    const orc_draw *x = (const orc_draw *)a, *y = (const orc_draw *)b;
    if (x->key != y->key) return x->key < y->key ? -1 : 1;
    return (x->pos > y->pos) - (x->pos < y->pos);
}

/* Random Attention's periodic cut: every generated token gets a fresh 64-bit
 * key for this step; the r smallest leave. The prompt is never touched. */
static void random_cut(orc_unit *u, int step)
{
    int n = 0;
    orc_draw *dr = (orc_draw *)malloc(sizeof(orc_draw) * (size_t)u->cap);
    for (int s = 0; s < u->cap; ++s) {
        if (u->pos[s] < u->prompt_len) continue; /* empty or prompt */
        dr[n].key = orc_random_key(u->seed, u->seq, u->layer, u->head, step, u->pos[s]);
        dr[n].pos = u->pos[s];
        dr[n].slot = s;
        n++;
    }
    qsort(dr, (size_t)n, sizeof(orc_draw), cmp_draw);
    for (int i = 0; i < u->r && i < n; ++i) u->pos[dr[i].slot] = -1;
    u->n_gen = n - (u->r < n ? u->r : n);
    u->n_cuts++;
    free(dr);
}

/* Two-pool H2O: admit the new token into `slot` in pool `new_pool` (slot ==
 * cap: the new token leaves), evicting what the slot held, and move the token
 * in slot `promote` (-1: none) to the heavy-hitter pool. Checked for
 * consistency with the pools' sizes; any such decision is accepted, so that
 * a caller can adopt another implementation's choice at a near-tie. */
int orc_commit_pools(orc_unit *u, int slot, int new_pool, int promote)
{
    if (!u->have_new || u->policy != ORC_H2O_POOLS) return ORC_ESTATE;
    if (slot < 0 || slot > u->cap || (new_pool != 0 && new_pool != 1)) return ORC_EINVAL;
    if (promote >= 0 && (promote >= u->cap || promote == slot || u->pos[promote] < 0 || u->pool[promote] != 0))
        return ORC_EINVAL;
    if (promote < -1 || (promote >= 0 && new_pool == 1) || (slot == u->cap && (promote >= 0 || new_pool == 1)))
        return ORC_EINVAL;
    int n_rec = 0, n_hh = 0;
    for (int s = 0; s < u->cap; ++s)
        if (u->pos[s] >= 0 && s != slot) { n_rec += u->pool[s] == 0; n_hh += u->pool[s] == 1; }
    if (promote >= 0) { n_rec--; n_hh++; }
    if (slot < u->cap) { if (new_pool) n_hh++; else n_rec++; }
    if (n_rec > u->n_recent || n_hh > u->n_heavy) return ORC_EINVAL;
    if (promote >= 0) u->pool[promote] = 1;
    u->last_promote = promote >= 0 ? promote : (new_pool ? -2 : -1);
    u->have_new = 0;
    if (slot == u->cap) { /* the new token leaves */
        u->last_victim_pos = u->new_pos;
        u->evicted_mass += u->score_new;
    } else {
        u->last_victim_pos = u->pos[slot];
        if (u->pos[slot] >= 0) u->evicted_mass += u->score[slot];
        u->pos[slot] = u->new_pos;
        u->pool[slot] = (signed char)new_pool;
        memcpy(u->k + (size_t)slot * u->d, u->k_new, sizeof(float) * (size_t)u->d);
        memcpy(u->v + (size_t)slot * u->d, u->v_new, sizeof(float) * (size_t)u->d);
        u->score[slot] = u->score_new;
    }
    if (u->is_prompt) u->prompt_len++;
    else u->t++;
    return ORC_OK;
}

int orc_commit(orc_unit *u, int slot)
{
    if (!u->have_new) return ORC_ESTATE;
    if (u->policy == ORC_H2O_POOLS) {
        if (slot != u->dec_slot) return ORC_EINVAL; /* orc_commit_pools takes another decision */
        return orc_commit_pools(u, slot, u->dec_pool, u->dec_promote);
    }
    if (slot < 0 || slot >= u->cap) return ORC_EINVAL;
    u->last_victim_pos = u->pos[slot];
    if (u->pos[slot] >= 0 && (u->policy == ORC_H2O || u->policy == ORC_H2O_BLOCK)) u->evicted_mass += u->score[slot];
    u->pos[slot] = u->new_pos;
    memcpy(u->k + (size_t)slot * u->d, u->k_new, sizeof(float) * (size_t)u->d);
    memcpy(u->v + (size_t)slot * u->d, u->v_new, sizeof(float) * (size_t)u->d);
    u->score[slot] = u->score_new;
    u->have_new = 0;
    if (u->is_prompt) {
        u->prompt_len++;
        return ORC_OK;
    }
    if (u->policy == ORC_RANDOM) {
        u->n_gen++;
        if (u->n_gen == u->budget + u->r) random_cut(u, u->t);
    }
    u->t++;
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Conveniences built only from the steps above.                             */
/* ------------------------------------------------------------------------ */

/* Append n prompt tokens ([n][d] each), one at a time. */
int orc_prefill(orc_unit *u, const float *k, const float *v, int n)
{
    for (int i = 0; i < n; ++i) {
        int rc = stage_prompt_token(u, k + (size_t)i * u->d, v + (size_t)i * u->d);
        if (rc) return rc;
        int slot = orc_choose(u);
        if (slot < 0) { u->have_new = 0; return ORC_ECAPACITY; }
        rc = orc_commit(u, slot);
        if (rc) return rc;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Q-seeded prefill (H2O).                                                   */
/* ------------------------------------------------------------------------ */

/* The prompt is scored by its own causal attention, then cut to the budget by
 * the greedy rule of Algorithm 1 ("h2o: heavy-hitter oracle" summary: the
 * score is the cumulative attention a token receives; remove the v whose
 * removal leaves the highest total):
 *   z_gij   = q_gi . k_j / sqrt(d)          for j <= i   (query i, key j)
 *   p_gij   = exp(z_gij - m_gi) / l_gi      softmax over j <= i
 *   score_j = (1/G) sum_g sum_{i >= j} p_gij
 * While more than K prompt tokens remain, remove the eligible v (n_sink <= pos
 * <= (P - 1) - n_recent) maximising F(T \ {v}); the scores do not change
 * between removals (no attention happens in between). The kept tokens fill
 * slots 0, 1, ... in ascending position order and keep their scores.
 * q is [G][P][d], k and v are [P][d]; scores_out (optional) receives the P
 * prompt scores before the cut. Only on an empty H2O unit. */
int orc_prefill_scored(orc_unit *u, const float *q, const float *k, const float *v, int P, double *scores_out)
{
    if (u->policy != ORC_H2O || u->prompt_len != 0 || u->t != 0 || u->have_new) return ORC_ESTATE;
    if (P < 1) return ORC_EINVAL;
    const int d = u->d, G = u->G;
    const double inv_sqrt_d = 1.0 / sqrt((double)d);
    double *score = (double *)calloc((size_t)P, sizeof(double));
    double *z = (double *)malloc(sizeof(double) * (size_t)P);
    char *alive = (char *)malloc((size_t)P);
    if (!score || !z || !alive) { free(score); free(z); free(alive); return ORC_ECAPACITY; }

    for (int g = 0; g < G; ++g) {
        for (int i = 0; i < P; ++i) {
            const float *qi = q + ((size_t)g * P + i) * d;
            double m = -INFINITY;
            for (int j = 0; j <= i; ++j) {
                double dot = 0.0;
                for (int e = 0; e < d; ++e) dot += (double)qi[e] * (double)k[(size_t)j * d + e];
                z[j] = dot * inv_sqrt_d;
                if (z[j] > m) m = z[j];
            }
            double l = 0.0;
            for (int j = 0; j <= i; ++j) l += exp(z[j] - m);
            for (int j = 0; j <= i; ++j) score[j] += exp(z[j] - m) / l;
        }
    }
    for (int j = 0; j < P; ++j) score[j] /= (double)G;
    if (scores_out) memcpy(scores_out, score, sizeof(double) * (size_t)P);

    /* Greedy cut to the budget, one removal at a time. */
    for (int j = 0; j < P; ++j) alive[j] = 1;
    int n_alive = P;
    const int last = P - 1;
    while (n_alive > u->budget) {
        double total = 0.0; /* F(T) */
        for (int j = 0; j < P; ++j)
            if (alive[j]) total += score[j];
        int best = -1, am = -1;
        double best_F = -INFINITY;
        for (int j = 0; j < P; ++j) {
            if (!alive[j] || !(j >= u->n_sink && j <= last - u->n_recent)) continue;
            double F = total - score[j];
            if (best < 0 || F > best_F || (F == best_F && (score[j] < score[best] || (score[j] == score[best] && j < best)))) {
                best = j;
                best_F = F;
            }
            if (am < 0 || score[j] < score[am] || (score[j] == score[am] && j < am)) am = j;
        }
        if (best < 0) break; /* nothing eligible: cannot happen when K = n_sink + n_heavy + n_recent */
        if (am != best) u->greedy_disagreements++;
        alive[best] = 0;
        u->evicted_mass += score[best];
        n_alive--;
    }

    int slot = 0;
    for (int j = 0; j < P && slot < u->cap; ++j) {
        if (!alive[j]) continue;
        u->pos[slot] = j;
        memcpy(u->k + (size_t)slot * d, k + (size_t)j * d, sizeof(float) * (size_t)d);
        memcpy(u->v + (size_t)slot * d, v + (size_t)j * d, sizeof(float) * (size_t)d);
        u->score[slot] = score[j];
        slot++;
    }
    u->prompt_len = P;
    free(score); free(z); free(alive);
    return ORC_OK;
}

/* The same prompt scores for the keys j >= j0 only: score_j needs the rows
 * i >= j, so only the rows i >= j0 are evaluated, each with its full softmax
 * over j' <= i. q is [G][P][d], k is [P][d]; out receives P - j0 values.
 * Independent of any unit: a sampled check of long prompts. */
int orc_prompt_tail_scores(const float *q, const float *k, int G, int P, int d, int j0, double *out)
{
    if (G < 1 || P < 1 || d < 1 || j0 < 0 || j0 >= P) return ORC_EINVAL;
    const double inv_sqrt_d = 1.0 / sqrt((double)d);
    double *z = (double *)malloc(sizeof(double) * (size_t)P);
    if (!z) return ORC_ECAPACITY;
    for (int j = j0; j < P; ++j) out[j - j0] = 0.0;
    for (int g = 0; g < G; ++g) {
        for (int i = j0; i < P; ++i) {
            const float *qi = q + ((size_t)g * P + i) * d;
            double m = -INFINITY;
            for (int j = 0; j <= i; ++j) {
                double dot = 0.0;
                for (int e = 0; e < d; ++e) dot += (double)qi[e] * (double)k[(size_t)j * d + e];
                z[j] = dot * inv_sqrt_d;
                if (z[j] > m) m = z[j];
            }
            double l = 0.0;
            for (int j = 0; j <= i; ++j) l += exp(z[j] - m);
            for (int j = j0; j <= i; ++j) out[j - j0] += exp(z[j] - m) / l;
        }
    }
    for (int j = j0; j < P; ++j) out[j - j0] /= (double)G;
    free(z);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* SnapKV prefill selection (H2O handle).                                    */
/* ------------------------------------------------------------------------ */

/* "Attention Sinks 与 KV Cache 淘汰策略" section 4.3 (SnapKV): after the prompt,
 * the last w prompt tokens (the observation window) vote for the prefix.
 *   votes_gj = sum over window queries i = P-w .. P-1 of head g of
 *              softmax_j(q_gi . k_j / sqrt(d)) over j <= i     (sum pooling)
 *   pooled_gj = max of votes_gj' over |j' - j| <= 3 within the prefix
 *              [0, P-w)                                          (max pooling, 7)
 *   each head g keeps its `topk` prefix positions with the largest pooled
 *   vote (ties: the newer position), the window is kept, and a KV head keeps
 *   the union over its G query heads.
 * The kept tokens fill slots 0, 1, ... in ascending position order; each
 * starts with score (1/G) sum_g votes_gj, the attention it received from the
 * window's queries. q_obs is [G][w][d] (the window's queries), k and v are
 * [P][d]; votes_out (optional) receives votes [G][P]. Only on an empty H2O
 * unit; ECAPACITY if the kept set does not fit the unit. */
int orc_prefill_snapkv(orc_unit *u, const float *q_obs, const float *k, const float *v, int P, int w, int topk,
                       double *votes_out)
{
    if (u->policy != ORC_H2O || u->prompt_len != 0 || u->t != 0 || u->have_new) return ORC_ESTATE;
    if (P < 1 || w < 1 || w >= P || topk < 0) return ORC_EINVAL;
    const int d = u->d, G = u->G, n_pre = P - w;
    const double inv_sqrt_d = 1.0 / sqrt((double)d);
    double *votes = (double *)calloc((size_t)G * P, sizeof(double));
    double *z = (double *)malloc(sizeof(double) * (size_t)P);
    double *pooled = (double *)malloc(sizeof(double) * (size_t)(n_pre > 0 ? n_pre : 1));
    char *kept = (char *)calloc((size_t)P, 1);
    char *taken = (char *)malloc((size_t)(n_pre > 0 ? n_pre : 1));
    if (!votes || !z || !pooled || !kept || !taken) {
        free(votes); free(z); free(pooled); free(kept); free(taken);
        return ORC_ECAPACITY;
    }
    for (int g = 0; g < G; ++g) {
        double *vg = votes + (size_t)g * P;
        for (int t = 0; t < w; ++t) {
            const int i = n_pre + t;
            const float *qi = q_obs + ((size_t)g * w + t) * d;
            double m = -INFINITY;
            for (int j = 0; j <= i; ++j) {
                double dot = 0.0;
                for (int e = 0; e < d; ++e) dot += (double)qi[e] * (double)k[(size_t)j * d + e];
                z[j] = dot * inv_sqrt_d;
                if (z[j] > m) m = z[j];
            }
            double l = 0.0;
            for (int j = 0; j <= i; ++j) l += exp(z[j] - m);
            for (int j = 0; j <= i; ++j) vg[j] += exp(z[j] - m) / l;
        }
        /* max pooling over the prefix, then this head's top-k, one at a time */
        for (int j = 0; j < n_pre; ++j) {
            double mx = -INFINITY;
            for (int jj = j - 3; jj <= j + 3; ++jj)
                if (jj >= 0 && jj < n_pre && vg[jj] > mx) mx = vg[jj];
            pooled[j] = mx;
            taken[j] = 0;
        }
        const int want = topk < n_pre ? topk : n_pre;
        for (int c = 0; c < want; ++c) {
            int best = -1;
            for (int j = 0; j < n_pre; ++j) {
                if (taken[j]) continue;
                if (best < 0 || pooled[j] > pooled[best] || (pooled[j] == pooled[best] && j > best)) best = j;
            }
            taken[best] = 1;
            kept[best] = 1;
        }
    }
    for (int j = n_pre; j < P; ++j) kept[j] = 1;
    if (votes_out) memcpy(votes_out, votes, sizeof(double) * (size_t)G * P);

    int n_kept = 0;
    for (int j = 0; j < P; ++j) n_kept += kept[j];
    int rc = ORC_OK;
    if (n_kept > u->cap) {
        rc = ORC_ECAPACITY;
    } else {
        int slot = 0;
        for (int j = 0; j < P; ++j) {
            if (!kept[j]) continue;
            double sc = 0.0;
            for (int g = 0; g < G; ++g) sc += votes[(size_t)g * P + j];
            u->pos[slot] = j;
            memcpy(u->k + (size_t)slot * d, k + (size_t)j * d, sizeof(float) * (size_t)d);
            memcpy(u->v + (size_t)slot * d, v + (size_t)j * d, sizeof(float) * (size_t)d);
            u->score[slot] = sc / (double)G;
            slot++;
        }
        u->prompt_len = P;
    }
    free(votes); free(z); free(pooled); free(kept); free(taken);
    return rc;
}

/* One full decode step with the oracle's own decision. Returns the slot taken
 * (two-pool H2O: the capacity when the new token itself left). */
int orc_step(orc_unit *u, const float *q, const float *k_new, const float *v_new, double *out)
{
    int rc = orc_attend(u, q, k_new, v_new, out);
    if (rc) return rc;
    int slot = orc_choose(u);
    if (slot < 0) { u->have_new = 0; return ORC_ECAPACITY; }
    rc = orc_commit(u, slot);
    return rc ? rc : slot;
}

/* Runs n_steps decode steps on each of n_units units, units spread over
 * n_threads threads (0 = all online cores). Inputs per unit u and step t:
 * q at q + ((u * n_steps + t) * G * d), k_new/v_new at ((u * n_steps + t) * d).
 * out (optional) like q, fp64. Returns 0 or the first error. */
typedef struct {
    orc_unit **units; int n_units, n_steps, tid, n_threads;
    const float *q, *k, *v; double *out; int rc;
} orc_job;

static void *run_job(void *arg)
{
    orc_job *j = (orc_job *)arg;
    for (int i = j->tid; i < j->n_units; i += j->n_threads) {
        orc_unit *u = j->units[i];
        size_t gd = (size_t)u->G * u->d;
        double *scratch = (double *)malloc(sizeof(double) * gd);
        for (int t = 0; t < j->n_steps; ++t) {
            size_t row = (size_t)i * j->n_steps + t;
            double *o = j->out ? j->out + row * gd : scratch;
            int rc = orc_step(u, j->q + row * gd, j->k + row * u->d, j->v + row * u->d, o);
            if (rc < 0) { j->rc = rc; break; }
        }
        free(scratch);
    }
    return NULL;
}

int orc_online_cores(void) { return (int)sysconf(_SC_NPROCESSORS_ONLN); }

int orc_run(orc_unit **units, int n_units, int n_steps, const float *q, const float *k, const float *v,
            double *out, int n_threads)
{
    if (n_threads <= 0) n_threads = orc_online_cores();
    if (n_threads > n_units) n_threads = n_units;
    if (n_threads < 1) n_threads = 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    orc_job *jobs = (orc_job *)calloc((size_t)n_threads, sizeof(orc_job));
    for (int i = 0; i < n_threads; ++i) {
        jobs[i] = (orc_job){units, n_units, n_steps, i, n_threads, q, k, v, out, 0};
        pthread_create(&th[i], NULL, run_job, &jobs[i]);
    }
    int rc = 0;
    for (int i = 0; i < n_threads; ++i) {
        pthread_join(th[i], NULL);
        if (jobs[i].rc && !rc) rc = jobs[i].rc;
    }
    free(th);
    free(jobs);
    return rc;
}
