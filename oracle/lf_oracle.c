/*
 * fp64 CPU oracle of one LongFlow decode step.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package's smoke check and the
 * CPU-baseline leg of the benchmark may load or run this file. The CUDA
 * library never calls it, and the two share no code: no headers, no helpers,
 * no tables.
 *
 * What it computes follows "LongFlow: Efficient KV Cache Compression for
 * Reasoning Models":
 *   - Fig. 2 (Left): the current token's K/V covers the slot chosen at the
 *     previous step; then the static KV and its Mask go to the kernel with Q,
 *     which returns the attention output and the slot to cover next.
 *   - Fig. 2 (Middle): the mask gates which cached slots take part.
 *   - Fig. 2 (Right): P.V is split in two steps. The intermediate G is the
 *     elementwise product G[h][j][c] = p[h][j] * v[j][c]; the output is its sum
 *     over slots, and LongFlowScore is read off G.
 *   - Fig. 1 caption and abstract: one token is evicted after every attention
 *     call, scored with the current query only.
 * The paper prints no formula for the score. This oracle uses the definition
 *   I_j = sum over the heads h of the KV group, sum over c, of |p[h][j] * v[j][c]|
 * with p the final normalised softmax weight. The slot to evict next is the
 * argmin of I_j over live slots whose age is at least W, ties to the lowest
 * slot index, -1 when no slot qualifies.
 *
 * Readings where the paper is silent (all shared with the CUDA library's
 * documentation, none shared as code):
 *   - mask: one int32 per (b, kvh, slot); negative = empty/masked, never
 *     attended or selected; >= 0 = age of the slot in decode steps.
 *   - the write: if 0 <= write_slot < S, the new K/V row replaces the slot, its
 *     age becomes 0 and the slot is live from then on; every other live slot
 *     ages by one (saturating). write_slot = -1 means no write, and no ageing.
 *     Any other value is counted as invalid and treated as -1.
 *   - write before attend: the current token takes part in this step's
 *     attention (Fig. 2 Left).
 *   - GQA: query head h uses KV head floor(h / g), g = Hq / Hkv.
 *   - scale multiplies the logits; nothing else (no RoPE, bias or softcap)
 *     happens inside the step.
 *   - a unit with no live slot writes an all-zero output.
 *
 * Arithmetic: bf16 inputs are widened exactly to double; everything after is
 * double. The output is returned in double, not rounded to bf16.
 *
 * Plain loops, no blocking, no fusion beyond what the definition states. One
 * OpenMP thread per (b, kvh) unit at a time.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* What a step returns besides the output (see lfo_decode_step_ex). */
typedef struct {
    int topk;           /* slots returned per unit */
    int fill_first;     /* empty slots are returned first, lowest index first */
    int mask_evicted;   /* returned slots get mask -1 */
    int attention_only; /* no score, no selection, no ageing */
} oracle_opts;

/* A selection candidate: class 0 = empty slot (fill), class 1 = scored slot. */
typedef struct {
    int cls;
    double score;
    int slot;
} candidate;

/* Ascending (class, score, slot): the plain order the selection follows. */
static int cmp_candidate(const void* pa, const void* pb) {
    const candidate* a = (const candidate*)pa;
    const candidate* b = (const candidate*)pb;
    if (a->cls != b->cls) return a->cls < b->cls ? -1 : 1;
    if (a->score != b->score) return a->score < b->score ? -1 : 1;
    return (a->slot > b->slot) - (a->slot < b->slot);
}

/* Widen a bf16 bit pattern to double (exact). */
static double bf16_to_double(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* One (b, kvh) unit. Returns 1 if its write slot was invalid, 0 otherwise,
 * -1 on allocation failure. */
static int oracle_unit(int b, int kvh, const uint16_t* q, uint16_t* k_cache, uint16_t* v_cache,
                       int32_t* mask, const uint16_t* new_k, const uint16_t* new_v,
                       const int32_t* write_slot, double* out, int32_t* next_slot,
                       double* p_out, double* score_out, int Hq, int Hkv, int d, int S, int W,
                       double scale, const oracle_opts* opt) {
    const int g = Hq / Hkv;
    const size_t unit = (size_t)b * Hkv + kvh;
    uint16_t* K = k_cache + unit * (size_t)S * d;
    uint16_t* V = v_cache + unit * (size_t)S * d;
    int32_t* age = mask + unit * (size_t)S;
    int invalid = 0;

    /* Step 1: the slot write (Fig. 2 Left). */
    int ws = write_slot[unit];
    if (ws != -1 && (ws < 0 || ws >= S)) {
        invalid = 1;
        ws = -1;
    }
    if (ws >= 0) {
        memcpy(K + (size_t)ws * d, new_k + unit * (size_t)d, sizeof(uint16_t) * (size_t)d);
        memcpy(V + (size_t)ws * d, new_v + unit * (size_t)d, sizeof(uint16_t) * (size_t)d);
        if (opt->attention_only) {
            /* Attention alone: the written slot is live; nothing else ages. */
            if (age[ws] < 0) age[ws] = 0;
        } else {
            for (int j = 0; j < S; ++j) {
                if (j == ws)
                    age[j] = 0;
                else if (age[j] >= 0 && age[j] < INT32_MAX)
                    age[j] += 1;
            }
        }
    }

    double* s = (double*)malloc(sizeof(double) * (size_t)S);
    double* p = (double*)malloc(sizeof(double) * (size_t)S);
    double* G = (double*)malloc(sizeof(double) * (size_t)S * d);
    double* I = (double*)calloc((size_t)S, sizeof(double));
    if (!s || !p || !G || !I) {
        free(s); free(p); free(G); free(I);
        return -1;
    }

    for (int h = 0; h < g; ++h) {
        const int hq = kvh * g + h;
        const uint16_t* qh = q + ((size_t)b * Hq + hq) * d;
        double* o = out + ((size_t)b * Hq + hq) * d;

        /* Step 2: logits S = scale * q . k over live slots (Fig. 2 Right). */
        double smax = -INFINITY;
        int nlive = 0;
        for (int j = 0; j < S; ++j) {
            if (age[j] < 0) continue;
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += bf16_to_double(qh[c]) * bf16_to_double(K[(size_t)j * d + c]);
            s[j] = scale * acc;
            if (s[j] > smax) smax = s[j];
            ++nlive;
        }

        /* Step 3: P = softmax(S) over live slots; masked slots weigh 0. */
        double l = 0.0;
        for (int j = 0; j < S; ++j) {
            p[j] = 0.0;
            if (age[j] < 0) continue;
            p[j] = exp(s[j] - smax);
            l += p[j];
        }
        for (int j = 0; j < S; ++j)
            if (age[j] >= 0) p[j] /= l;

        /* Step 4, first half of the split P.V: G[j][c] = p[j] * v[j][c]. */
        for (int j = 0; j < S; ++j)
            for (int c = 0; c < d; ++c)
                G[(size_t)j * d + c] =
                    (age[j] >= 0) ? p[j] * bf16_to_double(V[(size_t)j * d + c]) : 0.0;

        /* Step 4, second half: O[c] = sum_j G[j][c]. */
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int j = 0; j < S; ++j) acc += G[(size_t)j * d + c];
            o[c] = (nlive > 0) ? acc : 0.0;
        }

        /* Step 5, LongFlowScore read off G: I_j += sum_c |G[j][c]|. */
        for (int j = 0; j < S; ++j) {
            if (age[j] < 0) continue;
            double acc = 0.0;
            for (int c = 0; c < d; ++c) acc += fabs(G[(size_t)j * d + c]);
            I[j] += acc;
        }

        if (p_out)
            for (int j = 0; j < S; ++j) p_out[((size_t)b * Hq + hq) * S + j] = p[j];
    }

    if (score_out)
        for (int j = 0; j < S; ++j)
            score_out[unit * (size_t)S + j] = (age[j] >= 0) ? I[j] : INFINITY;

    /* Step 6: evict. The candidates are the live slots with age >= W (and,
     * when filling first, the empty slots, ranked before every score). They
     * are sorted by (class, I, slot) and the first topk are returned: topk = 1
     * is the argmin of I with ties to the lowest slot. */
    if (!opt->attention_only) {
        candidate* cand = (candidate*)malloc(sizeof(candidate) * (size_t)S);
        if (!cand) {
            free(s); free(p); free(G); free(I);
            return -1;
        }
        int nc = 0;
        for (int j = 0; j < S; ++j) {
            if (age[j] >= 0 && age[j] >= W) {
                cand[nc].cls = 1; cand[nc].score = I[j]; cand[nc].slot = j; ++nc;
            } else if (age[j] < 0 && opt->fill_first) {
                cand[nc].cls = 0; cand[nc].score = 0.0; cand[nc].slot = j; ++nc;
            }
        }
        qsort(cand, (size_t)nc, sizeof(candidate), cmp_candidate);
        for (int i = 0; i < opt->topk; ++i) {
            const int slot = (i < nc) ? cand[i].slot : -1;
            next_slot[unit * (size_t)opt->topk + i] = slot;
            if (slot >= 0 && opt->mask_evicted) age[slot] = -1;
        }
        free(cand);
    }

    free(s); free(p); free(G); free(I);
    return invalid;
}

/*
 * One decode step over the whole batch, with a choice of what it returns.
 *
 * q [B][Hq][d], new_k/new_v [B][Hkv][d]: bf16 bits. k_cache/v_cache
 * [B][Hkv][S][d] bf16 bits and mask [B][Hkv][S] are updated in place.
 * write_slot [B][Hkv]. out [B][Hq][d] double.
 * next_slots [B][Hkv][topk]: the topk candidates in ascending (class, score,
 * slot) order, -1 past the last; untouched when attention_only.
 * p_out [B][Hq][S] (optional): final softmax weights, 0 on masked slots.
 * score_out [B][Hkv][S] (optional): I_j on live slots, +inf on masked slots.
 * fill_first: empty slots are candidates ranked before every score (the
 * cache-fill phase). mask_evicted: returned slots get mask -1. topk > 1: the
 * periodic k-at-once compression. attention_only: write and attend only.
 * units/n_units (optional): process only these unit indices (b * Hkv + kvh);
 * outputs of other units are left untouched.
 *
 * Returns the number of invalid write slots seen (>= 0), -1 for bad arguments,
 * -2 if memory ran out.
 */
int lfo_decode_step_ex(const uint16_t* q, uint16_t* k_cache, uint16_t* v_cache, int32_t* mask,
                       const uint16_t* new_k, const uint16_t* new_v, const int32_t* write_slot,
                       double* out, int32_t* next_slots, double* p_out, double* score_out,
                       int B, int Hq, int Hkv, int d, int S, int W, float scale, int topk,
                       int fill_first, int mask_evicted, int attention_only, int nthreads,
                       const int32_t* units, int n_units) {
    if (!q || !k_cache || !v_cache || !mask || !new_k || !new_v || !write_slot || !out)
        return -1;
    if (!attention_only && !next_slots) return -1;
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || d < 1 || S < 1 || W < 0 || topk < 1)
        return -1;
    const int total = (units != NULL) ? n_units : B * Hkv;
    if (units != NULL)
        for (int i = 0; i < n_units; ++i)
            if (units[i] < 0 || units[i] >= B * Hkv) return -1;
    const oracle_opts opt = {topk, fill_first != 0, mask_evicted != 0, attention_only != 0};
    const double dscale = (double)scale;
    int invalid = 0, oom = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(+ : invalid, oom)
#endif
    for (int i = 0; i < total; ++i) {
        const int u = (units != NULL) ? units[i] : i;
        const int r = oracle_unit(u / Hkv, u % Hkv, q, k_cache, v_cache, mask, new_k, new_v,
                                  write_slot, out, next_slots, p_out, score_out, Hq, Hkv, d, S,
                                  W, dscale, &opt);
        if (r < 0)
            oom += 1;
        else
            invalid += r;
    }
    (void)nthreads;
    return oom ? -2 : invalid;
}

/* The LongFlow step as in the paper: one evicted slot per unit (the argmin). */
int lfo_decode_step(const uint16_t* q, uint16_t* k_cache, uint16_t* v_cache, int32_t* mask,
                    const uint16_t* new_k, const uint16_t* new_v, const int32_t* write_slot,
                    double* out, int32_t* next_slot, double* p_out, double* score_out, int B,
                    int Hq, int Hkv, int d, int S, int W, float scale, int nthreads,
                    const int32_t* units, int n_units) {
    if (!next_slot) return -1;
    return lfo_decode_step_ex(q, k_cache, v_cache, mask, new_k, new_v, write_slot, out, next_slot,
                              p_out, score_out, B, Hq, Hkv, d, S, W, scale, 1, 0, 0, 0, nthreads,
                              units, n_units);
}

/* Threads the oracle would use for nthreads <= 0. */
int lfo_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
