/*
 * Seeded synthetic top-k selection traces.
 *
 * This file is an INPUT GENERATOR: it stands in for a sparse-attention indexer
 * (DSA / NSA / Quest in "HiSparse: Scaling Sparse-Attention Decoding with
 * Hierarchical KV Cache Management", §3) that hands the KV-cache layer a list of
 * k distinct logical token positions per (request, layer, decode step).  It holds
 * none of the cache method's arithmetic: both the CPU oracle and the CUDA path
 * receive its output as plain int32 arrays.
 *
 * The blog summary of HiSparse (§4) says consecutive top-k sets overlap heavily
 * and drift slowly, and that recency predicts reuse.  The generator models that:
 *   step 0     : the newest position plus k-1 distinct uniform positions;
 *   step t > 0 : keep round(keep*k) entries of the previous list (uniformly
 *                chosen), add the newest position, refill to k with a mix of
 *                recency-biased draws (geometric offset back from the newest
 *                position, mean `recency_mean`) and uniform draws;
 *   burst      : every `burst_every` steps a contiguous span of round(burst_frac*k)
 *                positions, starting uniformly in a region at least `far_gap`
 *                tokens behind the newest, replaces that many entries;
 *   finally the list is shuffled (an indexer does not sort its output).
 *
 * Random numbers: xoshiro256** (Blackman and Vigna, "Scrambled linear
 * pseudorandom number generators", 2018), seeded with four outputs of
 * splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", 2014).  Both are written here from their published definitions.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct { uint64_t s[4]; } tg_rng;

static uint64_t tg_splitmix64(uint64_t *state) {
    uint64_t z = (*state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static uint64_t tg_rotl(uint64_t x, int r) { return (x << r) | (x >> (64 - r)); }

static uint64_t tg_next(tg_rng *g) {
    uint64_t *s = g->s;
    uint64_t out = tg_rotl(s[1] * 5u, 7) * 9u;
    uint64_t t = s[1] << 17;
    s[2] ^= s[0];
    s[3] ^= s[1];
    s[1] ^= s[2];
    s[0] ^= s[3];
    s[2] ^= t;
    s[3] = tg_rotl(s[3], 45);
    return out;
}

static void tg_seed(tg_rng *g, uint64_t seed) {
    uint64_t st = seed;
    for (int i = 0; i < 4; ++i) g->s[i] = tg_splitmix64(&st);
}

/* uniform integer in [0, n) by the high half of a 64x64-bit product */
static int64_t tg_below(tg_rng *g, int64_t n) {
    unsigned __int128 prod = (unsigned __int128)tg_next(g) * (unsigned __int128)(uint64_t)n;
    return (int64_t)(uint64_t)(prod >> 64);
}

/* uniform double in [0, 1) from the top 53 bits */
static double tg_unit(tg_rng *g) { return (double)(tg_next(g) >> 11) * (1.0 / 9007199254740992.0); }

typedef struct {
    int64_t ctx0;          /* positions [0, ctx0) exist before step 0 */
    int appends;           /* 1: the context grows by one token per step, appended before the step */
    int k;                 /* entries per list */
    int steps;
    double keep;           /* fraction of the previous list kept */
    double recency_mean;   /* mean geometric offset back from the newest position */
    double recency_share;  /* share of refill draws that are recency-biased */
    int burst_every;       /* 0 = no bursts */
    double burst_frac;
    int64_t far_gap;       /* a burst span starts at least this far behind the newest */
} tg_params;

/* byte-per-position membership set, cleared entry by entry */
typedef struct { uint8_t *in; } tg_set;

/* One trace: out[steps][k].  Returns 0, or -1 on bad parameters / no memory. */
static int tg_one(const tg_params *P, uint64_t seed, int32_t *out) {
    const int k = P->k;
    const int64_t maxpos = P->ctx0 + (P->appends ? P->steps : 0);
    if (k < 1 || P->ctx0 < 1 || k > P->ctx0 + (P->appends ? 1 : 0) || P->steps < 1) return -1;
    tg_rng g;
    tg_seed(&g, seed);
    uint8_t *in = (uint8_t *)calloc((size_t)maxpos + 1, 1);
    int32_t *cur = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
    int32_t *tmp = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
    if (!in || !cur || !tmp) { free(in); free(cur); free(tmp); return -1; }
    const double lq = (P->recency_mean > 1.0) ? log(1.0 - 1.0 / P->recency_mean) : 0.0;
    int len = 0;
    for (int t = 0; t < P->steps; ++t) {
        const int64_t n = P->ctx0 + (P->appends ? (int64_t)t + 1 : 0);
        const int32_t newest = (int32_t)(n - 1);
        if (t == 0) {
            len = 0;
            cur[len++] = newest;
            in[newest] = 1;
            while (len < k) {
                int64_t p = tg_below(&g, n);
                if (!in[p]) { in[p] = 1; cur[len++] = (int32_t)p; }
            }
        } else {
            int keep_n = (int)llround(P->keep * (double)k);
            if (keep_n < 0) keep_n = 0;
            if (keep_n > k) keep_n = k;
            for (int i = 0; i < keep_n; ++i) {  /* partial Fisher-Yates: a uniform keep_n-subset */
                int j = i + (int)tg_below(&g, k - i);
                int32_t s = cur[i]; cur[i] = cur[j]; cur[j] = s;
            }
            int newest_kept = 0;
            for (int i = 0; i < keep_n; ++i) newest_kept |= (cur[i] == newest);
            if (!newest_kept && keep_n == k) keep_n = k - 1;
            for (int i = 0; i < k; ++i) in[cur[i]] = 0;
            len = keep_n;
            for (int i = 0; i < len; ++i) in[cur[i]] = 1;
            if (!in[newest]) { in[newest] = 1; cur[len++] = newest; }
            while (len < k) {
                int placed = 0;
                if (tg_unit(&g) < P->recency_share && lq < 0.0) {
                    for (int tries = 0; tries < 64 && !placed; ++tries) {
                        double u = 1.0 - tg_unit(&g); /* (0, 1] */
                        int64_t d = 1 + (int64_t)floor(log(u) / lq);
                        int64_t p = (int64_t)newest - d;
                        if (p >= 0 && !in[p]) { in[p] = 1; cur[len++] = (int32_t)p; placed = 1; }
                    }
                }
                while (!placed) {
                    int64_t p = tg_below(&g, n);
                    if (!in[p]) { in[p] = 1; cur[len++] = (int32_t)p; placed = 1; }
                }
            }
            if (P->burst_every > 0 && t % P->burst_every == 0) {
                int span = (int)llround(P->burst_frac * (double)k);
                if (span > k - 1) span = k - 1;
                if (span > 0) {
                    int64_t hi = n - P->far_gap - span;
                    if (hi < 0) hi = 0;
                    if (hi + span > n - 1) hi = n - 1 - span;
                    if (hi < 0) hi = 0;
                    int64_t a = tg_below(&g, hi + 1);
                    for (int i = 0; i < len; ++i) in[cur[i]] = 0;
                    int m = 0;
                    for (int64_t p = a; p < a + span; ++p) { tmp[m++] = (int32_t)p; in[p] = 1; }
                    if (!in[newest]) { tmp[m++] = newest; in[newest] = 1; }
                    for (int i = 0; i < len && m < k; ++i) {
                        if (!in[cur[i]]) { in[cur[i]] = 1; tmp[m++] = cur[i]; }
                    }
                    /* the span can only shrink the list if it overlapped kept entries; refill uniformly */
                    while (m < k) {
                        int64_t p = tg_below(&g, n);
                        if (!in[p]) { in[p] = 1; tmp[m++] = (int32_t)p; }
                    }
                    memcpy(cur, tmp, sizeof(int32_t) * (size_t)k);
                    len = k;
                }
            }
        }
        for (int i = k - 1; i > 0; --i) {  /* full shuffle */
            int j = (int)tg_below(&g, i + 1);
            int32_t s = cur[i]; cur[i] = cur[j]; cur[j] = s;
        }
        memcpy(out + (size_t)t * (size_t)k, cur, sizeof(int32_t) * (size_t)k);
    }
    free(in); free(cur); free(tmp);
    return 0;
}

/*
 * Traces for a batch: out[steps][num_layers][num_requests][k] int32, the order in which a
 * decode step consumes them (one [R][k] block per layer).  The trace of (r, l)
 * uses seed base_seed + r * 65536 + l.
 */
int tg_drift_traces(uint64_t base_seed, int num_requests, int num_layers, int64_t ctx0, int appends,
                    int k, int steps, double keep, double recency_mean, double recency_share,
                    int burst_every, double burst_frac, int64_t far_gap, int32_t *out) {
    tg_params P = {ctx0, appends, k, steps, keep, recency_mean, recency_share, burst_every, burst_frac, far_gap};
    int32_t *one = (int32_t *)malloc(sizeof(int32_t) * (size_t)k * (size_t)steps);
    if (!one) return -1;
    for (int r = 0; r < num_requests; ++r) {
        for (int l = 0; l < num_layers; ++l) {
            if (tg_one(&P, base_seed + (uint64_t)r * 65536u + (uint64_t)l, one) != 0) { free(one); return -1; }
            for (int t = 0; t < steps; ++t) {
                int32_t *dst = out + (((size_t)t * (size_t)num_layers + (size_t)l) * (size_t)num_requests + (size_t)r) * (size_t)k;
                memcpy(dst, one + (size_t)t * (size_t)k, sizeof(int32_t) * (size_t)k);
            }
        }
    }
    free(one);
    return 0;
}

/* Raw generator output, for pinning the generators against their published test values. */
void tg_xoshiro_stream(uint64_t seed, int n, uint64_t *out) {
    tg_rng g;
    tg_seed(&g, seed);
    for (int i = 0; i < n; ++i) out[i] = tg_next(&g);
}

void tg_splitmix_stream(uint64_t seed, int n, uint64_t *out) {
    uint64_t st = seed;
    for (int i = 0; i < n; ++i) out[i] = tg_splitmix64(&st);
}
