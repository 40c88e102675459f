/*
 * CPU ORACLE -- test infrastructure only.
 *
 * A plain, slow, single-threaded restatement of what the HiSparse decode hot
 * path computes, written from the blog summary of "HiSparse: Scaling
 * Sparse-Attention Decoding with Hierarchical KV Cache Management"
 * (marsggbo.github.io, 2026-09-23).  Only the test suite, the package's smoke
 * check and the benchmark's CPU-baseline leg may load it; the product path never
 * does.  It shares no code, header or constant table with the CUDA library.
 *
 * One `orc_cache` simulates the fixed B-slot hot device buffer of ONE
 * (request, layer): a tag (logical position held, -1 = empty) and a recency
 * stamp (0 = empty) per slot, plus a clock.  Record payloads are not simulated
 * here; attention is computed from the authoritative history directly (the
 * exactness property of §3: the output over the hot buffer equals the output
 * over fully resident KV).
 *
 * Readings where the page is silent (each is listed with its reason in the
 * design notes of the repository):
 *   - which victims (§5 "parallel scan, select eviction slots", §4 LRU): the m
 *     candidates with the smallest key, key ties broken by lower slot index;
 *     key = stamp for LRU, FIFO and swap-vanilla (empty slots have stamp 0 and so
 *     go first), and for random: 0 for an empty slot, else 1 + the top 31 bits of
 *     splitmix64 at counter ((t*R + r)*L + l)*B + slot;
 *   - which miss goes to which victim: victims in ascending slot order are matched
 *     to the misses in top-k order;
 *   - stamps (§5 "hits promoted to MRU, fetched misses after the hits"): the hit
 *     of rank a among hits (top-k order) gets clock + a, the miss of rank q gets
 *     clock + h + q; FIFO stamps only misses (clock + q); then clock += k;
 *   - swap-vanilla (§4 "bring in only the current top-k, keep no hot set"): every
 *     candidate that is not a victim is emptied;
 *   - write-through append (§3 step (5)): the new record goes to the host
 *     history and into the slot that already holds its position, else the slot
 *     with the smallest key over all slots; stamp = clock, clock += 1;
 *   - invalid top-k entries (out of [0, C), or a repeat of an earlier entry) set
 *     an error bit and are treated as padding (-1);
 *   - a buffer grown on demand (§8: the coordinator allocates and grows the
 *     per-request, per-layer device cache as it is needed) holds only its first
 *     `cap` slots: resolve and append probe, evict and install among slots
 *     [0, cap) alone, the random key keeps its counter over all B slots; a
 *     buffer of fewer than k slots cannot take a step: resolve and append then
 *     set an error bit, change nothing and return -1 locations.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_LRU = 0, ORC_FIFO = 1, ORC_RANDOM = 2, ORC_SWAP = 3 };
enum { ORC_ERR_RANGE = 1, ORC_ERR_DUP = 2, ORC_ERR_CLOCK = 4, ORC_ERR_APPEND = 8, ORC_ERR_SLOTS = 128 };

typedef struct {
    int B, k, policy;
    int cap;                /* slots [0, cap) exist; B unless the buffer was grown on demand */
    uint64_t seed;
    int R, L, r, l;
    int64_t C;
    int32_t *tag;
    uint32_t *stamp;
    uint32_t clock;
    uint32_t nres;          /* resolves done so far: the step counter t of the random key */
    uint64_t hits, misses, appends;
    uint32_t err;
    int32_t *where;         /* [C]: index in the current top-k list, or -1 */
} orc_cache;

orc_cache *orc_cache_new(int B, int k, int policy, uint64_t seed, int R, int L, int r, int l, int64_t C) {
    if (B < 1 || k < 1 || k > B || C < 1 || policy < 0 || policy > 3) return NULL;
    orc_cache *c = (orc_cache *)calloc(1, sizeof(orc_cache));
    if (!c) return NULL;
    c->B = B; c->k = k; c->policy = policy; c->seed = seed; c->cap = B;
    c->R = R; c->L = L; c->r = r; c->l = l; c->C = C;
    c->tag = (int32_t *)malloc(sizeof(int32_t) * (size_t)B);
    c->stamp = (uint32_t *)calloc((size_t)B, sizeof(uint32_t));
    c->where = (int32_t *)malloc(sizeof(int32_t) * (size_t)C);
    if (!c->tag || !c->stamp || !c->where) { free(c->tag); free(c->stamp); free(c->where); free(c); return NULL; }
    for (int j = 0; j < B; ++j) c->tag[j] = -1;
    for (int64_t p = 0; p < C; ++p) c->where[p] = -1;
    c->clock = 1;
    return c;
}

/* the buffer now holds slots [0, cap), 0 <= cap <= B */
int orc_set_cap(orc_cache *c, int cap) {
    if (cap < 0 || cap > c->B) return -1;
    c->cap = cap;
    return 0;
}

void orc_cache_free(orc_cache *c) {
    if (!c) return;
    free(c->tag); free(c->stamp); free(c->where); free(c);
}

/* splitmix64's output function applied at counter n: mix(seed + n * golden gamma) */
static uint64_t orc_splitmix_at(uint64_t seed, uint64_t n) {
    uint64_t z = seed + n * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* eviction key of slot j (smaller = evicted first) */
static uint32_t orc_key(const orc_cache *c, int j) {
    if (c->policy == ORC_RANDOM) {
        if (c->tag[j] < 0) return 0;
        uint64_t n = (((uint64_t)c->nres * (uint64_t)c->R + (uint64_t)c->r) * (uint64_t)c->L + (uint64_t)c->l)
                         * (uint64_t)c->B + (uint64_t)j;
        return 1u + (uint32_t)(orc_splitmix_at(c->seed, n) >> 33);
    }
    return c->stamp[j];
}

typedef struct { uint32_t key; int32_t slot; } orc_ks;

static int orc_cmp_ks(const void *a, const void *b) {
    const orc_ks *x = (const orc_ks *)a, *y = (const orc_ks *)b;
    if (x->key != y->key) return x->key < y->key ? -1 : 1;
    return (x->slot > y->slot) - (x->slot < y->slot);
}

static int orc_cmp_int(const void *a, const void *b) {
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/*
 * valid[i] = 1 when S[i] is a usable selection: in [0, C) and not equal to any
 * earlier entry.  Returns the error bits for the bad entries.
 */
uint32_t orc_validate(const int32_t *S, int k, int64_t C, uint8_t *valid) {
    uint32_t err = 0;
    for (int i = 0; i < k; ++i) {
        valid[i] = 0;
        if (S[i] == -1) continue;
        if (S[i] < 0 || (int64_t)S[i] >= C) { err |= ORC_ERR_RANGE; continue; }
        int repeat = 0;
        for (int j = 0; j < i && !repeat; ++j) repeat = (S[j] == S[i]);
        if (repeat) { err |= ORC_ERR_DUP; continue; }
        valid[i] = 1;
    }
    return err;
}

/*
 * RESOLVE one step (§3 and §5 of the HiSparse summary): look the selected
 * positions up in the hot buffer, keep the hits, evict victims for the misses,
 * install the misses, update the stamps.  locs[i] = slot of S[i] after the step,
 * or -1 for padding / invalid entries.  Returns the number of misses, or -1 when
 * the buffer holds fewer than k slots.
 */
int orc_resolve(orc_cache *c, const int32_t *S, int32_t *locs) {
    const int B = c->cap, k = c->k;
    if (B < k) {  /* too few slots for a step */
        c->err |= ORC_ERR_SLOTS;
        for (int i = 0; i < k; ++i) locs[i] = -1;
        return -1;
    }
    uint8_t *valid = (uint8_t *)malloc((size_t)k);
    int32_t *hit_slot = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
    uint8_t *slot_hit = (uint8_t *)calloc((size_t)B, 1);
    orc_ks *cand = (orc_ks *)malloc(sizeof(orc_ks) * (size_t)B);
    int32_t *victims = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);

    c->err |= orc_validate(S, k, c->C, valid);
    if ((uint64_t)c->clock + (uint64_t)k >= 0xFFFFFFFFull) c->err |= ORC_ERR_CLOCK;

    /* hash of the selected positions: where[pos] = index in S */
    for (int i = 0; i < k; ++i) if (valid[i]) c->where[S[i]] = i;

    /* probe every slot */
    for (int i = 0; i < k; ++i) hit_slot[i] = -1;
    for (int j = 0; j < B; ++j) {
        int32_t t = c->tag[j];
        if (t >= 0 && c->where[t] >= 0) { hit_slot[c->where[t]] = j; slot_hit[j] = 1; }
    }
    int h = 0, m = 0;
    for (int i = 0; i < k; ++i) {
        if (!valid[i]) continue;
        if (hit_slot[i] >= 0) h++; else m++;
    }

    /* candidates: slots holding no selected position; the m with the smallest keys are victims */
    int nc = 0;
    for (int j = 0; j < B; ++j) if (!slot_hit[j]) { cand[nc].key = orc_key(c, j); cand[nc].slot = j; nc++; }
    qsort(cand, (size_t)nc, sizeof(orc_ks), orc_cmp_ks);
    for (int q = 0; q < m; ++q) victims[q] = cand[q].slot;
    qsort(victims, (size_t)m, sizeof(int32_t), orc_cmp_int);
    if (c->policy == ORC_SWAP) {
        for (int q = m; q < nc; ++q) { c->tag[cand[q].slot] = -1; c->stamp[cand[q].slot] = 0; }
    }

    /* install misses (top-k order -> ascending victim slots) and stamp */
    int a = 0, q = 0;
    for (int i = 0; i < k; ++i) {
        if (!valid[i]) { locs[i] = -1; continue; }
        if (hit_slot[i] >= 0) {
            int j = hit_slot[i];
            if (c->policy != ORC_FIFO) c->stamp[j] = c->clock + (uint32_t)a;
            locs[i] = j;
            a++;
        } else {
            int j = victims[q];
            c->tag[j] = S[i];
            c->stamp[j] = c->policy == ORC_FIFO ? c->clock + (uint32_t)q : c->clock + (uint32_t)h + (uint32_t)q;
            locs[i] = j;
            q++;
        }
    }
    c->clock += (uint32_t)k;
    c->hits += (uint64_t)h;
    c->misses += (uint64_t)m;
    c->nres += 1;
    for (int i = 0; i < k; ++i) if (valid[i]) c->where[S[i]] = -1;

    free(valid); free(hit_slot); free(slot_hit); free(cand); free(victims);
    return m;
}

/*
 * Write-through append of position p (§3 step (5)): returns the slot that now
 * holds p, or -1 (and an error bit) when p is outside [0, C) or the buffer holds
 * fewer than k slots.
 */
int orc_append(orc_cache *c, int64_t p) {
    if (p < 0 || p >= c->C) { c->err |= ORC_ERR_APPEND; return -1; }
    if ((uint64_t)c->clock + 1u >= 0xFFFFFFFFull) c->err |= ORC_ERR_CLOCK;
    if (c->cap < c->k) { c->err |= ORC_ERR_SLOTS; return -1; }
    int slot = -1;
    for (int j = 0; j < c->cap; ++j) if (c->tag[j] == (int32_t)p) slot = j;
    if (slot < 0) {
        slot = 0;
        uint32_t best = orc_key(c, 0);
        for (int j = 1; j < c->cap; ++j) {
            uint32_t kj = orc_key(c, j);
            if (kj < best) { best = kj; slot = j; }
        }
    }
    c->tag[slot] = (int32_t)p;
    c->stamp[slot] = c->clock;
    c->clock += 1;
    c->appends += 1;
    return slot;
}

void orc_get_slots(const orc_cache *c, int32_t *tag, uint32_t *stamp) {
    memcpy(tag, c->tag, sizeof(int32_t) * (size_t)c->B);
    memcpy(stamp, c->stamp, sizeof(uint32_t) * (size_t)c->B);
}

/* counters: [clock, nres, err, hits, misses, appends] */
void orc_get_counters(const orc_cache *c, uint64_t *out6) {
    out6[0] = c->clock; out6[1] = c->nres; out6[2] = c->err;
    out6[3] = c->hits; out6[4] = c->misses; out6[5] = c->appends;
}

/*
 * Belady's offline rule (§4: the policy that knows the future and evicts the
 * entry whose next use is farthest away).  Runs a whole no-append trace
 * S[T][k] on a B-slot buffer; misses[t] per step.  Victims: empty slots first
 * (lowest slot first), then positions never selected again (lowest slot
 * first), then the farthest next use.  Returns the total.
 */
int64_t orc_belady(int B, int k, int T, int64_t C, const int32_t *S, int32_t *misses) {
    int32_t *tag = (int32_t *)malloc(sizeof(int32_t) * (size_t)B);
    int64_t *next_use = (int64_t *)malloc(sizeof(int64_t) * (size_t)B);
    int32_t *where = (int32_t *)malloc(sizeof(int32_t) * (size_t)C);
    int64_t *nxt = (int64_t *)malloc(sizeof(int64_t) * (size_t)T * (size_t)k); /* next step selecting S[t][i] */
    int64_t *last = (int64_t *)malloc(sizeof(int64_t) * (size_t)C);
    uint8_t *valid = (uint8_t *)malloc((size_t)k);
    int32_t *hit_slot = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
    uint8_t *slot_hit = (uint8_t *)malloc((size_t)B);
    int64_t *ckey = (int64_t *)malloc(sizeof(int64_t) * (size_t)B);
    int32_t *cslot = (int32_t *)malloc(sizeof(int32_t) * (size_t)B);
    const int64_t NEVER = INT64_MAX / 4, EMPTY = INT64_MAX / 2;
    for (int j = 0; j < B; ++j) { tag[j] = -1; next_use[j] = EMPTY; }
    for (int64_t p = 0; p < C; ++p) { where[p] = -1; last[p] = NEVER; }
    for (int t = T - 1; t >= 0; --t) {
        orc_validate(S + (size_t)t * k, k, C, valid);
        for (int i = 0; i < k; ++i) {
            int32_t p = S[(size_t)t * k + i];
            if (!valid[i]) { nxt[(size_t)t * k + i] = NEVER; continue; }
            nxt[(size_t)t * k + i] = last[p];
        }
        for (int i = 0; i < k; ++i) if (valid[i]) last[S[(size_t)t * k + i]] = t;
    }
    int64_t total = 0;
    for (int t = 0; t < T; ++t) {
        const int32_t *St = S + (size_t)t * k;
        orc_validate(St, k, C, valid);
        for (int i = 0; i < k; ++i) if (valid[i]) where[St[i]] = i;
        for (int i = 0; i < k; ++i) hit_slot[i] = -1;
        for (int j = 0; j < B; ++j) {
            slot_hit[j] = 0;
            if (tag[j] >= 0 && where[tag[j]] >= 0) { hit_slot[where[tag[j]]] = j; slot_hit[j] = 1; }
        }
        int m = 0;
        for (int i = 0; i < k; ++i) if (valid[i] && hit_slot[i] < 0) m++;
        /* pick the m candidates with the largest next use (ties: lower slot) by repeated scans */
        int nc = 0;
        for (int j = 0; j < B; ++j) if (!slot_hit[j]) { ckey[nc] = next_use[j]; cslot[nc] = j; nc++; }
        int q = 0;
        for (int i = 0; i < k; ++i) {
            if (!valid[i]) continue;
            if (hit_slot[i] >= 0) { next_use[hit_slot[i]] = nxt[(size_t)t * k + i]; continue; }
            int best = -1;
            for (int x = 0; x < nc; ++x) {
                if (cslot[x] < 0) continue;
                if (best < 0 || ckey[x] > ckey[best]) best = x;
            }
            int j = cslot[best];
            cslot[best] = -1;
            tag[j] = St[i];
            next_use[j] = nxt[(size_t)t * k + i];
            q++;
        }
        for (int i = 0; i < k; ++i) if (valid[i]) where[St[i]] = -1;
        if (misses) misses[t] = m;
        total += m;
    }
    free(tag); free(next_use); free(where); free(nxt); free(last); free(valid);
    free(hit_slot); free(slot_hit); free(ckey); free(cslot);
    return total;
}

/* bf16 bit pattern -> double, exactly (a bf16 is the top half of an IEEE binary32) */
static double orc_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Exact attention of one request's queries over the selected positions (§3:
 * the selected set, scores and outputs are those of full-resident KV).
 *   q    : [Hq][Dqk] bf16 bits
 *   hist : [C][rec_elems] bf16 bits, the authoritative history of this (request, layer)
 *   S    : [k] positions (-1 = padding; invalid entries are ignored like padding)
 *   out  : [Hq][Dv] double
 * Record layout:
 *   MLA (kv_heads == 0): one shared latent of Dqk values; K = all Dqk, V = the first Dv.
 *   GQA (kv_heads  > 0): kv_heads blocks of [K (Dqk) | V (Dv)]; query head h reads
 *                        block h / (Hq / kv_heads).
 * logits_i = scale * <q_h, K_i>; p = softmax over the valid i; out_h = sum_i p_i V_i.
 * With no valid entry the output is 0.
 */
void orc_attention(int Hq, int kv_heads, int Dqk, int Dv, const uint16_t *q, const uint16_t *hist,
                   int64_t rec_elems, int64_t C, const int32_t *S, int k, double scale, double *out) {
    uint8_t *valid = (uint8_t *)malloc((size_t)k);
    double *logit = (double *)malloc(sizeof(double) * (size_t)k);
    orc_validate(S, k, C, valid);
    const int group = kv_heads > 0 ? Hq / kv_heads : Hq;
    for (int h = 0; h < Hq; ++h) {
        const int64_t koff = kv_heads > 0 ? (int64_t)(h / group) * (Dqk + Dv) : 0;
        const int64_t voff = kv_heads > 0 ? koff + Dqk : 0;
        double mx = -INFINITY;
        int any = 0;
        for (int i = 0; i < k; ++i) {
            if (!valid[i]) continue;
            const uint16_t *rec = hist + (int64_t)S[i] * rec_elems;
            double s = 0.0;
            for (int d = 0; d < Dqk; ++d) s += orc_bf16(q[(int64_t)h * Dqk + d]) * orc_bf16(rec[koff + d]);
            logit[i] = scale * s;
            if (logit[i] > mx) mx = logit[i];
            any = 1;
        }
        for (int d = 0; d < Dv; ++d) out[(int64_t)h * Dv + d] = 0.0;
        if (!any) continue;
        double den = 0.0;
        for (int i = 0; i < k; ++i) {
            if (!valid[i]) continue;
            double p = exp(logit[i] - mx);
            den += p;
            const uint16_t *rec = hist + (int64_t)S[i] * rec_elems;
            for (int d = 0; d < Dv; ++d) out[(int64_t)h * Dv + d] += p * orc_bf16(rec[voff + d]);
        }
        for (int d = 0; d < Dv; ++d) out[(int64_t)h * Dv + d] /= den;
    }
    free(valid); free(logit);
}
