/*
 * hs_oracle.c -- CPU oracle for HiSparse's fused per-layer swap-in resolution.
 *
 * TEST INFRASTRUCTURE. Only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg may load this file's library. It shares no code, header, table or
 * helper with the CUDA path; it is plain, single-threaded, slow-on-purpose C that a
 * reader can check against the pages by eye.
 *
 * What it computes (HiSparse paper abstract; blog commentary sections two and three):
 * every request keeps its full KV history in host memory and a small fixed-size
 * cache of S device slots; for each layer and decode step, the k selected positions
 * of a request are resolved by (1) hit detection through a position->slot page
 * table, (2) LRU replacement for the misses, (3) the page-table update and (4) the
 * host-to-device fetch of every missed entry. Only the placement of KV changes, so
 * the rows a consumer reads through the returned slots are the host rows.
 *
 * The pages leave the LRU order, its tie-break and the miss/victim pairing open.
 * This oracle takes the plainest reading that keeps the result deterministic:
 *   - recency is a per-request call counter t (0, 1, 2, ...); a slot never used
 *     has last_use = -1;
 *   - slots hit in this call are stamped t and cannot be evicted in it;
 *   - the misses, in ascending position order, take in order the non-hit slots
 *     with the smallest (last_use, slot index);
 *   - an evicted position is unmapped, the new one mapped and stamped t, and its
 *     host row copied into the slot.
 * Further readings of unstated cases:
 *   - a negative position is padding: it resolves to -1 and is neither hit nor miss;
 *   - a position >= C is an error: it resolves to -1, is skipped, and the call
 *     returns a status with ORC_ERR_RANGE set;
 *   - a position repeated within one row resolves to the same slot each time and
 *     counts once (misses are a set of positions); the status gets ORC_ERR_DUP.
 *
 * Replacement policies. LRU (above) is the method's policy; the blog commentary's
 * section on Fig. 3 compares it with policies that do not exploit locality, which
 * the pages do not name. Two such variants are kept for that comparison, each read
 * as the plainest policy of its kind:
 *   - FIFO: the stamp of a slot is the call that filled it; a hit does not restamp,
 *     so the victims are the non-hit slots in ascending (fill call, slot) order;
 *   - RANDOM: the victims are the non-hit slots in ascending (key, slot) order, the
 *     key of slot s at call t of request b being the high 32 bits of SplitMix64
 *     output number (t * 2^16 + s) of the stream whose seed is SplitMix64 output
 *     number b of the policy seed (Steele, Lea and Flood, "Fast splittable
 *     pseudorandom number generators", 2014: output n of seed x is
 *     mix(x + (n + 1) * 0x9E3779B97F4A7C15) with the 13th of Stafford's mixers);
 *     stamps are kept as under LRU. It needs S <= 65536.
 * Hits, misses, the miss order, pairing and page-table updates are the same for all.
 *
 * Parity is pinned (not to this code itself) by: a hand-worked trace, a textbook
 * single-access LRU cache (k = 1), an independently written recency-list LRU,
 * closed forms for the cold start, for S >= C and for S = k, the per-step miss
 * bound k - floor(keep * k), and the invariants of an exact cache. The variants
 * are pinned by Belady's textbook string (FIFO and LRU fault counts), a textbook
 * FIFO queue, SplitMix64's published outputs with victims recomputed from them, the
 * uniformity of RANDOM's victims, and the loop of S + 1 positions. The consumer is
 * pinned by the E4M3 definition and PyTorch's decoder, library softmax attention on small
 * cases, and closed forms (one entry, repeated entries, no valid entry, reordering).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_RANGE 1u
#define ORC_ERR_DUP 2u
#define ORC_EINVAL (-1)
#define ORC_ENOMEM (-2)
#define ORC_POLICY_LRU 0
#define ORC_POLICY_FIFO 1
#define ORC_POLICY_RANDOM 2

typedef struct {
    int R, C, S, E;
    int32_t* pt;  /* [R][C]    position -> slot, -1 when not resident */
    int32_t* tok; /* [R][S]    slot -> position, -1 when empty        */
    int32_t* lu;  /* [R][S]    last-use stamp, -1 when never used     */
    int32_t* t;   /* [R]       calls made so far for the request      */
    uint8_t* dev; /* [R][S][E] contents of the device slots           */
    int32_t* rid; /* [R]       request number of each row (RANDOM keys) */
    int32_t* len; /* [R]       positions each request has (C unless set: a shared pool) */
    int policy;   /* ORC_POLICY_*, LRU unless set                     */
    uint64_t seed;/* the RANDOM policy's seed                         */
} orc_state;

orc_state* orc_create(int R, int C, int S, int E) {
    if (R <= 0 || C <= 0 || S <= 0 || E <= 0) return NULL;
    orc_state* o = (orc_state*)calloc(1, sizeof(orc_state));
    if (!o) return NULL;
    o->R = R; o->C = C; o->S = S; o->E = E;
    o->pt = (int32_t*)malloc(sizeof(int32_t) * (size_t)R * C);
    o->tok = (int32_t*)malloc(sizeof(int32_t) * (size_t)R * S);
    o->lu = (int32_t*)malloc(sizeof(int32_t) * (size_t)R * S);
    o->t = (int32_t*)calloc((size_t)R, sizeof(int32_t));
    o->dev = (uint8_t*)calloc((size_t)R * S, (size_t)E);
    o->rid = (int32_t*)malloc(sizeof(int32_t) * (size_t)R);
    o->len = (int32_t*)malloc(sizeof(int32_t) * (size_t)R);
    if (!o->pt || !o->tok || !o->lu || !o->t || !o->dev || !o->rid || !o->len) {
        free(o->pt); free(o->tok); free(o->lu); free(o->t); free(o->dev); free(o->rid); free(o->len); free(o);
        return NULL;
    }
    for (int b = 0; b < R; ++b) { o->rid[b] = b; o->len[b] = C; }
    for (size_t i = 0; i < (size_t)R * C; ++i) o->pt[i] = -1;
    for (size_t i = 0; i < (size_t)R * S; ++i) { o->tok[i] = -1; o->lu[i] = -1; }
    return o;
}

void orc_destroy(orc_state* o) {
    if (!o) return;
    free(o->pt); free(o->tok); free(o->lu); free(o->t); free(o->dev); free(o->rid); free(o->len); free(o);
}

/*
 * A shared host pool holds requests of different lengths: request b has positions
 * [0, len) only (its history sits at its own extent of the pool; the caller passes that
 * extent as host_b), and a position >= len is out of range like one >= C. A request that
 * takes over row b is new: orc_reset_request empties its state (tables, stamps, call
 * counter, slot contents).
 */
int orc_set_len(orc_state* o, int b, int32_t len) {
    if (!o || b < 0 || b >= o->R || len < 0 || len > o->C) return ORC_EINVAL;
    o->len[b] = len;
    return 0;
}

int orc_reset_request(orc_state* o, int b) {
    if (!o || b < 0 || b >= o->R) return ORC_EINVAL;
    for (int p = 0; p < o->C; ++p) o->pt[(size_t)b * o->C + p] = -1;
    for (int s = 0; s < o->S; ++s) { o->tok[(size_t)b * o->S + s] = -1; o->lu[(size_t)b * o->S + s] = -1; }
    o->t[b] = 0;
    memset(o->dev + (size_t)b * o->S * o->E, 0, (size_t)o->S * o->E);
    return 0;
}

/* Replacement policy for the calls that follow (the state kept so far carries over). */
int orc_set_policy(orc_state* o, int policy, uint64_t seed) {
    if (!o || policy < ORC_POLICY_LRU || policy > ORC_POLICY_RANDOM) return ORC_EINVAL;
    if (policy == ORC_POLICY_RANDOM && o->S > 65536) return ORC_EINVAL;
    o->policy = policy;
    o->seed = seed;
    return 0;
}

/* Row b of this state follows request number id of a larger batch (the RANDOM
 * policy's draws depend on the request number; the default is b). */
int orc_set_request_id(orc_state* o, int b, int32_t id) {
    if (!o || b < 0 || b >= o->R || id < 0) return ORC_EINVAL;
    o->rid[b] = id;
    return 0;
}

/* SplitMix64 output number n (n = 0, 1, 2, ...) of the generator seeded with x. */
uint64_t orc_splitmix64(uint64_t x, uint64_t n) {
    uint64_t z = x + (n + 1u) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* The RANDOM policy's key of slot s at call t of request b. */
uint32_t orc_random_key(uint64_t seed, int b, int32_t t, int s) {
    const uint64_t stream = orc_splitmix64(seed, (uint64_t)b);
    return (uint32_t)(orc_splitmix64(stream, ((uint64_t)(uint32_t)t << 16) + (uint64_t)s) >> 32);
}

int32_t* orc_pt(orc_state* o) { return o->pt; }
int32_t* orc_tok(orc_state* o) { return o->tok; }
int32_t* orc_lu(orc_state* o) { return o->lu; }
int32_t* orc_t(orc_state* o) { return o->t; }
uint8_t* orc_dev(orc_state* o) { return o->dev; }

/* sort helpers (the library sort is a step of the definition, nothing more) */
static int cmp_int(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

typedef struct { int64_t key; int32_t slot; } cand_t;

static int cmp_cand(const void* a, const void* b) {
    const cand_t* x = (const cand_t*)a;
    const cand_t* y = (const cand_t*)b;
    if (x->key != y->key) return (x->key > y->key) - (x->key < y->key);
    return (x->slot > y->slot) - (x->slot < y->slot);
}

/*
 * Resolves one request b: host_b points at the request's history row 0 (rows are
 * host_stride bytes apart), sel_b at its k selected positions; writes out_b[k] and
 * *miss_b. Returns a status word (ORC_ERR_* bits) or a negative error.
 */
int orc_resolve_request(orc_state* o, int b, const uint8_t* host_b, size_t host_stride,
                        const int32_t* sel_b, int k, int32_t* out_b, int32_t* miss_b) {
    if (!o || b < 0 || b >= o->R || k <= 0 || k > o->S || !host_b || !sel_b || !out_b || !miss_b)
        return ORC_EINVAL;
    const int C = o->C, S = o->S, E = o->E;
    const int32_t lim = o->len[b];  /* positions this request has */
    int32_t* pt = o->pt + (size_t)b * C;
    int32_t* tok = o->tok + (size_t)b * S;
    int32_t* lu = o->lu + (size_t)b * S;
    uint8_t* dev = o->dev + (size_t)b * S * E;
    const int32_t t = o->t[b];
    int status = 0;

    char* hit = (char*)calloc((size_t)S, 1);        /* H: slots hit in this call   */
    int32_t* P = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);   /* missed positions */
    cand_t* V = (cand_t*)malloc(sizeof(cand_t) * (size_t)S);        /* eviction order   */
    if (!hit || !P || !V) { free(hit); free(P); free(V); return ORC_ENOMEM; }

    /* 1. hit detection through the page table */
    int np = 0;
    for (int j = 0; j < k; ++j) {
        int32_t p = sel_b[j];
        out_b[j] = -1;
        if (p < 0) continue;                         /* padding */
        if (p >= lim) { status |= ORC_ERR_RANGE; continue; }
        if (pt[p] >= 0) {
            out_b[j] = pt[p];
            hit[pt[p]] = 1;
        } else {
            P[np++] = p;
        }
    }

    /* 2. misses: the distinct missed positions in ascending order */
    qsort(P, (size_t)np, sizeof(int32_t), cmp_int);
    int m = 0;
    for (int i = 0; i < np; ++i) {
        if (m > 0 && P[m - 1] == P[i]) continue;
        P[m++] = P[i];
    }
    /* a position repeated in the row (hit or miss) is reported */
    {
        int32_t* Q = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
        if (!Q) { free(hit); free(P); free(V); return ORC_ENOMEM; }
        int nq = 0;
        for (int j = 0; j < k; ++j) if (sel_b[j] >= 0 && sel_b[j] < lim) Q[nq++] = sel_b[j];
        qsort(Q, (size_t)nq, sizeof(int32_t), cmp_int);
        for (int i = 1; i < nq; ++i) if (Q[i] == Q[i - 1]) status |= ORC_ERR_DUP;
        free(Q);
    }

    /* 3. eviction order of the slots not hit in this call: ascending (key, slot), the
     *    key being the stamp (LRU: last use; FIFO: fill) or the RANDOM policy's draw */
    int nv = 0;
    for (int s = 0; s < S; ++s) {
        if (hit[s]) continue;
        V[nv].key = o->policy == ORC_POLICY_RANDOM ? (int64_t)orc_random_key(o->seed, o->rid[b], t, s) : (int64_t)lu[s];
        V[nv].slot = s;
        ++nv;
    }
    qsort(V, (size_t)nv, sizeof(cand_t), cmp_cand);

    /* 4. the i-th miss takes the i-th victim: unmap, map, fetch */
    for (int i = 0; i < m; ++i) {
        int32_t v = V[i].slot;
        if (tok[v] >= 0) pt[tok[v]] = -1;
        pt[P[i]] = v;
        tok[v] = P[i];
        memcpy(dev + (size_t)v * E, host_b + (size_t)P[i] * host_stride, (size_t)E);
    }
    for (int j = 0; j < k; ++j) {
        int32_t p = sel_b[j];
        if (p >= 0 && p < lim && out_b[j] < 0) out_b[j] = pt[p];
    }

    /* 5. stamps and counters (FIFO keeps the fill call of a hit slot) */
    if (o->policy != ORC_POLICY_FIFO)
        for (int s = 0; s < S; ++s) if (hit[s]) lu[s] = t;
    for (int i = 0; i < m; ++i) lu[V[i].slot] = t;
    *miss_b = m;
    o->t[b] = t + 1;

    free(hit); free(P); free(V);
    return status;
}

/*
 * Resolves all B == R requests of one layer-step: host is [R][C] rows of
 * host_stride bytes, sel [R][k], out [R][k], miss [R]. Returns the OR of the
 * per-request status words, or a negative error.
 */
int orc_resolve(orc_state* o, const uint8_t* host, size_t host_stride, const int32_t* sel, int B,
                int k, int32_t* out, int32_t* miss) {
    if (!o || B != o->R || !host || !sel || !out || !miss) return ORC_EINVAL;
    int status = 0;
    for (int b = 0; b < B; ++b) {
        int rc = orc_resolve_request(o, b, host + (size_t)b * o->C * host_stride, host_stride,
                                     sel + (size_t)b * k, k, out + (size_t)b * k, miss + b);
        if (rc < 0) return rc;
        status |= rc;
    }
    return status;
}

/*
 * Decode-time append (blog commentary, opening and section two: the KV the decode no
 * longer needs on the GPU lives in host memory, which keeps each request's full
 * history; paper abstract: the full KV history is kept in host memory). The new entry
 * `row` of request b joins its history at position p: host_b[p] = row. If p is
 * resident (a rewrite of an entry already in a slot), the slot gets the row too, so the
 * cache stays exact. A negative p means no new entry; p >= C is a range error. The
 * replacement state (page table, stamps, steps) does not change: admitting the new
 * entry into a slot is a resolution that selects it.
 * Returns 0, ORC_ERR_RANGE, or a negative error.
 */
int orc_append(orc_state* o, int b, uint8_t* host_b, size_t host_stride, int32_t p, const uint8_t* row) {
    if (!o || b < 0 || b >= o->R || !host_b || !row) return ORC_EINVAL;
    if (p < 0) return 0;
    if (p >= o->len[b]) return ORC_ERR_RANGE;
    memcpy(host_b + (size_t)p * host_stride, row, (size_t)o->E);
    const int32_t s = o->pt[(size_t)b * o->C + p];
    if (s >= 0) memcpy(o->dev + ((size_t)b * o->S + s) * o->E, row, (size_t)o->E);
    return 0;
}


/*
 * ---------------------------------------------------------------------------------
 * The consumer: sparse attention over the resolved slots (the blog commentary, section
 * two: a resident entry takes part in the layer's computation directly; paper
 * abstract: only placement changes, so the consumer's outputs are unchanged).
 *
 * The pages fix no attention arithmetic; this is the plainest reading for the 656-byte
 * DSA-style entries of the DeepSeek sparse-attention family the pages evaluate, an
 * MLA decode in its absorbed form:
 *   entry bytes [0, 512)    e4m3 codes c_0..c_511 of the latent vector
 *               [512, 528)  four fp32 scales; scale g applies to codes 128g..128g+127
 *               [528, 656)  64 bf16 values of the rotary part
 *   key   K_j = (c_j * scale, rope_j)  in R^576,   value  V_j = c_j * scale  in R^512;
 *   for head h with query q_h in R^576 (bf16) and the selections j whose slot is >= 0:
 *   s_hj = sm_scale * <q_h, K_j>,  o_h = sum_j softmax_j(s_h) V_j,  lse_h = ln sum_j exp(s_hj).
 * A head with no valid selection gets o_h = 0 and lse_h = -inf. All arithmetic is fp64.
 * e4m3 is the OCP 8-bit floating point format E4M3: sign, 4 exponent bits with bias 7,
 * 3 mantissa bits, subnormals at exponent 0, no infinities, S.1111.111 is NaN.
 */
double orc_e4m3(uint8_t c) {
    const int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

double orc_bf16(uint16_t h) {
    const uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/*
 * Attention of request b over its selections: out_b[k] are the slots hs resolution
 * returned (negative = not a valid selection), q [H][576] bf16 bit patterns. Writes
 * o [H][512], lse [H], and absw [H][512] = sum_j softmax_j |V_j| (the scale of the
 * values each output averages, for error bounds). Needs E == 656.
 */
int orc_attend(const orc_state* o, int b, const uint16_t* q, int H, const int32_t* out_b, int k,
               double sm_scale, double* out, double* lse, double* absw) {
    if (!o || b < 0 || b >= o->R || o->E != 656 || !q || H <= 0 || !out_b || k <= 0 || !out || !lse || !absw)
        return ORC_EINVAL;
    const int S = o->S;
    double* K = (double*)malloc(sizeof(double) * (size_t)k * 576);
    double* s = (double*)malloc(sizeof(double) * (size_t)k);
    int* use = (int*)malloc(sizeof(int) * (size_t)k);
    if (!K || !s || !use) { free(K); free(s); free(use); return ORC_ENOMEM; }
    for (int j = 0; j < k; ++j) {
        const int32_t sl = out_b[j];
        use[j] = sl >= 0 && sl < S;
        if (!use[j]) continue;
        const uint8_t* row = o->dev + ((size_t)b * S + sl) * 656;
        for (int d = 0; d < 512; ++d) {
            float sc;
            memcpy(&sc, row + 512 + 4 * (d / 128), 4);
            K[(size_t)j * 576 + d] = orc_e4m3(row[d]) * (double)sc;
        }
        for (int d = 0; d < 64; ++d) {
            uint16_t h;
            memcpy(&h, row + 528 + 2 * d, 2);
            K[(size_t)j * 576 + 512 + d] = orc_bf16(h);
        }
    }
    for (int h = 0; h < H; ++h) {
        double mx = -INFINITY;
        for (int j = 0; j < k; ++j) {
            if (!use[j]) continue;
            double acc = 0.0;
            for (int d = 0; d < 576; ++d) acc += orc_bf16(q[(size_t)h * 576 + d]) * K[(size_t)j * 576 + d];
            s[j] = sm_scale * acc;
            if (s[j] > mx) mx = s[j];
        }
        double* oh = out + (size_t)h * 512;
        double* wh = absw + (size_t)h * 512;
        for (int d = 0; d < 512; ++d) { oh[d] = 0.0; wh[d] = 0.0; }
        if (mx == -INFINITY) { lse[h] = -INFINITY; continue; }
        double l = 0.0;
        for (int j = 0; j < k; ++j) if (use[j]) l += exp(s[j] - mx);
        for (int j = 0; j < k; ++j) {
            if (!use[j]) continue;
            const double w = exp(s[j] - mx) / l;
            for (int d = 0; d < 512; ++d) {
                oh[d] += w * K[(size_t)j * 576 + d];
                wh[d] += w * fabs(K[(size_t)j * 576 + d]);
            }
        }
        lse[h] = mx + log(l);
    }
    free(K); free(s); free(use);
    return 0;
}
