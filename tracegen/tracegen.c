/*
 * tracegen.c -- seeded synthetic inputs for the HiSparse swap-in resolution step.
 *
 * This module only MAKES INPUTS: decode-step top-k selections and the bytes of the
 * host-resident KV history. It holds none of the method's arithmetic (no hit test,
 * no page table, no LRU). Both the CPU oracle and the CUDA path consume what it
 * writes; neither is imported here.
 *
 * Stand-in for the pages' miss-count workload (HiSparse blog commentary, section
 * three: DeepSeek-V3.2, top-k = 2048, device buffers of 2048 / 4096 slots, a
 * long-context benchmark). Neither the model nor the dataset is available, so the
 * selections are drawn from a locality model instead:
 *   - step 0: k distinct positions drawn from a Zipf(s) law over ranks 1..C, each
 *     rank mapped through a per-request seeded permutation of [0, C);
 *   - step t >= 1: keep floor(pct * k / 100) positions of the previous selection
 *     (a uniform subset, partial Fisher-Yates) and refill to k with Zipf draws,
 *     redrawing any position already in the row;
 *   - optionally the `recent` positions C-recent .. C-1 are in every row (the
 *     most recent tokens of a DSA-style decode) and count toward the kept part;
 *   - each row is emitted in a seeded random order, not sorted.
 *   - "no-IO" traces: step 0 as above, every later step a fresh seeded permutation
 *     of step 0's row (so, once resident, every call is all hits).
 *
 * Random numbers: splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014; the 64-bit finaliser constants as published by
 * Vigna), one independent stream per (seed, config, request, layer). Bounded
 * integers use Lemire's multiply-shift, uniform doubles the top 53 bits.
 *
 * KV contents are counter based: every row's bytes are a pure function of
 * (seed, layer, request, position), so any row can be regenerated on its own.
 *   kind 0 (BF16): E/2 bf16 values ~ N(0,1)                       (tiny trace, Quest pages)
 *   kind 1 (DSA656): 512 e4m3 codes of N(0,1), 4 fp32 scales = 1.0, 64 bf16 N(0,1)
 *   kind 2 (RAW): uniformly random bytes
 * Normal deviates come from 65536-entry quantile tables (inverse normal CDF at the
 * midpoints (i + 1/2) / 65536), found by bisection on erfc; one 16-bit draw picks
 * one table entry. Value encodings use software round-to-nearest-even.
 *
 * Compile with -ffp-contract=off so that x86-64 and aarch64 agree bit for bit.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define TG_OK 0
#define TG_EINVAL (-1)
#define TG_ENOMEM (-2)

enum { TG_PURPOSE_TRACE = 1, TG_PURPOSE_KV = 2 };
enum { TG_KV_BF16 = 0, TG_KV_DSA656 = 1, TG_KV_RAW = 2 };

/* ------------------------------------------------------------------ RNG */

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline uint64_t sm64_next(uint64_t* s) {
    *s += 0x9E3779B97F4A7C15ull;
    return mix64(*s);
}

/* stream seed for one (seed, purpose, a, b, c) tuple: chained finalisers */
static uint64_t stream_seed(uint64_t seed, uint64_t purpose, uint64_t a, uint64_t b, uint64_t c) {
    uint64_t h = mix64(seed + 0x9E3779B97F4A7C15ull);
    h = mix64(h ^ (purpose + 0x632BE59BD9B4E019ull));
    h = mix64(h ^ (a + 0x8CB92BA72F3D8DD7ull));
    h = mix64(h ^ (b + 0xD1B54A32D192ED03ull));
    h = mix64(h ^ (c + 0xABC98388FB8FAC03ull));
    return h;
}

/* Lemire multiply-shift: an integer in [0, n) */
static inline uint32_t bounded(uint64_t* s, uint32_t n) {
    return (uint32_t)(((unsigned __int128)sm64_next(s) * n) >> 64);
}

static inline double uniform01(uint64_t* s) {
    return (double)(sm64_next(s) >> 11) * 0x1.0p-53;
}

/* ------------------------------------------------------------------ traces */

typedef struct {
    int B, C, k, T, keep_pct, recent, no_io, config, layer;
    double zipf_s;
    uint64_t seed;
    const double* cum; /* cum[i] = sum_{r=1}^{i+1} r^-s, i in [0, C) */
    int32_t* out;      /* [T][B][k] */
} trace_job;

/* smallest index i with cum[i] > x (x in [0, cum[C-1])) -> rank i+1 */
static int zipf_index(const double* cum, int C, double x) {
    int lo = 0, hi = C - 1;
    while (lo < hi) {
        int mid = lo + ((hi - lo) >> 1);
        if (cum[mid] > x) hi = mid; else lo = mid + 1;
    }
    return lo;
}

static void shuffle_i32(int32_t* a, int n, uint64_t* s) {
    for (int i = n - 1; i > 0; --i) {
        int j = (int)bounded(s, (uint32_t)(i + 1));
        int32_t tmp = a[i]; a[i] = a[j]; a[j] = tmp;
    }
}

#define BIT_GET(bm, p) ((bm)[(p) >> 6] >> ((p) & 63) & 1ull)
#define BIT_SET(bm, p) ((bm)[(p) >> 6] |= 1ull << ((p) & 63))
#define BIT_CLR(bm, p) ((bm)[(p) >> 6] &= ~(1ull << ((p) & 63)))

/* one request's whole trace; returns 0 or TG_ENOMEM */
static int trace_request(const trace_job* J, int b) {
    const int C = J->C, k = J->k, T = J->T, B = J->B;
    uint64_t st = stream_seed(J->seed, TG_PURPOSE_TRACE, (uint64_t)J->config, (uint64_t)b, (uint64_t)J->layer);
    int32_t* perm = (int32_t*)malloc(sizeof(int32_t) * (size_t)C);
    uint64_t* in_row = (uint64_t*)calloc((size_t)(C + 63) / 64, sizeof(uint64_t));
    int32_t* row = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
    int32_t* cand = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
    if (!perm || !in_row || !row || !cand) { free(perm); free(in_row); free(row); free(cand); return TG_ENOMEM; }

    for (int i = 0; i < C; ++i) perm[i] = i;
    shuffle_i32(perm, C, &st);
    const double total = J->cum[C - 1];
    const int recent = J->recent;
    const int keep = (int)(((int64_t)J->keep_pct * k) / 100);

    for (int t = 0; t < T; ++t) {
        int n = 0;
        if (t == 0 || !J->no_io) {
            if (t == 0) {
                for (int i = 0; i < recent; ++i) { int p = C - recent + i; row[n++] = p; BIT_SET(in_row, p); }
            } else {
                /* previous row is in `row` (internal order); in_row marks it */
                int nc = 0;
                for (int i = 0; i < k; ++i) {
                    int p = row[i];
                    BIT_CLR(in_row, p);
                    if (p >= C - recent) continue; /* the always-selected recent tail */
                    cand[nc++] = p;
                }
                for (int i = 0; i < recent; ++i) { int p = C - recent + i; row[n++] = p; BIT_SET(in_row, p); }
                int want = keep - recent;
                if (want > nc) want = nc;
                for (int i = 0; i < want; ++i) { /* partial Fisher-Yates: a uniform subset */
                    int j = i + (int)bounded(&st, (uint32_t)(nc - i));
                    int32_t tmp = cand[i]; cand[i] = cand[j]; cand[j] = tmp;
                    row[n++] = cand[i];
                    BIT_SET(in_row, cand[i]);
                }
            }
            while (n < k) { /* Zipf refill, redrawn until distinct */
                int r = zipf_index(J->cum, C, uniform01(&st) * total);
                int p = perm[r];
                if (BIT_GET(in_row, p)) continue;
                BIT_SET(in_row, p);
                row[n++] = p;
            }
            memcpy(cand, row, sizeof(int32_t) * (size_t)k);
        } else {
            memcpy(cand, row, sizeof(int32_t) * (size_t)k); /* no-IO: same set as step 0 */
        }
        shuffle_i32(cand, k, &st); /* emission order */
        memcpy(J->out + ((size_t)t * B + b) * (size_t)k, cand, sizeof(int32_t) * (size_t)k);
    }
    free(perm); free(in_row); free(row); free(cand);
    return TG_OK;
}

typedef struct { const trace_job* job; int b0, b1, step, rc; } trace_worker;

static void* trace_thread(void* arg) {
    trace_worker* w = (trace_worker*)arg;
    for (int b = w->b0; b < w->b1; b += w->step) {
        int rc = trace_request(w->job, b);
        if (rc) { w->rc = rc; break; }
    }
    return NULL;
}

/*
 * Writes a trace of T steps for B requests into out[T][B][k] (row-major int32).
 * keep_pct: kept percentage of the previous row (floor(keep_pct * k / 100) kept);
 * recent: number of always-selected tail positions (0 for none); no_io: 1 for the
 * all-hit trace. Returns 0, TG_EINVAL or TG_ENOMEM. Independent of nthreads.
 */
int tg_trace(int B, int C, int k, int T, int keep_pct, double zipf_s, int recent, int no_io,
             uint64_t seed, int config, int layer, int nthreads, int32_t* out) {
    if (B <= 0 || C <= 0 || k <= 0 || T <= 0 || k > C || keep_pct < 0 || keep_pct > 100 ||
        recent < 0 || recent > k || !(zipf_s > 0.0) || !out)
        return TG_EINVAL;
    if (recent > (int)(((int64_t)keep_pct * k) / 100) && T > 1 && !no_io) return TG_EINVAL;
    double* cum = (double*)malloc(sizeof(double) * (size_t)C);
    if (!cum) return TG_ENOMEM;
    double acc = 0.0;
    for (int r = 1; r <= C; ++r) { acc += pow((double)r, -zipf_s); cum[r - 1] = acc; }
    trace_job J = {B, C, k, T, keep_pct, recent, no_io, config, layer, zipf_s, seed, cum, out};
    if (nthreads < 1) nthreads = 1;
    if (nthreads > B) nthreads = B;
    trace_worker* ws = (trace_worker*)calloc((size_t)nthreads, sizeof(trace_worker));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!ws || !th) { free(ws); free(th); free(cum); return TG_ENOMEM; }
    int rc = TG_OK;
    for (int i = 0; i < nthreads; ++i) {
        ws[i].job = &J; ws[i].b0 = i; ws[i].b1 = B; ws[i].step = nthreads; ws[i].rc = 0;
        if (nthreads == 1 || pthread_create(&th[i], NULL, trace_thread, &ws[i]) != 0) {
            trace_thread(&ws[i]);
            th[i] = 0;
        }
    }
    for (int i = 0; i < nthreads; ++i) {
        if (th[i]) pthread_join(th[i], NULL);
        if (ws[i].rc) rc = ws[i].rc;
    }
    free(ws); free(th); free(cum);
    return rc;
}

/* ------------------------------------------------------------------ KV bytes */

static uint16_t q_bf16[65536]; /* bf16 bit patterns of N(0,1) quantiles */
static uint8_t q_e4m3[65536];  /* e4m3 codes of N(0,1) quantiles */
static pthread_once_t q_once = PTHREAD_ONCE_INIT;

/* standard normal quantile by bisection on Phi(x) = erfc(-x / sqrt 2) / 2 */
static double normal_quantile(double p) {
    double lo = -12.0, hi = 12.0;
    for (int it = 0; it < 200 && hi - lo > 1e-15; ++it) {
        double mid = 0.5 * (lo + hi);
        double cdf = 0.5 * erfc(-mid / sqrt(2.0));
        if (cdf < p) lo = mid; else hi = mid;
    }
    return 0.5 * (lo + hi);
}

static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t rounding = 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)((u + rounding) >> 16);
}

/* value of a non-negative e4m3 code c in [0, 126] (OCP FP8 E4M3: bias 7, no inf, 0x7F NaN) */
static double e4m3_value(int c) {
    int e = (c >> 3) & 15, m = c & 7;
    if (e == 0) return ldexp((double)m, -9);
    return ldexp(1.0 + m / 8.0, e - 7);
}

/* round-to-nearest-even onto the e4m3 grid, saturating at +-448 */
static uint8_t e4m3_rne(double x) {
    uint8_t sign = x < 0 ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    int lo = 0, hi = 126; /* largest code with value <= a */
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (e4m3_value(mid) <= a) lo = mid; else hi = mid - 1;
    }
    int c = lo;
    if (c < 126) {
        double d0 = a - e4m3_value(c), d1 = e4m3_value(c + 1) - a;
        if (d1 < d0 || (d1 == d0 && (c & 1))) c = c + 1;
    }
    return (uint8_t)(sign | c);
}

static void q_init(void) {
    for (int i = 0; i < 65536; ++i) {
        double x = normal_quantile((i + 0.5) / 65536.0);
        q_bf16[i] = f32_to_bf16_rne((float)x);
        q_e4m3[i] = e4m3_rne(x);
    }
}

static void kv_row(uint8_t* dst, int E, int kind, uint64_t seed, int layer, int b, int p) {
    uint64_t st = stream_seed(seed, TG_PURPOSE_KV, (uint64_t)layer, (uint64_t)b, (uint64_t)p);
    if (kind == TG_KV_RAW) {
        for (int o = 0; o < E; o += 8) {
            uint64_t r = sm64_next(&st);
            int n = E - o < 8 ? E - o : 8;
            memcpy(dst + o, &r, (size_t)n); /* little-endian on both targets */
        }
        return;
    }
    if (kind == TG_KV_DSA656) {
        for (int o = 0; o < 512; o += 4) {
            uint64_t r = sm64_next(&st);
            for (int q = 0; q < 4; ++q) dst[o + q] = q_e4m3[(r >> (16 * q)) & 0xFFFF];
        }
        const float one = 1.0f;
        for (int q = 0; q < 4; ++q) memcpy(dst + 512 + 4 * q, &one, 4);
        for (int o = 0; o < 64; o += 4) {
            uint64_t r = sm64_next(&st);
            for (int q = 0; q < 4; ++q) {
                uint16_t v = q_bf16[(r >> (16 * q)) & 0xFFFF];
                memcpy(dst + 528 + 2 * (o + q), &v, 2);
            }
        }
        return;
    }
    /* bf16 */
    int n = E / 2;
    for (int o = 0; o < n; o += 4) {
        uint64_t r = sm64_next(&st);
        for (int q = 0; q < 4 && o + q < n; ++q) {
            uint16_t v = q_bf16[(r >> (16 * q)) & 0xFFFF];
            memcpy(dst + 2 * (o + q), &v, 2);
        }
    }
}

static int kv_args_ok(int E, int kind) {
    if (E <= 0) return 0;
    if (kind == TG_KV_DSA656) return E == 656;
    if (kind == TG_KV_BF16) return (E % 2) == 0;
    return kind == TG_KV_RAW;
}

/* One row of (layer, b, p) into dst[0..E). Returns 0 or TG_EINVAL. */
int tg_kv_row(uint8_t* dst, int E, int kind, uint64_t seed, int layer, int b, int p) {
    if (!dst || !kv_args_ok(E, kind)) return TG_EINVAL;
    pthread_once(&q_once, q_init);
    kv_row(dst, E, kind, seed, layer, b, p);
    return TG_OK;
}

typedef struct {
    uint8_t* host; size_t stride; int B, C, E, kind, layer; uint64_t seed;
    int64_t r0, r1;
} kv_job;

static void* kv_thread(void* arg) {
    kv_job* j = (kv_job*)arg;
    for (int64_t r = j->r0; r < j->r1; ++r) {
        int b = (int)(r / j->C), p = (int)(r % j->C);
        kv_row(j->host + (size_t)r * j->stride, j->E, j->kind, j->seed, j->layer, b, p);
    }
    return NULL;
}

/*
 * Fills host[b][p][0..E) for all B x C rows (row pitch `stride` bytes, >= E) with
 * the counter-based contents of (seed, layer, b, p). Bytes beyond E in each row are
 * left untouched. Returns 0 or TG_EINVAL.
 */
int tg_fill_kv(uint8_t* host, size_t stride, int B, int C, int E, int kind, uint64_t seed,
               int layer, int nthreads) {
    if (!host || B <= 0 || C <= 0 || stride < (size_t)E || !kv_args_ok(E, kind)) return TG_EINVAL;
    pthread_once(&q_once, q_init);
    int64_t rows = (int64_t)B * C;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > rows) nthreads = (int)rows;
    kv_job jobs[256];
    pthread_t th[256];
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = (kv_job){host, stride, B, C, E, kind, layer, seed,
                           rows * i / nthreads, rows * (i + 1) / nthreads};
        if (nthreads == 1 || pthread_create(&th[i], NULL, kv_thread, &jobs[i]) != 0) {
            kv_thread(&jobs[i]);
            th[i] = 0;
        }
    }
    for (int i = 0; i < nthreads; ++i) if (th[i]) pthread_join(th[i], NULL);
    return TG_OK;
}
