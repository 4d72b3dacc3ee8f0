// hs_kernels.cu -- HiSparse swap-in resolution kernels for sm_103a.
//
// HiSparse resolves each layer's top-k selections in one fused step: hit detection,
// LRU replacement, the page-table update and the host-to-device fetch of the misses
// (paper abstract; blog commentary, sections two and three: hits are used in place,
// misses swapped in over LRU victims, the page table updated in the same step).
//
// The step is two kernels that run concurrently, chained by programmatic dependent
// launch (PDL) and synchronized per request through release/acquire flags:
//
// resolve_kernel -- one 512-thread CTA per request (resolve_role):
//   1. probe the page table for every selected position; hits are stamped and
//      answered in place, misses are marked in a shared position bitmap;
//   2. the probe lists every missed selection (position, index j in the row) in the
//      miss area as it finds it; right after the probe's barrier the list is
//      PUBLISHED (ready_pos): the source rows of the fetch are known from here on;
//   3. rank the misses by ascending position (a group prefix over the bitmap plus
//      popcounts), rank the non-hit slots by (last_use, slot) -- or, under the
//      comparison policies, by (fill call, slot) or (random draw, slot) -- with a stable LSD radix
//      sort whose digits are counted per warp (__match_any_sync ranks equal digits
//      inside a warp, an exclusive scan over the (digit, warp) table orders the warps),
//      pair the r-th miss with the r-th victim and answer the missed selections; the
//      answers name every row's slot, so they are PUBLISHED (ready_slot) before the
//      page table, slot tokens and stamps are updated.
// gather_kernel -- a persistent grid of one CTA per SM (fetch_role; held to 64 registers,
//   so that it fits beside a resolution CTA), launched right behind the resolution (PDL)
//   so that it is resident while the resolution runs. Each CTA owns
//   a share of one request's fetch list: it waits for ready_pos, issues the 16-byte
//   zero-copy loads of its rows from the mapped host store (coalesced, 8 in flight
//   per thread), waits for ready_slot only when it has to store, and writes each row
//   into the slot the resolution answered for it. The host-link transfer -- the only real cost of the step --
//   thus overlaps the victim ranking and the table updates, and uses every SM's load
//   slots, not just the CTAs of the requests. With more requests than SMs the
//   resolution fills the GPU, and the fetch grid runs after it instead.
// Flags carry a per-request call tag: each fetch CTA keeps a private counter for each
// (request, share) it serves and advances it once per call; the resolution reads share
// 0's counter of its request and tags the call's flags with counter + 1. A flag left
// from an earlier call never carries the tag a later fetch waits for (calls without a
// fetch publish nothing and advance nothing), and graph replays need no host reset.
// Every wait is bounded in time (global timer, the context's wait limit counted from the
// CTA's start): on expiry the CTA records HS_STATUS_TIMEOUT and skips, so no wait can
// hang the GPU.
//
// No tensor cores: nothing here is a contraction.
#include <cuda_runtime.h>
#include <stdint.h>

#include "hs_internal.h"

#define HS_STATUS_RANGE 1u
#define HS_STATUS_DUP 2u
#define HS_STATUS_STEP_LIMIT 4u
#define HS_STATUS_TIMEOUT 8u

namespace hs {
namespace {

constexpr int NT = kResolveThreads;
constexpr int NW = kResolveWarps;

__device__ __forceinline__ void pdl_wait_prerequisites() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gsrc) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed(uint32_t* p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// All threads' global writes so far become visible before *flag = value: the barrier
// orders them before thread 0's release store, which is cumulative. Called by every
// thread of the CTA; a no-op when `on` is false.
__device__ __forceinline__ void publish(uint32_t* flag, uint32_t value, bool on) {
    if (!on) return;
    __syncthreads();
    if (threadIdx.x == 0) st_release(flag, value);
}

// Thread 0 waits until (*flag & mask) == want and broadcasts the flag's value; the
// outcome is block-uniform. The wait gives up once the global timer passes `deadline`
// (the CTA's start plus the context's wait limit): it then records HS_STATUS_TIMEOUT
// and returns false. Polls follow one another without a pause: each flag has a line of
// its own, and one polling thread per CTA costs less than the latency a pause adds.
__device__ __forceinline__ bool wait_flag(const uint32_t* flag, uint32_t want, uint32_t mask, uint64_t deadline,
                                          uint32_t* status, uint32_t* bcast, uint32_t* value) {
    if (threadIdx.x == 0) {
        uint32_t ok = 1, v;
        while (((v = ld_acquire(flag)) & mask) != want) {
            if (global_ns() > deadline) {
                ok = 0;
                atomicOr(status, HS_STATUS_TIMEOUT);
                break;
            }
        }
        bcast[0] = ok;
        bcast[1] = v;
    }
    __syncthreads();
    const bool ok = bcast[0] != 0;
    *value = bcast[1];
    __syncthreads();
    return ok;
}

// Exclusive scan of one value per thread over a BT-thread block. `scratch` holds
// BT/32 + 1 words; *total receives the sum. All threads must call it (3 barriers).
template <int BT>
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* scratch, uint32_t* total) {
    constexpr int BW = BT / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < BW ? scratch[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < BW) scratch[lane] = w;
        if (lane == BW - 1) scratch[BW] = w;
    }
    __syncthreads();
    const uint32_t r = (warp == 0 ? 0u : scratch[warp - 1]) + x - v;
    *total = scratch[BW];
    __syncthreads();
    return r;
}

// SplitMix64 output number n (n = 0, 1, ...) of the generator seeded with x (Steele,
// Lea and Flood, "Fast splittable pseudorandom number generators", 2014: the state
// advances by the golden-ratio increment and each output is Stafford's 13th mixer of
// it), so any output is computed directly from (x, n): the RANDOM policy's draws.
__device__ __forceinline__ uint64_t splitmix64(uint64_t x, uint64_t n) {
    uint64_t z = x + (n + 1ull) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// Shared-memory plan of one request's resolution (byte offsets).
struct Plan {
    int CW, CG, SW;
    uint32_t posbm, gprefix, hitbm, keys, mpos, counts, scratch, sa, sb, fixed;
    __host__ __device__ Plan(int C, int S) {
        CW = ((C + 31) / 32 + kGroupWords - 1) / kGroupWords * kGroupWords;
        CG = CW / kGroupWords;
        SW = (S + 31) / 32;
        const uint32_t S4 = ((uint32_t)S * 4u + 15u) & ~15u;
        const uint32_t S2 = ((uint32_t)S * 2u + 15u) & ~15u;
        posbm = 0;
        gprefix = posbm + (uint32_t)CW * 4u;
        hitbm = gprefix + (((uint32_t)CG * 4u + 15u) & ~15u);
        keys = hitbm + (((uint32_t)SW * 4u + 15u) & ~15u);
        mpos = keys + S4;
        counts = mpos + S4;
        scratch = counts + (uint32_t)(kBins * NW) * 2u;
        sa = scratch + 48u * 4u;
        sb = sa + S2;
        fixed = sb + S2;
    }
};

// Selections j0 + q*NT + tid (q < 4) of one request's row (-1 past its end).
__device__ __forceinline__ void load_selections(const int32_t* __restrict__ selb, int k, int j0, int32_t (&p)[4]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int j = j0 + q * NT + (int)threadIdx.x;
        p[q] = j < k ? __ldg(selb + j) : -1;
    }
}

// One request's resolution state in shared memory, and the phases shared by both
// kernels. Every phase is called by all threads of the CTA.
struct Request {
    const Layout& L;
    const Plan& P;
    uint8_t* smem;
    int b, k;
    int32_t t;
    const int32_t* selb;
    int32_t* outb;
    int32_t* ptb;
    int32_t* tokb;
    int32_t* lub;
    int32_t* fpos;      // fetch list (global): positions of the missed selections ...
    int32_t* fsel;      // ... and their indices j in the row, in no particular order
    uint32_t* posbm;    // missed positions of this call
    uint32_t* gprefix;  // misses before each group of kGroupWords bitmap words
    uint32_t* hitbm;    // slots hit in this call
    uint32_t* keys;     // last_use of every slot as loaded at kernel start (key = value + 1)
    int32_t* mpos;      // missed positions in ascending order (rank -> position)
    uint16_t* counts;   // radix digit counts, [digit][warp]
    uint32_t* scratch;
    uint16_t* sa;
    uint16_t* sb;
    int lim;  // positions this request has: C, or its extent's length in a pooled store
    uint32_t m = 0, N = 0, miss_base = 0, cand_base = 0;
    int g0 = 0, g1 = 0, s0 = 0, s1 = 0;  // this thread's miss-bitmap groups and slot range
    const uint16_t* victims = nullptr;  // victims[r] = slot of the r-th miss

    __device__ Request(const Layout& L_, const Plan& P_, uint8_t* smem_, int b_, const int32_t* sel, int k_,
                       int32_t* out)
        : L(L_), P(P_), smem(smem_), b(b_), k(k_),
          lim(L_.row_len ? __ldg(L_.row_len + b_) : L_.C) {
        selb = sel + (size_t)b * k;
        outb = out + (size_t)b * k;
        ptb = L.pt + (size_t)b * L.C;
        tokb = L.tok + (size_t)b * L.S;
        lub = L.lu + (size_t)b * L.S;
        fpos = L.fpos + (size_t)b * L.S;
        fsel = L.fsel + (size_t)b * L.S;
        posbm = reinterpret_cast<uint32_t*>(smem + P.posbm);
        gprefix = reinterpret_cast<uint32_t*>(smem + P.gprefix);
        hitbm = reinterpret_cast<uint32_t*>(smem + P.hitbm);
        keys = reinterpret_cast<uint32_t*>(smem + P.keys);
        mpos = reinterpret_cast<int32_t*>(smem + P.mpos);
        counts = reinterpret_cast<uint16_t*>(smem + P.counts);
        scratch = reinterpret_cast<uint32_t*>(smem + P.scratch);
        sa = reinterpret_cast<uint16_t*>(smem + P.sa);
        sb = reinterpret_cast<uint16_t*>(smem + P.sb);
    }

    // Starts the asynchronous copy of the request's last-use stamps into keys[]: they
    // are only needed to rank victims, so the copy starts once the probe has found a miss
    // and lands while the misses are ranked (a call without a miss never reads them). A
    // hit slot's stamp may be copied before or after the probe restamped it; hit slots
    // are never candidates. Every exit path after it waits for it (drain()).
    __device__ void prefetch_stamps() {
        const int tid = threadIdx.x;
        const int S = L.S;
        if ((S & 3) == 0 && ((uintptr_t)lub & 15) == 0) {  // 16-byte chunks when aligned
            for (int i = tid; i < S / 4; i += NT) cp_async16(keys + 4 * i, lub + 4 * i);
        } else {
            for (int i = tid; i < S; i += NT) cp_async4(keys + i, lub + i);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    }

    // Clears the bitmaps and counters; no barrier.
    __device__ void start() {
        const int tid = threadIdx.x;
        for (int i = tid; i < P.CW; i += NT) posbm[i] = 0u;
        for (int i = tid; i < P.SW; i += NT) hitbm[i] = 0u;
        if (tid == 0) {
            scratch[2 * NW] = 0xffffffffu;  // running min / max of the candidates' keys
            scratch[2 * NW + 1] = 0u;
            scratch[2 * NW + 2] = 0u;       // entries of the fetch list
        }
    }

    // The page-table entries of the selections p (this thread's batch).
    __device__ __forceinline__ void load_slots(const int32_t (&p)[4], int32_t (&s)[4]) const {
        const int C = lim;
#pragma unroll
        for (int q = 0; q < 4; ++q) s[q] = (p[q] >= 0 && p[q] < C) ? ptb[p[q]] : -1;
    }

    // Loads the selections j0 + q*NT + tid (q < 4) and their page-table entries.
    __device__ __forceinline__ void load_batch(int j0, int32_t (&p)[4], int32_t (&s)[4]) const {
        load_selections(selb, k, j0, p);
        load_slots(p, s);
    }

    // The call is refused (the request reached its call limit): every selection -1.
    __device__ void refuse(int32_t* miss_counts) {
        for (int j = threadIdx.x; j < k; j += NT) outb[j] = -1;
        if (threadIdx.x == 0) {
            atomicOr(L.status, HS_STATUS_STEP_LIMIT);
            miss_counts[b] = 0;
        }
        drain();
    }

    // The answers that need no ranking -- hits (stamped, not evictable) and padding or
    // out-of-range selections -- are either written by the probe itself (`direct`) or by
    // write_direct() after the hand-off flags: none of them is read by the fetch, and
    // each flag's release waits for the writes before it. The caller chooses: deferred
    // when the request's previous call had misses (so this one likely has too), direct
    // otherwise (an all-hit call raises its flags without a release, and the probe's
    // writes then drain under its barrier), and always direct when the selections take
    // more than one batch (k > 4 * NT: they are no longer held in registers).
    __device__ __forceinline__ bool one_batch() const { return k <= 4 * NT; }

    // 1. hit detection, starting from the batch already loaded into p/s (t set).
    // Returns true (block-uniform) if any selection missed.
    __device__ bool probe(int32_t (&p)[4], int32_t (&s)[4], bool direct) {
        const int tid = threadIdx.x;
        const int C = lim;
        uint32_t st = 0;
        int any_miss = 0;
        for (int j0 = 0; j0 < k; j0 += 4 * NT) {
            if (j0 > 0) load_batch(j0, p, s);  // only when k > 4 * NT (then answers re-read)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int j = j0 + q * NT + tid;
                if (j >= k) continue;
                const int32_t pp = p[q], ss = s[q];
                if (ss >= 0) {  // hit: answered in place, stamped, not evictable
                    const uint32_t bit = 1u << (ss & 31);
                    if (atomicOr(&hitbm[ss >> 5], bit) & bit) st |= HS_STATUS_DUP;
                    if (direct) {
                        if (L.policy != kPolicyFifo) lub[ss] = t;  // FIFO keeps the fill call
                        outb[j] = ss;
                    }
                } else if (pp >= 0 && pp < C) {  // miss: marked, and listed for the fetch
                    const uint32_t bit = 1u << (pp & 31);
                    if (atomicOr(&posbm[pp >> 5], bit) & bit) st |= HS_STATUS_DUP;
                    any_miss = 1;
                    const uint32_t e = atomicAdd(&scratch[2 * NW + 2], 1u);
                    fpos[e] = pp;
                    fsel[e] = j;
                } else {  // padding, or out of range
                    if (pp >= C) st |= HS_STATUS_RANGE;
                    if (direct) outb[j] = -1;
                }
            }
        }
        if (st) atomicOr(L.status, st);
        return __syncthreads_or(any_miss) != 0;
    }

    // The hits' answers and stamps and the padding's -1 of this thread's batch, when the
    // probe left them (one batch only; see one_batch). A hit slot is never a victim, so
    // its stamp may land at any time during the call.
    __device__ void write_direct(const int32_t (&p)[4], const int32_t (&s)[4], bool direct) {
        if (direct) return;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int j = q * NT + threadIdx.x;
            if (j >= k) continue;
            if (s[q] >= 0) {
                if (L.policy != kPolicyFifo) lub[s[q]] = t;  // FIFO keeps the fill call
                outb[j] = s[q];
            } else if (p[q] < 0 || p[q] >= lim) {
                outb[j] = -1;
            }
        }
    }

    __device__ void drain() const { cp_async_wait_all(); }

    // Non-hit slots among [lo, hi) -- a range inside one bitmap word, or whole words.
    __device__ __forceinline__ uint32_t cand_bits(int lo, int hi) const {
        const uint32_t word = ~hitbm[lo >> 5];
        const int n = hi - lo;
        const uint32_t mask = n >= 32 ? 0xffffffffu : ((1u << n) - 1u) << (lo & 31);
        return word & mask;
    }

    // 2. miss count and ascending-position ranks; candidate count; mpos[] filled.
    __device__ void rank_misses() {
        const int tid = threadIdx.x;
        const int gpt = (P.CG + NT - 1) / NT;
        g0 = min(tid * gpt, P.CG);
        g1 = min(g0 + gpt, P.CG);
        // slots per thread: a power of two, so a thread's range never straddles a word
        // boundary unless it is made of whole words
        int spt = 1;
        while (spt * NT < L.S) spt <<= 1;
        s0 = min(tid * spt, L.S);
        s1 = min(s0 + spt, L.S);
        uint32_t nmiss = 0, ncand = 0;
        for (int g = g0; g < g1; ++g)
#pragma unroll
            for (int q = 0; q < kGroupWords; ++q) nmiss += __popc(posbm[g * kGroupWords + q]);
        for (int lo = s0; lo < s1; lo = min((lo | 31) + 1, s1)) ncand += __popc(cand_bits(lo, min((lo | 31) + 1, s1)));
        uint32_t total;
        const uint32_t excl = block_exclusive_scan<NT>((ncand << 16) | nmiss, scratch, &total);
        m = total & 0xffffu;
        N = total >> 16;
        miss_base = excl & 0xffffu;
        cand_base = excl >> 16;
        uint32_t r = miss_base;
        for (int g = g0; g < g1; ++g) {
            gprefix[g] = r;
            for (int q = 0; q < kGroupWords; ++q) {
                const int w = g * kGroupWords + q;
                uint32_t bits = posbm[w];
                while (bits) {
                    mpos[r++] = w * 32 + __ffs(bits) - 1;
                    bits &= bits - 1;
                }
            }
        }
        __syncthreads();
    }

    // 4a. eviction order of the non-hit slots: ascending (key, slot), the key being the
    // stamp + 1 (LRU: last use, FIFO: fill call) or the RANDOM policy's draw; sets victims.
    __device__ void rank_victims() {
        const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
        drain();  // the stamps copied after the probe have landed (this thread's part) ...
        __syncthreads();  // ... and everyone's
        const bool drawn = L.policy == kPolicyRandom;
        const uint64_t stream = drawn ? splitmix64(L.seed, (uint64_t)b) : 0ull;
        const uint64_t call = (uint64_t)(uint32_t)t << 16;
        uint32_t kmin = 0xffffffffu, kmax = 0u;
        {
            uint32_t c = cand_base;
            for (int lo = s0; lo < s1; lo = min((lo | 31) + 1, s1)) {
                uint32_t bits = cand_bits(lo, min((lo | 31) + 1, s1));
                while (bits) {
                    const int s = (lo & ~31) + __ffs(bits) - 1;
                    bits &= bits - 1;
                    sa[c++] = (uint16_t)s;
                    uint32_t key;
                    if (drawn) {  // the draw replaces the stamp as the sort key
                        key = (uint32_t)(splitmix64(stream, call + (uint64_t)s) >> 32);
                        keys[s] = key - 1u;
                    } else {
                        key = keys[s] + 1u;
                    }
                    kmin = min(kmin, key);
                    kmax = max(kmax, key);
                }
            }
        }
        kmin = __reduce_min_sync(0xffffffffu, kmin);
        kmax = __reduce_max_sync(0xffffffffu, kmax);
        uint32_t* kr = scratch + 2 * NW;  // [min, max], initialised in start()
        if (lane == 0) {
            atomicMin(kr, kmin);
            atomicMax(kr + 1, kmax);
        }
        __syncthreads();
        kmin = kr[0];
        kmax = kr[1];

        const uint32_t range = kmax - kmin;
        const int npass = range ? (32 - __clz(range) + kRadixBits - 1) / kRadixBits : 0;
        const int seg = (((int)N + NW - 1) / NW + 31) & ~31;
        const int e0 = min(warp * seg, (int)N), e1 = min(e0 + seg, (int)N);
        uint16_t* src = sa;
        uint16_t* dst = sb;
        for (int pass = 0; pass < npass; ++pass) {
            const int shift = pass * kRadixBits;
            for (int i = tid; i < kBins * NW / 2; i += NT) reinterpret_cast<uint32_t*>(counts)[i] = 0u;
            __syncthreads();
            for (int base = e0; base < e1; base += 32) {
                const int idx = base + lane;
                const bool v = idx < e1;
                const uint32_t d = v ? ((keys[src[idx]] + 1u - kmin) >> shift) & (kBins - 1) : (uint32_t)kBins;
                const uint32_t peers = __match_any_sync(0xffffffffu, d);
                if (v && lane == __ffs(peers) - 1) counts[d * NW + warp] += (uint16_t)__popc(peers);
            }
            __syncthreads();
            {
                constexpr int PER = kBins * NW / NT;  // 8 counts per thread
                uint16_t loc[PER];
                uint32_t sum = 0;
#pragma unroll
                for (int q = 0; q < PER; ++q) {
                    loc[q] = counts[tid * PER + q];
                    sum += loc[q];
                }
                uint32_t tot;
                uint32_t ex = block_exclusive_scan<NT>(sum, scratch, &tot);
#pragma unroll
                for (int q = 0; q < PER; ++q) {
                    counts[tid * PER + q] = (uint16_t)ex;
                    ex += loc[q];
                }
            }
            __syncthreads();
            for (int base = e0; base < e1; base += 32) {
                const int idx = base + lane;
                const bool v = idx < e1;
                const uint16_t sl = v ? src[idx] : (uint16_t)0;
                const uint32_t d = v ? ((keys[sl] + 1u - kmin) >> shift) & (kBins - 1) : (uint32_t)kBins;
                const uint32_t peers = __match_any_sync(0xffffffffu, d);
                if (v) dst[counts[d * NW + warp] + __popc(peers & lanemask_lt())] = sl;
                __syncwarp();
                if (v && lane == __ffs(peers) - 1) counts[d * NW + warp] += (uint16_t)__popc(peers);
                __syncwarp();
            }
            __syncthreads();
            uint16_t* tmp = src;
            src = dst;
            dst = tmp;
        }
        victims = src;
    }

    // 4b. pair, unmap, map, stamp.
    __device__ void apply() {
        for (uint32_t r = threadIdx.x; r < m; r += NT) {
            const int32_t p = mpos[r];
            const int32_t v = victims[r];
            const int32_t o = tokb[v];
            if (o >= 0) ptb[o] = -1;
            ptb[p] = v;
            tokb[v] = p;
            lub[v] = t;
        }
    }

    // 4c. answers for the missed selections (their rank through the bitmap).
    __device__ __forceinline__ void answer(int j, int32_t p) {
        if (p < 0 || p >= lim) return;
        const int w = p >> 5;
        const uint32_t bit = 1u << (p & 31);
        const uint32_t word = posbm[w];
        if (!(word & bit)) return;  // a hit, already answered
        const int g = w / kGroupWords;
        uint32_t rank = gprefix[g];
        for (int q = g * kGroupWords; q < w; ++q) rank += __popc(posbm[q]);
        rank += __popc(word & (bit - 1u));
        const int32_t v = victims[rank];
        outb[j] = v;
        if (L.jslot) L.jslot[(size_t)b * k + j] = v;  // the fetch's copy, in device memory
    }

    // p: the selections this thread probed in the first batch (still in registers).
    __device__ void answer_misses(const int32_t (&p)[4]) {
        if (k <= 4 * NT) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int j = q * NT + threadIdx.x;
                if (j < k) answer(j, p[q]);
            }
        } else {
            for (int j = threadIdx.x; j < k; j += NT) answer(j, __ldg(selb + j));
        }
    }

    __device__ void finish(int32_t* miss_counts, uint32_t misses) {
        if (threadIdx.x == 0) {
            miss_counts[b] = (int32_t)misses;
            L.step[b] = t + 1;
        }
    }
};

// The resolution of request b by one CTA. With `pub` (fetch CTAs serve this call) it
// publishes the request's fetch list after the probe and the answers once the victims
// are chosen.
// `prev_all_hit`: the request's previous call had no miss, as far as its list flag tells
// (a hint for where the hits' answers are written; see Request::one_batch).
__device__ __forceinline__ void resolve_role(const Layout& L, uint8_t* smem, int b, const int32_t* __restrict__ sel,
                                             int k, int32_t* __restrict__ out, int32_t* __restrict__ miss_counts,
                                             bool pub, int32_t (&p)[4], bool prev_all_hit) {
    const Plan P(L.C, L.S);
    Request R(L, P, smem, b, sel, k, out);
    int32_t s[4];
    R.load_slots(p, s);  // p: the first batch of selections, already loaded
    // the call's stamp and tag (read once by every thread; both only change between calls)
    const int32_t t0 = *(volatile const int32_t*)(L.step + b);
    const uint32_t ready = ld_relaxed(L.gcount + b) + 1u;
    const bool direct = !R.one_batch() || prev_all_hit;
    // ready_pos carries the tag's low half in its high half and the miss count in its
    // low half, so a fetch CTA learns both from the one acquire load it waits on.
    const uint32_t tag = (ready & 0xffffu) << 16;
    uint32_t* rpos = L.ready_pos + (size_t)b * kFlagStride;
    uint32_t* rslot = L.ready_slot + (size_t)b * kFlagStride;
    R.start();
    __syncthreads();  // bitmaps cleared
    // With nothing to fetch the flags order nothing (the fetch reads no list and stores
    // no row), so they are raised with plain stores: a release would first wait for this
    // thread's earlier writes, a fence on the no-IO path.
    if (t0 == INT32_MAX) {  // refused: the request reached its call limit
        R.refuse(miss_counts);
        if (pub && threadIdx.x == 0) {
            st_relaxed(rpos, tag);
            st_relaxed(rslot, ready);
        }
        return;
    }
    R.t = t0;
    if (!R.probe(p, s, direct)) {  // all hits: nothing to rank or fetch
        if (pub && threadIdx.x == 0) {
            st_relaxed(rpos, tag);
            st_relaxed(rslot, ready);
        }
        R.write_direct(p, s, direct);
        R.finish(miss_counts, 0);
        R.drain();
        return;
    }
    // The fetch list is complete (the probe ended with a barrier, and the release is
    // cumulative over it): the fetch of this request's rows can start now.
    if (pub && threadIdx.x == 0) st_release(rpos, tag | R.scratch[2 * NW + 2]);
    R.prefetch_stamps();
    R.rank_misses();
    R.rank_victims();
    R.answer_misses(p);
    publish(rslot, ready, pub);  // the answers name the slots: the rows can be stored
    R.write_direct(p, s, direct);
    R.apply();
    R.finish(miss_counts, R.m);
}

// One fetch CTA's share of request b: entries q, q + nq, q + 2nq, ... of its fetch
// list (position p, selection index j); the row of p goes to slot out[b][j].
__device__ __forceinline__ void fetch_rows(const Layout& L, const int32_t* out, int k, int b, uint32_t q,
                                           uint32_t nq, uint32_t ready, bool sync, uint64_t deadline,
                                           uint32_t* bcast) {
    constexpr int GT = kGatherThreads;
    uint32_t v;
    if (sync) {
        if (!wait_flag(L.ready_pos + (size_t)b * kFlagStride, (ready & 0xffffu) << 16, 0xffff0000u, deadline, L.status, bcast, &v))
            return;
    } else {  // launched after the resolution: its hand-off is complete
        v = ld_relaxed(L.ready_pos + (size_t)b * kFlagStride);
    }
    const uint32_t u = v & 0xffffu;  // entries in the fetch list
    const uint32_t cpr = (uint32_t)L.E >> 4;
    const uint32_t rows = u > q ? (u - q + nq - 1) / nq : 0u;
    const uint32_t n = rows * cpr;
    const int32_t* gpos = L.fpos + (size_t)b * L.S;
    const int32_t* gsel = L.fsel + (size_t)b * L.S;
    const int32_t* ob = (L.jslot ? L.jslot : out) + (size_t)b * k;
    const uint8_t* hb = L.host + (size_t)(L.row_base ? __ldg(L.row_base + b) : (int64_t)b * L.C) * L.host_stride;
    uint8_t* db = L.dev + (size_t)b * L.S * L.E;
    bool slots_known = false;
    for (uint32_t base = 0; base < n; base += GT * kGatherUnroll) {
        uint4 val[kGatherUnroll];
#pragma unroll
        for (int u8 = 0; u8 < kGatherUnroll; ++u8) {
            const uint32_t c = base + (uint32_t)u8 * GT + threadIdx.x;
            if (c < n) {
                const uint32_t lr = c / cpr, off = c - lr * cpr;
                const int32_t p = __ldcg(gpos + q + nq * lr);
                val[u8] = __ldcs(reinterpret_cast<const uint4*>(hb + (size_t)p * L.host_stride) + off);
            }
        }
        if (!slots_known) {  // the loads above are in flight while the victims are ranked
            if (sync && !wait_flag(L.ready_slot + (size_t)b * kFlagStride, ready, 0xffffffffu, deadline, L.status, bcast, &v)) return;
            slots_known = true;
        }
#pragma unroll
        for (int u8 = 0; u8 < kGatherUnroll; ++u8) {
            const uint32_t c = base + (uint32_t)u8 * GT + threadIdx.x;
            if (c < n) {
                const uint32_t lr = c / cpr, off = c - lr * cpr;
                const int32_t slot = __ldcg(ob + __ldcg(gsel + q + nq * lr));
                reinterpret_cast<uint4*>(db + (size_t)slot * L.E)[off] = val[u8];
            }
        }
    }
}

// Request b's fetch by nq CTAs (this one is share q). The CTA's own counter for
// (b, q) gives the call's tag and advances once the share is done.
__device__ __forceinline__ void fetch_request(const Layout& L, const int32_t* out, int k, int b, uint32_t q,
                                              uint32_t nq, bool sync, uint64_t deadline, uint32_t* bcast) {
    uint32_t* count = L.gcount + b + (size_t)q * L.R;
    const uint32_t ready = ld_relaxed(count) + 1u;
    fetch_rows(L, out, k, b, q, nq, ready, sync, deadline, bcast);
    __syncthreads();
    if (threadIdx.x == 0) *count = ready;
}

// Fetch CTA c of G: with G >= R, CTAs c = b (mod R) share request b's list; with fewer,
// each takes whole requests in turn.
// Fetch CTA c of G serving requests b0 .. b0 + nr - 1: with G >= nr, CTAs c = i (mod nr)
// share request b0 + i's list; with fewer, each takes whole requests in turn. Share q of
// request b keeps its call counter at gcount[b + q * R].
__device__ __forceinline__ void fetch_role(const Layout& L, const int32_t* out, int k, uint32_t c, uint32_t G,
                                           bool sync, uint32_t* bcast, uint32_t b0, uint32_t nr) {
    const uint64_t deadline = global_ns() + L.wait_ns;  // every wait of this CTA ends by then
    if (G >= nr) {  // several CTAs share each request
        const uint32_t i = c % nr;
        fetch_request(L, out, k, (int)(b0 + i), c / nr, (G - 1 - i) / nr + 1, sync, deadline, bcast);
    } else {  // each CTA takes whole requests
        for (uint32_t i = c; i < nr; i += G) fetch_request(L, out, k, (int)(b0 + i), 0, 1, sync, deadline, bcast);
    }
}

// The resolution of requests b0 .. b0 + gridDim.x - 1: one CTA per request. Launched as
// a programmatic dependent of the preceding grid. The selections are the caller's input,
// complete before the call was enqueued (a kernel that writes them lets this one start
// only when it finishes, or when it has signalled programmatic completion after writing
// them), so the first batch is loaded before the wait; nothing the previous call writes
// is read before that grid (and, through its own wait, the previous resolution) is done.
// A later chunk of a call's requests (`wait` = 0) does not wait: it is launched behind the
// first chunk's fetch, which starts only once every CTA of the first chunk has passed its
// wait -- the previous call is complete by then -- and its requests are disjoint from the
// earlier chunks', so it runs under their fetch.
__global__ void __launch_bounds__(kResolveThreads, 2)
resolve_kernel(const Layout L, const int32_t* __restrict__ sel, int k, int32_t* __restrict__ out,
               int32_t* __restrict__ miss_counts, int fetch, int b0, int wait) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int b = b0 + (int)blockIdx.x;
    int32_t p[4];
    load_selections(sel + (size_t)b * k, k, 0, p);
    // The previous call's miss count, from its list flag: only a hint (a stale value costs
    // time, not correctness), so it too is read before the wait.
    const uint32_t prev = ld_relaxed(L.ready_pos + (size_t)b * kFlagStride);
    if (wait) pdl_wait_prerequisites();
    pdl_launch_dependents();  // the fetch grid may start now; it synchronizes per request
    // Flags are raised only when a fetch grid follows (it advances the counters) and no
    // stall is being injected.
    resolve_role(L, smem, b, sel, k, out, miss_counts, fetch != 0 && !L.no_publish, p, (prev & 0xffffu) == 0);
}

// The fetch of a call, held to 64 registers so that it is resident beside a resolution CTA
// from the start. With `sync` it is a programmatic dependent of the resolution and waits
// for each request's flags; without, it runs after the resolution and reads the hand-off
// as it is.
__global__ void __launch_bounds__(kGatherThreads, 2)
gather_kernel(const Layout L, const int32_t* __restrict__ out, int k, int sync, int b0, int nr) {
    __shared__ uint32_t bcast[2];
    // The next call's resolution may be scheduled once every fetch CTA is resident (it
    // waits for this grid to finish before it reads anything).
    pdl_launch_dependents();
    fetch_role(L, out, k, blockIdx.x, gridDim.x, sync != 0, bcast, (uint32_t)b0, (uint32_t)nr);
    // This grid ends only after the resolution it serves: a successor that waits for this
    // grid then also sees every table update of that resolution.
    pdl_wait_prerequisites();
}

}  // namespace

size_t resolve_smem_bytes(int C, int S) { return Plan(C, S).fixed; }

size_t miss_area_bytes(int R, int S, int num_sms) {
    const size_t list = ((size_t)R * S * 4 + 15) & ~(size_t)15;
    const size_t per = (size_t)R * kFlagStride * 4;
    // share q of request b counts at b + q * R: a fetch grid of G = num_sms CTAs over a chunk
    // of nr requests gives each request ceil(G / nr) shares at most, which is at most
    // R + G counters in all when one chunk holds every request (R <= G) and at most 2R
    // when chunks hold at least G / 2 requests each (R > G; see chunk_requests)
    const size_t counters = (size_t)R + (size_t)(R > num_sms ? R : num_sms * kGatherCtasPerSm);
    return 2 * list + 2 * per + counters * 4;
}

void carve_miss_area(Layout& L, void* base) {
    uint8_t* p = static_cast<uint8_t*>(base);
    const size_t list = ((size_t)L.R * L.S * 4 + 15) & ~(size_t)15;
    const size_t per = (size_t)L.R * kFlagStride * 4;
    L.fpos = reinterpret_cast<int32_t*>(p);
    L.fsel = reinterpret_cast<int32_t*>(p + list);
    p += 2 * list;
    L.ready_pos = reinterpret_cast<uint32_t*>(p);
    L.ready_slot = reinterpret_cast<uint32_t*>(p + per);
    L.gcount = reinterpret_cast<uint32_t*>(p + 2 * per);
}

cudaError_t configure_kernels(int device) {
    // The attribute is per kernel, not per context: opt in to the device maximum once,
    // so that contexts of different sizes never lower each other's limit.
    int optin = 0;
    cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, resolve_kernel)) != cudaSuccess) return e;
    return cudaFuncSetAttribute(resolve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                optin - (int)fa.sharedSizeBytes);
}

cudaError_t launch_resolve(const Layout& L, cudaStream_t stream, const int32_t* sel, int k,
                           int32_t* out_slots, int32_t* miss_counts, bool fetch, int b0, int nr, bool wait) {
    // a programmatic dependent of whatever precedes it on the stream: it is scheduled early
    // only behind a grid that allows it (the previous call's fetch), and waits for that
    // grid's completion before its first read
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)nr);
    cfg.blockDim = dim3(kResolveThreads);
    cfg.dynamicSmemBytes = resolve_smem_bytes(L.C, L.S);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, resolve_kernel, L, sel, k, out_slots, miss_counts, fetch ? 1 : 0, b0,
                              wait ? 1 : 0);
}

cudaError_t launch_gather(const Layout& L, cudaStream_t stream, const int32_t* out_slots, int k, int num_sms,
                          bool pdl, int b0, int nr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(num_sms * kGatherCtasPerSm));
    cfg.blockDim = dim3(kGatherThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gather_kernel, L, out_slots, k, pdl ? 1 : 0, b0, nr);
}

}  // namespace hs
