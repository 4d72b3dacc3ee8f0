// hs_kernels.cu -- the two kernels of one HiSparse swap-in resolution step, sm_103a.
//
// HiSparse resolves each layer's top-k selections with one fused step: hit detection,
// LRU replacement, the page-table update and the host-to-device fetch (paper
// abstract; blog commentary, section three). Here the step is two kernels chained by
// programmatic dependent launch, so it stays one enqueue with no host round trip:
//
//  resolve_kernel  one CTA per request. Probes the page table for every selected
//                  position (hits are stamped and answered in place), marks misses
//                  in a position bitmap (ascending-position rank = prefix popcount),
//                  compacts the non-hit slots in slot order and ranks them by
//                  (last_use, slot) with a stable LSD radix sort whose digits are
//                  counted per warp (__match_any_sync ranks equal digits inside a
//                  warp, a per-(digit, warp) exclusive scan orders the warps), pairs
//                  the r-th miss with the r-th victim, updates page table / slot
//                  tokens / stamps, and writes the miss list (position, slot).
//  gather_kernel   a fixed persistent grid (2 CTAs per SM) that streams every miss
//                  row from the mapped host store into its HBM slot with coalesced
//                  16-byte loads, kGatherUnroll of them in flight per thread.
//
// No tensor cores: nothing here is a contraction. The resolution is latency bound
// (one dependent probe round plus shared-memory work); the fetch is bound by the
// host link.
#include <cuda_runtime.h>
#include <stdint.h>

#include "hs_internal.h"

#define HS_STATUS_RANGE 1u
#define HS_STATUS_DUP 2u
#define HS_STATUS_STEP_LIMIT 4u

namespace hs {
namespace {

__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Exclusive scan of one value per thread over an NT-thread block. `scratch` holds
// NT/32 + 1 words of shared memory; *total receives the block sum. Every thread
// of the block must call it (three barriers).
template <int NT>
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* scratch,
                                                         uint32_t* total) {
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < NW ? scratch[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < NW) scratch[lane] = w;
        if (lane == NW - 1) scratch[NW] = w;
    }
    __syncthreads();
    const uint32_t r = (warp == 0 ? 0u : scratch[warp - 1]) + x - v;
    *total = scratch[NW];
    __syncthreads();
    return r;
}

struct SmemPlan {
    int CW, CG, SW, S2;
    __host__ __device__ SmemPlan(int C, int S) {
        CW = ((C + 31) / 32 + kGroupWords - 1) / kGroupWords * kGroupWords;
        CG = CW / kGroupWords;
        SW = (S + 31) / 32;
        S2 = (S + 1) & ~1;
    }
    // word offsets
    __host__ __device__ int posbm() const { return 0; }
    __host__ __device__ int gprefix() const { return CW; }
    __host__ __device__ int hitbm() const { return CW + CG; }
    __host__ __device__ int keys(int) const { return CW + CG + SW; }
    __host__ __device__ int counts(int S) const { return keys(S) + S; }
    __host__ __device__ int scratch(int S) const { return counts(S) + kBins * kResolveWarps; }
    __host__ __device__ int slots(int S) const { return scratch(S) + 40; }
    __host__ __device__ size_t bytes(int S) const {
        return (size_t)slots(S) * 4 + (size_t)2 * S2 * sizeof(uint16_t);
    }
};

__global__ void __launch_bounds__(kResolveThreads, 2)
resolve_kernel(const Layout L, const int32_t* __restrict__ sel, int k, int32_t* __restrict__ out,
               int32_t* __restrict__ miss_counts) {
    constexpr int NT = kResolveThreads;
    extern __shared__ __align__(16) uint32_t smem[];
    const int C = L.C, S = L.S;
    const SmemPlan P(C, S);
    uint32_t* posbm = smem + P.posbm();     // missed positions of this call
    uint32_t* gprefix = smem + P.gprefix(); // misses before each group of kGroupWords words
    uint32_t* hitbm = smem + P.hitbm();     // slots hit in this call
    uint32_t* keys = smem + P.keys(S);      // last_use + 1 per slot; later miss positions by rank
    uint32_t* counts = smem + P.counts(S);  // radix digit counts, [digit][warp]
    uint32_t* scratch = smem + P.scratch(S);
    uint16_t* sa = reinterpret_cast<uint16_t*>(smem + P.slots(S));
    uint16_t* sb = sa + P.S2;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x;
    const int32_t* selb = sel + (size_t)b * k;
    int32_t* outb = out + (size_t)b * k;
    int32_t* ptb = L.pt + (size_t)b * C;
    int32_t* tokb = L.tok + (size_t)b * S;
    int32_t* lub = L.lu + (size_t)b * S;

    // The fetch kernel may be scheduled now; it waits for this grid to finish.
    pdl_launch_dependents();

    const int32_t t = L.step[b];
    for (int i = tid; i < P.CW; i += NT) posbm[i] = 0u;
    for (int i = tid; i < P.SW; i += NT) hitbm[i] = 0u;
    __syncthreads();

    if (t == INT32_MAX) {  // stamps would wrap: refuse the call for this request
        for (int j = tid; j < k; j += NT) outb[j] = -1;
        if (tid == 0) {
            atomicOr(L.status, HS_STATUS_STEP_LIMIT);
            miss_counts[b] = 0;
            L.mcnt[b] = 0;
        }
        return;
    }

    // ---- 1. hit detection: probe the page table, four selections per thread in flight
    uint32_t st = 0;
    int any_miss = 0;
    for (int j0 = 0; j0 < k; j0 += 4 * NT) {
        int32_t p[4], s[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int j = j0 + q * NT + tid;
            p[q] = j < k ? __ldg(selb + j) : -1;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) s[q] = (p[q] >= 0 && p[q] < C) ? ptb[p[q]] : -1;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int j = j0 + q * NT + tid;
            if (j >= k) continue;
            const int32_t pp = p[q], ss = s[q];
            if (ss >= 0) {  // hit: answered in place, stamped, not evictable
                const uint32_t bit = 1u << (ss & 31);
                if (atomicOr(&hitbm[ss >> 5], bit) & bit) st |= HS_STATUS_DUP;
                lub[ss] = t;
                outb[j] = ss;
            } else if (pp >= 0 && pp < C) {  // miss
                const uint32_t bit = 1u << (pp & 31);
                if (atomicOr(&posbm[pp >> 5], bit) & bit) st |= HS_STATUS_DUP;
                any_miss = 1;
            } else {  // padding, or out of range
                if (pp >= C) st |= HS_STATUS_RANGE;
                outb[j] = -1;
            }
        }
    }
    if (st) atomicOr(L.status, st);
    if (!__syncthreads_or(any_miss)) {  // all hits: nothing to rank or fetch
        if (tid == 0) {
            miss_counts[b] = 0;
            L.mcnt[b] = 0;
            L.step[b] = t + 1;
        }
        return;
    }

    // ---- 2. count misses per bitmap group and non-hit slots per hit-bitmap word
    const int gpt = (P.CG + NT - 1) / NT;
    const int g0 = min(tid * gpt, P.CG), g1 = min(g0 + gpt, P.CG);
    const int wpt = (P.SW + NT - 1) / NT;
    const int w0 = min(tid * wpt, P.SW), w1 = min(w0 + wpt, P.SW);
    const uint32_t tail_mask = (S & 31) ? ((1u << (S & 31)) - 1u) : 0xffffffffu;

    for (int s = tid; s < S; s += NT) keys[s] = (uint32_t)(lub[s] + 1);

    uint32_t nmiss = 0, ncand = 0;
    for (int g = g0; g < g1; ++g)
#pragma unroll
        for (int q = 0; q < kGroupWords; ++q) nmiss += __popc(posbm[g * kGroupWords + q]);
    for (int w = w0; w < w1; ++w) ncand += __popc(~hitbm[w] & (w == P.SW - 1 ? tail_mask : 0xffffffffu));

    // one scan for both counts: misses in the low 16 bits, candidates in the high 16
    uint32_t total;
    const uint32_t excl = block_exclusive_scan<NT>((ncand << 16) | nmiss, scratch, &total);
    const uint32_t m = total & 0xffffu, N = total >> 16;
    const uint32_t miss_base = excl & 0xffffu;

    {
        uint32_t r = miss_base;
        for (int g = g0; g < g1; ++g) {
            gprefix[g] = r;
#pragma unroll
            for (int q = 0; q < kGroupWords; ++q) r += __popc(posbm[g * kGroupWords + q]);
        }
    }

    // ---- 3. non-hit slots in slot order, and the range of their keys
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    {
        uint32_t c = excl >> 16;
        for (int w = w0; w < w1; ++w) {
            uint32_t bits = ~hitbm[w] & (w == P.SW - 1 ? tail_mask : 0xffffffffu);
            while (bits) {
                const int s = w * 32 + __ffs(bits) - 1;
                bits &= bits - 1;
                sa[c++] = (uint16_t)s;
                const uint32_t key = keys[s];
                kmin = min(kmin, key);
                kmax = max(kmax, key);
            }
        }
    }
    kmin = __reduce_min_sync(0xffffffffu, kmin);
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    if (lane == 0) {
        scratch[warp] = kmin;
        scratch[kResolveWarps + warp] = kmax;
    }
    __syncthreads();
    if (tid == 0) {
        uint32_t a = scratch[0], z = scratch[kResolveWarps];
        for (int i = 1; i < kResolveWarps; ++i) {
            a = min(a, scratch[i]);
            z = max(z, scratch[kResolveWarps + i]);
        }
        scratch[2 * kResolveWarps] = a;
        scratch[2 * kResolveWarps + 1] = z;
    }
    __syncthreads();
    kmin = scratch[2 * kResolveWarps];
    kmax = scratch[2 * kResolveWarps + 1];
    __syncthreads();  // scratch is reused by the scans below

    // ---- 4. LRU order: stable LSD radix sort of the candidates on last_use + 1
    const uint32_t range = kmax - kmin;
    const int npass = range ? (32 - __clz(range) + kRadixBits - 1) / kRadixBits : 0;
    const int seg = (((int)N + kResolveWarps - 1) / kResolveWarps + 31) & ~31;
    const int s0 = min(warp * seg, (int)N), s1 = min(s0 + seg, (int)N);
    uint16_t* src = sa;
    uint16_t* dst = sb;
    for (int pass = 0; pass < npass; ++pass) {
        const int shift = pass * kRadixBits;
        for (int i = tid; i < kBins * kResolveWarps; i += NT) counts[i] = 0u;
        __syncthreads();
        for (int base = s0; base < s1; base += 32) {
            const int idx = base + lane;
            const bool v = idx < s1;
            const uint32_t d = v ? ((keys[src[idx]] - kmin) >> shift) & (kBins - 1) : (uint32_t)kBins;
            const uint32_t peers = __match_any_sync(0xffffffffu, d);
            if (v && lane == __ffs(peers) - 1) counts[d * kResolveWarps + warp] += __popc(peers);
        }
        __syncthreads();
        {
            constexpr int PER = kBins * kResolveWarps / NT;
            uint32_t loc[PER], sum = 0;
#pragma unroll
            for (int q = 0; q < PER; ++q) {
                loc[q] = counts[tid * PER + q];
                sum += loc[q];
            }
            uint32_t tot;
            uint32_t ex = block_exclusive_scan<NT>(sum, scratch, &tot);
#pragma unroll
            for (int q = 0; q < PER; ++q) {
                counts[tid * PER + q] = ex;
                ex += loc[q];
            }
        }
        __syncthreads();
        for (int base = s0; base < s1; base += 32) {
            const int idx = base + lane;
            const bool v = idx < s1;
            const uint16_t sl = v ? src[idx] : (uint16_t)0;
            const uint32_t d = v ? ((keys[sl] - kmin) >> shift) & (kBins - 1) : (uint32_t)kBins;
            const uint32_t peers = __match_any_sync(0xffffffffu, d);
            if (v) dst[counts[d * kResolveWarps + warp] + __popc(peers & lanemask_lt())] = sl;
            __syncwarp();
            if (v && lane == __ffs(peers) - 1) counts[d * kResolveWarps + warp] += __popc(peers);
            __syncwarp();
        }
        __syncthreads();
        uint16_t* tmp = src;
        src = dst;
        dst = tmp;
    }
    const uint16_t* victims = src;  // victims[r] = the slot the r-th miss takes

    // ---- 5. misses by rank (ascending position), then unmap / map / stamp
    uint32_t* mpos = keys;  // keys are dead after the sort
    {
        uint32_t r = miss_base;
        for (int g = g0; g < g1; ++g)
            for (int q = 0; q < kGroupWords; ++q) {
                const int w = g * kGroupWords + q;
                uint32_t bits = posbm[w];
                while (bits) {
                    mpos[r++] = (uint32_t)(w * 32 + __ffs(bits) - 1);
                    bits &= bits - 1;
                }
            }
    }
    __syncthreads();
    int2* mlb = L.mlist + (size_t)b * S;
    for (uint32_t r = tid; r < m; r += NT) {
        const int32_t p = (int32_t)mpos[r];
        const int32_t v = victims[r];
        const int32_t o = tokb[v];
        if (o >= 0) ptb[o] = -1;
        ptb[p] = v;
        tokb[v] = p;
        lub[v] = t;
        mlb[r] = make_int2(p, v);
    }

    // ---- 6. answers for the missed selections
    for (int j = tid; j < k; j += NT) {
        const int32_t p = __ldg(selb + j);
        if (p < 0 || p >= C) continue;
        const int w = p >> 5;
        const uint32_t bit = 1u << (p & 31);
        const uint32_t word = posbm[w];
        if (!(word & bit)) continue;  // a hit, already answered
        const int g = w / kGroupWords;
        uint32_t rank = gprefix[g];
        for (int q = g * kGroupWords; q < w; ++q) rank += __popc(posbm[q]);
        rank += __popc(word & (bit - 1u));
        outb[j] = victims[rank];
    }
    if (tid == 0) {
        miss_counts[b] = (int32_t)m;
        L.mcnt[b] = (int32_t)m;
        L.step[b] = t + 1;
    }
}

__global__ void __launch_bounds__(kGatherThreads, kGatherCtasPerSm)
gather_kernel(const Layout L) {
    constexpr int NT = kGatherThreads;
    extern __shared__ __align__(16) uint32_t pref[];  // R + 1 row offsets, then scan scratch
    uint32_t* scratch = pref + L.R + 1;
    const int tid = threadIdx.x;
    const int R = L.R;

    pdl_wait_primary();  // the resolution kernel's miss list is complete and visible

    const int per = (R + NT - 1) / NT;
    const int r0 = min(tid * per, R), r1 = min(r0 + per, R);
    uint32_t sum = 0;
    for (int i = r0; i < r1; ++i) {
        const uint32_t c = (uint32_t)L.mcnt[i];
        pref[i] = c;
        sum += c;
    }
    uint32_t total;
    uint32_t ex = block_exclusive_scan<NT>(sum, scratch, &total);
    for (int i = r0; i < r1; ++i) {
        const uint32_t c = pref[i];
        pref[i] = ex;
        ex += c;
    }
    __syncthreads();

    const uint32_t cpr = (uint32_t)L.E >> 4;  // 16-byte chunks per row
    const uint32_t nchunks = total * cpr;
    const uint32_t T = gridDim.x * NT;
    for (uint32_t base = blockIdx.x * NT + tid; base < nchunks; base += T * kGatherUnroll) {
        uint4 val[kGatherUnroll];
        uint4* dptr[kGatherUnroll];
#pragma unroll
        for (int u = 0; u < kGatherUnroll; ++u) {
            const uint32_t c = base + (uint32_t)u * T;
            dptr[u] = nullptr;
            if (c < nchunks) {
                const uint32_t row = c / cpr, off = c - row * cpr;
                int lo = 0, hi = R - 1;  // the request: last b with pref[b] <= row
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (pref[mid] <= row) lo = mid; else hi = mid - 1;
                }
                const int2 e = L.mlist[(size_t)lo * L.S + (row - pref[lo])];
                const uint4* s = reinterpret_cast<const uint4*>(
                                     L.host + ((size_t)lo * L.C + (uint32_t)e.x) * L.host_stride) + off;
                dptr[u] = reinterpret_cast<uint4*>(L.dev + ((size_t)lo * L.S + (uint32_t)e.y) * L.E) + off;
                val[u] = __ldcs(s);
            }
        }
#pragma unroll
        for (int u = 0; u < kGatherUnroll; ++u)
            if (dptr[u]) *dptr[u] = val[u];
    }
}

}  // namespace

size_t resolve_smem_bytes(int C, int S) { return SmemPlan(C, S).bytes(S); }

size_t gather_smem_bytes(int R) { return (size_t)(R + 1 + kGatherThreads / 32 + 1) * 4; }

cudaError_t configure_kernels(int device) {
    // The attribute is per kernel, not per context: opt in to the device maximum once,
    // so that contexts of different sizes never lower each other's limit.
    int optin = 0;
    cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(resolve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
}

cudaError_t launch_resolve(const Layout& L, cudaStream_t stream, const int32_t* sel, int k,
                           int32_t* out_slots, int32_t* miss_counts) {
    resolve_kernel<<<L.R, kResolveThreads, resolve_smem_bytes(L.C, L.S), stream>>>(L, sel, k, out_slots,
                                                                                   miss_counts);
    return cudaGetLastError();
}

cudaError_t launch_gather(const Layout& L, cudaStream_t stream, int num_sms, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(num_sms * kGatherCtasPerSm));
    cfg.blockDim = dim3(kGatherThreads);
    cfg.dynamicSmemBytes = gather_smem_bytes(L.R);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gather_kernel, L);
}

}  // namespace hs
