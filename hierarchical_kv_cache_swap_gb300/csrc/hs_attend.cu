// hs_attend.cu -- the consumer: sparse MLA-style decode attention over the resolved
// slots, on the fifth-generation tensor cores (tcgen05) of sm_103a.
//
// After a resolution every selected entry sits in a device slot, and the layer's sparse
// attention reads it there (blog commentary, section two: a resident entry takes part
// in the computation directly; paper abstract: only KV placement changes, so outputs are
// unchanged). For the 656-byte entries of the DeepSeek sparse-attention family -- 512
// E4M3 latent codes with four fp32 block scales, then 64 bf16 rotary values -- the
// attention is an MLA decode in its absorbed form: key K_j = (latent_j, rope_j) in
// R^576, value V_j = latent_j in R^512, per head s_hj = sm_scale * <q_h, K_j> over the
// selections whose slot is valid, o_h = softmax(s_h) V, lse_h = ln sum_j exp(s_hj).
//
// attend_kernel: one CTA per (request b, key split s, value half v), 416 threads, one CTA
// per SM (222 KB of shared memory, 512 TMEM columns).
//   * Q [128 heads x 576] bf16 stays in shared memory for the whole CTA, in the 128-byte
//     swizzled K-major layout the MMA reads (heads beyond H are zero rows).
//   * 8 producer warps gather blocks of 32 selected entries through out_slots (one key
//     per lane, one 64-dimension slice per warp), decode the E4M3 codes times their
//     block scale to bf16 and store them swizzled into one of two stages: the stage is
//     K (K-major, 576 wide) for S = Q K^T and, read MN-major, V (256 wide, this CTA's
//     half) for O += P V -- one copy serves both products.
//   * one thread issues the MMAs: S (M=128 heads, N=32 keys, K=576) into TMEM, and
//     O += P V (M=128, N=256, K=32) with P read from TMEM; completion is signalled
//     through mbarriers by tcgen05.commit.
//   * 4 softmax warps (thread = head = TMEM lane) read S, keep a running maximum m (log2
//     domain) that moves only when a block's maximum exceeds it by more than 8 -- then O
//     (in TMEM) and the running sum are rescaled -- and write P = 2^(x - m) as bf16 into
//     TMEM; at the end they normalise O and write it with lse.
// With several key splits per request each CTA writes its normalised partial and its
// lse; combine_kernel merges them (weights exp(lse_s - lse)).
//
// Every wait on an mbarrier is bounded: on expiry the CTA records HS_STATUS_TIMEOUT,
// every role leaves its loop, the MMA thread waits (bounded) for its own MMAs, and the
// TMEM columns are freed before the CTA exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "hs_internal.h"

namespace hs {
namespace {

constexpr int kHeads = 128;    // MMA rows
constexpr int kDimK = 576;     // 512 latent + 64 rotary
constexpr int kDimV = 512;
constexpr int kHalfV = 256;    // value dimensions per CTA
constexpr int kBlk = 32;       // keys per stage
constexpr int kChunks = kDimK / 64;                  // 64-element (128-byte) swizzle columns
constexpr uint32_t kQChunk = kHeads * 128;           // bytes of one Q column chunk
constexpr uint32_t kKChunk = kBlk * 128;             // bytes of one stage column chunk
constexpr uint32_t kQBytes = kQChunk * kChunks;      // 147456
constexpr uint32_t kStageBytes = kKChunk * kChunks;  // 36864
constexpr int kSoftWarps = 4, kProdWarps = 8;
constexpr int kThreads = (kSoftWarps + kProdWarps + 1) * 32;  // 416
constexpr int kMmaWarp = kSoftWarps + kProdWarps;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256, kColP = 320;  // S[st] at 256+32st, P[st] at 320+16st
constexpr float kRescaleLog2 = 8.0f;
constexpr uint32_t kWaitLimit = 1u << 22;  // polls of an mbarrier before giving up

// barrier indices
enum { kQFull = 0, kKvFull = 1, kKvFree = 3, kSFull = 5, kPFull = 7, kPvDone = 9, kOFull = 11, kDrain = 12, kBars = 13 };

struct Smem {  // beyond Q and the two stages
    uint64_t bar[kBars];
    uint32_t vmask[2];  // valid keys of each stage
    uint32_t tmem;
    volatile int abort;
};
constexpr uint32_t kSmemBytes = 1024 + kQBytes + 2 * kStageBytes + sizeof(Smem);

struct AttendArgs {
    const uint8_t* dev;        // [R][S][656]
    int S;
    const uint16_t* q;         // [B][H][576] bf16
    int H;
    const int32_t* out_slots;  // [B][k]
    int k;
    int nsplit, keys_per_split;
    float scale_log2;          // sm_scale * log2(e)
    float* o;                  // nsplit == 1: [B][H][512]; else partials [B][nsplit][H][512]
    float* lse;                // nsplit == 1: [B][H];      else partials [B][nsplit][H]
    uint32_t* status;
};

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// ---------------------------------------------------------------- mbarriers
__device__ __forceinline__ void bar_init(uint64_t* b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint64_t* b) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool bar_try(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok) : "r"(su32(b)), "r"(parity) : "memory");
    return ok != 0;
}
// Waits for the phase of `parity` to complete; false (and the CTA aborted) on expiry or
// when another role has aborted.
__device__ __forceinline__ bool bar_wait(Smem* sm, uint64_t* b, uint32_t parity, uint32_t* status) {
    for (uint32_t i = 0; i < kWaitLimit; ++i) {
        if (bar_try(b, parity)) return true;
        if (sm->abort) return false;
    }
    sm->abort = 1;
    atomicOr(status, 8u /* HS_STATUS_TIMEOUT */);
    return false;
}

// The same wait taken by a whole warp whose next step is warp-collective: all lanes go on
// or none does.
__device__ __forceinline__ bool warp_wait(Smem* sm, uint64_t* b, uint32_t parity, uint32_t* status) {
    return __all_sync(0xffffffffu, bar_wait(sm, b, parity, status));
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) /* descriptor version */ |
           (2ull << 61) /* 128-byte swizzle */;
}
// kind::f16 instruction descriptor: D f32, A and B bf16, A K-major, B K- or MN-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile("{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
                 ::"r"(d), "l"(a), "l"(b), "r"(id), "r"(acc) : "memory");
}
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile("{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }"
                 ::"r"(d), "r"(a_tmem), "l"(b), "r"(id), "r"(acc) : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* b) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

#define HS_LD32(r, addr)                                                                                       \
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15," \
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"                    \
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),          \
                   "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),      \
                   "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),   \
                   "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),   \
                   "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])                                           \
                 : "r"(addr))
#define HS_ST32(addr, r)                                                                                       \
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14," \
                 "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"                   \
                 ::"r"(addr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),      \
                   "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), \
                   "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),          \
                   "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),          \
                   "r"(r[29]), "r"(r[30]), "r"(r[31])                                                          \
                 : "memory")
#define HS_ST16(addr, r)                                                                                       \
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14," \
                 "%15,%16};"                                                                                   \
                 ::"r"(addr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),      \
                   "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), \
                   "r"(r[15])                                                                                  \
                 : "memory")
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two E4M3 codes (low byte -> low half) to f16x2; the conversion is exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t c) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(c));
    return h;
}
// Eight codes (one 8-byte word) times `scale` -> eight bf16 (one 16-byte unit).
__device__ __forceinline__ uint4 decode8(uint32_t lo, uint32_t hi, float scale) {
    uint32_t w[4] = {lo & 0xFFFFu, lo >> 16, hi & 0xFFFFu, hi >> 16};
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t h = e4m3x2_to_f16x2((uint16_t)w[i]);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
        const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
        out[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

// Byte offset of 16-byte unit u (0..7) of row r in a 128-byte-swizzled column chunk.
__device__ __forceinline__ uint32_t swz(int r, int u) { return (uint32_t)(r * 128 + ((u ^ (r & 7)) << 4)); }

__global__ void __launch_bounds__(kThreads, 1) attend_kernel(const AttendArgs A) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = base;
    uint8_t* sK = base + kQBytes;  // stage st at sK + st * kStageBytes
    Smem* sm = reinterpret_cast<Smem*>(base + kQBytes + 2 * kStageBytes);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int v = blockIdx.x & 1;
    const int split = (blockIdx.x >> 1) % A.nsplit;
    const int b = (blockIdx.x >> 1) / A.nsplit;
    const int kbeg = split * A.keys_per_split;
    const int kend = min(A.k, kbeg + A.keys_per_split);
    const int nb = kend > kbeg ? (kend - kbeg + kBlk - 1) / kBlk : 0;

    if (tid == 0) {
        bar_init(&sm->bar[kQFull], kProdWarps * 32);
        for (int st = 0; st < 2; ++st) {
            bar_init(&sm->bar[kKvFull + st], kProdWarps * 32);
            bar_init(&sm->bar[kKvFree + st], 1);
            bar_init(&sm->bar[kSFull + st], 1);
            bar_init(&sm->bar[kPFull + st], kSoftWarps * 32);
            bar_init(&sm->bar[kPvDone + st], 1);
        }
        bar_init(&sm->bar[kOFull], 1);
        bar_init(&sm->bar[kDrain], 1);
        sm->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&sm->tmem)),
                     "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = sm->tmem;

    if (warp >= kSoftWarps && warp < kMmaWarp) {
        // ------------------------------------------------------------ producers
        const int pw = warp - kSoftWarps;  // the 64-dimension slice (and rotary unit) of this warp
        const int ptid = tid - kSoftWarps * 32;
        {  // Q, once: rows h < H of request b, zero rows beyond
            const uint4* qb = reinterpret_cast<const uint4*>(A.q + (size_t)b * A.H * kDimK);
            for (int u = ptid; u < kHeads * (kDimK / 8); u += kProdWarps * 32) {
                const int h = u / (kDimK / 8), cu = u - h * (kDimK / 8);
                const uint4 val = h < A.H ? __ldg(qb + (size_t)h * (kDimK / 8) + cu) : make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(sQ + (cu >> 3) * kQChunk + swz(h, cu & 7)) = val;
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            bar_arrive(&sm->bar[kQFull]);
        }
        const int32_t* slots = A.out_slots + (size_t)b * A.k;
        for (int i = 0; i < nb; ++i) {
            const int st = i & 1;
            const int j = kbeg + i * kBlk + lane;
            int32_t s = j < kend ? __ldg(slots + j) : -1;
            const bool valid = s >= 0 && s < A.S;
            uint4 c[4];
            uint4 rope = make_uint4(0, 0, 0, 0);
            float scale = 0.f;
            if (valid) {
                const uint8_t* row = A.dev + ((size_t)b * A.S + s) * 656;
                const uint4* cr = reinterpret_cast<const uint4*>(row + 64 * pw);
#pragma unroll
                for (int q = 0; q < 4; ++q) c[q] = __ldg(cr + q);
                scale = __ldg(reinterpret_cast<const float*>(row + 512) + (pw >> 1));
                rope = __ldg(reinterpret_cast<const uint4*>(row + 528) + pw);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) c[q] = make_uint4(0, 0, 0, 0);
            }
            if (i >= 2 && !bar_wait(sm, &sm->bar[kKvFree + st], ((i >> 1) & 1) ^ 1, A.status)) break;
            uint8_t* stg = sK + st * kStageBytes;
            uint8_t* col = stg + pw * kKChunk;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                *reinterpret_cast<uint4*>(col + swz(lane, 2 * q)) = decode8(c[q].x, c[q].y, scale);
                *reinterpret_cast<uint4*>(col + swz(lane, 2 * q + 1)) = decode8(c[q].z, c[q].w, scale);
            }
            *reinterpret_cast<uint4*>(stg + 8 * kKChunk + swz(lane, pw)) = rope;
            if (pw == 0) {
                const uint32_t m = __ballot_sync(0xffffffffu, valid);
                if (lane == 0) sm->vmask[st] = m;
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            bar_arrive(&sm->bar[kKvFull + st]);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issue (one thread)
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16(kHeads, kBlk, 0);
            const uint32_t id_o = idesc_bf16(kHeads, kHalfV, 1);
            const uint32_t q0 = su32(sQ), k0 = su32(sK);
            bool ok = bar_wait(sm, &sm->bar[kQFull], 0, A.status);
            auto do_pv = [&](int ib) -> bool {
                const int st = ib & 1;
                if (!bar_wait(sm, &sm->bar[kPFull + st], (ib >> 1) & 1, A.status)) return false;
                fence_after();
                const uint32_t vb = k0 + st * kStageBytes + (uint32_t)(4 * v) * kKChunk;
#pragma unroll
                for (int ks = 0; ks < kBlk / 16; ++ks)
                    mma_ts(tmem + kColO, tmem + kColP + 16 * st + 8 * ks,
                           smem_desc(vb + ks * 2048, kKChunk, 1024), id_o, (ib > 0 || ks > 0) ? 1u : 0u);
                mma_commit(&sm->bar[kKvFree + st]);
                mma_commit(&sm->bar[kPvDone + st]);
                return true;
            };
            for (int i = 0; ok && i < nb; ++i) {
                const int st = i & 1;
                if (!bar_wait(sm, &sm->bar[kKvFull + st], (i >> 1) & 1, A.status)) { ok = false; break; }
                fence_after();
                const uint32_t kb = k0 + st * kStageBytes;
#pragma unroll 4
                for (int kk = 0; kk < kDimK / 16; ++kk) {
                    const uint32_t c = kk >> 2, w = (kk & 3) * 32;
                    mma_ss(tmem + kColS + 32 * st, smem_desc(q0 + c * kQChunk + w, 16, 1024),
                           smem_desc(kb + c * kKChunk + w, 16, 1024), id_s, kk > 0 ? 1u : 0u);
                }
                mma_commit(&sm->bar[kSFull + st]);
                if (i > 0 && !do_pv(i - 1)) { ok = false; break; }
            }
            if (ok && nb > 0) ok = do_pv(nb - 1);
            if (ok) mma_commit(&sm->bar[kOFull]);
            // whatever happened, every MMA issued here completes before the columns are freed
            mma_commit(&sm->bar[kDrain]);
            for (uint32_t it = 0; it < kWaitLimit && !bar_try(&sm->bar[kDrain], 0); ++it) {
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax (thread = head row)
        const int h = tid;
        const uint32_t lrow = (uint32_t)(warp * 32) << 16;  // this warp's TMEM lanes
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int i = 0; i < nb; ++i) {
            const int st = i & 1, ph = (i >> 1) & 1;
            if (!warp_wait(sm, &sm->bar[kSFull + st], ph, A.status) ||
                !warp_wait(sm, &sm->bar[kKvFull + st], ph, A.status)) { ok = false; break; }
            fence_after();
            uint32_t r[32];
            HS_LD32(r, tmem + lrow + kColS + 32 * st);
            tmem_wait_ld();
            const uint32_t vm = sm->vmask[st];
            float x[32];
            float mb = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                x[j] = ((vm >> j) & 1u) ? __uint_as_float(r[j]) * A.scale_log2 : -INFINITY;
                mb = fmaxf(mb, x[j]);
            }
            const bool need = mb > m + kRescaleLog2 || (m == -INFINITY && mb > -INFINITY);
            const float m_new = need ? mb : m;
            if (i > 0 && __any_sync(0xffffffffu, need)) {
                // O holds blocks 0..i-1 once their last product is done: rescale it to m_new
                if (!warp_wait(sm, &sm->bar[kPvDone + ((i - 1) & 1)], ((i - 1) >> 1) & 1, A.status)) { ok = false; break; }
                fence_after();
                const float f = need ? ex2(m - m_new) : 1.f;  // m = -inf: O is zero so far
#pragma unroll 1
                for (int c0 = 0; c0 < kHalfV; c0 += 32) {
                    uint32_t o[32];
                    HS_LD32(o, tmem + lrow + kColO + c0);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
                    HS_ST32(tmem + lrow + kColO + c0, o);
                }
                tmem_wait_st();
                l *= f;
            }
            m = m_new;
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const float p0 = x[2 * c] == -INFINITY ? 0.f : ex2(x[2 * c] - m);
                const float p1 = x[2 * c + 1] == -INFINITY ? 0.f : ex2(x[2 * c + 1] - m);
                const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
                const float2 pr = __bfloat1622float2(pb);
                l += pr.x + pr.y;
                pk[c] = *reinterpret_cast<const uint32_t*>(&pb);
            }
            // P[st] was the operand of block i-2's product
            if (i >= 2 && !warp_wait(sm, &sm->bar[kPvDone + st], ((i - 2) >> 1) & 1, A.status)) { ok = false; break; }
            HS_ST16(tmem + lrow + kColP + 16 * st, pk);
            tmem_wait_st();
            fence_before();
            bar_arrive(&sm->bar[kPFull + st]);
        }
        if (ok && nb > 0 && warp_wait(sm, &sm->bar[kOFull], 0, A.status)) {
            fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            size_t orow;
            if (A.nsplit == 1) orow = ((size_t)b * A.H + h) * kDimV;
            else orow = (((size_t)b * A.nsplit + split) * A.H + h) * kDimV;
            float* dst = A.o + orow + kHalfV * v;
#pragma unroll 1
            for (int c0 = 0; c0 < kHalfV; c0 += 32) {
                uint32_t o[32];
                HS_LD32(o, tmem + lrow + kColO + c0);
                tmem_wait_ld();
                if (h < A.H) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4*>(dst + c0 + j) =
                            make_float4(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv,
                                        __uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv);
                }
            }
            if (v == 0 && h < A.H) {
                const float lse = l > 0.f ? (m + lg2(l)) * 0.69314718055994531f : -INFINITY;
                if (A.nsplit == 1) A.lse[(size_t)b * A.H + h] = lse;
                else A.lse[((size_t)b * A.nsplit + split) * A.H + h] = lse;
            }
        } else if (ok && nb == 0 && h < A.H) {  // no keys in this split
            size_t orow = A.nsplit == 1 ? ((size_t)b * A.H + h) * kDimV
                                        : (((size_t)b * A.nsplit + split) * A.H + h) * kDimV;
            for (int d = 0; d < kHalfV; ++d) A.o[orow + kHalfV * v + d] = 0.f;
            if (v == 0) {
                if (A.nsplit == 1) A.lse[(size_t)b * A.H + h] = -INFINITY;
                else A.lse[((size_t)b * A.nsplit + split) * A.H + h] = -INFINITY;
            }
        }
    }
    fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// Merges the key splits of one (request, head): weights exp(lse_s - lse).
__global__ void __launch_bounds__(128) combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                                                      int nsplit, int H, float* __restrict__ o, float* __restrict__ lse) {
    const int bh = blockIdx.x, b = bh / H, h = bh - b * H;
    float mx = -INFINITY;
    for (int s = 0; s < nsplit; ++s) mx = fmaxf(mx, part_lse[((size_t)b * nsplit + s) * H + h]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    if (mx > -INFINITY) {
        for (int s = 0; s < nsplit; ++s) {
            const float ls = part_lse[((size_t)b * nsplit + s) * H + h];
            const float w = ls == -INFINITY ? 0.f : expf(ls - mx);
            L += w;
            const float4 p = reinterpret_cast<const float4*>(part_o + (((size_t)b * nsplit + s) * H + h) * kDimV)[threadIdx.x];
            acc.x += w * p.x;
            acc.y += w * p.y;
            acc.z += w * p.z;
            acc.w += w * p.w;
        }
        const float inv = 1.f / L;
        acc = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
    reinterpret_cast<float4*>(o + ((size_t)b * H + h) * kDimV)[threadIdx.x] = acc;
    if (threadIdx.x == 0) lse[(size_t)b * H + h] = mx > -INFINITY ? mx + logf(L) : -INFINITY;
}

}  // namespace

size_t attend_smem_bytes() { return kSmemBytes; }

AttendPlan attend_plan(int B, int H, int k, int num_sms) {
    AttendPlan p;
    // one CTA per SM: B requests x 2 value halves x nsplit key splits, at least 64 keys each
    int nsplit = num_sms / (2 * B);
    if (nsplit < 1) nsplit = 1;
    const int max_split = (k + 63) / 64;
    if (nsplit > max_split) nsplit = max_split;
    int per = (k + nsplit - 1) / nsplit;
    per = (per + kBlk - 1) / kBlk * kBlk;
    nsplit = (k + per - 1) / per;
    p.nsplit = nsplit;
    p.keys_per_split = per;
    p.workspace_bytes = nsplit > 1 ? (size_t)B * nsplit * H * (kDimV + 1) * sizeof(float) : 0;
    return p;
}

cudaError_t configure_attend() {
    return cudaFuncSetAttribute(attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
}

cudaError_t launch_attend(const Layout& L, cudaStream_t stream, const uint16_t* q, int B, int H,
                          const int32_t* out_slots, int k, float sm_scale, float* o, float* lse,
                          void* workspace, const AttendPlan& plan) {
    AttendArgs a;
    a.dev = L.dev;
    a.S = L.S;
    a.q = q;
    a.H = H;
    a.out_slots = out_slots;
    a.k = k;
    a.nsplit = plan.nsplit;
    a.keys_per_split = plan.keys_per_split;
    a.scale_log2 = sm_scale * 1.4426950408889634f;
    a.status = L.status;
    float* part_o = nullptr;
    float* part_lse = nullptr;
    if (plan.nsplit > 1) {
        part_o = reinterpret_cast<float*>(workspace);
        part_lse = part_o + (size_t)B * plan.nsplit * H * kDimV;
        a.o = part_o;
        a.lse = part_lse;
    } else {
        a.o = o;
        a.lse = lse;
    }
    attend_kernel<<<B * plan.nsplit * 2, kThreads, kSmemBytes, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || plan.nsplit == 1) return e;
    combine_kernel<<<B * H, 128, 0, stream>>>(part_o, part_lse, plan.nsplit, H, o, lse);
    return cudaGetLastError();
}

}  // namespace hs
