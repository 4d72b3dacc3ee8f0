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
// attend_kernel: one CTA per (request b, key split s, value half v), 832 threads, one CTA
// per SM (209 KB of shared memory, 512 TMEM columns).
//   * Keys come in blocks of 256 selections, and the stages of a ring of four 48 KB
//     stages are filled in the order the MMAs consume them: per block nine K fills (256
//     keys x 64 dims, K-major; 8 latent chunks, then the rotary one) and four V fills (64
//     keys x this CTA's 256 value dims, read MN-major). A fill gathers its rows through
//     out_slots and decodes the E4M3 codes times their block scale to bf16 (the rotary
//     values are bf16 already and are copied as they are). 16 producer warps make six of
//     the K fills and the V fills; the 8 softmax warps, idle while a block's scores are
//     being multiplied, make the other three K fills of the block (latent chunks 2 and 5
//     and the rotary chunk) before they wait for its scores.
//   * Q [H x 576] bf16 is not kept resident: a K fill's stage also receives the matching
//     64-dimension column of Q (128 rows x 128 bytes) by one tensor-memory-access copy
//     (TMA, 128-byte swizzle, rows beyond H zero-filled) that lands on its own mbarrier;
//     one thread of its own warp issues these copies as soon as each stage is free.
//     Freeing Q's 147 KB of shared memory is what pays for the four-deep ring, so the
//     producers keep filling while the softmax runs.
//   * one thread issues the MMAs: S = Q K^T (M=128 heads, N=256 keys, K=16 per
//     instruction, 36 per block) into 256 TMEM columns, and O += P V (M=128, N=256 value
//     dims, K=16 keys, 16 per block) with P read from TMEM; completion is signalled through
//     mbarriers by tcgen05.commit. The widest N keeps the tensor core busy: an M=128
//     instruction takes ~200 cycles whatever N is (measured from N=32 to 256).
//   * 8 softmax warps in two groups of 128 keys (thread = head = TMEM lane in both) read
//     S, keep a running maximum m (log2 domain) that moves only when a block's maximum
//     exceeds it by more than 8 -- then O (in TMEM) and the running sums are rescaled --
//     and write P = 2^(x - m) as bf16 over the scores already read; at the end they
//     normalise O and write it with lse. Each group signals each half of its keys (64)
//     as soon as their P is written, and the product over those keys starts then, so
//     the P V MMAs run under the rest of the softmax.
// With several key splits per request each CTA writes its normalised partial and its
// lse; combine_kernel merges them (weights exp(lse_s - lse)). It is an ordinary launch:
// as a programmatic dependent started at the attention's beginning, its waiting blocks
// took the SMs the attention leaves free, which another stream's work (the next layer's
// resolution) needs.
//
// Every wait on an mbarrier is bounded in time (global timer, the context's wait limit
// counted from the CTA's start): on expiry the CTA records HS_STATUS_TIMEOUT, every role
// leaves its loop, the MMA thread waits (again bounded in time) for its own MMAs and the
// Q thread for its last copies, and the TMEM columns are freed before the CTA exits.
#include <cuda.h>  // CUtensorMap (the encoder is reached through the runtime's entry point)
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
constexpr int kBlk = 256;      // keys per block: the N of S = Q K^T
constexpr int kChunks = kDimK / 64;                  // 64-element (128-byte) swizzle columns
constexpr uint32_t kQChunk = kHeads * 128;           // bytes of one Q column chunk (16 KB)
constexpr uint32_t kKVBytes = 32768;                 // K chunk: 256 keys x 64 dims; V chunk: 64 keys x 256 dims
constexpr uint32_t kSlotBytes = kQChunk + kKVBytes;  // a stage: the Q chunk, then the K (or V) chunk
constexpr int kStages = 4;
constexpr int kKFills = kChunks;                     // K chunks per block (8 latent + 1 rotary)
constexpr int kVKeys = 64;                           // keys per V chunk
constexpr int kVFills = kBlk / kVKeys;               // V chunks per block
constexpr int kFills = kKFills + kVFills;            // stage fills per block
constexpr uint32_t kVSub = kVKeys * 128;             // bytes of one 64-dimension column of a V chunk
constexpr int kSoftWarps = 8, kProdWarps = 16;  // softmax: two groups of 4 warps, 128 keys each
constexpr int kMmaWarp = kSoftWarps + kProdWarps;  // then one warp for the Q copies
constexpr int kQWarp = kMmaWarp + 1;
constexpr int kThreads = (kQWarp + 1) * 32;  // 832
// The softmax warps, idle while a block's scores are being multiplied, fill three of its
// nine K chunks (latent chunks 2 and 5 and the rotary chunk); the producers fill the
// other six and the four V chunks.
constexpr int kHelp0 = 2, kHelp1 = 5, kHelp2 = 8;  // the softmax warps' K fills of a block, in order
constexpr int kProdFills = kFills - 3;    // the producers': the other six K fills, then V 9..12
__host__ __device__ constexpr int prod_fill(int j) {  // the producers' j-th fill of a block
    return j + (j >= kHelp0) + (j + 1 >= kHelp1) + (j + 2 >= kHelp2);
}
constexpr bool fills_split_once() {  // the two lists cover a block's 13 fills, each once
    int seen = (1 << kHelp0) | (1 << kHelp1) | (1 << kHelp2);
    for (int j = 0; j < kProdFills; ++j) {
        if ((seen >> prod_fill(j)) & 1) return false;
        seen |= 1 << prod_fill(j);
    }
    return seen == (1 << kFills) - 1 && kHelp2 == kKFills - 1;  // the last is the rotary chunk
}
static_assert(fills_split_once(), "fills of a block");
// Every writer's fills are at most 2 kStages apart, the window in which the parity waits on
// the free barriers stay unambiguous (see wait_free).
static_assert(kFills + kHelp0 - kHelp2 <= 2 * kStages && kHelp1 - kHelp0 <= 2 * kStages &&
                  kHelp2 - kHelp1 <= 2 * kStages,
              "the softmax warps' fills must stay within the free barriers' window");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256;  // O: 256 columns; S: 256 columns, P (bf16) written over its first 128
constexpr float kRescaleLog2 = 8.0f;
constexpr int kMaxSplitKeys = 2048;        // slots of one split staged in shared memory

// barrier indices
enum { kFull = 0 /* kStages: a stage's fill is written */, kFree = 4 /* 2 kStages: MMAs done with fill g, by g % 8 */,
       kQLand = 12 /* kStages: a stage's Q chunk has landed */, kSFull = 16, kPvDone = 17,
       kVmFull = 18 /* 2, by block parity */, kDrain = 20, kBmax = 21 /* 2, by block parity */, kLsum = 23,
       kPHalf = 24 /* 4: [softmax group][first or second half of its keys]: P written */, kBars = 28 };
static_assert(kFree == kFull + kStages && kQLand == kFree + 2 * kStages && kSFull == kQLand + kStages, "barrier map");

struct Smem {  // beyond Q and the stages
    int32_t slot[kMaxSplitKeys];  // this split's out_slots
    uint64_t bar[kBars];
    uint32_t vmask[2][kBlk / 32];  // valid keys of a block, by block parity
    float bmax[2][2][kHeads];      // [block parity][softmax group][head]: the groups' block maxima
    float lsum[2][kHeads];         // [softmax group][head]: the groups' running sums, at the end
    uint32_t tmem;
    volatile int abort;
};
constexpr uint32_t kSmemBytes = 1024 + kStages * kSlotBytes + sizeof(Smem);

struct AttendArgs {
    const uint8_t* dev;        // [R][S][656]
    int S;
    int H;
    const int32_t* out_slots;  // [B][k]
    int k;
    int nsplit, keys_per_split;
    float scale_log2;          // sm_scale * log2(e)
    float* o;                  // nsplit == 1: [B][H][512]; else partials [B][nsplit][H][512]
    float* lse;                // nsplit == 1: [B][H];      else partials [B][nsplit][H]
    uint32_t* status;
    uint64_t wait_ns;          // time limit of the CTA's waits (global-timer ns from its start)
    int stall;                 // tests: the producers withhold the first fill
};

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// ---------------------------------------------------------------- mbarriers
__device__ __forceinline__ void bar_init(uint64_t* b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive2(uint64_t* b) {  // counts as two arrivals
    asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0], 2; }" ::"r"(su32(b)) : "memory");
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
// Waits for the phase of `parity` to complete; false (and the CTA aborted) once the
// global timer passes `deadline` or when another role has aborted.
__device__ __forceinline__ bool bar_wait(Smem* sm, uint64_t* b, uint32_t parity, uint32_t* status, uint64_t deadline) {
    while (!bar_try(b, parity)) {
        if (sm->abort) return false;
        if (global_ns() > deadline) {
            sm->abort = 1;
            atomicOr(status, 8u /* HS_STATUS_TIMEOUT */);
            return false;
        }
    }
    return true;
}

// The same wait taken by a whole warp whose next step is warp-collective: all lanes go on
// or none does.
__device__ __forceinline__ bool warp_wait(Smem* sm, uint64_t* b, uint32_t parity, uint32_t* status, uint64_t deadline) {
    return __all_sync(0xffffffffu, bar_wait(sm, b, parity, status, deadline));
}

// Waits (bounded by `deadline` only, whatever the abort flag says) for in-flight
// asynchronous work -- a TMA copy or the CTA's MMAs -- that must land before the CTA
// releases its shared memory or tensor memory.
__device__ __forceinline__ void drain_wait(uint64_t* b, uint32_t parity, uint64_t deadline) {
    while (!bar_try(b, parity) && global_ns() <= deadline) {
    }
}

// The wait of a writer of fill g (of any role): the previous fill of its stage, g - 4, has
// been consumed. The MMA thread signals the consumption of fill g on barrier g % 8 -- two
// barriers per stage, used alternately -- so that a parity wait stays unambiguous for a
// writer whose previous write (or wait) was up to 8 fills earlier: the producers' fills
// are at most 3 apart, the softmax warps' 7 (from a block's rotary chunk to the next
// block's chunk 2), the Q thread's 5. With one barrier per stage, a writer returning after
// two phases of the stage could not tell them apart.
__device__ __forceinline__ bool wait_free(Smem* sm, int g, uint32_t* status, uint64_t deadline) {
    if (g < kStages) return true;
    const int p = g - kStages;
    return bar_wait(sm, &sm->bar[kFree + p % (2 * kStages)], (p / (2 * kStages)) & 1, status, deadline);
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void bar_expect_tx(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
// Box (64 dims, 128 heads, 1 request) of Q at (dim x, head 0, request z) into dst (1024-byte
// aligned), 128-byte swizzled; completion is counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_q(void* dst, const CUtensorMap* map, int x, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(su32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(0), "r"(z), "r"(su32(bar))
        : "memory");
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

// ---------------------------------------------------------------- stage fills
// A CTA's keys: request b's device rows and the split's slots, staged in shared memory.
struct Keys {
    const uint8_t* dev;
    int S, b, kbeg, kend;
    const int32_t* slot;
    __device__ __forceinline__ int32_t at(int j) const {  // key j of the split; -1 when past its end or invalid
        const int32_t s = kbeg + j < kend ? slot[j] : -1;
        return (s >= 0 && s < S) ? s : -1;
    }
    __device__ __forceinline__ const uint8_t* row(int32_t s) const { return dev + ((size_t)b * S + s) * 656; }
};
// The raw bytes one of NT threads decodes into a K chunk (256 keys x 64 dims): groups of
// 16 codes with their block scale. Thread t's keys are (t >> 2) + (NT / 4) w, its codes
// those of dimensions 64 f + 16 (t & 3) ... + 15: the 4 lanes of a key read 64 whole bytes.
template <int NT>
struct RawK {
    static constexpr int kItems = 1024 / NT;
    uint4 c[kItems];
    float scale[kItems];
};
template <int NT>
__device__ __forceinline__ void k_rows(const Keys& K, int t, int i, const uint8_t* (&rows)[1024 / NT]) {
#pragma unroll
    for (int w = 0; w < 1024 / NT; ++w) {
        const int32_t s = K.at(i * kBlk + (t >> 2) + (NT / 4) * w);
        rows[w] = s >= 0 ? K.row(s) : nullptr;  // nullptr: no key, zeros
    }
}
template <int NT>
__device__ __forceinline__ void k_load(const uint8_t* const (&rows)[1024 / NT], int t, int f, RawK<NT>& r) {
    const int off = 64 * f + 16 * (t & 3);
#pragma unroll
    for (int w = 0; w < RawK<NT>::kItems; ++w) {
        if (rows[w]) {
            r.c[w] = __ldg(reinterpret_cast<const uint4*>(rows[w] + off));
            r.scale[w] = __ldg(reinterpret_cast<const float*>(rows[w] + 512) + (off >> 7));
        } else {
            r.c[w] = make_uint4(0, 0, 0, 0);
            r.scale[w] = 0.f;
        }
    }
}
template <int NT>
__device__ __forceinline__ void k_store(uint8_t* stg, int t, const RawK<NT>& r) {
    const int q = t & 3;
#pragma unroll
    for (int w = 0; w < RawK<NT>::kItems; ++w) {
        const int key = (t >> 2) + (NT / 4) * w;
        *reinterpret_cast<uint4*>(stg + swz(key, 2 * q)) = decode8(r.c[w].x, r.c[w].y, r.scale[w]);
        *reinterpret_cast<uint4*>(stg + swz(key, 2 * q + 1)) = decode8(r.c[w].z, r.c[w].w, r.scale[w]);
    }
}
// The rotary chunk of block i (256 keys x 64 bf16, copied as it is) by NT threads with
// asynchronous 16-byte copies, 8 lanes per key; missing keys read as zero. Returns once
// the copies have landed.
template <int NT>
__device__ __forceinline__ void rope_copy(const Keys& K, uint8_t* stg, int t, int i) {
    const int u = t & 7;
#pragma unroll
    for (int w = 0; w < 2048 / NT; ++w) {
        const int key = (t >> 3) + (NT / 8) * w;
        const int32_t s = K.at(i * kBlk + key);
        const uint8_t* src = K.row(s >= 0 ? s : 0) + 528 + 16 * u;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(su32(stg + swz(key, u))), "l"(src),
                     "r"(s >= 0 ? 16u : 0u) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_all;" ::: "memory");
}

__global__ void __launch_bounds__(kThreads, 1) attend_kernel(const AttendArgs A, const __grid_constant__ CUtensorMap qmap) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = base;  // stage st at ring + st * kSlotBytes: Q chunk, then K (or V) chunk
    Smem* sm = reinterpret_cast<Smem*>(base + kStages * kSlotBytes);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int v = blockIdx.x & 1;
    const int split = (blockIdx.x >> 1) % A.nsplit;
    const int b = (blockIdx.x >> 1) / A.nsplit;
    const int kbeg = split * A.keys_per_split;
    const int kend = min(A.k, kbeg + A.keys_per_split);
    const int nb = kend > kbeg ? (kend - kbeg + kBlk - 1) / kBlk : 0;
    const uint64_t deadline = global_ns() + A.wait_ns;  // every wait of this CTA ends by then

    if (tid == 0) {
        for (int st = 0; st < kStages; ++st) {
            bar_init(&sm->bar[kFull + st], kProdWarps * 32);
            bar_init(&sm->bar[kFree + st], 1);
            bar_init(&sm->bar[kFree + kStages + st], 1);
            bar_init(&sm->bar[kQLand + st], 1);
        }
        bar_init(&sm->bar[kVmFull], kBlk / 32);
        bar_init(&sm->bar[kVmFull + 1], kBlk / 32);
        bar_init(&sm->bar[kSFull], 1);
        bar_init(&sm->bar[kPvDone], 1);
        bar_init(&sm->bar[kDrain], 1);
        bar_init(&sm->bar[kBmax], kSoftWarps * 32);
        bar_init(&sm->bar[kBmax + 1], kSoftWarps * 32);
        bar_init(&sm->bar[kLsum], kSoftWarps * 32);
        for (int j = 0; j < 4; ++j) bar_init(&sm->bar[kPHalf + j], kSoftWarps / 2 * 32);
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
        const int pw = warp - kSoftWarps;
        const int ptid = tid - kSoftWarps * 32;  // 0..511
        // the split's slots, staged once for the producers and the softmax warps
        const int32_t* slots = A.out_slots + (size_t)b * A.k;
        for (int j = ptid; j < kend - kbeg; j += kProdWarps * 32) sm->slot[j] = __ldg(slots + kbeg + j);
        asm volatile("bar.sync 1, %0;" ::"r"((kProdWarps + kSoftWarps) * 32) : "memory");
        const Keys K{A.dev, A.S, b, kbeg, kend, sm->slot};
        auto prefetch_block = [&](int i) {  // this warp's 32 rows of the block into L2
            if (i >= nb || ptid >= kBlk) return;
            const int32_t s = K.at(i * kBlk + ptid);
            if (s >= 0) asm volatile("cp.async.bulk.prefetch.L2.global [%0], 656;" ::"l"(K.row(s)) : "memory");
        };
        prefetch_block(0);
        // The producers' fills, in the order the MMAs consume them: per block six of the
        // K chunks (the softmax warps fill the other three) and the 4 V chunks. Loads are
        // spread so that the lanes of a warp read a few whole stretches of a row each (4
        // lanes x 16 bytes per key for a K chunk, 16 lanes for a V chunk): a warp-wide
        // load then touches 8 (or 2) rows rather than 32. The raw bytes of fill j + 2 are
        // requested before fill j is decoded; three register buffers rotate by unrolling,
        // so two fills' loads are always in flight.
        const int total = nb * kProdFills;
        const int vu = ptid & 15, vkey = ptid >> 4;  // V chunk: 16-dim unit of the half, key (+32 w)
        // This thread's K rows are the same for the latent fills of a block: they are
        // looked up once per block (a shared-memory read before every load would queue
        // behind the stage stores and delay the loads' issue).
        const uint8_t* krow[RawK<kProdWarps * 32>::kItems];
        int kblock = -1;
        auto issue = [&](int j, RawK<kProdWarps * 32>& r) {
            if (j >= total) return;
            const int i = j / kProdFills, f = prod_fill(j - i * kProdFills);
            if (f < kKFills) {
                if (i != kblock) {
                    k_rows<kProdWarps * 32>(K, ptid, i, krow);
                    kblock = i;
                }
                k_load<kProdWarps * 32>(krow, ptid, f, r);
                return;
            }
#pragma unroll
            for (int w = 0; w < RawK<kProdWarps * 32>::kItems; ++w) {
                const int32_t s = K.at(i * kBlk + (f - kKFills) * kVKeys + vkey + 32 * w);
                const int off = kHalfV * v + 16 * vu;
                if (s >= 0) {
                    const uint8_t* row = K.row(s);
                    r.c[w] = __ldg(reinterpret_cast<const uint4*>(row + off));
                    r.scale[w] = __ldg(reinterpret_cast<const float*>(row + 512) + (off >> 7));
                } else {
                    r.c[w] = make_uint4(0, 0, 0, 0);
                    r.scale[w] = 0.f;
                }
            }
        };
        auto process = [&](int j, const RawK<kProdWarps * 32>& r) -> bool {
            const int i = j / kProdFills, jj = j - i * kProdFills, f = prod_fill(jj);
            const int g = i * kFills + f;
            if (jj == 0 && pw < kBlk / 32) {  // a new block: its valid keys (32 per warp)
                const uint32_t m = __ballot_sync(0xffffffffu, K.at(i * kBlk + ptid) >= 0);
                if (lane == 0) {
                    sm->vmask[i & 1][pw] = m;
                    bar_arrive(&sm->bar[kVmFull + (i & 1)]);
                }
            }
            if (pw < kBlk / 32 && jj == pw) prefetch_block(i + 1);  // the next block's rows into L2
            const int st = g % kStages;
            if (!wait_free(sm, g, A.status, deadline)) return false;
            uint8_t* stg = ring + st * kSlotBytes + kQChunk;
            if (f < kKFills) {
                k_store<kProdWarps * 32>(stg, ptid, r);
            } else {
                uint8_t* col = stg + (vu >> 2) * kVSub;  // the 64-dim column of this unit
#pragma unroll
                for (int w = 0; w < RawK<kProdWarps * 32>::kItems; ++w) {
                    const int key = vkey + 32 * w;
                    *reinterpret_cast<uint4*>(col + swz(key, 2 * (vu & 3))) = decode8(r.c[w].x, r.c[w].y, r.scale[w]);
                    *reinterpret_cast<uint4*>(col + swz(key, 2 * (vu & 3) + 1)) = decode8(r.c[w].z, r.c[w].w, r.scale[w]);
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            if (!(A.stall && g == 0)) bar_arrive(&sm->bar[kFull + st]);
            return true;
        };
        RawK<kProdWarps * 32> r0, r1, r2;
        issue(0, r0);
        issue(1, r1);
        for (int j = 0; j < total; j += 3) {
            issue(j + 2, r2);
            if (!process(j, r0) || j + 1 >= total) break;
            issue(j + 3, r0);
            if (!process(j + 1, r1) || j + 2 >= total) break;
            issue(j + 4, r1);
            if (!process(j + 2, r2)) break;
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issue (one thread)
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16(kHeads, kBlk, 0);
            const uint32_t id_o = idesc_bf16(kHeads, kHalfV, 1);
            const uint32_t s0 = su32(ring);
            bool ok = true;
            uint32_t g = 0, qpar = 0;  // qpar: per stage, phase parity of the next Q copy to wait for
            for (int i = 0; ok && i < nb; ++i) {
                // S and P share columns: block i's scores wait until block i-1's product is done
                if (i > 0 && !bar_wait(sm, &sm->bar[kPvDone], (i - 1) & 1, A.status, deadline)) { ok = false; break; }
                for (int c = 0; c < kKFills; ++c, ++g) {
                    const int st = g % kStages;
                    if (!bar_wait(sm, &sm->bar[kFull + st], (g / kStages) & 1, A.status, deadline) ||
                        !bar_wait(sm, &sm->bar[kQLand + st], (qpar >> st) & 1u, A.status, deadline)) { ok = false; break; }
                    qpar ^= 1u << st;
                    fence_after();
                    const uint32_t qa = s0 + st * kSlotBytes, kb = qa + kQChunk;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_ss(tmem + kColS, smem_desc(qa + kk * 32, 16, 1024), smem_desc(kb + kk * 32, 16, 1024),
                               id_s, (c | kk) ? 1u : 0u);
                    mma_commit(&sm->bar[kFree + g % (2 * kStages)]);
                }
                if (!ok) break;
                mma_commit(&sm->bar[kSFull]);
                // P V in the order the softmax writes its halves: keys 0-63 and 128-191 (the
                // first half of each group's keys), then 64-127 and 192-255
                for (int j = 0; j < kVFills; ++j) {
                    const int vc = (j >> 1) | ((j & 1) << 1);  // 0, 2, 1, 3
                    if (!bar_wait(sm, &sm->bar[kPHalf + (vc >> 1) * 2 + (vc & 1)], i & 1, A.status, deadline)) { ok = false; break; }
                    const uint32_t gv = g + (uint32_t)vc;
                    const int st = gv % kStages;
                    if (!bar_wait(sm, &sm->bar[kFull + st], (gv / kStages) & 1, A.status, deadline)) { ok = false; break; }
                    fence_after();
                    const uint32_t vb = s0 + st * kSlotBytes + kQChunk;
#pragma unroll
                    for (int ks = 0; ks < kVKeys / 16; ++ks)
                        mma_ts(tmem + kColO, tmem + kColS + (kVKeys / 2) * vc + 8 * ks + (vc >= kVFills / 2 ? 64 : 0),
                               smem_desc(vb + ks * 2048, kVSub, 1024), id_o, (i > 0 || j > 0 || ks > 0) ? 1u : 0u);
                    mma_commit(&sm->bar[kFree + gv % (2 * kStages)]);
                }
                g += kVFills;
                if (!ok) break;
                mma_commit(&sm->bar[kPvDone]);
            }
            // whatever happened, every MMA issued here completes before the columns are freed
            mma_commit(&sm->bar[kDrain]);
            drain_wait(&sm->bar[kDrain], 0, global_ns() + A.wait_ns);
        }
        __syncwarp();
    } else if (warp == kQWarp) {
        // ------------------------------------------------------------ Q copies (one thread)
        // Each K fill's stage also receives the matching 64-dimension column of Q, by one TMA
        // copy issued as soon as the stage is free.
        if (lane == 0) {
            uint32_t qpar = 0, qout = 0;  // per stage: phase parity of its next Q copy; copies issued
            const int total = nb * kFills;
            for (int g = 0; g < total; ++g) {
                const int f = g % kFills, st = g % kStages;
                if (f >= kKFills) continue;
                if (!wait_free(sm, g, A.status, deadline)) break;
                bar_expect_tx(&sm->bar[kQLand + st], kQChunk);
                tma_load_q(ring + st * kSlotBytes, &qmap, 64 * f, b, &sm->bar[kQLand + st]);
                qpar ^= 1u << st;
                qout |= 1u << st;
            }
            // No Q copy may still be landing when the CTA exits (after an abort the MMA thread
            // may not have waited for the last ones): wait, bounded, for the last copy issued
            // into each stage.
            const uint64_t drain_by = global_ns() + A.wait_ns;
            for (int st = 0; st < kStages; ++st)
                if ((qout >> st) & 1u) drain_wait(&sm->bar[kQLand + st], ((qpar >> st) & 1u) ^ 1u, drain_by);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        // Two groups of 4 warps; thread = head row (its TMEM lane) in both. Group g reads the
        // scores of keys [128 g, 128 g + 128) and writes their P over its own first 64
        // columns of them (keys 0..127 -> columns 0..63, keys 128..255 -> 128..191), so
        // neither group overwrites scores the other has yet to read. The groups share the
        // block maximum through shared memory and keep partial running sums.
        const int grp = warp >> 2;
        const int h = tid & (kHeads - 1);
        const uint32_t lrow = (uint32_t)((warp & 3) * 32) << 16;  // this warp's TMEM lanes
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        asm volatile("bar.sync 1, %0;" ::"r"((kProdWarps + kSoftWarps) * 32) : "memory");  // slots staged
        const Keys K{A.dev, A.S, b, kbeg, kend, sm->slot};
        // Fill g's stage, once free (nullptr once the CTA has aborted); the caller stores into
        // it and calls close_fill.
        auto open_fill = [&](int g) -> uint8_t* {
            const int st = g % kStages;
            if (!__all_sync(0xffffffffu, wait_free(sm, g, A.status, deadline))) return nullptr;
            return ring + st * kSlotBytes + kQChunk;
        };
        auto close_fill = [&](int g) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            bar_arrive2(&sm->bar[kFull + g % kStages]);  // 256 threads stand for the producers' 512
        };
        for (int i = 0; i < nb; ++i) {
            {  // while the producers fill the rest of the block: its K chunks 2 and 5 and the rotary one
                constexpr int NT = kSoftWarps * 32;
                const uint8_t* hrow[RawK<NT>::kItems];
                k_rows<NT>(K, tid, i, hrow);
                RawK<NT> h0, h1;
                k_load<NT>(hrow, tid, kHelp0, h0);
                k_load<NT>(hrow, tid, kHelp1, h1);
                const int g0 = i * kFills;
                uint8_t* stg = open_fill(g0 + kHelp0);
                if (!stg) { ok = false; break; }
                k_store<NT>(stg, tid, h0);
                close_fill(g0 + kHelp0);
                if (!(stg = open_fill(g0 + kHelp1))) { ok = false; break; }
                k_store<NT>(stg, tid, h1);
                close_fill(g0 + kHelp1);
                if (!(stg = open_fill(g0 + kKFills - 1))) { ok = false; break; }
                rope_copy<NT>(K, stg, tid, i);
                close_fill(g0 + kKFills - 1);
            }
            if (!warp_wait(sm, &sm->bar[kSFull], i & 1, A.status, deadline) ||
                !warp_wait(sm, &sm->bar[kVmFull + (i & 1)], (i >> 1) & 1, A.status, deadline)) { ok = false; break; }
            fence_after();
            // pass 1: this group's part of the block maximum, then the block's
            float mb = -INFINITY;
#pragma unroll 1
            for (int ch = 4 * grp; ch < 4 * grp + 4; ++ch) {
                uint32_t r[32];
                HS_LD32(r, tmem + lrow + kColS + 32 * ch);
                tmem_wait_ld();
                const uint32_t vm = sm->vmask[i & 1][ch];
                if (vm == 0xffffffffu && A.scale_log2 > 0.f) {
                    // every key valid: the largest score, scaled once (a positive scale keeps
                    // the order of the rounded products, so the result is the same)
#pragma unroll
                    for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
                        for (int j = 0; j < w; ++j) r[j] = __float_as_uint(fmaxf(__uint_as_float(r[j]), __uint_as_float(r[j + w])));
                    mb = fmaxf(mb, __uint_as_float(r[0]) * A.scale_log2);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if ((vm >> j) & 1u) mb = fmaxf(mb, __uint_as_float(r[j]) * A.scale_log2);
                }
            }
            sm->bmax[i & 1][grp][h] = mb;
            bar_arrive(&sm->bar[kBmax + (i & 1)]);
            if (!warp_wait(sm, &sm->bar[kBmax + (i & 1)], (i >> 1) & 1, A.status, deadline)) { ok = false; break; }
            mb = fmaxf(sm->bmax[i & 1][0][h], sm->bmax[i & 1][1][h]);
            const bool need = mb > m + kRescaleLog2 || (m == -INFINITY && mb > -INFINITY);
            const float m_new = need ? mb : m;
            if (i > 0 && __any_sync(0xffffffffu, need)) {
                // O holds blocks 0..i-1 (their product is done: the scores of block i
                // were computed after it): each group rescales half of its columns to m_new
                if (!warp_wait(sm, &sm->bar[kPvDone], (i - 1) & 1, A.status, deadline)) { ok = false; break; }
                fence_after();
                const float f = need ? ex2(m - m_new) : 1.f;  // m = -inf: O is zero so far
#pragma unroll 1
                for (int c0 = (kHalfV / 2) * grp; c0 < (kHalfV / 2) * (grp + 1); c0 += 32) {
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
            // pass 2: P = 2^(x - m) in bf16, written over this group's scores already read
#pragma unroll 1
            for (int ch = 4 * grp; ch < 4 * grp + 4; ++ch) {
                uint32_t r[32];
                HS_LD32(r, tmem + lrow + kColS + 32 * ch);
                tmem_wait_ld();
                const uint32_t vm = sm->vmask[i & 1][ch];
                uint32_t pk[16];
                if (vm == 0xffffffffu) {  // every key valid
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float p0 = ex2(__uint_as_float(r[2 * c]) * A.scale_log2 - m);
                        const float p1 = ex2(__uint_as_float(r[2 * c + 1]) * A.scale_log2 - m);
                        const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
                        const float2 pr = __bfloat1622float2(pb);
                        l += pr.x + pr.y;
                        pk[c] = *reinterpret_cast<const uint32_t*>(&pb);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float p0 = ((vm >> (2 * c)) & 1u) ? ex2(__uint_as_float(r[2 * c]) * A.scale_log2 - m) : 0.f;
                        const float p1 = ((vm >> (2 * c + 1)) & 1u) ? ex2(__uint_as_float(r[2 * c + 1]) * A.scale_log2 - m) : 0.f;
                        const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
                        const float2 pr = __bfloat1622float2(pb);
                        l += pr.x + pr.y;
                        pk[c] = *reinterpret_cast<const uint32_t*>(&pb);
                    }
                }
                HS_ST16(tmem + lrow + kColS + 16 * ch + 64 * grp, pk);
                if (ch & 1) {  // 64 keys written: their part of P V may start
                    tmem_wait_st();
                    fence_before();
                    bar_arrive(&sm->bar[kPHalf + 2 * grp + ((ch >> 1) & 1)]);
                }
            }
        }
        // the running sum is the two groups' parts
        sm->lsum[grp][h] = l;
        bar_arrive(&sm->bar[kLsum]);
        if (ok && !warp_wait(sm, &sm->bar[kLsum], 0, A.status, deadline)) ok = false;
        l = sm->lsum[0][h] + sm->lsum[1][h];
        if (ok && nb > 0 && warp_wait(sm, &sm->bar[kPvDone], (nb - 1) & 1, A.status, deadline)) {
            fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            size_t orow;
            if (A.nsplit == 1) orow = ((size_t)b * A.H + h) * kDimV;
            else orow = (((size_t)b * A.nsplit + split) * A.H + h) * kDimV;
            float* dst = A.o + orow + kHalfV * v;
#pragma unroll 1
            for (int c0 = (kHalfV / 2) * grp; c0 < (kHalfV / 2) * (grp + 1); c0 += 32) {
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
            if (v == 0 && grp == 0 && h < A.H) {
                const float lse = l > 0.f ? (m + lg2(l)) * 0.69314718055994531f : -INFINITY;
                if (A.nsplit == 1) A.lse[(size_t)b * A.H + h] = lse;
                else A.lse[((size_t)b * A.nsplit + split) * A.H + h] = lse;
            }
        } else if (ok && nb == 0 && h < A.H) {  // no keys in this split
            size_t orow = A.nsplit == 1 ? ((size_t)b * A.H + h) * kDimV
                                        : (((size_t)b * A.nsplit + split) * A.H + h) * kDimV;
            for (int d = (kHalfV / 2) * grp; d < (kHalfV / 2) * (grp + 1); ++d) A.o[orow + kHalfV * v + d] = 0.f;
            if (v == 0 && grp == 0) {
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

// The driver's tensor-map encoder, looked up once through the runtime (no link against
// the driver library).
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiled encoder() {
    static const EncodeTiled fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult found;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &found) !=
                cudaSuccess ||
            found != cudaDriverEntryPointSuccess) {
            (void)cudaGetLastError();
            return (EncodeTiled) nullptr;
        }
        return reinterpret_cast<EncodeTiled>(f);
    }();
    return fn;
}

// Q [B][H][576] bf16 as a 3-D tensor (dims, heads, requests); one box is a 64-dimension
// column of all 128 head rows of one request (rows >= H read as zero), 128-byte swizzled
// as the MMA's K-major operand.
cudaError_t encode_q_map(CUtensorMap* map, const uint16_t* q, int B, int H) {
    const EncodeTiled enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)kDimK, (cuuint64_t)H, (cuuint64_t)B};
    const cuuint64_t strides[2] = {(cuuint64_t)kDimK * 2, (cuuint64_t)H * kDimK * 2};  // bytes, dims 1 and 2
    const cuuint32_t box[3] = {64, (cuuint32_t)kHeads, 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(q), dims, strides, box,
                           estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

size_t attend_smem_bytes() { return kSmemBytes; }

AttendPlan attend_plan(int B, int H, int k, int num_sms) {
    AttendPlan p;
    // one CTA per SM: B requests x 2 value halves x nsplit key splits, at least one
    // 256-key block each and at most the slots one CTA stages
    int nsplit = num_sms / (2 * B);
    if (nsplit < 1) nsplit = 1;
    const int max_split = (k + kBlk - 1) / kBlk;
    if (nsplit > max_split) nsplit = max_split;
    const int min_split = (k + kMaxSplitKeys - 1) / kMaxSplitKeys;
    if (nsplit < min_split) nsplit = min_split;
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
                          void* workspace, const AttendPlan& plan, bool stall) {
    CUtensorMap qmap;
    cudaError_t e = encode_q_map(&qmap, q, B, H);
    if (e != cudaSuccess) return e;
    AttendArgs a;
    a.dev = L.dev;
    a.S = L.S;
    a.H = H;
    a.out_slots = out_slots;
    a.k = k;
    a.nsplit = plan.nsplit;
    a.keys_per_split = plan.keys_per_split;
    a.scale_log2 = sm_scale * 1.4426950408889634f;
    a.status = L.status;
    a.wait_ns = L.wait_ns;
    a.stall = stall ? 1 : 0;
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
    attend_kernel<<<B * plan.nsplit * 2, kThreads, kSmemBytes, stream>>>(a, qmap);
    e = cudaGetLastError();
    if (e != cudaSuccess || plan.nsplit == 1) return e;
    combine_kernel<<<B * H, 128, 0, stream>>>(part_o, part_lse, plan.nsplit, H, o, lse);
    return cudaGetLastError();
}

}  // namespace hs
