// Internal interface between the C ABI (hs_api.cu) and the kernels (hs_kernels.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <climits>

namespace hs {

constexpr int kResolveThreads = 512;               // one CTA per request
constexpr int kResolveWarps = kResolveThreads / 32;
constexpr int kRadixBits = 8;                      // LSD digit width of the victim rank
constexpr int kBins = 1 << kRadixBits;
constexpr int kGroupWords = 8;                     // bitmap words per miss-rank prefix group
constexpr int kGatherThreads = 512;
constexpr int kGatherCtasPerSm = 1;
constexpr int kGatherUnroll = 8;                   // 16-byte loads in flight per thread

constexpr int kMaxSlots = 65535;                   // slot ids are kept as uint16 in shared memory
constexpr int kMaxRequests = 1 << 20;        // requests per context
// A request's two hand-off flags each sit on a 128-byte line of their own (stride in
// words): the fetch CTAs poll them while the resolution CTAs of other requests write
// theirs, and flags sharing a line delayed each other by microseconds.
constexpr int kFlagStride = 32;
// Every device wait gives up once the waiting CTA has run this long (global-timer
// nanoseconds from the CTA's start), records HS_STATUS_TIMEOUT and returns. A healthy
// wait lasts microseconds; the limit only bounds a lost hand-off (hs_set_wait_limit).
constexpr uint64_t kDefaultWaitNs = 20000000ull;   // 20 ms
constexpr uint64_t kMinWaitNs = 1000ull;
constexpr uint64_t kMaxWaitNs = 10000000000ull;    // 10 s

// The global timer (nanoseconds); the clock every bounded wait is measured on.
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Everything the two kernels need about one context.
// Replacement policies (values of HS_POLICY_*).
constexpr int kPolicyLru = 0;     // victims by ascending (last use, slot)
constexpr int kPolicyFifo = 1;    // victims by ascending (fill call, slot); hits keep their stamp
constexpr int kPolicyRandom = 2;  // victims by ascending (SplitMix64 draw, slot)

struct Layout {
    int R, C, S, E;
    size_t host_stride;
    const uint8_t* host;   // device-visible address of the mapped host store
    uint8_t* dev;          // [R][S][E]
    int32_t* pt;           // [R][C]
    int32_t* tok;          // [R][S]
    int32_t* lu;           // [R][S]
    int32_t* step;         // [R]
    uint32_t* status;      // device status word
    // miss area, shared by the two kernels of a call (carve_miss_area):
    int32_t* fpos;         // [R][S]: fetch list -- positions of the missed selections
    int32_t* fsel;         // [R][S]: ... and their indices j in the row (list order is arbitrary)
    uint32_t* ready_pos;   // [R][kFlagStride]: (tag mod 2^16) << 16 | list length, once request b's list is published
    uint32_t* ready_slot;  // [R][kFlagStride]: == tag once request b's answers (out_slots) are written
    uint32_t* gcount;      // [R + G]: fetch CTA counters; (b, share q) at b + q*R; tag = gcount[b] + 1
    const int64_t* row_base = nullptr;  // [R] pooled store: first row of request b (else b * C)
    const int32_t* row_len = nullptr;   // [R] pooled store: positions request b has (else C)
    // [R][k] device copy of the slots given to missed selections, which the fetch reads;
    // null: the fetch reads them from out_slots (which must then be device memory)
    int32_t* jslot = nullptr;
    int policy = kPolicyLru;  // replacement policy of the calls launched with this layout
    uint64_t seed = 0;        // kPolicyRandom's seed
    uint64_t wait_ns = kDefaultWaitNs;  // time limit of every device wait of a CTA
    // fault injection for tests (HS_FLAG_TEST_STALL): the resolution publishes nothing,
    // so a fetch grid waiting on its flags runs out of time
    int no_publish = 0;
};

// Bytes of the miss area for R requests of S slots, and its layout at `base`
// (16-byte aligned). An all-zero area is a valid initial state.
size_t miss_area_bytes(int R, int S, int num_sms);
void carve_miss_area(Layout& L, void* base);

// Dynamic shared memory of one request's resolution for (C, S).
size_t resolve_smem_bytes(int C, int S);

// Opt the kernels in to the device's maximum dynamic shared memory (the current
// device must be `device`); returns a CUDA error.
cudaError_t configure_kernels(int device);

// Enqueue the resolution of requests b0 .. b0 + nr - 1 (one CTA per request). With
// `fetch` (a fetch grid for them is enqueued next) it publishes each request's miss
// positions as soon as they are known and the victim slots once chosen. `wait` = false
// only for a later chunk of a call's requests (see chunk_requests).
cudaError_t launch_resolve(const Layout& L, cudaStream_t stream, const int32_t* sel, int k,
                           int32_t* out_slots, int32_t* miss_counts, bool fetch, int b0, int nr, bool wait);

// Enqueue the row fetch of requests b0 .. b0 + nr - 1 (a persistent grid of
// kGatherCtasPerSm CTAs per SM). With `pdl` it is chained to the preceding resolution by
// programmatic dependent launch and runs concurrently with it, starting on each
// request's rows as soon as they are published; without it, it runs after the
// resolution and reads the hand-off as is.
cudaError_t launch_gather(const Layout& L, cudaStream_t stream, const int32_t* out_slots, int k, int num_sms,
                          bool pdl, int b0, int nr);

// Chunks of a call: with more requests than SMs, the requests are resolved in
// ceil(R / num_sms) chunks of at most num_sms requests, each followed by its fetch grid;
// a chunk's resolution (one CTA per request, two per SM) then leaves room for its fetch
// grid, and the next chunk's resolution runs under the previous chunk's fetch.
inline int chunk_count(int R, int num_sms) { return R <= num_sms ? 1 : (R + num_sms - 1) / num_sms; }
inline void chunk_requests(int R, int nchunks, int i, int* b0, int* nr) {
    *b0 = (int)((long long)R * i / nchunks);
    *nr = (int)((long long)R * (i + 1) / nchunks) - *b0;
}

// Enqueue the consumer stand-in: sums[b] = sum (mod 2^64) of the 8-byte words of the
// k rows request b resolved to (slots < 0 skipped); zeroes sums first.
cudaError_t launch_checksum(const uint8_t* dev, int R, int S, int E, const int32_t* out_slots, int k,
                            unsigned long long* sums, int num_sms, cudaStream_t stream);

// Enqueue the decode-time append of kv[b] (device [R][E]) at positions[b] (device [R]).
cudaError_t launch_append(const Layout& L, cudaStream_t stream, const uint8_t* kv, const int32_t* positions);

// Sparse MLA-style decode attention over resolved slots (hs_attend.cu).
struct AttendPlan {
    int nsplit = 1;              // key splits per request
    int keys_per_split = 0;      // a multiple of the 32-key stage
    size_t workspace_bytes = 0;  // partial outputs when nsplit > 1
};
constexpr int kAttendEntryBytes = 656;
constexpr int kAttendMaxHeads = 128;
size_t attend_smem_bytes();
AttendPlan attend_plan(int B, int H, int k, int num_sms);
cudaError_t configure_attend();
// `stall` (tests only): the producers withhold their first fill, so the MMA thread's
// wait for it runs out of time and the kernel takes its abort path.
cudaError_t launch_attend(const Layout& L, cudaStream_t stream, const uint16_t* q, int B, int H,
                          const int32_t* out_slots, int k, float sm_scale, float* o, float* lse,
                          void* workspace, const AttendPlan& plan, bool stall = false);

// Set the calling thread's message for hs_last_error().
void record_error(const char* msg);

}  // namespace hs
