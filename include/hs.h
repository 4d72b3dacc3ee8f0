/*
 * hs.h -- C ABI of a GB300-native (sm_103a) HiSparse swap-in resolution library.
 *
 * HiSparse (paper abstract, "HiSparse: Turbocharging Sparse Attention with
 * Hierarchical Memory") keeps each request's full KV history in host memory and
 * bounds its decode footprint with a small, fixed-size GPU cache; a fused CUDA kernel
 * resolves each layer's top-k selections -- hit detection, LRU replacement and
 * host-to-device fetches -- inside the decode CUDA graph. The blog commentary
 * (sections two and three) adds that the same step updates the page table and that a
 * hit is used in place while a miss is swapped in over an LRU-chosen victim.
 *
 * One hs_ctx is one layer's cache for num_requests requests. It owns:
 *   host KV store   pinned + mapped host memory, [R][C] rows of hs_host_stride() bytes
 *                   (the first entry_bytes of each row are the entry);
 *   device buffer   HBM, [R][S] rows of entry_bytes bytes;
 *   page table      int32 [R][C] in HBM: position -> slot, -1 when not resident;
 *   slot tokens     int32 [R][S]: slot -> position, -1 when empty;
 *   last use        int32 [R][S]: per-slot recency stamp, -1 when never used;
 *   step            int32 [R]: calls made so far per request (the stamp of the next call);
 *   a miss area (miss lists and the flags that let the two kernels of a call
 *   overlap) and a device status word (internal).
 * R = num_requests, C = context_len, S = slots. Everything starts empty: page
 * table, slot tokens and last use at -1, step 0, device buffer zero.
 *
 * Replacement rule (the pages leave the order open; this is the deterministic
 * reading implemented, HS_POLICY_LRU, the default; hs_set_policy selects the FIFO and
 * random comparison policies): in a call with stamp t, slots hit by the selection are
 * stamped t and are not evictable; the distinct missed positions, in ascending
 * order, take in order the non-hit slots with the smallest (last_use, slot index);
 * the position a victim held is unmapped, the new one mapped and stamped t, and its
 * host row copied into the slot. A negative selection is padding (slot -1, neither
 * hit nor miss); a selection >= C (in a pooled context, >= the request's extent
 * length) yields slot -1 and sets HS_STATUS_RANGE; a position
 * repeated within one row resolves to the same slot each time, counts once, and sets
 * HS_STATUS_DUP.
 *
 * Error convention: functions returning int return HS_OK (0) or a negative HS_ERR_*;
 * hs_last_error() then describes the failure (per calling thread). Device-side input
 * problems never trap: they set bits of the status word (hs_get_status).
 * Threading: calls on one hs_ctx must not overlap on the GPU (state is per context);
 * different contexts are independent.
 */
#ifndef HS_H_
#define HS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct hs_ctx hs_ctx;
/* A CUDA stream (cudaStream_t); NULL is the legacy default stream. */
typedef struct CUstream_st* hs_stream_t;
/* A CUDA event (cudaEvent_t). */
typedef struct CUevent_st* hs_event_t;

#define HS_OK 0
#define HS_ERR_INVALID (-1) /* bad argument; nothing was enqueued */
#define HS_ERR_CUDA (-2)    /* a CUDA runtime call failed */
#define HS_ERR_NOMEM (-3)   /* host or device allocation failed */
#define HS_ERR_LIMIT (-4)   /* sizes beyond what this build supports */

/* device status bits (hs_get_status) */
#define HS_STATUS_RANGE 1u    /* a selection was >= context_len */
#define HS_STATUS_DUP 2u      /* a position appeared twice in one request's row */
#define HS_STATUS_STEP_LIMIT 4u /* a request reached 2^31-1 calls; the call was skipped */
#define HS_STATUS_TIMEOUT 8u    /* a device wait ran past the wait limit and gave up (see
                                   hs_set_wait_limit); the call's rows may be missing: hs_reset */

/* flags (hs_set_flags) */
#define HS_FLAG_NO_COPY 1u /* do all bookkeeping but skip the host->device row fetch */
/* Fault injection for tests, never for production: with it, hs_resolve's resolution
 * publishes nothing, so its overlapped fetch grid (contexts with num_requests <= the
 * SM count) waits for flags that are never raised, and hs_attend's producers withhold
 * their first fill, so its MMA issuer waits for a barrier that never completes. Every
 * such wait runs out after the wait limit: the kernels set HS_STATUS_TIMEOUT and
 * return, the context stays usable, and its cache contents are undefined until
 * hs_reset. A fetch that would not wait is not launched at all under this flag. */
#define HS_FLAG_TEST_STALL 2u

/*
 * hs_create -- one layer's cache for num_requests requests (paper abstract: full KV
 * history per request in host memory, a small fixed-size GPU cache per request).
 *   num_requests  R > 0 requests
 *   context_len   C > 0 positions of history per request (tokens, or pages)
 *   slots         S > 0 device slots per request (the GPU cache size)
 *   entry_bytes   E > 0 bytes per KV entry; a multiple of 16
 * Uses the calling thread's current CUDA device. Allocates everything up front
 * (R*C*E bytes of pinned host memory, R*S*E bytes of HBM, 4*R*(C+7S) + 268*R bytes of
 * tables, miss lists, flags and staging); hs_resolve allocates nothing. Returns NULL on failure (HS_ERR_INVALID,
 * HS_ERR_LIMIT, HS_ERR_NOMEM or HS_ERR_CUDA described by hs_last_error()). The caller
 * owns the handle and releases it with hs_destroy.
 */
hs_ctx* hs_create(int num_requests, int context_len, int slots, int entry_bytes);

/*
 * hs_create_with_host -- hs_create over a host store the caller owns and lends: the
 * caller keeps it alive (and does not free it) until hs_destroy returns. The store is
 * [R][C] rows host_stride bytes apart (a multiple of 16, >= entry_bytes), 16-byte
 * aligned, and must be pinned and mapped (cudaHostAlloc with cudaHostAllocMapped, or
 * cudaHostRegister with cudaHostRegisterMapped). Several contexts may share one store
 * (for example the layers of one model, or a pool sized by the deployment's
 * host-to-device ratio); the library only reads it. Same errors as hs_create.
 */
hs_ctx* hs_create_with_host(int num_requests, int context_len, int slots, int entry_bytes,
                            uint8_t* host_kv, size_t host_stride);

/*
 * hs_resolve -- the fused per-layer swap-in resolution (paper abstract: hit
 * detection, LRU replacement and host-to-device fetches for each layer's selections;
 * blog commentary section three: the same step updates the page table).
 *   stream        stream to enqueue on; the call is enqueue-only (no host sync, no
 *                 allocation), has a fixed launch shape and can be captured in a
 *                 CUDA graph; replays advance the per-request step counters
 *   selections    device int32 [B][k], row-major: request b's selected positions
 *   B             must equal num_requests
 *   k             0 < k <= slots
 *   out_slots     device int32 [B][k]: out_slots[b][j] is the slot now holding
 *                 selections[b][j] (-1 for padding or out-of-range); the entry's
 *                 bytes are at hs_device_kv() + ((size_t)b * S + slot) * E
 *   miss_counts   device int32 [B]: distinct missed positions of request b
 * The caller owns selections/out_slots/miss_counts and keeps them alive until the
 * enqueued work completes. The call's first kernel is a programmatic dependent of the
 * kernel before it on the stream and reads `selections` before waiting for that kernel:
 * a kernel that writes the selections and uses programmatic dependent launch itself
 * must signal completion to its dependents only after writing them (kernels that do not
 * use it have finished before this call starts). Returns HS_OK, HS_ERR_INVALID (nothing
 * enqueued) or HS_ERR_CUDA (a launch failed).
 */
int hs_resolve(hs_ctx* ctx, hs_stream_t stream, const int32_t* selections, int B, int k,
               int32_t* out_slots, int32_t* miss_counts);

/*
 * hs_resolve_host -- hs_resolve with HOST buffers; returns after the results are in
 * them (it waits for the stream). A page-locked buffer (cudaHostAlloc, cudaMallocHost,
 * or cudaHostRegister'ed and mapped; 4-byte aligned) is read or written by the kernels
 * in place over the host link, with no copy; any other host buffer (pageable memory) is
 * staged through device buffers preallocated by hs_create, with one copy each way. The
 * three buffers are classified independently. Same arguments and errors as hs_resolve.
 */
int hs_resolve_host(hs_ctx* ctx, hs_stream_t stream, const int32_t* selections_host, int B, int k,
                    int32_t* out_slots_host, int32_t* miss_counts_host);

/*
 * hs_resolve_profiled -- hs_resolve that records ev[0] before the resolution kernel,
 * ev[1] between it and the fetch kernel and ev[2] after the fetch (per-kernel timing
 * with events on the launching stream). The two kernels then run one after the other
 * instead of overlapping. ev entries must be valid events created on the context's
 * device. Results are identical to hs_resolve.
 */
int hs_resolve_profiled(hs_ctx* ctx, hs_stream_t stream, const int32_t* selections, int B, int k,
                        int32_t* out_slots, int32_t* miss_counts, hs_event_t ev[3]);

/*
 * hs_append -- decode-time append of new KV entries (blog commentary, opening: the KV
 * that does not need to stay on the GPU is offloaded to host memory; paper abstract:
 * each request's full KV history lives in host memory). Enqueues on `stream` a kernel
 * that writes kv[b] (device, [B][entry_bytes], 16-byte aligned) into the host store at
 * position positions[b] of request b (device int32 [B]; negative = no new entry for
 * that request) -- the writes cross the host link from the GPU -- and, when that
 * position is resident in a slot (a rewrite), into the slot as well, so the cache stays
 * exact. The replacement state does not change: to make a new entry resident, select it
 * in the next hs_resolve (or resolve it on its own). A position >= context_len sets
 * HS_STATUS_RANGE and is skipped. B must equal num_requests (at most 65535). Stream
 * ordered with hs_resolve on the same context. Returns HS_OK, HS_ERR_INVALID,
 * HS_ERR_LIMIT or HS_ERR_CUDA.
 */
int hs_append(hs_ctx* ctx, hs_stream_t stream, const uint8_t* kv, const int32_t* positions, int B);

/*
 * hs_attend -- the layer's consumer: sparse attention of every request over the slots
 * its selections resolved to (blog commentary, section two: a resident entry takes part
 * in the computation directly; paper abstract: only placement changes, so outputs are
 * unchanged). For the 656-byte entries of the DeepSeek sparse-attention family (the
 * context's entry_bytes must be 656): bytes [0,512) are E4M3 codes of the latent vector,
 * [512,528) four fp32 scales (scale g for codes 128g..128g+127), [528,656) 64 bf16 rotary
 * values. Key K_j = (latent_j * scale, rope_j) in R^576, value V_j = latent_j * scale in
 * R^512; for head h and the selections j with out_slots[b][j] >= 0:
 *   s_hj = sm_scale * <q_h, K_j>,  o[b][h] = sum_j softmax_j(s_h) V_j,  lse[b][h] = ln sum_j exp(s_hj).
 * A head with no valid selection gets o = 0 and lse = -inf.
 *   q          device bf16 [B][H][576], 16-byte aligned
 *   out_slots  device int32 [B][k] as written by hs_resolve (negative = not valid)
 *   o, lse     device fp32 [B][H][512] (16-byte aligned) and [B][H], overwritten
 *   workspace  device scratch of hs_attend_workspace() bytes (may be NULL when that is 0)
 * The latent codes are decoded to bf16 (code * scale rounded to nearest even), the
 * products run on the tensor cores with fp32 accumulation, and the softmax weights are
 * rounded to bf16 before the value product. B must equal num_requests, 1 <= H <= 128,
 * k >= 1. Enqueue-only: no allocation, no host synchronisation, graph-capturable. A
 * stalled pipeline sets HS_STATUS_TIMEOUT. Returns HS_OK, HS_ERR_INVALID or HS_ERR_CUDA.
 */
int hs_attend(hs_ctx* ctx, hs_stream_t stream, const void* q, int B, int H, const int32_t* out_slots, int k,
              float sm_scale, float* o, float* lse, void* workspace, size_t workspace_bytes);

/* hs_attend_workspace -- *bytes = the workspace hs_attend needs for (B, H, k) on this
 * context's device (0 when a request's keys fit one pass). Returns HS_OK or HS_ERR_INVALID. */
int hs_attend_workspace(hs_ctx* ctx, int B, int H, int k, size_t* bytes);

/*
 * hs_checksum_rows -- a stand-in for the sparse-attention consumer of a layer (blog
 * commentary, section two: a resident entry takes part in the computation directly).
 * Enqueues on `stream` a kernel that reads the k rows each request resolved to, through
 * out_slots (device int32 [B][k] from hs_resolve; negative slots are skipped), and
 * writes sums[b] = the sum modulo 2^64 of their 8-byte little-endian words (device
 * uint64 [B], overwritten). Used to measure the overlap of layer l+1's resolution with
 * layer l's consumer (paper abstract: exact layer-wise prefetching) and to check the
 * consumer's view against the host rows. B must equal num_requests (at most 65535),
 * 0 < k <= slots. Returns HS_OK, HS_ERR_INVALID, HS_ERR_LIMIT or HS_ERR_CUDA.
 */
int hs_checksum_rows(hs_ctx* ctx, hs_stream_t stream, const int32_t* out_slots, int B, int k,
                     uint64_t* sums);

/* hs_destroy -- synchronizes the device and frees everything; NULL is a no-op. */
void hs_destroy(hs_ctx* ctx);

/*
 * hs_reset -- enqueue a reset of all state to empty on `stream` (page table, slot
 * tokens and last use to -1, steps to 0, device buffer to zero, status cleared). The
 * host KV store is left as it is.
 */
int hs_reset(hs_ctx* ctx, hs_stream_t stream);

/* Host KV store: host pointer (also valid on the device through unified addressing)
 * to [R][C] rows of hs_host_stride() bytes. The caller writes the history here before
 * resolving; the library only reads it. */
uint8_t* hs_host_kv(hs_ctx* ctx);
size_t hs_host_stride(hs_ctx* ctx);

/* Device pointers to the state, for consumers and tests (layouts above). The device
 * buffer is read by the sparse-attention consumer; the tables should be treated as
 * read-only by callers. */
uint8_t* hs_device_kv(hs_ctx* ctx);
int32_t* hs_page_table(hs_ctx* ctx);
int32_t* hs_slot_token(hs_ctx* ctx);
int32_t* hs_last_use(hs_ctx* ctx);
int32_t* hs_step(hs_ctx* ctx);

/* hs_get_status -- synchronizes the device, then stores the OR of HS_STATUS_* bits
 * raised since the last hs_clear_status / hs_reset into *bits. */
int hs_get_status(hs_ctx* ctx, uint32_t* bits);
int hs_clear_status(hs_ctx* ctx);

/* hs_set_flags -- HS_FLAG_* bits for later calls (0 restores the default). */
int hs_set_flags(hs_ctx* ctx, unsigned flags);

/*
 * hs_set_wait_limit -- time limit, in nanoseconds of the GPU's global timer, of the
 * device waits of the kernels enqueued after it returns (hs_resolve's fetch grid waits
 * for its resolution's per-request flags; hs_attend's roles wait on shared-memory
 * barriers). A CTA's waits give up once it has run that long since it started; the
 * kernel then sets HS_STATUS_TIMEOUT and returns instead of spinning, so no lost
 * hand-off can hold the GPU. Default 20 ms (a healthy wait lasts microseconds); range
 * [1 us, 10 s]. Calls captured into a CUDA graph keep the limit they were captured
 * with. Not a timeout of the call as a whole: drains of in-flight copies after an
 * expiry take at most one more limit. Returns HS_OK or HS_ERR_INVALID.
 */
int hs_set_wait_limit(hs_ctx* ctx, uint64_t ns);

/* replacement policies (hs_set_policy) */
#define HS_POLICY_LRU 0    /* the method's: victims are the least recently used slots */
#define HS_POLICY_FIFO 1   /* victims are the slots filled longest ago; a hit does not renew */
#define HS_POLICY_RANDOM 2 /* victims are drawn at random among the slots not hit */

/*
 * hs_set_policy -- the replacement policy of the hs_resolve / hs_resolve_host /
 * hs_resolve_profiled calls enqueued after it returns (the blog commentary's Fig. 3
 * discussion: LRU against policies that do not exploit locality; the pages name none,
 * so the two plainest are offered for comparison). Everything but the choice of
 * victims is the same under every policy: hits, the ascending-position order of the
 * misses, the pairing of the r-th miss with the r-th victim, the page-table update.
 *   HS_POLICY_LRU     victims in ascending (last_use, slot); hits and fills stamp t
 *   HS_POLICY_FIFO    victims in ascending (last_use, slot), but a hit keeps its
 *                     stamp, which is therefore the call that filled the slot
 *   HS_POLICY_RANDOM  victims in ascending (key, slot) among the slots not hit, where
 *                     the key of slot s at call t of request b is the high 32 bits of
 *                     SplitMix64 output number t * 2^16 + s of the generator seeded
 *                     with SplitMix64 output number b of `seed` (Steele, Lea and Flood,
 *                     2014: output n of seed x is mix(x + (n + 1) * 0x9E3779B97F4A7C15),
 *                     mix being Stafford's 13th mixer); stamps are kept as under LRU
 * The state kept so far carries over (stamps mean the last use under LRU and RANDOM
 * and the fill call under FIFO from then on). Calls captured into a CUDA graph keep
 * the policy they were captured with. hs_resolve_noalloc always uses LRU.
 * Returns HS_OK or HS_ERR_INVALID (unknown policy).
 */
int hs_set_policy(hs_ctx* ctx, int policy, uint64_t seed);

/*
 * ---------------------------------------------------------------------------------
 * Capacity planning and the shared host pool (blog commentary, section on deployment
 * knobs: top_k, device_buffer_size and host_to_device_ratio set HiSparse's working range;
 * 2048 / 6144 / 10 for a disaggregated decode instance, a 4096 buffer with ratio 8 for a
 * colocated 8-GPU node). Host code only; nothing here touches a GPU.
 */
typedef struct {
    int top_k;                   /* selections per request, layer and step (k) */
    int device_buffer_size;      /* device slots per request and layer (S), >= top_k */
    double host_to_device_ratio; /* host pool rows / device pool rows, > 0 */
    int entry_bytes;             /* bytes of one KV entry (E) */
    int layers;                  /* layers, each with its own buffer and history */
    int64_t context_len;         /* positions of history a request reserves (C) */
    int64_t hbm_bytes;           /* device memory available to the caches */
    int64_t host_bytes;          /* pinned host memory available to the pool */
    double miss_fraction;        /* expected misses per step as a fraction of top_k, in [0, 1] */
    double link_gbs;             /* host-to-device bandwidth for the fetches (0: no estimate) */
} hs_plan_params;

typedef struct {
    int64_t device_bytes_per_request; /* all layers: buffer, page table, slot tables, miss lists */
    int64_t requests_by_device;       /* requests whose device state fits hbm_bytes */
    int64_t host_pool_rows;           /* ratio x requests_by_device x S, clamped to host_bytes */
    int64_t host_pool_bytes;          /* host_pool_rows x entry_bytes x layers */
    int64_t requests_by_host;         /* requests whose context_len rows fit the pool */
    int64_t requests;                 /* admissible concurrency: the smaller of the two */
    double miss_bytes_per_step;       /* host-to-device bytes of one decode step at that concurrency */
    double link_us_per_step;          /* that traffic at link_gbs (0 when link_gbs is 0) */
} hs_plan_result;

/* hs_plan -- fills *out from *in. Returns HS_OK or HS_ERR_INVALID (a value out of range). */
int hs_plan(const hs_plan_params* in, hs_plan_result* out);

/*
 * hs_pool -- the admission side of a shared host pool of `rows` rows: a request is
 * admitted by reserving a contiguous extent for its whole history (first fit: the free
 * extent with the lowest base that is long enough), and its extent is released when it
 * finishes (merged with free neighbours). The pool only does the bookkeeping; the rows
 * themselves are a pinned, mapped store the caller allocates (see hs_create_pooled).
 *   hs_pool_create   NULL if rows <= 0 or out of memory; hs_pool_destroy frees it.
 *   hs_pool_reserve  base row of a new extent of n > 0 rows, or -1 if none is long enough
 *                    (or the bookkeeping could not allocate).
 *   hs_pool_release  frees the extent reserved at `base`: HS_OK, HS_ERR_INVALID if no
 *                    extent starts there, or HS_ERR_NOMEM (the pool is left unchanged).
 *   hs_pool_free_rows, hs_pool_largest_free   free rows in total, and in one extent.
 */
typedef struct hs_pool hs_pool;
hs_pool* hs_pool_create(int64_t rows);
void hs_pool_destroy(hs_pool* pool);
int64_t hs_pool_reserve(hs_pool* pool, int64_t n);
int hs_pool_release(hs_pool* pool, int64_t base);
int64_t hs_pool_free_rows(const hs_pool* pool);
int64_t hs_pool_largest_free(const hs_pool* pool);

/*
 * hs_create_pooled -- hs_create over a shared host pool: the caller's pinned, mapped
 * store of pool_rows rows host_stride bytes apart (16-byte aligned, stride a multiple of
 * 16 >= entry_bytes; the caller keeps it alive until hs_destroy). Request b reads its
 * position p from row base[b] + p, and only positions p < len[b] exist (others are out of
 * range: slot -1, HS_STATUS_RANGE); context_len is the longest len allowed. Initially
 * every len is 0 (nothing admitted). Returns NULL on failure, as hs_create.
 */
hs_ctx* hs_create_pooled(int num_requests, int context_len, int slots, int entry_bytes, const void* host_pool,
                         int64_t pool_rows, size_t host_stride);

/*
 * hs_set_extents -- the extents of all num_requests requests of a pooled context (host
 * arrays base[R] >= 0, len[R] in [0, context_len], base + len <= pool_rows). Every request
 * whose extent changes is a new request: its cache state (page table, slots, stamps,
 * call counter, slot contents) is emptied. Enqueued on `stream` (copies from the caller's
 * arrays, which may be reused on return); an admission-time call, not meant to be
 * captured into a CUDA graph (its copies come from pageable memory). Returns HS_OK,
 * HS_ERR_INVALID or HS_ERR_CUDA.
 */
int hs_set_extents(hs_ctx* ctx, hs_stream_t stream, const int64_t* base, const int32_t* len);

/* Number of kernels one hs_resolve call enqueues under the current flags. */
int hs_kernels_per_call(hs_ctx* ctx);

/* Description of the calling thread's last failure ("" if none). */
const char* hs_last_error(void);

/*
 * hs_resolve_noalloc -- the same resolution as hs_resolve for callers that cannot
 * allocate device memory. The paper has no counterpart: it is a packaging of the
 * same step. Engines that own all GPU memory through their own pool allocator, and
 * code that sets itself up while a stream is being captured into a CUDA graph, cannot
 * call cudaMalloc, so they cannot use hs_create. Here the caller passes every buffer,
 * laid out as for a context (R = num_requests, C = context_len, S = slots,
 * E = entry_bytes):
 *   host_kv       device-visible address of the host store, [R][C] rows host_stride
 *                 bytes apart (memory from cudaHostAlloc can be passed as is under
 *                 unified addressing); 16-byte aligned, host_stride a multiple of 16
 *   device_kv     [R][S][E] bytes, 16-byte aligned
 *   page_table    int32 [R][C]; slot_token, last_use int32 [R][S]; step int32 [R]:
 *                 the caller initialises them to -1, -1, -1 and 0 for an empty cache
 *   selections, k, out_slots, miss_counts   as for hs_resolve (B = num_requests)
 *   status        device uint32 that collects HS_STATUS_* bits, or NULL
 * It allocates nothing and calls no allocating routine. Its two kernels run one after
 * the other (hs_resolve overlaps them). The miss list the two kernels
 * share lives in a fixed file-scope device array of HS_NOALLOC_SCRATCH_BYTES bytes,
 * which every GPU that loads this library keeps until the process exits; a call needs
 * about 8*R*S + 260*R + 4*G bytes of it, G = the GPU's SM count (up to 64 more for
 * alignment) and larger sizes fail with
 * HS_ERR_LIMIT before anything is enqueued. Every call on a device shares that device's copy of the array, so calls
 * whose work overlaps on the GPU (on two streams, say) race: serialise them. The array
 * keeps the last call's contents, which the next call continues from: besides the
 * lists every call rewrites, it holds per-request flags and counters; it starts zeroed at
 * load, which is a valid state, and needs no clearing between calls. The first call on a
 * device does a one-time set-up with that device current (it looks up the array's
 * device address and sets kernel attributes): make that first call before any stream
 * capture. Returns HS_OK or HS_ERR_* (hs_last_error() describes it).
 */
#define HS_NOALLOC_SCRATCH_BYTES (2u * 1024u * 1024u)
int hs_resolve_noalloc(hs_stream_t stream, int num_requests, int context_len, int slots,
                       int entry_bytes, const uint8_t* host_kv, size_t host_stride, uint8_t* device_kv,
                       int32_t* page_table, int32_t* slot_token, int32_t* last_use, int32_t* step,
                       const int32_t* selections, int k, int32_t* out_slots, int32_t* miss_counts,
                       uint32_t* status);

#ifdef __cplusplus
}
#endif

#endif /* HS_H_ */
