// hs_api.cu -- the C ABI of include/hs.h: allocation, argument checks, launches.
//
// HiSparse keeps each request's full KV history in host memory and a small fixed-size
// cache per request on the GPU, and resolves each layer's selections inside the
// decode CUDA graph (paper abstract). Accordingly everything is allocated once in
// hs_create, and hs_resolve only checks its arguments on the host and enqueues the
// two kernels: no host synchronisation, no allocation, a launch shape fixed by the
// context, so the call can be captured in a CUDA graph and replayed.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <new>

#include "hs.h"
#include "hs_internal.h"

struct hs_ctx {
    hs::Layout L;
    int device;
    int num_sms;
    unsigned flags;
    uint8_t* host_kv;      // host address of the pinned, mapped store
    bool owns_host;        // false when the caller lent the store (hs_create_with_host)
    void* miss_area;       // miss lists, counts and flags shared by the two kernels
    int32_t* stage_sel;    // [R][S] staging for hs_resolve_host
    int32_t* stage_out;    // [R][S]
    int32_t* stage_miss;   // [R]
    bool attend_ok;        // the attention kernel's shared memory fits this device
    int64_t pool_rows;     // > 0: the host store is a shared pool of that many rows
    int64_t* d_base;       // [R] device copies of the extents (pooled contexts)
    int32_t* d_len;        // [R]
    int64_t* ext_base;     // [R] host copies, to tell which requests change
    int32_t* ext_len;      // [R]
};

namespace {

thread_local char g_err[512];

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(HS_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

void free_ctx(hs_ctx* h) {
    if (!h) return;
    if (h->owns_host) cudaFreeHost(h->host_kv);
    cudaFree(h->L.dev);
    cudaFree(h->L.pt);
    cudaFree(h->L.tok);
    cudaFree(h->L.lu);
    cudaFree(h->L.step);
    cudaFree(h->miss_area);
    cudaFree(h->L.status);
    cudaFree(h->stage_sel);
    cudaFree(h->stage_out);
    cudaFree(h->stage_miss);
    cudaFree(h->L.jslot);
    cudaFree(h->d_base);
    cudaFree(h->d_len);
    free(h->ext_base);
    free(h->ext_len);
    delete h;
}

// The device address of a host buffer that kernels may access in place: page-locked
// memory mapped into the device's address space, 4-byte aligned. nullptr for pageable
// memory, device memory or anything the runtime does not know.
void* in_place(const void* p) {
    if ((reinterpret_cast<uintptr_t>(p) & 3u) != 0) return nullptr;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();  // not a pointer the runtime knows: clear the error it set
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

int check_call(hs_ctx* h, const void* sel, int B, int k, const void* out, const void* miss) {
    if (!h) return fail(HS_ERR_INVALID, "null context");
    if (!sel || !out || !miss) return fail(HS_ERR_INVALID, "null selections/out_slots/miss_counts");
    if (B != h->L.R) return fail(HS_ERR_INVALID, "B=%d but the context has %d requests", B, h->L.R);
    if (k <= 0 || k > h->L.S) return fail(HS_ERR_INVALID, "k=%d must be in [1, slots=%d]", k, h->L.S);
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != h->device)
        return fail(HS_ERR_INVALID, "current device %d is not the context's device %d", dev, h->device);
    return HS_OK;
}

int enqueue(hs_ctx* h, cudaStream_t s, const int32_t* sel, int k, int32_t* out, int32_t* miss,
            cudaEvent_t* ev) {
    const hs::Layout& L = h->L;
    const bool fetch = !(h->flags & HS_FLAG_NO_COPY);
    // A stalled resolution (tests) publishes nothing: only a fetch grid that waits for the
    // flags may follow it; one that reads the hand-off as is would read a stale one.
    h->L.no_publish = (h->flags & HS_FLAG_TEST_STALL) ? 1 : 0;
    cudaError_t e;
    if (ev || !fetch) {
        // per-kernel timing (events before, between and after), or bookkeeping only: the
        // resolution of every request in one grid, then (when fetching) the fetch after it
        if (ev && (e = cudaEventRecord(ev[0], s)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
        if ((e = hs::launch_resolve(L, s, sel, k, out, miss, fetch, 0, L.R, true)) != cudaSuccess)
            return cuda_fail(e, "resolution kernel launch");
        if (ev && (e = cudaEventRecord(ev[1], s)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
        if (fetch && !L.no_publish && (e = hs::launch_gather(L, s, out, k, h->num_sms, false, 0, L.R)) != cudaSuccess)
            return cuda_fail(e, "fetch kernel launch");
        if (ev && (e = cudaEventRecord(ev[2], s)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    } else {
        // chunks of at most num_sms requests, each resolution overlapped with its fetch
        const int n = hs::chunk_count(L.R, h->num_sms);
        for (int i = 0; i < n; ++i) {
            int b0, nr;
            hs::chunk_requests(L.R, n, i, &b0, &nr);
            if ((e = hs::launch_resolve(L, s, sel, k, out, miss, true, b0, nr, i == 0)) != cudaSuccess)
                return cuda_fail(e, "resolution kernel launch");
            if ((e = hs::launch_gather(L, s, out, k, h->num_sms, true, b0, nr)) != cudaSuccess)
                return cuda_fail(e, "fetch kernel launch");
        }
    }
    g_err[0] = 0;
    return HS_OK;
}

}  // namespace

void hs::record_error(const char* msg) { snprintf(g_err, sizeof g_err, "%s", msg); }

extern "C" {

const char* hs_last_error(void) { return g_err; }

}  // extern "C"

namespace {

// Shared by hs_create (host_kv == nullptr: allocate the store), hs_create_with_host and
// hs_create_pooled (pool_rows > 0: the store is a shared pool addressed through extents).
hs_ctx* create(int num_requests, int context_len, int slots, int entry_bytes, uint8_t* host_kv,
               size_t host_stride, int64_t pool_rows = 0) {
    const int R = num_requests, C = context_len, S = slots, E = entry_bytes;
    if (R <= 0 || C <= 0 || S <= 0 || E <= 0) {
        fail(HS_ERR_INVALID, "all sizes must be positive (R=%d C=%d S=%d E=%d)", R, C, S, E);
        return nullptr;
    }
    if (E % 16 != 0) {
        fail(HS_ERR_INVALID, "entry_bytes=%d must be a multiple of 16", E);
        return nullptr;
    }
    if (S > hs::kMaxSlots) {
        fail(HS_ERR_LIMIT, "slots=%d exceeds %d", S, hs::kMaxSlots);
        return nullptr;
    }
    if (R > hs::kMaxRequests) {
        fail(HS_ERR_LIMIT, "num_requests=%d exceeds %d", R, hs::kMaxRequests);
        return nullptr;
    }
    // the fetch indexes 16-byte chunks of the miss rows with 32-bit integers
    if ((unsigned long long)R * S * (E / 16) > (1ull << 31)) {
        fail(HS_ERR_LIMIT, "R*S*E=%llu bytes of device buffer exceed 32 GiB",
             (unsigned long long)R * S * E);
        return nullptr;
    }
    int dev = 0, sms = 0, smem_optin = 0, can_map = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&can_map, cudaDevAttrCanMapHostMemory, dev)) != cudaSuccess) {
        cuda_fail(e, "device query");
        return nullptr;
    }
    if (!can_map) {
        fail(HS_ERR_CUDA, "device %d cannot map host memory", dev);
        return nullptr;
    }
    const size_t need = hs::resolve_smem_bytes(C, S) + 64;  // + the kernel's static shared memory
    if (need > (size_t)smem_optin) {
        fail(HS_ERR_LIMIT, "context_len=%d / slots=%d need %zu B of shared memory per CTA (max %d)", C, S,
             need, smem_optin);
        return nullptr;
    }

    hs_ctx* h = new (std::nothrow) hs_ctx();  // value-initialised: every member zero
    if (!h) {
        fail(HS_ERR_NOMEM, "out of host memory");
        return nullptr;
    }
    h->device = dev;
    h->num_sms = sms;
    hs::Layout& L = h->L;
    L.R = R; L.C = C; L.S = S; L.E = E;
    L.host_stride = host_kv ? host_stride : (size_t)E;
    const size_t host_bytes = (size_t)R * C * L.host_stride;
    const size_t dev_bytes = (size_t)R * S * E;
    void* hp = host_kv;
    if (!host_kv) {
        if ((e = cudaHostAlloc(&hp, host_bytes, cudaHostAllocMapped | cudaHostAllocPortable)) != cudaSuccess) {
            fail(HS_ERR_NOMEM, "cudaHostAlloc of %zu bytes: %s", host_bytes, cudaGetErrorString(e));
            free_ctx(h);
            return nullptr;
        }
        h->owns_host = true;
    }
    h->host_kv = (uint8_t*)hp;
    void* hdev = nullptr;
    if ((e = cudaHostGetDevicePointer(&hdev, hp, 0)) != cudaSuccess) {
        cuda_fail(e, host_kv ? "cudaHostGetDevicePointer (the lent store must be pinned and mapped)"
                             : "cudaHostGetDevicePointer");
        free_ctx(h);
        return nullptr;
    }
    L.host = (const uint8_t*)hdev;

#define HS_ALLOC(ptr, bytes)                                                           \
    do {                                                                              \
        if ((e = cudaMalloc((void**)&(ptr), (bytes))) != cudaSuccess) {               \
            fail(HS_ERR_NOMEM, "cudaMalloc of %zu bytes: %s", (size_t)(bytes),        \
                 cudaGetErrorString(e));                                              \
            free_ctx(h);                                                              \
            return nullptr;                                                           \
        }                                                                             \
    } while (0)
    HS_ALLOC(L.dev, dev_bytes);
    HS_ALLOC(L.pt, sizeof(int32_t) * (size_t)R * C);
    HS_ALLOC(L.tok, sizeof(int32_t) * (size_t)R * S);
    HS_ALLOC(L.lu, sizeof(int32_t) * (size_t)R * S);
    HS_ALLOC(L.step, sizeof(int32_t) * (size_t)R);
    HS_ALLOC(h->miss_area, hs::miss_area_bytes(R, S, sms));
    hs::carve_miss_area(L, h->miss_area);
    HS_ALLOC(L.status, sizeof(uint32_t));
    HS_ALLOC(h->stage_sel, sizeof(int32_t) * (size_t)R * S);
    HS_ALLOC(h->stage_out, sizeof(int32_t) * (size_t)R * S);
    HS_ALLOC(h->stage_miss, sizeof(int32_t) * (size_t)R);
    HS_ALLOC(L.jslot, sizeof(int32_t) * (size_t)R * S);
    if (pool_rows > 0) {
        h->pool_rows = pool_rows;
        HS_ALLOC(h->d_base, sizeof(int64_t) * (size_t)R);
        HS_ALLOC(h->d_len, sizeof(int32_t) * (size_t)R);
        h->ext_base = (int64_t*)calloc((size_t)R, sizeof(int64_t));
        h->ext_len = (int32_t*)calloc((size_t)R, sizeof(int32_t));
        if (!h->ext_base || !h->ext_len) {
            fail(HS_ERR_NOMEM, "out of host memory");
            free_ctx(h);
            return nullptr;
        }
        if ((e = cudaMemset(h->d_base, 0, sizeof(int64_t) * (size_t)R)) != cudaSuccess ||
            (e = cudaMemset(h->d_len, 0, sizeof(int32_t) * (size_t)R)) != cudaSuccess) {
            cuda_fail(e, "cudaMemset");
            free_ctx(h);
            return nullptr;
        }
        L.row_base = h->d_base;
        L.row_len = h->d_len;
    }
#undef HS_ALLOC

    if ((e = hs::configure_kernels(dev)) != cudaSuccess) {
        cuda_fail(e, "kernel configuration");
        free_ctx(h);
        return nullptr;
    }
    {  // the attention consumer needs one SM's worth of shared memory
        int optin = 0;
        h->attend_ok = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess &&
                       (size_t)optin >= hs::attend_smem_bytes() && hs::configure_attend() == cudaSuccess;
        cudaGetLastError();
    }
    if (hs_reset(h, nullptr) != HS_OK) {
        free_ctx(h);
        return nullptr;
    }
    if ((e = cudaStreamSynchronize(nullptr)) != cudaSuccess) {
        cuda_fail(e, "initial reset");
        free_ctx(h);
        return nullptr;
    }
    g_err[0] = 0;
    return h;
}

}  // namespace

extern "C" {

hs_ctx* hs_create(int num_requests, int context_len, int slots, int entry_bytes) {
    return create(num_requests, context_len, slots, entry_bytes, nullptr, 0);
}

hs_ctx* hs_create_with_host(int num_requests, int context_len, int slots, int entry_bytes, uint8_t* host_kv,
                            size_t host_stride) {
    if (!host_kv || ((uintptr_t)host_kv & 15) || host_stride % 16 != 0 || host_stride < (size_t)entry_bytes ||
        entry_bytes <= 0) {
        fail(HS_ERR_INVALID, "host_kv must be 16-byte aligned and host_stride a multiple of 16 >= entry_bytes");
        return nullptr;
    }
    return create(num_requests, context_len, slots, entry_bytes, host_kv, host_stride);
}

hs_ctx* hs_create_pooled(int num_requests, int context_len, int slots, int entry_bytes, const void* host_pool,
                         int64_t pool_rows, size_t host_stride) {
    if (!host_pool || ((uintptr_t)host_pool & 15) || host_stride % 16 != 0 || host_stride < (size_t)entry_bytes ||
        entry_bytes <= 0 || pool_rows <= 0) {
        fail(HS_ERR_INVALID, "host_pool must be 16-byte aligned, pool_rows > 0 and host_stride a multiple of 16 "
                             ">= entry_bytes");
        return nullptr;
    }
    return create(num_requests, context_len, slots, entry_bytes, (uint8_t*)host_pool, host_stride, pool_rows);
}

int hs_set_extents(hs_ctx* h, hs_stream_t stream, const int64_t* base, const int32_t* len) {
    if (!h) return fail(HS_ERR_INVALID, "null context");
    if (h->pool_rows <= 0) return fail(HS_ERR_INVALID, "the context was not created on a pool");
    if (!base || !len) return fail(HS_ERR_INVALID, "null base/len");
    const hs::Layout& L = h->L;
    for (int b = 0; b < L.R; ++b)
        if (base[b] < 0 || len[b] < 0 || len[b] > L.C || base[b] + len[b] > h->pool_rows)
            return fail(HS_ERR_INVALID, "request %d: extent [%lld, +%d) outside [0, %lld) or len > %d", b,
                        (long long)base[b], len[b], (long long)h->pool_rows, L.C);
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e;
    for (int b = 0; b < L.R; ++b) {
        if (base[b] == h->ext_base[b] && len[b] == h->ext_len[b]) continue;
        // a new request in row b: its cache state starts empty
        if ((e = cudaMemsetAsync(L.pt + (size_t)b * L.C, 0xff, sizeof(int32_t) * (size_t)L.C, s)) != cudaSuccess ||
            (e = cudaMemsetAsync(L.tok + (size_t)b * L.S, 0xff, sizeof(int32_t) * (size_t)L.S, s)) != cudaSuccess ||
            (e = cudaMemsetAsync(L.lu + (size_t)b * L.S, 0xff, sizeof(int32_t) * (size_t)L.S, s)) != cudaSuccess ||
            (e = cudaMemsetAsync(L.step + b, 0, sizeof(int32_t), s)) != cudaSuccess ||
            (e = cudaMemsetAsync(L.dev + (size_t)b * L.S * L.E, 0, (size_t)L.S * L.E, s)) != cudaSuccess)
            return cuda_fail(e, "cudaMemsetAsync");
        h->ext_base[b] = base[b];
        h->ext_len[b] = len[b];
    }
    if ((e = cudaMemcpyAsync(h->d_base, h->ext_base, sizeof(int64_t) * (size_t)L.R, cudaMemcpyHostToDevice, s)) !=
            cudaSuccess ||
        (e = cudaMemcpyAsync(h->d_len, h->ext_len, sizeof(int32_t) * (size_t)L.R, cudaMemcpyHostToDevice, s)) !=
            cudaSuccess)
        return cuda_fail(e, "cudaMemcpyAsync");
    g_err[0] = 0;
    return HS_OK;
}

int hs_append(hs_ctx* h, hs_stream_t stream, const uint8_t* kv, const int32_t* positions, int B) {
    if (!h) return fail(HS_ERR_INVALID, "null context");
    if (!kv || !positions) return fail(HS_ERR_INVALID, "null kv/positions");
    if (B != h->L.R) return fail(HS_ERR_INVALID, "B=%d but the context has %d requests", B, h->L.R);
    if ((uintptr_t)kv & 15) return fail(HS_ERR_INVALID, "kv must be 16-byte aligned");
    if (B > 65535) return fail(HS_ERR_LIMIT, "hs_append handles at most 65535 requests");
    cudaError_t e = hs::launch_append(h->L, (cudaStream_t)stream, kv, positions);
    if (e != cudaSuccess) return cuda_fail(e, "append kernel launch");
    g_err[0] = 0;
    return HS_OK;
}

static int attend_check(hs_ctx* h, int B, int H, int k) {
    if (!h) return fail(HS_ERR_INVALID, "null context");
    if (h->L.E != hs::kAttendEntryBytes)
        return fail(HS_ERR_INVALID, "hs_attend needs %d-byte entries, the context has %d", hs::kAttendEntryBytes, h->L.E);
    if (B != h->L.R) return fail(HS_ERR_INVALID, "B=%d but the context has %d requests", B, h->L.R);
    if (H < 1 || H > hs::kAttendMaxHeads) return fail(HS_ERR_INVALID, "H=%d must be in [1, %d]", H, hs::kAttendMaxHeads);
    if (k < 1) return fail(HS_ERR_INVALID, "k=%d must be >= 1", k);
    if (!h->attend_ok) return fail(HS_ERR_INVALID, "the device cannot hold the attention kernel's shared memory");
    return HS_OK;
}

int hs_attend_workspace(hs_ctx* h, int B, int H, int k, size_t* bytes) {
    int rc = attend_check(h, B, H, k);
    if (rc != HS_OK) return rc;
    if (!bytes) return fail(HS_ERR_INVALID, "null bytes");
    *bytes = hs::attend_plan(B, H, k, h->num_sms).workspace_bytes;
    g_err[0] = 0;
    return HS_OK;
}

int hs_attend(hs_ctx* h, hs_stream_t stream, const void* q, int B, int H, const int32_t* out_slots, int k,
              float sm_scale, float* o, float* lse, void* workspace, size_t workspace_bytes) {
    int rc = attend_check(h, B, H, k);
    if (rc != HS_OK) return rc;
    if (!q || !out_slots || !o || !lse) return fail(HS_ERR_INVALID, "null q/out_slots/o/lse");
    if (((uintptr_t)q & 15) || ((uintptr_t)o & 15)) return fail(HS_ERR_INVALID, "q and o must be 16-byte aligned");
    const hs::AttendPlan plan = hs::attend_plan(B, H, k, h->num_sms);
    if (plan.workspace_bytes > 0 && (!workspace || workspace_bytes < plan.workspace_bytes || ((uintptr_t)workspace & 15)))
        return fail(HS_ERR_INVALID, "workspace of %zu bytes (16-byte aligned) needed, %zu given", plan.workspace_bytes,
                    workspace_bytes);
    cudaError_t e = hs::launch_attend(h->L, (cudaStream_t)stream, (const uint16_t*)q, B, H, out_slots, k, sm_scale, o,
                                      lse, workspace, plan, (h->flags & HS_FLAG_TEST_STALL) != 0);
    if (e != cudaSuccess) return cuda_fail(e, "attention kernel launch");
    g_err[0] = 0;
    return HS_OK;
}

int hs_checksum_rows(hs_ctx* h, hs_stream_t stream, const int32_t* out_slots, int B, int k, uint64_t* sums) {
    if (!h) return fail(HS_ERR_INVALID, "null context");
    if (!out_slots || !sums) return fail(HS_ERR_INVALID, "null out_slots/sums");
    if (B != h->L.R) return fail(HS_ERR_INVALID, "B=%d but the context has %d requests", B, h->L.R);
    if (k <= 0 || k > h->L.S) return fail(HS_ERR_INVALID, "k=%d must be in [1, slots=%d]", k, h->L.S);
    if (B > 65535) return fail(HS_ERR_LIMIT, "hs_checksum_rows handles at most 65535 requests");
    cudaError_t e = hs::launch_checksum(h->L.dev, B, h->L.S, h->L.E, out_slots, k, (unsigned long long*)sums,
                                        h->num_sms, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "checksum kernel launch");
    g_err[0] = 0;
    return HS_OK;
}

void hs_destroy(hs_ctx* h) {
    if (!h) return;
    cudaDeviceSynchronize();
    free_ctx(h);
}

int hs_reset(hs_ctx* h, hs_stream_t stream) {
    if (!h) return fail(HS_ERR_INVALID, "null context");
    cudaStream_t s = (cudaStream_t)stream;
    const hs::Layout& L = h->L;
    cudaError_t e;
    if ((e = cudaMemsetAsync(L.pt, 0xff, sizeof(int32_t) * (size_t)L.R * L.C, s)) != cudaSuccess ||
        (e = cudaMemsetAsync(L.tok, 0xff, sizeof(int32_t) * (size_t)L.R * L.S, s)) != cudaSuccess ||
        (e = cudaMemsetAsync(L.lu, 0xff, sizeof(int32_t) * (size_t)L.R * L.S, s)) != cudaSuccess ||
        (e = cudaMemsetAsync(L.step, 0, sizeof(int32_t) * (size_t)L.R, s)) != cudaSuccess ||
        (e = cudaMemsetAsync(h->miss_area, 0, hs::miss_area_bytes(L.R, L.S, h->num_sms), s)) != cudaSuccess ||
        (e = cudaMemsetAsync(L.status, 0, sizeof(uint32_t), s)) != cudaSuccess ||
        (e = cudaMemsetAsync(L.dev, 0, (size_t)L.R * L.S * L.E, s)) != cudaSuccess)
        return cuda_fail(e, "cudaMemsetAsync");
    return HS_OK;
}

int hs_resolve(hs_ctx* h, hs_stream_t stream, const int32_t* sel, int B, int k, int32_t* out,
               int32_t* miss) {
    int rc = check_call(h, sel, B, k, out, miss);
    if (rc != HS_OK) return rc;
    return enqueue(h, (cudaStream_t)stream, sel, k, out, miss, nullptr);
}

int hs_resolve_profiled(hs_ctx* h, hs_stream_t stream, const int32_t* sel, int B, int k, int32_t* out,
                        int32_t* miss, hs_event_t ev[3]) {
    int rc = check_call(h, sel, B, k, out, miss);
    if (rc != HS_OK) return rc;
    if (!ev || !ev[0] || !ev[1] || !ev[2]) return fail(HS_ERR_INVALID, "three events are required");
    cudaEvent_t cev[3] = {(cudaEvent_t)ev[0], (cudaEvent_t)ev[1], (cudaEvent_t)ev[2]};
    return enqueue(h, (cudaStream_t)stream, sel, k, out, miss, cev);
}

int hs_resolve_host(hs_ctx* h, hs_stream_t stream, const int32_t* sel_host, int B, int k,
                    int32_t* out_host, int32_t* miss_host) {
    int rc = check_call(h, sel_host, B, k, out_host, miss_host);
    if (rc != HS_OK) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    const size_t n = sizeof(int32_t) * (size_t)B * k;
    cudaError_t e;
    // Page-locked buffers are read and written by the kernels in place (over the
    // host link); pageable ones go through the context's device staging buffers.
    const int32_t* dsel = static_cast<const int32_t*>(in_place(sel_host));
    int32_t* dout = static_cast<int32_t*>(in_place(out_host));
    int32_t* dmiss = static_cast<int32_t*>(in_place(miss_host));
    if (!dsel) {
        if ((e = cudaMemcpyAsync(h->stage_sel, sel_host, n, cudaMemcpyHostToDevice, s)) != cudaSuccess)
            return cuda_fail(e, "selections host->device");
        dsel = h->stage_sel;
    }
    rc = enqueue(h, s, dsel, k, dout ? dout : h->stage_out, dmiss ? dmiss : h->stage_miss, nullptr);
    if (rc != HS_OK) return rc;
    if (!dout && (e = cudaMemcpyAsync(out_host, h->stage_out, n, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
        return cuda_fail(e, "out_slots device->host");
    if (!dmiss && (e = cudaMemcpyAsync(miss_host, h->stage_miss, sizeof(int32_t) * (size_t)B,
                                       cudaMemcpyDeviceToHost, s)) != cudaSuccess)
        return cuda_fail(e, "miss_counts device->host");
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    return HS_OK;
}

uint8_t* hs_host_kv(hs_ctx* h) { return h ? h->host_kv : nullptr; }
size_t hs_host_stride(hs_ctx* h) { return h ? h->L.host_stride : 0; }
uint8_t* hs_device_kv(hs_ctx* h) { return h ? h->L.dev : nullptr; }
int32_t* hs_page_table(hs_ctx* h) { return h ? h->L.pt : nullptr; }
int32_t* hs_slot_token(hs_ctx* h) { return h ? h->L.tok : nullptr; }
int32_t* hs_last_use(hs_ctx* h) { return h ? h->L.lu : nullptr; }
int32_t* hs_step(hs_ctx* h) { return h ? h->L.step : nullptr; }

int hs_get_status(hs_ctx* h, uint32_t* bits) {
    if (!h || !bits) return fail(HS_ERR_INVALID, "null argument");
    cudaError_t e;
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    if ((e = cudaMemcpy(bits, h->L.status, sizeof(uint32_t), cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e, "status read");
    return HS_OK;
}

int hs_clear_status(hs_ctx* h) {
    if (!h) return fail(HS_ERR_INVALID, "null context");
    cudaError_t e;
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    if ((e = cudaMemset(h->L.status, 0, sizeof(uint32_t))) != cudaSuccess) return cuda_fail(e, "status clear");
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    return HS_OK;
}

int hs_set_flags(hs_ctx* h, unsigned flags) {
    if (!h) return fail(HS_ERR_INVALID, "null context");
    if (flags & ~(unsigned)(HS_FLAG_NO_COPY | HS_FLAG_TEST_STALL))
        return fail(HS_ERR_INVALID, "unknown flags 0x%x", flags);
    h->flags = flags;
    return HS_OK;
}

int hs_set_wait_limit(hs_ctx* h, uint64_t ns) {
    if (!h) return fail(HS_ERR_INVALID, "null context");
    if (ns < hs::kMinWaitNs || ns > hs::kMaxWaitNs)
        return fail(HS_ERR_INVALID, "wait limit %llu ns outside [%llu, %llu]", (unsigned long long)ns,
                    (unsigned long long)hs::kMinWaitNs, (unsigned long long)hs::kMaxWaitNs);
    h->L.wait_ns = ns;
    return HS_OK;
}

int hs_set_policy(hs_ctx* h, int policy, uint64_t seed) {
    if (!h) return fail(HS_ERR_INVALID, "null context");
    if (policy != HS_POLICY_LRU && policy != HS_POLICY_FIFO && policy != HS_POLICY_RANDOM)
        return fail(HS_ERR_INVALID, "unknown policy %d", policy);
    h->L.policy = policy;
    h->L.seed = seed;
    return HS_OK;
}

int hs_kernels_per_call(hs_ctx* h) {
    if (!h) return fail(HS_ERR_INVALID, "null context");
    if (h->flags & HS_FLAG_NO_COPY) return 1;
    return 2 * hs::chunk_count(h->L.R, h->num_sms);
}

}  // extern "C"
