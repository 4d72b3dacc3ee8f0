// hs_noalloc.cu -- hs_resolve_noalloc: the resolution step with no allocation at all.
//
// Some callers cannot call cudaMalloc: engines that own all device memory through
// their own pool (a raw cudaMalloc would bypass their accounting and may synchronize
// the device), and code that sets itself up while a stream is being captured into a
// CUDA graph (allocation is not a stream operation and is refused during global
// capture). hs_create allocates, so such callers cannot use a context. This entry
// point takes every buffer from the caller instead; the only extra memory it needs,
// the per-call miss list that the resolution kernel hands to the fetch kernel, lives
// in the file-scope array below, which every GPU that loads this library holds
// until the process exits.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "hs.h"
#include "hs_internal.h"

namespace {

// The miss area of the two kernels (positions, slots, per-request flags), then one
// status word. Zero at load, which is a valid initial state.
static __device__ __align__(256) unsigned char g_noalloc_scratch[HS_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

struct DeviceSetup {
    std::mutex lock;
    bool ready = false;       // set only once every step below has succeeded
    void* scratch = nullptr;  // device address of g_noalloc_scratch on this device
    int num_sms = 0;
};
DeviceSetup g_setup[kMaxDevices];

int noalloc_fail(int code, const char* msg) {
    hs::record_error(msg);  // reported by hs_last_error()
    return code;
}

// Per device, with that device current: the array's device address (host code only
// sees a host-side stand-in under its name) and the kernels' shared-memory opt-in. The
// device counts as set up only after all of it succeeded; a failed attempt (a transient
// error, or a first call made while a stream is being captured) leaves it unset, and
// the next call tries again.
cudaError_t setup_device(int dev, DeviceSetup** out) {
    DeviceSetup& d = g_setup[dev];
    std::lock_guard<std::mutex> guard(d.lock);
    *out = &d;
    if (d.ready) return cudaSuccess;
    void* p = nullptr;
    int sms = 0;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = hs::configure_kernels(dev);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();  // do not leave the failure for the caller's next check
        return e;
    }
    d.scratch = p;
    d.num_sms = sms;
    d.ready = true;
    return cudaSuccess;
}

}  // namespace

extern "C" int hs_resolve_noalloc(hs_stream_t stream, int num_requests, int context_len, int slots,
                                  int entry_bytes, const uint8_t* host_kv, size_t host_stride,
                                  uint8_t* device_kv, int32_t* page_table, int32_t* slot_token,
                                  int32_t* last_use, int32_t* step, const int32_t* selections, int k,
                                  int32_t* out_slots, int32_t* miss_counts, uint32_t* status) {
    const int R = num_requests, C = context_len, S = slots, E = entry_bytes;
    if (R <= 0 || C <= 0 || S <= 0 || E <= 0 || E % 16 != 0)
        return noalloc_fail(HS_ERR_INVALID, "sizes must be positive and entry_bytes a multiple of 16");
    if (k <= 0 || k > S) return noalloc_fail(HS_ERR_INVALID, "k must be in [1, slots]");
    if (!host_kv || !device_kv || !page_table || !slot_token || !last_use || !step || !selections ||
        !out_slots || !miss_counts)
        return noalloc_fail(HS_ERR_INVALID, "null buffer");
    if (host_stride < (size_t)E || host_stride % 16 != 0 || ((uintptr_t)host_kv & 15) ||
        ((uintptr_t)device_kv & 15))
        return noalloc_fail(HS_ERR_INVALID,
                            "host_kv/device_kv must be 16-byte aligned and host_stride a multiple of 16 >= entry_bytes");
    if (S > hs::kMaxSlots || R > hs::kMaxRequests)
        return noalloc_fail(HS_ERR_LIMIT, "slots or num_requests beyond this build's limits");
    if ((unsigned long long)R * S * (E / 16) > (1ull << 31))
        return noalloc_fail(HS_ERR_LIMIT, "device buffer beyond 32 GiB");
    int nsm = 0;
    {
        int dv = -1;
        cudaError_t e0 = cudaGetDevice(&dv);
        if (e0 == cudaSuccess) e0 = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dv);
        if (e0 != cudaSuccess) return noalloc_fail(HS_ERR_CUDA, cudaGetErrorString(e0));
    }
    const size_t area = hs::miss_area_bytes(R, S, nsm);
    if (area + sizeof(uint32_t) > HS_NOALLOC_SCRATCH_BYTES)
        return noalloc_fail(HS_ERR_LIMIT,
                            "num_requests * slots too large for the fixed scratch array "
                            "(about 8*R*S + 260*R + 4*SMs bytes must fit in HS_NOALLOC_SCRATCH_BYTES)");
    int dev = -1, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return noalloc_fail(HS_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return noalloc_fail(HS_ERR_LIMIT, "device ordinal beyond 63");
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
        return noalloc_fail(HS_ERR_CUDA, cudaGetErrorString(e));
    if (hs::resolve_smem_bytes(C, S) + 64 > (size_t)optin)  // + static shared memory
        return noalloc_fail(HS_ERR_LIMIT, "context_len/slots need more shared memory than a CTA has");
    DeviceSetup* d = nullptr;
    if ((e = setup_device(dev, &d)) != cudaSuccess) return noalloc_fail(HS_ERR_CUDA, cudaGetErrorString(e));

    unsigned char* base = static_cast<unsigned char*>(d->scratch);
    hs::Layout L;
    L.R = R; L.C = C; L.S = S; L.E = E;
    L.host_stride = host_stride;
    L.host = host_kv;
    L.dev = device_kv;
    L.pt = page_table;
    L.tok = slot_token;
    L.lu = last_use;
    L.step = step;
    hs::carve_miss_area(L, base);
    L.status = status ? status : reinterpret_cast<uint32_t*>(base + area);
    cudaStream_t s = (cudaStream_t)stream;
    if ((e = hs::launch_resolve(L, s, selections, k, out_slots, miss_counts, true, 0, R, true)) != cudaSuccess)
        return noalloc_fail(HS_ERR_CUDA, cudaGetErrorString(e));
    // Callers with different sizes share this array, so the fetch CTAs' call counters
    // need not line up with a caller's requests: the fetch therefore runs after the
    // resolution here (no overlap) and reads the hand-off without waiting on flags.
    if ((e = hs::launch_gather(L, s, out_slots, k, d->num_sms, false, 0, R)) != cudaSuccess)
        return noalloc_fail(HS_ERR_CUDA, cudaGetErrorString(e));
    hs::record_error("");
    return HS_OK;
}
