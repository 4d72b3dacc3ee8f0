// Internal interface between the C ABI (hs_api.cu) and the kernels (hs_kernels.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace hs {

constexpr int kResolveThreads = 512;               // one CTA per request
constexpr int kResolveWarps = kResolveThreads / 32;
constexpr int kRadixBits = 8;                      // LSD digit width of the victim rank
constexpr int kBins = 1 << kRadixBits;
constexpr int kGroupWords = 8;                     // bitmap words per miss-rank prefix group
constexpr int kGatherThreads = 512;
constexpr int kGatherCtasPerSm = 2;
constexpr int kGatherUnroll = 8;                   // 16-byte loads in flight per thread

constexpr int kMaxSlots = 65535;                   // slot ids are kept as uint16 in shared memory
constexpr int kMaxRequestsGather = 16384;          // per-request miss prefix lives in shared memory

// Everything the two kernels need about one context.
struct Layout {
    int R, C, S, E;
    size_t host_stride;
    const uint8_t* host;   // device-visible address of the mapped host store
    uint8_t* dev;          // [R][S][E]
    int32_t* pt;           // [R][C]
    int32_t* tok;          // [R][S]
    int32_t* lu;           // [R][S]
    int32_t* step;         // [R]
    int2* mlist;           // [R][S]: (position, slot) of the r-th miss
    int32_t* mcnt;         // [R]: misses of the last call
    uint32_t* status;      // device status word
};

// Dynamic shared memory of the resolution kernel for (C, S).
size_t resolve_smem_bytes(int C, int S);
size_t gather_smem_bytes(int R);

// Opt the kernels in to the device's maximum dynamic shared memory (the current
// device must be `device`); returns a CUDA error.
cudaError_t configure_kernels(int device);

// Enqueue the resolution kernel (one CTA per request).
cudaError_t launch_resolve(const Layout& L, cudaStream_t stream, const int32_t* sel, int k,
                           int32_t* out_slots, int32_t* miss_counts);

// Enqueue the row fetch; `pdl` chains it to the preceding kernel by programmatic
// dependent launch.
cudaError_t launch_gather(const Layout& L, cudaStream_t stream, int num_sms, bool pdl);

// Set the calling thread's message for hs_last_error().
void record_error(const char* msg);

}  // namespace hs
