// hs_consume.cu -- the consumer stand-in and the decode-time append around the step.
//
// HiSparse's resolution leaves every selected entry in a device slot for the layer's
// sparse attention to read (blog commentary, section two: a resident entry takes part
// in the computation directly); for models that share one selection across layers,
// the next layer's resolution can run while this layer's consumer reads (paper
// abstract: exact layer-wise prefetching). The attention itself needs trained weights
// and is not built here; this kernel reads exactly what it would read -- the k rows of
// every request through out_slots -- and reduces them to one checksum per request, so
// that the two-stream overlap can be measured and the consumer's view checked.
//
// checksum_kernel: grid (parts, R); CTA (part, b) sums the 8-byte words of its share of
// request b's k * E / 16 sixteen-byte chunks (coalesced loads within each row) and adds
// its partial into sums[b]. Addition modulo 2^64 is associative and commutative, so the
// result does not depend on the order of the atomics.
#include <cuda_runtime.h>
#include <stdint.h>

#include "hs_internal.h"

namespace hs {
namespace {

constexpr int kConsumeThreads = 256;

__global__ void __launch_bounds__(kConsumeThreads)
checksum_kernel(const uint8_t* __restrict__ dev, int S, int E, const int32_t* __restrict__ out_slots, int k,
                unsigned long long* __restrict__ sums) {
    const int b = blockIdx.y;
    const uint32_t cpr = (uint32_t)E >> 4;
    const uint32_t n = (uint32_t)k * cpr;
    const uint32_t per = (n + gridDim.x - 1) / gridDim.x;
    const uint32_t c0 = blockIdx.x * per, c1 = min(c0 + per, n);
    const int32_t* ob = out_slots + (size_t)b * k;
    const uint8_t* db = dev + (size_t)b * S * E;
    unsigned long long acc = 0;
    for (uint32_t c = c0 + threadIdx.x; c < c1; c += kConsumeThreads) {
        const uint32_t j = c / cpr, off = c - j * cpr;
        const int32_t s = __ldg(ob + j);
        if (s < 0) continue;  // padding or an out-of-range selection
        const ulonglong2 v = __ldcs(reinterpret_cast<const ulonglong2*>(db + (size_t)s * E) + off);
        acc += v.x + v.y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    __shared__ unsigned long long part[kConsumeThreads / 32];
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long t = 0;
        for (int w = 0; w < kConsumeThreads / 32; ++w) t += part[w];
        atomicAdd(sums + b, t);
    }
}

constexpr int kAppendThreads = 256;

// Decode-time append: row kv[b] joins request b's history at position pos[b] in the
// host store (zero-copy stores over the host link; in a pooled store, row base[b] + p)
// and, when that position is resident, its device slot. Grid (parts, R); CTA (part, b) copies its share of the
// row's 16-byte chunks.
__global__ void __launch_bounds__(kAppendThreads)
append_kernel(const Layout L, const uint8_t* __restrict__ kv, const int32_t* __restrict__ pos) {
    const int b = blockIdx.y;
    const int32_t p = __ldg(pos + b);
    if (p < 0) return;  // no new entry for this request
    if (p >= (L.row_len ? __ldg(L.row_len + b) : L.C)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(L.status, 1u /* HS_STATUS_RANGE */);
        return;
    }
    const int32_t s = L.pt[(size_t)b * L.C + p];
    const uint32_t cpr = (uint32_t)L.E >> 4;
    const uint32_t per = (cpr + gridDim.x - 1) / gridDim.x;
    const uint32_t c0 = blockIdx.x * per, c1 = min(c0 + per, cpr);
    const uint4* src = reinterpret_cast<const uint4*>(kv + (size_t)b * L.E);
    const int64_t row = (L.row_base ? __ldg(L.row_base + b) : (int64_t)b * L.C) + p;
    uint4* host = reinterpret_cast<uint4*>(const_cast<uint8_t*>(L.host) + (size_t)row * L.host_stride);
    uint4* dev = s >= 0 ? reinterpret_cast<uint4*>(L.dev + ((size_t)b * L.S + s) * L.E) : nullptr;
    for (uint32_t c = c0 + threadIdx.x; c < c1; c += kAppendThreads) {
        const uint4 v = __ldg(src + c);
        host[c] = v;
        if (dev) dev[c] = v;
    }
}

}  // namespace

cudaError_t launch_append(const Layout& L, cudaStream_t stream, const uint8_t* kv, const int32_t* positions) {
    const uint32_t cpr = (uint32_t)L.E >> 4;
    uint32_t parts = (cpr + kAppendThreads * 4 - 1) / (kAppendThreads * 4);  // >= 4 chunks per thread
    if (parts < 1) parts = 1;
    append_kernel<<<dim3(parts, (unsigned)L.R), kAppendThreads, 0, stream>>>(L, kv, positions);
    return cudaGetLastError();
}

cudaError_t launch_checksum(const uint8_t* dev, int R, int S, int E, const int32_t* out_slots, int k,
                            unsigned long long* sums, int num_sms, cudaStream_t stream) {
    cudaError_t e = cudaMemsetAsync(sums, 0, sizeof(unsigned long long) * (size_t)R, stream);
    if (e != cudaSuccess) return e;
    const uint32_t n = (uint32_t)k * ((uint32_t)E >> 4);
    // about four CTAs per SM in total, none smaller than one chunk per thread
    uint32_t parts = (uint32_t)((4 * num_sms + R - 1) / R);
    const uint32_t max_parts = (n + kConsumeThreads - 1) / kConsumeThreads;
    if (parts > max_parts) parts = max_parts;
    if (parts < 1) parts = 1;
    checksum_kernel<<<dim3(parts, (unsigned)R), kConsumeThreads, 0, stream>>>(dev, S, E, out_slots, k, sums);
    return cudaGetLastError();
}

}  // namespace hs
