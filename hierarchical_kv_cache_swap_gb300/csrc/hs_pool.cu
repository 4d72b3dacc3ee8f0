// hs_pool.cu -- the host pool and the capacity planner around the resolution step (host
// code only).
//
// HiSparse keeps every request's full KV history in host memory and gives each request
// a fixed-size device buffer (paper abstract). Three knobs set its working range: the
// number of selections per step (top_k), the device buffer per request
// (device_buffer_size) and the size of the host pool relative to the device pool
// (host_to_device_ratio); the blog commentary (section on deployment knobs) quotes
// 2048 / 6144 / 10 for a disaggregated decode instance and a 4096 buffer with ratio 8 for
// a colocated 8-GPU node, and says they must be re-swept per context length, concurrency
// and link bandwidth.
//
// * hs_plan turns the knobs and the memory budgets into the concurrency they admit and
//   the host-link time a decode step needs.
// * hs_pool is the admission side of a shared host pool: one pinned store of rows that
//   requests of different lengths share. A request is admitted by reserving a contiguous
//   extent of rows for its whole history (first fit, lowest base first); releasing an
//   extent merges it with free neighbours. Contexts created with hs_create_pooled read
//   request b's position p from row base[b] + p of the pool.
#include <stdint.h>
#include <stdlib.h>

#include <algorithm>
#include <map>
#include <new>

#include "hs.h"

struct hs_pool {
    int64_t rows;
    std::map<int64_t, int64_t> free;  // base -> length of every free extent, disjoint, never adjacent
    std::map<int64_t, int64_t> used;  // base -> length of every reserved extent
    int64_t free_rows;
};

extern "C" {

hs_pool* hs_pool_create(int64_t rows) {
    if (rows <= 0) return nullptr;
    hs_pool* p = new (std::nothrow) hs_pool();
    if (!p) return nullptr;
    p->rows = rows;
    p->free[0] = rows;
    p->free_rows = rows;
    return p;
}

void hs_pool_destroy(hs_pool* p) { delete p; }

int64_t hs_pool_reserve(hs_pool* p, int64_t n) {
    if (!p || n <= 0) return -1;
    try {  // no exception crosses the C ABI: out of memory reads as "no extent"
        for (auto it = p->free.begin(); it != p->free.end(); ++it) {
            if (it->second < n) continue;
            const int64_t base = it->first, len = it->second;
            p->used[base] = n;  // first: if this throws, nothing has changed
            p->free.erase(it);
            if (len > n) p->free[base + n] = len - n;
            p->free_rows -= n;
            return base;
        }
    } catch (...) {
    }
    return -1;
}

int hs_pool_release(hs_pool* p, int64_t base) {
    if (!p) return HS_ERR_INVALID;
    auto u = p->used.find(base);
    if (u == p->used.end()) return HS_ERR_INVALID;
    // find the free neighbours first and insert the merged extent before erasing anything,
    // so that an allocation failure (the one insertion) leaves the pool as it was
    const int64_t n0 = u->second;
    auto next = p->free.lower_bound(base);
    const bool merge_next = next != p->free.end() && next->first == base + n0;
    auto prev = next;
    bool merge_prev = false;
    if (next != p->free.begin()) {
        prev = std::prev(next);
        merge_prev = prev->first + prev->second == base;
    }
    const int64_t b = merge_prev ? prev->first : base;
    const int64_t n = (merge_prev ? prev->second : 0) + n0 + (merge_next ? next->second : 0);
    if (merge_prev) {
        prev->second = n;  // grows in place: no allocation
    } else {
        try {
            p->free[b] = n;
        } catch (...) {
            return HS_ERR_NOMEM;
        }
    }
    if (merge_next) p->free.erase(next);
    p->used.erase(u);
    p->free_rows += n0;
    return HS_OK;
}

int64_t hs_pool_free_rows(const hs_pool* p) { return p ? p->free_rows : -1; }

int64_t hs_pool_largest_free(const hs_pool* p) {
    if (!p) return -1;
    int64_t m = 0;
    for (const auto& kv : p->free) m = std::max(m, kv.second);
    return m;
}

int hs_plan(const hs_plan_params* in, hs_plan_result* out) {
    if (!in || !out) return HS_ERR_INVALID;
    if (in->top_k <= 0 || in->device_buffer_size < in->top_k || in->host_to_device_ratio <= 0.0 ||
        in->entry_bytes <= 0 || in->layers <= 0 || in->context_len <= 0 || in->hbm_bytes < 0 ||
        in->host_bytes < 0 || in->miss_fraction < 0.0 || in->miss_fraction > 1.0 || in->link_gbs < 0.0)
        return HS_ERR_INVALID;
    const int64_t S = in->device_buffer_size, C = in->context_len, L = in->layers, E = in->entry_bytes;
    // device bytes of one request: per layer its S-slot buffer, its page table over the
    // context (4 B per position), slot tokens and stamps (8 B per slot), its miss list (8 B
    // per slot), the fetch's copy of the miss answers (4 B per slot), the staging of the
    // host-buffer entry point (8 B per slot), the two hand-off flags (a 128-byte line
    // each) and three 4-byte words (call counter, the fetch's call counter, the staged
    // miss count) -- what hs_create allocates per request, which a GPU test measures
    // (with more requests than SMs a request keeps a second fetch counter: 4 B more)
    const int64_t per_layer = S * E + 4 * C + 28 * S + 268;
    out->device_bytes_per_request = L * per_layer;
    out->requests_by_device = out->device_bytes_per_request > 0 ? in->hbm_bytes / out->device_bytes_per_request : 0;
    // the host pool is host_to_device_ratio times the device pool, in rows, clamped to the budget
    const double want_rows = in->host_to_device_ratio * (double)out->requests_by_device * (double)S;
    const int64_t budget_rows = in->host_bytes / (E * L);
    out->host_pool_rows = std::min((int64_t)want_rows, budget_rows);
    out->host_pool_bytes = out->host_pool_rows * E * L;
    out->requests_by_host = out->host_pool_rows / C;
    out->requests = std::min(out->requests_by_device, out->requests_by_host);
    // host-link traffic of one decode step: every layer of every request misses
    // miss_fraction of its top_k selections
    out->miss_bytes_per_step = (double)out->requests * (double)L * in->miss_fraction * (double)in->top_k * (double)E;
    out->link_us_per_step = in->link_gbs > 0.0 ? out->miss_bytes_per_step / (in->link_gbs * 1e3) : 0.0;
    return HS_OK;
}

}  // extern "C"
