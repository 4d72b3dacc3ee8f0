"""Capacity planning from the deployment knobs, restated plainly (test infrastructure).

The blog commentary's section on deployment knobs: top_k, device_buffer_size and
host_to_device_ratio set HiSparse's working range (2048 / 6144 / 10 for a disaggregated
decode instance). Reading taken: the host pool is host_to_device_ratio times the device
pool, counted in entries (rows); the device pool is the requests' S-slot buffers; every
admitted request reserves its whole history in the host pool.

What one request costs on the device per layer is not restated here: it is whatever the
library allocates, which a GPU test measures (cudaMemGetInfo around hs_create) and
compares with the planner's figure. This restatement takes that figure as an input and
checks the admission arithmetic built on it.
"""


def plan(top_k, device_buffer_size, host_to_device_ratio, entry_bytes, layers, context_len,
         hbm_bytes, host_bytes, miss_fraction, link_gbs, device_bytes_per_layer):
    S, C, L, E = device_buffer_size, context_len, layers, entry_bytes
    device_bytes = L * device_bytes_per_layer
    by_device = hbm_bytes // device_bytes
    rows = min(int(host_to_device_ratio * by_device * S), host_bytes // (E * L))
    by_host = rows // C
    requests = min(by_device, by_host)
    miss_bytes = requests * L * miss_fraction * top_k * E
    return {"device_bytes_per_request": device_bytes, "requests_by_device": by_device,
            "host_pool_rows": rows, "host_pool_bytes": rows * E * L, "requests_by_host": by_host,
            "requests": requests, "miss_bytes_per_step": miss_bytes,
            "link_us_per_step": miss_bytes / (link_gbs * 1e3) if link_gbs > 0 else 0.0}
