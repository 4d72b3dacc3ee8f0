"""The planner's device footprint against what hs_create really allocates.

hs_plan answers the deployment question of the blog commentary's section on deployment
knobs (top_k, device_buffer_size, host_to_device_ratio) by dividing the HBM budget by the
device bytes one request costs per layer. That figure must be what the library allocates,
so it is measured here: free device memory (cudaMemGetInfo) before and after hs_create of
a large context, divided by the number of requests. Three shapes vary the page table
(context length), the slot tables (slots) and the slot buffer (entry bytes), so a term the
planner drops or miscounts -- 4 bytes per slot is 6-8 % of these footprints -- shows up.
Allocation granularity (at most a couple of MiB per buffer, about a dozen buffers) spread
over 32768 requests is below 1 KB per request, so the bound is 1 % + 1 KB.
"""
import pytest
import torch

import hierarchical_kv_cache_swap_gb300 as hs

pytestmark = pytest.mark.gpu

R = 32768
SHAPES = [  # (context_len, slots, entry_bytes)
    (2048, 2048, 16),
    (8192, 2048, 16),
    (2048, 4096, 32),
]


def planned_bytes(C: int, S: int, E: int) -> int:
    return hs.plan(top_k=S, device_buffer_size=S, host_to_device_ratio=1.0, entry_bytes=E, layers=1,
                   context_len=C, hbm_bytes=1 << 40, host_bytes=1 << 40, miss_fraction=0.0,
                   link_gbs=0.0)["device_bytes_per_request"]


@pytest.mark.parametrize("C,S,E", SHAPES)
def test_planned_device_bytes_match_the_allocation(C, S, E):
    hs.build()
    torch.cuda.init()
    hs.Context(1, 64, 16, 16).close()  # the library's kernels are loaded before measuring
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    ctx = hs.Context(R, C, S, E)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    ctx.close()
    measured = (free0 - free1) / R
    planned = planned_bytes(C, S, E)
    assert abs(measured - planned) <= 0.01 * planned + 1024, (
        f"C={C} S={S} E={E}: hs_create allocates {measured:.0f} B per request, hs_plan counts {planned}")
