"""Shared driver for the GPU parity tests: run a trace through the CUDA path (via the
C ABI) and through the CPU oracle on the same seeded inputs, and compare.

Requests are independent, so the oracle may follow a sample of them: it gets each
sampled request's own host rows and selections and must reproduce, bit for bit, that
request's out_slots and miss counts at every step and its page table, slot tokens,
last-use stamps, step counter and device-slot bytes at the checkpoints.
"""
from __future__ import annotations

import numpy as np
import torch

import hierarchical_kv_cache_swap_gb300 as hs
import tracegen
from oracle import Oracle


class DeviceRun:
    """A context plus the whole trace resident on the device."""

    def __init__(self, w: tracegen.Workload, T: int, B: int | None = None, layer: int = 0,
                 sel: np.ndarray | None = None, fill: bool = True):
        self.w = w
        self.B = w.B if B is None else B
        self.T = T
        self.ctx = hs.Context(self.B, w.C, w.S, w.E)
        if fill:
            tracegen.fill_kv(self.ctx.host_kv_address(), self.ctx.host_stride, w, B=self.B, layer=layer)
        self.sel = tracegen.trace(w, T=T, B=self.B) if sel is None else sel
        self.sel_dev = torch.from_numpy(self.sel).cuda()
        self.out_dev = torch.full((T, self.B, w.k), -7, dtype=torch.int32, device="cuda")
        self.miss_dev = torch.full((T, self.B), -7, dtype=torch.int32, device="cuda")

    def step(self, t: int, stream=None) -> None:
        self.ctx.resolve(self.sel_dev[t], self.out_dev[t], self.miss_dev[t], stream=stream)

    def snapshot(self, rows) -> dict:
        rows = torch.as_tensor(rows, device="cuda", dtype=torch.long)
        return {
            "pt": self.ctx.page_table()[rows].cpu().numpy(),
            "tok": self.ctx.slot_token()[rows].cpu().numpy(),
            "lu": self.ctx.last_use()[rows].cpu().numpy(),
            "t": self.ctx.step()[rows].cpu().numpy(),
            "dev": self.ctx.device_kv()[rows].cpu().numpy(),
        }

    def close(self):
        self.ctx.close()


def run_and_compare(w: tracegen.Workload, T: int, B: int | None = None, sample=None,
                    checkpoints=None, layer: int = 0, run: DeviceRun | None = None,
                    policy: int = 0, seed: int = 0) -> dict:
    """Run T steps on the GPU, then replay the sampled requests on the oracle, both
    under replacement `policy` (0 LRU, 1 FIFO, 2 RANDOM with `seed`).

    Returns summary stats (total misses per sampled request). Raises AssertionError on
    the first difference.
    """
    own = run is None
    run = run or DeviceRun(w, T, B, layer=layer)
    B = run.B
    sample = list(range(B)) if sample is None else list(sample)
    checkpoints = sorted(set(checkpoints or [T - 1]))
    snaps = {}
    run.ctx.set_policy(policy, seed)
    for t in range(T):
        run.step(t)
        if t in checkpoints:
            snaps[t] = run.snapshot(sample)
    torch.cuda.synchronize()
    assert run.ctx.status() == 0
    out = run.out_dev[:, sample].cpu().numpy()
    miss = run.miss_dev[:, sample].cpu().numpy()

    o = Oracle(len(sample), w.C, w.S, w.E)
    o.set_policy(policy, seed)
    o.set_request_ids(sample)  # RANDOM's draws depend on the request number
    base = run.ctx.host_kv_address()
    row_bytes = w.C * run.ctx.host_stride
    for t in range(T):
        for i, b in enumerate(sample):
            o_out, o_m, st = o.resolve_request(i, base + b * row_bytes, run.ctx.host_stride,
                                               run.sel[t, b])
            assert st == 0
            if not np.array_equal(o_out, out[t, i]):
                bad = np.nonzero(o_out != out[t, i])[0][:8]
                raise AssertionError(f"{w.name}: out_slots differ at step {t}, request {b}, "
                                     f"j={bad.tolist()} gpu={out[t, i][bad].tolist()} "
                                     f"oracle={o_out[bad].tolist()}")
            assert o_m == miss[t, i], f"{w.name}: miss count step {t} request {b}: {miss[t, i]} vs {o_m}"
        if t in snaps:
            s = snaps[t]
            for name, ref in (("pt", o.pt), ("tok", o.tok), ("lu", o.lu), ("t", o.t)):
                if not np.array_equal(s[name], ref):
                    raise AssertionError(f"{w.name}: {name} differs after step {t}")
            for i in range(len(sample)):
                if not np.array_equal(s["dev"][i], o.dev_rows(i)):
                    raise AssertionError(f"{w.name}: device bytes differ after step {t}, request {sample[i]}")
    stats = {"misses": miss.sum(axis=0)}
    if own:
        run.close()
    return stats
