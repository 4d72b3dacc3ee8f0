"""Seeded synthetic inputs for the HiSparse swap-in resolution step.

This package only makes inputs (decode-step top-k selection traces and the bytes of
the host-resident KV history); it holds none of the method's arithmetic. Both the
CPU oracle and the CUDA path consume its output. The C source is ``tracegen.c``;
``build()`` compiles it in-tree with gcc.

The five workloads below carry the shapes of the HiSparse pages' setting (top-k =
2048 and 2048 / 4096 / 6144-slot device buffers from the blog commentary's section
three and its deployment knobs; DSA, NSA and Quest sparse-attention families from the
HiSparse paper abstract). Their selections stand in for a model's indexer output.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tracegen.c")
_LIB = os.path.join(_HERE, "libtracegen.so")

KV_BF16, KV_DSA656, KV_RAW = 0, 1, 2


@dataclass(frozen=True)
class Workload:
    """One synthetic decode workload: B requests x L layers over a context of C positions."""

    name: str
    config: int          # workload id, part of every random stream's seed
    B: int               # requests
    L: int               # layers (each layer has its own cache; selections are shared)
    C: int               # context positions per request (tokens, or pages)
    S: int               # device-buffer slots per request and layer
    k: int               # selected positions per request-step
    E: int               # bytes per KV entry
    kv_kind: int         # KV_BF16 / KV_DSA656 / KV_RAW
    T: int               # decode steps
    keep_pct: int        # percentage of the previous row that is kept
    zipf_s: float        # exponent of the refill law
    recent: int = 0      # always-selected tail positions
    seed: int = 0
    no_io: bool = False  # every step after the first repeats step 0's set

    @property
    def host_bytes(self) -> int:
        return self.B * self.C * self.E

    @property
    def device_bytes(self) -> int:
        return self.B * self.S * self.E


WORKLOADS = {
    # 1 request, bf16 entries of 576 values, 512 slots, k = 256, 80 % reuse
    "tiny": Workload("tiny", 1, B=1, L=1, C=4096, S=512, k=256, E=1152, kv_kind=KV_BF16,
                     T=64, keep_pct=80, zipf_s=1.1, seed=0),
    # DSA-style decode: 656-B entries (512 fp8 + 4 fp32 scales + 64 bf16), the 64 most
    # recent positions always selected, 90 % reuse
    "dsa": Workload("dsa", 2, B=32, L=1, C=32768, S=4096, k=2048, E=656, kv_kind=KV_DSA656,
                    T=256, keep_pct=90, zipf_s=1.1, recent=64, seed=1),
    # high-concurrency long context: 256 requests x 131072 positions (22 GB of host KV)
    "long": Workload("long", 4, B=256, L=1, C=131072, S=4096, k=2048, E=656, kv_kind=KV_DSA656,
                     T=64, keep_pct=85, zipf_s=1.05, seed=3),
    # Quest-style pages: 16 tokens x 8 heads x 128 dim x (K, V) in bf16 = 65536 B per page,
    # 8 layers sharing one selection of 128 pages, 256 pages of buffer per layer
    "quest": Workload("quest", 5, B=64, L=8, C=4096, S=256, k=128, E=65536, kv_kind=KV_BF16,
                      T=128, keep_pct=90, zipf_s=1.1, seed=4),
    # the DSA-style decode with 8 layers sharing one selection per step (for the
    # layer-wise overlap of resolution and attention)
    "dsa_layers": Workload("dsa_layers", 6, B=32, L=8, C=32768, S=4096, k=2048, E=656, kv_kind=KV_DSA656,
                           T=64, keep_pct=90, zipf_s=1.1, recent=64, seed=5),
}


def sweep_workload(S: int, keep_pct: int) -> Workload:
    """Buffer/locality sweep point: 64 requests, C = 65536, 656-B entries, k = 2048."""
    assert S in (2048, 4096, 6144) and keep_pct in (50, 80, 95)
    return Workload(f"sweep_S{S}_r{keep_pct}", 3, B=64, L=1, C=65536, S=S, k=2048, E=656,
                    kv_kind=KV_DSA656, T=128, keep_pct=keep_pct, zipf_s=1.1, seed=2)


def noio_workload(S: int = 4096) -> Workload:
    """The sweep's no-IO run: every call after the first re-selects step 0's set."""
    return replace(sweep_workload(S, 95), name=f"noio_S{S}", no_io=True)


def build(force: bool = False) -> str:
    """Compile tracegen.c into libtracegen.so next to it; returns the library path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-pthread", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.tg_trace.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_uint64,
                                 ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
        lib.tg_trace.restype = ctypes.c_int
        lib.tg_kv_row.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_uint64,
                                  ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.tg_kv_row.restype = ctypes.c_int
        lib.tg_fill_kv.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_uint64, ctypes.c_int,
                                   ctypes.c_int]
        lib.tg_fill_kv.restype = ctypes.c_int
        _lib = lib
    return _lib


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def trace(w: Workload, T: int | None = None, B: int | None = None, layer: int = 0) -> np.ndarray:
    """Selections of workload ``w`` as an int32 array [T][B][k] (one [B][k] row block per step).

    ``T``/``B`` override the step count / request count (requests 0..B-1 of the same
    streams; a shorter T is a prefix of the longer trace).
    """
    T = w.T if T is None else T
    B = w.B if B is None else B
    out = np.empty((T, B, w.k), dtype=np.int32)
    rc = _load().tg_trace(B, w.C, w.k, T, w.keep_pct, w.zipf_s, w.recent, int(w.no_io), w.seed,
                          w.config, layer, _threads(), out.ctypes.data)
    if rc != 0:
        raise ValueError(f"tg_trace failed ({rc}) for {w}")
    return out


def raw_trace(B: int, C: int, k: int, T: int, keep_pct: int, zipf_s: float, recent: int = 0,
              no_io: bool = False, seed: int = 0, config: int = 0, layer: int = 0) -> np.ndarray:
    """Trace with explicit parameters (small cases in tests)."""
    out = np.empty((T, B, k), dtype=np.int32)
    rc = _load().tg_trace(B, C, k, T, keep_pct, zipf_s, recent, int(no_io), seed, config, layer,
                          1, out.ctypes.data)
    if rc != 0:
        raise ValueError(f"tg_trace failed ({rc})")
    return out


def kv_row(w: Workload, b: int, p: int, layer: int = 0) -> np.ndarray:
    """The E bytes of request b's history row p (uint8)."""
    out = np.empty(w.E, dtype=np.uint8)
    rc = _load().tg_kv_row(out.ctypes.data, w.E, w.kv_kind, w.seed, layer, b, p)
    if rc != 0:
        raise ValueError("tg_kv_row failed")
    return out


def fill_kv(ptr: int, stride: int, w: Workload, B: int | None = None, layer: int = 0) -> None:
    """Fill a host buffer at address ``ptr`` laid out [B][C][stride] with w's KV history."""
    B = w.B if B is None else B
    rc = _load().tg_fill_kv(ptr, stride, B, w.C, w.E, w.kv_kind, w.seed, layer, _threads())
    if rc != 0:
        raise ValueError("tg_fill_kv failed")


def fill_kv_array(w: Workload, B: int | None = None, layer: int = 0) -> np.ndarray:
    """A new numpy array [B][C][E] holding w's KV history (small workloads only)."""
    B = w.B if B is None else B
    out = np.empty((B, w.C, w.E), dtype=np.uint8)
    fill_kv(out.ctypes.data, w.E, w, B=B, layer=layer)
    return out
