"""GB300-native HiSparse swap-in resolution: a thin Python binding over ``libhs.so``.

HiSparse (paper abstract) keeps every request's full KV history in host memory and a
small fixed-size cache of slots on the GPU; per layer and decode step one fused
resolution does hit detection, LRU replacement, the page-table update and the
host-to-device fetch of the misses. All of that runs in the library's CUDA kernels
(sm_103a) behind the C ABI of ``include/hs.h``; this module only marshals arguments
(torch tensors or raw addresses, streams, events) to those calls. There is no
fallback: if the compiled library is missing, loading fails with an error.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libhs.so")

HS_OK = 0
HS_ERR_INVALID = -1
HS_ERR_CUDA = -2
HS_ERR_NOMEM = -3
HS_ERR_LIMIT = -4
HS_STATUS_RANGE = 1
HS_STATUS_DUP = 2
HS_STATUS_STEP_LIMIT = 4
HS_STATUS_TIMEOUT = 8
HS_FLAG_NO_COPY = 1
HS_FLAG_TEST_STALL = 2
POLICY_LRU, POLICY_FIFO, POLICY_RANDOM = 0, 1, 2

# every symbol include/hs.h declares, with (restype, argtypes)
_VP, _I, _SZ, _U = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint
_I64, _F64 = ctypes.c_int64, ctypes.c_double


class PlanParams(ctypes.Structure):
    """hs_plan_params (include/hs.h)."""
    _fields_ = [("top_k", _I), ("device_buffer_size", _I), ("host_to_device_ratio", _F64),
                ("entry_bytes", _I), ("layers", _I), ("context_len", _I64), ("hbm_bytes", _I64),
                ("host_bytes", _I64), ("miss_fraction", _F64), ("link_gbs", _F64)]


class PlanResult(ctypes.Structure):
    """hs_plan_result (include/hs.h)."""
    _fields_ = [("device_bytes_per_request", _I64), ("requests_by_device", _I64), ("host_pool_rows", _I64),
                ("host_pool_bytes", _I64), ("requests_by_host", _I64), ("requests", _I64),
                ("miss_bytes_per_step", _F64), ("link_us_per_step", _F64)]

SIGNATURES = {
    "hs_create": (_VP, [_I, _I, _I, _I]),
    "hs_create_with_host": (_VP, [_I, _I, _I, _I, _VP, _SZ]),
    "hs_checksum_rows": (_I, [_VP, _VP, _VP, _I, _I, _VP]),
    "hs_append": (_I, [_VP, _VP, _VP, _VP, _I]),
    "hs_resolve": (_I, [_VP, _VP, _VP, _I, _I, _VP, _VP]),
    "hs_resolve_host": (_I, [_VP, _VP, _VP, _I, _I, _VP, _VP]),
    "hs_resolve_profiled": (_I, [_VP, _VP, _VP, _I, _I, _VP, _VP, _VP]),
    "hs_destroy": (None, [_VP]),
    "hs_reset": (_I, [_VP, _VP]),
    "hs_host_kv": (_VP, [_VP]),
    "hs_host_stride": (_SZ, [_VP]),
    "hs_device_kv": (_VP, [_VP]),
    "hs_page_table": (_VP, [_VP]),
    "hs_slot_token": (_VP, [_VP]),
    "hs_last_use": (_VP, [_VP]),
    "hs_step": (_VP, [_VP]),
    "hs_get_status": (_I, [_VP, ctypes.POINTER(ctypes.c_uint32)]),
    "hs_clear_status": (_I, [_VP]),
    "hs_set_flags": (_I, [_VP, _U]),
    "hs_set_policy": (_I, [_VP, _I, ctypes.c_uint64]),
    "hs_set_wait_limit": (_I, [_VP, ctypes.c_uint64]),
    "hs_attend": (_I, [_VP, _VP, _VP, _I, _I, _VP, _I, ctypes.c_float, _VP, _VP, _VP, ctypes.c_size_t]),
    "hs_attend_workspace": (_I, [_VP, _I, _I, _I, ctypes.POINTER(ctypes.c_size_t)]),
    "hs_kernels_per_call": (_I, [_VP]),
    "hs_plan": (_I, [ctypes.POINTER(PlanParams), ctypes.POINTER(PlanResult)]),
    "hs_pool_create": (_VP, [_I64]),
    "hs_pool_destroy": (None, [_VP]),
    "hs_pool_reserve": (_I64, [_VP, _I64]),
    "hs_pool_release": (_I, [_VP, _I64]),
    "hs_pool_free_rows": (_I64, [_VP]),
    "hs_pool_largest_free": (_I64, [_VP]),
    "hs_create_pooled": (_VP, [_I, _I, _I, _I, _VP, _I64, _SZ]),
    "hs_set_extents": (_I, [_VP, _VP, _VP, _VP]),
    "hs_last_error": (ctypes.c_char_p, []),
    "hs_resolve_noalloc": (_I, [_VP, _I, _I, _I, _I, _VP, _SZ, _VP, _VP, _VP, _VP, _VP, _VP, _I,
                                _VP, _VP, _VP]),
}


class HsError(RuntimeError):
    pass


_lib = None


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libhs.so in-tree with nvcc for sm_103a (see _nvcc.py)."""
    from . import _nvcc
    return _nvcc.build(force=force, verbose=verbose)


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libhs.so and declare its C signatures; raises if it has not been built."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise HsError(f"{path} is missing: build it first (hierarchical_kv_cache_swap_gb300.build())")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == LIB_PATH:
        _lib = lib
    return lib


def last_error() -> str:
    return (load_library().hs_last_error() or b"").decode()


_I32 = np.dtype(np.int32)


def _addr(x) -> int:
    """Device or host address of a torch tensor / numpy array / int."""
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        if x.flags.writeable and x.flags.c_contiguous and x.nbytes:
            return ctypes.addressof(ctypes.c_char.from_buffer(x))  # ~3x cheaper than .ctypes
        return x.ctypes.data
    return x.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class _DeviceArray:
    """Minimal __cuda_array_interface__ holder so torch can view library-owned memory."""

    def __init__(self, ptr: int, shape, typestr: str, owner):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (ptr, False), "version": 3, "strides": None}
        self._owner = owner


def plan(**params) -> dict:
    """hs_plan: the concurrency and host-link time the deployment knobs admit. Keywords are
    the fields of hs_plan_params; returns the fields of hs_plan_result as a dict."""
    lib = load_library()
    inp = PlanParams(**params)
    out = PlanResult()
    if lib.hs_plan(ctypes.byref(inp), ctypes.byref(out)) != HS_OK:
        raise HsError(f"hs_plan refused {params}")
    return {name: getattr(out, name) for name, _ in PlanResult._fields_}


class Pool:
    """Admission bookkeeping of a shared host pool of `rows` rows (hs_pool_*)."""

    def __init__(self, rows: int):
        self._lib = load_library()
        self.rows = rows
        self._h = self._lib.hs_pool_create(rows)
        if not self._h:
            raise HsError("hs_pool_create failed")

    def reserve(self, n: int) -> int:
        """Base row of a new extent of n rows, or -1 if none is long enough (first fit)."""
        return int(self._lib.hs_pool_reserve(self._h, n))

    def release(self, base: int) -> None:
        if self._lib.hs_pool_release(self._h, base) != HS_OK:
            raise HsError(f"no extent starts at {base}")

    def free_rows(self) -> int:
        return int(self._lib.hs_pool_free_rows(self._h))

    def largest_free(self) -> int:
        return int(self._lib.hs_pool_largest_free(self._h))

    def close(self) -> None:
        if getattr(self, "_h", None):
            self._lib.hs_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()


class Context:
    """One layer's cache for R requests (``hs_create``); release with close()."""

    def __init__(self, num_requests: int, context_len: int, slots: int, entry_bytes: int,
                 share_host_with: "Context | None" = None, pool=None):
        """share_host_with: borrow another context's host store (hs_create_with_host);
        that context must outlive this one. pool: (address, rows, stride) of a pinned host
        pool shared through extents (hs_create_pooled); the pool must outlive this one."""
        self._lib = load_library()
        self.R, self.C, self.S, self.E = num_requests, context_len, slots, entry_bytes
        self.pool_rows = 0
        if pool is not None:
            addr, rows, stride = pool
            self.pool_rows = rows
            self._h = self._lib.hs_create_pooled(num_requests, context_len, slots, entry_bytes, addr, rows, stride)
        elif share_host_with is None:
            self._h = self._lib.hs_create(num_requests, context_len, slots, entry_bytes)
        else:
            self._lender = share_host_with
            self._h = self._lib.hs_create_with_host(num_requests, context_len, slots, entry_bytes,
                                                    share_host_with.host_kv_address(),
                                                    share_host_with.host_stride)
        if not self._h:
            raise HsError(f"hs_create failed: {last_error()}")
        self.host_stride = int(self._lib.hs_host_stride(self._h))

    # ------------------------------------------------------------------ life cycle
    def close(self) -> None:
        if getattr(self, "_h", None):
            self._lib.hs_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def _check(self, rc: int, what: str) -> None:
        if rc != HS_OK:
            raise HsError(f"{what} failed ({rc}): {last_error()}")

    # ------------------------------------------------------------------ the step
    def resolve(self, selections, out_slots, miss_counts, stream=None) -> None:
        """Enqueue one resolution: selections/out_slots int32 [R, k], miss_counts int32 [R] (device)."""
        B, k = selections.shape
        self._check(self._lib.hs_resolve(self._h, _stream(stream), _addr(selections), B, k,
                                         _addr(out_slots), _addr(miss_counts)), "hs_resolve")

    def resolve_host(self, selections: np.ndarray, out_slots: np.ndarray, miss_counts: np.ndarray,
                     stream=None) -> None:
        """Resolve with host numpy buffers and wait. Page-locked buffers (e.g. views of
        pinned torch tensors) are accessed by the kernels in place; pageable ones are staged
        through device buffers."""
        for a in (selections, out_slots, miss_counts):
            if not isinstance(a, np.ndarray) or a.dtype != _I32 or not a.flags.c_contiguous:
                raise ValueError("resolve_host wants C-contiguous int32 numpy arrays")
        B, k = selections.shape
        if out_slots.shape != (B, k) or miss_counts.shape != (B,):
            raise ValueError(f"out_slots must be {(B, k)} and miss_counts {(B,)}")
        self._check(self._lib.hs_resolve_host(self._h, _stream(stream), _addr(selections), B, k,
                                              _addr(out_slots), _addr(miss_counts)),
                    "hs_resolve_host")

    def resolve_profiled(self, selections, out_slots, miss_counts, events, stream=None) -> None:
        """resolve() that records events[0..2] around the two kernels (torch.cuda.Event)."""
        B, k = selections.shape
        for e in events:  # torch creates the underlying CUDA event on first record
            if not e.cuda_event:
                e.record(stream if stream is not None else None)
        arr = (ctypes.c_void_p * 3)(*[e.cuda_event for e in events])
        self._check(self._lib.hs_resolve_profiled(self._h, _stream(stream), _addr(selections), B, k,
                                                  _addr(out_slots), _addr(miss_counts), arr),
                    "hs_resolve_profiled")

    def checksum_rows(self, out_slots, sums, stream=None) -> None:
        """Consumer stand-in: sums[b] = sum mod 2^64 of the 8-byte words of request b's
        resolved rows (out_slots int32 [R, k], sums a 64-bit tensor [R], device)."""
        B, k = out_slots.shape
        self._check(self._lib.hs_checksum_rows(self._h, _stream(stream), _addr(out_slots), B, k,
                                               _addr(sums)), "hs_checksum_rows")

    def append(self, kv, positions, stream=None) -> None:
        """Decode-time append: kv uint8 [R, E] and positions int32 [R] (device; negative =
        no new entry) into the host store (and resident slots)."""
        self._check(self._lib.hs_append(self._h, _stream(stream), _addr(kv), _addr(positions),
                                        positions.shape[0]), "hs_append")

    def attend_workspace(self, B: int, H: int, k: int) -> int:
        """Bytes of device scratch hs_attend needs for (B, H, k)."""
        n = ctypes.c_size_t(0)
        self._check(self._lib.hs_attend_workspace(self._h, B, H, k, ctypes.byref(n)), "hs_attend_workspace")
        return int(n.value)

    def attend(self, q, out_slots, o, lse, sm_scale: float, workspace=None, stream=None) -> None:
        """Sparse attention over the resolved slots: q bf16 [R, H, 576], out_slots int32
        [R, k], o float32 [R, H, 512] and lse float32 [R, H] (device); workspace: a device
        buffer of attend_workspace() bytes (None when that is 0)."""
        B, H, _ = q.shape
        k = out_slots.shape[1]
        ws, nbytes = (None, 0) if workspace is None else (_addr(workspace), workspace.numel() * workspace.element_size())
        self._check(self._lib.hs_attend(self._h, _stream(stream), _addr(q), B, H, _addr(out_slots), k,
                                        float(sm_scale), _addr(o), _addr(lse), ws, nbytes), "hs_attend")

    def reset(self, stream=None) -> None:
        self._check(self._lib.hs_reset(self._h, _stream(stream)), "hs_reset")

    def set_flags(self, flags: int) -> None:
        self._check(self._lib.hs_set_flags(self._h, flags), "hs_set_flags")

    def set_policy(self, policy: int, seed: int = 0) -> None:
        """Replacement policy (POLICY_LRU / POLICY_FIFO / POLICY_RANDOM) of later calls."""
        self._check(self._lib.hs_set_policy(self._h, policy, seed & (2**64 - 1)), "hs_set_policy")

    def set_wait_limit(self, ns: int) -> None:
        """Time limit (global-timer ns from a CTA's start) of the kernels' device waits."""
        self._check(self._lib.hs_set_wait_limit(self._h, int(ns)), "hs_set_wait_limit")

    def kernels_per_call(self) -> int:
        return int(self._lib.hs_kernels_per_call(self._h))

    def status(self) -> int:
        bits = ctypes.c_uint32(0)
        self._check(self._lib.hs_get_status(self._h, ctypes.byref(bits)), "hs_get_status")
        return int(bits.value)

    def clear_status(self) -> None:
        self._check(self._lib.hs_clear_status(self._h), "hs_clear_status")

    # ------------------------------------------------------------------ views
    def host_kv(self) -> np.ndarray:
        """The pinned host store as a writable numpy view [R, C, host_stride] (uint8), or
        [pool_rows, host_stride] for a pooled context."""
        rows = self.pool_rows if self.pool_rows else self.R * self.C
        buf = (ctypes.c_uint8 * (rows * self.host_stride)).from_address(self._lib.hs_host_kv(self._h))
        a = np.frombuffer(buf, dtype=np.uint8)
        return a.reshape(rows, self.host_stride) if self.pool_rows else a.reshape(self.R, self.C, self.host_stride)

    def set_extents(self, base, length, stream=None) -> None:
        """Pooled context: request b's history is rows base[b] .. base[b] + length[b] - 1 of
        the pool; a request whose extent changes starts empty."""
        b = np.ascontiguousarray(base, dtype=np.int64)
        n = np.ascontiguousarray(length, dtype=np.int32)
        self._check(self._lib.hs_set_extents(self._h, _stream(stream), b.ctypes.data, n.ctypes.data),
                    "hs_set_extents")

    def host_kv_address(self) -> int:
        return int(self._lib.hs_host_kv(self._h))

    def _dev(self, fn: str, shape, typestr: str):
        import torch
        return torch.as_tensor(_DeviceArray(getattr(self._lib, fn)(self._h), shape, typestr, self),
                               device="cuda")

    def device_kv(self):
        return self._dev("hs_device_kv", (self.R, self.S, self.E), "|u1")

    def page_table(self):
        return self._dev("hs_page_table", (self.R, self.C), "<i4")

    def slot_token(self):
        return self._dev("hs_slot_token", (self.R, self.S), "<i4")

    def last_use(self):
        return self._dev("hs_last_use", (self.R, self.S), "<i4")

    def step(self):
        return self._dev("hs_step", (self.R,), "<i4")
