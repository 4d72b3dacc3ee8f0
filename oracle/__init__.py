"""CPU oracle for HiSparse's fused per-layer swap-in resolution (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package. It shares nothing with the CUDA path: the arithmetic lives in
``hs_oracle.c`` (plain, single-threaded C, compiled here with gcc); this module only
marshals numpy arrays to it.

Reading of the method (HiSparse paper abstract: hit detection, LRU replacement and
host-to-device fetches resolve each layer's selections; blog commentary, section
two: a hit is used in place, a miss is swapped in and an LRU victim is evicted; section
three: the page table is updated in the same step) and of the points the pages leave
open (recency stamps, tie-break, pairing, padding, range errors, duplicates) is
written out at the top of ``hs_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "hs_oracle.c")
LIB = os.path.join(_HERE, "libhs_oracle.so")

ERR_RANGE = 1
ERR_DUP = 2
POLICY_LRU, POLICY_FIFO, POLICY_RANDOM = 0, 1, 2


def compile_oracle(src: str, out: str) -> str:
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra",
                           "-o", out, src])
    return out


def build(force: bool = False) -> str:
    """Compile hs_oracle.c into libhs_oracle.so next to it; returns the path."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        compile_oracle(SRC, tmp)
        os.replace(tmp, LIB)
    return LIB


_libs: dict[str, ctypes.CDLL] = {}


def load(path: str | None = None) -> ctypes.CDLL:
    path = build() if path is None else path
    lib = _libs.get(path)
    if lib is None:
        lib = ctypes.CDLL(path)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lib.orc_create.argtypes = [i32, i32, i32, i32]
        lib.orc_create.restype = vp
        lib.orc_destroy.argtypes = [vp]
        lib.orc_destroy.restype = None
        for name in ("orc_pt", "orc_tok", "orc_lu", "orc_t", "orc_dev"):
            getattr(lib, name).argtypes = [vp]
            getattr(lib, name).restype = vp
        lib.orc_resolve_request.argtypes = [vp, i32, vp, sz, vp, i32, vp, vp]
        lib.orc_resolve_request.restype = i32
        lib.orc_resolve.argtypes = [vp, vp, sz, vp, i32, i32, vp, vp]
        lib.orc_resolve.restype = i32
        lib.orc_append.argtypes = [vp, i32, vp, sz, i32, vp]
        lib.orc_append.restype = i32
        u64 = ctypes.c_uint64
        lib.orc_set_policy.argtypes = [vp, i32, u64]
        lib.orc_set_policy.restype = i32
        lib.orc_set_request_id.argtypes = [vp, i32, i32]
        lib.orc_set_request_id.restype = i32
        lib.orc_splitmix64.argtypes = [u64, u64]
        lib.orc_splitmix64.restype = u64
        lib.orc_random_key.argtypes = [u64, i32, i32, i32]
        lib.orc_random_key.restype = ctypes.c_uint32
        lib.orc_set_len.argtypes = [vp, i32, i32]
        lib.orc_set_len.restype = i32
        lib.orc_reset_request.argtypes = [vp, i32]
        lib.orc_reset_request.restype = i32
        f64 = ctypes.c_double
        lib.orc_e4m3.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3.restype = f64
        lib.orc_bf16.argtypes = [ctypes.c_uint16]
        lib.orc_bf16.restype = f64
        lib.orc_attend.argtypes = [vp, i32, vp, i32, vp, i32, f64, vp, vp, vp]
        lib.orc_attend.restype = i32
        _libs[path] = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def splitmix64(x: int, n: int) -> int:
    """SplitMix64 output number n of the generator seeded with x (the oracle's C)."""
    return int(load().orc_splitmix64(x & (2**64 - 1), n & (2**64 - 1)))


def e4m3(code: int) -> float:
    """Value of an OCP E4M3 code (the oracle's C)."""
    return float(load().orc_e4m3(code))


def random_key(seed: int, b: int, t: int, s: int) -> int:
    """The RANDOM policy's key of slot s at call t of request b (the oracle's C)."""
    return int(load().orc_random_key(seed & (2**64 - 1), b, t, s))


class Oracle:
    """State of R requests x (C positions, S slots, E-byte entries) for one layer."""

    def __init__(self, R: int, C: int, S: int, E: int, lib_path: str | None = None):
        self.R, self.C, self.S, self.E = R, C, S, E
        self._lib = load(lib_path)
        self._h = self._lib.orc_create(R, C, S, E)
        if not self._h:
            raise MemoryError("orc_create failed")

    def set_policy(self, policy: int, seed: int = 0) -> None:
        """Replacement policy (POLICY_LRU / FIFO / RANDOM) for the calls that follow."""
        if self._lib.orc_set_policy(self._h, policy, seed & (2**64 - 1)) != 0:
            raise ValueError(f"orc_set_policy({policy}) refused")

    def set_request_ids(self, ids) -> None:
        """Row b of this state stands for request ids[b] (RANDOM draws depend on it)."""
        for b, i in enumerate(ids):
            if self._lib.orc_set_request_id(self._h, b, int(i)) != 0:
                raise ValueError("orc_set_request_id refused")

    def set_len(self, b: int, n: int) -> None:
        """Request b has positions [0, n) only (a shared pool's extent length)."""
        if self._lib.orc_set_len(self._h, b, n) != 0:
            raise ValueError("orc_set_len refused")

    def reset_request(self, b: int) -> None:
        """A new request takes over row b: its state starts empty."""
        if self._lib.orc_reset_request(self._h, b) != 0:
            raise ValueError("orc_reset_request refused")

    def close(self) -> None:
        if self._h:
            self._lib.orc_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def _view(self, fn: str, dtype, shape) -> np.ndarray:
        addr = getattr(self._lib, fn)(self._h)
        n = int(np.prod(shape)) * np.dtype(dtype).itemsize
        buf = (ctypes.c_uint8 * n).from_address(addr)
        return np.frombuffer(buf, dtype=dtype).reshape(shape).copy()

    @property
    def pt(self) -> np.ndarray:
        return self._view("orc_pt", np.int32, (self.R, self.C))

    @property
    def tok(self) -> np.ndarray:
        return self._view("orc_tok", np.int32, (self.R, self.S))

    @property
    def lu(self) -> np.ndarray:
        return self._view("orc_lu", np.int32, (self.R, self.S))

    @property
    def t(self) -> np.ndarray:
        return self._view("orc_t", np.int32, (self.R,))

    @property
    def dev(self) -> np.ndarray:
        return self._view("orc_dev", np.uint8, (self.R, self.S, self.E))

    def dev_rows(self, b: int) -> np.ndarray:
        """Device-slot contents of request b only, [S][E]."""
        addr = self._lib.orc_dev(self._h) + b * self.S * self.E
        n = self.S * self.E
        buf = (ctypes.c_uint8 * n).from_address(addr)
        return np.frombuffer(buf, dtype=np.uint8).reshape(self.S, self.E).copy()

    def resolve(self, host, host_stride: int, sel: np.ndarray):
        """One layer-step for all R requests.

        host: a uint8 array [R][C][>=E] or an integer address of such a buffer (rows
        host_stride bytes apart); sel: int32 [R][k]. Returns (out_slots, miss_counts, status).
        """
        sel = np.ascontiguousarray(sel, dtype=np.int32)
        B, k = sel.shape
        out = np.empty((B, k), dtype=np.int32)
        miss = np.empty(B, dtype=np.int32)
        haddr = host if isinstance(host, int) else _ptr(host)
        rc = self._lib.orc_resolve(self._h, haddr, host_stride, _ptr(sel), B, k, _ptr(out),
                                   _ptr(miss))
        if rc < 0:
            raise ValueError(f"orc_resolve failed ({rc})")
        return out, miss, rc

    def resolve_request(self, b: int, host_b, host_stride: int, sel_b: np.ndarray):
        """One layer-step for request b alone (host_b: its row 0, array or address)."""
        sel_b = np.ascontiguousarray(sel_b, dtype=np.int32)
        k = sel_b.shape[0]
        out = np.empty(k, dtype=np.int32)
        miss = np.empty(1, dtype=np.int32)
        haddr = host_b if isinstance(host_b, int) else _ptr(host_b)
        rc = self._lib.orc_resolve_request(self._h, b, haddr, host_stride, _ptr(sel_b), k,
                                           _ptr(out), _ptr(miss))
        if rc < 0:
            raise ValueError(f"orc_resolve_request failed ({rc})")
        return out, int(miss[0]), rc

    def attend(self, b: int, q: np.ndarray, out_slots_b: np.ndarray, sm_scale: float):
        """Sparse attention of request b over the slots out_slots_b [k] (negative = not
        valid), q [H][576] as uint16 bf16 bit patterns. Returns (o [H][512], lse [H],
        absw [H][512]) in float64."""
        q = np.ascontiguousarray(q, dtype=np.uint16)
        sl = np.ascontiguousarray(out_slots_b, dtype=np.int32)
        H, k = q.shape[0], sl.shape[0]
        out = np.empty((H, 512))
        lse = np.empty(H)
        absw = np.empty((H, 512))
        rc = self._lib.orc_attend(self._h, b, _ptr(q), H, _ptr(sl), k, float(sm_scale), _ptr(out),
                                  _ptr(lse), _ptr(absw))
        if rc < 0:
            raise ValueError(f"orc_attend failed ({rc})")
        return out, lse, absw

    def append_request(self, b: int, host_b, host_stride: int, p: int, row: np.ndarray) -> int:
        """Decode-time append for request b alone: host_b is its history's row 0 (address or
        array); returns the status word."""
        row = np.ascontiguousarray(row, dtype=np.uint8)
        haddr = host_b if isinstance(host_b, int) else host_b.ctypes.data
        rc = self._lib.orc_append(self._h, b, haddr, host_stride, int(p), row.ctypes.data)
        if rc < 0:
            raise ValueError(f"orc_append failed ({rc})")
        return rc

    def append(self, host: np.ndarray, positions, rows: np.ndarray) -> int:
        """Decode-time append for all R requests: host [R][C][stride] (written), positions
        [R] (negative = none), rows [R][E]. Returns the OR of the status words."""
        rows = np.ascontiguousarray(rows, dtype=np.uint8)
        st = 0
        for b in range(self.R):
            hb = host[b]
            rc = self._lib.orc_append(self._h, b, hb.ctypes.data, host.shape[2], int(positions[b]),
                                      rows[b].ctypes.data)
            if rc < 0:
                raise ValueError(f"orc_append failed ({rc})")
            st |= rc
        return st
