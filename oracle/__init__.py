"""CPU oracle for the rank-sum reduce hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never links,
loads or calls it, and the two share no code: the oracle is plain,
single-threaded C (``oracle.c``) written from the pages' definitions, loaded
here with ctypes.

Arrays are passed as host buffers: numpy arrays, or CPU torch tensors (bf16
data is handled as its raw 16-bit storage).  Element types: "bf16", "fp16",
"fp32".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liboracle.so")
SRC_PATH = os.path.join(_HERE, "oracle.c")

DTYPE_CODE = {"bf16": 0, "fp16": 1, "fp32": 2}
ELEM_SIZE = {"bf16": 2, "fp16": 2, "fp32": 4}

_lock = threading.Lock()


def build(force: bool = False, src: str = SRC_PATH, out: str = LIB_PATH) -> str:
    """Compile an oracle source into a shared library with gcc (no fast-math,
    no FMA contraction).  The defaults build the oracle itself."""
    hdr = os.path.join(_HERE, "oracle.h")
    if force or not os.path.exists(out) or os.path.getmtime(out) < max(os.path.getmtime(src), os.path.getmtime(hdr)):
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-Wall", "-Wextra", "-I", _HERE, "-o", tmp, src, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def _bind(lib):
    i64, u16, u32, u64 = ctypes.c_int64, ctypes.c_uint16, ctypes.c_uint32, ctypes.c_uint64
    vp, pvp = ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)
    sig = {
        "orc_bf16_to_f32": (ctypes.c_float, [u16]),
        "orc_f16_to_f32": (ctypes.c_float, [u16]),
        "orc_f32_to_bf16": (u16, [ctypes.c_float]),
        "orc_f32_to_f16": (u16, [ctypes.c_float]),
        "orc_f64_to_bf16": (u16, [ctypes.c_double]),
        "orc_f64_to_f16": (u16, [ctypes.c_double]),
        "orc_f64_to_f32": (ctypes.c_float, [ctypes.c_double]),
        "orc_elem_size": (ctypes.c_int, [ctypes.c_int]),
        "orc_convert": (None, [vp, ctypes.c_int, vp, ctypes.c_int, i64]),
        "orc_reduce": (None, [ctypes.c_int, pvp, ctypes.c_int, i64, vp]),
        "orc_reduce_two_shot": (None, [ctypes.c_int, pvp, ctypes.c_int, i64, vp]),
        "orc_reduce_residual_rmsnorm": (None, [ctypes.c_int, pvp, vp, vp, ctypes.c_float, i64, i64,
                                               ctypes.c_int, vp, vp, vp, vp]),
        "orc_ll128_lines": (i64, [i64]),
        "orc_ll128_wire_bytes": (i64, [i64]),
        "orc_ll128_data_capacity": (i64, [i64]),
        "orc_ll128_encode": (None, [vp, i64, u64, vp]),
        "orc_ll128_decode_reduce": (i64, [ctypes.c_int, pvp, i64, ctypes.c_int, u64, vp, vp, i64]),
        "orc_ll_lines": (i64, [i64]),
        "orc_ll_wire_bytes": (i64, [i64]),
        "orc_ll_data_capacity": (i64, [i64]),
        "orc_ll_encode": (None, [vp, i64, u32, vp]),
        "orc_ll_decode_reduce": (i64, [ctypes.c_int, pvp, i64, ctypes.c_int, u32, vp, vp, i64]),
        "orc_lamport_fill": (None, [vp, i64]),
        "orc_lamport_push": (None, [vp, i64, vp]),
        "orc_lamport_reduce_residual_rmsnorm": (i64, [ctypes.c_int, vp, u64, i64, i64, vp, vp, ctypes.c_float,
                                                      vp, vp, vp, vp, i64]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


# --------------------------------------------------------------------------
# host-buffer marshalling
# --------------------------------------------------------------------------
def _as_host_array(a) -> np.ndarray:
    """Contiguous numpy view of a host buffer (numpy array or CPU torch tensor)."""
    if isinstance(a, np.ndarray):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("oracle needs C-contiguous host arrays")
        return a
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(a, torch.Tensor):
        if a.device.type != "cpu":
            raise ValueError("oracle takes host buffers only")
        if not a.is_contiguous():
            raise ValueError("oracle needs contiguous tensors")
        if a.dtype in (torch.bfloat16, torch.float16):
            return a.view(torch.int16).numpy()
        return a.numpy()
    raise TypeError(f"unsupported host buffer type {type(a)!r}")


def _ptr(a) -> int:
    return _as_host_array(a).ctypes.data


def _ptr_table(arrs):
    arr = (ctypes.c_void_p * len(arrs))(*[_ptr(a) for a in arrs])
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)), arr


def _nbytes(a) -> int:
    return _as_host_array(a).nbytes


KIND_CODE = {"bf16": 0, "fp16": 1, "fp32": 2, "fp64": 3}
_KIND_NP = {"bf16": np.uint16, "fp16": np.uint16, "fp32": np.float32, "fp64": np.float64}
class Oracle:
    """The oracle's operations, bound to one compiled oracle library."""

    def __init__(self, lib_path: str | None = None):
        if lib_path is None:
            lib_path = build()
        self.lib_path = lib_path
        self._lib = _bind(ctypes.CDLL(lib_path))

    def lib(self):
        """The loaded ctypes library."""
        return self._lib

    # --------------------------------------------------------------------------
    # the path's operations
    # --------------------------------------------------------------------------
    def reduce(self, xs, dtype: str, out) -> None:
        """ar = rne(sum_r x_r) elementwise, fp32 adds in rank order (see oracle.c)."""
        es = ELEM_SIZE[dtype]
        n = _nbytes(xs[0]) // es
        for a in list(xs) + [out]:
            if _nbytes(a) < n * es:
                raise ValueError("buffer too small")
        tbl, keep = _ptr_table(xs)
        self._lib.orc_reduce(len(xs), tbl, DTYPE_CODE[dtype], n, _ptr(out))
        del keep


    def reduce_two_shot(self, xs, dtype: str, out) -> None:
        """Two-shot bit pattern: each shard summed in its owner's rotated rank order."""
        es = ELEM_SIZE[dtype]
        n = _nbytes(xs[0]) // es
        if (n * es) % 16:
            raise ValueError("message bytes must be a multiple of 16")
        for a in list(xs) + [out]:
            if _nbytes(a) < n * es:
                raise ValueError("buffer too small")
        tbl, keep = _ptr_table(xs)
        self._lib.orc_reduce_two_shot(len(xs), tbl, DTYPE_CODE[dtype], n, _ptr(out))
        del keep


    def reduce_residual_rmsnorm(self, xs, residual, weight, eps: float, M: int, N: int, dtype: str,
                                residual_out, norm_out, ar_out=None, norm_f64=None) -> None:
        """Fused rank sum + residual add + RMSNorm over a row-major [M, N] problem."""
        es = ELEM_SIZE[dtype]
        need = M * N * es
        for a in list(xs) + [residual, residual_out, norm_out] + ([ar_out] if ar_out is not None else []):
            if _nbytes(a) < need:
                raise ValueError("buffer too small")
        if _nbytes(weight) < N * es:
            raise ValueError("weight too small")
        if norm_f64 is not None and (norm_f64.dtype != np.float64 or norm_f64.size < M * N):
            raise ValueError("norm_f64 must hold M*N float64")
        tbl, keep = _ptr_table(xs)
        self._lib.orc_reduce_residual_rmsnorm(
            len(xs), tbl, _ptr(residual), _ptr(weight), ctypes.c_float(eps), M, N, DTYPE_CODE[dtype],
            _ptr(ar_out) if ar_out is not None else None, _ptr(residual_out), _ptr(norm_out),
            norm_f64.ctypes.data if norm_f64 is not None else None)
        del keep


    def ll128_lines(self, data_bytes: int) -> int:
        return int(self._lib.orc_ll128_lines(data_bytes))


    def ll128_wire_bytes(self, data_bytes: int) -> int:
        return int(self._lib.orc_ll128_wire_bytes(data_bytes))


    def ll128_data_capacity(self, wire_bytes: int) -> int:
        return int(self._lib.orc_ll128_data_capacity(wire_bytes))


    def ll128_encode(self, data, data_bytes: int, flag: int, wire) -> None:
        if _nbytes(data) < data_bytes or _nbytes(wire) < self.ll128_wire_bytes(data_bytes):
            raise ValueError("buffer too small")
        self._lib.orc_ll128_encode(_ptr(data), data_bytes, flag, _ptr(wire))


    def _decode(self, fn, wires, data_bytes, dtype, flag, out, cap):
        stale = np.zeros((max(cap, 1), 2), dtype=np.uint32)
        tbl, keep = _ptr_table(wires)
        n = fn(len(wires), tbl, data_bytes, DTYPE_CODE[dtype], flag, _ptr(out), stale.ctypes.data, cap)
        del keep
        return int(n), stale[: min(int(n), cap)]


    def ll128_decode_reduce(self, wires, data_bytes: int, dtype: str, expected_flag: int, out, cap: int = 1 << 20):
        """Returns (n_stale, stale[k] = (rank, line)) in line-major order."""
        for w in wires:
            if _nbytes(w) < self.ll128_wire_bytes(data_bytes):
                raise ValueError("wire buffer too small")
        if _nbytes(out) < data_bytes:
            raise ValueError("output too small")
        return self._decode(self._lib.orc_ll128_decode_reduce, wires, data_bytes, dtype, expected_flag, out, cap)


    def ll_lines(self, data_bytes: int) -> int:
        return int(self._lib.orc_ll_lines(data_bytes))


    def ll_wire_bytes(self, data_bytes: int) -> int:
        return int(self._lib.orc_ll_wire_bytes(data_bytes))


    def ll_data_capacity(self, wire_bytes: int) -> int:
        return int(self._lib.orc_ll_data_capacity(wire_bytes))


    def ll_encode(self, data, data_bytes: int, flag: int, wire) -> None:
        if _nbytes(data) < data_bytes or _nbytes(wire) < self.ll_wire_bytes(data_bytes):
            raise ValueError("buffer too small")
        self._lib.orc_ll_encode(_ptr(data), data_bytes, flag, _ptr(wire))


    def ll_decode_reduce(self, wires, data_bytes: int, dtype: str, expected_flag: int, out, cap: int = 1 << 20):
        for w in wires:
            if _nbytes(w) < self.ll_wire_bytes(data_bytes):
                raise ValueError("wire buffer too small")
        if _nbytes(out) < data_bytes:
            raise ValueError("output too small")
        return self._decode(self._lib.orc_ll_decode_reduce, wires, data_bytes, dtype, expected_flag, out, cap)

    # Lamport one-shot push (bf16)
    LAMPORT_SENTINEL = 0x80008000

    def lamport_buffer_bytes(self, W: int, n: int) -> int:
        return 3 * W * n * 2

    def lamport_fill(self, words) -> None:
        self._lib.orc_lamport_fill(_ptr(words), _nbytes(words) // 4)

    def lamport_push(self, data, n: int, buffer, W: int, rank: int, round_: int) -> None:
        """Push rank's n bf16 values into its slot of region round % 3."""
        if _nbytes(buffer) < self.lamport_buffer_bytes(W, n) or _nbytes(data) < 2 * n:
            raise ValueError("buffer too small")
        off = ((round_ % 3) * W + rank) * n * 2
        self._lib.orc_lamport_push(_ptr(data), n, _ptr(buffer) + off)

    def lamport_reduce_residual_rmsnorm(self, W: int, buffer, round_: int, M: int, N: int, residual, weight,
                                        eps: float, residual_out, norm_out, ar_out=None, cap: int = 1 << 16):
        """Returns (n_stale, stale[k] = (rank, row))."""
        if _nbytes(buffer) < self.lamport_buffer_bytes(W, M * N):
            raise ValueError("buffer too small")
        stale = np.zeros((max(cap, 1), 2), dtype=np.uint32)
        n = self._lib.orc_lamport_reduce_residual_rmsnorm(
            W, _ptr(buffer), round_, M, N, _ptr(residual), _ptr(weight), ctypes.c_float(eps),
            _ptr(ar_out) if ar_out is not None else None, _ptr(residual_out), _ptr(norm_out), stale.ctypes.data, cap)
        return int(n), stale[: min(int(n), cap)]

    # conversions (used by the pins)
    def convert(self, src: np.ndarray, src_kind: str, dst_kind: str) -> np.ndarray:
        """Array conversion between bf16/fp16 (raw uint16 bits), fp32 and fp64."""
        src = np.ascontiguousarray(src)
        if src.dtype.itemsize != np.dtype(_KIND_NP[src_kind]).itemsize:
            raise ValueError("source itemsize does not match its kind")
        out = np.empty(src.shape, dtype=_KIND_NP[dst_kind])
        self._lib.orc_convert(src.ctypes.data, KIND_CODE[src_kind], out.ctypes.data, KIND_CODE[dst_kind], src.size)
        return out


    def f32_to_bf16(self, x: float) -> int:
        return int(self._lib.orc_f32_to_bf16(x))


    def f32_to_f16(self, x: float) -> int:
        return int(self._lib.orc_f32_to_f16(x))


    def f64_to_bf16(self, x: float) -> int:
        return int(self._lib.orc_f64_to_bf16(x))


    def f64_to_f16(self, x: float) -> int:
        return int(self._lib.orc_f64_to_f16(x))


    def f64_to_f32(self, x: float) -> float:
        return float(self._lib.orc_f64_to_f32(x))


    def bf16_to_f32(self, b: int) -> float:
        return float(self._lib.orc_bf16_to_f32(b))


    def f16_to_f32(self, h: int) -> float:
        return float(self._lib.orc_f16_to_f32(h))


_default = None


def default() -> "Oracle":
    """The oracle built from oracle.c (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle()
        return _default


def __getattr__(name):
    # module-level access to the default oracle's operations: oracle.reduce(...), ...
    if name.startswith("_"):
        raise AttributeError(name)
    return getattr(default(), name)
