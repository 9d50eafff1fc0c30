"""Python binding of libcar (include/car.h): argument marshalling only.

Every ``car_*`` function here has the name and arguments of the C entry point
and returns its status code; all work runs in libcar's CUDA kernels.  Device
buffers are passed as integer addresses (``tensor.data_ptr()``), streams as
integer handles (``torch.cuda.current_stream().cuda_stream``).

``Car`` is a small convenience wrapper over the same calls for torch tensors.
There is no CPU fallback: importing the binding without a built libcar.so
raises ImportError.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcar.so")

CAR_BF16, CAR_FP16, CAR_FP32 = 0, 1, 2
CAR_OK, CAR_ERR_ARG, CAR_ERR_ALIGN, CAR_ERR_SIZE, CAR_ERR_CUDA, CAR_ERR_STALE_FLAG, CAR_ERR_HANDLE, CAR_ERR_TIMEOUT = \
    range(8)
CAR_FUSED_AUTO, CAR_FUSED_ROWS, CAR_FUSED_PIPELINE = 0, 1, 2
CAR_STALE_LIST_MAX = 65536
CAR_MAX_ROW_BYTES = 64 * 1024
DTYPE_CODE = {"bf16": CAR_BF16, "fp16": CAR_FP16, "fp32": CAR_FP32}
ELEM_SIZE = {"bf16": 2, "fp16": 2, "fp32": 4}
STATUS_NAME = {CAR_OK: "CAR_OK", CAR_ERR_ARG: "CAR_ERR_ARG", CAR_ERR_ALIGN: "CAR_ERR_ALIGN",
               CAR_ERR_SIZE: "CAR_ERR_SIZE", CAR_ERR_CUDA: "CAR_ERR_CUDA",
               CAR_ERR_STALE_FLAG: "CAR_ERR_STALE_FLAG", CAR_ERR_HANDLE: "CAR_ERR_HANDLE",
               CAR_ERR_TIMEOUT: "CAR_ERR_TIMEOUT"}


class car_stale_report(ctypes.Structure):
    _fields_ = [("n_stale", ctypes.c_uint64), ("n_listed", ctypes.c_uint32), ("cap", ctypes.c_uint32),
                ("entries", ctypes.POINTER(ctypes.c_uint32 * 2))]


if not os.path.exists(LIB_PATH):
    raise ImportError(f"libcar.so is not built ({LIB_PATH}); run `python -c 'import __graft_entry__ as g; "
                      "g.build()'` or `python rank_sum_reduce_gb300/build.py`")

_lib = ctypes.CDLL(LIB_PATH)

_vp = ctypes.c_void_p
_pvp = ctypes.POINTER(ctypes.c_void_p)
_ctx_pp = ctypes.POINTER(ctypes.c_void_p)
_SIGS = {
    "car_create": (ctypes.c_int, [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, _ctx_pp]),
    "car_destroy": (ctypes.c_int, [_vp]),
    "car_reduce": (ctypes.c_int, [_vp, _pvp, _vp, _vp]),
    "car_reduce_two_shot": (ctypes.c_int, [_vp, _pvp, _vp, _vp]),
    "car_reduce_residual_rmsnorm": (ctypes.c_int, [_vp, _pvp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _vp]),
    "car_ll128_wire_bytes": (ctypes.c_size_t, [_vp]),
    "car_ll128_encode": (ctypes.c_int, [_vp, _vp, ctypes.c_uint64, _vp, _vp]),
    "car_ll128_decode_reduce": (ctypes.c_int, [_vp, _pvp, ctypes.c_uint64, ctypes.c_int, _vp, _vp]),
    "car_ll128_report": (ctypes.c_int, [_vp, ctypes.POINTER(car_stale_report)]),
    "car_ll_wire_bytes": (ctypes.c_size_t, [_vp]),
    "car_ll_encode": (ctypes.c_int, [_vp, _vp, ctypes.c_uint32, _vp, _vp]),
    "car_ll_decode_reduce": (ctypes.c_int, [_vp, _pvp, ctypes.c_uint32, ctypes.c_int, _vp, _vp]),
    "car_ll_report": (ctypes.c_int, [_vp, ctypes.POINTER(car_stale_report)]),
    "car_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "car_last_error": (ctypes.c_char_p, []),
    "car_tune_fused": (ctypes.c_int, [_vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "car_sync": (ctypes.c_int, [_vp, _vp]),
    "car_test_delay_partial": (ctypes.c_int, [_vp, ctypes.c_uint64, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64]),
    "car_lamport_buffer_bytes": (ctypes.c_size_t, [_vp]),
    "car_lamport_init": (ctypes.c_int, [_vp, _vp, _vp]),
    "car_lamport_push": (ctypes.c_int, [_vp, _vp, ctypes.c_int, ctypes.c_uint64, _vp, _vp]),
    "car_lamport_reduce_residual_rmsnorm": (ctypes.c_int, [_vp, _vp, ctypes.c_uint64, ctypes.c_int, _vp, _vp,
                                                           ctypes.c_float, _vp, _vp, _vp, _vp]),
    "car_lamport_report": (ctypes.c_int, [_vp, ctypes.POINTER(car_stale_report)]),
    "car_ll128_decode_reduce_noalloc": (ctypes.c_int, [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                                       _pvp, ctypes.c_uint64, ctypes.c_int, _vp, _vp,
                                                       ctypes.c_uint32, _vp]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

EXPORTED = tuple(_SIGS)


def lib():
    return _lib


def _table(ptrs):
    arr = (ctypes.c_void_p * len(ptrs))(*[int(p) for p in ptrs])
    return arr


# ---------------------------------------------------------------------------
# 1:1 wrappers of the C entry points
# ---------------------------------------------------------------------------
def car_create(W: int, M: int, N: int, dtype: int):
    """Returns (status, handle); handle is an int address or None."""
    out = ctypes.c_void_p()
    st = _lib.car_create(W, M, N, dtype, ctypes.byref(out))
    return st, out.value


def car_destroy(h) -> int:
    return _lib.car_destroy(h)


def car_reduce(h, inputs, ar_out: int, stream: int = 0) -> int:
    return _lib.car_reduce(h, _table(inputs) if inputs is not None else None, ar_out, stream)


def car_reduce_two_shot(h, inputs, ar_out: int, stream: int = 0) -> int:
    return _lib.car_reduce_two_shot(h, _table(inputs) if inputs is not None else None, ar_out, stream)


def car_reduce_residual_rmsnorm(h, inputs, residual: int, weight: int, eps: float, residual_out: int,
                                norm_out: int, ar_out: int | None, stream: int = 0) -> int:
    return _lib.car_reduce_residual_rmsnorm(h, _table(inputs) if inputs is not None else None, residual, weight,
                                            eps, residual_out, norm_out, ar_out, stream)


def car_ll128_wire_bytes(h) -> int:
    return int(_lib.car_ll128_wire_bytes(h))


def car_ll128_encode(h, data: int, flag: int, wire: int, stream: int = 0) -> int:
    return _lib.car_ll128_encode(h, data, flag, wire, stream)


def car_ll128_decode_reduce(h, wires, expected_flag: int, max_polls: int, ar_out: int, stream: int = 0) -> int:
    return _lib.car_ll128_decode_reduce(h, _table(wires) if wires is not None else None, expected_flag, max_polls,
                                        ar_out, stream)


def _report(fn, h, cap: int):
    entries = (ctypes.c_uint32 * 2 * max(cap, 1))()
    rep = car_stale_report(0, 0, cap, ctypes.cast(entries, ctypes.POINTER(ctypes.c_uint32 * 2)))
    st = fn(h, ctypes.byref(rep))
    pairs = [(entries[i][0], entries[i][1]) for i in range(rep.n_listed)]
    return st, int(rep.n_stale), pairs


def car_ll128_report(h, cap: int = CAR_STALE_LIST_MAX):
    """Returns (status, n_stale, [(rank, line), ...])."""
    return _report(_lib.car_ll128_report, h, cap)


def car_ll128_decode_reduce_noalloc(W: int, M: int, N: int, dtype: int, wires, expected_flag: int, max_polls: int,
                                    ar_out: int, stale_out: int, cap: int, stream: int = 0) -> int:
    """Handle-free LL128 decode-reduce that allocates nothing (see car.h):
    stale_out is a device buffer of 16 + 8*cap bytes."""
    return _lib.car_ll128_decode_reduce_noalloc(W, M, N, dtype, _table(wires) if wires is not None else None,
                                                expected_flag, max_polls, ar_out, stale_out, cap, stream)


def car_ll_wire_bytes(h) -> int:
    return int(_lib.car_ll_wire_bytes(h))


def car_ll_encode(h, data: int, flag: int, wire: int, stream: int = 0) -> int:
    return _lib.car_ll_encode(h, data, flag, wire, stream)


def car_ll_decode_reduce(h, wires, expected_flag: int, max_polls: int, ar_out: int, stream: int = 0) -> int:
    return _lib.car_ll_decode_reduce(h, _table(wires) if wires is not None else None, expected_flag, max_polls,
                                     ar_out, stream)


def car_ll_report(h, cap: int = CAR_STALE_LIST_MAX):
    return _report(_lib.car_ll_report, h, cap)


def car_lamport_buffer_bytes(h) -> int:
    return int(_lib.car_lamport_buffer_bytes(h))


def car_lamport_init(h, comm: int, stream: int = 0) -> int:
    return _lib.car_lamport_init(h, comm, stream)


def car_lamport_push(h, data: int, rank: int, round_: int, comm: int, stream: int = 0) -> int:
    return _lib.car_lamport_push(h, data, rank, round_, comm, stream)


def car_lamport_reduce_residual_rmsnorm(h, comm: int, round_: int, max_polls: int, residual: int, weight: int,
                                        eps: float, residual_out: int, norm_out: int, ar_out: int | None,
                                        stream: int = 0) -> int:
    return _lib.car_lamport_reduce_residual_rmsnorm(h, comm, round_, max_polls, residual, weight, eps,
                                                    residual_out, norm_out, ar_out, stream)


def car_lamport_report(h, cap: int = CAR_STALE_LIST_MAX):
    return _report(_lib.car_lamport_report, h, cap)


def car_status_string(st: int) -> str:
    return _lib.car_status_string(st).decode()


def car_last_error() -> str:
    return _lib.car_last_error().decode()


def car_tune_fused(h, kernel: int, cluster: int, threads: int, vpt: int) -> int:
    return _lib.car_tune_fused(h, kernel, cluster, threads, vpt)


def car_sync(h, stream: int = 0) -> int:
    return _lib.car_sync(h, stream)


def car_test_delay_partial(h, wait_limit_ns: int, cta: int, row: int, delay_ns: int) -> int:
    return _lib.car_test_delay_partial(h, wait_limit_ns, cta, row, delay_ns)


# ---------------------------------------------------------------------------
# torch convenience layer (still only marshalling)
# ---------------------------------------------------------------------------
class CarError(RuntimeError):
    def __init__(self, status: int, what: str):
        detail = car_last_error() if status == CAR_ERR_CUDA else ""
        super().__init__(f"{what}: {STATUS_NAME.get(status, status)} {detail}".strip())
        self.status = status


def check(status: int, what: str = "car") -> None:
    if status != CAR_OK:
        raise CarError(status, what)


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _ptr(t, nbytes: int, what: str, device=None) -> int:
    """Device pointer of a tensor the library will read or write `nbytes` of:
    it must be a contiguous CUDA tensor at least that large, on `device` when
    given (any dtype: the library sees bytes)."""
    if not t.is_cuda:
        raise ValueError(f"{what}: expected a CUDA tensor")
    if device is not None and t.device.index != device:
        raise ValueError(f"{what}: on cuda:{t.device.index}, the handle is on cuda:{device}")
    if not t.is_contiguous():
        raise ValueError(f"{what}: expected a contiguous tensor")
    if t.numel() * t.element_size() < nbytes:
        raise ValueError(f"{what}: {t.numel() * t.element_size()} bytes, the call needs {nbytes}")
    return t.data_ptr()


class Car:
    """A libcar handle for W rank buffers of [M, N] elements of one dtype.

    The methods take torch tensors and pass their device pointers to the C
    ABI; each tensor must be a contiguous CUDA tensor of at least the bytes
    the call reads or writes (ValueError otherwise)."""

    def __init__(self, W: int, M: int, N: int, dtype: str):
        st, h = car_create(W, M, N, DTYPE_CODE[dtype])
        check(st, "car_create")
        self.h, self.W, self.M, self.N, self.dtype = h, W, M, N, dtype
        self.D = M * N * ELEM_SIZE[dtype]      # bytes per rank
        import torch

        self.device = torch.cuda.current_device()

    def _p(self, t, nbytes: int, what: str) -> int:
        return _ptr(t, nbytes, what, self.device)

    def _ranks(self, ts, nbytes: int, what: str):
        if len(ts) != self.W:
            raise ValueError(f"{what}: {len(ts)} tensors for W = {self.W}")
        return [self._p(t, nbytes, f"{what}[{r}]") for r, t in enumerate(ts)]

    def close(self):
        if self.h is not None:
            check(car_destroy(self.h), "car_destroy")
            self.h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def ll128_wire_bytes(self) -> int:
        return car_ll128_wire_bytes(self.h)

    @property
    def ll_wire_bytes(self) -> int:
        return car_ll_wire_bytes(self.h)

    def reduce(self, xs, ar_out, stream=None):
        check(car_reduce(self.h, self._ranks(xs, self.D, "inputs"), self._p(ar_out, self.D, "ar_out"), _stream(stream)),
              "car_reduce")

    def reduce_two_shot(self, xs, ar_out, stream=None):
        check(car_reduce_two_shot(self.h, self._ranks(xs, self.D, "inputs"), self._p(ar_out, self.D, "ar_out"),
                                  _stream(stream)), "car_reduce_two_shot")

    def reduce_residual_rmsnorm(self, xs, residual, weight, eps, residual_out, norm_out, ar_out=None, stream=None):
        D = self.D
        check(car_reduce_residual_rmsnorm(self.h, self._ranks(xs, D, "inputs"), self._p(residual, D, "residual"),
                                          self._p(weight, D // self.M, "weight"), eps,
                                          self._p(residual_out, D, "residual_out"), self._p(norm_out, D, "norm_out"),
                                          self._p(ar_out, D, "ar_out") if ar_out is not None else None,
                                          _stream(stream)), "car_reduce_residual_rmsnorm")

    def ll128_encode(self, data, flag, wire, stream=None):
        check(car_ll128_encode(self.h, self._p(data, self.D, "data"), flag, self._p(wire, self.ll128_wire_bytes, "wire"),
                               _stream(stream)), "car_ll128_encode")

    def ll128_decode_reduce(self, wires, expected_flag, ar_out, max_polls=1, stream=None):
        check(car_ll128_decode_reduce(self.h, self._ranks(wires, self.ll128_wire_bytes, "wires"), expected_flag,
                                      max_polls, self._p(ar_out, self.D, "ar_out"), _stream(stream)),
              "car_ll128_decode_reduce")

    def ll128_report(self, cap=CAR_STALE_LIST_MAX):
        st, n, pairs = car_ll128_report(self.h, cap)
        if st not in (CAR_OK, CAR_ERR_STALE_FLAG):
            check(st, "car_ll128_report")
        return n, pairs

    def ll_encode(self, data, flag, wire, stream=None):
        check(car_ll_encode(self.h, self._p(data, self.D, "data"), flag, self._p(wire, self.ll_wire_bytes, "wire"),
                            _stream(stream)), "car_ll_encode")

    def ll_decode_reduce(self, wires, expected_flag, ar_out, max_polls=1, stream=None):
        check(car_ll_decode_reduce(self.h, self._ranks(wires, self.ll_wire_bytes, "wires"), expected_flag,
                                   max_polls, self._p(ar_out, self.D, "ar_out"), _stream(stream)),
              "car_ll_decode_reduce")

    def ll_report(self, cap=CAR_STALE_LIST_MAX):
        st, n, pairs = car_ll_report(self.h, cap)
        if st not in (CAR_OK, CAR_ERR_STALE_FLAG):
            check(st, "car_ll_report")
        return n, pairs

    @property
    def lamport_buffer_bytes(self) -> int:
        return car_lamport_buffer_bytes(self.h)

    def lamport_init(self, comm, stream=None):
        check(car_lamport_init(self.h, self._p(comm, self.lamport_buffer_bytes, "comm"), _stream(stream)),
              "car_lamport_init")

    def lamport_push(self, data, rank, round_, comm, stream=None):
        check(car_lamport_push(self.h, self._p(data, self.D, "data"), rank, round_,
                               self._p(comm, self.lamport_buffer_bytes, "comm"), _stream(stream)), "car_lamport_push")

    def lamport_reduce_residual_rmsnorm(self, comm, round_, residual, weight, eps, residual_out, norm_out,
                                        ar_out=None, max_polls=1, stream=None):
        D = self.D
        check(car_lamport_reduce_residual_rmsnorm(self.h, self._p(comm, self.lamport_buffer_bytes, "comm"), round_,
                                                  max_polls, self._p(residual, D, "residual"),
                                                  self._p(weight, D // self.M, "weight"), eps,
                                                  self._p(residual_out, D, "residual_out"), self._p(norm_out, D, "norm_out"),
                                                  self._p(ar_out, D, "ar_out") if ar_out is not None else None,
                                                  _stream(stream)), "car_lamport_reduce_residual_rmsnorm")

    def lamport_report(self, cap=CAR_STALE_LIST_MAX):
        st, n, pairs = car_lamport_report(self.h, cap)
        if st not in (CAR_OK, CAR_ERR_STALE_FLAG):
            check(st, "car_lamport_report")
        return n, pairs

    def tune_fused(self, kernel=CAR_FUSED_AUTO, cluster=0, threads=0, vpt=0):
        check(car_tune_fused(self.h, kernel, cluster, threads, vpt), "car_tune_fused")

    def sync(self, stream=None):
        check(car_sync(self.h, _stream(stream)), "car_sync")
