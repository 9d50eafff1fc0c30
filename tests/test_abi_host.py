"""Host-side checks of the C ABI: the library loads, exports every entry point
that include/car.h declares, and rejects bad arguments before touching CUDA.
No test here launches a kernel."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "car.h")


@pytest.fixture(scope="module")
def car():
    import __graft_entry__

    __graft_entry__.build()
    import rank_sum_reduce_gb300 as car

    return car


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(car_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ["car_create", "car_destroy", "car_reduce", "car_reduce_residual_rmsnorm", "car_ll128_encode",
                 "car_ll128_decode_reduce", "car_ll128_report", "car_ll_encode", "car_ll_decode_reduce"]:
        assert must in names


def test_library_exports_every_declared_symbol(car):
    lib = ctypes.CDLL(car.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in car.h but not exported"
    assert set(declared_functions()) == set(car.EXPORTED)


def test_status_strings(car):
    for st in range(8):
        assert car.car_status_string(st).startswith(car.STATUS_NAME[st])
    assert "unknown" in car.car_status_string(99)


@pytest.mark.parametrize("W,M,N,dtype,want", [
    (0, 1, 64, 0, 1), (17, 1, 64, 0, 1), (2, 0, 64, 0, 1), (2, 1, 0, 0, 1), (2, 1, 64, 7, 1),
    (2, 1, 4, 0, 3),          # 8 bytes per row: not a multiple of 16
    (2, 1, 6, 2, 3),          # 24 bytes per row
    (2, 1, 2**40, 0, 3),      # N*s beyond the int32 vector index
    (2, 2**60, 8, 0, 3),      # message size overflow
])
def test_create_rejects_bad_shapes_without_cuda(car, W, M, N, dtype, want):
    st, h = car.car_create(W, M, N, dtype)
    assert st == want and h is None


def test_create_needs_out_pointer(car):
    assert car.lib().car_create(2, 1, 64, 0, None) == car.CAR_ERR_ARG


def test_calls_on_bad_handles(car):
    bogus = 0x1000
    assert car.car_destroy(None) == car.CAR_ERR_HANDLE
    assert car.car_destroy(bogus) == car.CAR_ERR_HANDLE
    assert car.car_reduce(bogus, [0x10], 0x10) == car.CAR_ERR_HANDLE
    assert car.car_reduce_two_shot(bogus, [0x10], 0x10) == car.CAR_ERR_HANDLE
    assert car.car_reduce_residual_rmsnorm(bogus, [0x10], 16, 16, 1e-6, 16, 16, None) == car.CAR_ERR_HANDLE
    assert car.car_ll128_encode(bogus, 16, 7, 16) == car.CAR_ERR_HANDLE
    assert car.car_ll128_decode_reduce(bogus, [16], 7, 1, 16) == car.CAR_ERR_HANDLE
    assert car.car_ll_encode(bogus, 16, 7, 16) == car.CAR_ERR_HANDLE
    assert car.car_ll_decode_reduce(bogus, [16], 7, 1, 16) == car.CAR_ERR_HANDLE
    assert car.car_ll128_report(bogus)[0] == car.CAR_ERR_HANDLE
    assert car.car_ll_report(bogus)[0] == car.CAR_ERR_HANDLE
    assert car.car_tune_fused(bogus, car.CAR_FUSED_ROWS, 1, 32, 1) == car.CAR_ERR_HANDLE
    assert car.car_sync(bogus) == car.CAR_ERR_HANDLE
    assert car.car_ll128_wire_bytes(bogus) == 0 and car.car_ll_wire_bytes(bogus) == 0


def test_valid_create_without_a_gpu_reports_cuda_error(car):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the gpu tests")
    st, h = car.car_create(2, 4, 64, car.CAR_BF16)
    assert st == car.CAR_ERR_CUDA and h is None
    assert car.car_last_error() != ""
