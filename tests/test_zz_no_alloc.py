"""The allocation-free LL128 decode-reduce entry point.

Some callers cannot call cudaMalloc (allocator callbacks, processes whose
caching pool holds all free memory, paths that cannot take the
synchronisation an allocation implies), so they cannot create a handle.
car_ll128_decode_reduce_noalloc serves them with a stale-line log kept in a
fixed device array inside the library.  This test checks, through the C ABI,
that two calls in a row give the same output and the same stale report as
the handle-based entry point, that the second call does not see the first
call's stale lines, and that the calls change no device memory use.

The file is named to be collected last, so that a run stopping at the first
failure has already run every other test.
"""
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def car():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import rank_sum_reduce_gb300 as car

    return car


def _read_report(buf, cap):
    """stale_out layout: uint64 count, 8 reserved bytes, then (rank, line) uint32 pairs."""
    host = buf.cpu()
    n = int(host[:8].view(torch.int64).item())
    pairs = host[16:16 + 8 * cap].view(torch.int32).view(-1, 2)[: min(n, cap)].tolist()
    return n, {(int(r), int(k)) for r, k in pairs}


def test_noalloc_matches_handle_path_on_two_calls(car):
    dev = "cuda:0"
    W, M, N, dtype = 4, 37, 1000, "bf16"          # 74000 bytes per rank: 617 lines, odd, partial last line
    wl = workloads.custom(W, M, N, dtype, seed=123)
    xs = [workloads.make_x(wl, r, dev) for r in range(W)]
    D = wl.data_bytes
    L = oracle.ll128_lines(D)
    cap = 64
    handle = car.Car(W, M, N, dtype)
    wires = [torch.empty(handle.ll128_wire_bytes, dtype=torch.uint8, device=dev) for _ in range(W)]
    out_ref = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    out_na = torch.empty_like(out_ref)
    stale_buf = torch.zeros(16 + 8 * cap, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream().cuda_stream

    def noalloc_call(flag):
        st = car.car_ll128_decode_reduce_noalloc(W, M, N, car.CAR_BF16, [w.data_ptr() for w in wires], flag, 1,
                                                 out_na.data_ptr(), stale_buf.data_ptr(), cap, stream)
        assert st == car.CAR_OK, car.car_last_error()

    # warm both paths once (module loading happens on first use of each kernel)
    for x, wv in zip(xs, wires):
        handle.ll128_encode(x, 7, wv)
    handle.ll128_decode_reduce(wires, 7, out_ref)
    noalloc_call(7)
    old_flag = torch.tensor(list((6).to_bytes(8, "little")), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]

    plans = [  # two calls in a row with different stale sets
        {1: [0, 5, L - 1], 3: [5]},
        {0: [2], 2: [L // 2]},
    ]
    results = []
    for plan in plans:
        for x, wv in zip(xs, wires):
            handle.ll128_encode(x, 7, wv)
        for r, lines in plan.items():
            for k in lines:
                wires[r].view(L, 16, 8)[k, 15].copy_(old_flag)
        handle.ll128_decode_reduce(wires, 7, out_ref)
        n_ref, pairs_ref = handle.ll128_report()
        noalloc_call(7)
        torch.cuda.synchronize()
        n_na, pairs_na = _read_report(stale_buf, cap)
        results.append((plan, n_ref, set(pairs_ref), n_na, pairs_na, out_ref.cpu(), out_na.cpu()))
    free_after = torch.cuda.mem_get_info()[0]
    handle.close()

    for plan, n_ref, pairs_ref, n_na, pairs_na, o_ref, o_na in results:
        planted = {(r, k) for r, ks in plan.items() for k in ks}
        assert n_ref == n_na == len(planted)
        assert pairs_ref == pairs_na == planted
        assert torch.equal(o_na.view(torch.int16), o_ref.view(torch.int16))
    assert free_after == free_before, "device memory in use changed across the calls"


def test_noalloc_rejects_cap_beyond_its_array(car):
    x = torch.zeros(64, dtype=torch.uint8, device="cuda:0")
    st = car.car_ll128_decode_reduce_noalloc(1, 1, 8, car.CAR_BF16, [x.data_ptr()], 7, 1, x.data_ptr(),
                                             x.data_ptr(), car.CAR_STALE_LIST_MAX + 1, 0)
    assert st == car.CAR_ERR_SIZE
    assert "exceeds" in car.car_last_error()
