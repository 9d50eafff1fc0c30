"""The allocation-free LL128 decode-reduce entry point.

Some callers cannot call cudaMalloc (allocator callbacks, processes whose
caching pool holds all free memory, paths that cannot take the
synchronisation an allocation implies), so they cannot create a handle.
car_ll128_decode_reduce_noalloc serves them with a stale-line log kept in a
fixed device array inside the library.  This test checks, through the C ABI,
that two calls in a row give the same output and the same stale report as
the handle-based entry point and the oracle, that the second call does not see the first
call's stale lines, and that the calls change no device memory use.

The file is named to be collected last, so that a run stopping at the first
failure has already run every other test.
"""
import os
import subprocess

import numpy as np
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


def _other_compute_processes():
    """PIDs of other processes with a CUDA context on this machine's GPUs
    (None when nvidia-smi cannot tell)."""
    try:
        out = subprocess.run(["nvidia-smi", "--query-compute-apps=pid", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=30).stdout
    except Exception:
        return None
    return {int(t) for t in out.split() if t.strip().isdigit()} - {os.getpid()}


def _assert_no_device_memory_change(free_before, reserved_before):
    """This process allocated nothing: torch's pool is unchanged, and the
    device's free memory is unchanged unless another process shares the GPU."""
    assert torch.cuda.memory_reserved() == reserved_before, "torch's memory pool grew across the calls"
    free_after = torch.cuda.mem_get_info()[0]
    if free_after != free_before:
        others = _other_compute_processes()
        assert others, f"free device memory changed by {free_before - free_after} bytes with no other process"


def _oracle_decode(wires, D, dtype):
    """The oracle's decode of the wires as they are now: (stale count, stale
    set, output bytes)."""
    host_w = [wv.cpu().numpy() for wv in wires]
    ref = np.empty(D, dtype=np.uint8)
    n, lst = oracle.ll128_decode_reduce(host_w, D, dtype, 7, ref)
    return n, {tuple(int(v) for v in e) for e in lst.tolist()}, ref


def _bytes(t):
    return t.contiguous().view(-1).view(torch.uint8).cpu().numpy()


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
    free_before, reserved_before = torch.cuda.mem_get_info()[0], torch.cuda.memory_reserved()

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
        results.append((plan, n_ref, set(pairs_ref), n_na, pairs_na, out_ref.cpu(), out_na.cpu(),
                        _oracle_decode(wires, D, dtype)))
    torch.cuda.synchronize()
    _assert_no_device_memory_change(free_before, reserved_before)
    handle.close()

    for plan, n_ref, pairs_ref, n_na, pairs_na, o_ref, o_na, (n_or, pairs_or, b_or) in results:
        planted = {(r, k) for r, ks in plan.items() for k in ks}
        assert n_ref == n_na == n_or == len(planted)
        assert pairs_ref == pairs_na == pairs_or == planted
        assert torch.equal(o_na.view(torch.int16), o_ref.view(torch.int16))
        assert np.array_equal(_bytes(o_na), b_or)


def test_noalloc_rejects_cap_beyond_its_array(car):
    x = torch.zeros(64, dtype=torch.uint8, device="cuda:0")
    st = car.car_ll128_decode_reduce_noalloc(1, 1, 8, car.CAR_BF16, [x.data_ptr()], 7, 1, x.data_ptr(),
                                             x.data_ptr(), car.CAR_STALE_LIST_MAX + 1, 0)
    assert st == car.CAR_ERR_SIZE
    assert "exceeds" in car.car_last_error()


def _encode_with_stale(car, handle, xs, plan, flag=7, old=6):
    W = len(xs)
    L = (xs[0].numel() * xs[0].element_size() + 119) // 120
    wires = [torch.empty(handle.ll128_wire_bytes, dtype=torch.uint8, device="cuda:0") for _ in range(W)]
    for x, wv in zip(xs, wires):
        handle.ll128_encode(x, flag, wv)
    stale = torch.tensor(list(old.to_bytes(8, "little")), dtype=torch.uint8, device="cuda:0")
    for r, lines in plan.items():
        for k in lines:
            wires[r].view(L, 16, 8)[k, 15].copy_(stale)
    return wires


def test_noalloc_counts_every_stale_line_beyond_cap(car):
    """Five stale lines and room for two: the count says five, the two listed
    pairs are planted ones, and the output equals the handle path's."""
    dev = "cuda:0"
    W, M, N, cap = 3, 4, 1200, 2
    wl = workloads.custom(W, M, N, "bf16", seed=77)
    xs = [workloads.make_x(wl, r, dev) for r in range(W)]
    plan = {0: [1, 30], 1: [2], 2: [0, 79]}
    planted = {(r, k) for r, ks in plan.items() for k in ks}
    with car.Car(W, M, N, "bf16") as handle:
        wires = _encode_with_stale(car, handle, xs, plan)
        out_ref = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        handle.ll128_decode_reduce(wires, 7, out_ref)
        n_ref, pairs_ref = handle.ll128_report()
        out_na = torch.empty_like(out_ref)
        stale_buf = torch.full((16 + 8 * cap,), 0xAB, dtype=torch.uint8, device=dev)
        st = car.car_ll128_decode_reduce_noalloc(W, M, N, car.CAR_BF16, [w.data_ptr() for w in wires], 7, 1,
                                                 out_na.data_ptr(), stale_buf.data_ptr(), cap,
                                                 torch.cuda.current_stream().cuda_stream)
        assert st == car.CAR_OK, car.car_last_error()
        torch.cuda.synchronize()
    n_na, pairs_na = _read_report(stale_buf, cap)
    assert n_ref == n_na == len(planted) == 5
    assert set(pairs_ref) == planted and len(pairs_na) == cap and pairs_na <= planted
    assert torch.equal(out_na.view(torch.int16), out_ref.view(torch.int16))
    n_or, pairs_or, b_or = _oracle_decode(wires, wl.data_bytes, "bf16")
    assert n_or == 5 and pairs_or == planted and np.array_equal(_bytes(out_na), b_or)


def test_noalloc_fp32_sixteen_ranks_matches_handle_and_oracle(car):
    """fp32 at W=16 (its own occupancy entry and grid): output bit-exact with
    the handle path and with the oracle, on two calls with different stale
    sets, the second with a misaligned output."""
    dev = "cuda:0"
    W, M, N, cap = 16, 9, 1000, 16
    wl = workloads.custom(W, M, N, "fp32", seed=515)
    xs = [workloads.make_x(wl, r, dev) for r in range(W)]
    D = wl.data_bytes
    L = oracle.ll128_lines(D)
    stream = torch.cuda.current_stream().cuda_stream
    with car.Car(W, M, N, "fp32") as handle:
        for plan, off in (({3: [0, L - 1], 15: [L // 2]}, 0), ({0: [7], 9: [7, 8]}, 4)):
            wires = _encode_with_stale(car, handle, xs, plan)
            planted = {(r, k) for r, ks in plan.items() for k in ks}
            out_ref = torch.empty(M, N, dtype=torch.float32, device=dev)
            handle.ll128_decode_reduce(wires, 7, out_ref)
            n_ref, pairs_ref = handle.ll128_report()
            buf = torch.zeros(D + 32, dtype=torch.uint8, device=dev)
            stale_buf = torch.zeros(16 + 8 * cap, dtype=torch.uint8, device=dev)
            st = car.car_ll128_decode_reduce_noalloc(W, M, N, car.CAR_FP32, [w.data_ptr() for w in wires], 7, 1,
                                                     buf.data_ptr() + off, stale_buf.data_ptr(), cap, stream)
            assert st == car.CAR_OK, car.car_last_error()
            torch.cuda.synchronize()
            n_na, pairs_na = _read_report(stale_buf, cap)
            assert n_ref == n_na == len(planted) and set(pairs_ref) == pairs_na == planted
            got = buf[off:off + D].cpu().numpy()
            assert np.array_equal(got, out_ref.view(-1).view(torch.uint8).cpu().numpy())
            assert not buf[:off].any() and not buf[off + D:].any()
            host_w = [wv.cpu().numpy() for wv in wires]
            ref = np.empty(D, dtype=np.uint8)
            n_or, lst = oracle.ll128_decode_reduce(host_w, D, "fp32", 7, ref)
            assert n_or == len(planted) and {tuple(int(v) for v in e) for e in lst.tolist()} == planted
            assert np.array_equal(got, ref)


def test_noalloc_call_replayed_from_a_cuda_graph(car):
    """One allocation-free call captured in a CUDA graph (after a first call
    outside capture, which sets the device up): each replay reports exactly
    the stale lines planted for it, and its output equals the handle path's."""
    dev = "cuda:0"
    W, M, N, cap = 4, 7, 1000, 32
    wl = workloads.custom(W, M, N, "bf16", seed=606)
    xs = [workloads.make_x(wl, r, dev) for r in range(W)]
    L = oracle.ll128_lines(wl.data_bytes)
    with car.Car(W, M, N, "bf16") as handle:
        wires = [torch.empty(handle.ll128_wire_bytes, dtype=torch.uint8, device=dev) for _ in range(W)]
        out_na = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        out_ref = torch.empty_like(out_na)
        stale_buf = torch.zeros(16 + 8 * cap, dtype=torch.uint8, device=dev)
        ptrs = [w.data_ptr() for w in wires]
        side = torch.cuda.Stream()

        def call(stream):
            st = car.car_ll128_decode_reduce_noalloc(W, M, N, car.CAR_BF16, ptrs, 7, 1, out_na.data_ptr(),
                                                     stale_buf.data_ptr(), cap, stream)
            assert st == car.CAR_OK, car.car_last_error()

        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            call(side.cuda_stream)
            side.synchronize()
            with torch.cuda.graph(g, stream=side):
                call(torch.cuda.current_stream().cuda_stream)
        old = torch.tensor(list((6).to_bytes(8, "little")), dtype=torch.uint8, device=dev)
        for plan in ({1: [0, L - 1], 3: [2]}, {0: [5]}, {}):
            for x, wv in zip(xs, wires):
                handle.ll128_encode(x, 7, wv)
            for r, ks in plan.items():
                for k in ks:
                    wires[r].view(L, 16, 8)[k, 15].copy_(old)
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            n_na, pairs_na = _read_report(stale_buf, cap)
            handle.ll128_decode_reduce(wires, 7, out_ref)
            n_ref, pairs_ref = handle.ll128_report()
            planted = {(r, k) for r, ks in plan.items() for k in ks}
            assert n_na == n_ref == len(planted) and pairs_na == set(pairs_ref) == planted
            assert torch.equal(out_na.view(torch.int16), out_ref.view(torch.int16))
            n_or, pairs_or, b_or = _oracle_decode(wires, wl.data_bytes, "bf16")
            assert n_or == len(planted) and pairs_or == planted and np.array_equal(_bytes(out_na), b_or)
        del g
