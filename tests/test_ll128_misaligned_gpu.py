"""LL128 encode and decode-reduce on rank data that is not 16-byte aligned.

The data buffer (encode) and the output buffer (decode) may start at any
element offset from a 16-byte boundary; wires stay 16-byte aligned.  This is
the misaligned case that "LL128 对齐为何重要" measures for NCCL.  Wires must be
bit-identical to the oracle's and decoded bytes bit-identical to the oracle's
decode.  Canary bytes around the output must survive: the kernel may not
write outside [ar_out, ar_out + D).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
CANARY = 0xC5
PAD = 48


@pytest.fixture(scope="module")
def car():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import rank_sum_reduce_gb300 as car

    return car


def as_bytes(t):
    return t.detach().cpu().contiguous().view(torch.uint8).reshape(-1)


def oracle_wires(xs, D, flag):
    wb = oracle.ll128_wire_bytes(D)
    out = []
    for x in xs:
        wv = np.zeros(wb, dtype=np.uint8)
        oracle.ll128_encode(x, D, flag, wv)
        out.append(wv)
    return out


def offset_buffer(nbytes, offset, fill=CANARY):
    """A device byte buffer with `offset` bytes before and PAD bytes after a
    region of `nbytes`; returns (whole buffer, the region)."""
    base = torch.full((PAD + nbytes + PAD,), fill, dtype=torch.uint8, device=DEV)
    assert base.data_ptr() % 16 == 0
    start = PAD - (PAD % 16) + offset
    return base, base[start:start + nbytes]


def assert_canaries(base, region):
    b = base.cpu()
    start = region.data_ptr() - base.data_ptr()
    before, after = b[:start], b[start + region.numel():]
    assert bool((before == CANARY).all()), f"{int((before != CANARY).sum())} bytes written before the output"
    assert bool((after == CANARY).all()), f"{int((after != CANARY).sum())} bytes written after the output"


CASES = [
    # (W, M, N, dtype): one line, partial last line, odd and even line counts,
    # several warps, a tail shorter than a warp's 480 bytes
    (2, 1, 8, "bf16"), (1, 1, 120, "bf16"), (3, 1, 56, "bf16"), (2, 1, 64, "bf16"), (4, 3, 1000, "bf16"),
    (5, 7, 1544, "fp16"), (16, 5, 776, "bf16"), (8, 9, 1020, "fp32"), (2, 2, 60, "fp32"), (8, 31, 4096, "bf16"),
]
OFFSETS = {"bf16": [2, 4, 6, 8, 12, 14], "fp16": [4, 10], "fp32": [4, 8, 12]}


def cases():
    for W, M, N, dtype in CASES:
        for off in OFFSETS[dtype]:
            yield W, M, N, dtype, off


@pytest.mark.parametrize("W,M,N,dtype,off", list(cases()))
def test_encode_from_misaligned_data(car, W, M, N, dtype, off):
    wl = workloads.custom(W, M, N, dtype, seed=5000 + W + N + off)
    xs = [workloads.make_x(wl, r) for r in range(W)]
    D = wl.data_bytes
    flag = 0x0F1E2D3C4B5A6978
    want = oracle_wires(xs, D, flag)
    with car.Car(W, M, N, dtype) as c:
        for x, ref in zip(xs, want):
            _, data = offset_buffer(D, off)
            data.copy_(as_bytes(x).to(DEV))
            assert data.data_ptr() % 16 == off
            wire = torch.full((c.ll128_wire_bytes,), 0xEE, dtype=torch.uint8, device=DEV)
            c.ll128_encode(data, flag, wire)
            torch.cuda.synchronize()
            assert torch.equal(wire.cpu(), torch.from_numpy(ref)), "wire differs from the oracle's"


@pytest.mark.parametrize("W,M,N,dtype,off", list(cases()))
@pytest.mark.parametrize("n_stale", [0, 3])
def test_decode_into_misaligned_output(car, W, M, N, dtype, off, n_stale):
    wl = workloads.custom(W, M, N, dtype, seed=6000 + W + N + off)
    xs = [workloads.make_x(wl, r) for r in range(W)]
    D = wl.data_bytes
    flag = 9
    wires = oracle_wires(xs, D, flag)
    L = oracle.ll128_lines(D)
    g = torch.Generator().manual_seed(W * 131 + N + off)
    planted = set()
    for _ in range(n_stale):
        r, k = int(torch.randint(0, W, (1,), generator=g)), int(torch.randint(0, L, (1,), generator=g))
        if (r, k) not in planted:
            wires[r][k * 128 + 120] ^= 0x01              # 9 -> 8: the previous round's flag
            planted.add((r, k))
    ref = torch.empty_like(xs[0])
    n_ref, lst_ref = oracle.ll128_decode_reduce(wires, D, dtype, flag, ref)
    assert n_ref == len(planted) and {tuple(e) for e in lst_ref.tolist()} == planted
    with car.Car(W, M, N, dtype) as c:
        dw = [torch.from_numpy(wv).to(DEV) for wv in wires]
        base, out = offset_buffer(D, off)
        assert out.data_ptr() % 16 == off
        c.ll128_decode_reduce(dw, flag, out, max_polls=2)
        n, pairs = c.ll128_report()
        torch.cuda.synchronize()
        assert n == len(planted) and set(pairs) == planted
        got = out.cpu()
        want = as_bytes(ref)
        assert torch.equal(got, want), f"{int((got != want).sum())} of {D} output bytes differ from the oracle's"
        assert_canaries(base, out)


@pytest.mark.parametrize("off_in,off_out", [(2, 14), (8, 8), (12, 0), (0, 6)])
def test_round_trip_misaligned_to_misaligned(car, off_in, off_out):
    """CUDA encode from offset data, CUDA decode into an offset output; the
    result equals the oracle's rank sum of the same tensors."""
    W, M, N, dtype = 8, 64, 8192, "bf16"           # 1 MiB per rank
    wl = workloads.custom(W, M, N, dtype, seed=7000 + off_in * 16 + off_out)
    xs = [workloads.make_x(wl, r) for r in range(W)]
    D = wl.data_bytes
    want = torch.empty_like(xs[0])
    oracle.reduce(xs, dtype, want)
    with car.Car(W, M, N, dtype) as c:
        wires = [torch.empty(c.ll128_wire_bytes, dtype=torch.uint8, device=DEV) for _ in range(W)]
        keep = []
        for x, wv in zip(xs, wires):
            b, data = offset_buffer(D, off_in)
            data.copy_(as_bytes(x).to(DEV))
            keep.append(b)
            c.ll128_encode(data, 21, wv)
        base, out = offset_buffer(D, off_out)
        c.ll128_decode_reduce(wires, 21, out)
        n, _ = c.ll128_report()
        torch.cuda.synchronize()
        assert n == 0
        got = out.cpu()
        assert torch.equal(got, as_bytes(want))
        assert_canaries(base, out)


def test_noalloc_decode_into_misaligned_output(car):
    W, M, N, dtype = 3, 5, 1000, "bf16"
    wl = workloads.custom(W, M, N, dtype, seed=7100)
    xs = [workloads.make_x(wl, r) for r in range(W)]
    D = wl.data_bytes
    wires = oracle_wires(xs, D, 4)
    wires[1][3 * 128 + 120] = 3
    ref = torch.empty_like(xs[0])
    n_ref, _ = oracle.ll128_decode_reduce(wires, D, dtype, 4, ref)
    assert n_ref == 1
    dw = [torch.from_numpy(wv).to(DEV) for wv in wires]
    base, out = offset_buffer(D, 10)
    stale = torch.zeros(16 + 8 * 4, dtype=torch.uint8, device=DEV)
    st = car.car_ll128_decode_reduce_noalloc(W, M, N, car.CAR_BF16, [w.data_ptr() for w in dw], 4, 1,
                                             out.data_ptr(), stale.data_ptr(), 4,
                                             torch.cuda.current_stream().cuda_stream)
    assert st == car.CAR_OK, car.car_last_error()
    torch.cuda.synchronize()
    assert int(stale.cpu()[:8].view(torch.int64).item()) == 1
    assert torch.equal(out.cpu(), as_bytes(ref))
    assert_canaries(base, out)


def test_alignment_rules(car):
    """Element alignment is the floor for LL128 data and output; wires, and
    every pointer of the other calls, stay 16-byte aligned.  Rejected calls
    launch nothing."""
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device=DEV)
    p = buf.data_ptr()
    with car.Car(2, 1, 64, "bf16") as c:
        wire = c.ll128_wire_bytes
        assert car.car_ll128_encode(c.h, p + 1, 7, p + 4096) == car.CAR_ERR_ALIGN
        assert car.car_ll128_encode(c.h, p + 2, 7, p + 4096 + 8) == car.CAR_ERR_ALIGN
        assert car.car_ll128_decode_reduce(c.h, [p + 4096, p + 8192], 7, 1, p + 3) == car.CAR_ERR_ALIGN
        assert car.car_ll128_decode_reduce(c.h, [p + 4096 + 8, p + 8192], 7, 1, p + 2) == car.CAR_ERR_ALIGN
        assert car.car_ll_decode_reduce(c.h, [p + 4096, p + 8192], 7, 1, p + 2) == car.CAR_ERR_ALIGN
        assert car.car_reduce(c.h, [p + 2, p + 256], p + 512) == car.CAR_ERR_ALIGN
        assert wire <= 4096
    with car.Car(2, 1, 64, "fp32") as c:
        assert car.car_ll128_encode(c.h, p + 2, 7, p + 4096) == car.CAR_ERR_ALIGN
        assert car.car_ll128_decode_reduce(c.h, [p + 4096, p + 8192], 7, 1, p + 6) == car.CAR_ERR_ALIGN
    torch.cuda.synchronize()
    assert bool((buf.cpu() == 0).all())
