"""Lamport one-shot push format on the GPU against the oracle: push bits,
receive + fused residual/RMSNorm, stale rows, and region rotation."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SENTINEL = 0x80008000


@pytest.fixture(scope="module")
def car():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import rank_sum_reduce_gb300 as car

    return car


def _inputs(W, M, N, seed, neg_zero=True):
    wl = workloads.custom(W, M, N, "bf16", seed=seed)
    xs, res, w = workloads.make_inputs(wl)
    if neg_zero:   # put some -0.0 in to exercise the scrub
        xs[0].view(torch.int16).view(-1)[:5] = -32768
    return wl, xs, res, w


def _u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def test_push_scrubs_and_packs_like_the_oracle(car):
    W, M, N = 3, 4, 520
    wl, xs, _, _ = _inputs(W, M, N, 1)
    c = car.Car(W, M, N, "bf16")
    comm = torch.zeros(c.lamport_buffer_bytes, dtype=torch.uint8, device=DEV)
    c.lamport_init(comm)
    for r in range(W):
        c.lamport_push(xs[r].to(DEV), r, 5, comm)     # region 2
    torch.cuda.synchronize()
    want = np.zeros(3 * W * M * N, dtype=np.uint16)
    oracle.lamport_fill(want.view(np.uint32))
    for r in range(W):
        oracle.lamport_push(xs[r], M * N, want, W, r, 5)
    assert np.array_equal(comm.cpu().numpy().view(np.uint16), want)
    c.close()


@pytest.mark.parametrize("W,M,N", [(2, 1, 2048), (8, 1, 8192), (4, 3, 1544), (16, 2, 1024), (5, 400, 512),
                                   (8, 40, 8192), (3, 1, 8),
                                   # rows split over clusters of 8 and 4 for every row of a batch
                                   (8, 16, 8192), (4, 16, 4096)])
@pytest.mark.parametrize("missing", [False, True])
def test_round_matches_the_oracle(car, W, M, N, missing):
    wl, xs, res, w = _inputs(W, M, N, 10 + W + M)
    rnd = 7                                            # region 1; refills region 0
    c = car.Car(W, M, N, "bf16")
    comm = torch.empty(c.lamport_buffer_bytes, dtype=torch.uint8, device=DEV)
    c.lamport_init(comm)
    skip = W - 1 if missing else -1
    for r in range(W):
        if r != skip:
            c.lamport_push(xs[r].to(DEV), r, rnd, comm)
    host = np.zeros(3 * W * M * N, dtype=np.uint16)   # the oracle's copy of the same buffer
    oracle.lamport_fill(host.view(np.uint32))
    for r in range(W):
        if r != skip:
            oracle.lamport_push(xs[r], M * N, host, W, r, rnd)
    dres, dw = res.to(DEV), w.to(DEV)
    ro, no, ar = (torch.full_like(dres, 3.0) for _ in range(3))
    for polls in (1, 3):
        c.lamport_reduce_residual_rmsnorm(comm, rnd, dres, dw, wl.eps, ro, no, ar, max_polls=polls)
        n_stale, pairs = c.lamport_report()
        assert n_stale == (M if missing else 0)
        assert set(pairs) == ({(skip, m) for m in range(M)} if missing else set())
    c.sync()   # no bounded wait (split rows' partial exchange) ran out
    torch.cuda.synchronize()
    ref_ro, ref_no, ref_ar = (np.empty(M * N, dtype=np.uint16) for _ in range(3))
    n_ref, lst = oracle.lamport_reduce_residual_rmsnorm(W, host, rnd, M, N, res, w, wl.eps, ref_ro, ref_no, ref_ar)
    assert n_ref == n_stale and {tuple(e) for e in lst.tolist()} == set(pairs)
    assert np.array_equal(_u16(ar).ravel(), ref_ar) and np.array_equal(_u16(ro).ravel(), ref_ro)
    got = no.float().cpu().numpy().ravel().astype(np.float64)
    ref = torch.from_numpy(ref_no.view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2.0**-7 * np.abs(ref) + 1e-5)
    assert np.array_equal(comm.cpu().numpy().view(np.uint16), host)   # same refill, same untouched regions
    c.close()


def test_rounds_rotate_over_three_regions(car):
    """Six rounds on one buffer: every round sees only its own pushes; a round
    whose push is left out is reported stale instead of reusing old data."""
    W, M, N = 4, 6, 1024
    c = car.Car(W, M, N, "bf16")
    comm = torch.empty(c.lamport_buffer_bytes, dtype=torch.uint8, device=DEV)
    c.lamport_init(comm)
    host = np.zeros(3 * W * M * N, dtype=np.uint16)
    oracle.lamport_fill(host.view(np.uint32))
    for rnd in range(6):
        wl, xs, res, w = _inputs(W, M, N, 100 + rnd, neg_zero=False)
        skip = 2 if rnd == 4 else -1
        for r in range(W):
            if r != skip:
                c.lamport_push(xs[r].to(DEV), r, rnd, comm)
                oracle.lamport_push(xs[r], M * N, host, W, r, rnd)
        dres, dw = res.to(DEV), w.to(DEV)
        ro, no = torch.empty_like(dres), torch.empty_like(dres)
        c.lamport_reduce_residual_rmsnorm(comm, rnd, dres, dw, wl.eps, ro, no)
        n_stale, _ = c.lamport_report()
        ref_ro, ref_no = np.empty(M * N, dtype=np.uint16), np.empty(M * N, dtype=np.uint16)
        n_ref, _ = oracle.lamport_reduce_residual_rmsnorm(W, host, rnd, M, N, res, w, wl.eps, ref_ro, ref_no)
        assert n_stale == n_ref == (M if rnd == 4 else 0)
        assert np.array_equal(_u16(ro).ravel(), ref_ro)
        assert np.array_equal(comm.cpu().numpy().view(np.uint16), host)
    c.close()


def test_lamport_argument_errors(car):
    with car.Car(2, 2, 64, "fp16") as c:
        assert c.lamport_buffer_bytes == 0
        x = torch.zeros(1024, dtype=torch.uint8, device=DEV)
        assert car.car_lamport_init(c.h, x.data_ptr(), 0) == car.CAR_ERR_ARG
    with car.Car(2, 2, 64, "bf16") as c:
        x = torch.zeros(c.lamport_buffer_bytes + 64, dtype=torch.uint8, device=DEV)
        p = x.data_ptr()
        assert car.car_lamport_push(c.h, p, 2, 0, p, 0) == car.CAR_ERR_ARG
        assert car.car_lamport_push(c.h, p, -1, 0, p, 0) == car.CAR_ERR_ARG
        assert car.car_lamport_push(c.h, p + 8, 0, 0, p, 0) == car.CAR_ERR_ALIGN
        assert car.car_lamport_reduce_residual_rmsnorm(c.h, p, 0, 0, p, p, 1e-6, p, p, None, 0) == car.CAR_ERR_ARG


@pytest.mark.parametrize("max_polls", [1, 3])
def test_single_missing_words_make_only_their_rows_stale(car, max_polls):
    """Every rank pushes, then single 32-bit words of the receive region are
    put back to the sentinel, as if those words had not arrived yet: one in
    the middle of a row, one in a row's last 16-byte vector, one in the
    columns that CTA 3 of the row's 8-CTA cluster reduces (W=8, M=16,
    N=8192 bf16 takes clusters of 8, each CTA 128 of the row's 1024
    vectors), and one in the last vector of the last row.  The receive must
    report exactly those (rank, row) pairs, zero exactly those rows, and
    match the oracle's outputs and refilled buffer on the same buffer."""
    W, M, N = 8, 16, 8192
    wl, xs, res, w = _inputs(W, M, N, 4242)
    rnd = 4                                            # region 1; refills region 0
    c = car.Car(W, M, N, "bf16")
    comm = torch.empty(c.lamport_buffer_bytes, dtype=torch.uint8, device=DEV)
    c.lamport_init(comm)
    host = np.zeros(3 * W * M * N, dtype=np.uint16)
    oracle.lamport_fill(host.view(np.uint32))
    for r in range(W):
        c.lamport_push(xs[r].to(DEV), r, rnd, comm)
        oracle.lamport_push(xs[r], M * N, host, W, r, rnd)
    holes = {  # (rank, row): column of the first bf16 of the missing word
        (2, 5): N // 2 + 2,                            # middle of the row
        (7, 9): N - 4,                                 # the row's last 16-byte vector
        (0, 12): 3 * (N // 8) + 100,                   # inside CTA 3's columns
        (5, M - 1): N - 2,                             # last vector of the last row
    }
    region = rnd % 3
    dwords = comm.view(torch.int32)
    hwords = host.view(np.uint32)
    for (r, m), col in holes.items():
        word = ((region * W + r) * M * N + m * N + col) // 2
        dwords[word] = torch.tensor(SENTINEL, dtype=torch.int64).to(torch.int32).item()
        hwords[word] = SENTINEL
    torch.cuda.synchronize()
    dres, dw = res.to(DEV), w.to(DEV)
    ro, no, ar = (torch.full_like(dres, 3.0) for _ in range(3))
    c.lamport_reduce_residual_rmsnorm(comm, rnd, dres, dw, wl.eps, ro, no, ar, max_polls=max_polls)
    n_stale, pairs = c.lamport_report()
    c.sync()
    torch.cuda.synchronize()
    assert n_stale == len(holes) and set(pairs) == set(holes)
    ref_ro, ref_no, ref_ar = (np.empty(M * N, dtype=np.uint16) for _ in range(3))
    n_ref, lst = oracle.lamport_reduce_residual_rmsnorm(W, host, rnd, M, N, res, w, wl.eps, ref_ro, ref_no, ref_ar)
    assert n_ref == len(holes) and {tuple(int(v) for v in e) for e in lst.tolist()} == set(holes)
    assert np.array_equal(_u16(ar).ravel(), ref_ar) and np.array_equal(_u16(ro).ravel(), ref_ro)
    got = no.float().cpu().numpy().ravel().astype(np.float64)
    ref = torch.from_numpy(ref_no.view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2.0**-7 * np.abs(ref) + 1e-5)
    for _, m in holes:                                 # the stale rows are zero in every output
        assert not _u16(no).reshape(M, N)[m].any() and not _u16(ro).reshape(M, N)[m].any()
    assert np.array_equal(comm.cpu().numpy().view(np.uint16), host)
    c.close()
