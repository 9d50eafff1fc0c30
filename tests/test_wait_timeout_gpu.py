"""The bounded wait of the fused row kernel's split-row exchange, made to run
out on the GPU without any fault.

Rows split over a thread-block cluster exchange partial sums of squares; each
CTA waits for its peers' partials with a time limit (P2 "LL 如何发布和等待
flag": every spin checks for abort instead of spinning forever).  The test
hook car_test_delay_partial shortens that limit and makes one CTA push its
partial late, so its peers' waits run out: they flag the handle
(car_sync -> CAR_ERR_TIMEOUT), write NaN for their columns of that row's
norm_out, then wait, bounded again, until the late partial has landed.  Every
other output must still equal the oracle's, and the next call on the same
handle must be clean.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def car():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import rank_sum_reduce_gb300 as car

    return car


def _i16(t):
    return t.detach().cpu().contiguous().view(torch.int16)


def _norm_ok(got, ref):
    g = got.float().numpy().astype(np.float64)
    r = ref.float().numpy().astype(np.float64)
    return np.abs(g - r) <= 2.0**-7 * np.abs(r) + 1e-5


@pytest.mark.parametrize("W,M,N,shape,row,cta", [
    (8, 4, 8192, (8, 128, 1), 2, 3),      # clusters of 8, one row per cluster
    (8, 200, 8192, (2, 512, 1), 5, 1),    # clusters of 2 that take several rows each: later rows stay right
])
def test_late_partial_runs_the_wait_out_and_loses_only_that_row(car, W, M, N, shape, row, cta):
    wl = workloads.custom(W, M, N, "bf16", seed=300 + M)
    xs, res, w = workloads.make_inputs(wl)
    dx = [x.to(DEV) for x in xs]
    dres, dw = res.to(DEV), w.to(DEV)
    outs = [tuple(torch.empty_like(dres) for _ in range(3)) for _ in range(2)]
    stream = torch.cuda.current_stream().cuda_stream
    with car.Car(W, M, N, "bf16") as c:
        c.tune_fused(car.CAR_FUSED_ROWS, *shape)
        assert car.car_test_delay_partial(c.h, 50_000, cta, row, 2_000_000) == car.CAR_OK  # 50 us limit, 2 ms late
        ro, no, ar = outs[0]
        c.reduce_residual_rmsnorm(dx, dres, dw, wl.eps, ro, no, ar)
        assert car.car_sync(c.h, stream) == car.CAR_ERR_TIMEOUT
        assert car.car_sync(c.h, stream) == car.CAR_OK                # the flag was cleared
        assert car.car_test_delay_partial(c.h, 0, -1, 0, 0) == car.CAR_OK
        ro, no, ar = outs[1]
        c.reduce_residual_rmsnorm(dx, dres, dw, wl.eps, ro, no, ar)
        assert car.car_sync(c.h, stream) == car.CAR_OK
    torch.cuda.synchronize()
    ref_ar, ref_ro, ref_no = (torch.empty_like(res) for _ in range(3))
    oracle.reduce_residual_rmsnorm(xs, res, w, wl.eps, M, N, "bf16", ref_ro, ref_no, ar_out=ref_ar)
    cluster, threads, vpt = shape
    chunk = threads * vpt * 8                      # bf16 columns of one CTA
    mine = slice(cta * chunk, (cta + 1) * chunk)   # the delayed CTA's columns: its own total is complete
    for k, (ro, no, ar) in enumerate(outs):
        assert torch.equal(_i16(ar), _i16(ref_ar)) and torch.equal(_i16(ro), _i16(ref_ro)), f"call {k}"
        got, ref = no.cpu(), ref_no
        others = torch.ones(M, dtype=torch.bool)
        if k == 0:
            others[row] = False
            assert _norm_ok(got[row, mine], ref[row, mine]).all()
            lost = torch.ones(N, dtype=torch.bool)
            lost[mine] = False
            assert torch.isnan(got[row, lost].float()).all()
        assert _norm_ok(got[others], ref[others]).all(), f"call {k}: a row other than the delayed one changed"


def test_hook_rejects_out_of_range_values(car):
    with car.Car(8, 4, 8192, "bf16") as c:
        for args in ((999, 0, 0, 0), (2_000_000_000, 0, 0, 0), (50_000, 8, 0, 0), (50_000, 0, 4, 0),
                     (50_000, 0, -1, 0), (50_000, 0, 0, 200_000_000), (1, -1, 0, 0)):
            assert car.car_test_delay_partial(c.h, *args) == car.CAR_ERR_ARG, args
