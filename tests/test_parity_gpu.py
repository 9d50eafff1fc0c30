"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bar: ar, residual_out, LL/LL128 wires and decode-reduce results bit-exact;
norm_out within |gpu - ref| <= 2^-7 * |ref| + 1e-5 of the oracle's value in
the output type; stale-line reports equal as sets.  Inputs are seeded
synthetic tensors from workloads.py; every expected value comes from the
oracle or from the test's own planted stale lines.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

TOL_REL, TOL_ABS = 2.0**-7, 1e-5


def car_elem(dtype):
    return 4 if dtype == "fp32" else 2


@pytest.fixture(scope="module")
def car():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import rank_sum_reduce_gb300 as car

    return car


DEV = "cuda:0"


def bits(t):
    t = t.detach().cpu().contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16)
    if t.dtype == torch.float32:
        return t.view(torch.int32)
    return t


def assert_bits_equal(got, want, what):
    g, w = bits(got), bits(want)
    if not torch.equal(g, w):
        diff = (g != w).nonzero()
        first = tuple(diff[0].tolist())
        raise AssertionError(f"{what}: {diff.shape[0]} of {g.numel()} elements differ; first at "
                             f"{first}: got {int(g[first])} want {int(w[first])}")


def assert_norm_close(got, ref, what="norm_out"):
    g = got.detach().cpu().float().numpy().astype(np.float64).ravel()
    r = ref.detach().cpu().float().numpy().astype(np.float64).ravel()
    bad = np.abs(g - r) > TOL_REL * np.abs(r) + TOL_ABS
    assert not bad.any(), f"{what}: {bad.sum()} elements outside tolerance, first {np.nonzero(bad)[0][:5]}"


def oracle_fused(xs, res, w, eps, M, N, dtype):
    ar, ro, no = torch.empty_like(res), torch.empty_like(res), torch.empty_like(res)
    oracle.reduce_residual_rmsnorm(xs, res, w, eps, M, N, dtype, ro, no, ar_out=ar)
    return ar, ro, no


def oracle_reduce(xs, dtype):
    out = torch.empty_like(xs[0])
    oracle.reduce(xs, dtype, out)
    return out


# ---------------------------------------------------------------------------
# plain rank sum
# ---------------------------------------------------------------------------
REDUCE_CASES = [
    # (W, M, N, dtype): ragged tails over several 256-thread tiles, every instance
    (1, 3, 520, "bf16"), (2, 37, 1000, "bf16"), (3, 11, 776, "bf16"), (4, 64, 1032, "bf16"),
    (5, 9, 2056, "fp16"), (8, 33, 1000, "bf16"), (16, 7, 1544, "bf16"), (6, 13, 3000, "fp32"),
    (4, 17, 1020, "fp32"), (8, 21, 520, "fp16"), (16, 5, 4100, "fp32"), (2, 1, 8, "bf16"),
    (7, 1, 24, "fp16"), (2, 1, 4, "fp32"),
]


@pytest.mark.parametrize("W,M,N,dtype", REDUCE_CASES)
def test_reduce_bit_exact(car, W, M, N, dtype):
    wl = workloads.custom(W, M, N, dtype, seed=1000 + W * 7 + M)
    xs = [workloads.make_x(wl, r) for r in range(W)]
    dx = [x.to(DEV) for x in xs]
    out = torch.full_like(dx[0], float("nan"))
    with car.Car(W, M, N, dtype) as c:
        c.reduce(dx, out)
    torch.cuda.synchronize()
    assert_bits_equal(out, oracle_reduce(xs, dtype), "ar")


@pytest.mark.parametrize("W,M,N,dtype", REDUCE_CASES + [(8, 512, 8192, "bf16"), (3, 1, 8, "bf16"), (16, 1, 64, "fp32")])
def test_two_shot_bit_exact(car, W, M, N, dtype):
    """Owner-rotated sums, including part == 0 (fewer units than ranks) and a
    remainder for the last shard."""
    wl = workloads.custom(W, M, N, dtype, seed=7000 + W * 7 + M)
    xs = [workloads.make_x(wl, r) for r in range(W)]
    dx = [x.to(DEV) for x in xs]
    out = torch.full_like(dx[0], float("nan"))
    with car.Car(W, M, N, dtype) as c:
        c.reduce_two_shot(dx, out)
    torch.cuda.synchronize()
    want = torch.empty_like(xs[0])
    oracle.reduce_two_shot(xs, dtype, want)
    assert_bits_equal(out, want, "two-shot ar")


def test_reduce_output_may_alias_an_input(car):
    W, M, N = 8, 19, 1032
    wl = workloads.custom(W, M, N, "bf16", seed=5)
    xs = [workloads.make_x(wl, r) for r in range(W)]
    want = oracle_reduce(xs, "bf16")
    for k in (0, 5):
        dx = [x.to(DEV) for x in xs]
        with car.Car(W, M, N, "bf16") as c:
            c.reduce(dx, dx[k])
        torch.cuda.synchronize()
        assert_bits_equal(dx[k], want, f"ar aliased to input {k}")


def test_reduce_special_values(car):
    """-0 seeding, subnormal sums, overflow to inf, ties: the oracle decides."""
    W, M, N = 4, 1, 4096
    g = torch.Generator().manual_seed(3)
    pats = torch.randint(0, 65536, (W, M * N), generator=g, dtype=torch.int32).to(torch.int16)
    pats[:, :8] = torch.tensor([-32768, -32768, 0x0001, 0x0080, 0x7F7F, -129, 0x3F80, 0x3B80], dtype=torch.int16)
    xs = [p.view(torch.bfloat16).reshape(M, N).clone() for p in pats]
    keep = ~torch.isnan(torch.stack([x.float() for x in xs])).any(0)
    xs = [torch.where(keep, x, torch.zeros_like(x)) for x in xs]
    dx = [x.to(DEV) for x in xs]
    out = torch.empty_like(dx[0])
    with car.Car(W, M, N, "bf16") as c:
        c.reduce(dx, out)
    torch.cuda.synchronize()
    want = oracle_reduce(xs, "bf16")
    got_b, want_b = bits(out), bits(want)
    nan_both = torch.isnan(out.cpu().float()) & torch.isnan(want.float())
    assert torch.equal(got_b[~nan_both], want_b[~nan_both])


# ---------------------------------------------------------------------------
# fused rank sum + residual + RMSNorm
# ---------------------------------------------------------------------------
FUSED_CASES = [
    (2, 1, 2048, "bf16"), (8, 1, 8192, "bf16"), (8, 3, 1000, "bf16"), (4, 400, 512, "bf16"),
    (3, 5, 1544, "fp16"), (16, 2, 4096, "bf16"), (4, 7, 4096, "fp32"), (1, 9, 264, "bf16"),
    (5, 331, 776, "fp32"), (8, 310, 8192, "bf16"), (2, 1, 8, "bf16"), (7, 2, 16, "fp16"),
    (8, 2, 32768, "bf16"), (4, 1, 16384, "fp32"),
    # row kernel between a few rows and the pipeline's threshold: one CTA per
    # row with two vectors per thread (W=8), 1024 threads (W=4), a cluster of
    # two where no two-vector instance exists (W=16)
    (8, 64, 8192, "bf16"), (8, 180, 8192, "bf16"), (4, 150, 8192, "bf16"), (16, 40, 8192, "bf16"),
    # automatic clusters of 8 and 4 CTAs for every row of a small batch
    (8, 16, 8192, "bf16"), (2, 32, 8192, "bf16"), (8, 12, 4096, "fp16"),
    # many 8 KB rows: the row kernel (W=8 at two CTAs per SM) loops over rows, prefetching the next
    (8, 700, 4096, "bf16"), (4, 1000, 2048, "bf16"),
]


def _fused_inputs(W, M, N, dtype, seed):
    wl = workloads.custom(W, M, N, dtype, seed=seed)
    xs, res, w = workloads.make_inputs(wl)
    return wl, xs, res, w


@pytest.mark.parametrize("kernel", ["auto", "rows", "pipeline"])
@pytest.mark.parametrize("W,M,N,dtype", FUSED_CASES)
def test_fused_parity(car, W, M, N, dtype, kernel):
    wl, xs, res, w = _fused_inputs(W, M, N, dtype, seed=2000 + W + M)
    dx = [x.to(DEV) for x in xs]
    dres, dw = res.to(DEV), w.to(DEV)
    ro, no, ar = torch.empty_like(dres), torch.empty_like(dres), torch.empty_like(dres)
    with car.Car(W, M, N, dtype) as c:
        if kernel != "auto":
            c.tune_fused(car.CAR_FUSED_ROWS if kernel == "rows" else car.CAR_FUSED_PIPELINE)
        c.reduce_residual_rmsnorm(dx, dres, dw, wl.eps, ro, no, ar)
        c.sync()
    torch.cuda.synchronize()
    ref_ar, ref_ro, ref_no = oracle_fused(xs, res, w, wl.eps, M, N, dtype)
    assert_bits_equal(ar, ref_ar, "ar")
    assert_bits_equal(ro, ref_ro, "residual_out")
    assert_norm_close(no, ref_no)


SHAPES = [(1, 128, 1), (1, 256, 1), (1, 512, 2), (2, 512, 1), (4, 256, 1), (8, 128, 1), (8, 64, 2),
          (2, 256, 2), (4, 128, 2)]


@pytest.mark.parametrize("cluster,threads,vpt", SHAPES)
def test_fused_every_launch_shape(car, cluster, threads, vpt):
    """All shapes give the same ar/residual_out bits and norm within tolerance,
    on a problem where rows outnumber resident groups (row loop) and M = 1."""
    for W, M, N in ((8, 700, 8192), (8, 1, 8192), (4, 3, 4096)):
        wl, xs, res, w = _fused_inputs(W, M, N, "bf16", seed=77 + M)
        dx = [x.to(DEV) for x in xs]
        dres, dw = res.to(DEV), w.to(DEV)
        ro, no, ar = torch.empty_like(dres), torch.empty_like(dres), torch.empty_like(dres)
        with car.Car(W, M, N, "bf16") as c:
            V = N * 2 // 16
            if cluster * threads * vpt < V:
                assert car.car_tune_fused(c.h, car.CAR_FUSED_ROWS, cluster, threads, vpt) == car.CAR_ERR_SIZE
                continue
            c.tune_fused(car.CAR_FUSED_ROWS, cluster, threads, vpt)
            c.reduce_residual_rmsnorm(dx, dres, dw, wl.eps, ro, no, ar)
        torch.cuda.synchronize()
        ref_ar, ref_ro, ref_no = oracle_fused(xs, res, w, wl.eps, M, N, "bf16")
        assert_bits_equal(ar, ref_ar, "ar")
        assert_bits_equal(ro, ref_ro, "residual_out")
        assert_norm_close(no, ref_no)


PIPELINE_CASES = [
    # rows spread over every SM several times, partial last pass, every dtype, odd and large W
    (8, 700, 8192, "bf16"), (4, 333, 4096, "fp32"), (3, 401, 1544, "fp16"), (16, 160, 2048, "bf16"),
    (1, 155, 520, "bf16"), (5, 300, 16384, "bf16"), (2, 152, 8, "bf16"), (8, 2000, 1024, "bf16"),
]


@pytest.mark.parametrize("cluster", [1, 2])
@pytest.mark.parametrize("W,M,N,dtype", PIPELINE_CASES)
def test_fused_pipeline_many_rows(car, W, M, N, dtype, cluster):
    wl, xs, res, w = _fused_inputs(W, M, N, dtype, seed=5000 + W + M)
    dx = [x.to(DEV) for x in xs]
    dres, dw = res.to(DEV), w.to(DEV)
    ro, no, ar = torch.empty_like(dres), torch.empty_like(dres), torch.empty_like(dres)
    with car.Car(W, M, N, dtype) as c:
        V = N * car_elem(dtype) // 16
        if cluster == 2 and V % 2:
            assert car.car_tune_fused(c.h, car.CAR_FUSED_PIPELINE, 2, 0, 0) == car.CAR_ERR_SIZE
            return
        c.tune_fused(car.CAR_FUSED_PIPELINE, cluster)
        for _ in range(2):   # twice: the ring restarts cleanly on the next launch
            c.reduce_residual_rmsnorm(dx, dres, dw, wl.eps, ro, no, ar)
        c.sync()
    torch.cuda.synchronize()
    ref_ar, ref_ro, ref_no = oracle_fused(xs, res, w, wl.eps, M, N, dtype)
    assert_bits_equal(ar, ref_ar, "ar")
    assert_bits_equal(ro, ref_ro, "residual_out")
    assert_norm_close(no, ref_no)


def _degenerate_rows(W, M, N, seed):
    """bf16 inputs whose rows 0..4 are degenerate cases of the fused op, the
    rest ordinary: 0 all zero; 1 zero inputs over a constant residual; 2 every
    rank -0.0; 3 +inf in one rank; 4 zero inputs and residual (for eps = 0)."""
    g = torch.Generator().manual_seed(seed)
    xs = [torch.randn(M, N, generator=g).bfloat16() for _ in range(W)]
    res = torch.randn(M, N, generator=g).bfloat16()
    w = (torch.rand(N, generator=g) + 0.5).bfloat16()
    for x in xs:
        x[0] = 0.0
        x[1] = 0.0
        x[2] = -0.0
        x[4] = 0.0
    res[0] = 0.0
    res[1] = 0.375
    res[4] = 0.0
    xs[W - 1][3, N // 2] = float("inf")
    return xs, res, w


@pytest.mark.parametrize("kernel,M", [("rows", 6), ("cluster", 6), ("pipeline", 300)])
@pytest.mark.parametrize("eps", [1e-6, 0.0])
def test_fused_degenerate_rows(car, kernel, M, eps):
    """ar and residual_out bit-exact, norm_out within tolerance, and NaN in
    exactly the same places as the oracle (inf inputs; a zero row with eps 0)."""
    W, N = 3, 1024
    xs, res, w = _degenerate_rows(W, M, N, seed=77 + M)
    ref_ar, ref_ro, ref_no = oracle_fused(xs, res, w, eps, M, N, "bf16")
    dx = [x.to(DEV) for x in xs]
    ro, no, ar = (torch.empty(M, N, dtype=torch.bfloat16, device=DEV) for _ in range(3))
    with car.Car(W, M, N, "bf16") as c:
        if kernel == "cluster":
            c.tune_fused(car.CAR_FUSED_ROWS, 4, 32, 1)   # each row over 4 CTAs: the exchanged totals are inf / 0 too
        else:
            c.tune_fused(car.CAR_FUSED_ROWS if kernel == "rows" else car.CAR_FUSED_PIPELINE)
        c.reduce_residual_rmsnorm(dx, res.to(DEV), w.to(DEV), eps, ro, no, ar)
    torch.cuda.synchronize()
    assert_bits_equal(ar, ref_ar, "ar")
    assert_bits_equal(ro, ref_ro, "residual_out")
    got, ref = no.cpu().float(), ref_no.float()
    assert torch.equal(torch.isnan(got), torch.isnan(ref)), "NaN positions differ"
    # inf in one element: the row's statistic is inf, so rms = 0; that element
    # gives inf * 0 = NaN, every other element of the row 0
    assert bool(torch.isnan(ref[3, N // 2])) and int(torch.isnan(ref[3]).sum()) == 1
    assert bool((got[3][~torch.isnan(got[3])] == 0).all())
    assert bits(ar)[2].eq(-32768).all()                         # -0.0 ranks sum to -0.0 (seeded with rank 0)
    if eps > 0:
        assert bool((ref[0] == 0).all()) and bool((got[0] == 0).all())   # zero row: exactly 0
    else:
        assert bool(torch.isnan(ref[0]).all()) and bool(torch.isnan(ref[4]).all())  # 0 * rsqrt(0)
    keep = ~torch.isnan(ref)
    assert_norm_close(got[keep], ref[keep])


@pytest.mark.parametrize("W,M,N,dtype,kernel", [
    (4, 6, 2048, "bf16", "rows"),
    (8, 400, 8192, "bf16", "pipeline"),   # ranks 6, 7 and the residual loaded by the consumers
    (8, 400, 8192, "bf16", "pipeline_w7"),  # ar_out == the last rank, a register-loaded slice
    (4, 333, 4096, "fp32", "pipeline"),   # every slice through the bulk-copy ring
])
def test_fused_aliasing_and_no_ar(car, W, M, N, dtype, kernel):
    """residual_out == residual, and ar_out == one rank's input: each element
    is read before the same CTA writes it."""
    wl, xs, res, w = _fused_inputs(W, M, N, dtype, seed=31 + M)
    ref_ar, ref_ro, ref_no = oracle_fused(xs, res, w, wl.eps, M, N, dtype)
    tune = car.CAR_FUSED_ROWS if kernel == "rows" else car.CAR_FUSED_PIPELINE
    k = W - 1 if kernel == "pipeline_w7" else 2
    dx = [x.to(DEV) for x in xs]
    dres, dw = res.to(DEV), w.to(DEV)
    no = torch.empty_like(dres)
    with car.Car(W, M, N, dtype) as c:
        c.tune_fused(tune)
        c.reduce_residual_rmsnorm(dx, dres, dw, wl.eps, dres, no, None)   # residual_out == residual
    torch.cuda.synchronize()
    assert_bits_equal(dres, ref_ro, "residual_out in place")
    assert_norm_close(no, ref_no)
    dx = [x.to(DEV) for x in xs]
    dres = res.to(DEV)
    ro = torch.empty_like(dres)
    with car.Car(W, M, N, dtype) as c:
        c.tune_fused(tune)
        c.reduce_residual_rmsnorm(dx, dres, dw, wl.eps, ro, no, dx[k])   # ar_out == inputs[k]
    torch.cuda.synchronize()
    assert_bits_equal(dx[k], ref_ar, "ar in place")
    assert_bits_equal(ro, ref_ro, "residual_out")
    assert_norm_close(no, ref_no)


@pytest.mark.parametrize("W,M,dtype,kernel", [
    (16, 1, "bf16", "auto"),       # most ranks, one row split over a cluster
    (3, 5, "fp32", "rows"),        # one CTA per row
    (8, 200, "bf16", "auto"),      # more rows than SMs: the pipeline, with its ring cut to fit
    (8, 200, "fp16", "rows"),
    (2, 160, "bf16", "pipeline"),
])
def test_fused_at_the_longest_row(car, W, M, dtype, kernel):
    """Rows of exactly CAR_MAX_ROW_BYTES: every output element against the oracle."""
    N = car.CAR_MAX_ROW_BYTES // car_elem(dtype)
    wl, xs, res, w = _fused_inputs(W, M, N, dtype, seed=2600 + W + M)
    dx = [x.to(DEV) for x in xs]
    dres, dw = res.to(DEV), w.to(DEV)
    ro, no, ar = torch.empty_like(dres), torch.empty_like(dres), torch.empty_like(dres)
    with car.Car(W, M, N, dtype) as c:
        if kernel != "auto":
            c.tune_fused(car.CAR_FUSED_ROWS if kernel == "rows" else car.CAR_FUSED_PIPELINE)
        c.reduce_residual_rmsnorm(dx, dres, dw, wl.eps, ro, no, ar)
        c.sync()
    torch.cuda.synchronize()
    ref_ar, ref_ro, ref_no = oracle_fused(xs, res, w, wl.eps, M, N, dtype)
    assert_bits_equal(ar, ref_ar, "ar")
    assert_bits_equal(ro, ref_ro, "residual_out")
    assert_norm_close(no, ref_no)


def test_fused_rejects_rows_beyond_limit(car):
    N = car.CAR_MAX_ROW_BYTES // 2 + 8
    with car.Car(2, 1, N, "bf16") as c:
        x = torch.zeros(N, dtype=torch.bfloat16, device=DEV)
        st = car.car_reduce_residual_rmsnorm(c.h, [x.data_ptr()] * 2, x.data_ptr(), x.data_ptr(), 1e-6,
                                             x.data_ptr(), x.data_ptr(), None, 0)
        assert st == car.CAR_ERR_SIZE


def test_binding_rejects_unusable_tensors(car):
    """The torch layer checks what it hands the C ABI: CUDA, contiguous, and at
    least the bytes the call touches; the rank list has W entries."""
    W, M, N = 2, 4, 256
    xs = [torch.zeros(M, N, dtype=torch.bfloat16, device=DEV) for _ in range(W)]
    out = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    with car.Car(W, M, N, "bf16") as c:
        with pytest.raises(ValueError, match="CUDA"):
            c.reduce([xs[0].cpu(), xs[1]], out)
        with pytest.raises(ValueError, match="contiguous"):
            c.reduce([xs[0], torch.zeros(N, M, dtype=torch.bfloat16, device=DEV).t()], out)
        with pytest.raises(ValueError, match="needs"):
            c.reduce(xs, out.view(-1)[:-1])
        with pytest.raises(ValueError, match="W = 2"):
            c.reduce(xs[:1], out)
        wire = torch.empty(c.ll128_wire_bytes - 16, dtype=torch.uint8, device=DEV)
        with pytest.raises(ValueError, match="wire"):
            c.ll128_encode(xs[0], 7, wire)
        c.reduce(xs, out)   # a valid call still works
    torch.cuda.synchronize()
    assert bool((out == 0).all())


def test_argument_errors_launch_nothing(car):
    with car.Car(2, 2, 64, "bf16") as c:
        x = torch.zeros(2 * 64 + 8, dtype=torch.bfloat16, device=DEV)
        p = x.data_ptr()
        assert car.car_reduce(c.h, [p, p + 2], p) == car.CAR_ERR_ALIGN
        assert car.car_reduce(c.h, [p, 0], p) == car.CAR_ERR_ARG
        assert car.car_reduce(c.h, None, p) == car.CAR_ERR_ARG
        assert car.car_reduce(c.h, [p, p], p + 8) == car.CAR_ERR_ALIGN
        assert car.car_reduce_residual_rmsnorm(c.h, [p, p], p, p, float("nan"), p, p, None) == car.CAR_ERR_ARG
        assert car.car_reduce_residual_rmsnorm(c.h, [p, p], p, p, -1.0, p, p, None) == car.CAR_ERR_ARG
        assert car.car_ll128_decode_reduce(c.h, [p, p], 7, 0, p) == car.CAR_ERR_ARG
        assert car.car_ll_decode_reduce(c.h, [p, p], 7, 0, p) == car.CAR_ERR_ARG
        assert car.car_tune_fused(c.h, car.CAR_FUSED_ROWS, 3, 64, 1) == car.CAR_ERR_ARG
        assert car.car_tune_fused(c.h, car.CAR_FUSED_ROWS, 1, 48, 1) == car.CAR_ERR_ARG
        assert car.car_tune_fused(c.h, car.CAR_FUSED_PIPELINE, 4, 0, 0) == car.CAR_ERR_ARG
        assert car.car_tune_fused(c.h, car.CAR_FUSED_PIPELINE, 0, 64, 0) == car.CAR_ERR_ARG
        assert car.car_tune_fused(c.h, 9, 0, 0, 0) == car.CAR_ERR_ARG
        assert car.car_sync(c.h) == car.CAR_OK
        h = c.h
    assert car.car_destroy(h) == car.CAR_ERR_HANDLE   # already destroyed by the context manager
    assert car.car_reduce(h, [p, p], p) == car.CAR_ERR_HANDLE


# ---------------------------------------------------------------------------
# LL128 and LL
# ---------------------------------------------------------------------------
def _oracle_wires(fmt, xs, D, flag):
    wb = oracle.ll128_wire_bytes(D) if fmt == "ll128" else oracle.ll_wire_bytes(D)
    out = []
    for x in xs:
        wv = np.zeros(max(wb, 16), dtype=np.uint8)
        (oracle.ll128_encode if fmt == "ll128" else oracle.ll_encode)(x, D, flag, wv)
        out.append(wv)
    return out


WIRE_CASES = [
    # (W, M, N, dtype): lines odd/even, partial last line, single line, many pairs
    (2, 1, 8, "bf16"), (3, 1, 56, "bf16"), (2, 1, 64, "bf16"), (4, 3, 1000, "bf16"), (16, 5, 776, "bf16"),
    (5, 7, 1544, "fp16"), (8, 9, 1020, "fp32"), (1, 1, 120, "bf16"), (2, 2, 60, "fp32"), (8, 31, 4096, "bf16"),
    # 8 MiB per rank: more warps of work than the resident grid, so the grid-stride loops wrap
    (2, 1024, 4096, "bf16"),
]


@pytest.mark.parametrize("fmt", ["ll128", "ll"])
@pytest.mark.parametrize("W,M,N,dtype", WIRE_CASES)
def test_wire_encode_bit_exact(car, fmt, W, M, N, dtype):
    wl = workloads.custom(W, M, N, dtype, seed=3000 + W + N)
    xs = [workloads.make_x(wl, r) for r in range(W)]
    D = wl.data_bytes
    flag = 0x0123456789ABCDEF if fmt == "ll128" else 0x89ABCDEF
    want = _oracle_wires(fmt, xs, D, flag)
    with car.Car(W, M, N, dtype) as c:
        wb = c.ll128_wire_bytes if fmt == "ll128" else c.ll_wire_bytes
        assert wb == (oracle.ll128_wire_bytes(D) if fmt == "ll128" else oracle.ll_wire_bytes(D))
        for x, ref in zip(xs, want):
            wire = torch.full((wb,), 0xEE, dtype=torch.uint8, device=DEV)
            (c.ll128_encode if fmt == "ll128" else c.ll_encode)(x.to(DEV), flag, wire)
            torch.cuda.synchronize()
            assert torch.equal(wire.cpu(), torch.from_numpy(ref[:wb]))


@pytest.mark.parametrize("fmt", ["ll128", "ll"])
@pytest.mark.parametrize("W,M,N,dtype", WIRE_CASES)
@pytest.mark.parametrize("n_stale", [0, 3])
def test_wire_decode_reduce_bit_exact(car, fmt, W, M, N, dtype, n_stale):
    """Oracle-encoded wires (stale lines planted by the test) decoded by the
    CUDA path and by the oracle: same output bits, same stale set."""
    wl = workloads.custom(W, M, N, dtype, seed=4000 + W + N)
    xs = [workloads.make_x(wl, r) for r in range(W)]
    D = wl.data_bytes
    flag = 7
    wires = _oracle_wires(fmt, xs, D, flag)
    lines = oracle.ll128_lines(D) if fmt == "ll128" else oracle.ll_lines(D)
    line_bytes = 128 if fmt == "ll128" else 16
    flag_offsets = [120] if fmt == "ll128" else [4, 12]
    g = torch.Generator().manual_seed(N + W)
    planted = set()
    for i in range(n_stale):
        r = int(torch.randint(0, W, (1,), generator=g))
        k = int(torch.randint(0, lines, (1,), generator=g))
        if (r, k) in planted:
            continue
        off = flag_offsets[i % len(flag_offsets)]
        wires[r][k * line_bytes + off] ^= 0x02          # 7 -> 5: previous round's flag
        planted.add((r, k))
    ref = torch.empty_like(xs[0])
    n_ref, lst_ref = (oracle.ll128_decode_reduce if fmt == "ll128" else oracle.ll_decode_reduce)(
        wires, D, dtype, flag, ref)
    assert n_ref == len(planted) and {tuple(e) for e in lst_ref.tolist()} == planted
    with car.Car(W, M, N, dtype) as c:
        dw = [torch.from_numpy(wv[: (c.ll128_wire_bytes if fmt == "ll128" else c.ll_wire_bytes)]).to(DEV)
              for wv in wires]
        out = torch.full_like(xs[0], 3.0, device=DEV)
        for polls in (1, 4):
            (c.ll128_decode_reduce if fmt == "ll128" else c.ll_decode_reduce)(dw, flag, out, max_polls=polls)
            n, pairs = c.ll128_report() if fmt == "ll128" else c.ll_report()
            assert n == len(planted) and set(pairs) == planted
            assert_bits_equal(out, ref, f"{fmt} decode-reduce (max_polls={polls})")


def test_wire_report_cap_and_count(car):
    """More stale pairs than the caller's cap: the count is complete, the list
    holds cap distinct true entries."""
    W, M, N = 2, 4, 1200
    wl = workloads.custom(W, M, N, "bf16", seed=9)
    xs = [workloads.make_x(wl, r) for r in range(W)]
    D = wl.data_bytes
    with car.Car(W, M, N, "bf16") as c:
        wires = [torch.empty(c.ll128_wire_bytes, dtype=torch.uint8, device=DEV) for _ in range(W)]
        for x, wv in zip(xs, wires):
            c.ll128_encode(x.to(DEV), 6, wv)
        out = torch.empty_like(xs[0], device=DEV)
        c.ll128_decode_reduce(wires, 7, out)           # every line stale in every rank
        st, n, pairs = car.car_ll128_report(c.h, 10)
        assert st == car.CAR_ERR_STALE_FLAG and n == W * oracle.ll128_lines(D) and len(set(pairs)) == 10
        assert all(r < W and k < oracle.ll128_lines(D) for r, k in pairs)
        torch.cuda.synchronize()
        assert torch.count_nonzero(out.view(torch.int16)) == 0
        c.ll128_encode(xs[0].to(DEV), 7, wires[0])
        c.ll128_encode(xs[1].to(DEV), 7, wires[1])
        c.ll128_decode_reduce(wires, 7, out)
        assert car.car_ll128_report(c.h, 10)[:2] == (car.CAR_OK, 0)


# ---------------------------------------------------------------------------
# the configurations at full size, in the launch configuration bench.py uses
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["m1_w2", "m1_w8", "m512_w8", "m2048_w4_fp32"])
def test_workload_full_size(car, name):
    """Each configuration at full size, in bench.py's launch configuration
    (automatic kernel and shape): the plain reduce and the fused op against
    the oracle on every element of every output."""
    wl = workloads.WORKLOADS[name]
    W, M, N, dt = wl.W, wl.M, wl.N, wl.dtype
    dx, dres, dw = workloads.make_inputs(wl, DEV)
    ro, no = torch.empty_like(dres), torch.empty_like(dres)
    ar = torch.empty_like(dres) if wl.write_ar else None
    plain = torch.empty_like(dres)
    with car.Car(W, M, N, dt) as c:
        c.reduce(dx, plain)
        c.reduce_residual_rmsnorm(dx, dres, dw, wl.eps, ro, no, ar)
        c.sync()
    torch.cuda.synchronize()
    xs = [x.cpu() for x in dx]
    ref_ar, ref_ro, ref_no = oracle_fused(xs, dres.cpu(), dw.cpu(), wl.eps, M, N, dt)
    assert_bits_equal(plain, oracle_reduce(xs, dt), "plain reduce")
    if ar is not None:
        assert_bits_equal(ar, ref_ar, "ar")
    assert_bits_equal(ro, ref_ro, "residual_out")
    assert_norm_close(no, ref_no)


def _line_chunks(L, per=1 << 16):
    return [(k0, min(L, k0 + per)) for k0 in range(0, L, per)]


def _oracle_ll128_encode(data, D, flag, wire, pool):
    """The oracle's encode of one rank, cut at line boundaries: line k of a
    piece that starts at line k0 is line k0 + k of the whole message (every
    line holds its own 120 data bytes and flag), so the pieces run on
    several host threads."""
    def piece(k0, k1):
        d0, d1 = 120 * k0, min(D, 120 * k1)
        oracle.ll128_encode(data[d0:d1], d1 - d0, flag, wire[128 * k0:128 * k1])
    list(pool.map(lambda kk: piece(*kk), _line_chunks(oracle.ll128_lines(D))))


def _oracle_ll128_decode(wires, D, dtype, flag, out_u8, pool):
    """The oracle's validate + decode + reduce, cut at line boundaries as
    above; returns the stale (rank, line) pairs with whole-message line
    numbers."""
    def piece(k0, k1):
        d0, d1 = 120 * k0, min(D, 120 * k1)
        n, lst = oracle.ll128_decode_reduce([w[128 * k0:128 * k1] for w in wires], d1 - d0, dtype, flag,
                                            out_u8[d0:d1])
        assert n == len(lst)
        return {(int(r), int(k) + k0) for r, k in lst}
    stale = set()
    for part in pool.map(lambda kk: piece(*kk), _line_chunks(oracle.ll128_lines(D))):
        stale |= part
    return stale


def test_ll128_workload_full_size(car):
    """W=16, M=N=8192 bf16, flag 7, floor(L/4096) stale lines per rank:
    every wire byte of every rank equals the oracle's encode, and every
    output element and the stale set equal the oracle's validate + decode +
    reduce of its own wires with the same lines planted stale."""
    import concurrent.futures
    import os

    wl = workloads.WORKLOADS["ll128_w16"]
    W, M, N = wl.W, wl.M, wl.N
    D = wl.data_bytes
    L = oracle.ll128_lines(D)
    stale = workloads.stale_lines(L, W, wl.seed, wl.ll128_stale_every)
    old = list(wl.ll128_stale_flag.to_bytes(8, "little"))
    dx = [workloads.make_x(wl, r, DEV) for r in range(W)]
    with car.Car(W, M, N, "bf16") as c:
        wires = [torch.empty(c.ll128_wire_bytes, dtype=torch.uint8, device=DEV) for _ in range(W)]
        for x, wv in zip(dx, wires):
            c.ll128_encode(x, wl.ll128_flag, wv)
        torch.cuda.synchronize()
        pool = concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1)))
        owires = []
        for r in range(W):
            data = dx[r].cpu().view(-1).view(torch.uint8).numpy()
            ow = np.empty(c.ll128_wire_bytes, dtype=np.uint8)
            _oracle_ll128_encode(data, D, wl.ll128_flag, ow, pool)
            got = wires[r].cpu().numpy()
            if not np.array_equal(got, ow):
                first = int(np.nonzero(got != ow)[0][0])
                raise AssertionError(f"rank {r}: wire byte {first} (line {first // 128}) differs from the oracle's")
            owires.append(ow)
        for wv, ow, idx in zip(wires, owires, stale):
            wv.view(L, 16, 8)[idx.to(DEV), 15] = torch.tensor(old, dtype=torch.uint8, device=DEV)
            ow.reshape(L, 16, 8)[idx.numpy(), 15] = np.array(old, dtype=np.uint8)
        out = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
        c.ll128_decode_reduce(wires, wl.ll128_flag, out)
        n, pairs = c.ll128_report()
    torch.cuda.synchronize()
    planted = {(r, int(k)) for r, idx in enumerate(stale) for k in idx.tolist()}
    assert n == len(planted) == W * (L // 4096)
    assert set(pairs) == planted
    ref = np.empty(D, dtype=np.uint8)
    ref_stale = _oracle_ll128_decode(owires, D, "bf16", wl.ll128_flag, ref, pool)
    pool.shutdown()
    assert ref_stale == planted
    got = out.view(-1).view(torch.uint8).cpu().numpy()
    if not np.array_equal(got, ref):
        first = int(np.nonzero(got != ref)[0][0])
        raise AssertionError(f"output byte {first} (line {first // 120}) differs from the oracle's")


# ---------------------------------------------------------------------------
# launch ordering: programmatic dependent launch and CUDA-graph capture
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("M", [1, 3, 200])
def test_chained_calls_see_previous_outputs(car, M):
    """Back-to-back calls where each call's residual is the previous call's
    residual_out (and its rank 0 input the previous ar): every kernel waits
    for its predecessor before reading, so the chain equals the oracle chain."""
    W, N, steps = 4, 2048, 4
    wl, xs, res, w = _fused_inputs(W, M, N, "bf16", seed=900 + M)
    dx = [x.to(DEV) for x in xs]
    dres, dw = res.to(DEV), w.to(DEV)
    outs = [(torch.empty_like(dres), torch.empty_like(dres), torch.empty_like(dres)) for _ in range(steps)]
    with car.Car(W, M, N, "bf16") as c:
        cur_res, cur_x0 = dres, dx[0]
        for k in range(steps):
            ro, no, ar = outs[k]
            c.reduce_residual_rmsnorm([cur_x0] + dx[1:], cur_res, dw, wl.eps, ro, no, ar)
            cur_res, cur_x0 = ro, ar
        c.sync()
    torch.cuda.synchronize()
    ref_res, ref_x0 = res, xs[0]
    for k in range(steps):
        ref_ar, ref_ro, ref_no = oracle_fused([ref_x0] + xs[1:], ref_res, w, wl.eps, M, N, "bf16")
        ro, no, ar = outs[k]
        assert_bits_equal(ar, ref_ar, f"ar step {k}")
        assert_bits_equal(ro, ref_ro, f"residual_out step {k}")
        assert_norm_close(no, ref_no, f"norm_out step {k}")
        ref_res, ref_x0 = ref_ro, ref_ar


@pytest.mark.parametrize("M", [400, 700])
def test_chained_pipeline_calls_see_previous_outputs(car, M):
    """The pipelined fused kernel (more rows than SMs, 16 KB rows) behind a
    predecessor that writes its inputs: a plain reduce whose output is rank 0
    of the first fused call, then fused calls whose residual and rank 0 are
    the previous call's residual_out and ar.  Each launch may ask L2 for its
    first row while the predecessor still runs; every call must still read
    the predecessor's results."""
    W, N, steps = 8, 8192, 3
    wl, xs, res, w = _fused_inputs(W, M, N, "bf16", seed=960 + M)
    dx = [x.to(DEV) for x in xs]
    dres, dw = res.to(DEV), w.to(DEV)
    first = torch.full_like(dx[0], float("nan"))
    outs = [(torch.empty_like(dres), torch.empty_like(dres), torch.empty_like(dres)) for _ in range(steps)]
    with car.Car(W, M, N, "bf16") as c:
        c.reduce(dx, first)
        cur_res, cur_x0 = dres, first
        for k in range(steps):
            ro, no, ar = outs[k]
            c.reduce_residual_rmsnorm([cur_x0] + dx[1:], cur_res, dw, wl.eps, ro, no, ar)
            cur_res, cur_x0 = ro, ar
        c.sync()
    torch.cuda.synchronize()
    ref_res, ref_x0 = res, oracle_reduce(xs, "bf16")
    assert_bits_equal(first, ref_x0, "reduce before the chain")
    for k in range(steps):
        ref_ar, ref_ro, ref_no = oracle_fused([ref_x0] + xs[1:], ref_res, w, wl.eps, M, N, "bf16")
        ro, no, ar = outs[k]
        assert_bits_equal(ar, ref_ar, f"ar step {k}")
        assert_bits_equal(ro, ref_ro, f"residual_out step {k}")
        assert_norm_close(no, ref_no, f"norm_out step {k}")
        ref_res, ref_x0 = ref_ro, ref_ar


@pytest.mark.parametrize("M", [1919, 1920, 1921])
def test_ll128_encode_on_both_sides_of_the_streaming_size(car, M):
    """Aligned rank data whose wire reaches 32 MiB is encoded by the
    streaming instance (two loads in flight, evict-first stores), smaller
    data by the plain one: wires bit-identical to the oracle's below, at and
    above that size (N=8192 bf16; M=1921 ends in a partial line)."""
    N = 8192
    wl = workloads.custom(1, M, N, "bf16", seed=970 + M)
    x = workloads.make_x(wl, 0)
    D = wl.data_bytes
    with car.Car(1, M, N, "bf16") as c:
        wire = torch.empty(c.ll128_wire_bytes, dtype=torch.uint8, device=DEV)
        c.ll128_encode(x.to(DEV), 7, wire)
        torch.cuda.synchronize()
        assert (c.ll128_wire_bytes >= 32 << 20) == (M >= 1920)
    want = np.empty(oracle.ll128_wire_bytes(D), dtype=np.uint8)
    oracle.ll128_encode(x.view(-1).view(torch.uint8).numpy(), D, 7, want)
    got = wire.cpu().numpy()
    assert np.array_equal(got, want), f"first differing byte {int(np.nonzero(got != want)[0][0])}"


@pytest.mark.parametrize("kind", ["one_shot", "two_shot"])
@pytest.mark.parametrize("W,M,N", [(4, 33, 1032), (8, 512, 8192)])
def test_chained_reduces_see_previous_output(car, kind, W, M, N):
    """Back-to-back reduces where call k's rank-0 input is call k-1's output:
    each call's L2 prefetch runs before it waits for its predecessor, and
    every call must still read the predecessor's result."""
    steps = 4
    wl = workloads.custom(W, M, N, "bf16", seed=950 + W + M)
    xs = [workloads.make_x(wl, r) for r in range(W)]
    dx = [x.to(DEV) for x in xs]
    outs = [torch.full_like(dx[0], float("nan")) for _ in range(steps)]
    with car.Car(W, M, N, "bf16") as c:
        run = c.reduce if kind == "one_shot" else c.reduce_two_shot
        cur = dx[0]
        for k in range(steps):
            run([cur] + dx[1:], outs[k])
            cur = outs[k]
        c.sync()
    torch.cuda.synchronize()
    ref = xs[0]
    for k in range(steps):
        want = torch.empty_like(xs[0])
        (oracle.reduce if kind == "one_shot" else oracle.reduce_two_shot)([ref] + xs[1:], "bf16", want)
        assert_bits_equal(outs[k], want, f"{kind} step {k}")
        ref = want


@pytest.mark.parametrize("fmt", ["ll128", "ll"])
def test_graph_of_one_decode_reports_each_replay(car, fmt):
    """One decode captured in a CUDA graph: every replay, followed by a
    report, reports exactly the stale lines planted for that replay, and the
    output equals the oracle's decode of the same wires."""
    W, M, N = 3, 5, 1000
    wl = workloads.custom(W, M, N, "bf16", seed=1500)
    xs = [workloads.make_x(wl, r) for r in range(W)]
    D = wl.data_bytes
    lb = 128 if fmt == "ll128" else 16
    off = 120 if fmt == "ll128" else 4                   # the flag word (LL: flag1)
    with car.Car(W, M, N, "bf16") as c:
        nb = c.ll128_wire_bytes if fmt == "ll128" else c.ll_wire_bytes
        wires = [torch.empty(nb, dtype=torch.uint8, device=DEV) for _ in range(W)]
        enc = c.ll128_encode if fmt == "ll128" else c.ll_encode
        dec = c.ll128_decode_reduce if fmt == "ll128" else c.ll_decode_reduce
        rep = c.ll128_report if fmt == "ll128" else c.ll_report
        out = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        with torch.cuda.stream(side):
            dec(wires, 9, out, stream=side.cuda_stream)
            side.synchronize()
            rep()
            with torch.cuda.graph(g, stream=side):
                dec(wires, 9, out, stream=torch.cuda.current_stream().cuda_stream)
        L = nb // lb
        for trial, plan in enumerate(({0: [1, 7]}, {2: [0], 1: [L - 1, 3]}, {})):
            for x, wv in zip(xs, wires):
                enc(x.to(DEV), 9, wv)
            for r, ks in plan.items():
                for k in ks:
                    wires[r][k * lb + off] ^= 0x01
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()                       # the report waits only for the capture stream
            n, pairs = rep()
            planted = {(r, k) for r, ks in plan.items() for k in ks}
            assert n == len(planted) and set(pairs) == planted, f"replay {trial}"
            host = [wv.cpu().numpy() for wv in wires]
            ref = torch.empty_like(xs[0])
            (oracle.ll128_decode_reduce if fmt == "ll128" else oracle.ll_decode_reduce)(host, D, "bf16", 9, ref)
            assert_bits_equal(out, ref, f"{fmt} decode (replay {trial})")
        assert rep()[0] == 0                               # the report cleared what it returned
        del g


@pytest.mark.parametrize("M", [1, 400])
def test_graph_capture_replays_correctly(car, M):
    """Capture reduce + fused + LL128 encode/decode in one CUDA graph, change
    the inputs in place, replay: outputs follow the new inputs."""
    W, N = 8, 1024
    wl, xs, res, w = _fused_inputs(W, M, N, "bf16", seed=1300 + M)
    dx = [x.to(DEV) for x in xs]
    dres, dw = res.to(DEV), w.to(DEV)
    ar, ro, no, dec = (torch.empty_like(dres) for _ in range(4))
    c = car.Car(W, M, N, "bf16")
    wires = [torch.empty(c.ll128_wire_bytes, dtype=torch.uint8, device=DEV) for _ in range(W)]
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()

    def body(stream):
        c.reduce(dx, ar, stream=stream)
        c.reduce_residual_rmsnorm(dx, dres, dw, wl.eps, ro, no, stream=stream)
        for x, wv in zip(dx, wires):
            c.ll128_encode(x, 11, wv, stream=stream)
        c.ll128_decode_reduce(wires, 11, dec, stream=stream)

    with torch.cuda.stream(side):
        body(side.cuda_stream)
        side.synchronize()
        with torch.cuda.graph(g, stream=side):
            body(torch.cuda.current_stream().cuda_stream)
    for trial in range(2):
        new = workloads.make_inputs(workloads.custom(W, M, N, "bf16", seed=1400 + trial), "cpu")
        for d, h in zip(dx, new[0]):
            d.copy_(h)
        dres.copy_(new[1])
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        ref_ar, ref_ro, ref_no = oracle_fused(new[0], new[1], w, wl.eps, M, N, "bf16")
        assert_bits_equal(ar, ref_ar, "ar (graph)")
        assert_bits_equal(dec, ref_ar, "LL128 decode (graph)")
        assert_bits_equal(ro, ref_ro, "residual_out (graph)")
        assert_norm_close(no, ref_no, "norm_out (graph)")
    assert c.ll128_report()[0] == 0
    c.sync()
    c.close()
