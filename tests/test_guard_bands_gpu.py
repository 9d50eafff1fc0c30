"""Guard bands around every output: no kernel writes outside its buffers.

Each output sits inside a larger device buffer, 16-byte aligned, with bands
of a fixed byte before and after it.  After the call the bands must be
intact and the output must equal the oracle's.  Shapes are ragged: message
sizes that are not a whole number of CTA passes, rows split over clusters,
more rows than SMs, LL128 messages that end in a partial line.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
BAND = 512
FILL = 0xA5
TORCH = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


@pytest.fixture(scope="module")
def car():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import rank_sum_reduce_gb300 as car

    return car


class Guarded:
    """A device buffer of `nbytes` (viewed as `dtype` and `shape`) between two bands."""

    def __init__(self, nbytes, dtype=None, shape=None):
        self.nbytes = nbytes
        self.raw = torch.full((BAND + nbytes + BAND,), FILL, dtype=torch.uint8, device=DEV)
        inner = self.raw[BAND:BAND + nbytes]
        self.t = inner.view(dtype).view(shape) if dtype is not None else inner

    def check(self, what):
        host = self.raw.cpu()
        before, after = host[:BAND], host[BAND + self.nbytes:]
        assert bool((before == FILL).all()), f"{what}: {int((before != FILL).sum())} bytes written before the buffer"
        assert bool((after == FILL).all()), f"{what}: {int((after != FILL).sum())} bytes written after the buffer"


def _bits(t):
    t = t.detach().cpu().contiguous()
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


def _norm_ok(got, ref):
    g = got.detach().cpu().float().numpy().astype(np.float64)
    r = ref.detach().cpu().float().numpy().astype(np.float64)
    return bool(np.all(np.abs(g - r) <= 2.0**-7 * np.abs(r) + 1e-5))


@pytest.mark.parametrize("W,M,N,dtype", [(3, 7, 1000, "bf16"), (16, 5, 4100, "fp32"), (8, 513, 8192, "bf16"),
                                         (1, 1, 8, "fp16")])
def test_reduces_stay_inside_their_output(car, W, M, N, dtype):
    wl = workloads.custom(W, M, N, dtype, seed=3100 + M)
    xs = [workloads.make_x(wl, r) for r in range(W)]
    D = wl.data_bytes
    for kind in ("one_shot", "two_shot"):
        out = Guarded(D, TORCH[dtype], (M, N))
        with car.Car(W, M, N, dtype) as c:
            (c.reduce if kind == "one_shot" else c.reduce_two_shot)([x.to(DEV) for x in xs], out.t)
            c.sync()
        torch.cuda.synchronize()
        out.check(kind)
        want = torch.empty_like(xs[0])
        (oracle.reduce if kind == "one_shot" else oracle.reduce_two_shot)(xs, dtype, want)
        assert torch.equal(_bits(out.t), _bits(want)), kind


@pytest.mark.parametrize("W,M,N,dtype,kernel", [
    (8, 700, 8192, "bf16", "auto"),       # pipeline, partial last wave
    (4, 333, 4096, "fp32", "pipeline"),
    (3, 5, 1544, "fp16", "rows"),         # one CTA per row, ragged row
    (16, 2, 4096, "bf16", "rows"),        # rows split over a cluster
    (8, 16, 8192, "bf16", "auto"),        # clusters of 8, one row each
    (2, 1, 8, "bf16", "auto"),            # a single 16-byte vector
])
def test_fused_op_stays_inside_its_outputs(car, W, M, N, dtype, kernel):
    wl = workloads.custom(W, M, N, dtype, seed=3200 + M)
    xs, res, w = workloads.make_inputs(wl)
    D = wl.data_bytes
    ro, no, ar = (Guarded(D, TORCH[dtype], (M, N)) for _ in range(3))
    with car.Car(W, M, N, dtype) as c:
        if kernel != "auto":
            c.tune_fused(car.CAR_FUSED_ROWS if kernel == "rows" else car.CAR_FUSED_PIPELINE)
        c.reduce_residual_rmsnorm([x.to(DEV) for x in xs], res.to(DEV), w.to(DEV), wl.eps, ro.t, no.t, ar.t)
        c.sync()
    torch.cuda.synchronize()
    for g, name in ((ro, "residual_out"), (no, "norm_out"), (ar, "ar")):
        g.check(name)
    rar, rro, rno = (torch.empty_like(res) for _ in range(3))
    oracle.reduce_residual_rmsnorm(xs, res, w, wl.eps, M, N, dtype, rro, rno, ar_out=rar)
    assert torch.equal(_bits(ar.t), _bits(rar)) and torch.equal(_bits(ro.t), _bits(rro))
    assert _norm_ok(no.t, rno)


@pytest.mark.parametrize("fmt", ["ll128", "ll"])
@pytest.mark.parametrize("W,M,N,dtype", [(3, 7, 1000, "bf16"), (2, 3, 1164, "fp32"), (16, 2, 520, "fp16")])
def test_wire_kernels_stay_inside_their_buffers(car, fmt, W, M, N, dtype):
    """Encode writes only its wire, decode only its output (LL128 messages
    here end in a partial line), with a stale line planted in one rank."""
    wl = workloads.custom(W, M, N, dtype, seed=3300 + M + W)
    xs = [workloads.make_x(wl, r) for r in range(W)]
    D = wl.data_bytes
    with car.Car(W, M, N, dtype) as c:
        nb = c.ll128_wire_bytes if fmt == "ll128" else c.ll_wire_bytes
        enc = c.ll128_encode if fmt == "ll128" else c.ll_encode
        dec = c.ll128_decode_reduce if fmt == "ll128" else c.ll_decode_reduce
        rep = c.ll128_report if fmt == "ll128" else c.ll_report
        wires = [Guarded(nb) for _ in range(W)]
        for x, g in zip(xs, wires):
            enc(x.to(DEV), 5, g.t)
        torch.cuda.synchronize()
        for i, g in enumerate(wires):
            g.check(f"{fmt} wire {i}")
        line = 128 if fmt == "ll128" else 16
        flag_at = 120 if fmt == "ll128" else 4
        wires[W - 1].t[(nb // line - 1) * line + flag_at] ^= 0x01      # the last line of the last rank is stale
        out = Guarded(D, TORCH[dtype], (M, N))
        dec([g.t for g in wires], 5, out.t)
        n, pairs = rep()
    torch.cuda.synchronize()
    out.check(f"{fmt} decode output")
    assert n == 1 and set(pairs) == {(W - 1, nb // line - 1)}
    ref = torch.empty_like(xs[0])
    host = [g.t.cpu().numpy() for g in wires]
    n_ref, _ = (oracle.ll128_decode_reduce if fmt == "ll128" else oracle.ll_decode_reduce)(host, D, dtype, 5, ref)
    assert n_ref == 1 and torch.equal(_bits(out.t), _bits(ref))


def test_lamport_receive_stays_inside_its_outputs(car):
    W, M, N = 4, 3, 1544
    wl = workloads.custom(W, M, N, "bf16", seed=3400)
    xs, res, w = workloads.make_inputs(wl)
    D = wl.data_bytes
    with car.Car(W, M, N, "bf16") as c:
        comm = Guarded(c.lamport_buffer_bytes)
        c.lamport_init(comm.t)
        for r in range(W):
            c.lamport_push(xs[r].to(DEV), r, 2, comm.t)
        ro, no, ar = (Guarded(D, torch.bfloat16, (M, N)) for _ in range(3))
        c.lamport_reduce_residual_rmsnorm(comm.t, 2, res.to(DEV), w.to(DEV), wl.eps, ro.t, no.t, ar.t)
        n, _ = c.lamport_report()
        c.sync()
    torch.cuda.synchronize()
    assert n == 0
    for g, name in ((comm, "comm"), (ro, "residual_out"), (no, "norm_out"), (ar, "ar")):
        g.check(name)
    rar, rro, rno = (torch.empty_like(res) for _ in range(3))
    oracle.reduce_residual_rmsnorm(xs, res, w, wl.eps, M, N, "bf16", rro, rno, ar_out=rar)
    # pushes turn -0.0 into +0.0; N(0,1) data holds no -0.0, so the sums equal the fused op's
    assert torch.equal(_bits(ar.t), _bits(rar)) and torch.equal(_bits(ro.t), _bits(rro))
    assert _norm_ok(no.t, rno)
