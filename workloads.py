"""Seeded synthetic inputs for the rank-sum reduce hot path.

This module draws random numbers and lays out tensors; it holds none of the
method's arithmetic (no sums, no rounding choices, no wire formats).  Both the
CUDA path's tests/bench and the oracle's checks take their inputs from here.

Distributions follow the workload table of the configurations:

* ``m1_w2``   W=2,  M=1,    N=2048, bf16; x_r, residual ~ N(0,1); weight ~ U(0.5,1.5); eps 1e-6
* ``m1_w8``   W=8,  M=1,    N=8192, bf16; same distributions; eps 1e-6
* ``m512_w8`` W=8,  M=512,  N=8192, bf16; x_r ~ N(0,0.5), residual ~ N(0,1); eps 1e-5
* ``m2048_w4_fp32`` W=4, M=2048, N=4096, fp32; x_r ~ U(-1,1) with 1% of entries x1e3
* ``ll128_w16`` W=16, M=8192, N=8192, bf16; x_r ~ N(0,1); LL128 wire with flag 7,
  floor(L/4096) lines per rank carrying the stale flag 6

bf16/fp16 values are drawn in fp32 and cast by torch; the seed of every tensor
is derived from (workload seed, tensor role, rank) so that any subset of the
tensors can be regenerated on its own.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

TORCH_DTYPE = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}
ELEM_SIZE = {"bf16": 2, "fp16": 2, "fp32": 4}


@dataclass(frozen=True)
class Workload:
    name: str
    W: int
    M: int
    N: int
    dtype: str
    eps: float
    seed: int
    x_dist: str = "normal"      # "normal" | "uniform_outliers"
    x_sigma: float = 1.0
    outlier_p: float = 0.01
    outlier_scale: float = 1e3
    write_ar: bool = False      # the fused call also writes ar
    ll128_flag: int | None = None
    ll128_stale_flag: int | None = None
    ll128_stale_every: int | None = None
    notes: str = field(default="", compare=False)

    @property
    def data_bytes(self) -> int:
        return self.M * self.N * ELEM_SIZE[self.dtype]


WORKLOADS = {
    "m1_w2": Workload("m1_w2", W=2, M=1, N=2048, dtype="bf16", eps=1e-6, seed=0, write_ar=True,
                      notes="decode bs=1, two ranks; fused call writes ar, residual_out, norm_out"),
    "m1_w8": Workload("m1_w8", W=8, M=1, N=8192, dtype="bf16", eps=1e-6, seed=1,
                      notes="decode bs=1 latency regime, 16 KB per rank"),
    "m512_w8": Workload("m512_w8", W=8, M=512, N=8192, dtype="bf16", eps=1e-5, seed=2, x_sigma=0.5,
                        notes="8 MB per rank message; plain reduce and fused reduce+RMSNorm"),
    "m2048_w4_fp32": Workload("m2048_w4_fp32", W=4, M=2048, N=4096, dtype="fp32", eps=1e-6, seed=3,
                              x_dist="uniform_outliers", notes="fp32 with 1% outliers x1e3"),
    "ll128_w16": Workload("ll128_w16", W=16, M=8192, N=8192, dtype="bf16", eps=1e-6, seed=4,
                          ll128_flag=7, ll128_stale_flag=6, ll128_stale_every=4096,
                          notes="LL128 wire per rank, flag 7, 1/4096 lines stale (flag 6)"),
}

# tensor roles, mixed into the per-tensor seed
_ROLE = {"x": 1, "residual": 2, "weight": 3, "stale": 4, "outlier": 5}


def tensor_seed(seed: int, role: str, rank: int = 0) -> int:
    """Per-tensor seed: a fixed mix of (workload seed, role, rank)."""
    return (seed * 1_000_003 + _ROLE[role] * 10_007 + rank * 101 + 12345) & 0x7FFF_FFFF_FFFF


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, sigma, device, seed):
    return torch.randn(shape, generator=_gen(device, seed), device=device, dtype=torch.float32) * sigma


def _uniform(shape, lo, hi, device, seed):
    return torch.rand(shape, generator=_gen(device, seed), device=device, dtype=torch.float32) * (hi - lo) + lo


def make_x(wl: Workload, rank: int, device="cpu", M: int | None = None, N: int | None = None) -> torch.Tensor:
    """Rank r's contribution x_r, shape [M, N], in the workload's dtype."""
    M = wl.M if M is None else M
    N = wl.N if N is None else N
    s = tensor_seed(wl.seed, "x", rank)
    if wl.x_dist == "normal":
        v = _normal((M, N), wl.x_sigma, device, s)
    elif wl.x_dist == "uniform_outliers":
        v = _uniform((M, N), -1.0, 1.0, device, s)
        pick = _uniform((M, N), 0.0, 1.0, device, tensor_seed(wl.seed, "outlier", rank)) < wl.outlier_p
        v = torch.where(pick, v * wl.outlier_scale, v)
    else:
        raise ValueError(wl.x_dist)
    return v.to(TORCH_DTYPE[wl.dtype])


def make_residual(wl: Workload, device="cpu", M: int | None = None, N: int | None = None) -> torch.Tensor:
    M = wl.M if M is None else M
    N = wl.N if N is None else N
    return _normal((M, N), 1.0, device, tensor_seed(wl.seed, "residual")).to(TORCH_DTYPE[wl.dtype])


def make_weight(wl: Workload, device="cpu", N: int | None = None) -> torch.Tensor:
    N = wl.N if N is None else N
    return _uniform((N,), 0.5, 1.5, device, tensor_seed(wl.seed, "weight")).to(TORCH_DTYPE[wl.dtype])


def make_inputs(wl: Workload, device="cpu", M: int | None = None, N: int | None = None):
    """(xs, residual, weight) for the workload, optionally at another [M, N]."""
    xs = [make_x(wl, r, device, M, N) for r in range(wl.W)]
    return xs, make_residual(wl, device, M, N), make_weight(wl, device, N)


def custom(W: int, M: int, N: int, dtype: str, seed: int, eps: float = 1e-6, x_sigma: float = 1.0,
           x_dist: str = "normal") -> Workload:
    """An ad-hoc workload for parity cases (ragged tails, odd W, other dtypes)."""
    return Workload(f"custom_w{W}_m{M}_n{N}_{dtype}_s{seed}", W=W, M=M, N=N, dtype=dtype, eps=eps,
                    seed=seed, x_sigma=x_sigma, x_dist=x_dist)


def stale_lines(n_lines: int, W: int, seed: int, every: int) -> list[torch.Tensor]:
    """Per rank, floor(n_lines/every) distinct line indices (sorted), seeded per rank."""
    k = n_lines // every
    out = []
    for r in range(W):
        perm = torch.randperm(n_lines, generator=_gen("cpu", tensor_seed(seed, "stale", r)))
        out.append(torch.sort(perm[:k]).values)
    return out
