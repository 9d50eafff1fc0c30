"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, never against the oracle itself or the CUDA path.

Each test names the kind of pin it is:
  * library routine  -- numpy/torch conversions (IEEE round-half-to-even)
  * independent formulation -- frexp / rint / ldexp rounding, float64 exact sums
  * closed form      -- W identical ranks, integer-valued inputs, constant rows
  * brute force      -- every bf16 value against a structured partner set
  * page value       -- line layouts and buffer tables printed on the pages
                        (fixtures under tests/golden/)
  * reading          -- a documented reading of an ambiguous passage

Pages: P1 "SGLang Custom AllReduce v1 线程模型和工作原理细节"; P2 "NCCL 专家课程 14：
Simple、LL、LL128 的线格式、同步与真实性能边界"; P3 "0-custom-all-reduce"; P4 "用 Triton +
Symmetric Memory 写一个 AllReduce + RMSNorm 融合算子".
"""
import itertools
import os

import numpy as np
import pytest
import torch

from conftest import GOLDEN, read_golden

# ----------------------------------------------------------------------------
# test-side helpers (independent of oracle.c)
# ----------------------------------------------------------------------------
FMT = {"bf16": (8, -126, 127), "fp16": (11, -14, 15), "fp32": (24, -126, 127)}


def frexp_round(x, kind):
    """Round float64 values to a binary format by scaling: frexp -> rint -> ldexp.

    rint rounds half to even; scaling by powers of two is exact in float64 for
    every value reachable here, so this is a second, independent formulation of
    IEEE round-to-nearest-even with gradual underflow and overflow to inf."""
    p, emin, emax = FMT[kind]
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    fin = np.isfinite(x) & (x != 0)
    _, e = np.frexp(x[fin])
    E = e - 1
    q = np.maximum(E, emin) - (p - 1)
    r = np.ldexp(np.rint(np.ldexp(x[fin], -q)), q)
    big = np.abs(r) >= np.ldexp(1.0, emax + 1)
    r[big] = np.copysign(np.inf, r[big])
    out[fin] = r
    return out


def bits_of(value64, kind):
    """Bit pattern of a float64 value that is exactly representable in `kind`."""
    if kind == "bf16":
        return (value64.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    if kind == "fp16":
        return value64.astype(np.float16).view(np.uint16)
    return value64.astype(np.float32).view(np.uint32)


def torch_bf16_bits(f32):
    return torch.from_numpy(np.ascontiguousarray(f32, dtype=np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def all_patterns16():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)


def finite16(kind):
    p = all_patterns16()
    if kind == "bf16":
        f = (p.astype(np.uint32) << 16).view(np.float32)
    else:
        f = p.view(np.float16).astype(np.float32)
    return p[np.isfinite(f)]


def widen(bits, kind):
    if kind == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32)
    return bits.view(np.float16).astype(np.float32)


def same_bits_or_both_nan(a_bits, b_bits, kind):
    a, b = widen(a_bits, kind), widen(b_bits, kind)
    nan = np.isnan(a) & np.isnan(b)
    return np.all((a_bits == b_bits) | nan)


# ----------------------------------------------------------------------------
# conversions
# ----------------------------------------------------------------------------
def test_bf16_widening_every_pattern(orc):
    """library routine: torch's bf16 -> fp32 over all 2^16 patterns."""
    p = all_patterns16()
    got = orc.convert(p, "bf16", "fp32")
    ref = torch.from_numpy(p.view(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got.view(np.uint32)[~nan], ref.view(np.uint32)[~nan])


def test_f16_widening_every_pattern(orc):
    """library routine: numpy's float16 -> float32 over all 2^16 patterns."""
    p = all_patterns16()
    got = orc.convert(p, "fp16", "fp32")
    ref = p.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got.view(np.uint32)[~nan], ref.view(np.uint32)[~nan])


def _rounding_class_f32_for_bf16():
    """Every bf16 'kept' pattern x every class of dropped low half: 0, 1, just
    below half, exactly half (tie), just above half, all ones, and random."""
    hi = all_patterns16().astype(np.uint32)
    rng = np.random.default_rng(7)
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
    lows = np.concatenate([lows, rng.integers(0, 1 << 16, size=6, dtype=np.uint32)])
    u = (hi[:, None] << 16 | lows[None, :]).ravel()
    f = u.view(np.float32)
    return f[~np.isnan(f)]


def test_f32_to_bf16_every_rounding_class(orc):
    """library routine (torch RNE) and independent formulation (frexp/rint)."""
    f = _rounding_class_f32_for_bf16()
    got = orc.convert(f, "fp32", "bf16")
    assert np.array_equal(got, torch_bf16_bits(f))
    assert np.array_equal(got, bits_of(frexp_round(f.astype(np.float64), "bf16"), "bf16"))


def test_f32_to_f16_boundaries(orc):
    """library routine: numpy float32 -> float16 at every binary16 midpoint and
    its fp32 neighbours, plus random values over the whole fp32 range."""
    h = finite16("fp16")
    v = h.view(np.float16).astype(np.float64)
    v = np.unique(v)
    mids = (v[:-1] + v[1:]) / 2.0   # exact in float64, and in float32 as well
    m32 = mids.astype(np.float32)
    cands = [m32, np.nextafter(m32, np.float32(np.inf)), np.nextafter(m32, np.float32(-np.inf)),
             v.astype(np.float32)]
    rng = np.random.default_rng(11)
    cands.append(rng.integers(0, 1 << 32, size=200_000, dtype=np.uint64).astype(np.uint32).view(np.float32))
    cands.append(np.float32([65504.0, 65519.99, 65520.0, 65536.0, 2.0**-24, 2.0**-25, 3 * 2.0**-26,
                             2.0**-14, 1e-30, -1e-30]))
    f = np.concatenate(cands)
    f = f[~np.isnan(f)]
    with np.errstate(over="ignore"):
        ref = f.astype(np.float16).view(np.uint16)
    got = orc.convert(f, "fp32", "fp16")
    assert np.array_equal(got, ref)


def _doubles_for_narrowing(kind):
    rng = np.random.default_rng(13)
    p, emin, emax = FMT[kind]
    e = rng.integers(emin - p - 3, emax + 3, size=100_000)
    m = rng.uniform(1.0, 2.0, size=e.size) * rng.choice([-1.0, 1.0], size=e.size)
    x = np.ldexp(m, e)
    # exact ties: odd multiples of half a quantum in every binade
    k = rng.integers(1 << (p - 1), 1 << p, size=20_000)
    et = rng.integers(emin - p + 1, emax - p + 1, size=k.size)
    ties = np.ldexp(2.0 * k + 1.0, et - 1)
    return np.concatenate([x, ties, -ties, [0.0, -0.0, np.inf, -np.inf, 1e308, 5e-324]])


@pytest.mark.parametrize("kind", ["bf16", "fp16", "fp32"])
def test_f64_narrowing(orc, kind):
    """independent formulation for all three; numpy's correctly rounded
    float64 -> float32/float16 casts as a library routine for two of them."""
    x = _doubles_for_narrowing(kind)
    got = orc.convert(x, "fp64", kind)
    if kind == "fp32":
        got = got.view(np.uint32)
    want = bits_of(frexp_round(x, kind), kind)
    assert np.array_equal(got, want)
    if kind in ("fp16", "fp32"):
        with np.errstate(over="ignore"):
            lib = x.astype(np.float16 if kind == "fp16" else np.float32)
        assert np.array_equal(got, lib.view(np.uint16 if kind == "fp16" else np.uint32))


# ----------------------------------------------------------------------------
# one-shot rank sum  (P1 "1stage：kernel 全文与时间线", P3 "4. 求和")
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("kind", ["bf16", "fp16"])
@pytest.mark.parametrize("W", [1, 2, 3, 4, 8, 16])
def test_reduce_identical_ranks_is_W_times_x(orc, kind, W):
    """closed form: W identical ranks sum to W*x.  Every partial k*x of a
    16-bit value fits in fp32 exactly, so the only rounding is the last one."""
    x = finite16(kind)
    out = np.empty_like(x)
    orc.reduce([x] * W, kind, out)
    exact = widen(x, kind).astype(np.float64) * W
    with np.errstate(over="ignore"):
        f32 = exact.astype(np.float32)
        want = torch_bf16_bits(f32) if kind == "bf16" else f32.astype(np.float16).view(np.uint16)
    assert np.array_equal(out, want)


@pytest.mark.parametrize("W", [1, 2, 3])
def test_reduce_identical_ranks_fp32(orc, W):
    """closed form: for fp32, x+x is exact and (2x)+x is 3x rounded once."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal(50_000).astype(np.float32) * np.float32(1e3)
    out = np.empty_like(x)
    orc.reduce([x] * W, "fp32", out)
    assert np.array_equal(out.view(np.uint32), (x.astype(np.float64) * W).astype(np.float32).view(np.uint32))


@pytest.mark.parametrize("kind", ["bf16", "fp16", "fp32"])
def test_reduce_integer_values_exact_and_rank_order_free(orc, kind):
    """closed form: integer-valued inputs |v| <= 256 sum exactly in fp32 in any
    order, so the result is the integer sum rounded once, and permuting the
    ranks changes no bit."""
    rng = np.random.default_rng(5)
    W, n = 16, 40_000
    ints = rng.integers(-256, 257, size=(W, n))
    f = ints.astype(np.float32)
    xs = [torch_bf16_bits(f[r]) if kind == "bf16" else (f[r].astype(np.float16).view(np.uint16)
          if kind == "fp16" else f[r].copy()) for r in range(W)]
    out = np.empty_like(xs[0])
    orc.reduce(xs, kind, out)
    total = ints.sum(axis=0).astype(np.float32)
    want = torch_bf16_bits(total) if kind == "bf16" else (total.astype(np.float16).view(np.uint16)
                                                          if kind == "fp16" else total)
    assert np.array_equal(out.view(want.dtype), want)
    perm = rng.permutation(W)
    out2 = np.empty_like(out)
    orc.reduce([xs[i] for i in perm], kind, out2)
    assert np.array_equal(out, out2)


@pytest.mark.parametrize("kind", ["bf16", "fp16"])
def test_reduce_single_rank_is_identity(orc, kind):
    """closed form: W = 1 returns every finite input bit for bit (-0 included)."""
    x = finite16(kind)
    out = np.empty_like(x)
    orc.reduce([x], kind, out)
    assert np.array_equal(out, x)


@pytest.mark.parametrize("kind", ["bf16", "fp16"])
def test_reduce_pairs_brute_force(orc, kind):
    """brute force: every finite 16-bit value a against a structured set of
    partners b (every exponent, both signs, subnormals, extremes).  Independent
    formulation: a+b is exact in float64, and rounding that to fp32 equals the
    fp32 add (53 >= 2*24+2); then the library's rounding to the element type."""
    a = finite16(kind)
    p = all_patterns16()
    fin = finite16(kind)
    rng = np.random.default_rng(17)
    expo_reps = p[(p & 0x7F) == 0x01] if kind == "bf16" else p[(p & 0x3FF) == 0x001]
    b = np.unique(np.concatenate([fin[rng.integers(0, fin.size, 256)], np.intersect1d(expo_reps, fin),
                                  np.array([0x0000, 0x8000, 0x0001, 0x8001], dtype=np.uint16)]))
    A = np.repeat(a, b.size)
    B = np.tile(b, a.size)
    out = np.empty_like(A)
    orc.reduce([A, B], kind, out)
    with np.errstate(over="ignore", invalid="ignore"):
        s = (widen(A, kind).astype(np.float64) + widen(B, kind).astype(np.float64)).astype(np.float32)
        want = torch_bf16_bits(s) if kind == "bf16" else s.astype(np.float16).view(np.uint16)
    assert same_bits_or_both_nan(out, want, kind)


def test_reduce_negative_zero_seed(orc):
    """reading (P1's kernel seeds the accumulator with rank 0's value, P3's
    pseudocode with +0): all ranks -0 give -0; any +0 among them gives +0."""
    neg = np.full(4, 0x8000, dtype=np.uint16)
    pos = np.zeros(4, dtype=np.uint16)
    out = np.empty(4, dtype=np.uint16)
    orc.reduce([neg, neg, neg], "bf16", out)
    assert np.all(out == 0x8000)
    orc.reduce([neg, pos, neg], "bf16", out)
    assert np.all(out == 0x0000)


def test_reduce_keeps_subnormals(orc):
    """closed form: gradual underflow is kept (no flush to zero)."""
    x = np.float32([2.0**-140, 2.0**-149, -(2.0**-130)])
    out = np.empty_like(x)
    orc.reduce([x, x], "fp32", out)
    assert np.array_equal(out, np.float32([2.0**-139, 2.0**-148, -(2.0**-129)]))
    b = np.uint16([0x0001, 0x0040])           # bf16 subnormals 2^-133, 2^-127
    outb = np.empty_like(b)
    orc.reduce([b, b], "bf16", outb)
    assert np.array_equal(outb, np.uint16([0x0002, 0x0080]))


# ----------------------------------------------------------------------------
# fused reduce + residual + RMSNorm  (P4 "这个算子在算什么")
# ----------------------------------------------------------------------------
def _fused(orc, xs, res, w, eps, M, N, kind):
    ro = np.empty_like(res)
    no = np.empty_like(res)
    ar = np.empty_like(res)
    f64 = np.empty(M * N, dtype=np.float64)
    orc.reduce_residual_rmsnorm(xs, res, w, eps, M, N, kind, ro, no, ar_out=ar, norm_f64=f64)
    return ar, ro, no, f64.reshape(M, N)


def _bf16(f32):
    return torch_bf16_bits(np.asarray(f32, dtype=np.float32))


def test_fused_zero_x_passes_residual_through(orc):
    """closed form: x = +0 on every rank gives ar = +0 and residual_out equal
    to residual bit for bit (residual drawn without -0)."""
    rng = np.random.default_rng(19)
    M, N = 3, 256
    res = _bf16(rng.standard_normal(M * N))
    res[res == 0x8000] = 0
    w = _bf16(rng.uniform(0.5, 1.5, N))
    z = np.zeros(M * N, dtype=np.uint16)
    ar, ro, _, _ = _fused(orc, [z] * 4, res, w, 1e-6, M, N, "bf16")
    assert np.all(ar == 0)
    assert np.array_equal(ro, res)


@pytest.mark.parametrize("kind", ["bf16", "fp16", "fp32"])
def test_fused_zero_x_is_textbook_rmsnorm(orc, kind):
    """special case that is a textbook routine: with x = 0 the op is
    RMSNorm(residual) = residual / sqrt(mean(residual^2) + eps) * weight,
    written here with numpy in float64 as a division (the oracle multiplies by
    the reciprocal).  norm_out must be that value rounded once."""
    rng = np.random.default_rng(23)
    M, N, eps = 4, 512, 1e-5
    r64 = rng.standard_normal((M, N))
    w64 = rng.uniform(0.5, 1.5, N)
    if kind == "fp32":
        res, w = r64.astype(np.float32).ravel(), w64.astype(np.float32)
    elif kind == "fp16":
        res, w = r64.astype(np.float16).view(np.uint16).ravel(), w64.astype(np.float16).view(np.uint16)
    else:
        res, w = _bf16(r64.ravel()), _bf16(w64)
    z = np.zeros_like(res)
    _, _, no, f64 = _fused(orc, [z, z], res, w, eps, M, N, kind)
    rv = widen(res, kind).reshape(M, N).astype(np.float64) if kind != "fp32" else res.reshape(M, N).astype(np.float64)
    wv = widen(w, kind).astype(np.float64) if kind != "fp32" else w.astype(np.float64)
    eps32 = float(np.float32(eps))
    ref = rv / np.sqrt(np.mean(rv * rv, axis=1, keepdims=True) + eps32) * wv
    np.testing.assert_allclose(f64, ref, rtol=1e-13, atol=0)
    no_bits = no.view(np.uint32) if kind == "fp32" else no
    assert np.array_equal(no_bits, bits_of(frexp_round(f64.ravel(), kind), kind))


@pytest.mark.parametrize("c", [0.375, -1.5, 3.0, -0.125, 40.0])
def test_fused_constant_row_normalises_to_sign_times_weight(orc, c):
    """closed form: a constant row h = c gives (c / sqrt(c^2 + eps)) * w, which
    is sign(c) * w within eps / (2 c^2) relative."""
    N, eps = 1024, 1e-6
    rng = np.random.default_rng(29)
    x0 = _bf16(np.full(N, c))
    z = np.zeros(N, dtype=np.uint16)
    w = _bf16(rng.uniform(0.5, 1.5, N))
    _, ro, no, f64 = _fused(orc, [x0, z, z], z, w, eps, 1, N, "bf16")
    assert np.all(widen(ro, "bf16") == np.float32(c))
    wv = widen(w, "bf16").astype(np.float64)
    rel = np.abs(f64[0] - np.sign(c) * wv) / wv
    assert rel.max() <= float(np.float32(eps)) / (2 * c * c) * 1.0001 + 1e-15


def test_fused_scale_invariance(orc):
    """closed form: doubling every input (exact in bf16) doubles h and leaves
    norm_out unchanged up to the eps term: ratio - 1 <= eps / mean(h^2)."""
    rng = np.random.default_rng(31)
    M, N, eps = 2, 2048, 1e-6
    xs = [_bf16(rng.standard_normal(M * N)) for _ in range(3)]
    res = _bf16(rng.standard_normal(M * N))
    w = _bf16(rng.uniform(0.5, 1.5, N))
    dbl = lambda b: _bf16(widen(b, "bf16") * 2)  # noqa: E731
    _, ro1, _, f1 = _fused(orc, xs, res, w, eps, M, N, "bf16")
    _, ro2, _, f2 = _fused(orc, [dbl(x) for x in xs], dbl(res), w, eps, M, N, "bf16")
    assert np.array_equal(widen(ro2, "bf16"), 2 * widen(ro1, "bf16"))
    ms = np.mean(widen(ro1, "bf16").reshape(M, N).astype(np.float64) ** 2, axis=1, keepdims=True)
    assert np.all(np.abs(f2 / f1 - 1.0) <= float(np.float32(eps)) / ms + 1e-14)


def test_fused_single_column(orc):
    """closed form: N = 1 gives h / sqrt(h^2 + eps) * w."""
    vals = [0.5, -2.0, 1e-3, 7.0]
    for v in vals:
        x = _bf16([v])
        z = np.zeros(1, dtype=np.uint16)
        w = _bf16([1.25])
        _, ro, _, f64 = _fused(orc, [x, z], z, w, 1e-6, 1, 1, "bf16")
        h = float(widen(ro, "bf16")[0])
        eps32 = float(np.float32(1e-6))
        want = h / np.sqrt(h * h + eps32) * 1.25
        assert f64[0, 0] == pytest.approx(want, rel=1e-15)


def test_fused_rows_are_independent(orc):
    """closed form: each row's outputs equal a one-row call on that row alone
    (catches statistics leaking across rows or a wrong row stride)."""
    rng = np.random.default_rng(37)
    M, N = 5, 384
    xs = [_bf16(rng.standard_normal(M * N)) for _ in range(2)]
    res = _bf16(rng.standard_normal(M * N))
    w = _bf16(rng.uniform(0.5, 1.5, N))
    ar, ro, no, _ = _fused(orc, xs, res, w, 1e-6, M, N, "bf16")
    for m in range(M):
        sl = slice(m * N, (m + 1) * N)
        ar1, ro1, no1, _ = _fused(orc, [x[sl].copy() for x in xs], res[sl].copy(), w, 1e-6, 1, N, "bf16")
        assert np.array_equal(ar[sl], ar1) and np.array_equal(ro[sl], ro1) and np.array_equal(no[sl], no1)


def test_fused_residual_uses_unrounded_sum(orc):
    """reading (P4 "总体设计": fp32 sum, then add residual): h is formed from
    the fp32 rank sum before it is rounded to bf16.  x0 = 1, x1 = 2^-9,
    residual = 2^-8: the fp32 h is 1 + 3*2^-9 -> bf16 1 + 2^-7, while the
    rounded sum (1.0) + 2^-8 would tie down to 1.0."""
    x0, x1, r = _bf16([1.0]), _bf16([2.0**-9]), _bf16([2.0**-8])
    w = _bf16([1.0])
    ar, ro, _, _ = _fused(orc, [x0, x1], r, w, 1e-6, 1, 1, "bf16")
    assert ar[0] == 0x3F80                  # 1 + 2^-9 rounds to 1.0
    assert ro[0] == 0x3F81                  # 1 + 2^-7


# ----------------------------------------------------------------------------
# LL128 and LL wire formats  (P2)
# ----------------------------------------------------------------------------
def test_protocol_buffer_table(orc):
    """page value: default buffers and data per FIFO step (NCCL_STEPS = 8)."""
    rows = {}
    with open(os.path.join(GOLDEN, "protocol_buffers.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                name, *vals = line.split()
                rows[name] = vals
    ll = rows["LL"]
    ll128 = rows["LL128"]
    # columns: line_bytes, data_per_line, efficiency, default_buffer, wire_per_step, data_per_step
    for row, cap, wire in ((ll, orc.ll_data_capacity, orc.ll_wire_bytes),
                           (ll128, orc.ll128_data_capacity, orc.ll128_wire_bytes)):
        line, per_line, eff, buf, wire_step, data_step = row
        assert int(buf) // 8 == int(wire_step)
        assert cap(int(wire_step)) == int(data_step)
        assert cap(int(line)) == int(per_line)
        assert cap(int(line)) / int(line) == float(eff)
        assert wire(int(per_line)) == int(line)


def test_ll128_golden_lines(orc):
    """page value: the line layout worked from P2's definition (word 15 = flag)."""
    for case in read_golden("ll128_line.txt"):
        D = int(case["data_bytes"])
        flag = int(case["flag_hex"], 16)
        if case.get("data") == "iota":
            data = np.arange(D, dtype=np.uint8)
            want = np.concatenate([data, np.frombuffer(flag.to_bytes(8, "little"), dtype=np.uint8)])
        else:
            data = np.frombuffer(bytes.fromhex(case["data_hex"]), dtype=np.uint8).copy()
            want = np.frombuffer(bytes.fromhex(case["wire_hex"].replace(" ", "")), dtype=np.uint8)
        wire = np.full(orc.ll128_wire_bytes(D), 0xEE, dtype=np.uint8)
        orc.ll128_encode(data, D, flag, wire)
        assert np.array_equal(wire, want)


def test_ll_golden_line(orc):
    """page value: {data1, flag1, data2, flag2} for one 8-byte word."""
    (case,) = read_golden("ll_line.txt")
    data = np.frombuffer(bytes.fromhex(case["data_hex"]), dtype=np.uint8).copy()
    wire = np.zeros(16, dtype=np.uint8)
    orc.ll_encode(data, 8, int(case["flag"]), wire)
    assert wire.tobytes() == bytes.fromhex(case["wire_hex"].replace(" ", ""))
    # decode: data1 + (data2 << 32) gives back the word (W = 1, fp32 view of its two halves)
    out = np.zeros(2, dtype=np.float32)
    n, _ = orc.ll_decode_reduce([wire], 8, "fp32", int(case["flag"]), out)
    assert n == 0 and out.tobytes() == data.tobytes()


def _rand_bf16_bytes(rng, D):
    v = _bf16(rng.standard_normal(D // 2))
    return v


@pytest.mark.parametrize("fmt", ["ll128", "ll"])
def test_wire_round_trip_brute_force(orc, fmt):
    """brute force: for every even size D = 0..512 bytes, W = 1..3 and flags
    {0, 1, 2^31 or 2^63, all ones}: decode(encode(x)) reduces to exactly the
    plain rank sum of x, reports nothing stale, and for W = 1 returns x."""
    enc = orc.ll128_encode if fmt == "ll128" else orc.ll_encode
    dec = orc.ll128_decode_reduce if fmt == "ll128" else orc.ll_decode_reduce
    wb = orc.ll128_wire_bytes if fmt == "ll128" else orc.ll_wire_bytes
    top = 63 if fmt == "ll128" else 31
    flags = [0, 1, 1 << top, (1 << (top + 1)) - 1]
    rng = np.random.default_rng(41)
    for D in range(0, 514, 2):
        for W in (1, 2, 3):
            xs = [_rand_bf16_bytes(rng, D) for _ in range(W)]
            for flag in flags:
                wires = []
                for x in xs:
                    wire = np.zeros(max(wb(D), 1), dtype=np.uint8)
                    enc(x, D, flag, wire)
                    wires.append(wire)
                out = np.full(max(D // 2, 1), 0xDEAD, dtype=np.uint16)
                n, _ = dec(wires, D, "bf16", flag, out)
                assert n == 0
                want = np.empty_like(out)
                if D:
                    orc.reduce([x for x in xs], "bf16", want[: D // 2])
                    assert np.array_equal(out[: D // 2], want[: D // 2])
                    if W == 1:
                        assert np.array_equal(out[: D // 2], xs[0])


@pytest.mark.parametrize("fmt", ["ll128", "ll"])
def test_each_single_stale_line_detected_alone(orc, fmt):
    """brute force: every single (rank, line) whose flag is off is reported,
    alone; only that line's elements are zeroed, the rest equal the sum."""
    enc = orc.ll128_encode if fmt == "ll128" else orc.ll_encode
    dec = orc.ll128_decode_reduce if fmt == "ll128" else orc.ll_decode_reduce
    nl = orc.ll128_lines if fmt == "ll128" else orc.ll_lines
    line_bytes, data_per_line = (128, 120) if fmt == "ll128" else (16, 8)
    flag_off = 120 if fmt == "ll128" else 4
    D = 5 * data_per_line + 40 if fmt == "ll128" else 11 * 8
    rng = np.random.default_rng(43)
    W, flag = 3, 7
    xs = [_rand_bf16_bytes(rng, D) for _ in range(W)]
    base = []
    for x in xs:
        wire = np.zeros(nl(D) * line_bytes, dtype=np.uint8)
        enc(x, D, flag, wire)
        base.append(wire)
    full = np.empty(D // 2, dtype=np.uint16)
    orc.reduce(xs, "bf16", full)
    for r, k in itertools.product(range(W), range(nl(D))):
        wires = [b.copy() for b in base]
        wires[r][k * line_bytes + flag_off] ^= 0x01       # first flag byte off by one bit
        out = np.empty(D // 2, dtype=np.uint16)
        n, lst = dec(wires, D, "bf16", flag, out)
        assert n == 1 and lst.tolist() == [[r, k]]
        lo, hi = k * data_per_line // 2, min(D, (k + 1) * data_per_line) // 2
        assert np.all(out[lo:hi] == 0)
        keep = np.ones(D // 2, dtype=bool)
        keep[lo:hi] = False
        assert np.array_equal(out[keep], full[keep])


def test_ll_second_flag_alone_is_checked(orc):
    """page value: readLL waits until flag1 AND flag2 equal the expected flag,
    so a line with only flag2 off is stale too."""
    x = np.arange(8, dtype=np.uint8)
    wire = np.zeros(16, dtype=np.uint8)
    orc.ll_encode(x, 8, 9, wire)
    for off in (4, 12):
        bad = wire.copy()
        bad[off] = 8
        out = np.zeros(4, dtype=np.uint16)
        n, lst = orc.ll_decode_reduce([bad], 8, "bf16", 9, out)
        assert n == 1 and lst.tolist() == [[0, 0]] and np.all(out == 0)


def test_ll128_only_the_flag_word_is_checked(orc):
    """reading (P2: only the flag lane's second word is compared): a changed
    data word is not detected and flows into the sum."""
    rng = np.random.default_rng(47)
    D = 240
    x = _rand_bf16_bytes(rng, D)
    wire = np.zeros(orc.ll128_wire_bytes(D), dtype=np.uint8)
    orc.ll128_encode(x, D, 5, wire)
    wire[8] ^= 0x40                                    # word 1 of line 0
    out = np.empty(D // 2, dtype=np.uint16)
    n, _ = orc.ll128_decode_reduce([wire], D, "bf16", 5, out)
    assert n == 0 and out[4] != x[4] and np.array_equal(np.delete(out, 4), np.delete(x, 4))


def test_stale_list_cap(orc):
    """the count keeps going past the list's capacity; the list stops."""
    D = 120 * 10
    x = np.zeros(D // 2, dtype=np.uint16)
    wire = np.zeros(orc.ll128_wire_bytes(D), dtype=np.uint8)
    orc.ll128_encode(x, D, 3, wire)
    out = np.empty(D // 2, dtype=np.uint16)
    n, lst = orc.ll128_decode_reduce([wire, wire], D, "bf16", 4, out, cap=7)
    assert n == 20 and lst.shape == (7, 2)
    assert lst.tolist() == [[r, k] for k in range(10) for r in range(2)][:7]


# ----------------------------------------------------------------------------
# two-shot bit pattern  (P1 "2stage：分片、轮转、以及为什么没有出口 barrier")
# ----------------------------------------------------------------------------
def _owners(orc, W, units, probe_units):
    """For each probed unit, the ranks r such that the plain rank sum taken in
    the order r, r+1, ..., r-1 reproduces the two-shot result there.  fp32
    inputs spread over many binades make the order visible in the rounding;
    candidates are intersected over several independent draws."""
    n = units * 4
    owners = {u: set(range(W)) for u in probe_units}
    for seed in range(6):
        rng = np.random.default_rng(12345 + seed)
        xs = [(rng.standard_normal(n) * np.exp2(rng.integers(-12, 13, n))).astype(np.float32) for _ in range(W)]
        out = np.empty(n, dtype=np.float32)
        orc.reduce_two_shot(xs, "fp32", out)
        for u in probe_units:
            sl = slice(u * 4, (u + 1) * 4)
            for r in list(owners[u]):
                want = np.empty(4, dtype=np.float32)
                orc.reduce([xs[(r + k) % W][sl].copy() for k in range(W)], "fp32", want)
                if not np.array_equal(want.view(np.uint32), out[sl].view(np.uint32)):
                    owners[u].discard(r)
    return {u: sorted(c) for u, c in owners.items()}


def test_two_shot_shards_match_the_page(orc):
    """page value: a 512 KB message over 8 ranks has part = 4096 units; the
    owner (first rank of the sum) changes at unit 4096; the last rank owns the
    remainder."""
    (case,) = read_golden("two_shot_shards.txt")
    W, units = int(case["W"]), int(case["units"])
    assert int(case["message_bytes"]) // 16 == units and units // W == int(case["part"])
    keys = ("4095", "4096", "32767")
    owners = _owners(orc, W, units, [int(k) for k in keys])
    for key in keys:
        assert owners[int(key)] == [int(case[f"owner_of_unit_{key}"])]


@pytest.mark.parametrize("W,units", [(1, 7), (3, 10), (4, 2), (5, 23), (8, 8), (16, 40)])
def test_two_shot_is_rotated_one_shot_per_shard(orc, W, units):
    """closed form: each shard equals the plain rank sum over the rank list
    rotated to start at its owner; part = 0 gives everything to the last rank."""
    rng = np.random.default_rng(W * 100 + units)
    n = units * 4   # fp32: 4 elements per 16-byte unit, spread over many binades so order shows
    xs = [(rng.standard_normal(n) * np.exp2(rng.integers(-12, 13, n))).astype(np.float32) for _ in range(W)]
    out = np.empty(n, dtype=np.float32)
    orc.reduce_two_shot(xs, "fp32", out)
    part = units // W
    for u in range(units):
        owner = W - 1 if part == 0 else min(u // part, W - 1)
        rot = [xs[(owner + k) % W][u * 4:(u + 1) * 4].copy() for k in range(W)]
        want = np.empty(4, dtype=np.float32)
        orc.reduce(rot, "fp32", want)
        assert np.array_equal(out[u * 4:(u + 1) * 4].view(np.uint32), want.view(np.uint32))


def test_two_shot_equals_one_shot_on_exact_inputs(orc):
    """closed form: integer-valued inputs sum exactly in any order."""
    rng = np.random.default_rng(9)
    W, n = 6, 6000
    xs = [rng.integers(-256, 257, n).astype(np.float32) for _ in range(W)]
    a, b = np.empty(n, dtype=np.float32), np.empty(n, dtype=np.float32)
    orc.reduce(xs, "fp32", a)
    orc.reduce_two_shot(xs, "fp32", b)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("kind", ["fp32", "bf16"])
def test_reduce_is_sequential_fp32_adds_in_rank_order(orc, kind):
    """independent formulation: numpy float32 adds (IEEE binary32, round to
    nearest even), applied rank by rank from rank 0, then the library's
    rounding to the element type.  Values spread over many binades make the
    rank order visible in the rounding, so a reordered sum fails here."""
    rng = np.random.default_rng(77)
    W, n = 8, 20000
    f = [(rng.standard_normal(n) * np.exp2(rng.integers(-10, 11, n))).astype(np.float32) for _ in range(W)]
    xs = f if kind == "fp32" else [torch_bf16_bits(v) for v in f]
    vals = f if kind == "fp32" else [widen(b, "bf16") for b in xs]
    acc = vals[0].copy()
    for r in range(1, W):
        acc = (acc + vals[r]).astype(np.float32)
    out = np.empty_like(xs[0])
    orc.reduce(xs, kind, out)
    if kind == "fp32":
        assert np.array_equal(out.view(np.uint32), acc.view(np.uint32))
    else:
        assert np.array_equal(out, torch_bf16_bits(acc))
    rev = acc = vals[W - 1].copy()
    for r in range(W - 2, -1, -1):
        rev = (rev + vals[r]).astype(np.float32)
    assert not np.array_equal(rev.view(np.uint32), out.view(np.uint32) if kind == "fp32" else widen(out, kind).view(np.uint32))


# ----------------------------------------------------------------------------
# Lamport one-shot push  (P4 "方案二：Lamport（负零轮询）")
# ----------------------------------------------------------------------------
def _lamport_case():
    (case,) = read_golden("lamport.txt")
    return case


def test_lamport_sentinel_and_scrub_match_the_page(orc):
    """page value: sentinel 0x80008000, -0.0 scrubbed to +0.0, pair packing."""
    case = _lamport_case()
    assert orc.LAMPORT_SENTINEL == int(case["sentinel_hex"], 16)
    buf = np.zeros(4, dtype=np.uint32)
    orc.lamport_fill(buf)
    assert np.all(buf == int(case["sentinel_hex"], 16))
    pair = np.array([int(h, 16) for h in case["pair_hex"].split()], dtype=np.uint16)
    W, n = 1, 2
    comm = np.zeros(3 * W * n, dtype=np.uint16)
    orc.lamport_push(pair, n, comm, W, 0, 0)
    assert comm[:2].view(np.uint32)[0] == int(case["word_hex"], 16)


def test_lamport_push_never_writes_the_sentinel(orc):
    """brute force: every bf16 pattern as either half of a word; only -0.0
    changes (to +0.0), so no pushed word can equal the sentinel."""
    p = all_patterns16()
    n = p.size
    comm = np.zeros(3 * n, dtype=np.uint16)
    orc.lamport_push(p, n, comm, 1, 0, 0)
    got = comm[:n]
    want = p.copy()
    want[want == 0x8000] = 0
    assert np.array_equal(got, want)
    words = np.concatenate([got, got[::-1]]).reshape(-1, 2).copy().view(np.uint32)
    assert not np.any(words == orc.LAMPORT_SENTINEL)


def test_lamport_round_equals_fused_op_on_scrubbed_inputs(orc):
    """closed form through a pinned function: a complete round gives exactly
    the fused rank sum + residual + RMSNorm of the scrubbed inputs, reports
    nothing, and refills the previous round's region with the sentinel while
    leaving the next one alone."""
    rng = np.random.default_rng(51)
    W, M, N = 4, 3, 256
    xs = [_bf16(rng.standard_normal(M * N)) for _ in range(W)]
    xs[1][:7] = 0x8000                                     # some -0.0 to scrub
    res = _bf16(rng.standard_normal(M * N))
    w = _bf16(rng.uniform(0.5, 1.5, N))
    comm = np.zeros(3 * W * M * N, dtype=np.uint16)
    orc.lamport_fill(comm.view(np.uint32))
    rnd = 4                                                # region 1; refills region 0; region 2 untouched
    region = lambda k: comm[k * W * M * N:(k + 1) * W * M * N]  # noqa: E731
    region(0)[:] = 0x1234
    region(2)[:] = 0x5678
    for r in range(W):
        orc.lamport_push(xs[r], M * N, comm, W, r, rnd)
    ro, no, ar = (np.empty(M * N, dtype=np.uint16) for _ in range(3))
    n, _ = orc.lamport_reduce_residual_rmsnorm(W, comm, rnd, M, N, res, w, 1e-6, ro, no, ar)
    assert n == 0
    scrubbed = [np.where(x == 0x8000, 0, x).astype(np.uint16) for x in xs]
    ar2, ro2, no2 = (np.empty(M * N, dtype=np.uint16) for _ in range(3))
    orc.reduce_residual_rmsnorm(scrubbed, res, w, 1e-6, M, N, "bf16", ro2, no2, ar_out=ar2)
    assert np.array_equal(ar, ar2) and np.array_equal(ro, ro2) and np.array_equal(no, no2)
    assert np.all(region(0).view(np.uint32) == orc.LAMPORT_SENTINEL)   # (4 + 2) % 3 = 0
    assert np.all(region(2) == 0x5678)


@pytest.mark.parametrize("missing", [(0, 0, 0), (2, 1, 255), (1, 2, 128)])
def test_lamport_missing_word_makes_its_row_stale(orc, missing):
    """brute force on small inputs: one word still holding the sentinel makes
    exactly that (rank, row) stale; the row's outputs are 0; other rows are
    unaffected."""
    rng = np.random.default_rng(53)
    W, M, N = 3, 3, 256
    xs = [_bf16(rng.standard_normal(M * N)) for _ in range(W)]
    res = _bf16(rng.standard_normal(M * N))
    w = _bf16(rng.uniform(0.5, 1.5, N))
    comm = np.zeros(3 * W * M * N, dtype=np.uint16)
    orc.lamport_fill(comm.view(np.uint32))
    for r in range(W):
        orc.lamport_push(xs[r], M * N, comm, W, r, 0)
    rank, row, word = missing
    off = (rank * M * N + row * N + 2 * (word // 2))
    comm[off:off + 2] = [0x8000, 0x8000]
    ro, no, ar = (np.full(M * N, 7, dtype=np.uint16) for _ in range(3))
    n, lst = orc.lamport_reduce_residual_rmsnorm(W, comm, 0, M, N, res, w, 1e-6, ro, no, ar)
    assert n == 1 and lst.tolist() == [[rank, row]]
    sl = slice(row * N, (row + 1) * N)
    assert np.all(ro[sl] == 0) and np.all(no[sl] == 0) and np.all(ar[sl] == 0)
    keep = np.ones(M * N, dtype=bool)
    keep[sl] = False
    ro2, no2, ar2 = (np.empty(M * N, dtype=np.uint16) for _ in range(3))
    orc.reduce_residual_rmsnorm(xs, res, w, 1e-6, M, N, "bf16", ro2, no2, ar_out=ar2)
    assert np.array_equal(ro[keep], ro2[keep]) and np.array_equal(no[keep], no2[keep])
