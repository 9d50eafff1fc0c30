"""Exhaustive pin of the oracle's two-rank bf16 rank sum (CPU, about a
minute): every pair (a, b) of non-NaN bf16 values, 2^32 less the NaN
patterns, summed by the oracle and by a separate C check written here.

The check's formulation differs from the oracle's at both steps:
  * the add: a and b are exact in float64 and so is their sum's rounding to
    fp32 -- float((double)a + (double)b) equals the IEEE fp32 add because
    53 >= 2*24 + 2 (no harmful double rounding);
  * the narrowing: round-to-nearest-even to bf16 by the carry-add on the
    fp32 bit pattern, (u + 0x7FFF + ((u >> 16) & 1)) >> 16, instead of the
    oracle's rounding from an exact (sign, significand, exponent) value.
inf + -inf must give a NaN; NaN payloads are not pinned.
"""
import ctypes
import subprocess

CHECK_C = r"""
#include <stdint.h>
#include <string.h>

typedef void (*reduce_fn)(int, const void* const*, int, int64_t, void*);

static float widen(uint16_t h) {
  const uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}
static int is_nan16(uint16_t h) { return (h & 0x7F80u) == 0x7F80u && (h & 0x7Fu) != 0; }
static uint16_t narrow_rne(float f) {  /* f is not a NaN */
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)(u >> 16);  /* +-inf */
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* Returns the number of mismatching pairs; *compared gets the pairs checked. */
uint64_t check_all_pairs(reduce_fn reduce, int bf16_code, uint64_t* compared) {
  static uint16_t a[65536], b[65536], out[65536];
  uint64_t bad = 0, n = 0;
  for (uint32_t i = 0; i < 65536; i++) a[i] = (uint16_t)i;
  for (uint32_t j = 0; j < 65536; j++) {
    if (is_nan16((uint16_t)j)) continue;
    for (uint32_t i = 0; i < 65536; i++) b[i] = (uint16_t)j;
    const void* x[2] = {a, b};
    reduce(2, x, bf16_code, 65536, out);
    const double fb = (double)widen((uint16_t)j);
    for (uint32_t i = 0; i < 65536; i++) {
      if (is_nan16((uint16_t)i)) continue;
      const float s = (float)((double)widen((uint16_t)i) + fb);
      n++;
      if (s != s) {
        if (!is_nan16(out[i])) bad++;
      } else if (out[i] != narrow_rne(s)) {
        bad++;
      }
    }
  }
  *compared = n;
  return bad;
}
"""


def test_every_bf16_pair_sums_like_the_fp32_add(orc, tmp_path):
    src = tmp_path / "pairs_check.c"
    lib_path = tmp_path / "libpairs_check.so"
    src.write_text(CHECK_C)
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-shared", "-fPIC", str(src), "-o", str(lib_path)],
                   check=True)
    check = ctypes.CDLL(str(lib_path))
    check.check_all_pairs.restype = ctypes.c_uint64
    check.check_all_pairs.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_uint64)]
    reduce_ptr = ctypes.cast(orc.default().lib().orc_reduce, ctypes.c_void_p)
    compared = ctypes.c_uint64(0)
    bad = check.check_all_pairs(reduce_ptr, orc.DTYPE_CODE["bf16"], ctypes.byref(compared))
    non_nan = 65536 - 2 * 127                 # NaN patterns: exponent 0xFF, mantissa != 0, both signs
    assert compared.value == non_nan * non_nan
    assert bad == 0, f"{bad} of {compared.value} bf16 pairs differ from the fp32 add"
