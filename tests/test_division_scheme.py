"""The quantiser divides each element by its block divisor d with a
correctly rounded reciprocal and one FMA residual correction (Markstein's
scheme) instead of an IEEE division, and claims the result is the IEEE
quotient whenever 2^-70 <= d < 2^126, |x| >= 2^-96 and |q| >= 2^-100 (the
kernel takes the IEEE division outside that range).  This test restates
that arithmetic in C, compiled for the host with FMA contraction off, and
compares it with IEEE division on structured and random cases: every
positive BF16 x against divisors d = e4m3 * s, and random FP32 x and d with
mantissas near all-ones.  It does not run the CUDA code; the GPU parity
tests compare the kernel with the oracle bit for bit."""
import os
import subprocess
import tempfile

import pytest

SRC = r"""
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
static uint64_t st = 0x9E3779B97F4A7C15ull;
static uint64_t rnd(void) { st ^= st << 13; st ^= st >> 7; st ^= st << 17; return st; }
static float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static double e4m3(int b) { int e = (b >> 3) & 15, m = b & 7; return e ? ldexp(1.0 + m / 8.0, e - 7) : ldexp(m, -9); }
/* one residual correction, as in the kernel: q0 - RN(q0 d - x) * rd */
static float div_fast(float x, float d, float rd) {
  float q0 = x * rd;
  return fmaf(-fmaf(q0, d, -x), rd, q0);
}
static int in_range(float x, float d, float q) {
  return d >= 0x1p-70f && d < 0x1p126f && fabsf(x) >= 0x1p-96f && fabsf(q) >= 0x1p-100f;
}
int main(void) {
  long long n = 0, bad = 0;
  /* every positive BF16 x, d = e4m3 * s for structured and random s */
  for (int si = 0; si < 24; ++si) {
    uint32_t sm = si < 8 ? 0x7FFFFF - si : (si < 12 ? (uint32_t)(si - 8) : (uint32_t)(rnd() & 0x7FFFFF));
    int se = 90 + (int)(rnd() % 60);
    float s = u2f(sm | ((uint32_t)se << 23));
    for (int b = 1; b < 127; b += 3) {
      float d = (float)e4m3(b) * s, rd = 1.0f / d;
      for (uint32_t h = 1; h < 0x7F80; ++h) {
        float x = u2f(h << 16);
        if (x > 16.0f * d) break;
        float q = div_fast(x, d, rd), ref = x / d;
        if (!in_range(x, d, x * rd)) continue;
        ++n;
        if (f2u(q) != f2u(ref)) { if (bad < 5) printf("x=%a d=%a ref=%a got=%a\n", x, d, ref, q); ++bad; }
      }
    }
  }
  /* random FP32 x (the transform's outputs are not BF16), divisor mantissas near all-ones */
  for (long long it = 0; it < 20000000LL; ++it) {
    uint64_t r = rnd();
    uint32_t dm = (it & 3) == 0 ? (0x7FFFFF - (uint32_t)(r & 0xFF)) : (uint32_t)(r & 0x7FFFFF);
    float d = u2f(dm | ((uint32_t)(58 + (r >> 40) % 182) << 23));
    float x = u2f((uint32_t)rnd() & 0x7FFFFFFF);
    if (!isfinite(x)) continue;
    if (x > 9.0f * d) x = d * (float)((rnd() % 9000) / 1000.0);
    float rd = 1.0f / d;
    if (!in_range(x, d, x * rd)) continue;
    ++n;
    float q = div_fast(x, d, rd), ref = x / d;
    if (f2u(q) != f2u(ref)) { if (bad < 10) printf("x=%a d=%a ref=%a got=%a\n", x, d, ref, q); ++bad; }
    /* the negative side and signed zero */
    if (f2u(div_fast(-x, d, rd)) != f2u(-x / d)) ++bad;
  }
  if (f2u(div_fast(-0.0f, 3.0f, 1.0f / 3.0f)) != f2u(-0.0f)) ++bad;
  if (f2u(div_fast(0.0f, 3.0f, 1.0f / 3.0f)) != f2u(0.0f)) ++bad;
  printf("checked %lld mismatches %lld\n", n, bad);
  return bad != 0;
}
"""


def test_residual_corrected_division_is_ieee_in_range():
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "div.c")
        exe = os.path.join(d, "div")
        with open(c, "w") as f:
            f.write(SRC)
        try:
            subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-o", exe, c, "-lm"], check=True,
                           capture_output=True)
        except (OSError, subprocess.CalledProcessError) as e:
            pytest.skip("no host C compiler: %s" % e)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
        assert r.returncode == 0, r.stdout + r.stderr
        n = int(r.stdout.split()[1])
        assert n > 10_000_000, r.stdout


SRC_SCALE = r"""
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
static uint64_t st = 0xD1B54A32D192ED03ull;
static uint64_t rnd(void) { st ^= st << 13; st ^= st >> 7; st ^= st << 17; return st; }
static float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float div_fast(float x, float d, float rd) {
  float q0 = x * rd;
  return fmaf(-fmaf(q0, d, -x), rd, q0);
}
/* the block-scale argument as the kernel computes it: t = (bamax / 6) / s by
   two residual-corrected divisions when bamax >= 2^-93 and s in [2^-70,
   2^126), clamped at 2^100 (E4M3 saturates far below), else IEEE divisions */
static float t_fast(float x, float s) {
  float rs = 1.0f / s;
  if (s >= 0x1p-70f && s < 0x1p126f && x >= 0x1p-93f) {
    float d1 = div_fast(x, 6.0f, 0x1.555556p-3f);
    float t = div_fast(d1, s, rs);
    return t <= 0x1p100f ? t : 0x1p100f;
  }
  float t = (x / 6.0f) / s;  /* the IEEE path; E4M3 saturates above 464 either way */
  return t <= 0x1p100f ? t : 0x1p100f;
}
static float t_ieee(float x, float s) {
  float t = (x / 6.0f) / s;
  return t <= 0x1p100f ? t : 0x1p100f;
}
/* what decides an E4M3 code: equal values, or both below 2^-11 (code 0) */
static int same_code_input(float a, float b) {
  if (f2u(a) == f2u(b)) return 1;
  return a < 0x1p-11f && b < 0x1p-11f;
}
int main(void) {
  long long n = 0, bad = 0;
  if (0x1.555556p-3f != 1.0f / 6.0f) { printf("constant\n"); return 1; }
  /* every positive finite BF16 block maximum against structured and random s */
  for (int si = 0; si < 40; ++si) {
    uint32_t sm = si < 8 ? 0x7FFFFF - si : (si < 12 ? (uint32_t)(si - 8) : (uint32_t)(rnd() & 0x7FFFFF));
    int se = 1 + (int)(rnd() % 253);
    float s = u2f(sm | ((uint32_t)se << 23));
    for (uint32_t h = 1; h < 0x7F80; ++h) {
      float x = u2f(h << 16);
      ++n;
      float a = t_fast(x, s), b = t_ieee(x, s);
      if (!same_code_input(a, b)) { if (bad < 5) printf("x=%a s=%a ieee=%a got=%a\n", x, s, b, a); ++bad; }
    }
  }
  /* random FP32 block maxima (transform outputs) and random s */
  for (long long it = 0; it < 30000000LL; ++it) {
    uint64_t r = rnd();
    float x = u2f((uint32_t)(r & 0x7FFFFFFF));
    float s = u2f((uint32_t)((rnd() & 0x7FFFFF) | ((1 + rnd() % 253) << 23)));
    if (!isfinite(x)) continue;
    ++n;
    float a = t_fast(x, s), b = t_ieee(x, s);
    if (!same_code_input(a, b)) { if (bad < 10) printf("x=%a s=%a ieee=%a got=%a\n", x, s, b, a); ++bad; }
  }
  printf("checked %lld mismatches %lld\n", n, bad);
  return bad != 0;
}
"""


def test_block_scale_divisions_match_ieee():
    """The block-scale argument t = (bamax / 6) / s, as the quantiser computes
    it with two residual-corrected divisions (constant reciprocals of 6 and
    of s) and a clamp at 2^100, equals the IEEE value wherever the E4M3
    conversion can tell them apart (any value below 2^-11 encodes as 0)."""
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "scale.c")
        exe = os.path.join(d, "scale")
        with open(c, "w") as f:
            f.write(SRC_SCALE)
        try:
            subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-o", exe, c, "-lm"], check=True,
                           capture_output=True)
        except (OSError, subprocess.CalledProcessError) as e:
            pytest.skip("no host C compiler: %s" % e)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
        assert r.returncode == 0, r.stdout + r.stderr
        n = int(r.stdout.split()[1])
        assert n > 10_000_000, r.stdout
