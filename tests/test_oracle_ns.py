"""Pins for the oracle's Newton-Schulz step with NVFP4 products (CPU only).

Checked against facts fixed outside the oracle's code:
  * FP64 -> BF16 rounding: the result is the nearest BF16 value (its two
    neighbours are no closer), exact midpoints go to the even pattern, and on
    FP32 inputs it agrees with torch's FP32 -> BF16 conversion;
  * the FP32 combination a x + b y against numpy FP32 arithmetic;
  * a signed partial permutation matrix is a fixed point of the iteration
    whenever a + b + c = 1 (its polar factor is itself), and every NVFP4 step
    on it is exact, so the step must return it bit for bit, with A = I and
    B = (b + c) I along the way;
  * with (a, b, c) = (1, 0, 0) the step is the identity;
  * three steps from a well-conditioned random start stay close to the same
    three steps in plain FP64 arithmetic (the NVFP4 iteration error is a few
    percent; the pages report about 3 % with clipping).
"""
import numpy as np
import torch

import oracle


def _f(u16):
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).double().numpy()


def _bits(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


def _bf16_value(bits):
    return float(_f(np.array([bits], dtype=np.uint16))[0])


def test_bf16_rne_f64_is_nearest_with_ties_to_even():
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.standard_normal(2000) * np.exp2(rng.integers(-140, 120, 2000)),
                           rng.standard_normal(200) * 1e-40])
    for d in vals:
        b = oracle.bf16_rne_f64(d)
        v = _bf16_value(b)
        mag = b & 0x7FFF
        for nb in (mag - 1, mag + 1):
            if 0 <= nb < 0x7F80:
                w = _bf16_value(nb | (b & 0x8000))
                assert abs(d - v) <= abs(d - w)
                if abs(d - v) == abs(d - w):
                    assert (b & 1) == 0
    # exact midpoints between neighbouring BF16 values go to the even one
    for lo in (0x3F80, 0x3F81, 0x0001, 0x0002, 0x4B7F, 0x7F7E):
        mid = 0.5 * (_bf16_value(lo) + _bf16_value(lo + 1))
        assert oracle.bf16_rne_f64(mid) == (lo if lo % 2 == 0 else lo + 1)
        assert oracle.bf16_rne_f64(-mid) == 0x8000 | (lo if lo % 2 == 0 else lo + 1)
    # on FP32 values: one rounding, as torch's FP32 -> BF16 conversion
    f = rng.standard_normal(5000).astype(np.float32) * np.float32(3.7)
    got = np.array([oracle.bf16_rne_f64(float(v)) for v in f], dtype=np.uint16)
    assert np.array_equal(got, _bits(f))


def test_axpby_is_fp32_arithmetic_rounded_to_bf16():
    rng = np.random.default_rng(2)
    x = _bits(rng.standard_normal(4096))
    y = _bits(rng.standard_normal(4096) * 30)
    a, b = np.float32(1.875), np.float32(-0.3125)
    ref = (a * _f(x).astype(np.float32)) + (b * _f(y).astype(np.float32))
    assert np.array_equal(oracle.axpby_bf16(x, y, a, b), _bits(ref.astype(np.float32)))


QUINTIC = (15.0 / 8.0, -10.0 / 8.0, 3.0 / 8.0)  # degree-5 Newton-Schulz: f(s) = (15 s - 10 s^3 + 3 s^5) / 8


def _signed_partial_permutation(m, n, seed):
    rng = np.random.default_rng(seed)
    x = np.zeros((m, n), dtype=np.float32)
    cols = rng.permutation(n)[:m]
    x[np.arange(m), cols] = rng.choice([-1.0, 1.0], size=m)
    return _bits(x)


def test_partial_permutation_is_a_fixed_point():
    for m, n in ((32, 64), (64, 96)):
        x = _signed_partial_permutation(m, n, seed=m + n)
        out, tr = oracle.ns_step(x, *QUINTIC, p=100.0)
        assert np.array_equal(out, x)
        assert np.array_equal(_f(tr["a"]), np.eye(m))
        assert np.array_equal(_f(tr["a2"]), np.eye(m))
        assert np.array_equal(_f(tr["b"]), (QUINTIC[1] + QUINTIC[2]) * np.eye(m))
        # with a + b + c = 2 the step doubles it
        out2, _ = oracle.ns_step(x, 2.0 * QUINTIC[0], 2.0 * QUINTIC[1], 2.0 * QUINTIC[2], p=100.0)
        assert np.array_equal(_f(out2), 2.0 * _f(x))


def test_identity_coefficients_leave_the_iterate_unchanged():
    rng = np.random.default_rng(3)
    x = _bits(rng.standard_normal((64, 128)) * 0.01)
    out, _ = oracle.ns_step(x, 1.0, 0.0, 0.0, p=99.0)
    assert np.array_equal(_f(out), _f(x))


def _ns_fp64(x, a, b, c, steps):
    for _ in range(steps):
        A = x @ x.T
        x = a * x + (b * A + c * A @ A) @ x
    return x


def test_three_steps_track_the_fp64_iteration():
    rng = np.random.default_rng(4)
    m, n = 64, 192
    g = rng.standard_normal((m, n))
    x0 = g / np.linalg.norm(g)  # spectral norm <= Frobenius norm = 1
    x = _bits(x0)
    for _ in range(3):
        x, _ = oracle.ns_step(x, *QUINTIC, p=99.0)
    ref = _ns_fp64(_f(_bits(x0)), *QUINTIC, steps=3)
    err = np.linalg.norm(_f(x) - ref) / np.linalg.norm(ref)
    assert err < 0.08, err
    # and the iteration moved: the singular values grew toward 1
    assert np.linalg.svd(_f(x), compute_uv=False).min() > 2 * np.linalg.svd(x0, compute_uv=False).min()
