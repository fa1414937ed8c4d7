"""The amax passes take the largest magnitude of a transformed run,
x' = 1/4 * H16 * v, without forming x': after three butterfly stages they
keep RN(|a| + |b|) for each pair (a, b) of the last stage, whose two outputs
RN(a + b) and RN(a - b) have that larger magnitude, and scale the maximum by
1/4 once instead of every element.  Both steps rest on rounding to nearest
being monotonic and odd, so the result should equal the maximum of |x'|
formed the plain way bit for bit.  This test restates both computations in
FP32 with numpy (IEEE round to nearest even, subnormals kept) and compares
them on random runs of BF16 values and on runs built to stress the rounding:
ties, values next to the subnormal range, and magnitudes near overflow.  It
does not run the CUDA code; the GPU parity tests compare the kernels' tensor
scales with the oracle bit for bit."""
import numpy as np

F32 = np.float32


def _butterflies(v, strides):
    v = v.copy()
    for s in strides:
        for i in range(16):
            if i & s:
                continue
            a, b = v[:, i].copy(), v[:, i + s].copy()
            v[:, i] = a + b
            v[:, i + s] = a - b
    return v


def _plain(v):
    x = _butterflies(v, (1, 2, 4, 8)) * F32(0.25)
    return np.abs(x).view(np.uint32).max(axis=1)


def _shortcut(v):
    w = _butterflies(v, (1, 2, 4))
    pair = np.abs(w[:, :8]) + np.abs(w[:, 8:])
    m = np.abs(pair).view(np.uint32).max(axis=1)
    return np.abs(m.view(F32) * F32(0.25)).view(np.uint32)


def _bf16(bits):
    return (bits.astype(np.uint32) << 16).view(F32)


INF_BITS = np.array([np.inf], dtype=F32).view(np.uint32)[0]


def _agree(plain, short):
    """Bit-equal, or both at or above the bits of infinity (a transform that
    overflows can give NaN one way and infinity the other: inf - inf)."""
    return bool(np.all((plain == short) | ((plain >= INF_BITS) & (short >= INF_BITS))))


def test_random_bf16_runs():
    rng = np.random.default_rng(7)
    with np.errstate(over="ignore", invalid="ignore"):
        for scale_exp in (-140, -126, -100, -20, 0, 20, 100, 120):
            v = (rng.standard_normal((20000, 16)) * np.float64(2.0) ** scale_exp).astype(F32)
            v = _bf16(v.view(np.uint32) >> 16)  # BF16 inputs, as the kernels read them
            assert _agree(_plain(v), _shortcut(v)), scale_exp


def test_every_bf16_exponent_and_structured_runs():
    rng = np.random.default_rng(11)
    with np.errstate(over="ignore", invalid="ignore"):
        # random BF16 bit patterns over the whole finite range, mixed signs
        bits = rng.integers(0, 0x7F80, size=(200000, 16), dtype=np.uint32)
        bits |= (rng.integers(0, 2, size=bits.shape, dtype=np.uint32) << 15)
        v = _bf16(bits)
        assert _agree(_plain(v), _shortcut(v))
        # runs of equal magnitudes and signs chosen so that sums tie or cancel
        base = _bf16(rng.integers(0x0001, 0x7F7F, size=(50000, 1), dtype=np.uint32))
        signs = np.where(rng.integers(0, 2, size=(50000, 16)) == 1, F32(-1), F32(1))
        step = _bf16(rng.integers(0x3F80, 0x3F88, size=(50000, 16), dtype=np.uint32))
        v = (base * signs * step).astype(F32)
        plain, short = _plain(v), _shortcut(v)
        assert _agree(plain, short)
        finite = plain < INF_BITS
        assert finite.sum() > 40000 and np.array_equal(plain[finite], short[finite])


def test_zero_and_single_element_runs():
    v = np.zeros((3, 16), dtype=F32)
    v[1, 5] = F32(-3.0)
    v[2, 15] = F32(1e-45)  # the smallest subnormal
    assert np.array_equal(_plain(v), _shortcut(v))
    assert _shortcut(v)[1] == np.array([0.75], dtype=F32).view(np.uint32)[0]


def test_non_finite_runs_are_flagged_either_way():
    v = np.ones((3, 16), dtype=F32)
    v[0, 3] = np.inf
    v[1, 0], v[1, 8] = np.inf, -np.inf  # inf - inf: NaN one way, inf the other
    v[2, 7] = np.nan
    with np.errstate(invalid="ignore"):
        plain, short = _plain(v), _shortcut(v)
    assert (plain >= INF_BITS).all() and (short >= INF_BITS).all()
