"""Pins for the oracle's p99 clipping (CPU only): the nearest-rank percentile
on tensors whose magnitude counts are known in closed form, and clipping that
leaves values inside the bound untouched and bounds the rest."""
import numpy as np
import torch

import oracle


def _bits(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_percentile_on_known_counts():
    # 990 magnitudes of 1 and 10 of 100 (signs mixed): rank 990 is the last 1,
    # rank 991 the first 100
    x = np.concatenate([np.ones(990), np.full(10, 100.0)])
    x[::3] *= -1
    rng = np.random.default_rng(1)
    x = _bits(rng.permutation(x))
    assert oracle.abs_percentile_bf16(x, 99.0) == 1.0
    assert oracle.abs_percentile_bf16(x, 99.1) == 100.0
    assert oracle.abs_percentile_bf16(x, 100.0) == 100.0
    assert oracle.abs_percentile_bf16(x, 0.01) == 1.0


def test_percentile_of_a_ramp():
    # magnitudes 1..1024 (all exact in BF16 up to 256; beyond, distinct BF16
    # values in sorted order): the k-th smallest is the k-th value of the ramp
    vals = np.unique(torch.arange(1, 1025, dtype=torch.float32).to(torch.bfloat16).float().numpy())
    rng = np.random.default_rng(2)
    x = _bits(rng.permutation(np.concatenate([vals, -vals])))
    n = 2 * len(vals)
    k = int(np.ceil(0.99 * n))
    assert oracle.abs_percentile_bf16(x, 99.0) == vals[(k - 1) // 2]


def test_clip():
    x = _bits([-300.0, -2.5, 0.0, 1.0, 7.0, 1000.0])
    out = oracle.clip_bf16(x, 7.0)
    got = torch.from_numpy(out.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(got, [-7.0, -2.5, 0.0, 1.0, 7.0, 7.0])
