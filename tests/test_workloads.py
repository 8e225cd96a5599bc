"""The seeded input generators (CPU): what the workloads promise about their inputs."""
import numpy as np
import pytest
import torch

from lossless_invariant_bit_gb300 import workloads as wl


def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(3).standard_normal(200_000).astype(np.float32)
    x[:6] = [0.0, -0.0, 1.0, -2.5, 3.0e38, 1.0e-40]
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(wl.to_bf16_bits(x), ref)


def test_bf16_weight_rows_are_seeded_and_scaled():
    a = wl.bf16_weight_rows(64, 4096, seed=1, matrix=2)
    b = wl.bf16_weight_rows(64, 4096, seed=1, matrix=2)
    c = wl.bf16_weight_rows(64, 4096, seed=1, matrix=3)
    assert a.dtype == np.uint16 and a.shape == (64, 4096)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    v = (a.astype(np.uint32) << 16).view(np.float32)
    assert 0.018 < float(v.std()) < 0.022


@pytest.mark.parametrize("k", [0, 7, 31])
def test_invariant_pattern_bit_counts(k):
    for scattered in (False, True):
        keep, const = wl.invariant_pattern(96, k, scattered, seed=4)
        assert all(bin(int(x)).count("1") == 32 - k for x in keep)
        assert np.all(const & keep == 0)
