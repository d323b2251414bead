"""The seeded input generator: published SplitMix64 vectors, determinism,
counter-based slicing, and the distributions it claims."""
import numpy as np

import synthgen

GAMMA = 0x9E3779B97F4A7C15


def test_splitmix64_published_vectors():
    # SplitMix64 seeded with 1234567: the first three outputs of the published generator
    outs = [synthgen.splitmix64((1234567 + k * GAMMA) % 2**64) for k in range(3)]
    assert outs == [6457827717110365317, 3203168211198807973, 9817491932198370423]
    assert synthgen.splitmix64(0) == 0xE220A8397B1DCDAF


def test_counter_based_slices_and_determinism():
    full = synthgen.normal_f32(100_000, seed=7, sigma=1.0)
    part = synthgen.normal_f32(1000, seed=7, sigma=1.0, first=54_321)
    assert np.array_equal(full[54_321:55_321], part)
    assert np.array_equal(full, synthgen.normal_f32(100_000, seed=7, sigma=1.0))
    assert not np.array_equal(full, synthgen.normal_f32(100_000, seed=8, sigma=1.0))


def test_distributions():
    x = synthgen.normal_f32(1_000_000, seed=0, sigma=1e-3).astype(np.float64)
    assert abs(x.mean()) < 5e-6 and abs(x.std() - 1e-3) < 5e-6
    o = synthgen.normal_f32(1_000_000, seed=0, sigma=1e-3, outlier_p=1e-3, outlier_scale=100.0)
    frac = np.mean(np.abs(o) != np.abs(x.astype(np.float32)))
    assert 0.0007 < frac < 0.0013
    u = synthgen.uniform_f32(1_000_000, seed=1, lo=-1.0, hi=1.0)
    assert u.min() > -1 and u.max() < 1 and abs(u.mean()) < 5e-3
    k = synthgen.uniform_i32(1_000_000, seed=2, lo=-(2**20), hi=2**20)
    assert k.min() >= -(2**20) and k.max() <= 2**20 and k.min() < -(2**20) + 100 and k.max() > 2**20 - 100


def test_reduced_precision_is_library_rounding():
    import torch
    x = synthgen.normal_f32(10_000, seed=3, sigma=1e-4)
    b = synthgen.to_dtype(x, "bf16")
    assert np.array_equal(b, torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(synthgen.to_dtype(x, "f16"), x.astype(np.float16).view(np.uint16))


def test_gpt2_shapes():
    shapes = synthgen.gpt2_small_param_shapes()
    assert len(shapes) == 148
    assert sum(int(np.prod(s)) for _, s in shapes) == 124_439_808
