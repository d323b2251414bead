"""Pins of the oracle's number-format conversions (no GPU).

bf16 is checked against PyTorch's CPU conversion and fp16 against numpy's
(library routines); E4M3 against a brute-force nearest-value search over its
256 codes and the format's anchors. The patterns cover every sign/exponent/
top-fraction combination with the low bits that decide rounding (ties, just
below and above), plus random bit patterns.
"""
import numpy as np
import torch

import oracle

RNG = np.random.default_rng(1234)
LOWS = np.array([0x0000, 0x0001, 0x0FFF, 0x1000, 0x1001, 0x1FFF, 0x2000, 0x2001, 0x3000,
                 0x7FFF, 0x8000, 0x8001, 0xC000, 0xFFFF], dtype=np.uint32)


def _patterns():
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    grid = (hi[:, None] | LOWS[None, :]).ravel()
    rnd = RNG.integers(0, 1 << 32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
    return np.concatenate([grid, rnd]).view(np.float32)


def _same(a_bits, b_bits, is_nan):
    # NaN payloads are not part of the contract: compare the NaN class there
    return np.array_equal(a_bits[~is_nan], b_bits[~is_nan])


def test_bf16_matches_torch():
    x = _patterns()
    ours = oracle.f32_to_bf16(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert _same(ours, ref, nan)
    assert np.all(ours[nan] == 0x7FC0)


def test_f16_matches_numpy():
    x = _patterns()
    ours = oracle.f32_to_f16(x)
    with np.errstate(over="ignore", invalid="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert _same(ours, ref, nan)
    assert np.all(ours[nan] == 0x7E00)


def test_decoders_roundtrip_and_match_libraries():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    bf = oracle.bf16_to_f32(h)
    assert np.array_equal(bf.view(np.uint32), h.astype(np.uint32) << 16)
    f16 = oracle.f16_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    fin = ~np.isnan(ref)
    assert np.array_equal(f16[fin], ref[fin]) and np.all(np.isnan(f16[~fin]))
    assert np.array_equal(oracle.f32_to_f16(f16[fin]), h[fin])


def _e4m3_table():
    codes = np.arange(256, dtype=np.uint32).astype(np.uint8)
    return codes, oracle.e4m3_to_f32(codes)


def test_e4m3_anchors():
    codes, v = _e4m3_table()
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0           # largest finite
    assert v[0x08] == 2.0**-6                                # smallest normal
    assert v[0x01] == 2.0**-9                                # smallest subnormal
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])           # the only NaNs
    assert np.sum(np.isnan(v)) == 2 and not np.any(np.isinf(v))
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)                          # codes 0..126 increase
    assert np.array_equal(v[0x80:0xFF], -pos)                # sign bit mirrors
    assert v[0x80] == 0.0 and np.signbit(v[0x80])
    # every finite value converts back to its own code
    fin = ~np.isnan(v)
    assert np.array_equal(oracle.f32_to_e4m3(v[fin]), codes[fin])


def _brute_e4m3(x):
    """Nearest of the 127 non-negative finite E4M3 values; ties to the even code;
    saturate beyond 448; NaN -> 0x7F."""
    _, v = _e4m3_table()
    mags = v[:0x7F].astype(np.float64)
    a = np.abs(x.astype(np.float64))
    d = np.abs(a[:, None] - mags[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    k = np.where(cand.sum(axis=1) == 1, cand.argmax(axis=1),
                 np.where(cand[:, ::2].any(axis=1), 2 * cand[:, ::2].argmax(axis=1), cand.argmax(axis=1)))
    k = np.where(a > 448.0, 0x7E, k).astype(np.uint8)
    out = k | np.where(np.signbit(x), 0x80, 0).astype(np.uint8)
    return np.where(np.isnan(x), 0x7F, out).astype(np.uint8)


def test_e4m3_matches_brute_force():
    _, v = _e4m3_table()
    mags = np.sort(v[:0x7F])
    mids = ((mags[1:].astype(np.float64) + mags[:-1]) / 2).astype(np.float32)  # exact ties
    near = np.concatenate([np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    rnd = np.exp(RNG.uniform(np.log(2.0**-12), np.log(600.0), 200_000)).astype(np.float32)
    x = np.concatenate([mids, near, rnd, mags, [0.0, 448.0, 449.0, 464.0, 465.0, 1e30, np.inf, 2.0**-10,
                                               2.0**-11, 1e-45]]).astype(np.float32)
    x = np.concatenate([x, -x])
    assert np.array_equal(oracle.f32_to_e4m3(x), _brute_e4m3(x))
    assert oracle.f32_to_e4m3(np.array([np.nan], dtype=np.float32))[0] == 0x7F


def test_e4m3_matches_torch_within_range():
    # torch's float8_e4m3fn rounds to nearest even and does not saturate, so compare below 464
    x = RNG.uniform(-460, 460, 300_000).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.f32_to_e4m3(x), ref)
