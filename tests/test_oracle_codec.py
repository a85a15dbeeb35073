"""Pins the oracle's FP8 / bf16 codec by brute force and against independent
library casts (torch's float8_e4m3fn / float8_e5m2 / bfloat16 conversions are
round-to-nearest-even inside the finite range)."""
import math

import numpy as np
import pytest
import torch

import oracle as o


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_decode_all_codes_structure(fmt):
    vals = [o.decode(fmt, c) for c in range(256)]
    pos = vals[:128]
    maxc = 0x7E if fmt == o.E4M3 else 0x7B
    finite = pos[: maxc + 1]
    assert all(b > a for a, b in zip(finite, finite[1:])), "non-negative codes must increase"
    assert finite[0] == 0.0
    assert finite[1] == (2.0 ** -9 if fmt == o.E4M3 else 2.0 ** -16)      # smallest subnormal
    # negative half mirrors the positive half
    for c in range(128):
        a, b = vals[c], vals[c | 0x80]
        assert (math.isnan(a) and math.isnan(b)) or b == -a
    if fmt == o.E4M3:
        assert [c for c in range(256) if math.isnan(vals[c])] == [0x7F, 0xFF]
        assert not any(math.isinf(v) for v in vals)
    else:
        assert vals[0x7C] == math.inf and vals[0xFC] == -math.inf
        assert [c for c in range(256) if math.isnan(vals[c])] == [0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF]


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_encode_decode_roundtrip_all_codes(fmt):
    maxc = 0x7E if fmt == o.E4M3 else 0x7B
    for c in range(256):
        v = o.decode(fmt, c)
        if math.isnan(v):
            continue
        if math.isinf(v):                        # infinities saturate
            assert o.encode(fmt, v) == (maxc | (c & 0x80))
            continue
        assert o.encode(fmt, v) == c, hex(c)


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_saturation(fmt):
    fm = o.fmax(fmt)
    maxc = 0x7E if fmt == o.E4M3 else 0x7B
    for v in [fm, fm * 1.01, fm * 1.5, fm * 1000, 3e38, math.inf]:
        assert o.encode(fmt, v) == maxc
        assert o.encode(fmt, -v) == 0x80 | maxc
    assert o.encode(fmt, float("nan")) == 0x7F
    assert o.encode(fmt, -0.0) == 0x80
    assert o.encode(fmt, -1e-30) == 0x80


def _torch_fp8(fmt):
    return torch.float8_e4m3fn if fmt == o.E4M3 else torch.float8_e5m2


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_encode_matches_torch_cast_at_every_midpoint(fmt):
    """Every midpoint between neighbouring codes (exact in fp32), one fp32 ulp
    either side of it, and the codes themselves: the oracle's table encoder
    must agree with torch's RNE cast, which is an independent implementation."""
    maxc = 0x7E if fmt == o.E4M3 else 0x7B
    vals = np.array([o.decode(fmt, c) for c in range(maxc + 1)], dtype=np.float64)
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    assert np.all(mids.astype(np.float64) == (vals[:-1] + vals[1:]) / 2)
    pts = np.concatenate([vals.astype(np.float32), mids,
                          np.nextafter(mids, np.float32(np.inf)),
                          np.nextafter(mids, np.float32(-np.inf))])
    pts = np.concatenate([pts, -pts])
    ref = torch.from_numpy(pts).to(_torch_fp8(fmt)).view(torch.uint8).numpy()
    mine = np.array([o.encode(fmt, float(v)) for v in pts], dtype=np.uint8)
    assert np.array_equal(mine, ref)


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_encode_matches_torch_cast_random(fmt):
    rng = np.random.default_rng(7 + fmt)
    fm = o.fmax(fmt)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(fm / 8),
        (rng.standard_normal(20000) * 2.0 ** rng.integers(-24, 0, 20000)).astype(np.float32),
        rng.uniform(-fm * 0.999, fm * 0.999, 5000).astype(np.float32),
    ])
    x = x[np.abs(x) < fm]
    ref = torch.from_numpy(x).to(_torch_fp8(fmt)).view(torch.uint8).numpy()
    mine = np.array([o.encode(fmt, float(v)) for v in x], dtype=np.uint8)
    assert np.array_equal(mine, ref)


def test_bf16_matches_torch_and_fast_path():
    rng = np.random.default_rng(3)
    x = np.concatenate([
        rng.standard_normal(50000).astype(np.float32) * np.float32(1e3),
        (rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32)).view(np.float32),
        np.float32([257.0, 259.0, 0.0, -0.0, 3.4e38, -3.4e38, 1e-40, np.inf, -np.inf]),
    ])
    x = x[~np.isnan(x)]
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    mine = o.bf16_round_array(x)
    fast = o.bf16_round_array_fast(x)
    assert np.array_equal(mine, ref)
    assert np.array_equal(fast, ref)
