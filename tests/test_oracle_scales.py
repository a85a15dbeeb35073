"""Pins the oracle's amax, current-scale rules and the four quantisation
granularities against closed forms, invariants and brute force."""
import math

import numpy as np
import pytest

import oracle as o


def _enc_err_bound(fmt, p):
    """half the spacing of the format around |p| (p already scaled, |p| <= fmax)"""
    a = abs(float(p))
    if fmt == o.E4M3:
        e = max(math.floor(math.log2(a)) if a > 0 else -6, -6)
        return 2.0 ** (e - 3) / 2
    e = max(math.floor(math.log2(a)) if a > 0 else -14, -14)
    return 2.0 ** (e - 2) / 2


def test_amax_brute_force_and_nan():
    rng = np.random.default_rng(0)
    for n in [1, 2, 7, 128, 1000]:
        x = rng.standard_normal(n).astype(np.float32)
        assert o.amax(x) == np.max(np.abs(x))
    assert o.amax(np.zeros(5, np.float32)) == 0.0
    assert o.amax(np.float32([-3.0, 2.0])) == 3.0
    assert math.isnan(o.amax(np.float32([1.0, np.nan, 5.0])))


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_current_scale_closed_forms(fmt):
    fm = o.fmax(fmt)
    m, s = o.current_scale(fm / 4, fmt)
    assert m == 4.0 and s == 0.25
    m, s = o.current_scale(fm, fmt)
    assert m == 1.0 and s == 1.0
    for bad in [0.0, math.inf, math.nan]:
        assert o.current_scale(bad, fmt) == (1.0, 1.0)
    m, s = o.current_scale(3.0, fmt)
    assert m == np.float32(fm) / np.float32(3.0) and s == np.float32(3.0) / np.float32(fm)


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_tensor_current_invariants(fmt):
    rng = np.random.default_rng(1 + fmt)
    x = (rng.standard_normal((64, 96)) * 3).astype(np.float32)
    q, a, s, sat = o.quantize_tensor_current(x, fmt)
    maxc = 0x7E if fmt == o.E4M3 else 0x7B
    i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert q[i] & 0x7F == maxc                       # the amax element lands on +-fmax
    assert sat == 0
    m, _ = o.current_scale(a, fmt)
    deq = o.decode_array(fmt, q)
    p = x.astype(np.float32) * m
    for (r, c) in [(0, 0), (5, 7), (63, 95), i]:
        assert abs(deq[r, c] - float(p[r, c])) <= _enc_err_bound(fmt, p[r, c])
    assert np.all(np.sign(deq) * np.sign(x) >= 0)  # sign kept


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_power_of_two_rescale_is_exact(fmt):
    """Multiplying a tensor by 2^k multiplies its step s by 2^k and leaves the
    codes unchanged (the rule is scale-equivariant in binary)."""
    rng = np.random.default_rng(4)
    x = rng.standard_normal((4, 256)).astype(np.float32)
    for gran_fn in [o.quantize_tile1x128, o.quantize_mx32]:
        q0, s0, *_ = gran_fn(x, fmt)
        q1, s1, *_ = gran_fn(x * np.float32(8.0), fmt)
        assert np.array_equal(q0, q1)
        if gran_fn is o.quantize_mx32:
            assert np.array_equal(s1.astype(int), s0.astype(int) + 3)
        else:
            assert np.array_equal(s1, s0 * np.float32(8.0))


def test_tile_outlier_only_spoils_its_own_tile():
    """Week 14 absmax bullet: with per-block scales an outlier only hurts its
    own block.  A 1x128 tile with an outlier changes codes in that tile only."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 512)).astype(np.float32)
    q0, s0, a0, _ = o.quantize_tile1x128(x, o.E4M3)
    y = x.copy()
    y[1, 300] = 1000.0
    q1, s1, a1, _ = o.quantize_tile1x128(y, o.E4M3)
    diff = np.argwhere(q0 != q1)
    assert len(diff) > 0
    assert set(map(tuple, np.unique(np.stack([diff[:, 0], diff[:, 1] // 128], 1), axis=0))) == {(1, 2)}
    assert np.array_equal(np.argwhere(s0 != s1), np.array([[1, 2]]))
    assert a1[1, 2] == 1000.0


def test_tile_layout_rows_and_columns():
    """Scale layout s[r][c/128]: a tile whose values are all v gets s = v/448
    and every code is 0x7E; other tiles keep their own scale."""
    x = np.zeros((2, 384), np.float32)
    x[0, 0:128] = 3.0
    x[0, 128:256] = -5.0
    x[1, 256:384] = 0.5
    q, s, a, _ = o.quantize_tile1x128(x, o.E4M3)
    assert s.shape == (2, 3)
    assert s[0, 0] == np.float32(3.0) / np.float32(448.0)
    assert s[0, 1] == np.float32(5.0) / np.float32(448.0)
    assert s[1, 2] == np.float32(0.5) / np.float32(448.0)
    assert s[0, 2] == 1.0 and s[1, 0] == 1.0       # all-zero tiles
    assert np.all(q[0, 0:128] == 0x7E) and np.all(q[0, 128:256] == 0xFE)
    assert np.all(q[1, 256:] == 0x7E) and np.all(q[1, :256] == 0)


def test_block128_layout_and_outlier():
    rng = np.random.default_rng(6)
    x = (rng.standard_normal((256, 384)) * 0.02).astype(np.float32)
    q0, s0, a0, _ = o.quantize_block128(x, o.E4M3)
    assert s0.shape == (2, 3)
    for bi in range(2):
        for bj in range(3):
            blk = x[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]
            assert a0[bi, bj] == np.max(np.abs(blk))
            assert s0[bi, bj] == np.float32(np.max(np.abs(blk))) / np.float32(448.0)
    y = x.copy()
    y[130, 5] = 7.0                                     # block (1, 0)
    q1, s1, _, _ = o.quantize_block128(y, o.E4M3)
    changed = {(int(r) // 128, int(c) // 128) for r, c in np.argwhere(q0 != q1)}
    assert changed == {(1, 0)}
    assert np.array_equal(np.argwhere(s0 != s1), np.array([[1, 0]]))


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_mx_exponent_special_cases(fmt):
    emax = 8 if fmt == o.E4M3 else 15
    fm = o.fmax(fmt)
    for k in range(-20, 21):
        assert o.mx_scale_code(fm * 2.0 ** k, fmt) == 127 + k          # amax exactly fmax*2^k
        assert o.mx_scale_code(2.0 ** (emax + k), fmt) == 127 + k      # 1.0 * 2^(emax+k)
        just_above = float(np.nextafter(np.float32(fm * 2.0 ** k), np.float32(np.inf)))
        assert o.mx_scale_code(just_above, fmt) == 128 + k             # bumps by one
    assert o.mx_scale_code(0.0, fmt) == 127
    assert o.mx_scale_code(math.nan, fmt) == 0xFF
    assert o.mx_scale_code(math.inf, fmt) == 0xFF
    assert o.mx_scale_code(1e-45, fmt) == 0                            # clamped at 2^-127
    assert o.mx_scale_code(3e38, fmt) <= 254


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_mx_never_saturates_and_is_minimal(fmt):
    rng = np.random.default_rng(8)
    x = (rng.standard_normal((16, 256)) * 2.0 ** rng.integers(-30, 30, (16, 1))).astype(np.float32)
    x[3, 17] *= 100.0
    q, e, a, sat = o.quantize_mx32(x, fmt)
    assert sat == 0
    fm = o.fmax(fmt)
    for r in range(16):
        for t in range(8):
            amax = float(np.max(np.abs(x[r, 32 * t:32 * t + 32])))
            k = int(e[r, t]) - 127
            assert amax <= fm * 2.0 ** k                     # fits
            assert amax > fm * 2.0 ** (k - 1)                # smallest such power of two
            deq = o.decode_array(fmt, q[r, 32 * t:32 * t + 32]) * 2.0 ** k
            xs = x[r, 32 * t:32 * t + 32].astype(np.float64)
            bound = np.array([_enc_err_bound(fmt, v * 2.0 ** -k) for v in xs]) * 2.0 ** k
            assert np.all(np.abs(deq - xs) <= bound)


def test_sat_count_and_clipping():
    x = np.float32([1.0, 500.0, -448.0, 449.0, -1e6])
    q, sat = o.quantize_with_multiplier(x, 1.0, o.E4M3)
    assert sat == 3
    assert q.tolist() == [o.encode(o.E4M3, 1.0), 0x7E, 0xFE, 0x7E, 0xFE]


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_column_units_are_row_units_of_the_transpose(fmt):
    """Column tiles / column MX blocks of x are, by definition, the row units
    of x^T: codes, scales and amaxes must agree element for element."""
    rng = np.random.default_rng(12)
    x = (rng.standard_normal((256, 96)) * np.exp(rng.standard_normal((1, 96)))).astype(np.float32)
    x[5, 7] = 300.0
    q, s, a, sat = o.quantize_tile128x1(x, fmt)
    qt, st, at, satt = o.quantize_tile1x128(np.ascontiguousarray(x.T), fmt)
    assert np.array_equal(q, qt.T) and np.array_equal(s, st.T) and np.array_equal(a, at.T) and sat == satt
    q, e, a, sat = o.quantize_mx32_col(x, fmt)
    qt, et, at, satt = o.quantize_mx32(np.ascontiguousarray(x.T), fmt)
    assert np.array_equal(q, qt.T) and np.array_equal(e, et.T) and np.array_equal(a, at.T) and sat == satt


def test_column_tile_layout_closed_form():
    x = np.zeros((256, 3), np.float32)
    x[0:128, 0] = 2.0          # column 0, row block 0
    x[128:256, 2] = -7.0       # column 2, row block 1
    q, s, a, _ = o.quantize_tile128x1(x, o.E4M3)
    assert s.shape == (2, 3)
    assert s[0, 0] == np.float32(2.0) / np.float32(448.0) and s[1, 2] == np.float32(7.0) / np.float32(448.0)
    assert s[1, 0] == 1.0 and s[0, 2] == 1.0
    assert np.all(q[0:128, 0] == 0x7E) and np.all(q[128:, 2] == 0xFE)
    one = o.encode(o.E4M3, 1.0)
    assert np.array_equal(o.dequantize(np.full((256, 3), one, np.uint8), o.E4M3, o.GRAN_TILE_128x1, s),
                          np.repeat(s, 128, axis=0).astype(np.float64))
    e = np.array([[120, 130], [127, 140]], np.uint8)          # [R/32][C] for R = 64, C = 2
    assert np.array_equal(o.dequantize(np.full((64, 2), one, np.uint8), o.E4M3, o.GRAN_MX32_COL, e),
                          np.repeat(2.0 ** (e.astype(np.float64) - 127), 32, axis=0))


@pytest.mark.parametrize("gran", [o.GRAN_TILE_1x128, o.GRAN_MX32])
def test_fine_grained_backward_close_to_exact(gran):
    """The fine-grained forward / dgrad / wgrad of the oracle stay within the
    formats' precision of the exact float64 products (a dropped transpose or
    a mis-oriented scale would break this)."""
    rng = np.random.default_rng(13)
    M, K, N = 256, 384, 256
    x = rng.standard_normal((M, K)).astype(np.float32)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    dy = (rng.standard_normal((M, N)) * 1e-3).astype(np.float32)
    st, y = o.linear_fine_fwd(x, w, gran)
    dX, dW = o.linear_fine_bwd(st, dy, gran)
    x64, w64, d64 = x.astype(np.float64), w.astype(np.float64), dy.astype(np.float64)
    for got, exact in ((y, x64 @ w64.T), (dX, d64 @ w64), (dW, d64.T @ x64)):
        assert got.shape == exact.shape
        assert np.max(np.abs(got - exact)) / np.max(np.abs(exact)) < 0.1


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_mx_floor_rule_closed_form(fmt):
    """The floor rule is the ceiling rule minus one exactly when the block
    maximum's significand exceeds 1.75; only then does it clip."""
    fm = o.fmax(fmt)
    for k in range(-10, 11):
        exact = fm * 2.0 ** k                        # significand 1.75: same code, no clipping
        assert o.mx_scale_code_floor(exact, fmt) == o.mx_scale_code(exact, fmt)
        above = float(np.nextafter(np.float32(exact), np.float32(np.inf)))
        assert o.mx_scale_code_floor(above, fmt) == o.mx_scale_code(above, fmt) - 1
        one = 2.0 ** (k + 3)                         # significand 1.0
        assert o.mx_scale_code_floor(one, fmt) == o.mx_scale_code(one, fmt)
    x = np.full((1, 32), 1.0, np.float32)
    x[0, 0] = np.float32(1.9 * 2.0 ** 5)
    q, e, sat = o.quantize_mx32_floor(x, fmt)
    assert sat == 1 and (q[0, 0] & 0x7F) == (0x7E if fmt == o.E4M3 else 0x7B)
    _, _, _, sat_ceil = o.quantize_mx32(x, fmt)
    assert sat_ceil == 0


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_pow2_tiles_and_blocks(fmt):
    """A power-of-two 1x128 tile scale is the largest of its four MX-32 codes
    (the code is monotone in amax); a 128x128 block's is the largest over its
    tiles.  Codes are the cast with that exact power of two; nothing clips."""
    rng = np.random.default_rng(14)
    x = (rng.standard_normal((256, 384)) * np.exp(rng.standard_normal((256, 1)))).astype(np.float32)
    x[3, 200] = 5000.0
    q, e, sat = o.quantize_tile1x128_pow2(x, fmt)
    _, emx, _, _ = o.quantize_mx32(x, fmt)
    assert np.array_equal(e, emx.reshape(256, 3, 4).max(axis=2)) and sat == 0
    for (r, t) in [(0, 0), (3, 1), (255, 2)]:
        m = 2.0 ** -(int(e[r, t]) - 127)
        qq, _ = o.quantize_with_multiplier(x[r, 128 * t:128 * t + 128], np.float32(m), fmt)
        assert np.array_equal(q[r, 128 * t:128 * t + 128], qq)
    qb, eb, satb = o.quantize_block128_pow2(x, fmt)
    assert np.array_equal(eb, e.reshape(2, 128, 3).max(axis=1)) and satb == 0
    one = o.encode(fmt, 1.0)
    assert np.array_equal(o.dequantize(np.full((256, 384), one, np.uint8), fmt, o.GRAN_BLOCK_POW2, eb),
                          np.repeat(np.repeat(2.0 ** (eb.astype(np.float64) - 127), 128, 0), 128, 1))


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_pow2_column_tiles(fmt):
    """A power-of-two 128x1 column tile's code is the largest of the four
    column MX-32 codes it covers; the codes are the row tiles of x^T (the
    same rule on 128 consecutive values of a column); dequantising the code
    of 1.0 gives the tile's power of two."""
    rng = np.random.default_rng(16)
    x = (rng.standard_normal((256, 384)) * np.exp(rng.standard_normal((1, 384)))).astype(np.float32)
    x[200, 3] = 9000.0
    q, e, sat = o.quantize_tile128x1_pow2(x, fmt)
    _, emx, _, _ = o.quantize_mx32_col(x, fmt)
    assert e.shape == (2, 384) and sat == 0
    assert np.array_equal(e, emx.reshape(2, 4, 384).max(axis=1))
    qt, et, _ = o.quantize_tile1x128_pow2(np.ascontiguousarray(x.T), fmt)
    assert np.array_equal(q, qt.T) and np.array_equal(e, et.T)
    one = o.encode(fmt, 1.0)
    assert np.array_equal(o.dequantize(np.full((256, 384), one, np.uint8), fmt, o.GRAN_TILE_COL_POW2, e),
                          np.repeat(2.0 ** (e.astype(np.float64) - 127), 128, 0))


def test_layernorm_closed_forms():
    """Standardised output: every row has mean 0 and variance var/(var+eps)
    before the affine part; gamma scales and beta shifts column-wise; a
    constant row gives beta exactly."""
    rng = np.random.default_rng(15)
    x = (rng.standard_normal((8, 256)) * 3 + 2).astype(np.float32)
    x[5, :] = 7.0
    g = np.ones(256, np.float32)
    y, mu, rs = o.layernorm(x, g, None, 1e-5)
    assert np.allclose(mu, x.astype(np.float64).mean(axis=1), rtol=0, atol=1e-12)
    var = x.astype(np.float64).var(axis=1)
    assert np.allclose(rs, 1 / np.sqrt(var + 1e-5), rtol=1e-14)
    assert np.allclose(y.mean(axis=1), 0, atol=1e-12)
    assert np.allclose(y[:5].var(axis=1), var[:5] / (var[:5] + 1e-5), rtol=1e-12)
    gam = rng.uniform(0.5, 2, 256).astype(np.float32)
    bet = rng.standard_normal(256).astype(np.float32)
    y2, _, _ = o.layernorm(x, gam, bet, 1e-5)
    assert np.allclose(y2, y * gam + bet, rtol=1e-12, atol=1e-12)
    assert np.array_equal(y2[5], bet.astype(np.float64))


def test_ln_acceptable_codes_bracket():
    y = np.array([1.0, 67.9999, 68.0001, -3.0], dtype=np.float64)     # 68 = E4M3 midpoint of 64 and 72
    delta = np.full(4, 1e-3)
    near, lo, hi = o.ln_acceptable_codes(y, delta, 1.0, o.E4M3)
    r = o.code_rank
    assert np.all(r(lo) <= r(near)) and np.all(r(near) <= r(hi))
    assert lo[1] != hi[1] and lo[2] != hi[2]            # ambiguous next to the midpoint
    assert lo[0] == hi[0] and lo[3] == hi[3]            # unambiguous elsewhere
