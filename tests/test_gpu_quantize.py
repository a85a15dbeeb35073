"""GPU parity of amax, scale rules, casts and the delayed state against the
CPU oracle: codes, scales, amaxes and histories must match bit for bit."""
import numpy as np
import pytest
import torch

import oracle as o
import scaled_quantize_gemm_gb300 as sq
from scaled_quantize_gemm_gb300 import workloads as wl

from _helpers import codes, nan_aware_codes_equal, np32

pytestmark = pytest.mark.gpu
DEV = "cuda"
FMTS = [sq.E4M3, sq.E5M2]


def _u8(shape):
    return torch.empty(shape, dtype=torch.uint8, device=DEV)


def _f32(n):
    return torch.zeros(n, dtype=torch.float32, device=DEV)


def _all_bf16_patterns():
    return torch.arange(0, 65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).reshape(256, 256)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m", [1.0, 0.75, 3.0, 2.0 ** -10, 1e-3, 448.0 / 3.0, 57344.0 / 1000.0, 2.0 ** 20])
def test_every_bf16_pattern_every_multiplier(fmt, m):
    """All 65,536 bf16 bit patterns through the delayed per-tensor cast with a
    set multiplier: every code, the recorded amax and the clip count."""
    x = _all_bf16_patterns().to(DEV)
    H = 16
    st = _f32(H + 2)
    st[H] = float(np.float32(m))
    q = _u8((256, 256))
    sat = torch.zeros(1, dtype=torch.int64, device=DEV)
    sq.fp8_quantize(x, fmt, sq.TENSOR, q, delayed_state=st, history_len=H, sat_count=sat)
    torch.cuda.synchronize()
    xf = np32(x.cpu())
    ref, ref_sat = o.quantize_with_multiplier(xf, np.float32(m), fmt)
    assert nan_aware_codes_equal(codes(q), ref, fmt)
    assert np.isnan(float(st[0].item()))                     # the NaN patterns propagate into amax
    finite = xf[np.isfinite(xf)]
    ref_nonnan_sat = o.quantize_with_multiplier(xf[~np.isnan(xf)], np.float32(m), fmt)[1]
    assert int(sat.item()) == ref_nonnan_sat
    # amax over the non-NaN patterns
    st2 = _f32(H + 2)
    st2[H] = 1.0
    xs = x.view(-1)[~torch.isnan(x.view(-1))].contiguous()
    q2 = _u8(xs.numel())
    sq.fp8_quantize(xs, fmt, sq.TENSOR, q2, delayed_state=st2, history_len=H)
    torch.cuda.synchronize()
    assert float(st2[0].item()) == o.amax(np32(xs.cpu()))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(256, 256), (1000, 37), (1, 5), (3, 1024), (513, 256), (1024, 1031)])
def test_tensor_current(fmt, shape):
    a, _ = wl.w1_operands()
    x = torch.randn(shape, generator=torch.Generator().manual_seed(sum(shape)), dtype=torch.float32)
    if shape == (256, 256):
        x = a                                     # workload 1 operand, outliers of 30
    xd = x.to(DEV)
    q = _u8(shape)
    amax, s = _f32(1), _f32(1)
    sat = torch.zeros(1, dtype=torch.int64, device=DEV)
    sq.fp8_quantize(xd, fmt, sq.TENSOR, q, scales_out=s, amax_out=amax, sat_count=sat)
    torch.cuda.synchronize()
    rq, ra, rs, rsat = o.quantize_tensor_current(x.numpy(), fmt)
    assert np.array_equal(codes(q), rq)
    # amax * fp32(fmax / amax) can round one ulp above fmax, so current
    # scaling may saturate the elements equal to the amax (and only those):
    # the same count on both sides
    assert amax.item() == ra and s.item() == rs and int(sat.item()) == rsat
    assert rsat <= int(np.sum(np.abs(x.numpy()) == ra))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(256, 384), (16, 16), (272, 144), (128, 4096)])
def test_tensor_delayed_with_transpose(fmt, shape):
    R, C = shape
    x = wl.normal(shape, 2.5, 77 + R, "cpu")
    H = 16
    st = torch.tensor(o.state_init(H), device=DEV)
    st[H] = 60.0 if fmt == sq.E4M3 else 9000.0
    ref_state = st.cpu().numpy().copy()
    q, qT = _u8(shape), _u8((C, R))
    sq.fp8_quantize(x.to(DEV), fmt, sq.TENSOR, q, qT=qT, delayed_state=st, history_len=H)
    torch.cuda.synchronize()
    rq, _ = o.quantize_delayed(np32(x), fmt, ref_state)
    assert np.array_equal(codes(q), rq)
    assert np.array_equal(codes(qT), rq.T)
    assert st.cpu().numpy().tobytes() == ref_state.tobytes()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(300, 512), (1, 128), (64, 4096)])
def test_tile_1x128(fmt, shape):
    x = wl.student_t3(shape, 5 + shape[0])
    q = _u8(shape)
    s = _f32(shape[0] * shape[1] // 128)
    am = _f32(shape[0] * shape[1] // 128)
    sat = torch.zeros(1, dtype=torch.int64, device=DEV)
    sq.fp8_quantize(x.to(DEV), fmt, sq.TILE_1x128, q, scales_out=s, amax_out=am, sat_count=sat)
    torch.cuda.synchronize()
    rq, rs, ra, rsat = o.quantize_tile1x128(np32(x), fmt)
    assert np.array_equal(codes(q), rq)
    assert np.array_equal(s.cpu().numpy(), rs.ravel())
    assert np.array_equal(am.cpu().numpy(), ra.ravel())
    assert int(sat.item()) == rsat


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(384, 256), (128, 128)])
def test_block_128x128(fmt, shape):
    x = wl.normal(shape, 0.02, 9 + shape[0])
    x[5, 7] = 3.0
    q = _u8(shape)
    nb = (shape[0] // 128) * (shape[1] // 128)
    s, am = _f32(nb), _f32(nb)
    sq.fp8_quantize(x.to(DEV), fmt, sq.BLOCK_128x128, q, scales_out=s, amax_out=am)
    torch.cuda.synchronize()
    rq, rs, ra, _ = o.quantize_block128(np32(x), fmt)
    assert np.array_equal(codes(q), rq)
    assert np.array_equal(s.cpu().numpy(), rs.ravel())
    assert np.array_equal(am.cpu().numpy(), ra.ravel())


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(64, 1024), (3, 32), (17, 96)])
def test_mx32(fmt, shape):
    x = wl.with_scaled_fraction(shape, 0.01, 100.0, 3 + shape[0])
    x[0, :32] = 0.0                                         # all-zero block -> code 127
    x[1, :32] *= 2.0 ** -100                                # tiny block, exponent clamps
    q = _u8(shape)
    e = _u8(shape[0] * shape[1] // 32)
    am = _f32(shape[0] * shape[1] // 32)
    sat = torch.zeros(1, dtype=torch.int64, device=DEV)
    sq.fp8_quantize(x.to(DEV), fmt, sq.MX32, q, scales_out=e, amax_out=am, sat_count=sat)
    torch.cuda.synchronize()
    rq, re, ra, rsat = o.quantize_mx32(np32(x), fmt)
    assert np.array_equal(codes(q), rq)
    assert np.array_equal(e.cpu().numpy(), re.ravel())
    assert np.array_equal(am.cpu().numpy(), ra.ravel())
    assert int(sat.item()) == rsat == 0


@pytest.mark.parametrize("gran,shape", [(sq.TENSOR, (333, 17)), (sq.TILE_1x128, (5, 256)),
                                        (sq.BLOCK_128x128, (256, 128)), (sq.MX32, (7, 64))])
def test_amax_units(gran, shape):
    x = wl.normal(shape, 3.0, 41)
    n_units = {sq.TENSOR: 1, sq.TILE_1x128: shape[0] * shape[1] // 128,
               sq.BLOCK_128x128: (shape[0] // 128) * (shape[1] // 128), sq.MX32: shape[0] * shape[1] // 32}[gran]
    am = _f32(n_units)
    sq.fp8_amax(x.to(DEV), gran, am)
    torch.cuda.synchronize()
    xf = np32(x)
    if gran == sq.TENSOR:
        ref = np.float32([o.amax(xf)])
    elif gran == sq.TILE_1x128:
        ref = o.quantize_tile1x128(xf, 0)[2].ravel()
    elif gran == sq.BLOCK_128x128:
        ref = o.quantize_block128(xf, 0)[2].ravel()
    else:
        ref = o.quantize_mx32(xf, 0)[2].ravel()
    assert np.array_equal(am.cpu().numpy(), ref)


def test_empty_tensor():
    x = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    q = _u8((0, 64))
    amax, s = _f32(1), _f32(1)
    amax.fill_(5.0)
    s.fill_(5.0)
    sq.fp8_quantize(x, sq.E4M3, sq.TENSOR, q, scales_out=s, amax_out=amax)
    torch.cuda.synchronize()
    assert amax.item() == 0.0 and s.item() == 1.0


@pytest.mark.parametrize("algo", [sq.AMAX_MAX, sq.AMAX_MOST_RECENT])
def test_update_scale_multi_state_sequence(algo):
    """Three roles (x E4M3, W E4M3, dy E5M2 -- the HYBRID recipe), 25 steps of
    cast + end-of-step update with drifting and spiking tensors; histories,
    multipliers and steps must match the oracle bit for bit every step."""
    H = 16
    fmts = [sq.E4M3, sq.E4M3, sq.E5M2]
    states = torch.empty(3 * (H + 2), dtype=torch.float32, device=DEV)
    sq.fp8_scale_init(states, 3, H)
    ref = [o.state_init(H) for _ in range(3)]
    g = torch.Generator().manual_seed(0)
    for step in range(25):
        for r in range(3):
            std = (1.0 + step) if r == 0 else (0.02 if r == 1 else 1e-3)
            x = (torch.randn((64, 128), generator=g) * std).to(torch.bfloat16)
            if step == 7 and r == 0:
                x[3, 3] = 5000.0
            q = _u8((64, 128))
            st = states[r * (H + 2):(r + 1) * (H + 2)]
            sq.fp8_quantize(x.to(DEV), fmts[r], sq.TENSOR, q, delayed_state=st, history_len=H)
            rq, _ = o.quantize_delayed(np32(x), fmts[r], ref[r])
            torch.cuda.synchronize()
            assert np.array_equal(codes(q), rq), (step, r)
        sq.fp8_update_scale(states, 3, H, fmts, algo)
        for r in range(3):
            o.update_scale(ref[r], fmts[r], algo)
        torch.cuda.synchronize()
        assert states.cpu().numpy().tobytes() == np.concatenate(ref).tobytes(), step


def test_scale_init():
    st = torch.full((4 * 18,), 7.0, device=DEV)
    sq.fp8_scale_init(st, 4, 16)
    torch.cuda.synchronize()
    assert st.cpu().numpy().tobytes() == np.concatenate([o.state_init(16)] * 4).tobytes()


# ---------------------------------------------------------------- full-size workloads
def test_w3_tiles_and_blocks_full_size():
    x, w = wl.w3_operands(DEV)
    qx, qw = _u8(x.shape), _u8(w.shape)
    sx = _f32(4096 * 32)
    sw = _f32(32 * 32)
    sq.fp8_quantize(x, sq.E4M3, sq.TILE_1x128, qx, scales_out=sx)
    sq.fp8_quantize(w, sq.E4M3, sq.BLOCK_128x128, qw, scales_out=sw)
    torch.cuda.synchronize()
    rq, rs, _, _ = o.quantize_tile1x128(np32(x), sq.E4M3)
    assert np.array_equal(codes(qx), rq) and np.array_equal(sx.cpu().numpy(), rs.ravel())
    rq, rs, _, _ = o.quantize_block128(np32(w), sq.E4M3)
    assert np.array_equal(codes(qw), rq) and np.array_equal(sw.cpu().numpy(), rs.ravel())


def test_w4_mx_full_size():
    """Both operands of workload 4 (A and B, 8192 x 8192 with 0.1 % of
    entries x100) in MX-32 blocks: codes and E8M0 scales bit-exact."""
    for t in wl.w4_operands(DEV):
        q = _u8(t.shape)
        e = _u8(8192 * 256)
        sq.fp8_quantize(t, sq.E4M3, sq.MX32, q, scales_out=e)
        torch.cuda.synchronize()
        rq, re, _, _ = o.quantize_mx32(np32(t), sq.E4M3)
        assert np.array_equal(codes(q), rq) and np.array_equal(e.cpu().numpy(), re.ravel())


def test_w5_largest_cast_full_size():
    """The largest cast of the FFN step: the 16384 x 14336 gradient in E5M2
    with its transposed copy, delayed scaling."""
    M, N = 16384, 14336
    dy = wl.linear_dy(5, 0, 0, M, N, DEV)
    H = 16
    st = torch.tensor(o.state_init(H), device=DEV)
    st[H] = 57344.0 / 0.006
    ref_state = st.cpu().numpy().copy()
    q, qT = _u8((M, N)), _u8((N, M))
    sq.fp8_quantize(dy, sq.E5M2, sq.TENSOR, q, qT=qT, delayed_state=st, history_len=H)
    torch.cuda.synchronize()
    rq, _ = o.quantize_delayed(np32(dy), sq.E5M2, ref_state)
    gq = codes(q)
    assert np.array_equal(gq, rq)
    del gq
    gqt = codes(qT)
    assert np.array_equal(gqt, rq.T)
    assert st.cpu().numpy().tobytes() == ref_state.tobytes()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(128, 128), (384, 512)])
def test_mx32_tiled_scales(fmt, shape):
    from _helpers import mx_untile
    R, C = shape
    x = wl.with_scaled_fraction(shape, 0.01, 100.0, 31 + R)
    q = _u8(shape)
    e = _u8(R * C // 32)
    sq.fp8_quantize(x.to(DEV), fmt, sq.MX32_TILED, q, scales_out=e)
    torch.cuda.synchronize()
    rq, re, _, _ = o.quantize_mx32(np32(x), fmt)
    assert np.array_equal(codes(q), rq)
    assert np.array_equal(mx_untile(e.cpu().numpy(), R, C), re)


@pytest.mark.parametrize("H", [1, 1024])
def test_history_length_variants(H):
    """The tutorial's suggested amax_history_len=1024 (and the degenerate 1):
    40 steps of cast + update with a spike, bit-exact against the oracle."""
    states = torch.empty(2 * (H + 2), dtype=torch.float32, device=DEV)
    sq.fp8_scale_init(states, 2, H)
    ref = [o.state_init(H) for _ in range(2)]
    fmts = [sq.E4M3, sq.E5M2]
    g = torch.Generator().manual_seed(H)
    for step in range(40):
        for r in range(2):
            x = (torch.randn((32, 256), generator=g) * (1.0 + (step % 7))).to(torch.bfloat16)
            if step == 3:
                x[0, 0] = 3000.0
            q = _u8((32, 256))
            sq.fp8_quantize(x.to(DEV), fmts[r], sq.TENSOR, q, delayed_state=states[r * (H + 2):(r + 1) * (H + 2)],
                            history_len=H)
            o.quantize_delayed(np32(x), fmts[r], ref[r])
        sq.fp8_update_scale(states, 2, H, fmts)
        for r in range(2):
            o.update_scale(ref[r], fmts[r])
    torch.cuda.synchronize()
    assert states.cpu().numpy().tobytes() == np.concatenate(ref).tobytes()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(256, 384), (128, 144), (384, 128)])
def test_column_tiles_128x1(fmt, shape):
    R, C = shape
    x = wl.student_t3(shape, 61 + R + C)
    x[130 % R, 5] = 900.0
    q, qT = _u8(shape), _u8((C, R))
    s = _f32((R // 128) * C)
    sat = torch.zeros(1, dtype=torch.int64, device=DEV)
    sq.fp8_quantize(x.to(DEV), fmt, sq.TILE_128x1, q, qT=qT, scales_out=s, sat_count=sat)
    torch.cuda.synchronize()
    rq, rs, _, rsat = o.quantize_tile128x1(np32(x), fmt)
    assert np.array_equal(codes(q), rq)
    assert np.array_equal(codes(qT), rq.T)
    assert np.array_equal(s.cpu().numpy(), rs.ravel())
    assert int(sat.item()) == rsat


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(256, 384), (128, 128)])
def test_column_mx_blocks(fmt, shape):
    from _helpers import mx_untile
    R, C = shape
    x = wl.with_scaled_fraction(shape, 0.01, 100.0, 71 + R)
    x[32:64, 3] = 0.0
    qT = _u8((C, R))
    e = _u8(R * C // 32)
    sq.fp8_quantize(x.to(DEV), fmt, sq.MX32_COL_TILED, None, qT=qT, scales_out=e)
    torch.cuda.synchronize()
    rq, re, _, _ = o.quantize_mx32_col(np32(x), fmt)
    assert np.array_equal(codes(qT), rq.T)
    # the tiled scales belong to qT = [C][R]; canonical qT scales are re^T
    assert np.array_equal(mx_untile(e.cpu().numpy(), C, R), re.T)


@pytest.mark.parametrize("fmt", FMTS)
def test_block_128x128_with_transpose(fmt):
    x = wl.normal((256, 384), 0.02, 81)
    q, qT = _u8((256, 384)), _u8((384, 256))
    s = _f32(6)
    sq.fp8_quantize(x.to(DEV), fmt, sq.BLOCK_128x128, q, qT=qT, scales_out=s)
    torch.cuda.synchronize()
    rq, rs, _, _ = o.quantize_block128(np32(x), fmt)
    assert np.array_equal(codes(q), rq) and np.array_equal(codes(qT), rq.T)
    assert np.array_equal(s.cpu().numpy(), rs.ravel())


@pytest.mark.parametrize("fmt", FMTS)
def test_pow2_tiles_blocks_and_floor_mx(fmt):
    """Recipe variants: power-of-two 1x128 tiles, power-of-two 128x128 blocks
    and the OCP-floor MX rule, all with E8M0 codes in the tiled layout."""
    from _helpers import mx_untile
    R, C = 256, 384
    x = wl.with_scaled_fraction((R, C), 0.01, 100.0, 111)
    x[7, 40] = 1.9 * 2 ** 10                       # significand > 1.75: the floor rule clips it
    xd = x.to(DEV)
    xf = np32(x)
    q, e = _u8((R, C)), _u8(R * C // 32)
    sat = torch.zeros(1, dtype=torch.int64, device=DEV)
    sq.fp8_quantize(xd, fmt, sq.TILE_1x128_POW2, q, scales_out=e, sat_count=sat)
    torch.cuda.synchronize()
    rq, re, rsat = o.quantize_tile1x128_pow2(xf, fmt)
    assert np.array_equal(codes(q), rq) and int(sat.item()) == rsat == 0
    assert np.array_equal(mx_untile(e.cpu().numpy(), R, C), np.repeat(re, 4, axis=1))
    sq.fp8_quantize(xd, fmt, sq.BLOCK_128x128_POW2, q, scales_out=e)
    torch.cuda.synchronize()
    rq, re, _ = o.quantize_block128_pow2(xf, fmt)
    assert np.array_equal(codes(q), rq)
    assert np.array_equal(mx_untile(e.cpu().numpy(), R, C), np.repeat(np.repeat(re, 128, axis=0), 4, axis=1))
    sat.zero_()
    sq.fp8_quantize(xd, fmt, sq.MX32_FLOOR_TILED, q, scales_out=e, sat_count=sat)
    torch.cuda.synchronize()
    rq, re, rsat = o.quantize_mx32_floor(xf, fmt)
    assert np.array_equal(codes(q), rq) and int(sat.item()) == rsat >= 1
    assert np.array_equal(mx_untile(e.cpu().numpy(), R, C), re)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(256, 384), (128, 128), (384, 256), (640, 1152), (1152, 512)])
def test_rows_cols_pow2_tiles(fmt, shape):
    """Power-of-two 1x128 row tiles and 128x1 column tiles in one pass: codes
    bit-exact against the oracle's power-of-two quantisers; each tile's E8M0
    code fills the four 32-blocks it covers in the tiled layouts of x and
    x^T; an outlier and a NaN are planted."""
    from _helpers import mx_untile
    R, C = shape
    x = wl.student_t3(shape, 91 + R + C)
    x[3, 130 % C] = 700.0
    x[R - 1, 5] = float("nan")
    xd = x.to(DEV)
    q, qT = _u8(shape), _u8((C, R))
    rs, cs = _u8((R * C // 32,)), _u8((R * C // 32,))
    sq.fp8_quantize_rows_cols(xd, fmt, sq.TILE_1x128_POW2, q, rs, qT, cs)
    torch.cuda.synchronize()
    xf = np32(x)
    rq, re, _ = o.quantize_tile1x128_pow2(xf, fmt)
    cq, ce, _ = o.quantize_tile128x1_pow2(xf, fmt)
    assert np.array_equal(mx_untile(rs.cpu().numpy(), R, C), np.repeat(re, 4, axis=1))
    assert np.array_equal(mx_untile(cs.cpu().numpy(), C, R), np.repeat(ce.T, 4, axis=1))
    assert nan_aware_codes_equal(codes(q), rq, fmt)
    assert nan_aware_codes_equal(codes(qT), cq.T, fmt)


@pytest.mark.parametrize("unit", [sq.TILE_1x128, sq.MX32_TILED])
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(256, 384), (128, 128), (384, 256), (640, 1152), (1152, 512)])
def test_rows_cols_one_pass(unit, fmt, shape):
    """fp8_quantize_rows_cols gives bit-identical results to the two separate
    casts (row units into q, column units into qT), and matches the oracle's
    row-unit and column-unit quantisers; an outlier and a NaN are planted."""
    from _helpers import mx_untile
    R, C = shape
    x = wl.student_t3(shape, 81 + R + C)
    x[3, 130 % C] = 700.0
    x[R - 1, 5] = float("nan")
    xd = x.to(DEV)
    mx = unit == sq.MX32_TILED
    col_unit = sq.MX32_COL_TILED if mx else sq.TILE_128x1
    q, qT = _u8(shape), _u8((C, R))
    if mx:
        rs, cs = _u8((R * C // 32,)), _u8((R * C // 32,))
    else:
        rs, cs = _f32(R * (C // 128)), _f32((R // 128) * C)
    sq.fp8_quantize_rows_cols(xd, fmt, unit, q, rs, qT, cs)
    q2, qT2 = _u8(shape), _u8((C, R))
    rs2, cs2 = torch.empty_like(rs), torch.empty_like(cs)
    sq.fp8_quantize(xd, fmt, unit, q2, scales_out=rs2)
    sq.fp8_quantize(xd, fmt, col_unit, None, qT=qT2, scales_out=cs2)
    torch.cuda.synchronize()
    assert torch.equal(q, q2) and torch.equal(qT, qT2)
    assert torch.equal(rs.view(torch.uint8), rs2.view(torch.uint8))
    assert torch.equal(cs.view(torch.uint8), cs2.view(torch.uint8))
    # against the oracle
    xf = np32(x)
    if mx:
        rq, re, _, _ = o.quantize_mx32(xf, fmt)
        cq, ce, _, _ = o.quantize_mx32_col(xf, fmt)
        assert np.array_equal(mx_untile(rs.cpu().numpy(), R, C), re)
        assert np.array_equal(mx_untile(cs.cpu().numpy(), C, R), ce.T)
    else:
        rq, rsc, _, _ = o.quantize_tile1x128(xf, fmt)
        cq, csc, _, _ = o.quantize_tile128x1(xf, fmt)
        assert np.array_equal(rs.cpu().numpy().view(np.uint32), rsc.ravel().view(np.uint32))
        assert np.array_equal(cs.cpu().numpy().view(np.uint32), csc.ravel().view(np.uint32))
    assert nan_aware_codes_equal(codes(q), rq, fmt)
    assert nan_aware_codes_equal(codes(qT), cq.T, fmt)
