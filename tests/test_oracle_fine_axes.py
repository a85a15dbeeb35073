"""Oracle pin: the fine-grained backward scales each operand along its own
GEMM's contraction dimension ("Week 14. Scaling laws, precision, parallelism",
absmax bullet: 1x128 activation tiles and 128x128 weight blocks, the
DeepSeek-V3 granularity; MX blocks of 32).

The pages do not say along which axis the backward operands are re-scaled;
the reading taken is the contraction dimension of each GEMM (dgrad contracts
over N, wgrad over the tokens M).  One planted outlier per tensor must change
exactly one scale of each backward operand, at the unit the reading puts it
in, and nowhere else; a transposed reading (dy tiled along M for dgrad, or
along N for wgrad) would move or multiply the changed entries.  The backward
products are then the float64 products of exactly those operands.
"""
import numpy as np
import pytest

import oracle as o

M, N, K = 256, 384, 512
DY_AT, X_AT, W_AT = (130, 200), (70, 300), (260, 45)


def _inputs(seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32)
    w = (0.02 * rng.standard_normal((N, K))).astype(np.float32)
    dy = (1e-3 * rng.standard_normal((M, N))).astype(np.float32)
    return x, w, dy


def _operands(x, w, dy, gran):
    if gran == o.GRAN_TILE_1x128:
        qw, sw, _, _ = o.quantize_block128(w, o.E4M3)
        st = {"x": x, "w": w, "qw": qw, "sw": sw}
    elif gran == o.GRAN_TILE_POW2:
        qw, ew, _ = o.quantize_block128_pow2(w, o.E4M3)
        st = {"x": x, "w": w, "qw": qw, "sw": ew}
    else:
        st = {"x": x, "w": w}
    return o.linear_fine_bwd_operands(st, dy, gran, o.E5M2)


def _changed(a, b):
    return {tuple(int(v) for v in i) for i in np.argwhere(np.asarray(a) != np.asarray(b))}


# expected changed unit per operand, from the contraction-dimension reading
EXPECTED = {
    o.GRAN_TILE_1x128: {
        "dgrad_dy": ((M, N // 128), {(DY_AT[0], DY_AT[1] // 128)}),          # 1x128 along N
        "dgrad_w": ((N // 128, K // 128), {(W_AT[0] // 128, W_AT[1] // 128)}),  # W's 128x128 blocks
        "wgrad_dy": ((M // 128, N), {(DY_AT[0] // 128, DY_AT[1])}),          # 128x1 along M
        "wgrad_x": ((M // 128, K), {(X_AT[0] // 128, X_AT[1])}),             # 128x1 along M
    },
    o.GRAN_TILE_POW2: {      # the same units, power-of-two scales
        "dgrad_dy": ((M, N // 128), {(DY_AT[0], DY_AT[1] // 128)}),
        "dgrad_w": ((N // 128, K // 128), {(W_AT[0] // 128, W_AT[1] // 128)}),
        "wgrad_dy": ((M // 128, N), {(DY_AT[0] // 128, DY_AT[1])}),
        "wgrad_x": ((M // 128, K), {(X_AT[0] // 128, X_AT[1])}),
    },
    o.GRAN_MX32: {
        "dgrad_dy": ((M, N // 32), {(DY_AT[0], DY_AT[1] // 32)}),            # 32 along N
        "dgrad_w": ((N // 32, K), {(W_AT[0] // 32, W_AT[1])}),               # W, 32 along N
        "wgrad_dy": ((M // 32, N), {(DY_AT[0] // 32, DY_AT[1])}),            # 32 along M
        "wgrad_x": ((M // 32, K), {(X_AT[0] // 32, X_AT[1])}),               # 32 along M
    },
}


@pytest.mark.parametrize("gran", [o.GRAN_TILE_1x128, o.GRAN_TILE_POW2, o.GRAN_MX32])
def test_one_outlier_changes_exactly_its_unit_per_operand(gran):
    x, w, dy = _inputs(1)
    base = _operands(x, w, dy, gran)
    x2, w2, dy2 = x.copy(), w.copy(), dy.copy()
    dy2[DY_AT] = 0.5          # ~100x the gradient's spread
    x2[X_AT] = 60.0
    w2[W_AT] = 1.5
    spiked = _operands(x2, w2, dy2, gran)
    for name, (shape, where) in EXPECTED[gran].items():
        assert np.shape(spiked[name][1]) == shape, name
        assert _changed(base[name][1], spiked[name][1]) == where, name
        # the outlier itself is at the top of its unit's range: it maps to
        # (about) fmax of its format, so the other codes of that unit shrink
        fmax = o.fmax(o.E5M2 if "dy" in name else o.E4M3)
        at = {"dgrad_dy": DY_AT, "wgrad_dy": DY_AT, "wgrad_x": X_AT, "dgrad_w": W_AT}[name]
        fmt = o.E5M2 if "dy" in name else o.E4M3
        assert o.decode(fmt, int(spiked[name][0][at])) >= fmax / 2, name


@pytest.mark.parametrize("gran", [o.GRAN_TILE_1x128, o.GRAN_TILE_POW2, o.GRAN_MX32])
def test_backward_products_use_those_operands(gran):
    x, w, dy = _inputs(2)
    st, _ = o.linear_fine_fwd(x, w, gran)
    ops = o.linear_fine_bwd_operands(st, dy, gran, o.E5M2)
    dX, dW = o.linear_fine_bwd(st, dy, gran, o.E5M2)
    assert np.array_equal(dX, ops["dgrad_dy"][2] @ ops["dgrad_w"][2])
    assert np.array_equal(dW, ops["wgrad_dy"][2].T @ ops["wgrad_x"][2])
    # and they approximate the exact backward of the unquantised tensors
    ex = dy.astype(np.float64) @ w.astype(np.float64)
    ew = dy.astype(np.float64).T @ x.astype(np.float64)
    assert np.max(np.abs(dX - ex)) <= 0.1 * np.max(np.abs(ex))
    assert np.max(np.abs(dW - ew)) <= 0.1 * np.max(np.abs(ew))


def test_transposed_reading_would_differ():
    """The pin distinguishes the axes: quantising dy for dgrad in column
    tiles (along M) puts the spike's scale at a different unit."""
    x, w, dy = _inputs(3)
    dy2 = dy.copy()
    dy2[DY_AT] = 0.5
    _, s_rows, _, _ = o.quantize_tile1x128(dy, o.E5M2)
    _, s_rows2, _, _ = o.quantize_tile1x128(dy2, o.E5M2)
    _, s_cols, _, _ = o.quantize_tile128x1(dy, o.E5M2)
    _, s_cols2, _, _ = o.quantize_tile128x1(dy2, o.E5M2)
    assert _changed(s_rows, s_rows2) == {(130, 1)}
    assert _changed(s_cols, s_cols2) == {(1, 200)}
