"""Pins the oracle's dequantisation and GEMM reference.

The GEMM is a float64 product of exactly dequantised operands; these tests
pin the contraction (A [M,K] times B [N,K] over K), the scale layouts and the
output rounding against exact integer arithmetic and tiny brute force.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle as o


def _codes_of_small_ints(rng, shape, fmt, lo=-8, hi=8):
    v = rng.integers(lo, hi + 1, shape)
    q = np.vectorize(lambda t: o.encode(fmt, float(t)))(v).astype(np.uint8)
    return v, q


@pytest.mark.parametrize("fa,fb", [(o.E4M3, o.E4M3), (o.E5M2, o.E4M3)])
def test_integer_operands_exact(fa, fb):
    """Small integers are exact in both formats; with unit scales the GEMM is an
    integer matrix product (computed here in int64, a different code path)."""
    rng = np.random.default_rng(0)
    M, N, K = 17, 23, 300
    va, qa = _codes_of_small_ints(rng, (M, K), fa)
    vb, qb = _codes_of_small_ints(rng, (N, K), fb)
    ah = o.dequantize(qa, fa, o.GRAN_TENSOR, 1.0)
    bh = o.dequantize(qb, fb, o.GRAN_TENSOR, 1.0)
    assert np.array_equal(ah, va) and np.array_equal(bh, vb)
    r = o.gemm_ref(ah, bh)
    assert np.array_equal(r, (va.astype(np.int64) @ vb.astype(np.int64).T).astype(np.float64))


def test_identity_b_returns_dequantised_a():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((9, 32)).astype(np.float32)
    qa, amax, s, _ = o.quantize_tensor_current(x, o.E4M3)
    ah = o.dequantize(qa, o.E4M3, o.GRAN_TENSOR, s)
    one = o.encode(o.E4M3, 1.0)
    qb = np.where(np.eye(32, dtype=bool), one, 0).astype(np.uint8)
    r = o.gemm_ref(ah, o.dequantize(qb, o.E4M3, o.GRAN_TENSOR, 1.0))
    assert np.array_equal(r, ah)


def test_brute_force_fractions_tiny():
    """3x5x7 with distinct values: exact rational sum-of-products in pure
    Python loops must equal the float64 reference (exact here)."""
    rng = np.random.default_rng(2)
    M, N, K = 3, 5, 7
    qa = rng.integers(0, 0x7E, (M, K)).astype(np.uint8)
    qb = rng.integers(0, 0x7B, (N, K)).astype(np.uint8)
    ah = o.dequantize(qa, o.E4M3, o.GRAN_TENSOR, 0.5)
    bh = o.dequantize(qb, o.E5M2, o.GRAN_TENSOR, 0.25)
    r = o.gemm_ref(ah, bh, bias=np.float32([1, 2, 3, 4, 5]))
    for i in range(M):
        for j in range(N):
            acc = Fraction(j + 1)
            for k in range(K):
                acc += Fraction(o.decode(o.E4M3, int(qa[i, k]))) * Fraction(1, 2) * \
                       Fraction(o.decode(o.E5M2, int(qb[j, k]))) * Fraction(1, 4)
            assert float(acc) == r[i, j]


def test_dequant_scale_layouts():
    """A code of 1.0 everywhere dequantises to the expanded scale grid."""
    one4 = o.encode(o.E4M3, 1.0)
    R, C = 256, 384
    q = np.full((R, C), one4, np.uint8)
    rng = np.random.default_rng(3)
    s_tile = rng.uniform(0.1, 2, (R, C // 128)).astype(np.float32)
    assert np.array_equal(o.dequantize(q, o.E4M3, o.GRAN_TILE_1x128, s_tile),
                          np.repeat(s_tile, 128, axis=1).astype(np.float64))
    s_blk = rng.uniform(0.1, 2, (R // 128, C // 128)).astype(np.float32)
    assert np.array_equal(o.dequantize(q, o.E4M3, o.GRAN_BLOCK_128x128, s_blk),
                          np.repeat(np.repeat(s_blk, 128, axis=0), 128, axis=1).astype(np.float64))
    e = rng.integers(100, 150, (R, C // 32)).astype(np.uint8)
    assert np.array_equal(o.dequantize(q, o.E4M3, o.GRAN_MX32, e),
                          np.repeat(2.0 ** (e.astype(np.float64) - 127), 32, axis=1))


def test_quantize_then_gemm_close_to_fp64_product():
    """End-to-end sanity: per-tensor E4M3 quantisation of N(0,1) operands keeps
    the product within the format's relative precision (2^-4 per element, far
    less after averaging over K)."""
    rng = np.random.default_rng(4)
    a = rng.standard_normal((64, 512)).astype(np.float32)
    b = rng.standard_normal((48, 512)).astype(np.float32)
    qa, _, sa, _ = o.quantize_tensor_current(a, o.E4M3)
    qb, _, sb, _ = o.quantize_tensor_current(b, o.E4M3)
    r = o.gemm_ref(o.dequantize(qa, o.E4M3, 0, sa), o.dequantize(qb, o.E4M3, 0, sb))
    exact = a.astype(np.float64) @ b.astype(np.float64).T
    assert np.max(np.abs(r - exact)) / np.max(np.abs(exact)) < 0.05


def test_epilogue_rounding():
    r = np.array([[257.0, 1.0 + 2 ** -30, -3.0]])
    f = o.epilogue(r, out_bf16=False)
    assert f.dtype == np.float32 and f[0, 1] == 1.0
    b = o.epilogue(r, out_bf16=True)
    assert b.dtype == np.uint16
    assert o.bf16_bits_to_f32(b).tolist() == [[256.0, 1.0, -3.0]]


def test_linear_delayed_exact_on_representable_inputs():
    """The delayed linear layer end to end.  Each role's state gets its own
    power-of-two multiplier m and scale s = 1/m (x: 2, W: 4, dy: 8), and the
    inputs are small integers, so every scaled value is exact in its format:
    x*2 within +-16 in E4M3, W*4 multiples of 4 within +-32 in E4M3, dy*8
    multiples of 8 within +-32 in E5M2.  The forward, dgrad and wgrad must
    then be the exact integer products R = x W^T, dX = dy W, dW = dy^T x, on
    non-square shapes where a transposed operand, a scale taken from the
    wrong role or the wrong format would show.  Each cast also records its
    tensor's amax in history slot 0."""
    rng = np.random.default_rng(5)
    M, K, N, H = 6, 5, 7, 4
    xi = rng.integers(-8, 9, (M, K))
    wi = rng.integers(-8, 9, (N, K))
    di = rng.integers(-4, 5, (M, N))
    states = []
    for m in (2.0, 4.0, 8.0):
        st = o.state_init(H)
        st[H], st[H + 1] = m, 1.0 / m
        states.append(st)
    sx, sw, sd = states
    qx, fx, qw, fw, r = o.linear_fwd_delayed(xi.astype(np.float32), wi.astype(np.float32), sx, sw)
    assert (fx, fw) == (0.5, 0.25)
    _, fd, dX, dW = o.linear_bwd_delayed(di.astype(np.float32), sd, o.E5M2, qx, fx, qw, fw)
    assert fd == 0.125
    assert np.array_equal(r, xi @ wi.T)
    assert np.array_equal(dX, di @ wi)
    assert np.array_equal(dW, di.T @ xi)
    assert (sx[0], sw[0], sd[0]) == (np.abs(xi).max(), np.abs(wi).max(), np.abs(di).max())
