"""GPU parity of the tcgen05 FP8 GEMM against the oracle's float64 product of
the dequantised operands (tolerance in tests/_helpers.py), plus closed forms
that must come out exact."""
import numpy as np
import pytest
import torch

import oracle as o
import scaled_quantize_gemm_gb300 as sq
from scaled_quantize_gemm_gb300 import workloads as wl

from _helpers import assert_gemm_close, codes, gemm_error, np32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _int_codes(rng, shape, fmt, lo, hi):
    v = rng.integers(lo, hi + 1, shape)
    table = {t: o.encode(fmt, float(t)) for t in range(lo, hi + 1)}
    q = np.vectorize(table.get)(v).astype(np.uint8)
    return v, q


def _one(v=1.0):
    return torch.tensor([v], dtype=torch.float32, device=DEV)


def _gemm_t(qa, fa, sa, qb, fb, sb, out_dtype, bias=None):
    M, N = qa.shape[0], qb.shape[0]
    D = torch.empty((M, N), dtype=out_dtype, device=DEV)
    sq.fp8_gemm(qa, fa, sa, sq.TENSOR, qb, fb, sb, sq.TENSOR, D, bias=bias)
    torch.cuda.synchronize()
    return D


@pytest.mark.parametrize("fa,fb", [(sq.E4M3, sq.E4M3), (sq.E5M2, sq.E4M3), (sq.E4M3, sq.E5M2), (sq.E5M2, sq.E5M2)])
def test_integer_operands_exact(fa, fb):
    """Small integers are exact codes; with unit scales every partial sum is an
    integer below 2^24, so fp32 accumulation must reproduce the int64 product."""
    rng = np.random.default_rng(1)
    M, N, K = 256, 512, 384
    va, qa = _int_codes(rng, (M, K), fa, -8, 8)
    vb, qb = _int_codes(rng, (N, K), fb, -8, 8)
    D = _gemm_t(torch.from_numpy(qa).to(DEV), fa, _one(), torch.from_numpy(qb).to(DEV), fb, _one(), torch.float32)
    exact = (va.astype(np.int64) @ vb.astype(np.int64).T).astype(np.float32)
    assert np.array_equal(D.cpu().numpy(), exact)


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 128), (4096, 5120, 128)])
def test_multi_wave_exact(M, N, K):
    """Several waves of 256x256 tiles on the persistent CTA pairs, with a
    last, partial wave (4096^2: 256 tiles, 28 left after three waves of 76
    pairs; 4096 x 5120: 320 tiles, 16 left).  Integer operands and unit
    scales make every output exact, so a tile scheduled onto the wrong pair,
    rows or columns shows."""
    rng = np.random.default_rng(7)
    va, qa = _int_codes(rng, (M, K), sq.E4M3, -8, 8)
    vb, qb = _int_codes(rng, (N, K), sq.E4M3, -8, 8)
    D = _gemm_t(torch.from_numpy(qa).to(DEV), sq.E4M3, _one(), torch.from_numpy(qb).to(DEV), sq.E4M3, _one(),
                torch.float32)
    exact = va.astype(np.float64) @ vb.astype(np.float64).T      # integers far below 2^53
    assert np.array_equal(D.cpu().numpy().astype(np.float64), exact)


def test_identity_b():
    rng = np.random.default_rng(2)
    M, K = 384, 256
    qa = rng.integers(0, 256, (M, K)).astype(np.uint8)
    qa[(qa & 0x7F) == 0x7F] = 0x10                        # no NaN codes
    one = o.encode(o.E4M3, 1.0)
    qb = np.where(np.eye(K, dtype=bool), one, 0).astype(np.uint8)
    D = _gemm_t(torch.from_numpy(qa).to(DEV), sq.E4M3, _one(0.5), torch.from_numpy(qb).to(DEV), sq.E4M3, _one(),
                torch.float32)
    ref = o.dequantize(qa, o.E4M3, o.GRAN_TENSOR, 0.5).astype(np.float32)
    assert np.array_equal(D.cpu().numpy(), ref)


def test_accumulation_width_long_k():
    """K = 16384 with integer operands 0..16 (exact in E4M3): every running sum
    is an integer below 2^22 and exact in fp32, so the result must be exact --
    a narrow accumulator (the week-14 page's ~14-bit FP8 accumulator note)
    would lose the low bits of these ~2^21 sums."""
    rng = np.random.default_rng(3)
    M, N, K = 128, 256, 16384
    va, qa = _int_codes(rng, (M, K), o.E4M3, 0, 16)
    vb, qb = _int_codes(rng, (N, K), o.E4M3, 0, 16)
    D = _gemm_t(torch.from_numpy(qa).to(DEV), sq.E4M3, _one(), torch.from_numpy(qb).to(DEV), sq.E4M3, _one(),
                torch.float32)
    exact = (va.astype(np.int64) @ vb.astype(np.int64).T)
    assert 2 ** 20 < exact.max() < 2 ** 22
    assert np.array_equal(D.cpu().numpy().astype(np.int64), exact)


def _quant_tensor(x, fmt):
    xd = x.to(DEV)
    q = torch.empty(x.shape, dtype=torch.uint8, device=DEV)
    amax = torch.zeros(1, device=DEV)
    s = torch.zeros(1, device=DEV)
    sq.fp8_quantize(xd, fmt, sq.TENSOR, q, scales_out=s, amax_out=amax)
    return q, s


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (200, 136, 80), (384, 768, 1024), (1, 8, 16), (130, 264, 144)])
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_per_tensor_vs_oracle(M, N, K, out):
    a = wl.normal((M, K), 1.0, 11 + M, dtype=torch.float32)
    b = wl.normal((N, K), 1.0, 12 + N, dtype=torch.float32)
    qa, sa = _quant_tensor(a, sq.E4M3)
    qb, sb = _quant_tensor(b, sq.E4M3)
    bias = torch.randn(N, generator=torch.Generator().manual_seed(5)).to(DEV) if M == 384 else None
    D = _gemm_t(qa, sq.E4M3, sa, qb, sq.E4M3, sb, out, bias=bias)
    R = o.gemm_ref(o.dequantize(codes(qa), 0, 0, sa.item()), o.dequantize(codes(qb), 0, 0, sb.item()),
                   bias=None if bias is None else bias.cpu().numpy())
    assert_gemm_close(D, R)


def test_w1_per_tensor_current_linear():
    """Workload 1: A, B 256x256 fp32 with outliers of 30, per-tensor current
    E4M3, M=N=K=256, fp32 output."""
    a, b = wl.w1_operands()
    qa, sa = _quant_tensor(a, sq.E4M3)
    qb, sb = _quant_tensor(b, sq.E4M3)
    D = _gemm_t(qa, sq.E4M3, sa, qb, sq.E4M3, sb, torch.float32)
    rqa, _, rsa, _ = o.quantize_tensor_current(a.numpy(), o.E4M3)
    rqb, _, rsb, _ = o.quantize_tensor_current(b.numpy(), o.E4M3)
    assert np.array_equal(codes(qa), rqa) and np.array_equal(codes(qb), rqb)
    R = o.gemm_ref(o.dequantize(rqa, 0, 0, rsa), o.dequantize(rqb, 0, 0, rsb))
    assert_gemm_close(D, R)
    assert gemm_error(D, R) < 1e-5


def test_k_zero_and_m_zero():
    qa = torch.empty((64, 0), dtype=torch.uint8, device=DEV)
    qb = torch.empty((32, 0), dtype=torch.uint8, device=DEV)
    bias = torch.arange(32, dtype=torch.float32, device=DEV)
    D = torch.full((64, 32), 7.0, device=DEV)
    sq.fp8_gemm(qa, 0, _one(), 0, qb, 0, _one(), 0, D, bias=bias, M=64, N=32, K=0)
    torch.cuda.synchronize()
    assert torch.equal(D, bias.expand(64, 32))
    E = torch.full((0, 32), 1.0, device=DEV)
    sq.fp8_gemm(torch.empty((0, 16), dtype=torch.uint8, device=DEV), 0, _one(), 0,
                torch.zeros((32, 16), dtype=torch.uint8, device=DEV), 0, _one(), 0, E, M=0, N=32, K=16)
    torch.cuda.synchronize()


def _quant_tile_block(x, w):
    M, K = x.shape
    N = w.shape[0]
    qx = torch.empty((M, K), dtype=torch.uint8, device=DEV)
    qw = torch.empty((N, K), dtype=torch.uint8, device=DEV)
    sx = torch.empty(M * (K // 128), dtype=torch.float32, device=DEV)
    sw = torch.empty((N // 128) * (K // 128), dtype=torch.float32, device=DEV)
    sq.fp8_quantize(x.to(DEV), sq.E4M3, sq.TILE_1x128, qx, scales_out=sx)
    sq.fp8_quantize(w.to(DEV), sq.E4M3, sq.BLOCK_128x128, qw, scales_out=sw)
    return qx, sx, qw, sw


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 384, 1024), (200, 256, 512)])
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_tile_block_promotion_vs_oracle(M, N, K, out):
    x = wl.student_t3((M, K), 21 + M)
    w = wl.normal((N, K), 0.02, 22 + N)
    qx, sx, qw, sw = _quant_tile_block(x, w)
    D = torch.empty((M, N), dtype=out, device=DEV)
    sq.fp8_gemm(qx, sq.E4M3, sx, sq.TILE_1x128, qw, sq.E4M3, sw, sq.BLOCK_128x128, D)
    torch.cuda.synchronize()
    R = o.gemm_ref(o.dequantize(codes(qx), 0, o.GRAN_TILE_1x128, sx.cpu().numpy().reshape(M, K // 128)),
                   o.dequantize(codes(qw), 0, o.GRAN_BLOCK_128x128, sw.cpu().numpy().reshape(N // 128, K // 128)))
    assert_gemm_close(D, R)


@pytest.mark.parametrize("M,N,K", [(328, 640, 512), (128, 1152, 384)])
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_tile_block_promotion_bias_ragged_tiles(M, N, K, out):
    """Promotion with bias, N % 256 == 128 (the last 256-wide tile holds one
    weight block and columns past N) and a ragged M."""
    x = wl.student_t3((M, K), 31 + M)
    w = wl.normal((N, K), 0.02, 32 + N)
    bias = wl.normal((N,), 0.5, 33 + N, dtype=torch.float32).to(DEV)
    qx, sx, qw, sw = _quant_tile_block(x, w)
    D = torch.empty((M, N), dtype=out, device=DEV)
    sq.fp8_gemm(qx, sq.E4M3, sx, sq.TILE_1x128, qw, sq.E4M3, sw, sq.BLOCK_128x128, D, bias=bias)
    torch.cuda.synchronize()
    R = o.gemm_ref(o.dequantize(codes(qx), 0, o.GRAN_TILE_1x128, sx.cpu().numpy().reshape(M, K // 128)),
                   o.dequantize(codes(qw), 0, o.GRAN_BLOCK_128x128, sw.cpu().numpy().reshape(N // 128, K // 128)),
                   bias=bias.cpu().numpy())
    assert_gemm_close(D, R)


def _sample_rows(M, n, seed):
    return np.sort(np.random.default_rng(seed).choice(M, size=n, replace=False))


def test_w3_full_size_sampled_rows():
    """Workload 3 at full size (M=N=K=4096, bf16 out) in the launch
    configuration the bench times.  The reference is built from the oracle's
    own 1x128 / 128x128 quantisation of the inputs (which must equal the
    GPU's codes and scales); 256 sampled rows of the product checked."""
    x, w = wl.w3_operands(DEV)
    qx, sx, qw, sw = _quant_tile_block(x, w)
    D = torch.empty((4096, 4096), dtype=torch.bfloat16, device=DEV)
    sq.fp8_gemm(qx, sq.E4M3, sx, sq.TILE_1x128, qw, sq.E4M3, sw, sq.BLOCK_128x128, D)
    torch.cuda.synchronize()
    rqx, rsx, _, _ = o.quantize_tile1x128(np32(x), o.E4M3)
    rqw, rsw, _, _ = o.quantize_block128(np32(w), o.E4M3)
    assert np.array_equal(codes(qx), rqx) and np.array_equal(sx.cpu().numpy(), rsx.ravel())
    assert np.array_equal(codes(qw), rqw) and np.array_equal(sw.cpu().numpy(), rsw.ravel())
    rows = _sample_rows(4096, 256, 3)
    ah = o.dequantize(rqx[rows], 0, o.GRAN_TILE_1x128, rsx[rows])
    bh = o.dequantize(rqw, 0, o.GRAN_BLOCK_128x128, rsw)
    assert_gemm_close(D[rows], o.gemm_ref(ah, bh))


def test_w5_forward_gemm_full_size_sampled_rows():
    """The FFN up-projection of workload 5 (M=16384, K=4096, N=14336, bf16
    out) at full size, current per-tensor scaling; the reference comes from
    the oracle's own quantisation of x and W (equal to the GPU's codes and
    scales); 128 sampled rows against it."""
    M, K, N = 16384, 4096, 14336
    x = wl.linear_x(5, 0, 0, M, K, DEV)
    w = wl.linear_w(5, 0, N, K, DEV)
    qx, sx = _quant_tensor(x, sq.E4M3)
    qw, sw = _quant_tensor(w, sq.E4M3)
    D = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    sq.fp8_gemm(qx, sq.E4M3, sx, sq.TENSOR, qw, sq.E4M3, sw, sq.TENSOR, D)
    torch.cuda.synchronize()
    rqx, _, rsx, _ = o.quantize_tensor_current(np32(x), o.E4M3)
    rqw, _, rsw, _ = o.quantize_tensor_current(np32(w), o.E4M3)
    assert np.array_equal(codes(qx), rqx) and np.float32(sx.item()) == rsx
    assert np.array_equal(codes(qw), rqw) and np.float32(sw.item()) == rsw
    rows = _sample_rows(M, 128, 5)
    ah = o.dequantize(rqx[rows], 0, 0, rsx)
    bh = o.dequantize(rqw, 0, 0, rsw)
    assert_gemm_close(D[rows], o.gemm_ref(ah, bh))


# ---------------------------------------------------------------- MX-32 block scaling
def _quant_mx(x):
    R, C = x.shape
    q = torch.empty((R, C), dtype=torch.uint8, device=DEV)
    e = torch.empty(R * C // 32, dtype=torch.uint8, device=DEV)
    sq.fp8_quantize(x.to(DEV), sq.E4M3, sq.MX32_TILED, q, scales_out=e)
    return q, e


def _mx_gemm(qa, ea, qb, eb, out):
    D = torch.empty((qa.shape[0], qb.shape[0]), dtype=out, device=DEV)
    sq.fp8_gemm(qa, sq.E4M3, ea, sq.MX32_TILED, qb, sq.E4M3, eb, sq.MX32_TILED, D)
    torch.cuda.synchronize()
    return D


def test_mx_gemm_bias_vs_oracle():
    """MX-32 GEMM with bias (fp32 out), N % 256 == 128."""
    from _helpers import mx_untile
    M, N, K = 256, 640, 512
    a = wl.normal((M, K), 1.0, 41)
    b = wl.normal((N, K), 1.0, 42)
    bias = wl.normal((N,), 2.0, 43, dtype=torch.float32).to(DEV)
    qa, ea = _quant_mx(a)
    qb, eb = _quant_mx(b)
    D = torch.empty((M, N), dtype=torch.float32, device=DEV)
    sq.fp8_gemm(qa, sq.E4M3, ea, sq.MX32_TILED, qb, sq.E4M3, eb, sq.MX32_TILED, D, bias=bias)
    torch.cuda.synchronize()
    ah = o.dequantize(codes(qa), 0, o.GRAN_MX32, mx_untile(ea.cpu().numpy(), M, K))
    bh = o.dequantize(codes(qb), 0, o.GRAN_MX32, mx_untile(eb.cpu().numpy(), N, K))
    assert_gemm_close(D, o.gemm_ref(ah, bh, bias=bias.cpu().numpy()))


def test_mx_unit_scales_integer_exact():
    """E8M0 code 127 (= 1.0) everywhere and small-integer codes: the
    block-scaled MMA must reproduce the int64 product exactly."""
    rng = np.random.default_rng(7)
    M, N, K = 256, 384, 512
    va, qa = _int_codes(rng, (M, K), o.E4M3, -8, 8)
    vb, qb = _int_codes(rng, (N, K), o.E4M3, -8, 8)
    ea = torch.full((M * K // 32,), 127, dtype=torch.uint8, device=DEV)
    eb = torch.full((N * K // 32,), 127, dtype=torch.uint8, device=DEV)
    D = _mx_gemm(torch.from_numpy(qa).to(DEV), ea, torch.from_numpy(qb).to(DEV), eb, torch.float32)
    assert np.array_equal(D.cpu().numpy(), (va.astype(np.int64) @ vb.astype(np.int64).T).astype(np.float32))


def test_mx_power_of_two_scales_select_the_right_block():
    """One non-unit scale per operand at a time: a 2^k on row r, 32-block t of
    A must scale exactly the products of that block (checks the scale
    factors' row and K placement in tensor memory, and the per-MMA byte id)."""
    from _helpers import mx_untile
    rng = np.random.default_rng(8)
    M, N, K = 256, 256, 256
    va, qa = _int_codes(rng, (M, K), o.E4M3, -4, 4)
    vb, qb = _int_codes(rng, (N, K), o.E4M3, -4, 4)
    ta = np.full((M, K // 32), 127, np.uint8)
    tb = np.full((N, K // 32), 127, np.uint8)
    ta[37, 5] = 129      # x4
    ta[200, 0] = 126     # x0.5
    ta[99, 7] = 130      # x8
    tb[150, 3] = 128     # x2
    tb[3, 6] = 125       # x0.25

    def tile(can, R, C):
        out = np.zeros(R * C // 32, np.uint8)
        r = np.arange(R)[:, None]
        t = np.arange(C // 32)[None, :]
        off = ((r // 128) * (C // 128) + t // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (t % 4)
        out[off] = can
        assert np.array_equal(mx_untile(out, R, C), can)
        return out

    ea = torch.from_numpy(tile(ta, M, K)).to(DEV)
    eb = torch.from_numpy(tile(tb, N, K)).to(DEV)
    D = _mx_gemm(torch.from_numpy(qa).to(DEV), ea, torch.from_numpy(qb).to(DEV), eb, torch.float32)
    ah = va * np.repeat(2.0 ** (ta.astype(np.float64) - 127), 32, axis=1)
    bh = vb * np.repeat(2.0 ** (tb.astype(np.float64) - 127), 32, axis=1)
    assert np.array_equal(D.cpu().numpy().astype(np.float64), ah @ bh.T)


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 384, 512), (384, 256, 1024), (256, 384, 1536),
                                   (640, 256, 1536), (384, 640, 1152)])
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_mx_vs_oracle(M, N, K, out):
    from _helpers import mx_untile
    a = wl.with_scaled_fraction((M, K), 1e-3, 100.0, 41 + M)
    b = wl.with_scaled_fraction((N, K), 1e-3, 100.0, 42 + N)
    qa, ea = _quant_mx(a)
    qb, eb = _quant_mx(b)
    D = _mx_gemm(qa, ea, qb, eb, out)
    R = o.gemm_ref(o.dequantize(codes(qa), 0, o.GRAN_MX32, mx_untile(ea.cpu().numpy(), M, K)),
                   o.dequantize(codes(qb), 0, o.GRAN_MX32, mx_untile(eb.cpu().numpy(), N, K)))
    assert_gemm_close(D, R)


def test_w4_mx_full_size_sampled_rows():
    """Workload 4 at full size: A, B 8192 x 8192 with 0.1 % of entries x100,
    MX-32 E4M3, bf16 out.  The reference comes from the oracle's own MX-32
    quantisation of A and B (equal to the GPU's codes and, untiled, its E8M0
    scales); 128 sampled rows against it."""
    from _helpers import mx_untile
    a, b = wl.w4_operands(DEV)
    qa, ea = _quant_mx(a)
    qb, eb = _quant_mx(b)
    D = _mx_gemm(qa, ea, qb, eb, torch.bfloat16)
    rqa, rea, _, _ = o.quantize_mx32(np32(a), o.E4M3)
    rqb, reb, _, _ = o.quantize_mx32(np32(b), o.E4M3)
    del a, b
    assert np.array_equal(codes(qa), rqa) and np.array_equal(mx_untile(ea.cpu().numpy(), 8192, 8192), rea)
    assert np.array_equal(codes(qb), rqb) and np.array_equal(mx_untile(eb.cpu().numpy(), 8192, 8192), reb)
    rows = _sample_rows(8192, 128, 9)
    ah = o.dequantize(rqa[rows], 0, o.GRAN_MX32, rea[rows])
    bh = o.dequantize(rqb, 0, o.GRAN_MX32, reb)
    assert_gemm_close(D[rows], o.gemm_ref(ah, bh))


@pytest.mark.parametrize("Mt,N,K,with_bias", [(256, 384, 256, False), (384, 256, 512, False),
                                              (512, 208, 640, True), (128, 144, 1152, True)])
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_column_tile_gemm_vs_oracle(Mt, N, K, with_bias, out):
    """Mode for wgrad: both operands are the transposed codes of 128x1
    column-tile quantisations (contraction over the original rows Mt); the
    GEMM's N (here K) ragged at the 256-wide tile, GEMM M (here N) ragged at
    128, with and without bias."""
    dy = wl.normal((Mt, N), 1e-3, 91 + Mt)
    x = wl.student_t3((Mt, K), 92 + K)
    bias = wl.normal((K,), 1e-3, 93 + K, dtype=torch.float32).to(DEV) if with_bias else None
    qdT = torch.empty((N, Mt), dtype=torch.uint8, device=DEV)
    qxT = torch.empty((K, Mt), dtype=torch.uint8, device=DEV)
    sd = torch.empty((Mt // 128) * N, dtype=torch.float32, device=DEV)
    sx = torch.empty((Mt // 128) * K, dtype=torch.float32, device=DEV)
    sq.fp8_quantize(dy.to(DEV), sq.E5M2, sq.TILE_128x1, None, qT=qdT, scales_out=sd)
    sq.fp8_quantize(x.to(DEV), sq.E4M3, sq.TILE_128x1, None, qT=qxT, scales_out=sx)
    D = torch.empty((N, K), dtype=out, device=DEV)
    sq.fp8_gemm(qdT, sq.E5M2, sd, sq.TILE_128x1, qxT, sq.E4M3, sx, sq.TILE_128x1, D, bias=bias)
    torch.cuda.synchronize()
    rqd, rsd, _, _ = o.quantize_tile128x1(np32(dy), o.E5M2)
    rqx, rsx, _, _ = o.quantize_tile128x1(np32(x), o.E4M3)
    R = o.gemm_ref(o.dequantize(rqd, o.E5M2, o.GRAN_TILE_128x1, rsd).T,
                   o.dequantize(rqx, o.E4M3, o.GRAN_TILE_128x1, rsx).T,
                   bias=None if bias is None else bias.cpu().numpy())
    assert_gemm_close(D, R)


@pytest.mark.parametrize("M,N,K", [(256, 384, 512), (4096, 4096, 4096)])
def test_pow2_tiles_blocks_on_block_scaled_mma(M, N, K):
    """Power-of-two 1x128 tiles x power-of-two 128x128 blocks run on the
    block-scaled MMA (no promotion): parity with the oracle's product of the
    exactly dequantised operands (sampled rows at the full workload-3 size)."""
    x = wl.student_t3((M, K), 121 + M)
    w = wl.normal((N, K), 0.02, 122 + N)
    qx, qw = torch.empty((M, K), dtype=torch.uint8, device=DEV), torch.empty((N, K), dtype=torch.uint8, device=DEV)
    ex = torch.empty(M * K // 32, dtype=torch.uint8, device=DEV)
    ew = torch.empty(N * K // 32, dtype=torch.uint8, device=DEV)
    sq.fp8_quantize(x.to(DEV), sq.E4M3, sq.TILE_1x128_POW2, qx, scales_out=ex)
    sq.fp8_quantize(w.to(DEV), sq.E4M3, sq.BLOCK_128x128_POW2, qw, scales_out=ew)
    D = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    sq.fp8_gemm(qx, sq.E4M3, ex, sq.TILE_1x128_POW2, qw, sq.E4M3, ew, sq.BLOCK_128x128_POW2, D)
    torch.cuda.synchronize()
    rqx, rex, _ = o.quantize_tile1x128_pow2(np32(x), o.E4M3)
    rqw, rew, _ = o.quantize_block128_pow2(np32(w), o.E4M3)
    assert np.array_equal(codes(qx), rqx) and np.array_equal(codes(qw), rqw)
    rows = _sample_rows(M, min(M, 128), 11)
    ah = o.dequantize(rqx[rows], o.E4M3, o.GRAN_TILE_POW2, rex[rows])
    bh = o.dequantize(rqw, o.E4M3, o.GRAN_BLOCK_POW2, rew)
    assert_gemm_close(D[rows], o.gemm_ref(ah, bh))


# ---------------------------------------------------------------- MN-major operands
@pytest.mark.parametrize("a_mn,b_mn", [(False, True), (True, False), (True, True)])
@pytest.mark.parametrize("M,N,K,with_bias", [(256, 384, 512, False), (272, 400, 144, True), (128, 128, 16, False),
                                             (528, 256, 1040, True), (720, 592, 1328, True), (96, 1008, 416, False)])
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_mn_major_operands(a_mn, b_mn, M, N, K, with_bias, out):
    """fp8_gemm_layout with A stored [K][M] and/or B stored [K][N]: bit-identical
    to fp8_gemm on the same codes stored K-major, and within tolerance of the
    oracle's product (ragged tiles in M, N and K, with and without bias)."""
    a = wl.normal((M, K), 1.0, 131 + M, dtype=torch.float32)
    b = wl.normal((N, K), 1.0, 132 + N, dtype=torch.float32)
    qa, sa = _quant_tensor(a, sq.E5M2)
    qb, sb = _quant_tensor(b, sq.E4M3)
    bias = wl.normal((N,), 1.0, 133 + N, dtype=torch.float32).to(DEV) if with_bias else None
    ref = _gemm_t(qa, sq.E5M2, sa, qb, sq.E4M3, sb, out, bias=bias)
    A = qa.t().contiguous() if a_mn else qa
    B = qb.t().contiguous() if b_mn else qb
    D = torch.empty((M, N), dtype=out, device=DEV)
    sq.fp8_gemm_layout(A, sq.E5M2, sa, sq.MN_MAJOR if a_mn else sq.K_MAJOR, B, sq.E4M3, sb,
                       sq.MN_MAJOR if b_mn else sq.K_MAJOR, D, M, N, K, bias=bias)
    torch.cuda.synchronize()
    assert torch.equal(D.view(torch.uint8), ref.view(torch.uint8))
    R = o.gemm_ref(o.dequantize(codes(qa), o.E5M2, 0, sa.item()), o.dequantize(codes(qb), o.E4M3, 0, sb.item()),
                   bias=None if bias is None else bias.cpu().numpy())
    assert_gemm_close(D, R)


def test_mn_major_integer_operands_exact():
    """Integer-valued codes, unit scales, both operands MN-major: the int64
    product exactly."""
    rng = np.random.default_rng(12)
    M, N, K = 256, 512, 384
    va, qa = _int_codes(rng, (M, K), o.E4M3, -8, 8)
    vb, qb = _int_codes(rng, (N, K), o.E5M2, -8, 8)
    D = torch.empty((M, N), dtype=torch.float32, device=DEV)
    sq.fp8_gemm_layout(torch.from_numpy(np.ascontiguousarray(qa.T)).to(DEV), sq.E4M3, _one(), sq.MN_MAJOR,
                       torch.from_numpy(np.ascontiguousarray(qb.T)).to(DEV), sq.E5M2, _one(), sq.MN_MAJOR, D, M, N, K)
    torch.cuda.synchronize()
    assert np.array_equal(D.cpu().numpy(), (va.astype(np.int64) @ vb.astype(np.int64).T).astype(np.float32))


def test_mn_major_rejects_unaligned_rows():
    qa = torch.zeros((64, 40), dtype=torch.uint8, device=DEV)      # A [K][M] with M = 40
    qb = torch.zeros((64, 32), dtype=torch.uint8, device=DEV)
    D = torch.empty((40, 32), dtype=torch.float32, device=DEV)
    with pytest.raises(sq.Fp8Error) as e:
        sq.fp8_gemm_layout(qa, sq.E4M3, _one(), sq.MN_MAJOR, qb, sq.E4M3, _one(), sq.MN_MAJOR, D, 40, 32, 64)
    assert e.value.code == sq.ERR_UNSUPPORTED


# ---------------------------------------------------------------- GEMM with the output cast fused
@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (False, True), (True, True)])
@pytest.mark.parametrize("M,N,K,with_bias", [(256, 384, 512, False), (272, 400, 144, True), (528, 256, 1040, True)]
                         + [(432, 896, 1488, False), (304, 128, 928, True), (688, 800, 992, False)])
@pytest.mark.parametrize("qfmt", [sq.E4M3, sq.E5M2])
def test_gemm_cast_equals_gemm_then_cast(a_mn, b_mn, M, N, K, with_bias, qfmt):
    """fp8_gemm_cast: D bit-identical to fp8_gemm_layout's, the codes and the
    delayed state bit-identical to fp8_quantize (TENSOR, delayed) of that D
    run afterwards -- including a ragged M with bias, whose rows past M must
    not enter the amax (the last three shapes: seeded random draws)."""
    H = 16
    a = wl.normal((M, K), 1.0, 141 + M, dtype=torch.float32)
    b = wl.normal((N, K), 1.0, 142 + N, dtype=torch.float32)
    qa, sa = _quant_tensor(a, sq.E4M3)
    qb, sb = _quant_tensor(b, sq.E4M3)
    bias = wl.normal((N,), 3.0, 143 + N, dtype=torch.float32).to(DEV) if with_bias else None
    A = qa.t().contiguous() if a_mn else qa
    B = qb.t().contiguous() if b_mn else qb
    la, lb = (sq.MN_MAJOR if a_mn else sq.K_MAJOR), (sq.MN_MAJOR if b_mn else sq.K_MAJOR)
    st0 = torch.tensor(o.state_init(H), device=DEV)
    st0[H] = 448.0 / 7.0 if qfmt == sq.E4M3 else 57344.0 / 7.0     # a multiplier under which some outputs saturate
    st0[3] = 2.5                                                     # older history entries stay put
    # reference: the GEMM, then the delayed cast of its bf16 output
    D_ref = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    sq.fp8_gemm_layout(A, sq.E4M3, sa, la, B, sq.E4M3, sb, lb, D_ref, M, N, K, bias=bias)
    st_ref = st0.clone()
    q_ref = torch.empty((M, N), dtype=torch.uint8, device=DEV)
    sq.fp8_quantize(D_ref, qfmt, sq.TENSOR, q_ref, delayed_state=st_ref, history_len=H)
    # fused
    D = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    q = torch.empty((M, N), dtype=torch.uint8, device=DEV)
    st = st0.clone()
    sq.fp8_gemm_cast(A, sq.E4M3, sa, la, B, sq.E4M3, sb, lb, D, M, N, K, q, qfmt, st, H, bias=bias)
    torch.cuda.synchronize()
    assert torch.equal(D.view(torch.int16), D_ref.view(torch.int16))
    assert torch.equal(q, q_ref)
    assert st.cpu().numpy().tobytes() == st_ref.cpu().numpy().tobytes()
    # and against the oracle's cast of the same bf16 output
    rst = st0.cpu().numpy().copy()
    rq, _ = o.quantize_delayed(np32(D), qfmt, rst)
    assert np.array_equal(codes(q), rq) and rst.tobytes() == st.cpu().numpy().tobytes()


def test_gemm_cast_rejects_n_not_multiple_of_16():
    qa = torch.zeros((64, 32), dtype=torch.uint8, device=DEV)
    qb = torch.zeros((40, 32), dtype=torch.uint8, device=DEV)     # N = 40: not a multiple of 16
    D = torch.empty((64, 40), dtype=torch.bfloat16, device=DEV)
    q = torch.empty((64, 40), dtype=torch.uint8, device=DEV)
    st = torch.tensor(o.state_init(16), device=DEV)
    with pytest.raises(sq.Fp8Error) as e:
        sq.fp8_gemm_cast(qa, sq.E4M3, _one(), sq.K_MAJOR, qb, sq.E4M3, _one(), sq.K_MAJOR, D, 64, 40, 32, q, sq.E4M3,
                         st, 16)
    assert e.value.code == sq.ERR_UNSUPPORTED
