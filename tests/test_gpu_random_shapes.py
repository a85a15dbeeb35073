"""Seeded random shapes through every GEMM mode and the fine-grained linear
layers, against the oracle: the quantised operands bit-exact where the
quantiser is the oracle's, every output within the GEMM tolerance.  The
shapes are drawn from the ranges each mode accepts (ragged row counts,
tile counts that leave partial waves, K that leaves partial scale groups),
so layout edge cases that fixed parametrisations miss get exercised."""
import numpy as np
import pytest
import torch

import oracle as o
import scaled_quantize_gemm_gb300 as sq
from scaled_quantize_gemm_gb300 import workloads as wl

from _helpers import assert_gemm_close, codes, mx_untile, np32

pytestmark = pytest.mark.gpu
DEV = "cuda"
U8 = dict(dtype=torch.uint8, device=DEV)
F32 = dict(dtype=torch.float32, device=DEV)


def _shapes(seed, n, m_step, n_step, k_step, m_max=640, n_max=896, k_max=1152):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        out.append((int(rng.integers(1, m_max // m_step + 1)) * m_step,
                    int(rng.integers(1, n_max // n_step + 1)) * n_step,
                    int(rng.integers(1, k_max // k_step + 1)) * k_step))
    return out


@pytest.mark.parametrize("M,N,K", _shapes(1, 6, 1, 8, 16))
def test_per_tensor_random(M, N, K):
    a = wl.normal((M, K), 1.0, 31 + M, dtype=torch.float32)
    b = wl.normal((N, K), 1.0, 32 + N, dtype=torch.float32)
    qa, qb = torch.empty((M, K), **U8), torch.empty((N, K), **U8)
    sa, sb, aa, ab = (torch.empty(1, **F32) for _ in range(4))
    sq.fp8_quantize(a.to(DEV), sq.E4M3, sq.TENSOR, qa, scales_out=sa, amax_out=aa)
    sq.fp8_quantize(b.to(DEV), sq.E5M2, sq.TENSOR, qb, scales_out=sb, amax_out=ab)
    out = torch.bfloat16 if (M + N) % 2 else torch.float32
    D = torch.empty((M, N), dtype=out, device=DEV)
    sq.fp8_gemm(qa, sq.E4M3, sa, sq.TENSOR, qb, sq.E5M2, sb, sq.TENSOR, D)
    torch.cuda.synchronize()
    rqa, _, rsa, _ = o.quantize_tensor_current(a.numpy(), o.E4M3)
    rqb, _, rsb, _ = o.quantize_tensor_current(b.numpy(), o.E5M2)
    assert np.array_equal(codes(qa), rqa) and np.array_equal(codes(qb), rqb)
    assert_gemm_close(D, o.gemm_ref(o.dequantize(rqa, o.E4M3, 0, rsa), o.dequantize(rqb, o.E5M2, 0, rsb)))


@pytest.mark.parametrize("M,N,K", _shapes(2, 6, 1, 128, 128))
def test_tile_block_promotion_random(M, N, K):
    x = wl.student_t3((M, K), 41 + M)
    w = wl.normal((N, K), 0.02, 42 + N)
    qx, qw = torch.empty((M, K), **U8), torch.empty((N, K), **U8)
    sx = torch.empty(M * (K // 128), **F32)
    sw = torch.empty((N // 128) * (K // 128), **F32)
    sq.fp8_quantize(x.to(DEV), sq.E4M3, sq.TILE_1x128, qx, scales_out=sx)
    sq.fp8_quantize(w.to(DEV), sq.E4M3, sq.BLOCK_128x128, qw, scales_out=sw)
    D = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    sq.fp8_gemm(qx, sq.E4M3, sx, sq.TILE_1x128, qw, sq.E4M3, sw, sq.BLOCK_128x128, D)
    torch.cuda.synchronize()
    rqx, rsx, _, _ = o.quantize_tile1x128(np32(x), o.E4M3)
    rqw, rsw, _, _ = o.quantize_block128(np32(w), o.E4M3)
    assert np.array_equal(codes(qx), rqx) and np.array_equal(codes(qw), rqw)
    assert_gemm_close(D, o.gemm_ref(o.dequantize(rqx, 0, o.GRAN_TILE_1x128, rsx),
                                    o.dequantize(rqw, 0, o.GRAN_BLOCK_128x128, rsw)))


@pytest.mark.parametrize("M,N,K", _shapes(3, 6, 128, 128, 128))
def test_mx_random(M, N, K):
    a = wl.with_scaled_fraction((M, K), 1e-3, 100.0, 51 + M)
    b = wl.with_scaled_fraction((N, K), 1e-3, 100.0, 52 + N)
    qa, qb = torch.empty((M, K), **U8), torch.empty((N, K), **U8)
    ea, eb = torch.empty(M * K // 32, **U8), torch.empty(N * K // 32, **U8)
    sq.fp8_quantize(a.to(DEV), sq.E4M3, sq.MX32_TILED, qa, scales_out=ea)
    sq.fp8_quantize(b.to(DEV), sq.E4M3, sq.MX32_TILED, qb, scales_out=eb)
    out = torch.bfloat16 if (M // 128 + N // 128) % 2 else torch.float32
    D = torch.empty((M, N), dtype=out, device=DEV)
    sq.fp8_gemm(qa, sq.E4M3, ea, sq.MX32_TILED, qb, sq.E4M3, eb, sq.MX32_TILED, D)
    torch.cuda.synchronize()
    rqa, rea, _, _ = o.quantize_mx32(np32(a), o.E4M3)
    rqb, reb, _, _ = o.quantize_mx32(np32(b), o.E4M3)
    assert np.array_equal(codes(qa), rqa) and np.array_equal(mx_untile(ea.cpu().numpy(), M, K), rea)
    assert np.array_equal(codes(qb), rqb) and np.array_equal(mx_untile(eb.cpu().numpy(), N, K), reb)
    assert_gemm_close(D, o.gemm_ref(o.dequantize(rqa, 0, o.GRAN_MX32, rea), o.dequantize(rqb, 0, o.GRAN_MX32, reb)))


@pytest.mark.parametrize("gran", [sq.TILE_1x128, sq.TILE_1x128_POW2, sq.MX32])
@pytest.mark.parametrize("M,N,K", _shapes(4, 3, 128, 128, 128))
def test_fine_linear_random(gran, M, N, K):
    x = wl.student_t3((M, K), 61 + M)
    w = wl.normal((N, K), 0.02, 62 + N)
    dy = wl.normal((M, N), 1e-3, 63 + K)
    ws = torch.empty(sq.fp8_linear_workspace_bytes(M, N, K, gran), **U8)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    dx = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    dw = torch.empty((N, K), **F32)
    sq.fp8_linear_fwd(x.to(DEV), w.to(DEV), y, ws, gran=gran)
    sq.fp8_linear_bwd(dy.to(DEV), dx, dw, ws, K, gran=gran)
    torch.cuda.synchronize()
    og = {sq.TILE_1x128: o.GRAN_TILE_1x128, sq.TILE_1x128_POW2: o.GRAN_TILE_POW2, sq.MX32: o.GRAN_MX32}[gran]
    st, Y = o.linear_fine_fwd(np32(x), np32(w), og)
    dX, dW = o.linear_fine_bwd(st, np32(dy), og, o.E5M2)
    assert_gemm_close(y, Y)
    assert_gemm_close(dx, dX)
    assert_gemm_close(dw, dW)
    assert sq.fp8_device_status(True) == 0
