"""The Python binding checks each buffer's dtype, contiguity and size before
it hands a raw pointer to the C ABI (which cannot see sizes), so a wrong
buffer raises instead of being written out of bounds.  CPU tensors suffice:
every check runs before the library is called."""
import pytest
import torch

import scaled_quantize_gemm_gb300 as sq

bf16, f32, u8 = torch.bfloat16, torch.float32, torch.uint8


def test_linear_bwd_rejects_a_bf16_or_short_weight_gradient():
    M, N, K = 64, 48, 32
    dy = torch.zeros((M, N), dtype=bf16)
    dx = torch.zeros((M, K), dtype=bf16)
    ws = torch.zeros(1024, dtype=u8)
    with pytest.raises(TypeError, match="dw"):
        sq.fp8_linear_bwd(dy, dx, torch.zeros((N, K), dtype=bf16), ws, K)     # dW is fp32
    with pytest.raises(ValueError, match="dw"):
        sq.fp8_linear_bwd(dy, dx, torch.zeros((N, K - 1), dtype=f32), ws, K)
    with pytest.raises(ValueError, match="dx"):
        sq.fp8_linear_bwd(dy, torch.zeros((M, K - 8), dtype=bf16), torch.zeros((N, K), dtype=f32), ws, K)


def test_linear_fwd_checks_output_and_states():
    M, N, K = 64, 48, 32
    x, w = torch.zeros((M, K), dtype=bf16), torch.zeros((N, K), dtype=bf16)
    ws = torch.zeros(1024, dtype=u8)
    with pytest.raises(ValueError, match="y"):
        sq.fp8_linear_fwd(x, w, torch.zeros((M, N - 1), dtype=bf16), ws)
    with pytest.raises(ValueError, match="x_state"):
        sq.fp8_linear_fwd(x, w, torch.zeros((M, N), dtype=bf16), ws, x_state=torch.zeros(17),
                          w_state=torch.zeros(18), history_len=16)
    with pytest.raises(ValueError, match="contiguous"):
        sq.fp8_linear_fwd(torch.zeros((K, M), dtype=bf16).t(), w, torch.zeros((M, N), dtype=bf16), ws)


def test_gemm_and_quantize_check_sizes():
    A, B = torch.zeros((64, 32), dtype=u8), torch.zeros((48, 32), dtype=u8)
    one = torch.ones(1)
    with pytest.raises(ValueError, match="D"):
        sq.fp8_gemm(A, sq.E4M3, one, sq.TENSOR, B, sq.E4M3, one, sq.TENSOR, torch.zeros((64, 47), dtype=f32))
    with pytest.raises(TypeError, match="A"):
        sq.fp8_gemm(A.float(), sq.E4M3, one, sq.TENSOR, B, sq.E4M3, one, sq.TENSOR, torch.zeros((64, 48)))
    x = torch.zeros((256, 256), dtype=bf16)
    with pytest.raises(ValueError, match="q"):
        sq.fp8_quantize(x, sq.E4M3, sq.TENSOR, torch.zeros(256 * 255, dtype=u8))
    with pytest.raises(ValueError, match="scales_out"):
        sq.fp8_quantize(x, sq.E4M3, sq.TILE_1x128, torch.zeros((256, 256), dtype=u8),
                        scales_out=torch.zeros(256 * 2 - 1))
    with pytest.raises(ValueError, match="scales_out"):
        sq.fp8_quantize(x, sq.E4M3, sq.MX32_TILED, torch.zeros((256, 256), dtype=u8),
                        scales_out=torch.zeros(256 * 8 - 1, dtype=u8))


def test_scale_state_calls_check_sizes():
    with pytest.raises(ValueError, match="states"):
        sq.fp8_scale_init(torch.zeros(18), 2, 16)          # two states need 36 floats
    with pytest.raises(ValueError, match="formats"):
        sq.fp8_update_scale(torch.zeros(36), 2, 16, [sq.E4M3])
