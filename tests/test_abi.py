"""The C-ABI library builds for sm_103a, loads, exports every entry point the
header declares, and rejects bad arguments on the host before touching the
GPU (these tests make no compute call)."""
import ctypes

import pytest

import scaled_quantize_gemm_gb300 as sq
from scaled_quantize_gemm_gb300 import build as sqbuild


@pytest.fixture(scope="module")
def L():
    sqbuild.build()
    return sq.lib()


def test_exports_every_declared_symbol(L):
    names = sq.declared_symbols()
    assert set(names) >= {"fp8_amax", "fp8_update_scale", "fp8_quantize", "fp8_gemm",
                          "fp8_linear_fwd", "fp8_linear_bwd", "fp8_last_error",
                          "fp8_scale_init", "fp8_linear_workspace_bytes", "fp8_device_status"}
    for n in names:
        assert hasattr(L, n), n
    assert L.fp8_abi_version() == 7


def test_null_and_enum_validation(L):
    P = ctypes.c_void_p
    fake = P(4096)      # aligned, never dereferenced: validation fails first
    assert L.fp8_amax(None, 0, 4, 4, 0, fake, None) == sq.ERR_INVALID_ARG
    assert b"null" in L.fp8_last_error()
    assert L.fp8_amax(fake, 7, 4, 4, 0, fake, None) == sq.ERR_INVALID_ARG
    assert L.fp8_amax(fake, 0, -1, 4, 0, fake, None) == sq.ERR_INVALID_ARG
    assert L.fp8_amax(P(4097), 0, 4, 4, 0, fake, None) == sq.ERR_MISALIGNED
    assert L.fp8_amax(fake, 0, 4, 100, sq.TILE_1x128, fake, None) == sq.ERR_UNSUPPORTED
    assert L.fp8_amax(fake, 0, 100, 128, sq.BLOCK_128x128, fake, None) == sq.ERR_UNSUPPORTED
    assert L.fp8_amax(fake, 0, 4, 48, sq.MX32, fake, None) == sq.ERR_UNSUPPORTED


def test_quantize_validation(L):
    P = ctypes.c_void_p
    f = P(4096)
    q = L.fp8_quantize
    # current per-tensor needs amax_out and scales_out
    assert q(f, 0, 4, 4, 0, 0, None, 0, f, None, None, None, None, None) == sq.ERR_INVALID_ARG
    # bad format
    assert q(f, 0, 4, 4, 3, 0, None, 0, f, None, f, f, None, None) == sq.ERR_INVALID_ARG
    # transposed copy needs multiples of 16
    assert q(f, 0, 8, 32, 0, 0, f, 16, f, f, None, None, None, None) == sq.ERR_UNSUPPORTED
    # transposed copy / delayed state only per tensor
    assert q(f, 0, 128, 128, 0, sq.TILE_1x128, None, 0, f, f, f, None, None, None) == sq.ERR_UNSUPPORTED
    assert q(f, 0, 128, 128, 0, sq.TILE_1x128, f, 16, f, None, f, None, None, None) == sq.ERR_UNSUPPORTED
    # column units: qT required, bf16 only, rows % 128
    assert q(f, 0, 256, 128, 0, sq.TILE_128x1, None, 0, None, None, f, None, None, None) == sq.ERR_INVALID_ARG
    assert q(f, 1, 256, 128, 0, sq.TILE_128x1, None, 0, None, f, f, None, None, None) == sq.ERR_UNSUPPORTED
    assert q(f, 0, 200, 128, 0, sq.TILE_128x1, None, 0, None, f, f, None, None, None) == sq.ERR_UNSUPPORTED
    assert q(f, 0, 256, 96, 0, sq.MX32_COL_TILED, None, 0, None, f, f, None, None, None) == sq.ERR_UNSUPPORTED
    # missing scales for a block granularity
    assert q(f, 0, 128, 128, 0, sq.MX32, None, 0, f, None, None, None, None, None) == sq.ERR_INVALID_ARG
    # bad history length
    assert q(f, 0, 16, 16, 0, 0, f, 0, f, None, None, None, None, None) == sq.ERR_INVALID_ARG
    # misaligned sat counter
    assert q(f, 0, 16, 16, 0, 0, f, 16, f, None, None, None, P(4100), None) == sq.ERR_MISALIGNED


def test_gemm_validation(L):
    P = ctypes.c_void_p
    f = P(4096)
    g = L.fp8_gemm
    assert g(None, 0, f, 0, f, 0, f, 0, 128, 128, 128, None, f, 0, None) == sq.ERR_INVALID_ARG
    assert g(f, 0, f, 0, f, 0, f, 0, 128, 124, 128, None, f, 0, None) == sq.ERR_UNSUPPORTED   # N % 8
    assert g(f, 0, f, 0, f, 0, f, 0, 128, 128, 120, None, f, 0, None) == sq.ERR_UNSUPPORTED   # K % 16
    assert g(f, 0, f, 1, f, 0, f, 2, 128, 128, 64, None, f, 0, None) == sq.ERR_UNSUPPORTED    # K % 128
    assert g(f, 0, f, 0, f, 0, f, 3, 128, 128, 128, None, f, 0, None) == sq.ERR_UNSUPPORTED   # mixed pair
    assert g(f, 2, f, 0, f, 0, f, 0, 128, 128, 128, None, f, 0, None) == sq.ERR_INVALID_ARG   # format
    assert g(f, 0, f, 0, P(4104), 0, f, 0, 128, 128, 128, None, f, 0, None) == sq.ERR_MISALIGNED


def test_linear_validation_and_workspace(L):
    P = ctypes.c_void_p
    f = P(4096)
    ws = sq.fp8_linear_workspace_bytes(256, 512, 384)
    # per tensor: the codes of x, W and dy (+ scalars), 256-byte aligned; the
    # backward reads them MN-major, so no transposed copies are kept
    assert 256 * 384 + 512 * 384 + 256 * 512 <= ws < 2 * (256 * 384 + 512 * 384 + 256 * 512)
    assert ws % 256 == 0
    # the fine-grained layouts also keep the column-unit codes
    assert sq.fp8_linear_workspace_bytes(256, 512, 384, sq.TILE_1x128) >= 2 * (256 * 384 + 512 * 384 + 256 * 512)
    assert sq.fp8_linear_workspace_bytes(256, 512, 384, sq.BLOCK_128x128) == 0
    fwd = L.fp8_linear_fwd
    assert fwd(f, f, 256, 512, 384, 0, 0, f, None, 16, f, ws, None, f, 0, None) == sq.ERR_INVALID_ARG  # one state
    assert fwd(f, f, 256, 512, 384, 0, 0, None, None, 0, f, ws - 1, None, f, 0, None) == sq.ERR_INVALID_ARG
    assert fwd(f, f, 256, 512, 384, 0, 0, None, None, 0, P(4096 + 16), ws, None, f, 0, None) == sq.ERR_MISALIGNED
    assert fwd(f, f, 200, 512, 384, 1, 0, None, None, 0, f, 1 << 30, None, f, 0, None) == sq.ERR_UNSUPPORTED
    bwd = L.fp8_linear_bwd
    assert bwd(f, 256, 512, 384, 0, 5, None, 0, f, ws, f, f, None) == sq.ERR_INVALID_ARG       # recipe
    assert bwd(f, 256, 512, 384, 9, 0, None, 0, f, ws, f, f, None) == sq.ERR_INVALID_ARG       # gran
    assert bwd(f, 256, 512, 384, 1, 0, f, 16, f, 1 << 30, f, f, None) == sq.ERR_UNSUPPORTED   # delayed + tiles
    # the fine-grained layouts hold the column-unit codes and scales of x, W and dy too
    assert sq.fp8_linear_workspace_bytes(256, 512, 384, sq.TILE_1x128) >= 2 * (256 * 384 + 512 * 384 + 256 * 512)
    assert sq.fp8_linear_workspace_bytes(256, 512, 384, sq.MX32) >= 2 * (256 * 384 + 512 * 384 + 256 * 512)


def test_update_scale_validation(L):
    P = ctypes.c_void_p
    fm = (ctypes.c_int * 2)(0, 5)
    assert L.fp8_update_scale(P(4096), 2, 16, fm, 0, None) == sq.ERR_INVALID_ARG
    fm = (ctypes.c_int * 2)(0, 1)
    assert L.fp8_update_scale(P(4096), 2, 16, fm, 9, None) == sq.ERR_INVALID_ARG
    assert L.fp8_update_scale(P(4096), 2, 0, fm, 0, None) == sq.ERR_INVALID_ARG
    assert L.fp8_scale_init(None, 2, 16, None) == sq.ERR_INVALID_ARG


def test_valid_call_without_gpu_reports_cuda_error(L):
    """On a machine without a GPU a well-formed call fails with a CUDA status
    (never a silent CPU fallback)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    P = ctypes.c_void_p
    r = L.fp8_amax(P(4096), 0, 16, 16, 0, P(8192), None)
    assert r == sq.ERR_CUDA
    assert b"device" in L.fp8_last_error()


def test_binding_raises_when_library_missing(monkeypatch, tmp_path):
    monkeypatch.setattr(sq, "LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(sq, "_lib", None)
    with pytest.raises(RuntimeError, match="no fallback"):
        sq.lib()


def test_layernorm_validation(L):
    """gamma, beta, mean and rstd are read as 128-bit vectors: 16-byte
    alignment is required; M, K must be multiples of 16."""
    P, c = ctypes.c_void_p, ctypes
    f = P(4096)
    ln = L.fp8_layernorm_quantize
    args = lambda gamma, M=32, K=64: (f, gamma, f, c.c_float(1e-5), M, K, sq.E4M3, f, 16, f, f, f, f, None)
    assert ln(*args(P(4096 + 4))) == sq.ERR_MISALIGNED
    assert b"16-byte" in L.fp8_last_error()
    assert ln(*args(f, M=24)) == sq.ERR_UNSUPPORTED
    assert ln(*args(None)) == sq.ERR_INVALID_ARG


def test_rows_cols_validation(L):
    P = ctypes.c_void_p
    f = P(4096)
    rc = L.fp8_quantize_rows_cols
    assert rc(f, 128, 128, sq.E4M3, sq.TENSOR, f, f, f, f, None, None) == sq.ERR_INVALID_ARG
    assert rc(f, 128, 96, sq.E4M3, sq.TILE_1x128, f, f, f, f, None, None) == sq.ERR_UNSUPPORTED
    assert rc(P(4100), 128, 128, sq.E4M3, sq.TILE_1x128, f, f, f, f, None, None) == sq.ERR_MISALIGNED
    assert rc(f, 128, 128, sq.E4M3, sq.MX32_TILED, f, P(4100), f, f, None, None) == sq.ERR_MISALIGNED
    assert rc(None, 128, 128, sq.E4M3, sq.TILE_1x128, f, f, f, f, None, None) == sq.ERR_INVALID_ARG
