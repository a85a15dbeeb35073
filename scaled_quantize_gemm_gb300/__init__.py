"""Python binding of the sm_103a FP8 scaled-linear library (libfp8sq.so).

Argument marshalling only: every function forwards torch tensors' device
pointers and the current CUDA stream to the extern "C" entry point of the
same name declared in ``include/fp8sq.h``; all of the path's arithmetic runs
in the library's CUDA kernels.  There is no fallback: if the library has not
been built (``__graft_entry__.build()``) the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

E4M3, E5M2 = 0, 1
BF16, F32 = 0, 1
TENSOR, TILE_1x128, BLOCK_128x128, MX32, MX32_TILED, TILE_128x1, MX32_COL_TILED = 0, 1, 2, 3, 4, 5, 6
TILE_1x128_POW2, BLOCK_128x128_POW2, MX32_FLOOR_TILED = 7, 8, 9
AMAX_MAX, AMAX_MOST_RECENT = 0, 1
RECIPE_HYBRID, RECIPE_E4M3 = 0, 1
K_MAJOR, MN_MAJOR = 0, 1
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_MISALIGNED, ERR_WRONG_ARCH, ERR_CUDA, ERR_TIMEOUT = 0, -1, -2, -3, -4, -5, -6

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libfp8sq.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "fp8sq.h")

_lock = threading.Lock()
_lib = None


class Fp8Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


def state_floats(history_len: int) -> int:
    return history_len + 2


def lib() -> ctypes.CDLL:
    """Load libfp8sq.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                                   "(the FP8 path has no fallback)")
            L = ctypes.CDLL(LIB_PATH)
            c = ctypes
            P, I, I64, Z = c.c_void_p, c.c_int, c.c_int64, c.c_size_t
            sig = {
                "fp8_abi_version": (I, []),
                "fp8_last_error": (c.c_char_p, []),
                "fp8_device_status": (I, [I]),
                "fp8_selftest_wait_timeout": (I, [I, P, P]),
                "fp8_amax": (I, [P, I, I64, I64, I, P, P]),
                "fp8_scale_init": (I, [P, I, I, P]),
                "fp8_update_scale": (I, [P, I, I, P, I, P]),
                "fp8_quantize": (I, [P, I, I64, I64, I, I, P, I, P, P, P, P, P, P]),
                "fp8_quantize_rows_cols": (I, [P, I64, I64, I, I, P, P, P, P, P, P]),
                "fp8_gemm": (I, [P, I, P, I, P, I, P, I, I64, I64, I64, P, P, I, P]),
                "fp8_gemm_layout": (I, [P, I, P, I, P, I, P, I, I64, I64, I64, P, P, I, P]),
                "fp8_gemm_cast": (I, [P, I, P, I, P, I, P, I, I64, I64, I64, P, P, P, I, P, I, P]),
                "fp8_linear_workspace_bytes": (Z, [I64, I64, I64, I]),
                "fp8_linear_fwd": (I, [P, P, I64, I64, I64, I, I, P, P, I, P, Z, P, P, I, P]),
                "fp8_linear_bwd": (I, [P, I64, I64, I64, I, I, P, I, P, Z, P, P, P]),
                "fp8_linear_fwd_noalloc": (I, [P, P, I64, I64, I64, P, P, I, P]),
                "fp8_layernorm_quantize": (I, [P, P, P, c.c_float, I64, I64, I, P, I, P, P, P, P, P]),
                "fp8_layernorm_linear_fwd": (I, [P, P, P, c.c_float, P, I64, I64, I64, P, P, I, P, Z, P, P, P, P,
                                                 I, P]),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


_torch = None
_raw_stream = None


def _t():
    global _torch
    if _torch is None:
        import torch
        _torch = torch
    return _torch


def _current_stream() -> int:
    """The current CUDA stream of the current device as a raw handle.  The
    binding asks for it on every call, so it takes torch's direct accessor
    (a fraction of a microsecond) where torch has it, else the public one."""
    global _raw_stream
    if _raw_stream is None:
        torch = _t()
        torch.cuda.init()
        C = torch._C
        if hasattr(C, "_cuda_getCurrentRawStream") and hasattr(C, "_cuda_getDevice"):
            get, dev = C._cuda_getCurrentRawStream, C._cuda_getDevice
            _raw_stream = lambda: get(dev())
        else:
            _raw_stream = lambda: torch.cuda.current_stream().cuda_stream
    return _raw_stream()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return _current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code: int):
    if code != OK:
        raise Fp8Error(code, lib().fp8_last_error().decode())


def _need(t, name: str, dtype=None, nbytes: int = None):
    """The C ABI takes raw pointers and cannot see a buffer's size: check here
    that each tensor is contiguous, of the documented dtype and large enough,
    so a wrong buffer raises instead of being written out of bounds."""
    if t is None:
        raise ValueError(f"{name} is required")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, the library expects {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if nbytes is not None and t.numel() * t.element_size() < nbytes:
        raise ValueError(f"{name}: {t.numel() * t.element_size()} bytes, needs {nbytes}")


def _opt(t, name: str, dtype=None, nbytes: int = None):
    if t is not None:
        _need(t, name, dtype, nbytes)


def _units(gran: int, R: int, C: int) -> int:
    """number of scaling units of an R x C tensor (include/fp8sq.h)"""
    if gran == TENSOR:
        return 1
    if gran == TILE_1x128:
        return R * (C // 128)
    if gran == BLOCK_128x128:
        return ((R + 127) // 128) * ((C + 127) // 128)
    if gran == TILE_128x1:
        return (R // 128) * C
    return R * C // 32          # MX-32 blocks (and the power-of-two codes in their tiled layout)


def _scale_bytes(gran: int, R: int, C: int) -> int:
    """bytes of the scales fp8_quantize writes: fp32 per unit, or one E8M0
    byte per 32-element block"""
    if gran in (TENSOR, TILE_1x128, BLOCK_128x128, TILE_128x1):
        return 4 * _units(gran, R, C)
    return R * C // 32


def _dtype_code(t) -> int:
    torch = _t()
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}")


# ---------------------------------------------------------------- entry points
def fp8_amax(x, gran: int, amax_out, stream=None) -> None:
    R, C = (x.shape[0], x.shape[1]) if x.dim() == 2 else (1, x.numel())
    _need(x, "x")
    _need(amax_out, "amax_out", _t().float32, 4 * _units(gran, R, C))
    _check(lib().fp8_amax(_ptr(x), _dtype_code(x), R, C, gran, _ptr(amax_out), _stream(stream)))


def fp8_scale_init(states, n_states: int, history_len: int, stream=None) -> None:
    _need(states, "states", _t().float32, 4 * n_states * (history_len + 2))
    _check(lib().fp8_scale_init(_ptr(states), n_states, history_len, _stream(stream)))


def fp8_update_scale(states, n_states: int, history_len: int, formats, algo: int = AMAX_MAX,
                     stream=None) -> None:
    _need(states, "states", _t().float32, 4 * n_states * (history_len + 2))
    if len(formats) < n_states:
        raise ValueError(f"formats: {len(formats)} entries for {n_states} states")
    arr = (ctypes.c_int * max(1, n_states))(*formats)
    _check(lib().fp8_update_scale(_ptr(states), n_states, history_len, arr, algo, _stream(stream)))


def fp8_quantize(x, format: int, gran: int, q, qT=None, scales_out=None, amax_out=None,
                 delayed_state=None, history_len: int = 0, sat_count=None, stream=None) -> None:
    R, C = (x.shape[0], x.shape[1]) if x.dim() == 2 else (1, x.numel())
    T = _t()
    _need(x, "x")
    _opt(q, "q", T.uint8, R * C)
    _opt(qT, "qT", T.uint8, R * C)
    _opt(scales_out, "scales_out", None, _scale_bytes(gran, R, C))
    _opt(delayed_state, "delayed_state", T.float32, 4 * (history_len + 2))
    _check(lib().fp8_quantize(_ptr(x), _dtype_code(x), R, C, format, gran, _ptr(delayed_state), history_len,
                              _ptr(q), _ptr(qT), _ptr(scales_out), _ptr(amax_out), _ptr(sat_count),
                              _stream(stream)))


def fp8_quantize_rows_cols(x, format: int, unit: int, q, row_scales, qT, col_scales, sat_count=None,
                           stream=None) -> None:
    R, C = x.shape
    T = _t()
    _need(x, "x", T.bfloat16)
    _need(q, "q", T.uint8, R * C)
    _need(qT, "qT", T.uint8, R * C)
    _need(row_scales, "row_scales", None, _scale_bytes(unit, R, C))
    _need(col_scales, "col_scales", None,
          _scale_bytes(TILE_128x1 if unit == TILE_1x128 else MX32_COL_TILED, R, C))
    _check(lib().fp8_quantize_rows_cols(_ptr(x), R, C, format, unit, _ptr(q), _ptr(row_scales), _ptr(qT),
                                        _ptr(col_scales), _ptr(sat_count), _stream(stream)))


def fp8_gemm(A, a_format: int, a_scale, a_gran: int, B, b_format: int, b_scale, b_gran: int,
             D, bias=None, M: int = None, N: int = None, K: int = None, stream=None) -> None:
    M = A.shape[0] if M is None else M
    K = A.shape[1] if K is None else K
    N = B.shape[0] if N is None else N
    T = _t()
    _need(A, "A", T.uint8, M * K)
    _need(B, "B", T.uint8, N * K)
    _need(D, "D", None, M * N * (2 if D.dtype == T.bfloat16 else 4))
    _opt(bias, "bias", T.float32, 4 * N)
    _check(lib().fp8_gemm(_ptr(A), a_format, _ptr(a_scale), a_gran, _ptr(B), b_format, _ptr(b_scale), b_gran,
                          M, N, K, _ptr(bias), _ptr(D), _dtype_code(D), _stream(stream)))


def fp8_gemm_layout(A, a_format: int, a_scale, a_major: int, B, b_format: int, b_scale, b_major: int,
                    D, M: int, N: int, K: int, bias=None, stream=None) -> None:
    """Per-tensor-scaled GEMM with K-major or MN-major operands: A [M][K]
    or [K][M], B [N][K] or [K][N] (a_major / b_major K_MAJOR or MN_MAJOR)."""
    T = _t()
    _need(A, "A", T.uint8, M * K)
    _need(B, "B", T.uint8, N * K)
    _need(D, "D", None, M * N * (2 if D.dtype == T.bfloat16 else 4))
    _need(a_scale, "a_scale", T.float32, 4)
    _need(b_scale, "b_scale", T.float32, 4)
    _opt(bias, "bias", T.float32, 4 * N)
    _check(lib().fp8_gemm_layout(_ptr(A), a_format, _ptr(a_scale), a_major, _ptr(B), b_format, _ptr(b_scale),
                                 b_major, M, N, K, _ptr(bias), _ptr(D), _dtype_code(D), _stream(stream)))


def fp8_gemm_cast(A, a_format: int, a_scale, a_major: int, B, b_format: int, b_scale, b_major: int,
                  D, M: int, N: int, K: int, q_out, q_format: int, q_state, history_len: int, bias=None,
                  stream=None) -> None:
    """fp8_gemm_layout with a bf16 D whose epilogue also casts D to FP8
    codes q_out [M][N] with the delayed per-tensor state q_state."""
    T = _t()
    _need(A, "A", T.uint8, M * K)
    _need(B, "B", T.uint8, N * K)
    _need(D, "D", T.bfloat16, 2 * M * N)
    _need(a_scale, "a_scale", T.float32, 4)
    _need(b_scale, "b_scale", T.float32, 4)
    _need(q_out, "q_out", T.uint8, M * N)
    _need(q_state, "q_state", T.float32, 4 * (history_len + 2))
    _opt(bias, "bias", T.float32, 4 * N)
    _check(lib().fp8_gemm_cast(_ptr(A), a_format, _ptr(a_scale), a_major, _ptr(B), b_format, _ptr(b_scale),
                               b_major, M, N, K, _ptr(bias), _ptr(D), _ptr(q_out), q_format, _ptr(q_state),
                               history_len, _stream(stream)))


def fp8_linear_workspace_bytes(M: int, N: int, K: int, gran: int = TENSOR) -> int:
    return int(lib().fp8_linear_workspace_bytes(M, N, K, gran))


def fp8_linear_fwd(x, w, y, workspace, gran: int = TENSOR, recipe: int = RECIPE_HYBRID,
                   x_state=None, w_state=None, history_len: int = 0, bias=None, stream=None) -> None:
    M, K = x.shape
    N = w.shape[0]
    T = _t()
    _need(x, "x", T.bfloat16)
    _need(w, "w", T.bfloat16, 2 * N * K)
    _need(y, "y", None, M * N * (2 if y.dtype == T.bfloat16 else 4))
    _need(workspace, "workspace", T.uint8)
    _opt(x_state, "x_state", T.float32, 4 * (history_len + 2))
    _opt(w_state, "w_state", T.float32, 4 * (history_len + 2))
    _opt(bias, "bias", T.float32, 4 * N)
    _check(lib().fp8_linear_fwd(_ptr(x), _ptr(w), M, N, K, gran, recipe, _ptr(x_state), _ptr(w_state),
                                history_len, _ptr(workspace), workspace.numel() * workspace.element_size(),
                                _ptr(bias), _ptr(y), _dtype_code(y), _stream(stream)))


def fp8_linear_bwd(dy, dx, dw, workspace, K: int, gran: int = TENSOR, recipe: int = RECIPE_HYBRID,
                   dy_state=None, history_len: int = 0, stream=None) -> None:
    M, N = dy.shape
    T = _t()
    _need(dy, "dy", T.bfloat16)
    _need(dx, "dx", T.bfloat16, 2 * M * K)
    _need(dw, "dw", T.float32, 4 * N * K)
    _need(workspace, "workspace", T.uint8)
    _opt(dy_state, "dy_state", T.float32, 4 * (history_len + 2))
    _check(lib().fp8_linear_bwd(_ptr(dy), M, N, K, gran, recipe, _ptr(dy_state), history_len, _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _ptr(dx), _ptr(dw),
                                _stream(stream)))


def fp8_layernorm_quantize(x, gamma, beta, eps: float, format: int, q, qT, mu, rstd, delayed_state,
                           history_len: int, stream=None) -> None:
    M, K = x.shape
    T = _t()
    _need(x, "x", T.bfloat16)
    _need(gamma, "gamma", T.float32, 4 * K)
    _opt(beta, "beta", T.float32, 4 * K)
    _opt(q, "q", T.uint8, M * K)
    _opt(qT, "qT", T.uint8, M * K)
    _need(mu, "mu", T.float32, 4 * M)
    _need(rstd, "rstd", T.float32, 4 * M)
    _opt(delayed_state, "delayed_state", T.float32, 4 * (history_len + 2))
    _check(lib().fp8_layernorm_quantize(_ptr(x), _ptr(gamma), _ptr(beta), eps, M, K, format, _ptr(delayed_state),
                                        history_len, _ptr(q), _ptr(qT), _ptr(mu), _ptr(rstd), _stream(stream)))


def fp8_layernorm_linear_fwd(x, gamma, beta, eps: float, w, y, workspace, mu, rstd, x_state, w_state,
                             history_len: int, bias=None, stream=None) -> None:
    M, K = x.shape
    N = w.shape[0]
    T = _t()
    _need(x, "x", T.bfloat16)
    _need(gamma, "gamma", T.float32, 4 * K)
    _opt(beta, "beta", T.float32, 4 * K)
    _need(w, "w", T.bfloat16, 2 * N * K)
    _need(y, "y", None, M * N * (2 if y.dtype == T.bfloat16 else 4))
    _need(workspace, "workspace", T.uint8)
    _need(mu, "mu", T.float32, 4 * M)
    _need(rstd, "rstd", T.float32, 4 * M)
    _opt(x_state, "x_state", T.float32, 4 * (history_len + 2))
    _opt(w_state, "w_state", T.float32, 4 * (history_len + 2))
    _opt(bias, "bias", T.float32, 4 * N)
    _check(lib().fp8_layernorm_linear_fwd(_ptr(x), _ptr(gamma), _ptr(beta), eps, _ptr(w), M, N, K, _ptr(x_state),
                                          _ptr(w_state), history_len, _ptr(workspace),
                                          workspace.numel() * workspace.element_size(), _ptr(mu), _ptr(rstd),
                                          _ptr(bias), _ptr(y), _dtype_code(y), _stream(stream)))


def fp8_linear_fwd_noalloc(x, w, y, bias=None, stream=None) -> None:
    """Forward linear with current per-tensor scaling and no allocation: the
    scratch is the library's static device array (see include/fp8sq.h)."""
    M, K = x.shape
    N = w.shape[0]
    T = _t()
    _need(x, "x", T.bfloat16)
    _need(w, "w", T.bfloat16, 2 * N * K)
    _need(y, "y", None, M * N * (2 if y.dtype == T.bfloat16 else 4))
    _opt(bias, "bias", T.float32, 4 * N)
    _check(lib().fp8_linear_fwd_noalloc(_ptr(x), _ptr(w), M, N, K, _ptr(bias), _ptr(y), _dtype_code(y),
                                        _stream(stream)))


def fp8_selftest_wait_timeout(limit_us: int, waited_out, stream=None) -> None:
    _check(lib().fp8_selftest_wait_timeout(limit_us, _ptr(waited_out), _stream(stream)))


def fp8_device_status(clear: bool = True) -> int:
    return lib().fp8_device_status(1 if clear else 0)


def declared_symbols() -> list:
    """Names of the entry points declared FP8SQ_API in include/fp8sq.h."""
    import re
    txt = open(HEADER).read()
    return re.findall(r"FP8SQ_API\s+[\w\s\*]+?\b(fp8_\w+)\s*\(", txt)
