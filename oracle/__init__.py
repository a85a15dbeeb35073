"""CPU oracle for the FP8 scaled-linear path -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product library never does, and the two
share no code.  The bit-level work (codec, amax, scale rules, quantizers,
delayed state, dequantisation) is plain C in ``fp8_oracle.c``; this module
loads it with ctypes and adds the GEMM reference, which is a float64
matrix product of the exactly dequantised operands (a library matmul used as
one step, with no blocking or reordering of its own).

Sources are cited by page title and section:
  "Transformer Scaling" (lab.mindcaptain.ai reading 06) -- Part 01, core
  vocabulary, worked example;
  "Week 14. Scaling laws, precision, parallelism" -- absmax, FP8 and
  accumulation-precision bullets, bf16 paragraph;
  "Accelerating Transformer Training with NVIDIA Transformer Engine" --
  DelayedScaling recipe and the fp8_meta dump.

Parity status: every function is pinned by tests under ``tests/`` (worked
examples, brute force over all codes, closed forms, library special cases),
except the choices the pages leave open and the tests can only fix by
convention: the E8M0 exponent rule, the order of the amax history, and the
output dtypes (these are "parity unpinned" against the pages and pinned only
against their own closed forms).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

E4M3, E5M2 = 0, 1
ALGO_MAX, ALGO_MOST_RECENT = 0, 1
GRAN_TENSOR, GRAN_TILE_1x128, GRAN_BLOCK_128x128, GRAN_MX32 = 0, 1, 2, 3
GRAN_TILE_128x1, GRAN_MX32_COL = 4, 5   # column units (128 or 32 consecutive rows of a column)
GRAN_TILE_POW2, GRAN_BLOCK_POW2 = 6, 7   # 1x128 / 128x128 units with power-of-two (E8M0) scales
GRAN_TILE_COL_POW2 = 8                   # 128x1 column units with power-of-two (E8M0) scales
FMAX = {E4M3: 448.0, E5M2: 57344.0}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile fp8_oracle.c with the host C compiler (no fast-math, no FMA
    contraction, OpenMP for the row loops)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            c = ctypes
            P = c.c_void_p
            sig = {
                "orc_decode": (c.c_double, [c.c_int, c.c_uint8]),
                "orc_encode": (c.c_uint8, [c.c_int, c.c_float]),
                "orc_fmax": (c.c_double, [c.c_int]),
                "orc_max_code": (c.c_int, [c.c_int]),
                "orc_bf16_from_f32": (c.c_uint16, [c.c_float]),
                "orc_f32_from_bf16": (c.c_float, [c.c_uint16]),
                "orc_amax": (c.c_float, [P, c.c_int64]),
                "orc_current_scale": (None, [c.c_float, c.c_int, P, P]),
                "orc_quantize_tensor_current": (c.c_int64, [P, c.c_int64, c.c_int, P, P, P]),
                "orc_quantize_with_multiplier": (c.c_int64, [P, c.c_int64, c.c_float, c.c_int, P]),
                "orc_quantize_tile1x128": (c.c_int64, [P, c.c_int64, c.c_int64, c.c_int, P, P, P]),
                "orc_quantize_block128": (c.c_int64, [P, c.c_int64, c.c_int64, c.c_int, P, P, P]),
                "orc_mx_scale_code": (c.c_uint8, [c.c_float, c.c_int]),
                "orc_quantize_tile128x1": (c.c_int64, [P, c.c_int64, c.c_int64, c.c_int, P, P, P]),
                "orc_mx_scale_code_floor": (c.c_uint8, [c.c_float, c.c_int]),
                "orc_layernorm": (None, [P, c.c_int64, c.c_int64, P, P, c.c_double, P, P, P]),
                "orc_quantize_mx32_floor": (c.c_int64, [P, c.c_int64, c.c_int64, c.c_int, P, P]),
                "orc_quantize_tile1x128_pow2": (c.c_int64, [P, c.c_int64, c.c_int64, c.c_int, P, P]),
                "orc_quantize_tile128x1_pow2": (c.c_int64, [P, c.c_int64, c.c_int64, c.c_int, P, P]),
                "orc_quantize_block128_pow2": (c.c_int64, [P, c.c_int64, c.c_int64, c.c_int, P, P]),
                "orc_quantize_mx32_col": (c.c_int64, [P, c.c_int64, c.c_int64, c.c_int, P, P, P]),
                "orc_quantize_mx32": (c.c_int64, [P, c.c_int64, c.c_int64, c.c_int, P, P, P]),
                "orc_state_init": (None, [P, c.c_int]),
                "orc_quantize_delayed": (c.c_int64, [P, c.c_int64, c.c_int, P, c.c_int, P]),
                "orc_update_scale": (None, [P, c.c_int, c.c_int, c.c_int]),
                "orc_dequantize": (None, [P, c.c_int64, c.c_int64, c.c_int, c.c_int, P, P]),
                "orc_int8_absmax": (None, [P, c.c_int64, P, P]),
                "orc_fp8_running_sum": (c.c_float, [c.c_int, c.c_float, c.c_int, c.c_int, P]),
            }
            for name, (res, args) in sig.items():
                f = getattr(lib, name)
                f.restype = res
                f.argtypes = args
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _f32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


# ---------------------------------------------------------------- input views
def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float32 values."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- codec
def decode(fmt: int, code: int) -> float:
    return _load().orc_decode(fmt, code)


def encode(fmt: int, v: float) -> int:
    return _load().orc_encode(fmt, float(np.float32(v)))


def decode_array(fmt: int, q: np.ndarray) -> np.ndarray:
    table = np.array([decode(fmt, c) for c in range(256)], dtype=np.float64)
    return table[np.asarray(q, dtype=np.uint8)]


def fmax(fmt: int) -> float:
    return _load().orc_fmax(fmt)


def bf16_from_f32(v: float) -> int:
    return _load().orc_bf16_from_f32(float(np.float32(v)))


def bf16_round_array(x: np.ndarray) -> np.ndarray:
    """fp32 array -> bf16 bit patterns (uint16), element by element."""
    f = _load().orc_bf16_from_f32
    flat = _f32(x).ravel()
    out = np.fromiter((f(float(v)) for v in flat), dtype=np.uint16, count=flat.size)
    return out.reshape(np.shape(x))


def bf16_round_array_fast(x: np.ndarray) -> np.ndarray:
    """Same rule as ``orc_bf16_from_f32`` (ties to even on the dropped 16
    bits), vectorised for large outputs; checked against the C routine by the
    oracle tests."""
    b = _f32(x).view(np.uint32)
    upper = (b >> 16).astype(np.uint32)
    lower = b & 0xFFFF
    up = (lower > 0x8000) | ((lower == 0x8000) & ((upper & 1) == 1))
    res = (upper + up.astype(np.uint32)).astype(np.uint16)
    nan = np.isnan(_f32(x))
    res[nan] = (upper[nan] | 0x40).astype(np.uint16)
    return res


# ---------------------------------------------------------------- amax / scales
def amax(x) -> float:
    a = _f32(x)
    return float(_load().orc_amax(_p(a), a.size))


def current_scale(a: float, fmt: int):
    m = ctypes.c_float()
    s = ctypes.c_float()
    _load().orc_current_scale(float(np.float32(a)), fmt, ctypes.byref(m), ctypes.byref(s))
    return np.float32(m.value), np.float32(s.value)


def mx_scale_code(a: float, fmt: int) -> int:
    return int(_load().orc_mx_scale_code(float(np.float32(a)), fmt))


# ---------------------------------------------------------------- quantizers
def quantize_tensor_current(x, fmt: int):
    """-> (q uint8 same shape, amax, s, n_saturated)"""
    a = _f32(x)
    q = np.empty(a.shape, dtype=np.uint8)
    am = ctypes.c_float()
    s = ctypes.c_float()
    sat = _load().orc_quantize_tensor_current(_p(a), a.size, fmt, _p(q), ctypes.byref(am), ctypes.byref(s))
    return q, np.float32(am.value), np.float32(s.value), int(sat)


def quantize_with_multiplier(x, m: float, fmt: int):
    a = _f32(x)
    q = np.empty(a.shape, dtype=np.uint8)
    sat = _load().orc_quantize_with_multiplier(_p(a), a.size, float(np.float32(m)), fmt, _p(q))
    return q, int(sat)


def quantize_tile1x128(x, fmt: int):
    """x[R][C], C % 128 == 0 -> (q, s[R][C/128], amax[R][C/128], n_sat)"""
    a = _f32(x)
    R, C = a.shape
    assert C % 128 == 0
    q = np.empty((R, C), dtype=np.uint8)
    s = np.empty((R, C // 128), dtype=np.float32)
    am = np.empty((R, C // 128), dtype=np.float32)
    sat = _load().orc_quantize_tile1x128(_p(a), R, C, fmt, _p(q), _p(s), _p(am))
    return q, s, am, int(sat)


def quantize_block128(x, fmt: int):
    """x[R][C], R, C % 128 == 0 -> (q, s[R/128][C/128], amax, n_sat)"""
    a = _f32(x)
    R, C = a.shape
    assert R % 128 == 0 and C % 128 == 0
    q = np.empty((R, C), dtype=np.uint8)
    s = np.empty((R // 128, C // 128), dtype=np.float32)
    am = np.empty((R // 128, C // 128), dtype=np.float32)
    sat = _load().orc_quantize_block128(_p(a), R, C, fmt, _p(q), _p(s), _p(am))
    return q, s, am, int(sat)


def quantize_mx32(x, fmt: int):
    """x[R][C], C % 32 == 0 -> (q, e8m0[R][C/32] uint8, amax, n_sat)"""
    a = _f32(x)
    R, C = a.shape
    assert C % 32 == 0
    q = np.empty((R, C), dtype=np.uint8)
    e = np.empty((R, C // 32), dtype=np.uint8)
    am = np.empty((R, C // 32), dtype=np.float32)
    sat = _load().orc_quantize_mx32(_p(a), R, C, fmt, _p(q), _p(e), _p(am))
    return q, e, am, int(sat)


def quantize_tile128x1(x, fmt: int):
    """column tiles: x[R][C], R % 128 == 0 -> (q [R][C], s[R/128][C], amax, n_sat)"""
    a = _f32(x)
    R, C = a.shape
    assert R % 128 == 0
    q = np.empty((R, C), dtype=np.uint8)
    s = np.empty((R // 128, C), dtype=np.float32)
    am = np.empty((R // 128, C), dtype=np.float32)
    sat = _load().orc_quantize_tile128x1(_p(a), R, C, fmt, _p(q), _p(s), _p(am))
    return q, s, am, int(sat)


def quantize_mx32_col(x, fmt: int):
    """column MX blocks: x[R][C], R % 32 == 0 -> (q [R][C], e8m0 [R/32][C], amax, n_sat)"""
    a = _f32(x)
    R, C = a.shape
    assert R % 32 == 0
    q = np.empty((R, C), dtype=np.uint8)
    e = np.empty((R // 32, C), dtype=np.uint8)
    am = np.empty((R // 32, C), dtype=np.float32)
    sat = _load().orc_quantize_mx32_col(_p(a), R, C, fmt, _p(q), _p(e), _p(am))
    return q, e, am, int(sat)


def mx_scale_code_floor(a: float, fmt: int) -> int:
    return int(_load().orc_mx_scale_code_floor(float(np.float32(a)), fmt))


def _e8m0_quantizer(name, shape_fn):
    def f(x, fmt: int):
        a = _f32(x)
        R, C = a.shape
        q = np.empty((R, C), dtype=np.uint8)
        e = np.empty(shape_fn(R, C), dtype=np.uint8)
        sat = getattr(_load(), name)(_p(a), R, C, fmt, _p(q), _p(e))
        return q, e, int(sat)
    return f


# recipe variants: OCP-floor MX exponent; power-of-two 1x128 / 128x128 scales
quantize_mx32_floor = _e8m0_quantizer("orc_quantize_mx32_floor", lambda R, C: (R, C // 32))
quantize_tile1x128_pow2 = _e8m0_quantizer("orc_quantize_tile1x128_pow2", lambda R, C: (R, C // 128))
quantize_block128_pow2 = _e8m0_quantizer("orc_quantize_block128_pow2", lambda R, C: (R // 128, C // 128))
quantize_tile128x1_pow2 = _e8m0_quantizer("orc_quantize_tile128x1_pow2", lambda R, C: (R // 128, C))


def layernorm(x, gamma, beta=None, eps: float = 1e-5):
    """-> (y float64 [R][K], mean float64 [R], rstd float64 [R])"""
    a = _f32(x)
    R, K = a.shape
    g = _f32(gamma)
    b = None if beta is None else _f32(beta)
    y = np.empty((R, K), dtype=np.float64)
    mu = np.empty(R, dtype=np.float64)
    rs = np.empty(R, dtype=np.float64)
    _load().orc_layernorm(_p(a), R, K, _p(g), _p(b), float(eps), _p(y), _p(mu), _p(rs))
    return y, mu, rs


def ln_acceptable_codes(y: np.ndarray, delta: np.ndarray, m: float, fmt: int):
    """Codes reachable from a LayerNorm output known to within +-delta of the
    exact y (the reduction order of an implementation is not specified):
    (nearest code of fp32(y) * m, lowest and highest code over the interval).
    Casting is monotone, so every code in between is reachable too."""
    yf = y.astype(np.float32)
    m32 = np.float32(m)
    lo = (y - delta).astype(np.float32)
    hi = (y + delta).astype(np.float32)
    def enc(v):
        q, _ = quantize_with_multiplier(v, m32, fmt)
        return q
    return enc(yf), enc(lo), enc(hi)


def code_rank(q: np.ndarray) -> np.ndarray:
    """Order-preserving integer for FP8 codes (sign-magnitude -> signed)."""
    q = q.astype(np.int32)
    return np.where(q & 0x80, -(q & 0x7F), q & 0x7F)


# ---------------------------------------------------------------- delayed state
def state_init(H: int) -> np.ndarray:
    st = np.empty(H + 2, dtype=np.float32)
    _load().orc_state_init(_p(st), H)
    return st


def quantize_delayed(x, fmt: int, state: np.ndarray):
    """Casts with state's multiplier and records amax in state[0] (in place)."""
    a = _f32(x)
    assert state.dtype == np.float32 and state.flags.c_contiguous
    H = state.size - 2
    q = np.empty(a.shape, dtype=np.uint8)
    sat = _load().orc_quantize_delayed(_p(a), a.size, fmt, _p(state), H, _p(q))
    return q, int(sat)


def update_scale(state: np.ndarray, fmt: int, algo: int = ALGO_MAX) -> None:
    assert state.dtype == np.float32 and state.flags.c_contiguous
    _load().orc_update_scale(_p(state), state.size - 2, fmt, algo)


# ---------------------------------------------------------------- dequant + GEMM
def dequantize(q: np.ndarray, fmt: int, gran: int, scales) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    R, C = q.shape
    if gran in (GRAN_MX32, GRAN_MX32_COL, GRAN_TILE_POW2, GRAN_BLOCK_POW2, GRAN_TILE_COL_POW2):
        sc = np.ascontiguousarray(scales, dtype=np.uint8)
    else:
        sc = np.ascontiguousarray(np.atleast_1d(np.asarray(scales, dtype=np.float32)))
    out = np.empty((R, C), dtype=np.float64)
    _load().orc_dequantize(_p(q), R, C, fmt, gran, _p(sc), _p(out))
    return out


def gemm_ref(a_hat: np.ndarray, b_hat: np.ndarray, bias=None) -> np.ndarray:
    """R[i][j] = sum_k a_hat[i][k] * b_hat[j][k] in float64 (A [M,K], B [N,K],
    both K-contiguous, the layout of a linear layer y = x W^T); bias is added
    in float64.  Returns float64."""
    r = np.asarray(a_hat, dtype=np.float64) @ np.asarray(b_hat, dtype=np.float64).T
    if bias is not None:
        r = r + np.asarray(bias, dtype=np.float64)[None, :]
    return r


def epilogue(r: np.ndarray, out_bf16: bool) -> np.ndarray:
    """Output rounding: fp32 of the exact result; bf16 is then the RNE of that
    fp32 (bit patterns, uint16)."""
    f = r.astype(np.float32)
    return bf16_round_array_fast(f) if out_bf16 else f


# ---------------------------------------------------------------- linear layer
# y = x W^T with per-tensor delayed scaling under the HYBRID recipe
# ("Transformer Scaling", Part 01: E4M3 for forward weights/activations, E5M2
# for gradients; Transformer Engine tutorial: te.Linear under fp8_autocast).
# Backward: dx = dy W (contraction over N), dW = dy^T x (contraction over M).
# Per-tensor codes transpose exactly, so the transposed operands are the
# transposes of the forward codes.
def linear_fwd_delayed(x, w, x_state, w_state):
    """-> (qx, sx, qw, sw, R) with R = xhat what^T in float64; the states'
    history slot 0 records the amaxes (in place)."""
    H = x_state.size - 2
    sx, sw = np.float32(x_state[H + 1]), np.float32(w_state[H + 1])
    qx, _ = quantize_delayed(x, E4M3, x_state)
    qw, _ = quantize_delayed(w, E4M3, w_state)
    r = gemm_ref(dequantize(qx, E4M3, GRAN_TENSOR, sx), dequantize(qw, E4M3, GRAN_TENSOR, sw))
    return qx, sx, qw, sw, r


def linear_bwd_delayed(dy, dy_state, dy_fmt, qx, sx, qw, sw, rows=None, wrows=None):
    """-> (qdy, sdy, dX, dW) in float64.  rows / wrows: optional row subsets
    of dX (over M) and dW (over N) to evaluate (sampled checks)."""
    H = dy_state.size - 2
    sdy = np.float32(dy_state[H + 1])
    qdy, _ = quantize_delayed(dy, dy_fmt, dy_state)
    dyh = dequantize(qdy, dy_fmt, GRAN_TENSOR, sdy)
    xh = dequantize(qx, E4M3, GRAN_TENSOR, sx)
    wh = dequantize(qw, E4M3, GRAN_TENSOR, sw)
    a = dyh if rows is None else dyh[rows]
    dX = gemm_ref(a, wh.T)
    at = dyh.T if wrows is None else dyh.T[wrows]
    dW = gemm_ref(at, xh.T)
    return qdy, sdy, dX, dW


# Fine-grained scaling ("Week 14", absmax bullet: 1x128 activation tiles and
# 128x128 weight blocks, as in DeepSeek-V3; MX blocks of 32).  Each GEMM
# operand is quantised along that GEMM's contraction dimension: the forward
# contracts over K (x rows, W rows), dgrad over N (dy rows; W's columns: the
# 128x128 blocks of W^T are W's blocks transposed, and MX W is re-quantised
# in column blocks), wgrad over the tokens M (dy and x in column units).
def linear_fine_fwd(x, w, gran: int):
    """gran GRAN_TILE_1x128 (x tiles, W blocks), GRAN_TILE_POW2 (the same
    units with power-of-two scales) or GRAN_MX32 -> (state, R) with state
    holding what the backward needs (the forward's W codes / scales)."""
    if gran == GRAN_TILE_1x128:
        qx, sx, _, _ = quantize_tile1x128(x, E4M3)
        qw, sw, _, _ = quantize_block128(w, E4M3)
        r = gemm_ref(dequantize(qx, E4M3, GRAN_TILE_1x128, sx), dequantize(qw, E4M3, GRAN_BLOCK_128x128, sw))
        return {"x": x, "qw": qw, "sw": sw, "w": w}, r
    if gran == GRAN_TILE_POW2:
        qx, ex, _ = quantize_tile1x128_pow2(x, E4M3)
        qw, ew, _ = quantize_block128_pow2(w, E4M3)
        r = gemm_ref(dequantize(qx, E4M3, GRAN_TILE_POW2, ex), dequantize(qw, E4M3, GRAN_BLOCK_POW2, ew))
        return {"x": x, "qw": qw, "sw": ew, "w": w}, r
    qx, ex, _, _ = quantize_mx32(x, E4M3)
    qw, ew, _, _ = quantize_mx32(w, E4M3)
    r = gemm_ref(dequantize(qx, E4M3, GRAN_MX32, ex), dequantize(qw, E4M3, GRAN_MX32, ew))
    return {"x": x, "w": w}, r


def linear_fine_bwd_operands(st, dy, gran: int, dy_fmt: int = E4M3):
    """The four operands of the fine-grained backward, each quantised along
    its own GEMM's contraction dimension.  Returns {name: (codes, scales,
    dequantised float64)} with every matrix in its original orientation
    (dy [M][N], W [N][K], x [M][K]):
      dgrad_dy  dy in units along N   (1x128 tiles [M][N/128] / MX-32 [M][N/32])
      dgrad_w   W in units along N    (the forward's 128x128 blocks [N/128][K/128] /
                                       MX-32 column blocks [N/32][K])
      wgrad_dy  dy in units along M   (128x1 column tiles [M/128][N] / [M/32][N])
      wgrad_x   x in units along M    (128x1 column tiles [M/128][K] / [M/32][K])"""
    x, w = st["x"], st["w"]
    if gran == GRAN_TILE_POW2:
        qd, ed, _ = quantize_tile1x128_pow2(dy, dy_fmt)
        qdc, edc, _ = quantize_tile128x1_pow2(dy, dy_fmt)
        qxc, exc, _ = quantize_tile128x1_pow2(x, E4M3)
        return {
            "dgrad_dy": (qd, ed, dequantize(qd, dy_fmt, GRAN_TILE_POW2, ed)),
            "dgrad_w": (st["qw"], st["sw"], dequantize(st["qw"], E4M3, GRAN_BLOCK_POW2, st["sw"])),
            "wgrad_dy": (qdc, edc, dequantize(qdc, dy_fmt, GRAN_TILE_COL_POW2, edc)),
            "wgrad_x": (qxc, exc, dequantize(qxc, E4M3, GRAN_TILE_COL_POW2, exc)),
        }
    if gran == GRAN_TILE_1x128:
        qd, sd, _, _ = quantize_tile1x128(dy, dy_fmt)
        qdc, sdc, _, _ = quantize_tile128x1(dy, dy_fmt)
        qxc, sxc, _, _ = quantize_tile128x1(x, E4M3)
        return {
            "dgrad_dy": (qd, sd, dequantize(qd, dy_fmt, GRAN_TILE_1x128, sd)),
            "dgrad_w": (st["qw"], st["sw"], dequantize(st["qw"], E4M3, GRAN_BLOCK_128x128, st["sw"])),
            "wgrad_dy": (qdc, sdc, dequantize(qdc, dy_fmt, GRAN_TILE_128x1, sdc)),
            "wgrad_x": (qxc, sxc, dequantize(qxc, E4M3, GRAN_TILE_128x1, sxc)),
        }
    qd, ed, _, _ = quantize_mx32(dy, dy_fmt)
    qwc, ewc, _, _ = quantize_mx32_col(w, E4M3)
    qdc, edc, _, _ = quantize_mx32_col(dy, dy_fmt)
    qxc, exc, _, _ = quantize_mx32_col(x, E4M3)
    return {
        "dgrad_dy": (qd, ed, dequantize(qd, dy_fmt, GRAN_MX32, ed)),
        "dgrad_w": (qwc, ewc, dequantize(qwc, E4M3, GRAN_MX32_COL, ewc)),
        "wgrad_dy": (qdc, edc, dequantize(qdc, dy_fmt, GRAN_MX32_COL, edc)),
        "wgrad_x": (qxc, exc, dequantize(qxc, E4M3, GRAN_MX32_COL, exc)),
    }


def linear_fine_bwd(st, dy, gran: int, dy_fmt: int = E4M3):
    """-> (dX, dW) float64 for the fine-grained recipes: dX = dy W over N,
    dW = dy^T x over M, on the operands of linear_fine_bwd_operands."""
    ops = linear_fine_bwd_operands(st, dy, gran, dy_fmt)
    dX = gemm_ref(ops["dgrad_dy"][2], ops["dgrad_w"][2].T)
    dW = gemm_ref(ops["wgrad_dy"][2].T, ops["wgrad_x"][2].T)
    return dX, dW


# ---------------------------------------------------------------- worked-example helpers
def int8_absmax(x):
    a = _f32(x)
    q = np.empty(a.shape, dtype=np.int8)
    step = ctypes.c_float()
    _load().orc_int8_absmax(_p(a), a.size, _p(q), ctypes.byref(step))
    return q, np.float32(step.value)


def fp8_running_sum(fmt: int, term: float, n: int, promote: int):
    stall = ctypes.c_int()
    total = _load().orc_fp8_running_sum(fmt, float(term), n, promote, ctypes.byref(stall))
    return float(total), int(stall.value)
