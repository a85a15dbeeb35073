"""Shared test helpers: tensor conversion and the GEMM tolerance check.

GEMM tolerance (the 1e-3 bound on maximum relative error): for fp32 output,
max|C - R| <= 1e-3 * max|R|, R the oracle's float64 result.  For bf16 output
the output rounding itself is up to half a bf16 ulp (2^-8 relative), so each
element must satisfy |C - R| <= 1e-3 * max|R| + ulp_bf16(C) / 2: C is the
bf16 rounding of a value within the 1e-3 bound.

Beside that norm-style bound, every check also takes the elementwise relative
error max |C_ij - R_ij| / |R_ij| over the elements with |R_ij| >= 1e-2 max|R|
(small outputs, which the norm bound barely constrains: it lets an element at
1e-2 max|R| be 10 % off).  It must stay within ELEM_TOL_F32 for fp32 outputs
(fp32 accumulation error only) and within ELEM_TOL_BF16 for bf16 outputs
(half a bf16 ulp, 2^-8 of the value, plus the same accumulation slack).  With SQ_ERR_REPORT=<path> set, each check appends one
JSON line (test, shape, dtype, both errors) to that file.
"""
import json
import os

import numpy as np
import torch

import oracle as o


def np32(t: torch.Tensor) -> np.ndarray:
    """torch (bf16/fp32, any device) -> exact float32 numpy."""
    return t.detach().float().cpu().numpy()


def codes(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.uint8)


def bf16_half_ulp(c: np.ndarray) -> np.ndarray:
    a = np.abs(c.astype(np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7) / 2


def gemm_error(C: torch.Tensor, R: np.ndarray) -> float:
    """max|C - R| / max|R| (the reported relative error)."""
    c = C.detach().float().cpu().numpy().astype(np.float64)
    den = float(np.max(np.abs(R)))
    return float(np.max(np.abs(c - R))) / (den if den > 0 else 1.0)


ELEM_FLOOR = 1e-2          # elements with |R_ij| >= ELEM_FLOOR * max|R| enter the elementwise error
# fp32 accumulation error only: measured at most 3.8e-5 (K = 16384, the FFN
# wgrad) and below 8e-6 for K <= 4096 on the GB300
ELEM_TOL_F32 = 1e-4
# the bf16 output rounding is up to half an ulp, 2^-8 of the value, plus the
# same accumulation slack
ELEM_TOL_BF16 = 2.0 ** -8 + 1e-4


def elementwise_rel_error(c: np.ndarray, R: np.ndarray, floor: float = ELEM_FLOOR) -> float:
    """max |c_ij - R_ij| / |R_ij| over |R_ij| >= floor * max|R| (0 if none)."""
    a = np.abs(R)
    if a.size == 0:
        return 0.0
    mask = a >= floor * float(a.max())
    if not np.any(mask) or float(a.max()) == 0.0:
        return 0.0
    return float(np.max(np.abs(c[mask] - R[mask]) / a[mask]))


def _report(C: torch.Tensor, norm_err: float, elem_err: float):
    path = os.environ.get("SQ_ERR_REPORT")
    if not path:
        return
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    with open(path, "a") as f:
        f.write(json.dumps({"test": test, "shape": list(C.shape), "dtype": str(C.dtype).replace("torch.", ""),
                            "norm_err": norm_err, "elem_err": elem_err}) + "\n")


def assert_gemm_close(C: torch.Tensor, R: np.ndarray, tol: float = 1e-3):
    c = C.detach().float().cpu().numpy().astype(np.float64)
    assert c.shape == R.shape
    assert np.all(np.isfinite(c)), "non-finite output"
    scale = float(np.max(np.abs(R))) if R.size else 0.0
    bound = tol * scale
    if C.dtype == torch.bfloat16:
        bound = bound + bf16_half_ulp(c)
    err = np.abs(c - R)
    bad = err > bound
    if np.any(bad):
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{int(bad.sum())} elements out of tolerance; first at {tuple(i)}: "
                             f"got {c[tuple(i)]!r}, oracle {R[tuple(i)]!r}, max|R| {scale}")
    norm_err = float(err.max()) / scale if scale > 0 else 0.0
    elem_err = elementwise_rel_error(c, R)
    _report(C, norm_err, elem_err)
    etol = ELEM_TOL_BF16 if C.dtype == torch.bfloat16 else ELEM_TOL_F32
    assert elem_err <= etol, f"elementwise relative error {elem_err:.3e} over |R| >= {ELEM_FLOOR} max|R| " \
                             f"exceeds {etol:.3e}"


def nan_aware_codes_equal(gpu: np.ndarray, ref: np.ndarray, fmt: int) -> bool:
    """bit-exact, except that any NaN code matches any NaN code"""
    table = np.array([np.isnan(o.decode(fmt, c)) for c in range(256)])
    g_nan, r_nan = table[gpu], table[ref]
    if not np.array_equal(g_nan, r_nan):
        return False
    return bool(np.array_equal(gpu[~g_nan], ref[~r_nan]))


def mx_untile(tiled: np.ndarray, R: int, C: int) -> np.ndarray:
    """Tiled MX scale layout (include/fp8sq.h, FP8SQ_MX32_TILED) -> the
    canonical [R][C/32] layout, by the header's index formula."""
    r = np.arange(R)[:, None]
    t = np.arange(C // 32)[None, :]
    off = ((r // 128) * (C // 128) + t // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (t % 4)
    return np.asarray(tiled).reshape(-1)[off]
