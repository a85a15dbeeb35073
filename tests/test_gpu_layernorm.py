"""LayerNorm fused into the FP8 cast (te.LayerNormLinear's normalisation),
against the oracle's float64 LayerNorm.

The row statistics are fp32 reductions in an order the pages do not fix, so a
code may legitimately differ from the exact LayerNorm's code where y * m
lies within the reductions' rounding error of a midpoint between two codes.
The check: mean and rstd within fp32 reduction error; every code inside the
bracket of codes reachable from y +- delta, with delta = 2^-14 (|t gamma| +
|gamma| + |beta|), t the standardised value (a bound 8x looser than the
fp32 error of the reductions at K <= 4096); at least 99 % of codes equal to
the exact LayerNorm's nearest code; the transposed copy exact; the recorded
amax within 1e-5 of the exact one.
"""
import numpy as np
import pytest
import torch

import oracle as o
import scaled_quantize_gemm_gb300 as sq
from scaled_quantize_gemm_gb300 import workloads as wl

from _helpers import assert_gemm_close, codes, np32

pytestmark = pytest.mark.gpu
DEV = "cuda"
EPS = 1e-5


def _inputs(M, K, seed):
    g = torch.Generator().manual_seed(seed)
    x = (wl.normal((M, K), 2.0, seed, dtype=torch.float32) + 0.7).to(torch.bfloat16)
    gamma = torch.rand(K, generator=g) + 0.5
    beta = torch.randn(K, generator=g) * 0.1
    return x, gamma, beta


def _check_ln_codes(x, gamma, beta, q, mu, rstd, m, fmt):
    xf = np32(x)
    y, mu_o, rs_o = o.layernorm(xf, gamma.numpy(), beta.numpy(), EPS)
    mu_g, rs_g = mu.cpu().numpy().astype(np.float64), rstd.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(mu_g - mu_o) <= 1e-5 * (np.abs(mu_o) + 1.0 / rs_o))
    assert np.all(np.abs(rs_g / rs_o - 1.0) <= 2e-5)
    t = (xf.astype(np.float64) - mu_o[:, None]) * rs_o[:, None]
    g64, b64 = gamma.numpy().astype(np.float64), beta.numpy().astype(np.float64)
    delta = 2.0 ** -14 * (np.abs(t * g64) + np.abs(g64) + np.abs(b64))
    near, lo, hi = o.ln_acceptable_codes(y, delta, m, fmt)
    gq = codes(q)
    r = o.code_rank
    assert np.all((r(lo) <= r(gq)) & (r(gq) <= r(hi))), "a code outside the reachable bracket"
    assert np.mean(gq == near) >= 0.99
    return y


@pytest.mark.parametrize("fmt", [sq.E4M3, sq.E5M2])
@pytest.mark.parametrize("M,K", [(256, 768), (128, 4096), (272, 144)])
def test_layernorm_fused_cast(fmt, M, K):
    x, gamma, beta = _inputs(M, K, 7 + K)
    H = 16
    st = torch.tensor(o.state_init(H), device=DEV)
    m = 448.0 / 6.0 if fmt == sq.E4M3 else 57344.0 / 6.0
    st[H] = float(np.float32(m))
    q, qT = torch.empty((M, K), dtype=torch.uint8, device=DEV), torch.empty((K, M), dtype=torch.uint8, device=DEV)
    mu, rstd = torch.empty(M, device=DEV), torch.empty(M, device=DEV)
    sq.fp8_layernorm_quantize(x.to(DEV), gamma.to(DEV), beta.to(DEV), EPS, fmt, q, qT, mu, rstd, st, H)
    torch.cuda.synchronize()
    y = _check_ln_codes(x, gamma, beta, q, mu, rstd, np.float32(m), fmt)
    assert np.array_equal(codes(qT), codes(q).T)
    assert abs(float(st[0].item()) / np.max(np.abs(y)) - 1.0) <= 1e-5


def test_layernorm_linear_forward_and_backward():
    """LayerNormLinear forward (LN cast, W cast, GEMM) over three delayed
    steps, then the linear backward from the same workspace."""
    M, K, N, H = 256, 768, 512, 16
    w = wl.normal((N, K), 0.02, 3).to(DEV)
    states = torch.empty(3 * (H + 2), device=DEV)
    sq.fp8_scale_init(states, 3, H)
    st = [states[i * (H + 2):(i + 1) * (H + 2)] for i in range(3)]
    ws = torch.empty(sq.fp8_linear_workspace_bytes(M, N, K), dtype=torch.uint8, device=DEV)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    dx = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    dw = torch.empty((N, K), dtype=torch.float32, device=DEV)
    mu, rstd = torch.empty(M, device=DEV), torch.empty(M, device=DEV)
    ref_w = o.state_init(H)
    for step in range(3):
        x, gamma, beta = _inputs(M, K, 30 + step)
        dy = wl.normal((M, N), 1e-3, 40 + step).to(DEV)
        m_x = float(st[0][H].item())
        s_x = np.float32(st[0][H + 1].item())
        sq.fp8_layernorm_linear_fwd(x.to(DEV), gamma.to(DEV), beta.to(DEV), EPS, w, y, ws, mu, rstd, st[0], st[1], H)
        sq.fp8_linear_bwd(dy, dx, dw, ws, K, dy_state=st[2], history_len=H)
        torch.cuda.synchronize()
        # LayerNorm codes of x, checked against the exact LayerNorm
        yln, _, _ = o.layernorm(np32(x), gamma.numpy(), beta.numpy(), EPS)
        near, _, _ = o.ln_acceptable_codes(yln, np.zeros_like(yln), m_x, o.E4M3)
        qw, _ = o.quantize_delayed(np32(w), o.E4M3, ref_w)
        s_w = np.float32(ref_w[H + 1])
        R = o.gemm_ref(o.dequantize(near, o.E4M3, 0, s_x), o.dequantize(qw, o.E4M3, 0, s_w))
        assert_gemm_close(y, R)
        sq.fp8_update_scale(states, 3, H, [sq.E4M3, sq.E4M3, sq.E5M2])
        o.update_scale(ref_w, o.E4M3)
        torch.cuda.synchronize()
        assert np.all(np.isfinite(dx.float().cpu().numpy())) and np.all(np.isfinite(dw.cpu().numpy()))
