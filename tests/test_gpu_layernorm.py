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
    # + 2^-20 |y|: room for a multiplier a few ulps away from m (the GPU's
    # own, derived from its fp32 amax history)
    delta = 2.0 ** -14 * (np.abs(t * g64) + np.abs(g64) + np.abs(b64)) + 2.0 ** -20 * np.abs(y)
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
    """LayerNormLinear forward (LN cast, W cast, GEMM) then the linear
    backward from the same workspace, over four delayed steps.

    The W and dy states are bit-exact against the oracle's every step.  The x
    state follows the exact (float64) LayerNorm's amax: every history entry
    within 1e-5 of the oracle's, and the update rule applied exactly to the
    GPU's own history.  The LayerNorm codes (re-derived by the same cast on a
    copy of the pre-step state) sit inside the reachable bracket of the exact
    LayerNorm under the oracle's multiplier; y, dx and dW are then compared
    with the oracle's float64 products of those codes, the oracle's W codes
    and the oracle's own dy codes."""
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
    qln, qlnT = torch.empty((M, K), dtype=torch.uint8, device=DEV), torch.empty((K, M), dtype=torch.uint8, device=DEV)
    mu2, rstd2 = torch.empty(M, device=DEV), torch.empty(M, device=DEV)
    ref_x, ref_w, ref_dy = o.state_init(H), o.state_init(H), o.state_init(H)
    wf = np32(w)
    for step in range(4):
        x, gamma, beta = _inputs(M, K, 30 + step)
        # a gradient spike at step 2 moves the dy scale through its history
        dy = wl.normal((M, N), 1e-3 * (30.0 if step == 2 else 1.0), 40 + step).to(DEV)
        xd, gd, bd = x.to(DEV), gamma.to(DEV), beta.to(DEV)
        pre_x = st[0].clone()
        sq.fp8_layernorm_linear_fwd(xd, gd, bd, EPS, w, y, ws, mu, rstd, st[0], st[1], H)
        sq.fp8_linear_bwd(dy, dx, dw, ws, K, dy_state=st[2], history_len=H)
        # the LayerNorm codes the forward used: the same cast, from a copy of
        # the pre-step x state
        sq.fp8_layernorm_quantize(xd, gd, bd, EPS, sq.E4M3, qln, qlnT, mu2, rstd2, pre_x, H)
        torch.cuda.synchronize()
        m_x_gpu = np.float32(st[0][H].item())
        s_x_gpu = np.float32(st[0][H + 1].item())
        m_x, s_x = np.float32(ref_x[H]), np.float32(ref_x[H + 1])
        assert abs(m_x_gpu / m_x - 1.0) <= 1e-5 and abs(s_x_gpu / s_x - 1.0) <= 1e-5, step
        yln = _check_ln_codes(x, gamma, beta, qln, mu, rstd, m_x, o.E4M3)
        assert np.array_equal(codes(mu2.view(torch.uint8)), codes(mu.view(torch.uint8)))
        # oracle: W and dy codes and their states (bit-exact below)
        qw, _ = o.quantize_delayed(wf, o.E4M3, ref_w)
        s_w = np.float32(ref_w[H + 1])
        qd, _ = o.quantize_delayed(np32(dy), o.E5M2, ref_dy)
        s_d = np.float32(ref_dy[H + 1])
        ref_x[0] = np.float32(np.max(np.abs(yln)))
        xh = o.dequantize(codes(qln), o.E4M3, o.GRAN_TENSOR, s_x_gpu)
        wh = o.dequantize(qw, o.E4M3, o.GRAN_TENSOR, s_w)
        dh = o.dequantize(qd, o.E5M2, o.GRAN_TENSOR, s_d)
        assert_gemm_close(y, o.gemm_ref(xh, wh))
        assert_gemm_close(dx, o.gemm_ref(dh, wh.T))
        assert_gemm_close(dw, o.gemm_ref(dh.T, xh.T))
        # end of step: update, then compare the states
        gpu_x_before = st[0].cpu().numpy().copy()
        sq.fp8_update_scale(states, 3, H, [sq.E4M3, sq.E4M3, sq.E5M2])
        for ref, fmt in ((ref_x, o.E4M3), (ref_w, o.E4M3), (ref_dy, o.E5M2)):
            o.update_scale(ref, fmt)
        o.update_scale(gpu_x_before, o.E4M3)
        torch.cuda.synchronize()
        got = states.cpu().numpy()
        gx, gw, gd_ = got[:H + 2], got[H + 2:2 * (H + 2)], got[2 * (H + 2):]
        assert gw.tobytes() == ref_w.tobytes(), step
        assert gd_.tobytes() == ref_dy.tobytes(), step
        assert gx.tobytes() == gpu_x_before.tobytes(), step          # the update rule, exactly
        nz = ref_x[:H] > 0
        assert np.array_equal(gx[:H] > 0, nz)
        assert np.all(np.abs(gx[:H][nz] / ref_x[:H][nz] - 1.0) <= 1e-5), step


def _random_ln_shapes(seed, n):
    """seeded (rows, width) pairs, both multiples of 16, widths up to 6000"""
    rng = np.random.default_rng(seed)
    return [(int(rng.integers(1, 129)) * 16, int(rng.integers(1, 376)) * 16, bool(i % 2)) for i in range(n)]


@pytest.mark.parametrize("fmt", [sq.E4M3, sq.E5M2])
@pytest.mark.parametrize("M,K,with_beta", [(272, 144, True), (4096, 4096, True), (2064, 1040, False),
                                           (64, 4112, True), (48, 16, True), (32, 2064, False)]
                         + _random_ln_shapes(5, 4))
def test_layernorm_single_pass_matches_two_pass(fmt, M, K, with_beta):
    """Without a transposed copy the LayerNorm cast runs in one pass (each
    row held in registers from the statistics to the codes, rows of up to
    4096); with one it runs as a statistics kernel and a tiled cast.  Both
    take the same fp32 reductions in the same order and the same per-element
    arithmetic, so the codes, mean, rstd, the recorded amax and the reported
    scale are bit-identical.  The shapes: an odd number of 8-element chunks
    per row (144), the largest single-pass row (4096) over more rows than
    one wave of CTAs holds, no beta, a row too long for the single pass
    (4112, both calls take the two-pass path), a row of two chunks (16) and
    one where a few threads hold a second chunk (2064)."""
    x, gamma, beta = _inputs(M, K, 90 + K)
    beta = beta if with_beta else None
    H = 16
    xd, gd = x.to(DEV), gamma.to(DEV)
    bd = beta.to(DEV) if beta is not None else None
    out = []
    for with_qT in (False, True):
        st = torch.tensor(o.state_init(H), device=DEV)
        st[H] = float(np.float32(17.25))
        st[H + 1] = float(np.float32(1.0 / 17.25))
        q = torch.full((M, K), 0x55, dtype=torch.uint8, device=DEV)
        qT = torch.empty((K, M), dtype=torch.uint8, device=DEV) if with_qT else None
        mu, rstd = torch.full((M,), 7.0, device=DEV), torch.full((M,), 7.0, device=DEV)
        sq.fp8_layernorm_quantize(xd, gd, bd, EPS, fmt, q, qT, mu, rstd, st, H)
        torch.cuda.synchronize()
        out.append((codes(q), mu.cpu().numpy().tobytes(), rstd.cpu().numpy().tobytes(), st.cpu().numpy().tobytes()))
    for a, b in zip(out[0], out[1]):
        assert np.array_equal(a, b) if isinstance(a, np.ndarray) else a == b
    # and the single pass against the exact LayerNorm, as for the two-pass
    # cast (on the first and last 256 rows)
    rows = torch.cat([torch.arange(min(M, 256)), torch.arange(max(M - 256, min(M, 256)), M)])
    beta_c = beta if beta is not None else torch.zeros(K)
    q1 = torch.from_numpy(out[0][0])[rows]
    mu1 = torch.from_numpy(np.frombuffer(out[0][1], dtype=np.float32).copy())[rows]
    rs1 = torch.from_numpy(np.frombuffer(out[0][2], dtype=np.float32).copy())[rows]
    _check_ln_codes(x[rows], gamma, beta_c, q1, mu1, rs1, np.float32(17.25), fmt)


def test_layernorm_non_finite_rows_agree():
    """A row holding an inf (its mean is inf, its variance NaN) and a row
    holding a NaN normalise to NaN everywhere: both LayerNorm paths must give
    the same codes, statistics and recorded amax (the NaN), bit for bit, and
    the finite rows must be unaffected."""
    M, K, H = 64, 768, 16
    x, gamma, beta = _inputs(M, K, 5)
    x[3, 17] = float("inf")
    x[40, 5] = float("nan")
    xd, gd, bd = x.to(DEV), gamma.to(DEV), beta.to(DEV)
    out = []
    for with_qT in (False, True):
        st = torch.tensor(o.state_init(H), device=DEV)
        q = torch.empty((M, K), dtype=torch.uint8, device=DEV)
        qT = torch.empty((K, M), dtype=torch.uint8, device=DEV) if with_qT else None
        mu, rstd = torch.empty(M, device=DEV), torch.empty(M, device=DEV)
        sq.fp8_layernorm_quantize(xd, gd, bd, EPS, sq.E4M3, q, qT, mu, rstd, st, H)
        torch.cuda.synchronize()
        out.append((codes(q), mu.cpu().numpy().tobytes(), rstd.cpu().numpy().tobytes(), st.cpu().numpy().tobytes()))
    for a, b in zip(out[0], out[1]):
        assert np.array_equal(a, b) if isinstance(a, np.ndarray) else a == b
    st = np.frombuffer(out[0][3], dtype=np.float32)
    assert np.isnan(st[0])
    q = out[0][0]
    assert np.all((q[3] & 0x7F) == 0x7F) and np.all((q[40] & 0x7F) == 0x7F)     # NaN codes
    finite = [r for r in range(M) if r not in (3, 40)]
    assert np.all((q[finite] & 0x7F) != 0x7F)
