"""GPU parity of the FP8 linear layer (forward, dgrad, wgrad) under the
HYBRID delayed-scaling recipe and under current / fine-grained scaling:
histories and multipliers bit-exact every step, outputs within tolerance."""
import numpy as np
import pytest
import torch

import oracle as o
import scaled_quantize_gemm_gb300 as sq
from scaled_quantize_gemm_gb300 import workloads as wl

from _helpers import assert_gemm_close, codes, np32

pytestmark = pytest.mark.gpu
DEV = "cuda"


class Layer:
    """device buffers of one linear layer under delayed scaling"""

    def __init__(self, M, K, N, H=16):
        self.M, self.K, self.N, self.H = M, K, N, H
        self.states = torch.empty(3 * (H + 2), dtype=torch.float32, device=DEV)
        sq.fp8_scale_init(self.states, 3, H)
        self.ws = torch.empty(sq.fp8_linear_workspace_bytes(M, N, K), dtype=torch.uint8, device=DEV)
        self.y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
        self.dx = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
        self.dw = torch.empty((N, K), dtype=torch.float32, device=DEV)

    def st(self, i):
        return self.states[i * (self.H + 2):(i + 1) * (self.H + 2)]

    def step(self, x, w, dy, recipe=sq.RECIPE_HYBRID):
        sq.fp8_linear_fwd(x, w, self.y, self.ws, recipe=recipe, x_state=self.st(0), w_state=self.st(1),
                          history_len=self.H)
        sq.fp8_linear_bwd(dy, self.dx, self.dw, self.ws, self.K, recipe=recipe, dy_state=self.st(2),
                          history_len=self.H)


FORMATS = [sq.E4M3, sq.E4M3, sq.E5M2]       # x, W, dy under HYBRID


def _oracle_step(ref, x, w, dy, rows=None, wrows=None, dy_fmt=o.E5M2):
    qx, sx, qw, sw, Y = o.linear_fwd_delayed(np32(x), np32(w), ref[0], ref[1])
    if rows is not None:
        Y = Y[rows]
    _, _, dX, dW = o.linear_bwd_delayed(np32(dy), ref[2], dy_fmt, qx, sx, qw, sw, rows=rows, wrows=wrows)
    return Y, dX, dW


@pytest.mark.parametrize("M,K,N", [(256, 384, 512), (128, 128, 128), (272, 144, 400), (848, 1232, 688), (64, 2048, 96)])
def test_delayed_hybrid_steps(M, K, N):
    L = Layer(M, K, N)
    ref = [o.state_init(16) for _ in range(3)]
    w = wl.normal((N, K), 0.02, 3).to(DEV)
    for step in range(4):
        x = wl.normal((M, K), 1.0 + step, 10 + step).to(DEV)
        dy = wl.normal((M, N), 1e-3, 20 + step).to(DEV)
        L.step(x, w, dy)
        Y, dX, dW = _oracle_step(ref, x, w, dy)
        sq.fp8_update_scale(L.states, 3, 16, FORMATS)
        for r in range(3):
            o.update_scale(ref[r], FORMATS[r])
        torch.cuda.synchronize()
        assert_gemm_close(L.y, Y)
        assert_gemm_close(L.dx, dX)
        assert_gemm_close(L.dw, dW)
        assert L.states.cpu().numpy().tobytes() == np.concatenate(ref).tobytes(), step


@pytest.mark.parametrize("M,K,N", [(256, 384, 512), (272, 144, 400)])
def test_delayed_e4m3_only_recipe(M, K, N):
    """The E4M3-only recipe (Transformer Engine tutorial, closing suggestions:
    Format.E4M3 instead of HYBRID) under delayed scaling: the gradient's state
    is an E4M3 state (fmax 448) too.  Six steps with H = 16, a gradient spike
    at step 3; all three histories bit-exact every step."""
    H = 16
    L = Layer(M, K, N, H)
    ref = [o.state_init(H) for _ in range(3)]
    fmts = [sq.E4M3, sq.E4M3, sq.E4M3]
    w = wl.normal((N, K), 0.02, 13).to(DEV)
    for step in range(6):
        x = wl.normal((M, K), 1.0 + 0.5 * step, 110 + step).to(DEV)
        dy = wl.normal((M, N), 1e-3 * (20.0 if step == 3 else 1.0), 120 + step).to(DEV)
        L.step(x, w, dy, recipe=sq.RECIPE_E4M3)
        Y, dX, dW = _oracle_step(ref, x, w, dy, dy_fmt=o.E4M3)
        sq.fp8_update_scale(L.states, 3, H, fmts)
        for r in range(3):
            o.update_scale(ref[r], o.E4M3)
        torch.cuda.synchronize()
        assert_gemm_close(L.y, Y)
        assert_gemm_close(L.dx, dX)
        assert_gemm_close(L.dw, dW)
        assert L.states.cpu().numpy().tobytes() == np.concatenate(ref).tobytes(), step


def test_current_scaling_linear():
    M, K, N = 256, 256, 384
    x = wl.normal((M, K), 2.0, 1).to(DEV)
    w = wl.normal((N, K), 0.02, 2).to(DEV)
    dy = wl.normal((M, N), 1e-3, 3).to(DEV)
    ws = torch.empty(sq.fp8_linear_workspace_bytes(M, N, K), dtype=torch.uint8, device=DEV)
    y = torch.empty((M, N), dtype=torch.float32, device=DEV)
    dx = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    dw = torch.empty((N, K), dtype=torch.float32, device=DEV)
    sq.fp8_linear_fwd(x, w, y, ws)
    sq.fp8_linear_bwd(dy, dx, dw, ws, K, recipe=sq.RECIPE_E4M3)
    torch.cuda.synchronize()
    qx, _, sx, _ = o.quantize_tensor_current(np32(x), o.E4M3)
    qw, _, sw, _ = o.quantize_tensor_current(np32(w), o.E4M3)
    qd, _, sd, _ = o.quantize_tensor_current(np32(dy), o.E4M3)
    xh, wh, dh = (o.dequantize(qx, 0, 0, sx), o.dequantize(qw, 0, 0, sw), o.dequantize(qd, 0, 0, sd))
    assert_gemm_close(y, o.gemm_ref(xh, wh))
    assert_gemm_close(dx, o.gemm_ref(dh, wh.T))
    assert_gemm_close(dw, o.gemm_ref(dh.T, xh.T))


def test_tile_block_linear_forward():
    M, K, N = 256, 512, 384
    x = wl.student_t3((M, K), 4).to(DEV)
    w = wl.normal((N, K), 0.02, 5).to(DEV)
    ws = torch.empty(sq.fp8_linear_workspace_bytes(M, N, K, sq.TILE_1x128), dtype=torch.uint8, device=DEV)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    sq.fp8_linear_fwd(x, w, y, ws, gran=sq.TILE_1x128)
    torch.cuda.synchronize()
    qx, sx, _, _ = o.quantize_tile1x128(np32(x), o.E4M3)
    qw, sw, _, _ = o.quantize_block128(np32(w), o.E4M3)
    R = o.gemm_ref(o.dequantize(qx, 0, o.GRAN_TILE_1x128, sx), o.dequantize(qw, 0, o.GRAN_BLOCK_128x128, sw))
    assert_gemm_close(y, R)


def test_w2_minigpt_20_steps():
    """Workload 2: M = 2048 tokens (8 x 256), 768->2304, 768->3072, 3072->768,
    HYBRID delayed scaling, H = 16, max, 20 steps with the activation std
    drifting from 1 to 8.  All nine histories are compared bit for bit after
    every step; outputs on 64 sampled rows (and 64 sampled dW rows) per step."""
    wk = wl.WORKLOADS[2]
    layers, refs, ws_ = [], [], []
    for li, lin in enumerate(wk.linears):
        layers.append(Layer(wk.tokens, lin.in_features, lin.out_features, wk.history_len))
        refs.append([o.state_init(wk.history_len) for _ in range(3)])
        ws_.append(wl.linear_w(2, li, lin.out_features, lin.in_features, DEV))
    rng = np.random.default_rng(0)
    for step in range(wk.steps):
        for li, lin in enumerate(wk.linears):
            L = layers[li]
            x = wl.linear_x(2, li, step, wk.tokens, lin.in_features, DEV, std=wl.w2_sigma(step, wk.steps))
            dy = wl.linear_dy(2, li, step, wk.tokens, lin.out_features, DEV)
            L.step(x, ws_[li], dy)
            rows = np.sort(rng.choice(wk.tokens, 64, replace=False))
            wrows = np.sort(rng.choice(lin.out_features, 64, replace=False))
            Y, dX, dW = _oracle_step(refs[li], x, ws_[li], dy, rows=rows, wrows=wrows)
            torch.cuda.synchronize()
            assert_gemm_close(L.y[rows], Y)
            assert_gemm_close(L.dx[rows], dX)
            assert_gemm_close(L.dw[wrows], dW)
        for li in range(3):
            sq.fp8_update_scale(layers[li].states, 3, wk.history_len, FORMATS)
            for r in range(3):
                o.update_scale(refs[li][r], FORMATS[r])
        torch.cuda.synchronize()
        for li in range(3):
            assert layers[li].states.cpu().numpy().tobytes() == np.concatenate(refs[li]).tobytes(), (step, li)


def test_w5_ffn_step_full_size():
    """Workload 5 at full size, all 10 steps, through the bench's own step
    (bench.FFNStep: the granular calls chained as in a training step, x ->
    linear 0 -> y0 -> linear 1; dy -> linear 1's dgrad and wgrad -> dx1 ->
    linear 0's dgrad and wgrad, with W1, dy and dx1 cast on the side stream
    beside the GEMMs), HYBRID delayed scaling, H = 16.

    After every step: the codes of all six casts equal the oracle's over the
    whole tensor, y, dx and dW match the oracle on 32 sampled rows per GEMM,
    and all six histories are bit-exact after the update.  Each linear's
    input is the GPU's own output of the previous linear (checked there)."""
    import bench
    wk = wl.WORKLOADS[5]
    M, H = wk.tokens, wk.history_len
    step = bench.FFNStep(torch.device(DEV), n_input_sets=wk.steps)
    (K0, N0), (K1, N1) = step.lin
    B0, B1 = step.buf
    Wf = [np32(w) for w in step.W]
    ref = [o.state_init(H) for _ in range(6)]
    fmts = [o.E4M3, o.E4M3, o.E5M2] * 2
    rng = np.random.default_rng(1)

    def check_cast(src, fmt, si, q):
        s_used = np.float32(ref[si][H + 1])              # the state's scale before the cast
        rq, _ = o.quantize_delayed(np32(src), fmt, ref[si])
        assert np.array_equal(codes(q), rq), ("codes", si)
        return rq, s_used

    for s_ in range(wk.steps):
        step.step(s_)
        torch.cuda.synchronize()
        x, dy = step.inputs[s_]
        qx0, sx0 = check_cast(x, o.E4M3, 0, B0["qx"])
        qw0, sw0 = check_cast(step.W[0], o.E4M3, 1, B0["qw"])
        qw1, sw1 = check_cast(step.W[1], o.E4M3, 4, B1["qw"])
        qd1, sd1 = check_cast(dy, o.E5M2, 5, B1["qdy"])
        qx1, sx1 = check_cast(B0["y"], o.E4M3, 3, B1["qx"])
        qd0, sd0 = check_cast(B1["dx"], o.E5M2, 2, B0["qdy"])
        for (B, qx, sx, qw, sw, qd, sd, K, N) in ((B0, qx0, sx0, qw0, sw0, qd0, sd0, K0, N0),
                                                  (B1, qx1, sx1, qw1, sw1, qd1, sd1, K1, N1)):
            rows = np.sort(rng.choice(M, 32, replace=False))
            wrows = np.sort(rng.choice(N, 32, replace=False))
            wh = o.dequantize(qw, o.E4M3, o.GRAN_TENSOR, sw)
            assert_gemm_close(B["y"][rows], o.gemm_ref(o.dequantize(qx[rows], o.E4M3, o.GRAN_TENSOR, sx), wh))
            assert_gemm_close(B["dx"][rows], o.gemm_ref(o.dequantize(qd[rows], o.E5M2, o.GRAN_TENSOR, sd), wh.T))
            dcols = o.dequantize(np.ascontiguousarray(qd[:, wrows].T), o.E5M2, o.GRAN_TENSOR, sd)
            xh = o.dequantize(qx, o.E4M3, o.GRAN_TENSOR, sx)
            assert_gemm_close(B["dw"][wrows], o.gemm_ref(dcols, xh.T))
            del xh, dcols
        for i in range(6):
            o.update_scale(ref[i], fmts[i])
        assert step.states.cpu().numpy().tobytes() == np.concatenate(ref).tobytes(), s_
    assert sq.fp8_device_status(True) == 0


def test_w5_linear_api_full_size():
    """Workload 5 at full size through fp8_linear_fwd / fp8_linear_bwd (the
    calls the end-to-end leg of the bench times), two steps; histories
    bit-exact, 32 sampled rows of y, dx and dW per linear."""
    wk = wl.WORKLOADS[5]
    rng = np.random.default_rng(2)
    layers, refs, ws_ = [], [], []
    for li, lin in enumerate(wk.linears):
        layers.append(Layer(wk.tokens, lin.in_features, lin.out_features, wk.history_len))
        refs.append([o.state_init(wk.history_len) for _ in range(3)])
        ws_.append(wl.linear_w(5, li, lin.out_features, lin.in_features, DEV))
    for step in range(2):
        for li, lin in enumerate(wk.linears):
            L = layers[li]
            x = wl.linear_x(5, li, step, wk.tokens, lin.in_features, DEV)
            dy = wl.linear_dy(5, li, step, wk.tokens, lin.out_features, DEV)
            L.step(x, ws_[li], dy)
            rows = np.sort(rng.choice(wk.tokens, 32, replace=False))
            wrows = np.sort(rng.choice(lin.out_features, 32, replace=False))
            Y, dX, dW = _oracle_step(refs[li], x, ws_[li], dy, rows=rows, wrows=wrows)
            torch.cuda.synchronize()
            assert_gemm_close(L.y[rows], Y)
            assert_gemm_close(L.dx[rows], dX)
            assert_gemm_close(L.dw[wrows], dW)
            del x, dy
        for li in range(2):
            sq.fp8_update_scale(layers[li].states, 3, wk.history_len, FORMATS)
            for r in range(3):
                o.update_scale(refs[li][r], FORMATS[r])
        torch.cuda.synchronize()
        for li in range(2):
            assert layers[li].states.cpu().numpy().tobytes() == np.concatenate(refs[li]).tobytes(), (step, li)


def test_mx_linear_forward():
    M, K, N = 256, 512, 384
    x = wl.with_scaled_fraction((M, K), 1e-3, 100.0, 6).to(DEV)
    w = wl.normal((N, K), 0.02, 7).to(DEV)
    ws = torch.empty(sq.fp8_linear_workspace_bytes(M, N, K, sq.MX32), dtype=torch.uint8, device=DEV)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    sq.fp8_linear_fwd(x, w, y, ws, gran=sq.MX32)
    torch.cuda.synchronize()
    qx, ex, _, _ = o.quantize_mx32(np32(x), o.E4M3)
    qw, ew, _, _ = o.quantize_mx32(np32(w), o.E4M3)
    R = o.gemm_ref(o.dequantize(qx, 0, o.GRAN_MX32, ex), o.dequantize(qw, 0, o.GRAN_MX32, ew))
    assert_gemm_close(y, R)


@pytest.mark.parametrize("gran", [sq.TILE_1x128, sq.TILE_1x128_POW2, sq.MX32])
@pytest.mark.parametrize("recipe", [sq.RECIPE_E4M3, sq.RECIPE_HYBRID])
def test_fine_grained_linear_forward_and_backward(gran, recipe):
    """1x128 / 128x128 (with fp32 or power-of-two scales, and MX-32) forward,
    dgrad and wgrad, each operand quantised along its own contraction
    dimension, against the oracle."""
    M, K, N = 256, 384, 512
    x = wl.student_t3((M, K), 101).to(DEV)
    w = wl.normal((N, K), 0.02, 102).to(DEV)
    dy = wl.normal((M, N), 1e-3, 103).to(DEV)
    ws = torch.empty(sq.fp8_linear_workspace_bytes(M, N, K, gran), dtype=torch.uint8, device=DEV)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    dx = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    dw = torch.empty((N, K), dtype=torch.float32, device=DEV)
    sq.fp8_linear_fwd(x, w, y, ws, gran=gran)
    sq.fp8_linear_bwd(dy, dx, dw, ws, K, gran=gran, recipe=recipe)
    torch.cuda.synchronize()
    og = {sq.TILE_1x128: o.GRAN_TILE_1x128, sq.TILE_1x128_POW2: o.GRAN_TILE_POW2, sq.MX32: o.GRAN_MX32}[gran]
    st, Y = o.linear_fine_fwd(np32(x), np32(w), og)
    dX, dW = o.linear_fine_bwd(st, np32(dy), og, o.E5M2 if recipe == sq.RECIPE_HYBRID else o.E4M3)
    assert_gemm_close(y, Y)
    assert_gemm_close(dx, dX)
    assert_gemm_close(dw, dW)


def _fine_forward_operands(x, w, og):
    """The oracle's forward operands of the fine-grained recipes, dequantised,
    and the backward state (W's codes and scales for the tile recipes)."""
    if og == o.GRAN_TILE_1x128:
        qx, sx, _, _ = o.quantize_tile1x128(x, o.E4M3)
        qw, sw, _, _ = o.quantize_block128(w, o.E4M3)
        return (o.dequantize(qx, o.E4M3, og, sx), o.dequantize(qw, o.E4M3, o.GRAN_BLOCK_128x128, sw),
                {"x": x, "w": w, "qw": qw, "sw": sw})
    if og == o.GRAN_TILE_POW2:
        qx, ex, _ = o.quantize_tile1x128_pow2(x, o.E4M3)
        qw, ew, _ = o.quantize_block128_pow2(w, o.E4M3)
        return (o.dequantize(qx, o.E4M3, og, ex), o.dequantize(qw, o.E4M3, o.GRAN_BLOCK_POW2, ew),
                {"x": x, "w": w, "qw": qw, "sw": ew})
    qx, ex, _, _ = o.quantize_mx32(x, o.E4M3)
    qw, ew, _, _ = o.quantize_mx32(w, o.E4M3)
    return o.dequantize(qx, o.E4M3, og, ex), o.dequantize(qw, o.E4M3, og, ew), {"x": x, "w": w}


@pytest.mark.parametrize("gran", [sq.TILE_1x128, sq.TILE_1x128_POW2, sq.MX32])
def test_fine_grained_linear_full_size_sampled_rows(gran):
    """Workload 3's shapes and data (M = N = K = 4096: Student-t x, N(0, 0.02)
    W, N(0, 1e-3) dy) through fp8_linear_fwd / fp8_linear_bwd in the launch
    configuration the bench times: y, dx and dW on 32 sampled rows each
    against the oracle's products of its own operands (HYBRID: dy in E5M2)."""
    n = 4096
    x, w = wl.w3_operands(DEV)
    dy = wl.normal((n, n), 1e-3, wl.seed_of(3, 0, wl.ROLE_DY), DEV)
    ws = torch.empty(sq.fp8_linear_workspace_bytes(n, n, n, gran), dtype=torch.uint8, device=DEV)
    y = torch.empty((n, n), dtype=torch.bfloat16, device=DEV)
    dx = torch.empty((n, n), dtype=torch.bfloat16, device=DEV)
    dw = torch.empty((n, n), dtype=torch.float32, device=DEV)
    sq.fp8_linear_fwd(x, w, y, ws, gran=gran)
    sq.fp8_linear_bwd(dy, dx, dw, ws, n, gran=gran)
    torch.cuda.synchronize()
    og = {sq.TILE_1x128: o.GRAN_TILE_1x128, sq.TILE_1x128_POW2: o.GRAN_TILE_POW2, sq.MX32: o.GRAN_MX32}[gran]
    xh, wh, st = _fine_forward_operands(np32(x), np32(w), og)
    ops = o.linear_fine_bwd_operands(st, np32(dy), og, o.E5M2)
    rng = np.random.default_rng(33)
    ry, rx, rw = (np.sort(rng.choice(n, size=32, replace=False)) for _ in range(3))
    assert_gemm_close(y[ry], o.gemm_ref(xh[ry], wh))
    assert_gemm_close(dx[rx], ops["dgrad_dy"][2][rx] @ ops["dgrad_w"][2])
    assert_gemm_close(dw[rw], ops["wgrad_dy"][2][:, rw].T @ ops["wgrad_x"][2])
    assert sq.fp8_device_status(True) == 0
