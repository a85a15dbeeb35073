"""The linear-layer path captured in a CUDA graph: no call of the forward,
backward or scale update synchronises or allocates, so a whole training
step (delayed scaling, amax histories included) can be captured once and
replayed.  Replays on fresh inputs must give bit-identical outputs and
states to the same steps run eagerly."""
import numpy as np
import pytest
import torch

import scaled_quantize_gemm_gb300 as sq
from scaled_quantize_gemm_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"
H = 16
FORMATS = [sq.E4M3, sq.E4M3, sq.E5M2]


class Step:
    def __init__(self, M, K, N):
        self.M, self.K, self.N = M, K, N
        self.states = torch.empty(3 * (H + 2), dtype=torch.float32, device=DEV)
        sq.fp8_scale_init(self.states, 3, H)
        self.ws = torch.empty(sq.fp8_linear_workspace_bytes(M, N, K), dtype=torch.uint8, device=DEV)
        self.x = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
        self.w = torch.empty((N, K), dtype=torch.bfloat16, device=DEV)
        self.dy = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
        self.y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
        self.dx = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
        self.dw = torch.empty((N, K), dtype=torch.float32, device=DEV)

    def st(self, i):
        return self.states[i * (H + 2):(i + 1) * (H + 2)]

    def run(self):
        sq.fp8_linear_fwd(self.x, self.w, self.y, self.ws, x_state=self.st(0), w_state=self.st(1), history_len=H)
        sq.fp8_linear_bwd(self.dy, self.dx, self.dw, self.ws, self.K, dy_state=self.st(2), history_len=H)
        sq.fp8_update_scale(self.states, 3, H, FORMATS)


def _inputs(M, K, N, step):
    return (wl.normal((M, K), 1.0 + step, 300 + step, DEV), wl.normal((N, K), 0.02, 400, DEV),
            wl.normal((M, N), 1e-3, 500 + step, DEV))


@pytest.mark.parametrize("M,K,N", [(2048, 768, 2304), (272, 144, 400)])
def test_linear_step_graph_replay_matches_eager(M, K, N):
    steps = 4
    eager = Step(M, K, N)
    outs = []
    for s in range(steps):
        x, w, dy = _inputs(M, K, N, s)
        eager.x.copy_(x); eager.w.copy_(w); eager.dy.copy_(dy)
        eager.run()
        outs.append((eager.y.clone(), eager.dx.clone(), eager.dw.clone(), eager.states.clone()))
    torch.cuda.synchronize()

    g_step = Step(M, K, N)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):          # first calls (one-time queries) outside the capture
        g_step.run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    sq.fp8_scale_init(g_step.states, 3, H)  # start from the same state as the eager run
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g_step.run()
    # capturing does not execute: the state is still the initial one
    torch.cuda.synchronize()
    for s in range(steps):
        x, w, dy = _inputs(M, K, N, s)
        g_step.x.copy_(x); g_step.w.copy_(w); g_step.dy.copy_(dy)
        graph.replay()
        torch.cuda.synchronize()
        y, dx, dw, st = outs[s]
        assert torch.equal(g_step.y, y), s
        assert torch.equal(g_step.dx, dx), s
        assert torch.equal(g_step.dw, dw), s
        assert np.array_equal(g_step.states.cpu().numpy().view(np.uint32), st.cpu().numpy().view(np.uint32)), s
    assert sq.fp8_device_status(True) == sq.OK


@pytest.mark.parametrize("gran", [sq.TILE_1x128, sq.TILE_1x128_POW2, sq.MX32])
def test_fine_grained_linear_graph_replay_matches_eager(gran):
    """The fine-grained recipes (current scaling per unit, fp32 or
    power-of-two tile scales, MX-32) captured once: replays on fresh inputs
    give bit-identical y, dx and dW to eager calls."""
    M, K, N = 256, 384, 512
    steps = 3
    ws = torch.empty(sq.fp8_linear_workspace_bytes(M, N, K, gran), dtype=torch.uint8, device=DEV)
    x = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    w = torch.empty((N, K), dtype=torch.bfloat16, device=DEV)
    dy = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    dx = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    dw = torch.empty((N, K), dtype=torch.float32, device=DEV)

    def run():
        sq.fp8_linear_fwd(x, w, y, ws, gran=gran)
        sq.fp8_linear_bwd(dy, dx, dw, ws, K, gran=gran)

    def inputs(s):
        return (wl.student_t3((M, K), 600 + s, DEV), wl.normal((N, K), 0.02, 700 + s, DEV),
                wl.normal((M, N), 1e-3, 800 + s, DEV))

    outs = []
    for s in range(steps):
        a, b, c = inputs(s)
        x.copy_(a); w.copy_(b); dy.copy_(c)
        run()
        outs.append((y.clone(), dx.clone(), dw.clone()))
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):          # first calls (one-time queries) outside the capture
        run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    for s in range(steps):
        a, b, c = inputs(s)
        x.copy_(a); w.copy_(b); dy.copy_(c)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, outs[s][0]), s
        assert torch.equal(dx, outs[s][1]), s
        assert torch.equal(dw, outs[s][2]), s
    assert sq.fp8_device_status(True) == sq.OK
