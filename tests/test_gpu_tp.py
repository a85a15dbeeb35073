"""The column-parallel FP8 linear's per-rank path on the GPU (LibraryOps:
delayed per-tensor casts and FP8 GEMMs through the C ABI), in a
tensor-parallel group of one rank on NCCL: the gathered output, the input
gradient (fp32, all-reduced) and the weight gradient against the oracle,
histories bit-exact every step.  The two-rank exchange logic is covered on
CPU ranks (tests/test_tp_gloo.py); this run uses one GPU."""
import datetime
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

import oracle as o
import scaled_quantize_gemm_gb300 as sq
from scaled_quantize_gemm_gb300 import tp
from scaled_quantize_gemm_gb300 import workloads as wl

from _helpers import assert_gemm_close, np32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_column_parallel_linear_one_rank_matches_oracle():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                            timeout=datetime.timedelta(seconds=120), device_id=torch.device(DEV, 0))
    try:
        M, K, N, H = 256, 384, 512, 16
        w = wl.normal((N, K), 0.02, 71).to(DEV)
        layer = tp.ColumnParallelFP8Linear(tp.shard_rows(w, 0, 1), M, history_len=H)
        ref = [o.state_init(H) for _ in range(3)]
        qo, so = torch.empty((128, K), dtype=torch.uint8, device=DEV), torch.empty(1, device=DEV)
        ao = torch.empty(1, device=DEV)
        for step in range(4):
            x = wl.normal((M, K), 1.0 + step, 72 + step).to(DEV)
            dy = wl.normal((M, N), 1e-3 * (30.0 if step == 2 else 1.0), 80 + step).to(DEV)
            handle = layer.forward_async(x)
            # independent work in the window: another cast of the same input
            sq.fp8_quantize(x[:128], sq.E4M3, sq.TENSOR, qo, scales_out=so, amax_out=ao)
            y = handle.wait()
            dx, dw = layer.backward(dy)
            layer.end_step()
            torch.cuda.synchronize()
            qx, sx, qw, sw, Y = o.linear_fwd_delayed(np32(x), np32(w), ref[0], ref[1])
            _, _, dX, dW = o.linear_bwd_delayed(np32(dy), ref[2], o.E5M2, qx, sx, qw, sw)
            for r, f in zip(ref, (o.E4M3, o.E4M3, o.E5M2)):
                o.update_scale(r, f)
            assert_gemm_close(y, Y)
            assert_gemm_close(dx, dX)
            assert_gemm_close(dw, dW)
            assert layer.ops.states.cpu().numpy().tobytes() == np.concatenate(ref).tobytes(), step
        assert sq.fp8_device_status(True) == 0
    finally:
        dist.destroy_process_group()


def test_row_parallel_linear_one_rank_matches_oracle():
    """The row-parallel linear's per-rank path (fp32 partial output through
    the library's GEMM, then the all-reduce) in a group of one rank on NCCL:
    the output, the input gradient and the weight gradient against the
    oracle, histories bit-exact every step."""
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                            timeout=datetime.timedelta(seconds=120), device_id=torch.device(DEV, 0))
    try:
        M, K, N, H = 256, 512, 384, 16
        w = wl.normal((N, K), 0.02, 91).to(DEV)
        layer = tp.RowParallelFP8Linear(tp.shard_cols(w, 0, 1), M, history_len=H)
        ref = [o.state_init(H) for _ in range(3)]
        for step in range(4):
            x = wl.normal((M, K), 1.0 + step, 92 + step).to(DEV)
            dy = wl.normal((M, N), 1e-3 * (30.0 if step == 1 else 1.0), 96 + step).to(DEV)
            work, y = layer.forward(tp.shard_cols(x, 0, 1), async_op=True)
            work.wait()
            dx, dw = layer.backward(dy)
            layer.end_step()
            torch.cuda.synchronize()
            assert y.dtype == torch.float32
            qx, sx, qw, sw, Y = o.linear_fwd_delayed(np32(x), np32(w), ref[0], ref[1])
            _, _, dX, dW = o.linear_bwd_delayed(np32(dy), ref[2], o.E5M2, qx, sx, qw, sw)
            for r, f in zip(ref, (o.E4M3, o.E4M3, o.E5M2)):
                o.update_scale(r, f)
            assert_gemm_close(y, Y)
            assert_gemm_close(dx, dX)
            assert_gemm_close(dw, dW)
            assert layer.ops.states.cpu().numpy().tobytes() == np.concatenate(ref).tobytes(), step
        assert sq.fp8_device_status(True) == 0
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("gran,og", [(sq.TILE_1x128, o.GRAN_TILE_1x128), (sq.TILE_1x128_POW2, o.GRAN_TILE_POW2),
                                     (sq.MX32, o.GRAN_MX32)])
def test_data_parallel_fine_grained_one_rank_matches_oracle(gran, og):
    """The data-parallel linear's per-rank path under a fine-grained recipe
    (FineOps: fp8_linear_fwd / fp8_linear_bwd) in a group of one rank on
    NCCL: y, dx and the all-reduced dW against the oracle."""
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                            timeout=datetime.timedelta(seconds=120), device_id=torch.device(DEV, 0))
    try:
        M, K, N = 256, 384, 512
        w = wl.normal((N, K), 0.02, 191).to(DEV)
        layer = tp.DataParallelFP8Linear(w, M, gran=gran)
        assert isinstance(layer.ops, tp.FineOps)
        for step in range(2):
            x = wl.student_t3((M, K), 192 + step).to(DEV)
            dy = wl.normal((M, N), 1e-3, 196 + step).to(DEV)
            y = layer.forward(x)
            dx, dw = layer.backward(dy)
            layer.end_step()
            torch.cuda.synchronize()
            st, Y = o.linear_fine_fwd(np32(x), np32(w), og)
            dX, dW = o.linear_fine_bwd(st, np32(dy), og, o.E5M2)
            assert_gemm_close(y, Y)
            assert_gemm_close(dx, dX)
            assert_gemm_close(dw, dW)
        assert sq.fp8_device_status(True) == 0
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("gran,og", [(sq.TILE_1x128, o.GRAN_TILE_1x128), (sq.TILE_1x128_POW2, o.GRAN_TILE_POW2),
                                     (sq.MX32, o.GRAN_MX32)])
def test_row_parallel_fine_grained_one_rank_matches_oracle(gran, og):
    """The row-parallel linear's per-rank path under a fine-grained recipe
    (FineOps: fp32 partial output, then the all-reduce) in a group of one
    rank on NCCL: y, dx and dW against the oracle."""
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                            timeout=datetime.timedelta(seconds=120), device_id=torch.device(DEV, 0))
    try:
        M, K, N = 256, 512, 384
        w = wl.normal((N, K), 0.02, 291).to(DEV)
        layer = tp.RowParallelFP8Linear(tp.shard_cols(w, 0, 1), M, gran=gran)
        assert isinstance(layer.ops, tp.FineOps)
        for step in range(2):
            x = wl.student_t3((M, K), 292 + step).to(DEV)
            dy = wl.normal((M, N), 1e-3, 296 + step).to(DEV)
            work, y = layer.forward(tp.shard_cols(x, 0, 1), async_op=True)
            work.wait()
            dx, dw = layer.backward(dy)
            layer.end_step()
            torch.cuda.synchronize()
            assert y.dtype == torch.float32
            st, Y = o.linear_fine_fwd(np32(x), np32(w), og)
            dX, dW = o.linear_fine_bwd(st, np32(dy), og, o.E5M2)
            assert_gemm_close(y, Y)
            assert_gemm_close(dx, dX)
            assert_gemm_close(dw, dW)
        assert sq.fp8_device_status(True) == 0
    finally:
        dist.destroy_process_group()
