"""Column-parallel FP8 linear ("Transformer Scaling", "04 · Put it back into
code -- Program model": local linear, asynchronous all-gather, independent
work in the window, wait at the first consumer) on two CPU ranks with gloo.

Each rank's arithmetic runs in the oracle (an implementation of the layer's
five per-rank operations on numpy), so what is under test is the host-side
tensor-parallel logic of scaled_quantize_gemm_gb300.tp: W sharded along N,
the gathered output, the summed input gradient, the local weight gradient,
and the amax all-reduce that keeps every rank's delayed-scaling state
bit-identical.  Every step is compared with the unsharded layer computed by
the same oracle operations on one rank.  A run that skips the amax
all-reduce must diverge (the W shards have different amaxes)."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
M, K, N, H, STEPS = 64, 96, 128, 8, 4


class OracleOps:
    """The per-rank operations of a column-parallel linear on the CPU
    oracle: delayed per-tensor casts (x, W in E4M3, dy in E5M2) and float64
    products of the dequantised codes."""

    def __init__(self, H):
        import oracle as o
        self.o = o
        self.H = H
        self.st = [o.state_init(H) for _ in range(3)]
        self.fmts = [o.E4M3, o.E4M3, o.E5M2]

    def forward(self, x, w):
        o, H = self.o, self.H
        sx, sw = np.float32(self.st[0][H + 1]), np.float32(self.st[1][H + 1])
        qx, _ = o.quantize_delayed(x.numpy(), o.E4M3, self.st[0])
        qw, _ = o.quantize_delayed(w.numpy(), o.E4M3, self.st[1])
        self.xh = o.dequantize(qx, o.E4M3, o.GRAN_TENSOR, sx)
        self.wh = o.dequantize(qw, o.E4M3, o.GRAN_TENSOR, sw)
        return torch.from_numpy(o.gemm_ref(self.xh, self.wh))

    def forward_partial(self, x, w):
        return self.forward(x, w)

    def backward(self, dy):
        o, H = self.o, self.H
        sd = np.float32(self.st[2][H + 1])
        qd, _ = o.quantize_delayed(dy.numpy(), o.E5M2, self.st[2])
        dh = o.dequantize(qd, o.E5M2, o.GRAN_TENSOR, sd)
        return torch.from_numpy(o.gemm_ref(dh, self.wh.T)), torch.from_numpy(o.gemm_ref(dh.T, self.xh.T))

    def recorded_amax(self):
        return torch.tensor([s[0] for s in self.st], dtype=torch.float32)

    def set_recorded_amax(self, a):
        for s, v in zip(self.st, a.numpy()):
            s[0] = v

    def update_scale(self):
        for s, f in zip(self.st, self.fmts):
            self.o.update_scale(s, f)

    def state_bytes(self):
        return np.concatenate(self.st).tobytes()


def _inputs(step):
    g = torch.Generator().manual_seed(10 + step)
    x = (torch.randn((M, K), generator=g) * (1.0 + step)).to(torch.bfloat16).float()
    dy = (torch.randn((M, N), generator=g) * 1e-3 * (40.0 if step == 2 else 1.0)).to(torch.bfloat16).float()
    return x, dy


def _weights():
    g = torch.Generator().manual_seed(3)
    w = (torch.randn((N, K), generator=g) * 0.02)
    w[N - 5, 7] = 0.5            # one rank's shard has a much larger amax
    return w.to(torch.bfloat16).float()


def _worker(rank, ws, port, sync, out):
    try:
        _work(rank, ws, port, sync, out)
    except BaseException as e:          # report instead of leaving the parent waiting
        import traceback
        out.put((rank, "error: " + "".join(traceback.format_exception(e))))
        raise


def _work(rank, ws, port, sync, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    from scaled_quantize_gemm_gb300 import tp
    dist.init_process_group("gloo", rank=rank, world_size=ws, timeout=__import__("datetime").timedelta(seconds=60))
    try:
        w = _weights()
        ops = OracleOps(H)
        layer = tp.ColumnParallelFP8Linear(tp.shard_rows(w, rank, ws), M, history_len=H, ops=ops)
        other = OracleOps(H)            # an independent linear for the overlap window
        rec = []
        for step in range(STEPS):
            x, dy = _inputs(step)
            handle = layer.forward_async(x)
            independent = other.forward(x, w[:16])        # runs while the gather is in flight
            y = handle.wait().clone()
            dx, dw = layer.backward(dy)
            if sync:
                layer.end_step()
            else:
                ops.update_scale()                         # the planted omission
            rec.append((y.numpy(), dx.numpy(), dw.numpy(), ops.state_bytes(), independent.shape))
        out.put((rank, rec))
    finally:
        dist.destroy_process_group()


def _unsharded():
    w = _weights()
    ops = OracleOps(H)
    rec = []
    for step in range(STEPS):
        x, dy = _inputs(step)
        y = ops.forward(x, w)
        dx, dw = ops.backward(dy)
        ops.update_scale()
        rec.append((y.numpy(), dx.numpy(), dw.numpy(), ops.state_bytes()))
    return rec


def _run(sync):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    procs = [ctx.Process(target=_worker, args=(r, 2, port, sync, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(2):
        rank, rec = out.get(timeout=180)
        assert not isinstance(rec, str), rec
        res[rank] = rec
    for p in procs:
        p.join(60)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    return res


def _close(a, b):
    scale = max(np.max(np.abs(b)), 1e-300)
    return np.max(np.abs(a - b)) <= 1e-12 * scale


def test_column_parallel_matches_unsharded_layer():
    res = _run(sync=True)
    ref = _unsharded()
    half = N // 2
    for step in range(STEPS):
        y_r, dx_r, dw_r, st_r = ref[step]
        for rank in range(2):
            y, dx, dw, st, ind = res[rank][step]
            assert ind == (M, 16)
            assert st == st_r, (step, rank)                       # states bit-identical to the unsharded layer
            assert _close(y, y_r), (step, rank)                   # the gathered output
            assert _close(dx, dx_r), (step, rank)                 # the summed input gradient
            assert _close(dw, dw_r[rank * half:(rank + 1) * half]), (step, rank)


def test_without_amax_allreduce_the_states_diverge():
    res = _run(sync=False)
    ref = _unsharded()
    # after the first update the shard without the large weight holds a
    # different W multiplier from the unsharded layer
    assert res[0][0][3] != ref[0][3] or res[1][0][3] != ref[0][3]
    assert res[0][0][3] != res[1][0][3]


def test_shard_helpers():
    sys.path.insert(0, ROOT)
    from scaled_quantize_gemm_gb300 import tp
    w = torch.arange(24, dtype=torch.float32).reshape(6, 4)
    assert torch.equal(torch.cat([tp.shard_rows(w, r, 3) for r in range(3)]), w)
    t = torch.arange(24, dtype=torch.float32).reshape(4, 6)
    assert torch.equal(torch.cat([tp.shard_cols(t, r, 2) for r in range(2)], dim=1), t)
    parts = torch.stack([tp.shard_cols(t, r, 3) for r in range(3)])
    assert torch.equal(tp.GatherHandle(None, parts, 4, 6).wait(), t)


# ---------------------------------------------------------------- row-parallel
def _row_inputs(step):
    g = torch.Generator().manual_seed(50 + step)
    x = (torch.randn((M, N), generator=g) * (1.0 + step)).to(torch.bfloat16).float()   # the layer's K = N here
    x[5, N - 3] = 40.0 * (1.0 + step)                 # the second rank's shard of x holds the largest entry
    dy = (torch.randn((M, K), generator=g) * 1e-3).to(torch.bfloat16).float()
    return x, dy


def _row_weights():
    g = torch.Generator().manual_seed(4)
    w = (torch.randn((K, N), generator=g) * 0.02)
    w[3, 2] = 0.7                                     # the first rank's shard of W holds the largest entry
    return w.to(torch.bfloat16).float()


def _row_worker(rank, ws, port, sync, out):
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        sys.path.insert(0, ROOT)
        from scaled_quantize_gemm_gb300 import tp
        dist.init_process_group("gloo", rank=rank, world_size=ws, timeout=__import__("datetime").timedelta(seconds=60))
        try:
            w = _row_weights()
            ops = OracleOps(H)
            layer = tp.RowParallelFP8Linear(tp.shard_cols(w, rank, ws), M, history_len=H, ops=ops)
            rec = []
            for step in range(STEPS):
                x, dy = _row_inputs(step)
                work, y = layer.forward(tp.shard_cols(x, rank, ws), async_op=True)
                work.wait()
                dx, dw = layer.backward(dy)
                if sync:
                    layer.end_step()
                else:
                    ops.update_scale()
                rec.append((y.numpy().copy(), dx.numpy(), dw.numpy(), ops.state_bytes()))
            out.put((rank, rec))
        finally:
            dist.destroy_process_group()
    except BaseException as e:
        import traceback
        out.put((rank, "error: " + "".join(traceback.format_exception(e))))
        raise


def _row_run(sync):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    procs = [ctx.Process(target=_row_worker, args=(r, 2, port, sync, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(2):
        rank, rec = out.get(timeout=180)
        assert not isinstance(rec, str), rec
        res[rank] = rec
    for p in procs:
        p.join(60)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    return res


def _row_unsharded():
    w = _row_weights()
    ops = OracleOps(H)
    rec = []
    for step in range(STEPS):
        x, dy = _row_inputs(step)
        y = ops.forward(x, w)
        dx, dw = ops.backward(dy)
        ops.update_scale()
        rec.append((y.numpy(), dx.numpy(), dw.numpy(), ops.state_bytes()))
    return rec


def test_row_parallel_matches_unsharded_layer():
    """Row-parallel (W [K_out][N] sharded along its input dimension, x
    sharded the same way): the all-reduced output, each rank's input- and
    weight-gradient columns, and the delayed-scaling states (bit-identical
    to the unsharded layer's, through the amax all-reduce)."""
    res = _row_run(sync=True)
    ref = _row_unsharded()
    half = N // 2
    for step in range(STEPS):
        y_r, dx_r, dw_r, st_r = ref[step]
        for rank in range(2):
            y, dx, dw, st = res[rank][step]
            assert st == st_r, (step, rank)
            assert _close(y, y_r), (step, rank)
            assert _close(dx, dx_r[:, rank * half:(rank + 1) * half]), (step, rank)
            assert _close(dw, dw_r[:, rank * half:(rank + 1) * half]), (step, rank)


def test_row_parallel_without_amax_allreduce_diverges():
    res = _row_run(sync=False)
    ref = _row_unsharded()
    assert res[0][0][3] != res[1][0][3]
    assert res[0][0][3] != ref[0][3] or res[1][0][3] != ref[0][3]


# ---------------------------------------------------------------- data-parallel
def _dp_worker(rank, ws, port, sync, out):
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        sys.path.insert(0, ROOT)
        from scaled_quantize_gemm_gb300 import tp
        dist.init_process_group("gloo", rank=rank, world_size=ws, timeout=__import__("datetime").timedelta(seconds=60))
        try:
            w = _weights()
            ops = OracleOps(H)
            layer = tp.DataParallelFP8Linear(w, M // ws, history_len=H, ops=ops)
            rows = slice(rank * (M // ws), (rank + 1) * (M // ws))
            rec = []
            for step in range(STEPS):
                x, dy = _inputs(step)
                if step == 1:
                    x[M - 2, 9] = 300.0                   # only the second rank's rows hold this spike
                y = layer.forward(x[rows].contiguous())
                dx, dw, work = layer.backward(dy[rows].contiguous(), async_op=True)
                work.wait()
                if sync:
                    layer.end_step()
                else:
                    ops.update_scale()
                rec.append((y.numpy(), dx.numpy(), dw.numpy().copy(), ops.state_bytes()))
            out.put((rank, rec))
        finally:
            dist.destroy_process_group()
    except BaseException as e:
        import traceback
        out.put((rank, "error: " + "".join(traceback.format_exception(e))))
        raise


def _dp_run(sync):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    procs = [ctx.Process(target=_dp_worker, args=(r, 2, port, sync, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(2):
        rank, rec = out.get(timeout=180)
        assert not isinstance(rec, str), rec
        res[rank] = rec
    for p in procs:
        p.join(60)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    return res


def _dp_unsharded():
    w = _weights()
    ops = OracleOps(H)
    rec = []
    for step in range(STEPS):
        x, dy = _inputs(step)
        if step == 1:
            x[M - 2, 9] = 300.0
        y = ops.forward(x, w)
        dx, dw = ops.backward(dy)
        ops.update_scale()
        rec.append((y.numpy(), dx.numpy(), dw.numpy(), ops.state_bytes()))
    return rec


def test_data_parallel_matches_unsharded_layer():
    """Data-parallel (W replicated, batch rows sharded): each rank's output
    and input-gradient rows, the all-reduced weight gradient, and the
    states bit-identical to the full-batch layer's through the amax
    all-reduce (a spike in the second rank's rows moves the x history)."""
    res = _dp_run(sync=True)
    ref = _dp_unsharded()
    half = M // 2
    for step in range(STEPS):
        y_r, dx_r, dw_r, st_r = ref[step]
        for rank in range(2):
            y, dx, dw, st = res[rank][step]
            assert st == st_r, (step, rank)
            assert _close(y, y_r[rank * half:(rank + 1) * half]), (step, rank)
            assert _close(dx, dx_r[rank * half:(rank + 1) * half]), (step, rank)
            assert _close(dw, dw_r), (step, rank)


def test_data_parallel_without_amax_allreduce_diverges():
    res = _dp_run(sync=False)
    assert res[0][1][3] != res[1][1][3]


# ---------------------------------------------------------------- data-parallel, fine-grained recipes
class OracleFineOps:
    """The per-rank operations of a data-parallel linear under a
    fine-grained recipe on the CPU oracle (current scaling per unit, float64
    products of the dequantised operands); no delayed state."""

    def __init__(self, gran):
        import oracle as o
        self.o, self.gran = o, gran

    def forward(self, x, w):
        self.st, r = self.o.linear_fine_fwd(x.numpy(), w.numpy(), self.gran)
        return torch.from_numpy(r)

    def forward_partial(self, x, w):
        return self.forward(x, w)

    def backward(self, dy):
        dX, dW = self.o.linear_fine_bwd(self.st, dy.numpy(), self.gran, self.o.E5M2)
        return torch.from_numpy(dX), torch.from_numpy(dW)

    def recorded_amax(self):
        return torch.zeros(0, dtype=torch.float32)

    def set_recorded_amax(self, a):
        pass

    def update_scale(self):
        pass


FM, FK, FN = 256, 384, 256      # fine-grained units need multiples of 128 (128 batch rows per rank)


def _fine_inputs(step):
    g = torch.Generator().manual_seed(50 + step)
    x = (torch.randn((FM, FK), generator=g) * (1.0 + step)).to(torch.bfloat16).float()
    x[FM - 3, 17] = 90.0 * (step + 1)            # an outlier in the second rank's rows
    dy = (torch.randn((FM, FN), generator=g) * 1e-3).to(torch.bfloat16).float()
    w = (torch.randn((FN, FK), generator=torch.Generator().manual_seed(51)) * 0.02).to(torch.bfloat16).float()
    return x, w, dy


def _fine_dp_worker(rank, ws, port, gran, out):
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        sys.path.insert(0, ROOT)
        from scaled_quantize_gemm_gb300 import tp
        dist.init_process_group("gloo", rank=rank, world_size=ws, timeout=__import__("datetime").timedelta(seconds=60))
        try:
            rows = slice(rank * (FM // ws), (rank + 1) * (FM // ws))
            rec = []
            for step in range(2):
                x, w, dy = _fine_inputs(step)
                layer = tp.DataParallelFP8Linear(w, FM // ws, ops=OracleFineOps(gran))
                y = layer.forward(x[rows].contiguous())
                dx, dw = layer.backward(dy[rows].contiguous())
                layer.end_step()
                rec.append((y.numpy(), dx.numpy(), dw.numpy().copy()))
            out.put((rank, rec))
        finally:
            dist.destroy_process_group()
    except BaseException as e:
        import traceback
        out.put((rank, "error: " + "".join(traceback.format_exception(e))))
        raise


@pytest.mark.parametrize("gran_name", ["GRAN_TILE_1x128", "GRAN_TILE_POW2", "GRAN_MX32"])
def test_data_parallel_fine_grained_matches_full_batch(gran_name):
    """Data-parallel under the fine-grained recipes: each rank's output and
    input-gradient rows and the summed weight gradient equal the full-batch
    layer's (every quantisation unit lies inside one rank's rows or is the
    same on every rank, so the codes and scales are the full batch's)."""
    import oracle as o
    gran = getattr(o, gran_name)
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    procs = [ctx.Process(target=_fine_dp_worker, args=(r, 2, port, gran, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(2):
        rank, rec = out.get(timeout=180)
        assert not isinstance(rec, str), rec
        res[rank] = rec
    for p in procs:
        p.join(60)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    half = FM // 2
    for step in range(2):
        x, w, dy = _fine_inputs(step)
        st, Y = o.linear_fine_fwd(x.numpy(), w.numpy(), gran)
        dX, dW = o.linear_fine_bwd(st, dy.numpy(), gran, o.E5M2)
        for rank in range(2):
            y, dx, dw = res[rank][step]
            assert np.array_equal(y, Y[rank * half:(rank + 1) * half]), (step, rank)
            assert np.array_equal(dx, dX[rank * half:(rank + 1) * half]), (step, rank)
            assert _close(dw, dW), (step, rank)


# ---------------------------------------------------------------- row-parallel, fine-grained recipes
RM, RK, RN = 128, 512, 256      # each rank's K/P = 256 columns: whole 1x128 tiles and 128x128 blocks


def _fine_row_inputs(step):
    g = torch.Generator().manual_seed(70 + step)
    x = (torch.randn((RM, RK), generator=g) * (1.0 + step)).to(torch.bfloat16).float()
    x[9, RK - 5] = 70.0 * (step + 1)             # an outlier in the second rank's columns
    dy = (torch.randn((RM, RN), generator=g) * 1e-3).to(torch.bfloat16).float()
    w = (torch.randn((RN, RK), generator=torch.Generator().manual_seed(71)) * 0.02).to(torch.bfloat16).float()
    return x, w, dy


def _fine_row_worker(rank, ws, port, gran, out):
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        sys.path.insert(0, ROOT)
        from scaled_quantize_gemm_gb300 import tp
        dist.init_process_group("gloo", rank=rank, world_size=ws, timeout=__import__("datetime").timedelta(seconds=60))
        try:
            rec = []
            for step in range(2):
                x, w, dy = _fine_row_inputs(step)
                layer = tp.RowParallelFP8Linear(tp.shard_cols(w, rank, ws), RM, ops=OracleFineOps(gran))
                y = layer.forward(tp.shard_cols(x, rank, ws))
                dx, dw = layer.backward(dy)
                layer.end_step()
                rec.append((y.numpy().copy(), dx.numpy(), dw.numpy()))
            out.put((rank, rec))
        finally:
            dist.destroy_process_group()
    except BaseException as e:
        import traceback
        out.put((rank, "error: " + "".join(traceback.format_exception(e))))
        raise


@pytest.mark.parametrize("gran_name", ["GRAN_TILE_1x128", "GRAN_TILE_POW2", "GRAN_MX32"])
def test_row_parallel_fine_grained_matches_full_layer(gran_name):
    """Row-parallel under the fine-grained recipes with K/P a multiple of
    128: the summed partial outputs equal the full layer's output up to the
    order of the sum over K, and each rank's input- and weight-gradient
    columns equal the full layer's exactly (the contraction of dgrad runs
    over N and that of wgrad over M, neither sharded; every unit of x and W
    lies inside one rank's columns and dy is the same on every rank)."""
    import oracle as o
    gran = getattr(o, gran_name)
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    procs = [ctx.Process(target=_fine_row_worker, args=(r, 2, port, gran, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(2):
        rank, rec = out.get(timeout=180)
        assert not isinstance(rec, str), rec
        res[rank] = rec
    for p in procs:
        p.join(60)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    half = RK // 2
    for step in range(2):
        x, w, dy = _fine_row_inputs(step)
        st, Y = o.linear_fine_fwd(x.numpy(), w.numpy(), gran)
        dX, dW = o.linear_fine_bwd(st, dy.numpy(), gran, o.E5M2)
        for rank in range(2):
            y, dx, dw = res[rank][step]
            assert _close(y, Y), (step, rank)
            assert np.array_equal(dx, dX[:, rank * half:(rank + 1) * half]), (step, rank)
            assert np.array_equal(dw, dW[:, rank * half:(rank + 1) * half]), (step, rank)
