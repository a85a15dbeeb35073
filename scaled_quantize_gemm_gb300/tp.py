"""Tensor-parallel column-parallel FP8 linear ("Transformer Scaling",
Part 03 and "04 · Put it back into code -- Program model": each TP rank
computes a local linear, launches an all-gather of its output asynchronously,
runs independent work in the window, and waits at the first consumer of the
gathered result).

W [N][K] is sharded along N: rank r owns rows [r N/P, (r+1) N/P).  Per step,
with per-tensor delayed scaling under the HYBRID recipe:

  forward   y_r = x W_r^T          (x replicated; the rank's own FP8 GEMM on
                                    local operands only)
            y   = all-gather_r(y_r) (asynchronous; a handle is returned)
  backward  dx  = sum_r dy_r W_r    (dy_r = the rank's N-columns of dy; the
                                    partial products are all-reduced, summed)
            dW_r = dy_r^T x         (local, no exchange)
  step end  the amax just recorded in each state's history slot 0 is
            all-reduced (max) before the scale update, so every rank's
            x, W and dy states stay bit-identical, and equal to the states of
            the unsharded layer (the amax of a sharded tensor is the max of
            its shards' amaxes).

Row-parallel (RowParallelFP8Linear), the partner of a column-parallel
layer: W [N][K] sharded along K, rank r owning columns [r K/P, (r+1) K/P),
and the input arriving sharded the same way (the column-parallel layer's
output columns):

  forward   y = sum_r x_r W_r^T   (each rank's product in fp32, then one
                                   all-reduce (sum) of the partial outputs)
  backward  dx_r = dy W_r         (dy replicated; local, no exchange)
            dW_r = dy^T x_r       (local)
  step end  the same amax all-reduce (max) as above: x_r and W_r are shards
            of x and W, and dy is the same on every rank.

Data-parallel (DataParallelFP8Linear): W replicated, the batch sharded along
M (rank r owns rows [r M/P, (r+1) M/P) of x and dy):

  forward   y_r = x_r W^T         (local)
  backward  dx_r = dy_r W         (local)
            dW = sum_r dy_r^T x_r (the local products all-reduced, sum)
  step end  the amax all-reduce (max): x and dy are sharded, W identical.

The data-parallel and row-parallel linears also run the fine-grained
recipes (FineOps:
current scaling per 1x128 tile / 128x128 block, with fp32 or power-of-two
scales, or per MX-32 block).  Every unit lies inside one rank's rows (1x128
tiles and MX blocks along a row; wgrad's 128-row column tiles and 32-row
column blocks inside the rank's M_local rows, a multiple of 128) or is the
same on every rank (W's blocks), so each rank computes exactly the scales and
codes of the full-batch layer and there is no amax to exchange; dW is summed
as above.  Row-parallel likewise, with K/P a multiple of 128 (x's tiles and
W's blocks inside one rank's columns, dy the same everywhere); the fp32
partial outputs are summed as above.

The exchange steps are torch.distributed collectives on the given process
group; the arithmetic of each rank runs in `ops`.  The default `ops`
(LibraryOps) is this library's CUDA path through the C ABI; a caller may
pass another implementation of the same five methods (the tests drive the
orchestration on CPU ranks this way).
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def shard_rows(w: torch.Tensor, rank: int, world: int) -> torch.Tensor:
    """Rows [rank N/P, (rank+1) N/P) of w [N][K] (N % P == 0), contiguous."""
    n = w.shape[0]
    if n % world:
        raise ValueError(f"N = {n} is not divisible by the tensor-parallel size {world}")
    step = n // world
    return w[rank * step:(rank + 1) * step].contiguous()


def shard_cols(t: torch.Tensor, rank: int, world: int) -> torch.Tensor:
    """Columns [rank N/P, (rank+1) N/P) of t [M][N], contiguous (the rank's
    part of the output gradient of a column-parallel linear)."""
    n = t.shape[1]
    if n % world:
        raise ValueError(f"N = {n} is not divisible by the tensor-parallel size {world}")
    step = n // world
    return t[:, rank * step:(rank + 1) * step].contiguous()


class GatherHandle:
    """An all-gather in flight: `wait()` blocks (on the host for CPU
    collectives, on the current stream for device ones) until the gathered
    output may be read, and returns it as y [M][N]."""

    def __init__(self, work, parts: torch.Tensor, M: int, N: int):
        self._work = work
        self._parts = parts          # [P][M][N/P], rank-major
        self._M, self._N = M, N
        self._out = None

    def wait(self) -> torch.Tensor:
        if self._out is None:
            if self._work is not None:
                self._work.wait()
            # rank-major [P][M][N/P] -> [M][N]: rank r's block is columns [r N/P, (r+1) N/P)
            self._out = self._parts.permute(1, 0, 2).reshape(self._M, self._N)
        return self._out


class LibraryOps:
    """Per-rank arithmetic on this library's CUDA path: per-tensor delayed
    casts and FP8 GEMMs through the C ABI (the backward reads the codes
    MN-major), states in one device block of three (x, W, dy)."""

    def __init__(self, M: int, N_local: int, K: int, history_len: int, device, recipe_e4m3: bool = False):
        import scaled_quantize_gemm_gb300 as sq
        self.sq = sq
        self.H = history_len
        self.M, self.N, self.K = M, N_local, K
        u8 = dict(dtype=torch.uint8, device=device)
        self.qx = torch.empty((M, K), **u8)
        self.qw = torch.empty((N_local, K), **u8)
        self.qdy = torch.empty((M, N_local), **u8)
        self.states = torch.empty(3 * (history_len + 2), dtype=torch.float32, device=device)
        sq.fp8_scale_init(self.states, 3, history_len)
        self.dy_fmt = sq.E4M3 if recipe_e4m3 else sq.E5M2
        self.formats = [sq.E4M3, sq.E4M3, self.dy_fmt]

    def _st(self, i):
        return self.states[i * (self.H + 2):(i + 1) * (self.H + 2)]

    def _s(self, i):
        j = i * (self.H + 2) + self.H + 1
        return self.states[j:j + 1]

    def forward(self, x: torch.Tensor, w_local: torch.Tensor, out_dtype=torch.bfloat16) -> torch.Tensor:
        sq, H = self.sq, self.H
        sq.fp8_quantize(x, sq.E4M3, sq.TENSOR, self.qx, delayed_state=self._st(0), history_len=H)
        sq.fp8_quantize(w_local, sq.E4M3, sq.TENSOR, self.qw, delayed_state=self._st(1), history_len=H)
        y = torch.empty((self.M, self.N), dtype=out_dtype, device=x.device)
        sq.fp8_gemm(self.qx, sq.E4M3, self._s(0), sq.TENSOR, self.qw, sq.E4M3, self._s(1), sq.TENSOR, y)
        return y

    def forward_partial(self, x_local: torch.Tensor, w_local: torch.Tensor) -> torch.Tensor:
        """The rank's partial output of a row-parallel linear, fp32 (summed
        across the group afterwards)."""
        return self.forward(x_local, w_local, out_dtype=torch.float32)

    def backward(self, dy_local: torch.Tensor):
        """-> (dx partial fp32 [M][K], dW_local fp32 [N/P][K])"""
        sq, H = self.sq, self.H
        sq.fp8_quantize(dy_local, self.dy_fmt, sq.TENSOR, self.qdy, delayed_state=self._st(2), history_len=H)
        dx = torch.empty((self.M, self.K), dtype=torch.float32, device=dy_local.device)
        dw = torch.empty((self.N, self.K), dtype=torch.float32, device=dy_local.device)
        # the forward's codes as they are: W and (for wgrad) dy and x MN-major
        sq.fp8_gemm_layout(self.qdy, self.dy_fmt, self._s(2), sq.K_MAJOR, self.qw, sq.E4M3, self._s(1), sq.MN_MAJOR,
                           dx, self.M, self.K, self.N)
        sq.fp8_gemm_layout(self.qdy, self.dy_fmt, self._s(2), sq.MN_MAJOR, self.qx, sq.E4M3, self._s(0), sq.MN_MAJOR,
                           dw, self.N, self.K, self.M)
        return dx, dw

    def recorded_amax(self) -> torch.Tensor:
        """history slot 0 of the x, W and dy states (3 floats, a copy)"""
        H = self.H
        return self.states[0::H + 2][:3].clone()

    def set_recorded_amax(self, a: torch.Tensor) -> None:
        H = self.H
        self.states[0::H + 2][:3].copy_(a)

    def update_scale(self) -> None:
        self.sq.fp8_update_scale(self.states, 3, self.H, self.formats)


class FineOps:
    """Per-rank arithmetic of a data-parallel linear under a fine-grained
    recipe (gran TILE_1x128, TILE_1x128_POW2 or MX32; current scaling per
    unit) through fp8_linear_fwd / fp8_linear_bwd: y and dx bf16, dW fp32.
    There is no delayed state, so nothing is recorded or exchanged at the
    step's end."""

    def __init__(self, M: int, N: int, K: int, gran: int, device, recipe_e4m3: bool = False):
        import scaled_quantize_gemm_gb300 as sq
        self.sq = sq
        self.M, self.N, self.K, self.gran = M, N, K, gran
        self.recipe = sq.RECIPE_E4M3 if recipe_e4m3 else sq.RECIPE_HYBRID
        nbytes = sq.fp8_linear_workspace_bytes(M, N, K, gran)
        if nbytes == 0:
            raise ValueError(f"granularity {gran} is not a linear-layer recipe")
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=device)

    def forward(self, x: torch.Tensor, w: torch.Tensor, out_dtype=torch.bfloat16) -> torch.Tensor:
        y = torch.empty((self.M, self.N), dtype=out_dtype, device=x.device)
        self.sq.fp8_linear_fwd(x, w, y, self.ws, gran=self.gran, recipe=self.recipe)
        return y

    def forward_partial(self, x_local: torch.Tensor, w_local: torch.Tensor) -> torch.Tensor:
        """The rank's partial output of a row-parallel linear, fp32 (summed
        across the group afterwards)."""
        return self.forward(x_local, w_local, out_dtype=torch.float32)

    def backward(self, dy: torch.Tensor):
        """-> (dx bf16 [M][K], dW fp32 [N][K])"""
        dx = torch.empty((self.M, self.K), dtype=torch.bfloat16, device=dy.device)
        dw = torch.empty((self.N, self.K), dtype=torch.float32, device=dy.device)
        self.sq.fp8_linear_bwd(dy, dx, dw, self.ws, self.K, gran=self.gran, recipe=self.recipe)
        return dx, dw

    def recorded_amax(self) -> torch.Tensor:
        return torch.zeros(0, dtype=torch.float32, device=self.ws.device)

    def set_recorded_amax(self, a: torch.Tensor) -> None:
        pass

    def update_scale(self) -> None:
        pass


class ColumnParallelFP8Linear:
    """One column-parallel FP8 linear of a TP group (see the module text).

    w_local: this rank's rows of W ([N/P][K]).  `ops` defaults to LibraryOps
    on w_local's device."""

    def __init__(self, w_local: torch.Tensor, M: int, history_len: int = 16, group=None, ops=None,
                 recipe_e4m3: bool = False):
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.w = w_local
        self.M = M
        self.N_local, self.K = w_local.shape
        self.N = self.N_local * self.world
        self.ops = ops if ops is not None else LibraryOps(M, self.N_local, self.K, history_len, w_local.device,
                                                          recipe_e4m3)

    def forward_async(self, x: torch.Tensor) -> GatherHandle:
        """Local linear, then an asynchronous all-gather of its output along
        N; run independent work before calling wait() on the handle."""
        y_local = self.ops.forward(x, self.w)
        # rank-major concatenation along the first dimension: [P M][N/P]
        parts = torch.empty((self.world * self.M, self.N_local), dtype=y_local.dtype, device=y_local.device)
        work = dist.all_gather_into_tensor(parts, y_local.contiguous(), group=self.group, async_op=True)
        return GatherHandle(work, parts.view(self.world, self.M, self.N_local), self.M, self.N)

    def backward(self, dy: torch.Tensor):
        """dy: the full output gradient [M][N] (replicated) or this rank's
        columns [M][N/P].  Returns (dx fp32 [M][K], summed over the group;
        dW_local fp32 [N/P][K])."""
        dy_local = dy if dy.shape[1] == self.N_local else shard_cols(dy, self.rank, self.world)
        dx, dw = self.ops.backward(dy_local)
        dist.all_reduce(dx, op=dist.ReduceOp.SUM, group=self.group)
        return dx, dw

    def end_step(self) -> None:
        """All-reduce (max) the amaxes the step recorded, then update the
        scales: every rank ends the step with the same x, W and dy states."""
        a = self.ops.recorded_amax()
        dist.all_reduce(a, op=dist.ReduceOp.MAX, group=self.group)
        self.ops.set_recorded_amax(a)
        self.ops.update_scale()


class RowParallelFP8Linear:
    """One row-parallel FP8 linear of a TP group (see the module text).

    w_local: this rank's columns of W ([N][K/P]); the forward takes this
    rank's columns of x ([M][K/P]).  `ops` defaults to LibraryOps on
    w_local's device (its N is the full N, its K the local K/P), or FineOps
    when a fine-grained `gran` is given (K/P a multiple of 128: every 1x128
    tile of x and 128x128 block of W then lies inside one rank's columns, and
    dy's units are the same on every rank)."""

    def __init__(self, w_local: torch.Tensor, M: int, history_len: int = 16, group=None, ops=None,
                 recipe_e4m3: bool = False, gran: int = 0):
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.w = w_local
        self.M = M
        self.N, self.K_local = w_local.shape
        self.K = self.K_local * self.world
        if ops is None:
            ops = (LibraryOps(M, self.N, self.K_local, history_len, w_local.device, recipe_e4m3) if gran == 0
                   else FineOps(M, self.N, self.K_local, gran, w_local.device, recipe_e4m3))
        self.ops = ops

    def forward(self, x_local: torch.Tensor, async_op: bool = False):
        """The rank's partial product, then an all-reduce (sum) of it: y
        [M][N] fp32 on every rank.  With async_op the all-reduce is left in
        flight and (work, y) is returned; y may be read after work.wait()."""
        y = self.ops.forward_partial(x_local, self.w)
        work = dist.all_reduce(y, op=dist.ReduceOp.SUM, group=self.group, async_op=async_op)
        return (work, y) if async_op else y

    def backward(self, dy: torch.Tensor):
        """dy: the full output gradient [M][N] (the same on every rank).
        Returns (dx_local [M][K/P], fp32 under the per-tensor recipe, bf16
        under a fine-grained one; dW_local fp32 [N][K/P]); no exchange."""
        return self.ops.backward(dy)

    def end_step(self) -> None:
        """All-reduce (max) the amaxes the step recorded, then update the
        scales: every rank ends the step with the same x, W and dy states
        (a fine-grained recipe records none)."""
        a = self.ops.recorded_amax()
        if a.numel():
            dist.all_reduce(a, op=dist.ReduceOp.MAX, group=self.group)
            self.ops.set_recorded_amax(a)
        self.ops.update_scale()


class DataParallelFP8Linear:
    """One data-parallel FP8 linear (see the module text): every rank holds
    all of W [N][K] and its own M_local rows of the batch.  `ops` defaults to
    LibraryOps on w's device (its M is the local batch), or FineOps when a
    fine-grained `gran` is given."""

    def __init__(self, w: torch.Tensor, M_local: int, history_len: int = 16, group=None, ops=None,
                 recipe_e4m3: bool = False, gran: int = 0):
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.w = w
        self.N, self.K = w.shape
        if ops is None:
            ops = (LibraryOps(M_local, self.N, self.K, history_len, w.device, recipe_e4m3) if gran == 0
                   else FineOps(M_local, self.N, self.K, gran, w.device, recipe_e4m3))
        self.ops = ops

    def forward(self, x_local: torch.Tensor) -> torch.Tensor:
        """y_local [M_local][N] (bf16 on the library path); no exchange."""
        return self.ops.forward(x_local, self.w)

    def backward(self, dy_local: torch.Tensor, async_op: bool = False):
        """dx_local [M_local][K] (local) and dW [N][K] fp32 summed over the
        group.  With async_op the all-reduce of dW is left in flight and
        (dx_local, dW, work) is returned; dW may be read after work.wait()."""
        dx, dw = self.ops.backward(dy_local)
        work = dist.all_reduce(dw, op=dist.ReduceOp.SUM, group=self.group, async_op=async_op)
        return (dx, dw, work) if async_op else (dx, dw)

    def end_step(self) -> None:
        """All-reduce (max) the amaxes the step recorded, then update the
        scales: every rank ends the step with the same x, W and dy states
        (a fine-grained recipe records none)."""
        a = self.ops.recorded_amax()
        if a.numel():
            dist.all_reduce(a, op=dist.ReduceOp.MAX, group=self.group)
            self.ops.set_recorded_amax(a)
        self.ops.update_scale()
