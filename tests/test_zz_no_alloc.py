"""fp8_linear_fwd_noalloc -- the forward FP8 linear for callers that cannot
allocate device memory (a framework that owns every byte through its own pool,
or a plugin that must not call cudaMalloc because it can synchronise the
device).  Its scratch is the library's static 32 MiB device array instead of a
workspace.

Called twice in a row through the C ABI.  Each output must be bit-identical
to the workspace-based fp8_linear_fwd (current per-tensor scaling, same
inputs: the same casts and the same GEMM), and within the GEMM tolerance of
the oracle's product of its own current-scaled codes.  The first call draws x
with std 8 and the second with std 1 at a larger shape: the per-tensor amax is
a max-reduction, so an amax slot left over from the first call in the shared
array would raise the second call's scale and change its codes, which both
comparisons would catch.
"""
import numpy as np
import pytest
import torch

import oracle as o
import scaled_quantize_gemm_gb300 as sq
from scaled_quantize_gemm_gb300 import workloads as wl

from _helpers import assert_gemm_close, np32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _workspace_entry(x, w, out_dtype, bias=None):
    M, K = x.shape
    N = w.shape[0]
    ws = torch.empty(sq.fp8_linear_workspace_bytes(M, N, K), dtype=torch.uint8, device=DEV)
    y = torch.empty((M, N), dtype=out_dtype, device=DEV)
    sq.fp8_linear_fwd(x, w, y, ws, bias=bias)
    return y


def _oracle(x, w, bias=None):
    qx, _, sx, _ = o.quantize_tensor_current(np32(x), o.E4M3)
    qw, _, sw, _ = o.quantize_tensor_current(np32(w), o.E4M3)
    return o.gemm_ref(o.dequantize(qx, o.E4M3, o.GRAN_TENSOR, sx), o.dequantize(qw, o.E4M3, o.GRAN_TENSOR, sw),
                      bias=None if bias is None else bias.cpu().numpy())


def test_noalloc_matches_workspace_entry_on_two_calls():
    # large amax first, then a smaller amax at a larger shape
    cases = [((256, 512, 384), 8.0, torch.float32, True), ((512, 768, 1024), 1.0, torch.bfloat16, False)]
    for i, ((M, K, N), std, out, with_bias) in enumerate(cases):
        x = wl.normal((M, K), std, 500 + i).to(DEV)
        w = wl.normal((N, K), 0.02, 600 + i).to(DEV)
        bias = wl.normal((N,), 1.0, 700 + i, dtype=torch.float32).to(DEV) if with_bias else None
        y = torch.empty((M, N), dtype=out, device=DEV)
        sq.fp8_linear_fwd_noalloc(x, w, y, bias=bias)
        ref = _workspace_entry(x, w, out, bias=bias)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.uint8 if out == torch.bfloat16 else torch.int32),
                           ref.view(torch.uint8 if out == torch.bfloat16 else torch.int32)), f"call {i}"
        assert_gemm_close(y, _oracle(x, w, bias))
    assert sq.fp8_device_status(True) == 0


def test_noalloc_rejects_sizes_beyond_the_scratch():
    M, K, N = 8192, 4096, 16
    x = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    w = torch.empty((N, K), dtype=torch.bfloat16, device=DEV)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(sq.Fp8Error) as e:
        sq.fp8_linear_fwd_noalloc(x, w, y)
    assert e.value.code == sq.ERR_UNSUPPORTED
    assert "static scratch holds" in str(e.value)
