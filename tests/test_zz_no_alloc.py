"""fp8_linear_fwd_noalloc -- the forward FP8 linear for callers that cannot
allocate device memory (a framework that owns every byte through its own pool,
or a plugin that must not call cudaMalloc because it can synchronise the
device).  Its scratch is the library's static 32 MiB device array instead of a
workspace.

Called twice in a row through the C ABI; each output must match the
workspace-based fp8_linear_fwd (current per-tensor scaling, same inputs)
within the GEMM tolerance of the other tests.  The second call reuses the
array the first one left behind, so it also checks that nothing stale (the
amax slots) leaks from one call into the next.
"""
import numpy as np
import pytest
import torch

import scaled_quantize_gemm_gb300 as sq
from scaled_quantize_gemm_gb300 import workloads as wl

from _helpers import assert_gemm_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _reference(x, w, out_dtype, bias=None):
    M, K = x.shape
    N = w.shape[0]
    ws = torch.empty(sq.fp8_linear_workspace_bytes(M, N, K), dtype=torch.uint8, device=DEV)
    y = torch.empty((M, N), dtype=out_dtype, device=DEV)
    sq.fp8_linear_fwd(x, w, y, ws, bias=bias)
    return y


def test_noalloc_matches_workspace_entry_on_two_calls():
    # second call: larger amax than the first, then smaller shapes: a stale
    # amax left in the shared array would change the second call's scales
    cases = [((512, 768, 1024), 1.0, torch.bfloat16), ((256, 512, 384), 8.0, torch.float32)]
    for i, ((M, K, N), std, out) in enumerate(cases):
        x = wl.normal((M, K), std, 500 + i).to(DEV)
        w = wl.normal((N, K), 0.02, 600 + i).to(DEV)
        bias = torch.randn(N, generator=torch.Generator().manual_seed(i)).to(DEV) if i == 1 else None
        y = torch.empty((M, N), dtype=out, device=DEV)
        sq.fp8_linear_fwd_noalloc(x, w, y, bias=bias)
        ref = _reference(x, w, out, bias=bias)
        torch.cuda.synchronize()
        assert_gemm_close(y, ref.double().cpu().numpy())
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
