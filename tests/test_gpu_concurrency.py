"""Concurrent callers: two host threads, each on its own stream, run the
linear layer at a size where the backward runs dgrad and wgrad side by side
(its wgrad on the calling thread's own side stream).  Every thread's
outputs must equal a single-threaded run on the same inputs bit for bit: the
per-thread side streams and the library's per-device caches keep the calls
apart, and stream order still holds from each caller's point of view."""
import threading

import pytest
import torch

import scaled_quantize_gemm_gb300 as sq
from scaled_quantize_gemm_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(x, w, dy, out, stream, reps):
    """`reps` current-scaled forward + backward calls on `stream`."""
    M, K = x.shape
    N = w.shape[0]
    ws = torch.empty(sq.fp8_linear_workspace_bytes(M, N, K), dtype=torch.uint8, device=DEV)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            sq.fp8_linear_fwd(x, w, out["y"], ws)
            sq.fp8_linear_bwd(dy, out["dx"], out["dw"], ws, K)
    stream.synchronize()


def _buffers(M, K, N):
    return {"y": torch.empty((M, N), dtype=torch.bfloat16, device=DEV),
            "dx": torch.empty((M, K), dtype=torch.bfloat16, device=DEV),
            "dw": torch.empty((N, K), dtype=torch.float32, device=DEV)}


@pytest.mark.parametrize("M,K,N", [(2048, 768, 2304), (2048, 3072, 768)])
def test_two_threads_two_streams_bit_exact(M, K, N):
    # 768 -> 2304 runs dgrad and wgrad side by side; 3072 -> 768 runs them in
    # order (the two grids do not fit on the device together)
    x = wl.normal((M, K), 1.0, 900, DEV)
    w = wl.normal((N, K), 0.02, 901, DEV)
    dy = wl.normal((M, N), 1e-3, 902, DEV)
    ref = _buffers(M, K, N)
    _run(x, w, dy, ref, torch.cuda.Stream(), 1)

    outs = [_buffers(M, K, N) for _ in range(2)]
    errors = []

    def worker(i):
        try:
            _run(x, w, dy, outs[i], torch.cuda.Stream(), 8)
        except Exception as e:   # surfaced below, in the test's own thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for out in outs:
        for k in ("y", "dx", "dw"):
            assert torch.equal(out[k], ref[k]), k
    assert sq.fp8_device_status(True) == sq.OK
