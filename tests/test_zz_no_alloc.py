"""The workspace-free GEMV entry point, for callers that cannot allocate device memory
(plugins whose host runtime owns all GPU memory, or paths that cannot afford cudaMalloc's
implicit synchronisation).  Its scratch is a fixed array inside the library shared by all
calls, so two calls in a row must both match the workspace entry point, and the second
must not see state left by the first.  Both entry points run the same kernel with the same
plan, so their outputs agree bit for bit.  Collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import dev_bf16, qlib, to_f64

pytestmark = pytest.mark.gpu


def _plan_mode(n):
    """The GEMV's work split for n rows on this GPU (the host planner's rule): 'whole' (one
    row tile per CTA), 'cluster' (few row tiles, split over clusters) or 'stream-k' (tiles
    split across CTAs, finished through the tickets and partial sums of the scratch)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nt = (n + 127) // 128
    if nt < sms and nt * 8 >= sms * 7:
        return "whole"
    if nt * 2 <= sms:
        return "cluster"
    return "stream-k"


@pytest.mark.parametrize("fmt,n,k,m,residual", [
    (wl.NVFP4, 1000, 1280, 3, True),
    (wl.Q6K, 640, 1536, 1, False),
    (wl.MXFP4, 17408 // 8, 5120, 4, True),
    # more row tiles than SMs: stream-K, whose split tiles use the array's tickets and
    # partial-sum region
    (wl.NVFP4, 32768, 512, 4, True),
    (wl.Q6K, 170 * 128 - 5, 512, 2, False),
])
def test_static_workspace_matches_workspace_entry_on_two_calls(fmt, n, k, m, residual):
    q = qlib()
    w = wl.weight(fmt, n, k, seed=41)
    pw = q.PackedWeight.from_logical(w)
    stream = torch.cuda.current_stream().cuda_stream
    if n >= 20000:
        assert _plan_mode(n) == "stream-k"
    rows = np.unique(np.concatenate([np.arange(0, n, max(1, n // 700)), [n - 1]]))
    assert q.qgemv_static_ws_status(stream) == 0  # a clean start (or a previous call's clean end)
    for call in range(2):
        x = wl.activations(m, k, seed=50 + call)
        res = wl.activations(m, n, seed=60 + call, stream="residual") if residual else None
        xt = dev_bf16(x)
        rt = dev_bf16(res) if residual else None
        ref = q.gemv(pw, xt, rt)  # the existing entry point, own workspace
        out = torch.empty((m, (n + 7) // 8 * 8), dtype=torch.bfloat16, device="cuda")[:, :n]
        out.fill_(float("nan"))
        q.qgemv_static_ws(pw.desc, xt.data_ptr(), m, xt.stride(0), None if rt is None else rt.data_ptr(),
                          0 if rt is None else rt.stride(0), out.data_ptr(), out.stride(0), stream)
        torch.cuda.synchronize()
        assert q.qgemv_static_ws_status(stream) == 0
        got, want = to_f64(out), to_f64(ref)
        assert np.all(np.isfinite(got))
        assert np.array_equal(got, want), f"call {call}: {np.count_nonzero(got != want)} outputs differ"
        ref_o, _ = oracle.gemv_rows(w, x, rows, res)
        tol = oracle.tolerance(w, x, res, rows=rows, ref=ref_o)
        assert np.all(np.abs(got[:, rows] - ref_o) <= tol)


def test_static_workspace_validates_on_host():
    q = qlib()
    w = q.qg_weight(wl.NVFP4, 0, 256, 100, 0x1000, 0x2000, None, 1.0, 0.0)  # K not a multiple of 16
    assert q.lib().qgemv_static_ws(ctypes.byref(w), 0x3000, 1, 256, None, 0, 0x4000, 256, None) == 1
    w = q.qg_weight(wl.NVFP4, 0, 256, 256, 0x1000, 0x2000, None, 1.0, 0.0)
    assert q.lib().qgemv_static_ws(ctypes.byref(w), 0x3000, 5, 256, None, 0, 0x4000, 256, None) == 2
    assert q.lib().qgemv_static_ws_status(None, None) == 1
