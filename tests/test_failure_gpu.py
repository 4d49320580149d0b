"""Failure detection on the GPU without a fault: a bounded mbarrier wait that nothing
completes runs out, the kernel records QG_ERR_TIMEOUT in the workspace status word and
returns; the host reads the status, and the context keeps working afterwards."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import dev_bf16, qlib, to_f64

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    q = qlib()
    ws = q.Workspace(256)
    q.qg_selftest_wait_timeout(ws.ptr, ws.nbytes, 0)
    assert q.STATUS[ws.status()] == "QG_ERR_TIMEOUT"
    assert ws.status() == 0  # reading the status clears it
    # the context is still usable: a GEMV right after matches the oracle
    w, x, _ = wl.gemv_case(wl.NVFP4, 256, 512, 2, seed=5)
    pw = q.PackedWeight.from_logical(w)
    y = q.gemv(pw, dev_bf16(x))
    torch.cuda.synchronize()
    ref, _ = oracle.gemv(w, x)
    tol = oracle.tolerance(w, x, None, ref=ref)
    assert np.all(np.abs(to_f64(y) - ref) <= tol)
