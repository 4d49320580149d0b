"""GPU parity of the GEMV on activations with extreme magnitude structure, through the C ABI.

The GEMV stages activations in 16-bit form with a power-of-two scale; these cases check
that no magnitude pattern breaks the stated bound 2e-3 * ||x_m|| * max_n ||w_n|| (plus one
output ulp): values 2^20 .. 2^30 apart inside one 16-input quarter, all-zero quarters next
to quarters near 2^100, bf16 subnormals, values near bf16's largest finite number, and the
non-finite policy (an inf or NaN activation makes every output of its token non-finite --
which of NaN and +-inf is not specified -- and leaves the other tokens untouched)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import dev_bf16, qlib, to_f64

pytestmark = pytest.mark.gpu

ALL = [wl.MLX_AFFINE4_G64, wl.MXFP4, wl.NVFP4, wl.Q6K, wl.Q5_0, wl.Q5_1, wl.Q5_K]
N, K = 300, 1280  # three row tiles (the last ragged), 20 input groups; K a multiple of 256


@pytest.fixture(scope="module")
def q():
    return qlib()


def _run(q, w, x, m):
    pw = q.PackedWeight.from_logical(w)
    y = q.gemv(pw, dev_bf16(x))
    torch.cuda.synchronize()
    return to_f64(y)


@pytest.mark.parametrize("fmt", ALL)
@pytest.mark.parametrize("m", [1, 4])
@pytest.mark.parametrize("kind", ["spread", "zero_next_to_huge", "subnormal", "near_max"])
def test_gemv_extreme_magnitudes(q, fmt, m, kind):
    w = wl.weight(fmt, N, K, seed=71)
    x = wl.activations_edge(m, K, kind, seed=73 + m)
    got = _run(q, w, x, m)
    ref, _ = oracle.gemv(w, x)
    inf = np.isinf(ref)
    assert np.array_equal(got[inf], ref[inf]), "an overflowing exact result is the same infinity"
    fin = ~inf
    assert np.all(np.isfinite(got[fin])), f"{np.count_nonzero(~np.isfinite(got[fin]))} non-finite outputs"
    tol = oracle.tolerance(w, x, ref=ref)
    err = np.abs(got - ref)
    bad = fin & ~(err <= tol)
    assert not bad.any(), f"{bad.sum()} outputs out of tolerance, worst excess {np.max((err - tol)[bad])}"


@pytest.mark.parametrize("fmt", ALL)
def test_gemv_nonfinite_policy(q, fmt):
    m = 4
    w = wl.weight(fmt, N, K, seed=79)
    x = wl.activations_edge(m, K, "nonfinite", seed=83)
    got = _run(q, w, x, m)
    ref, _ = oracle.gemv(w, x)
    xv = oracle.bf16_value(x)
    bad_tok = ~np.all(np.isfinite(xv), axis=1)
    assert bad_tok.tolist() == [False, True, True, True]
    assert not np.isfinite(ref[bad_tok]).any()  # IEEE arithmetic: every such output is inf or NaN
    assert not np.isfinite(got[bad_tok]).any()
    ok = ~bad_tok
    tol = oracle.tolerance(w, x[ok], ref=ref[ok])
    assert np.all(np.abs(got[ok] - ref[ok]) <= tol)
