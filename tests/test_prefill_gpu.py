"""GPU parity of the prefill GEMM (tcgen05 tensor cores) against the CPU oracle,
called through the C ABI (qgemm with more than 4 token rows)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import dev_bf16, qlib, to_f64

pytestmark = pytest.mark.gpu

ALL = [wl.MLX_AFFINE4_G64, wl.MXFP4, wl.NVFP4, wl.Q6K, wl.Q5_0, wl.Q5_1, wl.Q5_K]
# (n, k, tokens): several 128-row tiles, ragged rows, ragged token tiles (256 per tile),
# K that is not a multiple of the 64-deep stage for the small-block formats
SHAPES = {
    wl.MLX_AFFINE4_G64: [(300, 640, 5), (256, 1024, 300), (128, 64, 17)],
    wl.MXFP4: [(300, 640, 260), (1024, 2048, 96), (257, 96, 33)],
    wl.NVFP4: [(300, 208, 300), (1000, 1280, 600), (129, 512, 7)],
    wl.Q6K: [(300, 768, 130), (640, 1536, 257), (129, 256, 5)],
    wl.Q5_0: [(300, 640, 5), (256, 1024, 300), (129, 96, 17)],
    wl.Q5_1: [(300, 160, 260), (1024, 2048, 96), (257, 512, 33)],
    wl.Q5_K: [(300, 768, 130), (640, 1536, 257), (129, 256, 5)],
}


@pytest.fixture(scope="module")
def q():
    return qlib()


def _run(q, w, x, res, pw=None, ws=None):
    pw = pw or q.PackedWeight.from_logical(w)
    xt = dev_bf16(x)
    rt = dev_bf16(res) if res is not None else None
    y = q.gemm(pw, xt, rt, workspace=ws)
    torch.cuda.synchronize()
    return to_f64(y), pw


@pytest.mark.parametrize("fmt", ALL)
def test_prefill_small_shapes(q, fmt):
    for i, (n, k, t) in enumerate(SHAPES[fmt]):
        w, x, res = wl.gemv_case(fmt, n, k, t, seed=200 + i, residual=(i % 2 == 0))
        ws = q.Workspace(q.qg_gemm_workspace_size(fmt, n, k, t))
        got, _ = _run(q, w, x, res, ws=ws)
        ref, _ = oracle.gemv(w, x, res)
        tol = oracle.tolerance(w, x, res, ref=ref)
        err = np.abs(got - ref)
        assert np.all(np.isfinite(got))
        assert np.all(err <= tol), f"{fmt} {n}x{k} t={t}: {np.sum(err > tol)} out of tolerance, worst {np.max(err - tol)}"
        assert ws.status() == 0


def test_prefill_deterministic(q):
    w, x, res = wl.gemv_case(wl.NVFP4, 1000, 1280, 600, seed=7, residual=True)
    pw = q.PackedWeight.from_logical(w)
    a, _ = _run(q, w, x, res, pw=pw)
    b, _ = _run(q, w, x, res, pw=pw)
    assert np.array_equal(a, b)


def test_qgemm_dispatches_small_m_to_gemv(q):
    w, x, res = wl.gemv_case(wl.MXFP4, 1024, 2048, 3, seed=8, residual=True)
    pw = q.PackedWeight.from_logical(w)
    got, _ = _run(q, w, x, res, pw=pw)
    ref_gemv = to_f64(q.gemv(pw, dev_bf16(x), dev_bf16(res)))
    torch.cuda.synchronize()
    assert np.array_equal(got, ref_gemv)


def test_prefill_matches_gemv_at_five_rows(q):
    # five tokens take the tensor-core path; the first four must agree with the GEMV
    # within the tolerance (different summation orders)
    w, x, _ = wl.gemv_case(wl.NVFP4, 512, 1024, 5, seed=9)
    pw = q.PackedWeight.from_logical(w)
    got, _ = _run(q, w, x, None, pw=pw)
    ref4 = to_f64(q.gemv(pw, dev_bf16(x[:4])))
    tol = oracle.tolerance(w, x[:4])
    assert np.all(np.abs(got[:4] - ref4) <= 2 * tol)


def test_prefill_full_size_sampled(q):
    """NVFP4 17408 x 5120 against 8192 tokens (the prefill benchmark size): every output
    of sampled tokens and rows against the oracle."""
    cfg = wl.PREFILL
    n, k, t = cfg["n"], cfg["k"], cfg["tokens"]
    w = wl.weight(wl.NVFP4, n, k, seed=0)
    x = wl.activations(t, k, seed=3)
    got, _ = _run(q, w, x, None)
    rng = np.random.default_rng(4)
    toks = np.unique(np.concatenate([[0, 255, 256, t - 1], rng.integers(0, t, 60)]))
    rows = np.unique(np.concatenate([[0, 127, 128, n - 1], rng.integers(0, n, 508)]))
    ref, _ = oracle.gemv_rows(w, x[toks], rows)
    tol = oracle.tolerance(w, x[toks], rows=rows, ref=ref)
    err = np.abs(got[np.ix_(toks, rows)] - ref)
    assert np.all(err <= tol), f"{np.sum(err > tol)} out of tolerance"


@pytest.mark.parametrize("n,k,t", [(17408, 5120, 128), (5120, 17408, 128), (5120, 17408, 300), (17408, 5120, 16)])
def test_small_token_gemm_full_size_sampled(q, n, k, t):
    """The benchmark matrices against one token tile (the small-token GEMM: 136 row tiles over
    all of K, or 40 row tiles with K split over clusters of 3) and against 300 tokens (the
    256-token GEMM with K split): sampled rows of every token against the oracle."""
    w = wl.weight(wl.NVFP4, n, k, seed=0)
    x = wl.activations(t, k, seed=5)
    got, _ = _run(q, w, x, None)
    rng = np.random.default_rng(6)
    rows = np.unique(np.concatenate([[0, 127, 128, n - 1], rng.integers(0, n, 124)]))
    ref, _ = oracle.gemv_rows(w, x, rows)
    tol = oracle.tolerance(w, x, rows=rows, ref=ref)
    err = np.abs(got[:, rows] - ref)
    assert np.all(np.isfinite(got))
    assert np.all(err <= tol), f"{np.sum(err > tol)} out of tolerance"


@pytest.mark.parametrize("t", [5, 16, 17, 64, 65, 128, 129, 255, 256, 257])
def test_token_count_boundaries(q, t):
    """Every token-tile width of the small-token GEMM (16/32/64/128) and the switch to the
    256-token GEMM, with a residual, on a weight whose few row tiles split K over clusters."""
    w, x, res = wl.gemv_case(wl.NVFP4, 384, 1024, t, seed=60 + t, residual=True)
    ws = q.Workspace(q.qg_gemm_workspace_size(wl.NVFP4, 384, 1024, t))
    got, _ = _run(q, w, x, res, ws=ws)
    ref, _ = oracle.gemv(w, x, res)
    err = np.abs(got - ref)
    assert np.all(err <= oracle.tolerance(w, x, res, ref=ref))
    assert ws.status() == 0


@pytest.mark.parametrize("fmt,t", [(wl.Q5_K, 128), (wl.Q5_0, 1000), (wl.Q5_1, 40)])
def test_prefill_q5_full_size_sampled(q, fmt, t):
    """The 5-bit formats at the 17408 x 5120 gate/up size against one small-token tile, several
    256-token tiles and 40 tokens: every token of sampled rows against the oracle."""
    n, k = 17408, 5120
    w = wl.weight(fmt, n, k, seed=0)
    x = wl.activations(t, k, seed=7)
    got, _ = _run(q, w, x, None)
    rng = np.random.default_rng(8)
    rows = np.unique(np.concatenate([[0, 127, 128, n - 1], rng.integers(0, n, 60)]))
    ref, _ = oracle.gemv_rows(w, x, rows)
    err = np.abs(got[:, rows] - ref)
    assert np.all(err <= oracle.tolerance(w, x, rows=rows, ref=ref)), f"{fmt} t={t}"
