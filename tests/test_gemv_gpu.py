"""GPU parity: dequantisation bit-exact and GEMV within tolerance of the CPU oracle,
called through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import dev_bf16, qlib, to_f64

pytestmark = pytest.mark.gpu

ALL = [wl.MLX_AFFINE4_G64, wl.MXFP4, wl.NVFP4, wl.Q6K, wl.Q5_0, wl.Q5_1, wl.Q5_K]
# several 128 x 64 tiles, ragged row tails, padded K (NVFP4 208 = 13 blocks, MXFP4 96)
SMALL = {
    wl.MLX_AFFINE4_G64: [(300, 640), (128, 64), (1000, 1280)],
    wl.MXFP4: [(300, 640), (257, 96), (1024, 2048)],
    wl.NVFP4: [(300, 208), (1000, 1280), (129, 512)],
    wl.Q6K: [(300, 768), (129, 256), (640, 1536)],
    wl.Q5_0: [(300, 640), (257, 96), (1000, 1280)],
    wl.Q5_1: [(300, 160), (129, 512), (640, 1536)],
    wl.Q5_K: [(300, 768), (129, 256), (640, 1536)],
}


@pytest.fixture(scope="module")
def q():
    return qlib()


@pytest.mark.parametrize("fmt", ALL)
def test_dequant_bit_exact(q, fmt):
    for n, k in SMALL[fmt]:
        w = wl.weight(fmt, n, k, seed=n * 7 + k)
        pw = q.PackedWeight.from_logical(w)
        got32 = to_f64(q.dequant(pw, q.OUT_F32))
        assert np.array_equal(got32, oracle.dequant(w).astype(np.float64)), (fmt, n, k)
        got16 = to_f64(q.dequant(pw, q.OUT_BF16))
        assert np.array_equal(got16, oracle.dequant_operand_bf16(w)), (fmt, n, k)


def _check(q, w, x, res, m, pw=None, ws=None, rows=None):
    pw = pw or q.PackedWeight.from_logical(w)
    xt = dev_bf16(x)
    rt = dev_bf16(res) if res is not None else None
    y = q.gemv(pw, xt, rt, workspace=ws)
    torch.cuda.synchronize()
    got = to_f64(y)
    if rows is None:
        ref, _ = oracle.gemv(w, x, res)
        tol = oracle.tolerance(w, x, res, ref=ref)
    else:
        ref, _ = oracle.gemv_rows(w, x, rows, res)
        got = got[:, rows]
        tol = oracle.tolerance(w, x, res, rows=rows, ref=ref)
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got))
    bad = err > tol
    assert not bad.any(), f"{bad.sum()} outputs out of tolerance, worst {np.max(err - tol)}"
    return got, ref


@pytest.mark.parametrize("fmt", ALL)
@pytest.mark.parametrize("m", [1, 2, 3, 4])
def test_gemv_small_shapes(q, fmt, m):
    for i, (n, k) in enumerate(SMALL[fmt]):
        w, x, res = wl.gemv_case(fmt, n, k, m, seed=100 + i, residual=(i % 2 == 1))
        _check(q, w, x, res, m)


@pytest.mark.parametrize("fmt", ALL)
def test_gemv_deterministic_and_workspace_reset(q, fmt):
    n, k = SMALL[fmt][-1]
    w, x, res = wl.gemv_case(fmt, n, k, 3, seed=5, residual=True)
    pw = q.PackedWeight.from_logical(w)
    ws = q.Workspace(q.qg_gemv_workspace_size(fmt, n, k, 3))
    xt, rt = dev_bf16(x), dev_bf16(res)
    a = q.gemv(pw, xt, rt, workspace=ws).clone()
    b = q.gemv(pw, xt, rt, workspace=ws).clone()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert ws.status() == 0
    # tickets are back at zero after every call
    hdr = 256
    nt = (n + 127) // 128
    cnt = ws.buf[hdr:hdr + 4 * nt].view(torch.int32)
    assert int(cnt.abs().sum()) == 0


def test_gemv_zero_and_identity_like_inputs(q):
    # x = 0 gives exactly the residual; a one-hot x picks one column of W
    n, k = 256, 512
    w = wl.weight(wl.NVFP4, n, k, seed=9)
    x = np.zeros((2, k), np.uint16)
    res = wl.activations(2, n, seed=9, stream="residual")
    got, ref = _check(q, w, x, res, 2)
    assert np.array_equal(got, oracle.bf16_value(res))
    x1 = np.zeros((1, k), np.uint16)
    x1[0, 77] = 0x3F80  # 1.0
    got, _ = _check(q, w, x1, None, 1)
    col = oracle.dequant(w)[:, 77].astype(np.float64)
    assert np.array_equal(got[0], oracle.round_to_bf16(col))


FULL = [
    ("mlx_affine4_g64_5120x5120", (1,)),
    ("nvfp4_gate_up_17408x5120", (1, 2, 3, 4)),
    ("nvfp4_down_5120x17408", (1, 4)),
    ("q6k_5120x6144", (1, 4)),
    ("q6k_output_248320x5120", (1, 4)),
    ("q5_k_gate_up_17408x5120", (1, 4)),
    ("q5_k_down_5120x17408", (1, 3)),
    ("q5_k_out_5120x6144", (2,)),
    ("q5_0_gate_up_17408x5120", (1, 4)),
    ("q5_1_gate_up_17408x5120", (1, 2)),
]


@pytest.mark.parametrize("name,ms", FULL)
def test_gemv_full_size_sampled_rows(q, name, ms):
    cfg = wl.WORKLOADS.get(name) or wl.WORKLOADS_Q5[name]
    fmt, n, k = cfg["fmt"], cfg["n"], cfg["k"]
    w = wl.weight(fmt, n, k, seed=0)
    pw = q.PackedWeight.from_logical(w)
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, n - 1], rng.integers(0, n, 251)]))
    for m in ms:
        x = wl.activations(m, k, seed=m)
        res = wl.activations(m, n, seed=m, stream="residual") if cfg["residual"] else None
        _check(q, w, x, res, m, pw=pw, rows=rows)


# The three ways a GEMV is cut across the SMs (152 on GB300): one whole 128-row tile per CTA
# (row tiles close to the SM count: 136 here), row tiles split over thread-block clusters
# with the partials summed in the first CTA's shared memory (few row tiles: 20 here), and
# stream-K with tickets (more row tiles than SMs: 160 here).  Every output is checked, twice
# in a row on one workspace (bit-identical).
PARTITIONS = [("whole_row_tiles", wl.NVFP4, 136 * 128, 256), ("cluster_split", wl.MXFP4, 20 * 128 - 37, 1024),
              ("stream_k", wl.MLX_AFFINE4_G64, 160 * 128, 512), ("stream_k_q6k", wl.Q6K, 170 * 128 - 5, 512),
              ("stream_k_q5k", wl.Q5_K, 170 * 128 - 5, 512), ("cluster_split_q5_1", wl.Q5_1, 20 * 128 - 9, 1056),
              ("whole_row_tiles_q5_0", wl.Q5_0, 136 * 128 - 100, 288)]


@pytest.mark.parametrize("name,fmt,n,k", PARTITIONS)
@pytest.mark.parametrize("m", [1, 4])
def test_gemv_partition_modes(q, name, fmt, n, k, m):
    w, x, res = wl.gemv_case(fmt, n, k, m, seed=900 + m, residual=(m == 4))
    pw = q.PackedWeight.from_logical(w)
    ws = q.Workspace(q.qg_gemv_workspace_size(fmt, n, k, m))
    got, _ = _check(q, w, x, res, m, pw=pw, ws=ws)
    got2, _ = _check(q, w, x, res, m, pw=pw, ws=ws)
    assert np.array_equal(got, got2)
    assert ws.status() == 0


MIN_K = {wl.MLX_AFFINE4_G64: 64, wl.MXFP4: 32, wl.NVFP4: 16, wl.Q6K: 256, wl.Q5_0: 32, wl.Q5_1: 32, wl.Q5_K: 256}


@pytest.mark.parametrize("fmt", ALL)
def test_degenerate_shapes(q, fmt):
    """One output row, the format's smallest K (one block), and one row below a tile: every
    M through the GEMV and 5 and 200 tokens through the tensor-core GEMMs, against the oracle."""
    k = MIN_K[fmt]
    for n in (1, 127):
        for m in (1, 2, 3, 4, 5, 200):
            w, x, res = wl.gemv_case(fmt, n, k, m, seed=n * 10 + m, residual=(m % 2 == 0))
            pw = q.PackedWeight.from_logical(w)
            xt, rt = dev_bf16(x), (dev_bf16(res) if res is not None else None)
            y = q.gemv(pw, xt, rt) if m <= 4 else q.gemm(pw, xt, rt)
            torch.cuda.synchronize()
            ref, _ = oracle.gemv(w, x, res)
            err = np.abs(to_f64(y) - ref)
            assert np.all(err <= oracle.tolerance(w, x, res, ref=ref)), (fmt, n, m)
