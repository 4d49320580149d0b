"""GPU parity of the W4A4 path (activations quantised to NVFP4, TurboEXL3 article §2.2)
against the CPU oracle, through the C ABI: the activation quantiser bit for bit (codes,
E4M3 scales, the bf16 expansion), the W4A4 GEMM within the error bound."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests import pins
from tests.gpu_util import dev_bf16, qlib, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    return qlib()


def _bits(t) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _unpack(packed: np.ndarray, k: int) -> np.ndarray:
    out = np.empty((packed.shape[0], k), dtype=np.uint8)
    out[:, 0::2] = packed[:, :k // 2] & 0xF
    out[:, 1::2] = packed[:, :k // 2] >> 4
    return out


def _activations(m: int, k: int, seed: int) -> np.ndarray:
    """Seeded bf16 activations with rows of different magnitudes, and special blocks in the
    first rows: every E2M1 rounding tie (block maximum 6, so the scale is 1 at act_scale 1),
    negative zeros, an all-zero block and a block of tiny values."""
    x = pins.bf16_value_np(wl.activations(m, k, seed=seed)) * np.exp2(
        np.random.default_rng(seed).integers(-8, 9, (m, 1)))
    if k >= 64 and m >= 2:
        ties = np.array([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0, 0.5])
        x[0, :16] = ties
        x[0, 16:32] = -0.0
        x[0, 32:48] = 0.0
        x[1, :16] *= 1e-30
    return wl.bf16_bits_from_f32(x.astype(np.float32))


def _quant_gpu(q, bits, act_scale):
    xt = dev_bf16(bits)
    codes, scales, xe = q.quant_act_nvfp4(xt, act_scale)
    torch.cuda.synchronize()
    return _unpack(codes.cpu().numpy(), bits.shape[1]), scales.cpu().numpy(), _bits(xe)


def _check_quant(q, bits, act_scale, rows=None):
    codes, scales, xe = _quant_gpu(q, bits, act_scale)
    rows = np.arange(bits.shape[0]) if rows is None else np.asarray(rows)
    c_ref, s_ref, xe_ref, _ = oracle.quantize_act_nvfp4(bits[rows], act_scale)
    xe_ref_bits = (xe_ref.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    assert np.array_equal(scales[rows], s_ref), act_scale
    bad = np.argwhere(codes[rows] != c_ref)
    assert bad.size == 0, (act_scale, bad[:5])
    assert np.array_equal(xe[rows], xe_ref_bits), act_scale


@pytest.mark.parametrize("m,k", [(1, 5120), (7, 2048), (300, 1024), (2, 64)])
@pytest.mark.parametrize("act_scale", [1.0, 0.37, 1e-6, 1e3])
def test_quant_act_bit_exact(q, m, k, act_scale):
    """1e-6 saturates most block scales at 448 (codes clamp at 6); 1e3 sends them to E4M3
    subnormals and zero (whole blocks quantise to zero)."""
    _check_quant(q, _activations(m, k, seed=m * 7 + k), act_scale)


def test_quant_act_full_prefill_size_sampled(q):
    """8192 tokens x 5120 (the prefill workload): the whole matrix on the GPU, sampled rows
    (independent of each other) against the oracle."""
    bits = _activations(8192, 5120, seed=5)
    rows = np.random.default_rng(1).choice(8192, 48, replace=False)
    rows[:3] = [0, 1, 8191]
    _check_quant(q, bits, 0.5, rows=rows)


def test_quant_act_optional_outputs_and_errors(q):
    bits = _activations(4, 256, seed=9)
    xt = dev_bf16(bits)
    xe = torch.empty((4, 256), dtype=torch.bfloat16, device="cuda")
    q.qg_quant_act_nvfp4(xt.data_ptr(), 4, 256, xt.stride(0), 1.0, None, 0, None, 0, xe.data_ptr(), 256)
    torch.cuda.synchronize()
    _, _, xe_ref, _ = oracle.quantize_act_nvfp4(bits, 1.0)
    assert np.array_equal(_bits(xe), (xe_ref.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16))
    with pytest.raises(q.QGError):
        q.qg_quant_act_nvfp4(xt.data_ptr(), 4, 250, xt.stride(0), 1.0, None, 0, None, 0, xe.data_ptr(), 256)
    with pytest.raises(q.QGError):
        q.qg_quant_act_nvfp4(xt.data_ptr(), 4, 256, xt.stride(0), float("nan"), None, 0, None, 0, xe.data_ptr(), 256)


def _w4a4_tol(w, xq, ref):
    wmax = float(np.max(oracle.row_norms(w)))
    return 2e-3 * np.linalg.norm(xq, axis=1)[:, None] * wmax + 2.0 ** -7 * np.abs(ref)


@pytest.mark.parametrize("n,k,m,act_scale", [(300, 208, 1, 1.0), (384, 1024, 4, 0.02), (1000, 1280, 40, 0.5),
                                             (300, 512, 300, 3.0), (129, 512, 7, 0.1)])
def test_w4a4_gemm_parity(q, n, k, m, act_scale):
    """1..4 rows through the GEMV, 5..128 the small-token GEMM, more the prefill GEMM; ragged
    row tiles and token tiles; a residual on every other case."""
    w, _, res = wl.gemv_case(wl.NVFP4, n, k, m, seed=n + m, residual=(m % 2 == 0))
    bits = _activations(m, k, seed=n + k + m)
    pw = q.PackedWeight.from_logical(w)
    y = q.gemm_w4a4(pw, dev_bf16(bits), act_scale, None if res is None else dev_bf16(res))
    torch.cuda.synchronize()
    got = to_f64(y)
    ref, _, xq = oracle.gemm_w4a4(w, bits, act_scale, res)
    tol = _w4a4_tol(w, xq, ref)
    if res is not None:
        tol = tol + 2.0 ** -7 * np.abs(oracle.bf16_value(res))
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    assert np.all(err <= tol), (float(np.max(err / tol)), np.unravel_index(np.argmax(err / tol), err.shape))


@pytest.mark.parametrize("m", [4, 128, 1024])
def test_w4a4_full_size_sampled(q, m):
    """NVFP4 17408 x 5120 at 4, 128 and 1024 tokens (GEMV, small-token GEMM, prefill GEMM):
    every output on the GPU, sampled output rows against the oracle."""
    w = wl.weight(wl.NVFP4, 17408, 5120, seed=3)
    bits = _activations(m, 5120, seed=m)
    pw = q.PackedWeight.from_logical(w)
    ws = q.Workspace(q.qgemm_w4a4_workspace_size(wl.NVFP4, 17408, 5120, m))
    y = q.gemm_w4a4(pw, dev_bf16(bits), 0.25, workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    rows = np.random.default_rng(m).choice(17408, 96, replace=False)
    rows[:2] = [0, 17407]
    got = to_f64(y)[:, rows]
    ref, _, xq = oracle.gemm_w4a4(w, bits, 0.25, rows=rows)
    wmax = float(np.max(oracle.row_norms(w, rows)))
    tol = 2e-3 * np.linalg.norm(xq, axis=1)[:, None] * wmax + 2.0 ** -7 * np.abs(ref)
    assert np.all(np.abs(got - ref) <= tol)


@pytest.mark.parametrize("m", [3, 40, 300])
def test_w4a4_on_exact_activations_equals_w4a16(q, m):
    """Activations NVFP4 represents exactly, at a power-of-two tensor scale: both calls form
    the same exact products.  At 1..4 rows W4A4 runs the W4A16 GEMV on the exact expansion
    and returns its outputs bit for bit; from 5 rows it multiplies the FP4 codes on the
    block-scaled tensor cores, whose fp32 sums may round in another order, so both sides
    are held to the oracle's bound."""
    w = wl.weight(wl.NVFP4, 384, 1024, seed=m)
    bits, _, _ = pins.exact_nvfp4_activations(m, 1024, 0.25, seed=m)
    pw = q.PackedWeight.from_logical(w)
    xt = dev_bf16(bits)
    y4 = q.gemm_w4a4(pw, xt, 0.25)
    y16 = q.gemm(pw, xt)
    torch.cuda.synchronize()
    if m <= 4:
        assert torch.equal(y4.contiguous().view(torch.int16), y16.contiguous().view(torch.int16))
    else:
        ref, _ = oracle.gemv(w, bits)
        tol = oracle.tolerance(w, bits, ref=ref)
        assert np.all(np.abs(to_f64(y4) - ref) <= tol)
        assert np.all(np.abs(to_f64(y16) - ref) <= tol)


@pytest.mark.parametrize("n,k,m", [(257, 208, 300), (640, 1280, 513), (128, 64, 5), (1000, 4096, 260)])
def test_w4a4_fp4_tensor_core_shapes(q, n, k, m):
    """The block-scaled FP4 GEMM (5 or more rows): K tails inside a 256-deep stage and inside a
    64-deep tile (K = 208, 64), several token tiles with a ragged last one, ragged row tiles, a
    residual; every output against the oracle, and two calls bit for bit."""
    w, _, res = wl.gemv_case(wl.NVFP4, n, k, m, seed=n + k, residual=True)
    bits = _activations(m, k, seed=m + k)
    pw = q.PackedWeight.from_logical(w)
    xt, rt = dev_bf16(bits), dev_bf16(res)
    ws = q.Workspace(q.qgemm_w4a4_workspace_size(wl.NVFP4, n, k, m))
    y1 = q.gemm_w4a4(pw, xt, 0.3, rt, workspace=ws).clone()
    y2 = q.gemm_w4a4(pw, xt, 0.3, rt, workspace=ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    assert torch.equal(y1.contiguous().view(torch.int16), y2.contiguous().view(torch.int16))
    got = to_f64(y1)
    ref, _, xq = oracle.gemm_w4a4(w, bits, 0.3, res)
    tol = _w4a4_tol(w, xq, ref) + 2.0 ** -7 * np.abs(oracle.bf16_value(res))
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got))
    assert np.all(err <= tol), (float(np.max(err / tol)), np.unravel_index(np.argmax(err / tol), err.shape))
