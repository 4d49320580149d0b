"""GPU parity of the mixture-of-experts prefill chain (route, grouped tensor-core gate/up
GEMM with SwiGLU in its epilogue, grouped down GEMM, weighted finish) against the CPU
oracle, through the C ABI.  Covers every format, ragged per-expert tiles (one tile, several
192-pair tiles, a remainder), the shared expert as extra tiles, a ragged hidden size, the
smallest token count that takes this chain, and the 512-expert, 8192-token layer on
sampled tokens."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_util import dev_bf16, grouped_rows, h_tolerance, moe_tolerance, qlib, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    return qlib()


def _run(q, layer, x, lg, k, reps=1, workspace=None):
    pm = q.PackedMoE(layer)
    ids, w, rws = q.route(torch.from_numpy(np.ascontiguousarray(lg)).cuda(), k)
    if workspace is None:
        workspace = q.Workspace(q.qmoe_workspace_size(pm.desc, x.shape[0], k))
    outs = [q.moe_ffn(pm, dev_bf16(x), w, rws, workspace=workspace) for _ in range(reps)]
    torch.cuda.synchronize()
    assert workspace.status() == 0
    return outs, ids


def _check(got, ref, tol):
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got))
    assert np.all(err <= tol), f"{np.sum(err > tol)} of {err.size} out of tolerance, worst {np.max(err - tol)}"


@pytest.mark.parametrize("fmt", [wl.MXFP4, wl.NVFP4, wl.MLX_AFFINE4_G64, wl.Q6K])
def test_moe_prefill_small(q, fmt):
    E, k, t = 16, 4, 300
    H, F = (512, 256) if fmt == wl.Q6K else (256, 128)
    layer = wl.moe_layer(fmt, E, H, F, seed=400 + fmt, shared=True)
    x = wl.moe_tokens(t, H, seed=401)
    lg = wl.router_logits(t, E, seed=402)
    (out, out2), _ = _run(q, layer, x, lg, k, reps=2)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))  # no atomics in any sum
    ref = oracle.moe_forward(layer, x, lg, k)
    _check(to_f64(out), ref, moe_tolerance(oracle, layer, x, lg, k, ref))


@pytest.mark.parametrize("skew", [False, True])
def test_moe_prefill_multi_tile(q, skew):
    """Experts with more than 192 pairs split into several tiles plus a remainder; with
    skew every token's first choice is expert 3 (1100 pairs: 5 full tiles + 140)."""
    E, H, F, k, t = 8, 256, 128, 2, 1100
    layer = wl.moe_layer(wl.MXFP4, E, H, F, seed=410, shared=True)
    x = wl.moe_tokens(t, H, seed=411)
    lg = wl.router_logits(t, E, seed=412)
    if skew:
        lg = lg.copy()
        lg[:, 3] += 8.0
    (out,), ids = _run(q, layer, x, lg, k)
    counts = np.bincount(ids.cpu().numpy().ravel(), minlength=E)
    assert counts.max() > 192
    ref = oracle.moe_forward(layer, x, lg, k)
    _check(to_f64(out), ref, moe_tolerance(oracle, layer, x, lg, k, ref))


@pytest.mark.parametrize("t", [5, 17, 193])
def test_moe_prefill_small_token_counts(q, t):
    """The smallest count past the GEMV chain, a ragged count and one past a 192-token
    shared-expert tile."""
    E, H, F, k = 12, 256, 128, 3
    layer = wl.moe_layer(wl.NVFP4, E, H, F, seed=420 + t, shared=True)
    x = wl.moe_tokens(t, H, seed=421)
    lg = wl.router_logits(t, E, seed=422)
    (out,), _ = _run(q, layer, x, lg, k)
    ref = oracle.moe_forward(layer, x, lg, k)
    _check(to_f64(out), ref, moe_tolerance(oracle, layer, x, lg, k, ref))


def test_moe_prefill_without_shared(q):
    E, H, F, k, t = 8, 256, 128, 3, 77
    layer = wl.moe_layer(wl.MXFP4, E, H, F, seed=430, shared=False)
    x = wl.moe_tokens(t, H, seed=431)
    lg = wl.router_logits(t, E, seed=432)
    (out,), _ = _run(q, layer, x, lg, k)
    ref = oracle.moe_forward(layer, x, lg, k)
    _check(to_f64(out), ref, moe_tolerance(oracle, layer, x, lg, k, ref))


def test_moe_prefill_ragged_hidden(q):
    """hidden = 208 (NVFP4, 16-wide blocks): the gate/up K ends inside a 64-deep stage, so
    the gathered rows are zero-filled past it; the down projection's last 128-row tile is
    partial."""
    E, H, F, k, t = 6, 208, 128, 2, 90
    layer = wl.moe_layer(wl.NVFP4, E, H, F, seed=440, shared=True)
    x = wl.moe_tokens(t, H, seed=441)
    lg = wl.router_logits(t, E, seed=442)
    (out,), _ = _run(q, layer, x, lg, k)
    ref = oracle.moe_forward(layer, x, lg, k)
    _check(to_f64(out), ref, moe_tolerance(oracle, layer, x, lg, k, ref))


def test_moe_prefill_full_config_sampled(q):
    """The MoE prefill layer: 512 MXFP4 experts, hidden 2048, FFN 512, top-10, shared
    expert, 8192 tokens (about 160 pairs per expert); the oracle checks sampled tokens at
    both ends and across a shared-tile boundary; the run is repeated bit for bit."""
    c = wl.MOE_PREFILL
    layer = wl.moe_layer(c["fmt"], c["n_experts"], c["hidden"], c["ffn"], seed=0, shared=True)
    x = wl.moe_tokens(c["tokens"], c["hidden"], seed=30)
    lg = wl.router_logits(c["tokens"], c["n_experts"], seed=31)
    (out, out2), _ = _run(q, layer, x, lg, c["topk"], reps=2)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    got = to_f64(out)
    assert np.all(np.isfinite(got))
    tokens = np.array([0, 255, 256, 8191])
    ref = oracle.moe_forward(layer, x, lg, c["topk"], tokens=tokens)
    _check(got[tokens], ref, moe_tolerance(oracle, layer, x, lg, c["topk"], ref, tokens=tokens))


@pytest.mark.parametrize("fmt,shared", [(wl.MXFP4, True), (wl.NVFP4, False)])
def test_moe_prefill_staged(q, fmt, shared):
    """qgemm_grouped one stage at a time on the tensor-core chain: h against the oracle's h,
    the combined output bit-identical to the fused qmoe_ffn chain."""
    E, H, F, k, t = 16, 256, 128, 4, 257
    layer = wl.moe_layer(fmt, E, H, F, seed=430 + fmt, shared=shared)
    x = wl.moe_tokens(t, H, seed=431)
    lg = wl.router_logits(t, E, seed=432)
    pm = q.PackedMoE(layer)
    ids, w, rws = q.route(torch.from_numpy(lg).cuda(), k)
    xd = dev_bf16(x)
    fused = q.moe_ffn(pm, xd, w, rws)
    h = q.moe_stage(pm, q.QG_MOE_GATE_UP_SWIGLU, xd, t, k, rws)
    out = q.moe_stage(pm, q.QG_MOE_DOWN_COMBINE, h, t, k, rws, topk_w=w)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), fused.view(torch.int16))
    _, _, _, _, inter = oracle.moe_forward(layer, x, lg, k, with_intermediates=True)
    rows = grouped_rows(ids.cpu().numpy(), shared)
    href = np.stack([inter[r][2] for r in rows])
    _check(to_f64(h), href, h_tolerance(oracle, layer, x, inter, rows))


@pytest.mark.parametrize("fmt", [wl.MXFP4, wl.Q6K])
def test_moe_prefill_shared_gate(q, fmt):
    """The shared expert weighed by its sigmoid gate on the tensor-core chain: against the
    oracle, staged = fused bit for bit, a saturated gate (+100) = no gate bit for bit."""
    E, k, t = 16, 4, 200
    H, F = (512, 256) if fmt == wl.Q6K else (256, 128)
    layer = wl.moe_layer(fmt, E, H, F, seed=440 + fmt, shared=True)
    x = wl.moe_tokens(t, H, seed=441)
    lg = wl.router_logits(t, E, seed=442)
    gl = wl.shared_gate_logits(t, seed=443)
    pm = q.PackedMoE(layer)
    ids, w, rws = q.route(torch.from_numpy(lg).cuda(), k)
    xd = dev_bf16(x)
    gd = torch.from_numpy(gl).cuda()
    out = q.moe_ffn(pm, xd, w, rws, shared_gate=gd)
    h = q.moe_stage(pm, q.QG_MOE_GATE_UP_SWIGLU, xd, t, k, rws)
    staged = q.moe_stage(pm, q.QG_MOE_DOWN_COMBINE, h, t, k, rws, topk_w=w, shared_gate=gd)
    sat = q.moe_ffn(pm, xd, w, rws, shared_gate=torch.full((t,), 100.0, device="cuda"))
    plain = q.moe_ffn(pm, xd, w, rws)
    torch.cuda.synchronize()
    assert torch.equal(staged.view(torch.int16), out.view(torch.int16))
    assert torch.equal(sat.view(torch.int16), plain.view(torch.int16))
    ref = oracle.moe_forward(layer, x, lg, k, shared_gate=gl)
    _check(to_f64(out), ref, moe_tolerance(oracle, layer, x, lg, k, ref))
