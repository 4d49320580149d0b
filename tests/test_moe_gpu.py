"""GPU parity of the mixture-of-experts decode chain (route, grouped gate/up GEMV, SwiGLU,
grouped down GEMV, weighted finish) against the CPU oracle, through the C ABI."""
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


def _route(q, lg):
    lt = torch.from_numpy(np.ascontiguousarray(lg, dtype=np.float32)).cuda()
    ids, w, ws = q.route(lt, TOPK[0])
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy(), ws


TOPK = [10]


@pytest.mark.parametrize("t,e,k", [(1, 512, 10), (4, 512, 10), (3, 64, 4), (32, 512, 10), (300, 128, 6), (8192, 512, 10)])
def test_route_matches_oracle(q, t, e, k):
    lg = wl.router_logits(t, e, seed=t + e + k)
    lt = torch.from_numpy(np.ascontiguousarray(lg)).cuda()
    ids, w, ws = q.route(lt, k)
    torch.cuda.synchronize()
    rid, rp = oracle.route(lg, k)
    assert np.array_equal(ids.cpu().numpy(), rid)  # integer decisions from the same fp32 logits
    assert np.allclose(w.cpu().numpy(), rp, rtol=2e-6, atol=1e-7)
    ids2, w2, _ = q.route(lt, k)
    torch.cuda.synchronize()
    assert torch.equal(ids, ids2) and torch.equal(w, w2)


def test_route_ties_go_to_lower_index(q):
    lg = np.zeros((4, 64), np.float32)
    lg[:, 10] = 1.0
    lg[:, 20] = 1.0
    lg[2, :] = 0.5
    # -0 ties with +0 (lower index first); NaN sorts below every number
    lg[3, :] = -1.0
    lg[3, 7] = -0.0
    lg[3, 2] = 0.0
    lg[3, 9] = np.nan
    lt = torch.from_numpy(lg).cuda()
    ids, w, _ = q.route(lt, 3)
    torch.cuda.synchronize()
    rid, rp = oracle.route(lg, 3)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert list(rid[3]) == [2, 7, 0]
    assert np.allclose(w.cpu().numpy(), rp, rtol=2e-6, atol=1e-7)


def _clustered_logits(t, e, k, seed):
    """Router logits whose winners crowd into few residues mod 32 (experts e, e+32, e+64, ...),
    the ones a warp-wide top-k that gives each lane the experts of one residue finds hardest:
    token 0 has all k winners on one residue, token 1 three on one residue and the rest on
    another, token 2 exactly three on one residue (k = 3 case) and token 3 ties on one
    residue."""
    rng = np.random.default_rng(seed)
    lg = rng.standard_normal((t, e)).astype(np.float32)
    lane = 5
    same = [lane + 32 * i for i in range(e // 32)]
    for i, ex in enumerate(same[:k]):
        lg[0, ex] = 10.0 - 0.5 * i
    if t > 1:
        for i, ex in enumerate(same[:3]):
            lg[1, ex] = 9.0 - i
        for i in range(k - 3):
            lg[1, 17 + 32 * (i % (e // 32))] = 5.0 - 0.25 * i + (0.01 if i >= e // 32 else 0.0) * i
    if t > 2:
        lg[2, same[:3]] = [8.0, 7.5, 7.25]
    if t > 3:
        lg[3, same[: min(k + 2, len(same))]] = 3.0  # ties: lower experts first
    return lg


@pytest.mark.parametrize("t,e,k", [(4, 512, 10), (4, 512, 4), (3, 512, 3), (4, 128, 6), (2, 64, 4)])
def test_route_winners_on_one_residue(q, t, e, k):
    """Top-k whose winners share a residue mod 32: ids equal to the oracle's, weights within
    rounding, for the router launch and for the router inside the decode chain's gate/up
    launch (same ids and weights byte for byte)."""
    lg = _clustered_logits(t, e, k, seed=700 + t + e + k)
    lt = torch.from_numpy(np.ascontiguousarray(lg)).cuda()
    ids, w, _ = q.route(lt, k)
    torch.cuda.synchronize()
    rid, rp = oracle.route(lg, k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.allclose(w.cpu().numpy(), rp, rtol=2e-6, atol=1e-7)
    H, F = 256, 128
    layer = wl.moe_layer(wl.MXFP4, e, H, F, seed=701, shared=False)
    pm = q.PackedMoE(layer)
    xd = dev_bf16(wl.moe_tokens(t, H, seed=702))
    _, ids_b, w_b, _ = q.moe_forward(pm, xd, lt, k)
    torch.cuda.synchronize()
    assert torch.equal(ids, ids_b) and torch.equal(w, w_b)


@pytest.mark.parametrize("fmt,e,h,f,k,shared", [(wl.MXFP4, 16, 256, 128, 4, True), (wl.NVFP4, 64, 1024, 512, 10, True),
                                                 (wl.Q6K, 8, 512, 256, 1, False), (wl.MLX_AFFINE4_G64, 32, 256, 384, 2, True),
                                                 (wl.MXFP4, 64, 2048, 512, 10, True)])
def test_moe_decode_tokens_share_experts(q, fmt, e, h, f, k, shared):
    """Four tokens that all chose the same experts (the fewest groups, so the longest row-tile
    splits over CTAs and the most output parts): the decode chain against the oracle, and the
    routed and pre-routed chains byte for byte."""
    t = 4
    layer = wl.moe_layer(fmt, e, h, f, seed=720 + k, shared=shared)
    x = wl.moe_tokens(t, h, seed=721)
    lg = np.repeat(wl.router_logits(1, e, seed=722), t, axis=0)
    lg[2] *= 0.5  # the same ranking, other weights
    pm = q.PackedMoE(layer)
    xd, lt = dev_bf16(x), torch.from_numpy(np.ascontiguousarray(lg)).cuda()
    ids, w, rws = q.route(lt, k)
    out_a = q.moe_ffn(pm, xd, w, rws)
    out_b, ids_b, w_b, _ = q.moe_forward(pm, xd, lt, k)
    torch.cuda.synchronize()
    assert torch.equal(ids, ids_b) and torch.equal(w, w_b)
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    ref = oracle.moe_forward(layer, x, lg, k)
    err = np.abs(to_f64(out_b) - ref)
    assert np.all(err <= moe_tolerance(oracle, layer, x, lg, k, ref))


@pytest.mark.parametrize("fmt", [wl.MXFP4, wl.NVFP4, wl.MLX_AFFINE4_G64, wl.Q6K])
@pytest.mark.parametrize("t", [1, 2, 4])
def test_moe_decode_small(q, fmt, t):
    E, H, F, k = 16, 512 if fmt == wl.Q6K else 256, 256 if fmt == wl.Q6K else 128, 4
    layer = wl.moe_layer(fmt, E, H, F, seed=300 + fmt, shared=True)
    x = wl.moe_tokens(t, H, seed=301)
    lg = wl.router_logits(t, E, seed=302)
    pm = q.PackedMoE(layer)
    lt = torch.from_numpy(lg).cuda()
    ids, w, rws = q.route(lt, k)
    out = q.moe_ffn(pm, dev_bf16(x), w, rws)
    torch.cuda.synchronize()
    got = to_f64(out)
    ref = oracle.moe_forward(layer, x, lg, k)
    tol = moe_tolerance(oracle, layer, x, lg, k, ref)
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got))
    assert np.all(err <= tol), f"{np.sum(err > tol)} out of tolerance, worst {np.max(err - tol)}"


def test_moe_decode_without_shared(q):
    E, H, F, k, t = 8, 256, 128, 3, 4
    layer = wl.moe_layer(wl.MXFP4, E, H, F, seed=310, shared=False)
    x = wl.moe_tokens(t, H, seed=311)
    lg = wl.router_logits(t, E, seed=312)
    pm = q.PackedMoE(layer)
    ids, w, rws = q.route(torch.from_numpy(lg).cuda(), k)
    out = q.moe_ffn(pm, dev_bf16(x), w, rws)
    torch.cuda.synchronize()
    ref = oracle.moe_forward(layer, x, lg, k)
    assert np.all(np.abs(to_f64(out) - ref) <= moe_tolerance(oracle, layer, x, lg, k, ref))


def test_moe_decode_full_config(q):
    """The MoE decode benchmark layer: 512 MXFP4 experts, hidden 2048, FFN 512, top-10,
    shared expert, 4 tokens; two routings in a row on one workspace (deterministic)."""
    c = wl.MOE_DECODE
    layer = wl.moe_layer(c["fmt"], c["n_experts"], c["hidden"], c["ffn"], seed=0, shared=True)
    pm = q.PackedMoE(layer)
    ws = q.Workspace(q.qmoe_workspace_size(pm.desc, c["tokens"], c["topk"]))
    for rep in range(2):
        x = wl.moe_tokens(c["tokens"], c["hidden"], seed=10 + rep)
        lg = wl.router_logits(c["tokens"], c["n_experts"], seed=20 + rep)
        ids, w, rws = q.route(torch.from_numpy(lg).cuda(), c["topk"])
        out = q.moe_ffn(pm, dev_bf16(x), w, rws, workspace=ws)
        out2 = q.moe_ffn(pm, dev_bf16(x), w, rws, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
        ref = oracle.moe_forward(layer, x, lg, c["topk"])
        tol = moe_tolerance(oracle, layer, x, lg, c["topk"], ref)
        err = np.abs(to_f64(out) - ref)
        assert np.all(err <= tol), f"rep {rep}: {np.sum(err > tol)} out of tolerance"
        assert ws.status() == 0


@pytest.mark.parametrize("fmt", [wl.MXFP4, wl.Q6K])
@pytest.mark.parametrize("t,shared", [(1, True), (4, True), (3, False)])
def test_moe_decode_staged(q, fmt, t, shared):
    """qgemm_grouped one stage at a time: h against the oracle's h of the same (token,
    expert), and the combined output bit-identical to the fused qmoe_ffn chain."""
    E, k = 16, 4
    H, F = (512, 256) if fmt == wl.Q6K else (256, 128)
    layer = wl.moe_layer(fmt, E, H, F, seed=320 + fmt, shared=shared)
    x = wl.moe_tokens(t, H, seed=321)
    lg = wl.router_logits(t, E, seed=322)
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
    assert h.shape[0] == len(rows)
    href = np.stack([inter[r][2] for r in rows])
    err = np.abs(to_f64(h) - href)
    tol = h_tolerance(oracle, layer, x, inter, rows)
    assert np.all(err <= tol), f"{np.sum(err > tol)} h values out of tolerance"


@pytest.mark.parametrize("fmt,t", [(wl.MXFP4, 1), (wl.MXFP4, 4), (wl.NVFP4, 3)])
def test_moe_decode_shared_gate(q, fmt, t):
    """The shared expert weighed by its sigmoid gate (fp32 logits per token): against the
    oracle, the staged chain bit-identical to the fused one, and a saturated gate (+100)
    bit-identical to no gate."""
    E, H, F, k = 16, 256, 128, 4
    layer = wl.moe_layer(fmt, E, H, F, seed=330 + t, shared=True)
    x = wl.moe_tokens(t, H, seed=331)
    lg = wl.router_logits(t, E, seed=332)
    gl = wl.shared_gate_logits(t, seed=333)
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
    tol = moe_tolerance(oracle, layer, x, lg, k, ref)
    err = np.abs(to_f64(out) - ref)
    assert np.all(err <= tol), f"{np.sum(err > tol)} out of tolerance, worst {np.max(err - tol)}"


@pytest.mark.parametrize("t,e,k,shared,fmt", [(1, 16, 4, True, wl.MXFP4), (2, 64, 10, True, wl.NVFP4),
                                              (4, 512, 10, True, wl.MXFP4), (3, 32, 16, False, wl.MLX_AFFINE4_G64),
                                              (4, 16, 16, True, wl.Q6K), (6, 16, 4, True, wl.MXFP4)])
def test_moe_forward_routes_inside_the_chain(q, t, e, k, shared, fmt):
    """qmoe_forward (router and FFN in one call; at 1-4 tokens the gate/up launch routes the
    tokens itself) against qmoe_route + qmoe_ffn on fresh zeroed workspaces: the same output,
    ids, weights and router workspace, byte for byte; and the output against the oracle."""
    H, F = (512, 256) if fmt == wl.Q6K else (256, 128)
    layer = wl.moe_layer(fmt, e, H, F, seed=340 + t, shared=shared)
    x = wl.moe_tokens(t, H, seed=341)
    lg = wl.router_logits(t, e, seed=342)
    if t == 4 and e == 16:
        lg[1] = lg[0]  # two tokens with the same experts: groups of several rows
    pm = q.PackedMoE(layer)
    xd, lt = dev_bf16(x), torch.from_numpy(np.ascontiguousarray(lg)).cuda()
    gl = torch.from_numpy(wl.shared_gate_logits(t, seed=343)).cuda() if shared else None
    rws_a = q.Workspace(q.qmoe_route_workspace_size(t, e, k))
    ids_a, w_a, _ = q.route(lt, k, workspace=rws_a)
    out_a = q.moe_ffn(pm, xd, w_a, rws_a, shared_gate=gl)
    rws_b = q.Workspace(q.qmoe_route_workspace_size(t, e, k))
    out_b, ids_b, w_b, _ = q.moe_forward(pm, xd, lt, k, route_ws=rws_b, shared_gate=gl)
    torch.cuda.synchronize()
    assert torch.equal(ids_a, ids_b) and torch.equal(w_a, w_b)
    assert torch.equal(rws_a.buf, rws_b.buf)
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    ref = oracle.moe_forward(layer, x, lg, k, shared_gate=None if gl is None else gl.cpu().numpy())
    err = np.abs(to_f64(out_b) - ref)
    assert np.all(err <= moe_tolerance(oracle, layer, x, lg, k, ref))
