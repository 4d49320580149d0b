"""Planted mistakes in the oracle (on the CPU) must be caught by the pins.

Each case patches one oracle function with a plausible bug (dropped term, wrong
sign, wrong constant, transposed operand, double rounding, wrong tie-break) and
checks that at least one pin fails.
"""
import sys

import numpy as np
import torch

import oracle
import workloads as wl
from tests import pins

F = sys.modules["oracle.formats"]
G = sys.modules["oracle.gemv"]  # the package re-exports a function under the same name
MO = sys.modules["oracle.moe"]


def _fails(fn, *a, **kw):
    try:
        fn(*a, **kw)
    except (AssertionError, ValueError):
        return True
    return False


def test_e2m1_sign_dropped(monkeypatch):
    orig = F.e2m1_value
    monkeypatch.setattr(oracle, "e2m1_value", lambda c: np.abs(orig(c)))
    assert _fails(pins.check_e2m1, oracle)


def test_e2m1_magnitudes_swapped(monkeypatch):
    orig = F.e2m1_value

    def bad(c):
        c = np.asarray(c)
        swapped = np.where((c & 7) == 3, (c & 8) | 4, np.where((c & 7) == 4, (c & 8) | 3, c))
        return orig(swapped)
    monkeypatch.setattr(oracle, "e2m1_value", bad)
    assert _fails(pins.check_e2m1, oracle)


def test_e4m3_wrong_bias(monkeypatch):
    monkeypatch.setattr(oracle, "e4m3fn_value", lambda b: F.e4m3fn_value(b) / 2)
    assert _fails(pins.check_e4m3, oracle)


def test_e8m0_off_by_one(monkeypatch):
    monkeypatch.setattr(oracle, "e8m0_value", lambda b: F.e8m0_value(np.asarray(b) + 1))
    assert _fails(pins.check_e8m0, oracle)


def test_bf16_double_rounding(monkeypatch):
    def via_fp32(v):
        t = torch.from_numpy(np.asarray(v, np.float64).astype(np.float32)).to(torch.bfloat16)
        return t.to(torch.float64).numpy()
    monkeypatch.setattr(oracle, "round_to_bf16", via_fp32)
    assert _fails(pins.check_bf16_rounding, oracle)


def _patch_exact(monkeypatch, fmt_target, transform):
    orig = F._exact_values

    def bad(fmt, codes, scales, aux, ts):
        v = orig(fmt, codes, scales, aux, ts)
        return transform(v, fmt, codes, scales, aux, ts) if fmt == fmt_target else v
    monkeypatch.setattr(F, "_exact_values", bad)


def test_q6k_zero_point_31(monkeypatch):
    def t(v, fmt, codes, scales, aux, ts):
        sc = np.repeat(np.asarray(scales, np.int8).astype(np.float64), 16, axis=1)
        d = np.repeat(np.asarray(aux, np.float16).astype(np.float64), 256, axis=1)
        return d * sc * (np.asarray(codes, np.float64) - 31.0)
    _patch_exact(monkeypatch, wl.Q6K, t)
    assert _fails(pins.check_q6k_operand, oracle)
    assert _fails(pins.check_dequant_exact, oracle, wl.Q6K)


def test_nvfp4_tensor_scale_dropped(monkeypatch):
    _patch_exact(monkeypatch, wl.NVFP4, lambda v, fmt, c, s, a, ts: v / float(np.float32(ts)))
    assert _fails(pins.check_dequant_exact, oracle, wl.NVFP4)


def test_mlx_bias_sign_flipped(monkeypatch):
    def t(v, fmt, codes, scales, aux, ts):
        b = np.repeat(np.asarray(aux, np.float16).astype(np.float64), 64, axis=1)
        return v - 2 * b
    _patch_exact(monkeypatch, wl.MLX_AFFINE4_G64, t)
    assert _fails(pins.check_dequant_exact, oracle, wl.MLX_AFFINE4_G64)


def test_mxfp4_scale_block_16_instead_of_32(monkeypatch):
    def t(v, fmt, codes, scales, aux, ts):
        s = np.repeat(F.e8m0_value(scales), 16, axis=1)
        s = np.concatenate([s, s], axis=1)[:, :np.asarray(codes).shape[1]]
        return F.e2m1_value(codes) * s
    _patch_exact(monkeypatch, wl.MXFP4, t)
    assert _fails(pins.check_dequant_exact, oracle, wl.MXFP4)


def test_gemv_residual_dropped(monkeypatch):
    orig = G.gemv_rows
    monkeypatch.setattr(oracle, "gemv", lambda w, x, res=None: orig(w, x, np.arange(w.n), None))
    assert _fails(pins.check_gemv_brute_force, oracle, wl.NVFP4, 4, True)


def test_gemv_transposed_operand(monkeypatch):
    def bad(w, x, res=None):
        w32 = F.dequant(w).astype(np.float64)
        v = F.bf16_value(x) @ w32  # W instead of W^T
        return F.round_to_bf16(v), v
    monkeypatch.setattr(oracle, "gemv", bad)
    assert _fails(pins.check_gemv_brute_force, oracle, wl.MXFP4, 1, False)


def test_gemv_wrong_sign(monkeypatch):
    orig = G.gemv_rows

    def bad(w, x, res=None):
        y, v = orig(w, x, np.arange(w.n), res)
        return -y, -v
    monkeypatch.setattr(oracle, "gemv", bad)
    assert _fails(pins.check_dense_special_case, oracle, wl.MLX_AFFINE4_G64)


def test_route_ties_to_higher_index(monkeypatch):
    def bad(logits, topk):
        lg = np.asarray(logits, np.float32)[:, ::-1]
        ids, p = MO.route(lg, topk)
        return lg.shape[1] - 1 - ids, p
    monkeypatch.setattr(oracle, "route", bad)
    assert _fails(pins.check_route_brute_force, oracle)


def test_route_softmax_over_all_experts(monkeypatch):
    def bad(logits, topk):
        ids, _ = MO.route(logits, topk)
        lg = np.asarray(logits, np.float64)
        z = np.exp(lg - lg.max(axis=1, keepdims=True))
        z = z / z.sum(axis=1, keepdims=True)
        return ids, np.take_along_axis(z, ids, axis=1)
    monkeypatch.setattr(oracle, "route", bad)
    assert _fails(pins.check_route_brute_force, oracle)


def test_moe_shared_expert_dropped(monkeypatch):
    orig = MO.moe_forward

    def bad(layer, x, lg, topk, tokens=None, with_intermediates=False):
        l2 = wl.MoELayer(layer.fmt, layer.n_experts, layer.hidden, layer.ffn, layer.gate_up, layer.down, None, None)
        return orig(l2, x, lg, topk, tokens, with_intermediates)
    monkeypatch.setattr(oracle, "moe_forward", bad)
    assert _fails(pins.check_moe_composition, oracle)


def test_moe_routing_weights_dropped(monkeypatch):
    # the finish sums the experts' outputs without their softmax weights
    orig = MO.route
    monkeypatch.setattr(MO, "route", lambda lg, k: (orig(lg, k)[0], np.ones_like(orig(lg, k)[1])))
    assert _fails(pins.check_moe_composition, oracle)


def test_moe_routing_weights_on_the_wrong_slots(monkeypatch):
    # each expert's output weighed by another slot's weight (the slot order reversed)
    orig = MO.route
    monkeypatch.setattr(MO, "route", lambda lg, k: (orig(lg, k)[0], orig(lg, k)[1][:, ::-1]))
    assert _fails(pins.check_moe_composition, oracle)


def test_moe_h_not_rounded_to_bf16(monkeypatch):
    # the mid hands h to the down projection without its 16-bit rounding
    monkeypatch.setattr(MO, "swiglu_bf16", lambda g, u: MO.silu(g) * np.asarray(u, dtype=np.float64))
    assert _fails(pins.check_moe_composition, oracle)


def test_moe_swiglu_swapped(monkeypatch):
    orig = MO.swiglu_bf16
    monkeypatch.setattr(MO, "swiglu_bf16", lambda g, u: orig(u, g))
    assert _fails(pins.check_moe_composition, oracle)


def test_sigmoid_sign_flipped(monkeypatch):
    orig = MO.sigmoid
    monkeypatch.setattr(MO, "sigmoid", lambda l: orig(-np.asarray(l, np.float64)))
    monkeypatch.setattr(oracle, "sigmoid", lambda l: orig(-np.asarray(l, np.float64)))
    assert _fails(pins.check_sigmoid, oracle)
    assert _fails(pins.check_moe_shared_gate, oracle)


def test_shared_gate_on_the_routed_sum(monkeypatch):
    orig = MO.moe_forward

    def bad(layer, x, lg, topk, tokens=None, with_intermediates=False, shared_gate=None):
        if shared_gate is None or layer.shared_gate_up is None:
            return orig(layer, x, lg, topk, tokens, with_intermediates)
        routed = wl.MoELayer(layer.fmt, layer.n_experts, layer.hidden, layer.ffn, layer.gate_up, layer.down, None, None)
        a_r = orig(routed, x, lg, topk, tokens, True)[1]
        a_s = orig(layer, x, lg, topk, tokens, True)
        g = MO.sigmoid(np.asarray(shared_gate, np.float32))[:, None]
        acc = g * a_r + (a_s[1] - a_r)  # the gate on the routed experts instead of the shared one
        out = F.round_to_bf16(acc)
        return (out, acc) + tuple(a_s[2:]) if with_intermediates else out
    monkeypatch.setattr(oracle, "moe_forward", bad)
    assert _fails(pins.check_moe_shared_gate, oracle)


def test_q5_0_zero_point_15(monkeypatch):
    def t(v, fmt, codes, scales, aux, ts):
        d = np.repeat(np.asarray(scales, np.float16).astype(np.float64), 32, axis=1)
        return d * (np.asarray(codes, np.float64) - 15.0)
    _patch_exact(monkeypatch, wl.Q5_0, t)
    assert _fails(pins.check_q5_operand, oracle)
    assert _fails(pins.check_dequant_exact, oracle, wl.Q5_0)


def test_q5_k_min_added(monkeypatch):
    def t(v, fmt, codes, scales, aux, ts):
        sm = np.asarray(scales, np.uint8).astype(np.float64)
        dd = np.asarray(aux, np.float16).astype(np.float64)
        return np.repeat(dd[:, :, 0], 256, axis=1) * np.repeat(sm[:, :, 0], 32, axis=1) * np.asarray(codes, np.float64) \
            + np.repeat(dd[:, :, 1], 256, axis=1) * np.repeat(sm[:, :, 1], 32, axis=1)
    _patch_exact(monkeypatch, wl.Q5_K, t)
    assert _fails(pins.check_dequant_exact, oracle, wl.Q5_K)


def test_q5_1_scale_and_min_swapped(monkeypatch):
    def t(v, fmt, codes, scales, aux, ts):
        d = np.repeat(np.asarray(scales, np.float16).astype(np.float64), 32, axis=1)
        m = np.repeat(np.asarray(aux, np.float16).astype(np.float64), 32, axis=1)
        return m * np.asarray(codes, np.float64) + d
    _patch_exact(monkeypatch, wl.Q5_1, t)
    assert _fails(pins.check_dense_special_case, oracle, wl.Q5_1)
    assert _fails(pins.check_dequant_exact, oracle, wl.Q5_1)


def test_q5_operand_fifth_bit_at_bit_9(monkeypatch):
    def bad(code):
        c = np.asarray(code).astype(np.uint16) & 0x1F
        return (np.uint16(0x3C00) | ((c & 0xF) << 4) | ((c >> 4) << 9)).astype(np.uint16)
    monkeypatch.setattr(oracle, "q5_half_operand_bits", bad)
    assert _fails(pins.check_q5_operand, oracle)


A = sys.modules["oracle.act_quant"]


def _both(monkeypatch, name, fn):
    monkeypatch.setattr(oracle, name, fn)
    monkeypatch.setattr(A, name, fn)


def test_e2m1_encode_ties_down(monkeypatch):
    def bad(q):
        q = np.asarray(q, dtype=np.float32)
        a = np.minimum(np.abs(q.astype(np.float64)), 6.0)
        d = np.abs(a[..., None] - A._E2M1_GRID)
        mag = np.argmax(d == d.min(axis=-1, keepdims=True), axis=-1).astype(np.uint8)  # lower of two
        return mag | (np.signbit(q).astype(np.uint8) << 3)
    _both(monkeypatch, "e2m1_encode", bad)
    assert _fails(pins.check_e2m1_encode, oracle)


def test_e4m3_encode_truncates(monkeypatch):
    def bad(r):
        r = np.asarray(r, dtype=np.float64)
        return np.array([np.searchsorted(A._E4M3_GRID, v, side="right") - 1 for v in r.ravel()],
                        dtype=np.uint8).reshape(r.shape)
    _both(monkeypatch, "e4m3_encode", bad)
    assert _fails(pins.check_e4m3_encode, oracle)


def test_act_quant_divisor_four(monkeypatch):
    orig = A.e4m3_encode
    monkeypatch.setattr(A, "e4m3_encode", lambda r: orig(np.asarray(r, np.float32) * np.float32(1.5)))
    assert _fails(pins.check_act_quant_round_trip, oracle)
    assert _fails(pins.check_act_quant_nearest, oracle)


def test_act_quant_sign_dropped(monkeypatch):
    orig = A.quantize_act_nvfp4

    def bad(x, a):
        c, s, xe, xq = orig(x, a)
        return c & 7, s, np.abs(xe), np.abs(xq)
    _both(monkeypatch, "quantize_act_nvfp4", bad)
    assert _fails(pins.check_act_quant_round_trip, oracle)


def test_act_quant_tensor_scale_dropped(monkeypatch):
    orig = A.quantize_act_nvfp4

    def bad(x, a):
        c, s, xe, xq = orig(x, a)
        return c, s, xe, xe
    _both(monkeypatch, "quantize_act_nvfp4", bad)
    assert _fails(pins.check_act_quant_round_trip, oracle)
    assert _fails(pins.check_w4a4_reduces_to_w4a16, oracle)


def test_w4a4_skips_activation_quantisation(monkeypatch):
    def bad(w, x, a, res=None, rows=None):
        y, v = G.gemv(w, x, res)
        return y, v, None
    _both(monkeypatch, "gemm_w4a4", bad)
    assert _fails(pins.check_w4a4_brute_force, oracle)


# ----------------------------------------------------------------- the parity bound itself
def _bad_tolerance(xnorm_axis=1, reduce=np.max, sample_max=False, keep_res=True):
    """A copy of the oracle's tolerance with one planted change (the same steps otherwise)."""
    def tol(w, x_bits, res_bits=None, rows=None, max_row_norm=None, ref=None):
        x64 = oracle.bf16_value(x_bits)
        xn = np.linalg.norm(x64, axis=xnorm_axis)
        norms = G.row_norms(w, rows if sample_max else None)
        wmax = float(reduce(norms)) if max_row_norm is None else float(max_row_norm)
        ncols = w.n if rows is None else len(rows)
        t = np.repeat((2e-3 * xn * wmax)[:, None], ncols, axis=1) if xn.shape[0] == x64.shape[0] \
            else np.repeat((2e-3 * xn[: x64.shape[0]] * wmax)[:, None], ncols, axis=1)
        if ref is not None:
            t = t + 2.0 ** -7 * np.abs(np.asarray(ref, dtype=np.float64))
        elif res_bits is not None and keep_res:
            r = oracle.bf16_value(res_bits) if rows is None else oracle.bf16_value(np.asarray(res_bits)[:, rows])
            t = t + 2.0 ** -7 * np.abs(r)
        return t
    return tol


def test_row_norms_over_columns(monkeypatch):
    def cols(w, rows=None):
        return np.linalg.norm(oracle.dequant(w).astype(np.float64), axis=0)
    monkeypatch.setattr(G, "row_norms", cols)
    monkeypatch.setattr(oracle, "row_norms", cols)
    assert _fails(pins.check_tolerance_base, oracle)


def test_tolerance_mean_row_norm(monkeypatch):
    monkeypatch.setattr(oracle, "tolerance", _bad_tolerance(reduce=np.mean))
    assert _fails(pins.check_tolerance_base, oracle)


def test_tolerance_activation_norm_over_inputs(monkeypatch):
    monkeypatch.setattr(oracle, "tolerance", _bad_tolerance(xnorm_axis=0))
    assert _fails(pins.check_tolerance_base, oracle)


def test_tolerance_max_over_sampled_rows_only(monkeypatch):
    monkeypatch.setattr(oracle, "tolerance", _bad_tolerance(sample_max=True))
    assert _fails(pins.check_tolerance_base, oracle)


def test_tolerance_residual_term_dropped(monkeypatch):
    monkeypatch.setattr(oracle, "tolerance", _bad_tolerance(keep_res=False))
    assert _fails(pins.check_tolerance_base, oracle)


def test_tolerance_copy_is_faithful():
    """The unmutated copy above passes the pin, so each mutation's failure is its own."""
    import pytest
    mp = pytest.MonkeyPatch()
    try:
        mp.setattr(oracle, "tolerance", _bad_tolerance())
        pins.check_tolerance_base(oracle)
    finally:
        mp.undo()
