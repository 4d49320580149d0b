"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each ``check_*`` takes the oracle package (or a copy with a planted mistake) and
raises AssertionError when the oracle disagrees with the pin.  The normal tests
run them on the real oracle; ``test_oracle_mutations.py`` runs them on oracles
with planted mistakes and expects them to fail.
"""
from __future__ import annotations

import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import torch

import workloads as wl

_HERE = os.path.dirname(os.path.abspath(__file__))
with open(os.path.join(_HERE, "golden", "page_facts.json")) as _f:
    FACTS = json.load(_f)

FMT_KEY = {wl.MLX_AFFINE4_G64: "mlx_affine4_g64", wl.MXFP4: "mxfp4", wl.NVFP4: "nvfp4", wl.Q6K: "q6k",
           wl.Q5_0: "q5_0", wl.Q5_1: "q5_1", wl.Q5_K: "q5_k"}
Q5 = (wl.Q5_0, wl.Q5_1, wl.Q5_K)


def shape_for(fmt, n, k_small):
    """A test shape: formats with a 256-weight super-block need K = 256."""
    return (n, 256) if fmt in (wl.Q6K, wl.Q5_K) else (n, k_small)


# ----------------------------------------------------------------- exact helpers
def frac_round_bf16(fr: Fraction) -> Fraction:
    """Exact round-to-nearest-even of a rational to bf16 (8 significant bits,
    subnormal quantum 2**-133); returns +-inf as float('inf') for overflow."""
    if fr == 0:
        return Fraction(0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** (e - 1) > a:
        e -= 1
    while Fraction(2) ** e <= a:
        e += 1
    q = max(e - 8, -133)
    s = a / (Fraction(2) ** q)
    fl = math.floor(s)
    rem = s - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    r = fl * Fraction(2) ** q
    if r >= Fraction(2) ** 128:
        return sign * float("inf")
    return sign * r


def e2m1_from_page(code: int) -> Fraction:
    """E2M1 value from the page's magnitude set: codes 0..7 take the magnitudes in
    increasing order, bit 3 is the sign."""
    mags = [Fraction(str(v)) for v in FACTS["e2m1_magnitudes"]["value"]]
    v = mags[code & 7]
    return -v if code & 8 else v


def torch_e4m3(byte: int) -> Fraction:
    t = torch.tensor([byte], dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    return Fraction(float(t.item()))


def torch_e8m0(byte: int) -> Fraction:
    t = torch.tensor([byte], dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64)
    return Fraction(float(t.item()))


def exact_weight(w, n: int, k: int) -> Fraction:
    """Exact real value of weight (n, k) written from the format definitions with
    library decoders (numpy fp16, torch fp8) and the page's E2M1 table."""
    c = int(w.codes[n, k])
    if w.fmt == wl.MLX_AFFINE4_G64:
        return Fraction(float(w.scales[n, k // 64])) * c + Fraction(float(w.aux[n, k // 64]))
    if w.fmt == wl.MXFP4:
        return e2m1_from_page(c) * torch_e8m0(int(w.scales[n, k // 32]))
    if w.fmt == wl.NVFP4:
        return Fraction(float(np.float32(w.tensor_scale))) * torch_e4m3(int(w.scales[n, k // 16])) * e2m1_from_page(c)
    if w.fmt == wl.Q6K:
        return Fraction(float(w.aux[n, k // 256])) * int(w.scales[n, k // 16]) * (c - 32)
    if w.fmt == wl.Q5_0:  # GGML Q5_0: d (code - 16)
        return Fraction(float(w.scales[n, k // 32])) * (c - FACTS["_not_from_pages"]["q5_zero_point"]["q5_0"])
    if w.fmt == wl.Q5_1:  # GGML Q5_1: d code + m
        return Fraction(float(w.scales[n, k // 32])) * c + Fraction(float(w.aux[n, k // 32]))
    if w.fmt == wl.Q5_K:  # GGML Q5_K: d sc code - dmin mn
        sc, mn = int(w.scales[n, k // 32, 0]), int(w.scales[n, k // 32, 1])
        d, dmin = Fraction(float(w.aux[n, k // 256, 0])), Fraction(float(w.aux[n, k // 256, 1]))
        return d * sc * c - dmin * mn
    raise ValueError(w.fmt)


def bf16_frac(bits: int) -> Fraction:
    return Fraction(float(np.array([int(bits) << 16], dtype=np.uint32).view(np.float32)[0]))


# ----------------------------------------------------------------- pins
def check_e2m1(o):
    vals = o.e2m1_value(np.arange(16))
    mags = sorted(set(np.abs(vals).tolist()))
    assert mags == [float(v) for v in FACTS["e2m1_magnitudes"]["value"]], mags
    assert np.all(np.diff(vals[:8]) > 0), "codes 0..7 must increase"
    assert np.array_equal(vals[8:], -vals[:8]), "bit 3 is the sign"
    assert np.all(np.signbit(vals[8:])), "codes 8..15 carry the sign bit"


def check_e8m0(o):
    b = np.arange(256)
    got = o.e8m0_value(b)
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert got[127] == 1.0 and np.isnan(got[255])


def check_e4m3(o):
    got = o.e4m3fn_value(np.arange(256))
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.nanmax(got) == 448.0


def check_bf16_rounding(o, seed=1):
    rng = np.random.default_rng(seed)
    # fp32 inputs: torch's fp32 -> bf16 cast rounds once, so both must agree exactly
    a = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),  # subnormals
        np.clip(rng.standard_normal(2000) * 3e38, -3.4e38, 3.4e38).astype(np.float32),  # near overflow
        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -133, 3 * 2 ** -134], np.float32),
    ])
    ref = torch.from_numpy(a).to(torch.bfloat16).to(torch.float64).numpy()
    got = o.round_to_bf16(a.astype(np.float64))
    assert np.array_equal(got, ref), np.nonzero(got != ref)[0][:5]
    # one rounding from fp64: 1 + 2^-8 + 2^-30 rounds up, while fp32 first would make a tie -> 1.0
    v = 1.0 + 2.0 ** -8 + 2.0 ** -30
    assert o.round_to_bf16(np.array([v]))[0] == 1.0 + 2.0 ** -7


def check_bpw(o):
    page = FACTS["bits_per_weight"]["value"]
    for fmt, key in [(wl.MLX_AFFINE4_G64, "mlx_affine4_g64"), (wl.MXFP4, "mxfp4"), (wl.NVFP4, "nvfp4")]:
        assert o.bits_per_weight(fmt) == page[key], key
        c, s, a = o.packed_sizes(fmt, 1024, 2048)
        assert (c + s + a) * 8 / (1024 * 2048) == page[key], key
    q = FACTS["q6k_output_layer"]
    c, s, a = o.packed_sizes(wl.Q6K, q["n"], q["k"])
    total = c + s + a
    assert total == q["n"] * q["k"] * o.bits_per_weight(wl.Q6K) / 8
    assert round(total / 1e9, 2) == q["gigabytes"], total
    for fmt in Q5:  # the GGML block sizes (bytes per block of weights)
        nbytes, nweights = FACTS["_not_from_pages"]["q5_block_bytes"][FMT_KEY[fmt]]
        assert o.bits_per_weight(fmt) == nbytes * 8 / nweights, fmt
        c, s, a = o.packed_sizes(fmt, 1024, 2048)
        assert (c + s + a) * 8 / (1024 * 2048) == nbytes * 8 / nweights, fmt


def check_q6k_operand(o):
    f = FACTS["q6k_operand"]
    codes = np.arange(64)
    half = o.q6k_half_operand_bits(codes).view(np.float16)
    assert np.array_equal(half.astype(np.float64), 1.0 + codes / 64.0)
    diff = (half - np.float16(f["subtract"])).astype(np.float64)  # fp16 arithmetic
    assert np.array_equal(diff, (codes - f["zero_point"]) / 64.0)
    # the oracle's Q6_K dequantisation must use the same zero point
    w = wl.QWeight(wl.Q6K, 1, 256, codes=np.tile(np.arange(64, dtype=np.uint8), 4)[None, :],
                   scales=np.ones((1, 16), np.int8), aux=np.ones((1, 1), np.float16))
    got = o.dequant(w)[0].astype(np.float64)
    assert np.array_equal(got, 64.0 * np.tile(diff, 4))


def check_q5_operand(o):
    """The 5-bit operand is 1 + code/64 for every 5-bit code, and Q5_0's dequantisation
    uses zero point 16 (GGML; the page's "as ZeroAsMin": d (code - 16) = d code - 16 d)."""
    f = FACTS["q5_operand"]
    codes = np.arange(f["max_exact_code"] + 1)
    bits = o.q5_half_operand_bits(codes)
    assert np.array_equal(bits.view(np.float16).astype(np.float64), f["operand_base"] + codes * f["operand_step"])
    assert np.array_equal((bits >> f["fifth_bit"]) & 1, codes >> 4)
    zp = FACTS["_not_from_pages"]["q5_zero_point"]["q5_0"]
    w = wl.QWeight(wl.Q5_0, 1, 64, codes=np.tile(np.arange(32, dtype=np.uint8), 2)[None, :],
                   scales=np.ones((1, 2), np.float16))
    assert np.array_equal(o.dequant(w)[0].astype(np.float64), np.tile(np.arange(32) - zp, 2).astype(np.float64))
    # ZeroAsMin: the same weights as a Q5_1 block with m = -16 d
    w1 = wl.QWeight(wl.Q5_1, 1, 64, codes=w.codes, scales=np.full((1, 2), 0.25, np.float16),
                    aux=np.full((1, 2), -zp * 0.25, np.float16))
    w0 = wl.QWeight(wl.Q5_0, 1, 64, codes=w.codes, scales=np.full((1, 2), 0.25, np.float16))
    assert np.array_equal(o.dequant(w1), o.dequant(w0))


def check_q6k_old_seed(seed=3):
    """(128 + c) operands seeded with -160 * sum(x) give the same exact dot as (c - 32)."""
    f = FACTS["q6k_old_seed"]
    rng = np.random.default_rng(seed)
    for _ in range(20):
        c = rng.integers(0, 64, f["chain"])
        x = [Fraction(int(v), 1024) for v in rng.integers(-4096, 4096, f["chain"])]
        old = sum((f["operand_offset"] + int(ci)) * xi for ci, xi in zip(c, x)) + f["seed_per_input"] * sum(x)
        new = sum((int(ci) - FACTS["q6k_operand"]["zero_point"]) * xi for ci, xi in zip(c, x))
        assert old == new


def check_dequant_exact(o, fmt, seed=5):
    n, k = shape_for(fmt, 8, 128)
    w = wl.weight(fmt, n, k, seed)
    got = o.dequant(w)
    for i in range(n):
        for j in range(k):
            ex = exact_weight(w, i, j)
            assert Fraction(float(ex)) == ex  # exactly representable in fp64
            assert got[i, j] == np.float32(float(ex)), (fmt, i, j)


def check_gemv_brute_force(o, fmt, m, residual, seed=7):
    n, k = shape_for(fmt, 16, 64)
    w, x, res = wl.gemv_case(fmt, n, k, m, seed=seed, residual=residual)
    y, v = o.gemv(w, x, res)
    w32 = o.dequant(w)
    for mi in range(m):
        for ni in range(n):
            terms = [Fraction(float(w32[ni, kk])) * bf16_frac(x[mi, kk]) for kk in range(k)]
            ex = sum(terms, Fraction(0))
            if res is not None:
                ex += bf16_frac(res[mi, ni])
            mag = float(sum(abs(t) for t in terms)) + (abs(float(bf16_frac(res[mi, ni]))) if res is not None else 0)
            bound = (k + 2) * 2.0 ** -52 * mag
            assert abs(Fraction(float(v[mi, ni])) - ex) <= Fraction(bound), (fmt, mi, ni)
            lo, hi = frac_round_bf16(ex - Fraction(bound)), frac_round_bf16(ex + Fraction(bound))
            if lo == hi:
                assert Fraction(float(y[mi, ni])) == lo, (fmt, mi, ni, float(y[mi, ni]), float(lo))
            else:
                assert Fraction(float(y[mi, ni])) in (lo, hi)


def check_dense_special_case(o, fmt, seed=11):
    """Unit scales reduce every format to a dense matmul of its integer / E2M1 values."""
    (n, k), m = shape_for(fmt, 32, 128), 3
    w, x, _ = wl.gemv_case(fmt, n, k, m, seed=seed)
    if fmt == wl.MLX_AFFINE4_G64:
        w.scales = np.ones_like(w.scales)
        w.aux = np.zeros_like(w.aux)
        dense = w.codes.astype(np.float64)
    elif fmt == wl.MXFP4:
        w.scales = np.full_like(w.scales, 127)
        dense = np.vectorize(lambda c: float(e2m1_from_page(int(c))))(w.codes)
    elif fmt == wl.NVFP4:
        w.scales = np.full_like(w.scales, 0x38)  # E4M3 1.0
        w.tensor_scale = 1.0
        dense = np.vectorize(lambda c: float(e2m1_from_page(int(c))))(w.codes)
    elif fmt == wl.Q6K:
        w.scales = np.ones_like(w.scales)
        w.aux = np.ones_like(w.aux)
        dense = w.codes.astype(np.float64) - 32.0
    elif fmt == wl.Q5_0:
        w.scales = np.ones_like(w.scales)
        dense = w.codes.astype(np.float64) - 16.0
    elif fmt == wl.Q5_1:
        w.scales = np.ones_like(w.scales)
        w.aux = np.zeros_like(w.aux)
        dense = w.codes.astype(np.float64)
    else:  # Q5_K: sc = 1, mn = 0, d = 1
        w.scales = np.stack([np.ones_like(w.scales[..., 0]), np.zeros_like(w.scales[..., 1])], axis=-1)
        w.aux = np.ones_like(w.aux)
        dense = w.codes.astype(np.float64)
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(torch.float64)
    ref = torch.matmul(xt, torch.from_numpy(dense).T).numpy()
    _, v = o.gemv(w, x)
    assert np.allclose(v, ref, rtol=1e-12, atol=1e-12)


def check_route_brute_force(o, seed=13):
    rng = np.random.default_rng(seed)
    for _ in range(30):
        t, e, kk = 3, 8, 3
        lg = rng.integers(-3, 3, size=(t, e)).astype(np.float32)  # many ties
        ids, p = o.route(lg, kk)
        for ti in range(t):
            # rank-based definition: e is kept iff fewer than k experts beat it
            beats = [sum(1 for f in range(e) if lg[ti, f] > lg[ti, g] or (lg[ti, f] == lg[ti, g] and f < g))
                     for g in range(e)]
            chosen = [g for g in range(e) if beats[g] < kk]
            assert sorted(ids[ti].tolist()) == chosen
            assert [beats[g] for g in ids[ti]] == list(range(kk)), "descending order, ties to lower index"
            z = np.exp(lg[ti, ids[ti]].astype(np.float64) - lg[ti, ids[ti]].max())
            assert np.allclose(p[ti], z / z.sum(), rtol=1e-15)
    # permutation invariance of the weights
    lg = rng.standard_normal((5, 64)).astype(np.float32)
    perm = rng.permutation(64)
    ids, p = o.route(lg, 10)
    ids2, p2 = o.route(lg[:, perm], 10)
    assert np.array_equal(perm[ids2], ids) and np.array_equal(p, p2)
    assert np.allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-15)


def check_route_statistics(o):
    r = FACTS["routing"]
    e, kk, t = r["experts"], r["topk"], r["decode_rows"]
    closed = e * (1 - (1 - kk / e) ** t)
    lg = wl.router_logits(t, e, seed=17, sets=3000)
    distinct = [len(np.unique(o.route(lg[s], kk)[0])) for s in range(lg.shape[0])]
    mean = float(np.mean(distinct))
    assert abs(mean - closed) < 0.15, (mean, closed)
    assert round(mean) == r["distinct_experts_synthetic"]
    big = wl.router_logits(r["prefill_tokens"], e, seed=19)
    ids, _ = o.route(big, kk)
    counts = np.bincount(ids.ravel(), minlength=e)
    assert counts.sum() / e == r["tokens_per_expert"]
    assert counts.min() > 80 and counts.max() < 260  # binomial(8192, 10/512) spread


def check_silu(o, seed=23):
    assert o.silu(np.array([0.0]))[0] == 0.0
    assert o.silu(np.array([60.0]))[0] == 60.0
    assert abs(o.silu(np.array([-60.0]))[0]) < 1e-24
    g = np.random.default_rng(seed).standard_normal(1000) * 6
    ref = torch.nn.functional.silu(torch.from_numpy(g)).numpy()
    assert np.allclose(o.silu(g), ref, rtol=1e-14, atol=0)


def check_sigmoid(o, seed=24):
    """sigmoid(0) = 1/2, the symmetry sigmoid(l) + sigmoid(-l) = 1, saturation, and the
    library routine on random logits."""
    assert o.sigmoid(np.array([0.0]))[0] == 0.5
    assert o.sigmoid(np.array([800.0]))[0] == 1.0 and o.sigmoid(np.array([-800.0]))[0] == 0.0
    l = np.random.default_rng(seed).standard_normal(1000) * 8
    assert np.allclose(o.sigmoid(l) + o.sigmoid(-l), 1.0, rtol=0, atol=1e-15)
    ref = torch.sigmoid(torch.from_numpy(l)).numpy()
    assert np.allclose(o.sigmoid(l), ref, rtol=1e-14, atol=0)


def check_moe_shared_gate(o, seed=30):
    """The shared expert's sigmoid gate scales only the shared expert's output: with the
    routed-only sum a_r (no shared expert) and the ungated sum a_s, the gated sum is
    a_r + sigmoid(l) (a_s - a_r) per token; a zero logit halves the shared output, and a
    very large logit gives the ungated layer."""
    layer = wl.moe_layer(wl.MXFP4, 6, 64, 32, seed=seed, shared=True)
    routed = wl.MoELayer(layer.fmt, 6, 64, 32, layer.gate_up, layer.down, None, None)
    x = wl.moe_tokens(4, 64, seed=seed)
    lg = wl.router_logits(4, 6, seed=seed)
    gate = np.array([0.0, 1.5, -2.25, 100.0], np.float32)
    a_r = o.moe_forward(routed, x, lg, topk=2, with_intermediates=True)[1]
    a_s = o.moe_forward(layer, x, lg, topk=2, with_intermediates=True)[1]
    out, a_g = o.moe_forward(layer, x, lg, topk=2, with_intermediates=True, shared_gate=gate)[:2]
    sg = 1.0 / (1.0 + np.exp(-gate.astype(np.float64)))
    assert np.allclose(a_g, a_r + sg[:, None] * (a_s - a_r), rtol=1e-12, atol=1e-12)
    assert np.allclose(a_g[0], a_r[0] + 0.5 * (a_s[0] - a_r[0]), rtol=1e-12, atol=1e-12)
    assert np.array_equal(a_g[3], a_s[3])
    assert np.array_equal(out, o.round_to_bf16(a_g))
    ungated = o.moe_forward(layer, x, lg, topk=2)
    assert np.array_equal(o.moe_forward(layer, x, lg, topk=2, shared_gate=np.full(4, 100.0, np.float32)), ungated)


def _expert_by_gemv(o, gu, dn, x_row, f):
    """One expert on one token through the dense GEMV oracle: gate/up GEMV (fp32 outputs),
    h = bf16(silu(g)·u), down GEMV of h (fp64 value before rounding)."""
    _, v = o.gemv(gu, x_row)
    g, u = v[0, :f].astype(np.float32), v[0, f:].astype(np.float32)
    h = o.round_to_bf16(o.silu(g) * u.astype(np.float64))
    return o.gemv(dn, o.bf16_bits_of(h)[None, :])[1][0]


def check_moe_composition(o, seed=29):
    """The MoE chain against the dense GEMV oracle: top-1 routing (p = 1) through one
    expert equals gate/up GEMV -> SwiGLU -> down GEMV; top-3 routing equals the sum of the
    three experts' chains, each times its own slot's softmax weight, plus the shared
    expert's; and relabelling the experts (with the logits) leaves the output unchanged."""
    layer = wl.moe_layer(wl.MXFP4, 6, 64, 32, seed=seed, shared=True)
    x = wl.moe_tokens(3, 64, seed=seed)
    lg = wl.router_logits(3, 6, seed=seed)
    out = o.moe_forward(layer, x, lg, topk=1)
    ids, p = o.route(lg, 1)
    assert np.all(p == 1.0)
    for t in range(3):
        acc = np.zeros(64)
        for gu, dn in [(layer.gate_up[ids[t, 0]], layer.down[ids[t, 0]]), (layer.shared_gate_up, layer.shared_down)]:
            acc += _expert_by_gemv(o, gu, dn, x[t:t + 1], 32)
        assert np.array_equal(out[t], o.round_to_bf16(acc)), t
    # top-3 on logits with well-separated values (a different order per token): distinct
    # weights per slot, so a weight on the wrong slot or no weight shows
    rng = np.random.default_rng(seed)
    lg3 = np.stack([rng.permutation(np.array([2.0, 1.0, 0.25, -0.5, -1.0, -2.0], np.float32)) for _ in range(3)])
    _, acc3, ids3, _, _ = o.moe_forward(layer, x, lg3, topk=3, with_intermediates=True)
    rids, rp = o.route(lg3, 3)
    assert np.array_equal(ids3, rids)
    assert np.all(np.abs(np.diff(rp, axis=1)) > 1e-3)
    for t in range(3):
        want = _expert_by_gemv(o, layer.shared_gate_up, layer.shared_down, x[t:t + 1], 32)
        for j in range(3):
            e = int(rids[t, j])
            want = want + rp[t, j] * _expert_by_gemv(o, layer.gate_up[e], layer.down[e], x[t:t + 1], 32)
        assert np.allclose(acc3[t], want, rtol=1e-12, atol=1e-12 * np.max(np.abs(want))), t
    perm = np.random.default_rng(seed).permutation(6)  # new index i holds old expert perm[i]
    layer2 = wl.MoELayer(layer.fmt, 6, 64, 32, [layer.gate_up[j] for j in perm], [layer.down[j] for j in perm],
                         layer.shared_gate_up, layer.shared_down)
    lg2 = wl.router_logits(3, 6, seed=seed + 1)
    a1 = o.moe_forward(layer, x, lg2, topk=3, with_intermediates=True)[1]
    a2 = o.moe_forward(layer2, x, lg2[:, perm], topk=3, with_intermediates=True)[1]
    assert np.allclose(a1, a2, rtol=1e-12, atol=0)
    # all experts, equal logits: p = 1/E for every slot
    eq = np.zeros((3, 6), np.float32)
    _, p = o.route(eq, 6)
    assert np.allclose(p, 1 / 6, rtol=1e-15)


def check_operand_bf16(o, fmt, seed=31):
    """The bf16 prefill operand: exact for the E2M1 formats (rounding changes nothing and
    the NVFP4 tensor scale times the operand rounds to the fp32 weight); one extra
    rounding of the fp32 weight for MLX affine, Q6_K and the 5-bit formats."""
    n, k = shape_for(fmt, 8, 128)
    w = wl.weight(fmt, n, k, seed)
    op = o.dequant_operand_bf16(w)
    w32 = o.dequant(w).astype(np.float64)
    if fmt in (wl.MXFP4, wl.NVFP4):
        exact = np.array([[float(exact_weight(w, i, j) / (Fraction(float(np.float32(w.tensor_scale)))
                                                            if fmt == wl.NVFP4 else 1)) for j in range(k)]
                          for i in range(n)])
        assert np.array_equal(op, exact)
        ts = float(np.float32(w.tensor_scale)) if fmt == wl.NVFP4 else 1.0
        assert np.array_equal((op * ts).astype(np.float32).astype(np.float64), w32)
    else:
        ref = torch.from_numpy(w32.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
        assert np.array_equal(op, ref)


def check_tolerance_output_ulp(o, seed=37):
    """The output term of the tolerance, max(2**-7 |ref|, 2**-133), is at least the gap
    between ref and either bf16 neighbour (so two sides rounding one exact value to
    neighbouring bf16 numbers stay inside it) -- for normal outputs and for bf16's
    subnormals, whose spacing is 2**-133 -- and is a strict bound: a flip of two ulps is
    outside it."""
    rng = np.random.default_rng(seed)
    v = o.round_to_bf16(np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-3, 4, 2000),
                                        rng.standard_normal(500) * 2.0 ** -128,  # subnormal bf16
                                        rng.standard_normal(100) * 2.0 ** -125]))
    v = v[v != 0]
    bits = o.bf16_bits_of(v).astype(np.int32)
    up = o.bf16_value((bits + 1).astype(np.uint16))    # next bf16 away from zero (sign-magnitude)
    down = o.bf16_value((bits - 1).astype(np.uint16))  # next bf16 toward zero
    gap = np.maximum(2.0 ** -7 * np.abs(v), 2.0 ** -133)
    assert np.all(np.abs(up) > np.abs(v)) and np.all(np.abs(down) < np.abs(v))
    assert np.all(np.abs(up - v) <= gap)
    assert np.all(np.abs(v - down) <= gap)
    assert np.all(np.abs(up - down) > gap)  # two ulps apart: outside the term
    sub = np.abs(v) < 2.0 ** -126
    assert sub.sum() > 100 and np.all(np.abs(up - v)[sub] == 2.0 ** -133)
    w = wl.weight(wl.NVFP4, 4, 64, seed)
    x = wl.activations(2, 64, seed)
    ref, _ = o.gemv(w, x)
    tol = o.tolerance(w, x, ref=ref)
    base = o.tolerance(w, x)
    assert np.allclose(tol - base, np.maximum(2.0 ** -7 * np.abs(ref), 2.0 ** -133), rtol=1e-12, atol=0)


def _exact_norm(values) -> float:
    """sqrt of an exact rational sum of squares, correctly rounded to fp64 (the integer
    square root of the scaled sum fixes 60 bits before the one rounding)."""
    s = sum((Fraction(v) * Fraction(v) for v in values), Fraction(0))
    if s == 0:
        return 0.0
    e = (s.numerator.bit_length() - s.denominator.bit_length()) // 2 - 62
    scaled = s / (Fraction(4) ** e)  # s = scaled * 2^(2e), scaled ~ 2^124
    r = math.isqrt(scaled.numerator // scaled.denominator)
    return math.ldexp(float(r), e)


def check_tolerance_base(o, seed=67):
    """The stated bound 2e-3 * ||x_m||_2 * max_n ||w_n||_2, pinned with norms taken here in
    exact rational arithmetic from the format definitions (``exact_weight``) and the bf16
    activation values:
      - ``row_norms`` returns one norm per output row n of the N x K weight, in row order;
      - the base term (no residual, no ``ref``) is that product for every output of row m;
      - with ``rows=`` the max still runs over every row of w (the bound is the weight's,
        not the sample's), and the residual term 2**-7 |res| follows the selected columns.
    A norm over the wrong axis, a mean for the max, a sample-only max or a dropped residual
    term each fail one of these."""
    for fmt in (wl.NVFP4, wl.Q6K, wl.MLX_AFFINE4_G64):
        n, k = shape_for(fmt, 12, 64)
        m = 3
        w, x, res = wl.gemv_case(fmt, n, k, m, seed=seed, residual=True)
        # row 5 made clearly the largest (its scales raised), so a max over a sample that
        # skips it differs from the max over the weight
        if fmt == wl.NVFP4:  # every block of row 5 at twice the largest scale (E4M3 byte + 8)
            w.scales[5] = int(w.scales.max()) + 8
        elif fmt == wl.Q6K:
            w.aux[5] = (2.0 * w.aux.astype(np.float32).max()).astype(w.aux.dtype)
        else:
            w.scales[5] = (w.scales[5].astype(np.float32) * 4).astype(w.scales.dtype)
            w.aux[5] = (w.aux[5].astype(np.float32) * 4).astype(w.aux.dtype)
        wn = np.array([_exact_norm(exact_weight(w, i, j) for j in range(k)) for i in range(n)])
        xn = np.array([_exact_norm(bf16_frac(x[mi, j]) for j in range(k)) for mi in range(m)])
        assert int(np.argmax(wn)) == 5, wn
        got = np.asarray(o.row_norms(w), dtype=np.float64)
        assert got.shape == (n,), got.shape
        assert np.allclose(got, wn, rtol=1e-6, atol=0), (fmt, got, wn)
        sub = np.array([0, 2, 9])  # excludes the largest row
        assert np.allclose(np.asarray(o.row_norms(w, sub)), wn[sub], rtol=1e-6, atol=0)
        want = 2e-3 * xn[:, None] * wn.max()
        base = np.asarray(o.tolerance(w, x), dtype=np.float64)
        assert base.shape == (m, n), base.shape
        assert np.allclose(base, np.repeat(want, n, axis=1), rtol=1e-6, atol=0), fmt
        tr = np.asarray(o.tolerance(w, x, res_bits=res, rows=sub), dtype=np.float64)
        rv = np.array([[float(bf16_frac(res[mi, c])) for c in sub] for mi in range(m)])
        assert tr.shape == (m, sub.size), tr.shape
        assert np.allclose(tr, want + 2.0 ** -7 * np.abs(rv), rtol=1e-6, atol=0), fmt


# ----------------------------------------------------------------- W4A4 (activations to NVFP4)
def _e2m1_closed_form(v: np.ndarray) -> np.ndarray:
    """Nearest-even E2M1 magnitude by a closed form: below 2 the grid has step 1/2, from
    2 to 4 step 1, from 4 step 2 up to 6; np.round rounds half to even, and at each step
    change the even neighbour is the power of two."""
    a = np.abs(v.astype(np.float64))
    return np.where(a < 2, np.round(2 * a) / 2, np.where(a < 4, np.round(a), np.minimum(6.0, 2 * np.round(a / 2))))


def check_e2m1_encode(o, seed=41):
    """E2M1 encoding: each code's own value maps back to it; midpoints, their fp32
    neighbours and random values match the closed form; the sign bit follows the input's."""
    codes = np.arange(16)
    assert np.array_equal(o.e2m1_encode(o.e2m1_value(codes).astype(np.float32)), codes)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float32)
    mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)
    rng = np.random.default_rng(seed)
    v = np.concatenate([grid, mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(100)),
                        rng.uniform(0, 9, 4000).astype(np.float32), np.float32([7.0, 1e30])])
    v = np.concatenate([v, -v]).astype(np.float32)
    got = o.e2m1_encode(v)
    want = _e2m1_closed_form(v)
    mag = np.abs(np.vectorize(lambda c: float(e2m1_from_page(int(c))))(got))
    assert np.array_equal(mag, want), v[mag != want][:8]
    assert np.array_equal((got >> 3) & 1, np.signbit(v).astype(np.uint8))
    assert int(o.e2m1_encode(np.float32([-0.0]))[0]) == 8 and int(o.e2m1_encode(np.float32([0.1]))[0]) == 0


def check_e4m3_encode(o, seed=43):
    """E4M3 encoding: every finite code maps back to itself; values up to 448 (midpoints,
    their fp32 neighbours, log-uniform draws) match torch's float8_e4m3fn conversion
    (round to nearest even); larger values saturate at 448 (0x7E)."""
    codes = np.arange(0x7F)
    assert np.array_equal(o.e4m3_encode(o.e4m3fn_value(codes).astype(np.float32)), codes)
    vals = o.e4m3fn_value(codes)
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)
    rng = np.random.default_rng(seed)
    v = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)),
                        np.exp2(rng.uniform(-12, np.log2(448.0), 4000)).astype(np.float32)])
    v = v[v <= 448].astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = o.e4m3_encode(v)
    assert np.array_equal(got, ref), v[got != ref][:8]
    assert np.all(o.e4m3_encode(np.float32([448.0, 460.0, 464.0, 1e4, 3e38])) == 0x7E)
    assert int(o.e4m3_encode(np.float32([0.0]))[0]) == 0


def exact_nvfp4_activations(m: int, k: int, act_scale: float, seed: int):
    """Activations that NVFP4 represents exactly: x = act_scale * E4M3(S) * E2M1(c) per
    block of 16 with one magnitude-6 code per block, act_scale a power of two.  Built
    with torch's E4M3 decoder and the page's E2M1 table; returns (x bf16 bits, c, S)."""
    rng = np.random.default_rng(seed)
    c = rng.integers(0, 16, (m, k)).astype(np.uint8)
    c[c == 8] = 0  # -0 has no exact rational: keep zeros positive here (check_e2m1_encode pins -0)
    blocks = c.reshape(m, k // 16, 16)
    pos = rng.integers(0, 16, (m, k // 16))
    sign = rng.integers(0, 2, (m, k // 16)).astype(np.uint8) << 3
    np.put_along_axis(blocks, pos[..., None], (7 | sign)[..., None], axis=2)
    s = rng.integers(0x10, 0x70, (m, k // 16)).astype(np.uint8)
    sv = np.vectorize(lambda b: float(torch_e4m3(int(b))))(s)
    ev = np.vectorize(lambda q: float(e2m1_from_page(int(q))))(c)
    x = act_scale * np.repeat(sv, 16, axis=1) * ev
    bits = (x.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    assert np.array_equal(bf16_value_np(bits), x), "the construction must be bf16-exact"
    return bits, c, s


def bf16_value_np(bits) -> np.ndarray:
    return (np.asarray(bits).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def check_act_quant_round_trip(o, seed=47):
    """Activations NVFP4 represents exactly (one magnitude-6 code per block) come back as
    the same codes, the same E4M3 scales and the same values, for several power-of-two
    tensor scales.  A wrong block size, divisor, scale order or sign rule breaks it."""
    for i, a in enumerate((1.0, 0.125, 32.0)):
        bits, c, s = exact_nvfp4_activations(3, 96, a, seed + i)
        codes, scales, xe, xq = o.quantize_act_nvfp4(bits, a)
        assert np.array_equal(scales, s), a
        assert np.array_equal(codes, c), a
        assert np.array_equal(xq, bf16_value_np(bits)), a
        assert np.array_equal(xe, bf16_value_np(bits) / a), a


def check_act_quant_nearest(o, seed=53):
    """On arbitrary activations: each block's scale is a nearest E4M3 value to
    amax / (6 act_scale), and each quantised value is a nearest point of its block's grid
    act_scale * E4M3(S) * (+-E2M1) to x (up to the fp32 rounding of the division), with
    x's sign; all-zero blocks give zero scales and codes."""
    rng = np.random.default_rng(seed)
    m, k = 4, 256
    x = rng.standard_normal((m, k)) * np.exp2(rng.integers(-12, 12, (m, 1)))
    x[1, :16] = 0.0
    x[2, 16:32] *= 1e-30  # far below act_scale * 2**-9 * 6: the scale rounds to 0
    bits = wl.bf16_bits_from_f32(x.astype(np.float32))
    xv = bf16_value_np(bits)
    grid_e4 = np.array([float(torch_e4m3(b)) for b in range(0x7F)])
    grid_e2 = np.array([float(e2m1_from_page(c)) for c in range(8)])
    for a in (1.0, 0.37, 3e-3):
        codes, scales, xe, xq = o.quantize_act_nvfp4(bits, a)
        for i in range(m):
            for b in range(k // 16):
                blk = xv[i, 16 * b:16 * b + 16]
                r = np.abs(blk).max() / (6 * float(np.float32(a)))
                sf = float(torch_e4m3(int(scales[i, b])))
                assert abs(sf - r) <= np.min(np.abs(grid_e4 - r)) * (1 + 1e-6) + 1e-300, (a, i, b)
                step = float(np.float32(a)) * sf
                for j in range(16):
                    xj, qj = blk[j], xq[i, 16 * b + j]
                    best = np.min(np.abs(step * grid_e2 - abs(xj)))
                    assert abs(abs(qj) - abs(xj)) <= best + 2.0 ** -20 * abs(xj) + 1e-300, (a, i, b, j)
                    assert qj == 0 or np.sign(qj) == np.sign(xj)
                    assert ((codes[i, 16 * b + j] >> 3) & 1) == int(np.signbit(xj))
        assert np.all(scales[1, 0] == 0) and np.all(codes[1, :16] == 0)
        assert scales[2, 1] == 0 and np.all(xq[2, 16:32] == 0)


def check_w4a4_reduces_to_w4a16(o, seed=59):
    """With activations NVFP4 represents exactly, the W4A4 GEMM is the W4A16 GEMM of the
    same activations, bit for bit (a residual included)."""
    w = wl.weight(wl.NVFP4, 48, 96, seed)
    for a in (1.0, 0.25):
        bits, _, _ = exact_nvfp4_activations(3, 96, a, seed + 1)
        res = wl.activations(3, 48, seed=seed + 2, stream="residual")
        y4, v4, _ = o.gemm_w4a4(w, bits, a, res)
        y16, v16 = o.gemv(w, bits, res)
        assert np.array_equal(y4, y16) and np.allclose(v4, v16, rtol=1e-15, atol=0)


def check_w4a4_brute_force(o, seed=61):
    """W4A4 outputs against exact rationals: sum_k fp32(w) * act_scale * E4M3(S) * E2M1(c)
    with the scales and codes the oracle chose (those are pinned above), one bf16 rounding."""
    w = wl.weight(wl.NVFP4, 6, 32, seed)
    bits = wl.activations(2, 32, seed=seed + 1)
    a = 0.37
    y, v, _ = o.gemm_w4a4(w, bits, a)
    codes, scales, _, _ = o.quantize_act_nvfp4(bits, a)
    w32 = o.dequant(w)
    af = Fraction(float(np.float32(a)))
    for mi in range(2):
        for ni in range(6):
            terms = [Fraction(float(w32[ni, kk])) * af * torch_e4m3(int(scales[mi, kk // 16]))
                     * e2m1_from_page(int(codes[mi, kk])) for kk in range(32)]
            ex = sum(terms, Fraction(0))
            bound = 34 * 2.0 ** -52 * float(sum(abs(t) for t in terms))
            assert abs(Fraction(float(v[mi, ni])) - ex) <= Fraction(bound), (mi, ni)
            lo, hi = frac_round_bf16(ex - Fraction(bound)), frac_round_bf16(ex + Fraction(bound))
            assert Fraction(float(y[mi, ni])) in (lo, hi), (mi, ni)
