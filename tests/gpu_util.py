"""Helpers for the GPU parity tests: build/load the library, move logical inputs to the device."""
from __future__ import annotations

import numpy as np
import torch

_built = False


def qlib():
    """Build (if stale) and load the C library; returns the binding module."""
    global _built
    import prefill_dequant_gemv_gb300 as q
    from prefill_dequant_gemv_gb300 import build as b
    if not _built:
        b.build()
        _built = True
    q.lib()
    return q


def dev_bf16(bits: np.ndarray, device="cuda"):
    """bf16 bit patterns [r, c] -> device bf16 tensor view [r, c] whose row stride is a multiple of 8."""
    r, c = bits.shape
    cp = (c + 7) // 8 * 8
    host = np.zeros((r, cp), dtype=np.uint16)
    host[:, :c] = bits
    t = torch.from_numpy(host.view(np.int16)).view(torch.bfloat16).to(device)
    return t[:, :c]


def to_f64(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def moe_tolerance(o, layer, x, lg, topk, out_ref, tokens=None, pair_bf16=None):
    """Per-element bound for a mixture-of-experts output (rows = `tokens`, all by default):
    each expert's down output within the GEMV bound of its (bf16) input h plus one bf16 ulp
    of h (rounding flips between the two sides), weighted by p; plus one output ulp.
    pair_bf16 (default: more than 4 tokens, the prefill chain): each down output is also
    rounded to bf16 before the weighted sum -- half an ulp, at most 2^-9 of the value; the
    bound takes 2^-8 of the oracle's value so that it also covers the kernel's value lying
    within the GEMV bound of it."""
    if pair_bf16 is None:
        pair_bf16 = x.shape[0] > 4
    _, _, ids, p, inter = o.moe_forward(layer, x, lg, topk, tokens=tokens, with_intermediates=True)
    toks = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens)
    tol = np.zeros((toks.size, layer.hidden))
    rn = {}
    pr = 2.0 ** -8 if pair_bf16 else 0.0
    for i, t in enumerate(toks):
        for j in range(topk):
            e = int(ids[t, j])
            if e not in rn:
                rn[e] = float(np.max(o.row_norms(layer.down[e])))
            _, _, h, d = inter[(int(t), e)]
            tol[i] += p[t, j] * ((2e-3 + 2.0 ** -8) * np.linalg.norm(h) * rn[e] + pr * np.abs(d))
        if layer.shared_down is not None:
            _, _, h, d = inter[(int(t), -1)]
            tol[i] += (2e-3 + 2.0 ** -8) * np.linalg.norm(h) * float(np.max(o.row_norms(layer.shared_down))) \
                + pr * np.abs(d)
    return tol + 2.0 ** -7 * np.abs(out_ref)


def grouped_rows(ids, with_shared: bool):
    """(token, expert) of each row of the staged gate/up output: the (token, slot) pairs with
    experts ascending and tokens ascending within an expert, then one shared row per token
    (expert -1)."""
    t, k = ids.shape
    pairs = sorted((int(ids[i, j]), i) for i in range(t) for j in range(k))
    rows = [(i, e) for e, i in pairs]
    if with_shared:
        rows += [(i, -1) for i in range(t)]
    return rows


def h_tolerance(o, layer, x, inter, rows):
    """Per-element bound for the staged h = bf16(silu(g)·u) rows: g and u each within the GEMV
    bound D = 2e-3·||x_t||·max_n||w_n|| of the gate/up weight, propagated through silu(g)·u
    (|d silu/dg| <= 1.1), plus one bf16 ulp of h (a rounding flip between the two sides)."""
    xv = o.bf16_value(x)
    rn = {}
    tol = []
    for t, e in rows:
        w = layer.shared_gate_up if e < 0 else layer.gate_up[e]
        if e not in rn:
            rn[e] = float(np.max(o.row_norms(w)))
        d = 2e-3 * np.linalg.norm(xv[t]) * rn[e]
        g, u, h, _ = inter[(t, e)]
        silu = g / (1.0 + np.exp(-np.clip(g, -80.0, None)))
        tol.append((1.1 * np.abs(u) + np.abs(silu) + 1.1 * d) * d + 2.0 ** -7 * np.abs(h))
    return np.array(tol)
