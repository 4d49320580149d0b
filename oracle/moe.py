"""Reference mixture-of-experts FFN (oracle; test infrastructure only).

Steps, in the order of the TurboEXL3 article §4.1 (prefill chain) and §4.2
(decode chain):

1. Route: each token keeps its top-k experts by router logit and weighs them by
   a softmax over those k logits (§4.2 names the router's top-k and softmax).
   Reading: ties go to the lower expert index; the softmax is over the k kept
   logits (the same as a softmax over all experts renormalised over the k).
2. Gate and up: one projection of 2F rows per expert; rows 0..F-1 are the gate,
   rows F..2F-1 the up projection (reading).  Each output is the fp64 dot
   product rounded to fp32.
3. Mid: SwiGLU in 32-bit or wider, h = silu(gate) * up, rounded to bf16 as the
   16-bit input of the down projection (§4.1 "Mid").
4. Down: the expert's H x F projection of h, fp64.
5. Finish: the score-weighted sum of each token's k expert outputs plus the
   shared expert's output times its sigmoid gate, rounded to bf16 once (§4.1
   "Finish"; §4.2 names the shared expert's sigmoid gate, a multiply and an add).
   Reading: the gate is sigmoid(l_t) of one logit per token, which the caller
   supplies as it supplies the router's logits; without gate logits the shared
   expert enters with weight 1.
"""
from __future__ import annotations

import numpy as np

from .formats import bf16_value, dequant, round_to_bf16


def route(logits, topk: int):
    """(ids [T, topk] int64 in descending-logit order, p [T, topk] fp64 softmax
    weights) from fp32 logits [T, E]."""
    lg = np.asarray(logits, dtype=np.float32)
    t, e = lg.shape
    if not 1 <= topk <= e:
        raise ValueError("topk out of range")
    order = np.argsort(-lg.astype(np.float64), axis=1, kind="stable")[:, :topk]
    sel = np.take_along_axis(lg, order, axis=1).astype(np.float64)
    z = np.exp(sel - sel[:, :1])
    p = z / z.sum(axis=1, keepdims=True)
    return order.astype(np.int64), p


def sigmoid(l) -> np.ndarray:
    """sigmoid(l) = 1 / (1 + exp(-l)) in fp64."""
    l = np.asarray(l, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-l))


def silu(g) -> np.ndarray:
    """silu(g) = g / (1 + exp(-g)) in fp64."""
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def swiglu_bf16(g, u) -> np.ndarray:
    """h = RN_bf16(silu(g) * u) with the product in fp64 (§4.1 "Mid")."""
    return round_to_bf16(silu(g) * np.asarray(u, dtype=np.float64))


def expert_ffn(gu_w32: np.ndarray, dn_w32: np.ndarray, x64: np.ndarray):
    """One expert on token rows x64 [T, H]: returns (g, u, h, d) with g, u fp32-rounded
    [T, F], h bf16-exact [T, F] and d the fp64 down output [T, H]."""
    f = gu_w32.shape[0] // 2
    gu = (x64 @ gu_w32.astype(np.float64).T).astype(np.float32).astype(np.float64)
    g, u = gu[:, :f], gu[:, f:]
    h = swiglu_bf16(g, u)
    d = h @ dn_w32.astype(np.float64).T
    return g, u, h, d


def moe_forward(layer, x_bits, logits, topk: int, tokens=None, with_intermediates: bool = False,
                shared_gate=None):
    """out bits-exact fp64 values [len(tokens), H] for the selected tokens (all by default).

    out[t] = RN_bf16( sum_j p[t, j] * down_{e_j}(h_{t, e_j}) + g_t * shared(h_{t, s}) ),
    g_t = sigmoid(shared_gate[t]) (fp32 logits [T]) or 1 when shared_gate is None."""
    x64_all = bf16_value(x_bits)
    ids, p = route(logits, topk)
    tokens = np.arange(x64_all.shape[0]) if tokens is None else np.asarray(tokens, dtype=np.int64)
    acc = np.zeros((tokens.size, layer.hidden), dtype=np.float64)
    inter = {}
    # one dequantisation per expert that the selected tokens use
    for e in np.unique(ids[tokens]):
        rows_t, slots = np.nonzero(ids[tokens] == e)
        gu32, dn32 = dequant(layer.gate_up[e]), dequant(layer.down[e])
        g, u, h, d = expert_ffn(gu32, dn32, x64_all[tokens[rows_t]])
        acc[rows_t] += p[tokens[rows_t], slots][:, None] * d
        if with_intermediates:
            for i, (r, s) in enumerate(zip(rows_t, slots)):
                inter[(int(tokens[r]), int(e))] = (g[i], u[i], h[i], d[i])
    if layer.shared_gate_up is not None:
        g, u, h, d = expert_ffn(dequant(layer.shared_gate_up), dequant(layer.shared_down), x64_all[tokens])
        if shared_gate is None:
            acc += d
        else:
            lg = np.asarray(shared_gate, dtype=np.float32)[tokens]
            acc += sigmoid(lg)[:, None] * d
        if with_intermediates:
            for i, t in enumerate(tokens):
                inter[(int(t), -1)] = (g[i], u[i], h[i], d[i])
    out = round_to_bf16(acc)
    if with_intermediates:
        return out, acc, ids, p, inter
    return out
