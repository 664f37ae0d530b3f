"""Float64 oracle of one W4A8 MXFP4 MoE decode layer (router, experts, combine).

Test infrastructure (see ``oracle/__init__.py``).

Sources (page title, section):

* "Three MoE Inference Optimizations NVIDIA Measured on DGX Spark", section "Decoding was
  memory-bound on a 124-billion-parameter model at batch size 1": a token is routed to
  eight of 512 routed experts alongside one shared expert (also runbyai.xyz/posts/593,
  paragraph 2).
* same page, section "Humming MXFP4 kernels compile at run time for the model's real
  shapes": W4A8 MXFP4 experts, moe_intermediate_size 768.
* same page, section "Multi-token prediction turns each verification into four tokens":
  verifying four positions activates up to 32 experts; each selected expert is needed
  once per window, whatever number of its tokens (the union of the selections).

Readings taken where the pages are silent (each is listed in the design notes):

* R1 scoring: softmax over the router logits, top-k by logit (ties to the lower expert
  index), the k selected weights renormalised to sum to one; no bias, no group limit,
  routed scaling factor 1. The renormalised softmax over k selected entries equals the
  softmax of the k selected logits, which is what ``route`` computes.
* R2 router input: the bf16 hidden state before FP8 quantisation, float accumulation.
* R3 MXFP4 layout: 32 contiguous K elements share one E8M0 scale; in a packed byte the
  low nibble holds the even K index; gate rows 0..I-1 and up rows I..2I-1 of ``w13``.
* R4 W4A8: the expert input x is quantised per token to E4M3 with one float32 scale
  (amax/448); the SwiGLU output h is quantised the same way per (token, expert) before
  the down projection, so both expert GEMMs see 8-bit activations.
* R5 SwiGLU: h = silu(gate) * up, silu(g) = g / (1 + exp(-g)).
* R6 combine: y = sum over the token's k experts of gate weight * expert output, plus
  the shared expert's output with weight 1 (plus an optional residual).
"""

from __future__ import annotations

import numpy as np

from .formats import (E2M1_LUT, E4M3_LUT, e8m0_to_float, quantize_fp8_lastdim)

# ----------------------------------------------------------------------------- router


def topk_desc(values, k: int) -> np.ndarray:
    """Indices of the k largest entries of each row, largest first, ties -> lower index."""
    v = np.asarray(values, dtype=np.float64)
    out = np.empty(v.shape[:-1] + (k,), dtype=np.int64)
    flat_v = v.reshape(-1, v.shape[-1])
    flat_o = out.reshape(-1, k)
    idx = np.arange(v.shape[-1])
    for r in range(flat_v.shape[0]):
        order = np.lexsort((idx, -flat_v[r]))   # primary: -value, secondary: index
        flat_o[r] = order[:k]
    return out


def router_logits(x, wr) -> np.ndarray:
    """z[t, e] = sum_h x[t, h] * Wr[e, h] in float64 (reading R2: bf16 x before quantisation)."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(wr, dtype=np.float64).T


def route(z, top_k: int):
    """Top-k selection and renormalised softmax gates (reading R1).

    Returns (ids int64 [M, k] in descending logit order, gates float64 [M, k]).
    """
    ids = topk_desc(z, top_k)
    sel = np.take_along_axis(np.asarray(z, dtype=np.float64), ids, axis=-1)
    ex = np.exp(sel - sel.max(axis=-1, keepdims=True))
    return ids, ex / ex.sum(axis=-1, keepdims=True)


def gates_for(z, ids) -> np.ndarray:
    """Renormalised softmax weights of given selections (used when routing is imposed)."""
    sel = np.take_along_axis(np.asarray(z, dtype=np.float64), np.asarray(ids), axis=-1)
    ex = np.exp(sel - sel.max(axis=-1, keepdims=True))
    return ex / ex.sum(axis=-1, keepdims=True)


def expert_union(ids) -> np.ndarray:
    """The distinct experts selected by any token of the window, ascending."""
    return np.unique(np.asarray(ids).reshape(-1))


# ----------------------------------------------------------------------------- MXFP4


def mxfp4_dequant(q, s) -> np.ndarray:
    """Dequantise packed MXFP4 rows to float64 (reading R3).

    q: uint8 [..., R, K/2], low nibble = even K index. s: uint8 E8M0 [..., R, K/32].
    Returns float64 [..., R, K] = e2m1(code) * 2^(scale - 127) for the code's 32-block.
    """
    q = np.asarray(q, dtype=np.uint8)
    s = np.asarray(s, dtype=np.uint8)
    lo = E2M1_LUT[q & 0xF]
    hi = E2M1_LUT[q >> 4]
    w = np.stack([lo, hi], axis=-1).reshape(q.shape[:-1] + (q.shape[-1] * 2,))
    sc = np.repeat(e8m0_to_float(s), 32, axis=-1)
    return w * sc


def mx_gemv(q, s, a_codes, a_scale) -> np.ndarray:
    """sum_b 2^(E_b-127) sum_{k in b} e2m1(W[r,k]) * e4m3(a[k]), times the activation scale."""
    a = E4M3_LUT[np.asarray(a_codes, dtype=np.uint8)]
    return float(a_scale) * (mxfp4_dequant(q, s) @ a)


# ----------------------------------------------------------------------------- expert


def act_quant(x):
    """Per-token E4M3 quantisation of the expert input (reading R4); x: [M, H] bf16 values."""
    return quantize_fp8_lastdim(x)


def expert_gate_up(w13_q, w13_s, xq, sx):
    """gate[j], up[j] of one expert for one token: rows 0..I-1 gate, I..2I-1 up (R3)."""
    v = mx_gemv(w13_q, w13_s, xq, sx)
    inter = v.shape[0] // 2
    return v[:inter], v[inter:]


def swiglu(gate, up) -> np.ndarray:
    """h = silu(gate) * up in float64 (reading R5)."""
    gate = np.asarray(gate, dtype=np.float64)
    return gate / (1.0 + np.exp(-gate)) * np.asarray(up, dtype=np.float64)


def h_quant(h):
    """E4M3 quantisation of a SwiGLU output vector (reading R4): the float64 h is first
    rounded to float32, then the float32 quantiser of ``quantize_fp8_lastdim`` applies."""
    return quantize_fp8_lastdim(np.asarray(h, dtype=np.float64).astype(np.float32))


def expert_down(w2_q, w2_s, hq, s_h) -> np.ndarray:
    """y_e[r] = s_h * sum_b 2^(E_b-127) sum_{j in b} e2m1(W2[r, j]) * e4m3(hq[j])."""
    return mx_gemv(w2_q, w2_s, hq, s_h)


def expert_forward(wq13, ws13, wq2, ws2, xq, sx):
    """One expert on one token: returns dict(gate, up, h, hq, s_h, y)."""
    gate, up = expert_gate_up(wq13, ws13, xq, sx)
    h = swiglu(gate, up)
    hq, s_h = h_quant(h)
    y = expert_down(wq2, ws2, hq, s_h)
    return dict(gate=gate, up=up, h=h, hq=hq, s_h=float(s_h), y=y)


# ----------------------------------------------------------------------------- layer


def moe_layer(x, wr, experts, shared, top_k: int, topk_override=None, residual=None):
    """One MoE decode layer for M tokens.

    x: [M, H] float32 holding bf16 values. wr: [E, H] router weight (bf16 values).
    experts: callable e -> (w13_q, w13_s, w2_q, w2_s) of routed expert e (so a caller can
    regenerate only the selected experts). shared: the same 4-tuple or None.
    topk_override: optional [M, k] expert ids that replace the top-k selection; the gates
    are then the renormalised softmax of the router logits at those ids.
    residual: optional [M, H] added to the output.

    Returns a dict of every intermediate: xq, sx, logits, ids, gates, union, per-(token,
    expert) results, y (float64 [M, H]).
    """
    x = np.asarray(x, dtype=np.float32)
    m = x.shape[0]
    xq, sx = act_quant(x)
    z = router_logits(x, wr)
    if topk_override is None:
        ids, gates = route(z, top_k)
    else:
        ids = np.asarray(topk_override, dtype=np.int64)
        gates = gates_for(z, ids)
    union = expert_union(ids)
    cache = {}

    def get(e):
        if e not in cache:
            cache[e] = experts(int(e))
        return cache[e]

    per = {}
    y = np.zeros((m, x.shape[1]), dtype=np.float64)
    for t in range(m):
        for i in range(ids.shape[1]):
            e = int(ids[t, i])
            r = expert_forward(*get(e), xq[t], sx[t])
            per[(t, e)] = r
            y[t] += gates[t, i] * r["y"]
        if shared is not None:
            r = expert_forward(*shared, xq[t], sx[t])
            per[(t, "shared")] = r
            y[t] += r["y"]
    if residual is not None:
        y = y + np.asarray(residual, dtype=np.float64)
    return dict(xq=xq, sx=sx, logits=z, ids=ids, gates=gates, union=union, per=per, y=y)
