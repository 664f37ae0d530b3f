"""Float64 oracle of the full decode-step weight stream: L MoE layers, then the FP8 head.

Test infrastructure (see ``oracle/__init__.py``).

Sources (page title, section): "Three MoE Inference Optimizations NVIDIA Measured on DGX
Spark", section "Decoding was memory-bound on a 124-billion-parameter model at batch
size 1": 42 layers, each with an MoE block, then the vocabulary projection, read in full
for every generated token; runbyai.xyz/posts/593, paragraph 2.

Reading R10 (listed in the design notes): the stack keeps a bf16 residual stream r and
uses a pre-norm, as a decoder does; attention is left out.

    x_l     = bf16( RMSNorm(r_l) ),   RMSNorm(v) = v / sqrt(mean(v^2) + 1e-6), unit gain
    r_{l+1} = bf16( r_l + MoE_l(x_l) )
    logits  = LMHead( bf16( RMSNorm(r_L) ) )

Without a norm the expert outputs (standard deviation ~40 for a unit input with these
weight distributions) would overflow the residual stream within a few layers.
"""

from __future__ import annotations

import numpy as np

from .formats import round_f64_to_bf16
from .moe import moe_layer
from . import lm_head as _head

RMS_EPS = 1e-6


def rmsnorm_bf16(r, eps: float = RMS_EPS) -> np.ndarray:
    """bf16(r / sqrt(mean(r^2) + eps)) per row, computed in float64, rounded once."""
    r = np.asarray(r, dtype=np.float64)
    inv = 1.0 / np.sqrt(np.mean(r * r, axis=-1, keepdims=True) + eps)
    return round_f64_to_bf16(r * inv)


def residual_add_bf16(r, y) -> np.ndarray:
    """bf16(r + y) with the sum taken in float64 and rounded once."""
    return round_f64_to_bf16(np.asarray(r, dtype=np.float64) + np.asarray(y, dtype=np.float64))


def layer_step(r, layer, top_k: int, topk_override=None):
    """One layer of the stack on residual r: returns (r_next, x, moe_result)."""
    x = rmsnorm_bf16(r)
    res = moe_layer(x, layer["wr"], layer["experts"], layer["shared"], top_k,
                    topk_override=topk_override)
    return residual_add_bf16(r, res["y"]), x, res


def decode_step(r0, layers, head_q, head_scale, top_k: int, k_vocab: int = 29):
    """The whole decode step: returns dict(r=[r_0..r_L], x_final, logits, argmax, topk)."""
    rs = [np.asarray(r0, dtype=np.float32)]
    for layer in layers:
        r_next, _, _ = layer_step(rs[-1], layer, top_k)
        rs.append(r_next)
    xf = rmsnorm_bf16(rs[-1])
    logits = _head.lm_head_fp8_logits(head_q, head_scale, xf)
    idx = _head.topk(logits, k_vocab)
    return dict(r=rs, x_final=xf, logits=logits, argmax=idx[:, 0], topk=idx)
