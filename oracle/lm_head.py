"""Float64 oracle of the online-FP8 LM head: quantisation, GEMV, argmax and top-k.

Test infrastructure (see ``oracle/__init__.py``).

Sources (page title, section):

* "Three MoE Inference Optimizations NVIDIA Measured on DGX Spark", section "Online FP8
  quantization halves the LM head weight reads": the BF16 head (157,184 x 2,560) is
  quantised with a dynamic FP8 configuration when the head is constructed, halving the
  bytes read per generated token.
* runbyai.xyz/posts/593, paragraph 3: ~402 million weights, ~805 MB per token in BF16,
  ~400 MB in FP8.
* same blog page, section "GSM8K measured a 42.5% throughput gain across 1,319
  questions": sampling keeps the top_k = 29 tokens; the synthetic run decodes greedily
  (argmax).

Readings (listed in the design notes):

* R7 scale granularity: one float32 scale per vocabulary row, scale = amax/448.
* R8 activations of the head: the bf16 hidden state is used as is (W8A16); the logit of
  row v is scale_v * sum_h e4m3(q[v, h]) * x[h].
* R9 order: descending logit, ties to the lower vocabulary index.
"""

from __future__ import annotations

import numpy as np

from .formats import E4M3_LUT, quantize_fp8_lastdim
from .moe import topk_desc


def quantize_lm_head(w) -> tuple[np.ndarray, np.ndarray]:
    """Row-wise dynamic FP8 quantisation of the head weight (readings R7; float32 steps).

    w: [V, H] float32 holding bf16 values. Returns (q uint8 [V, H], scale float32 [V]).
    """
    return quantize_fp8_lastdim(w)


def lm_head_fp8_logits(q, scale, x, rows=None, chunk: int = 8192) -> np.ndarray:
    """logits[t, v] = scale_v * sum_h e4m3(q[v, h]) * x[t, h], float64 (reading R8).

    ``rows`` optionally restricts the output to a subset of vocabulary rows (returned in
    that order); otherwise all rows are computed in chunks of ``chunk`` rows.
    """
    x = np.asarray(x, dtype=np.float64)
    q = np.asarray(q)
    scale = np.asarray(scale, dtype=np.float64)
    if rows is not None:
        rows = np.asarray(rows)
        w = E4M3_LUT[q[rows]] * scale[rows, None]
        return x @ w.T
    v = q.shape[0]
    out = np.empty((x.shape[0], v), dtype=np.float64)
    for r0 in range(0, v, chunk):
        r1 = min(v, r0 + chunk)
        w = E4M3_LUT[q[r0:r1]] * scale[r0:r1, None]
        out[:, r0:r1] = x @ w.T
    return out


def lm_head_bf16_logits(w, x, rows=None, chunk: int = 8192) -> np.ndarray:
    """logits[t, v] = sum_h w[v, h] * x[t, h] in float64 on the unquantised bf16 head."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w)
    if rows is not None:
        return x @ np.asarray(w[np.asarray(rows)], dtype=np.float64).T
    out = np.empty((x.shape[0], w.shape[0]), dtype=np.float64)
    for r0 in range(0, w.shape[0], chunk):
        r1 = min(w.shape[0], r0 + chunk)
        out[:, r0:r1] = x @ np.asarray(w[r0:r1], dtype=np.float64).T
    return out


def topk(logits, k: int) -> np.ndarray:
    """Top-k vocabulary indices per token, descending, ties -> lower index (reading R9)."""
    return topk_desc(logits, k)


def argmax(logits) -> np.ndarray:
    """Greedy token per row: the first entry of the descending order."""
    return topk_desc(logits, 1)[:, 0]
