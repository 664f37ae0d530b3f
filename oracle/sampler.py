"""Float64 oracle of the decode-time sampler on the LM head's top-k: temperature, nucleus
(top_p) truncation and one inverse-CDF draw.

Test infrastructure (see ``oracle/__init__.py``).

Sources (page title, section):

* "Three MoE Inference Optimizations NVIDIA Measured on DGX Spark", section
  "GSM8K measured a 42.5% throughput gain across 1,319 questions": the evaluation samples
  at temperature 0.6 with top_p 0.95 and top_k 29.
* runbyai.xyz/posts/593, paragraph 6: the same three settings, against greedy decoding on
  the synthetic run.

The pages name the three settings and nothing else. Readings (listed in the design notes):

* S1 order: the head's top_k candidates (descending logit, ties to the lower id) are
  scaled by 1/temperature and normalised with a softmax over those k only.
* S2 nucleus: the smallest prefix of the candidates whose probability mass reaches top_p
  is kept (the candidate that crosses top_p stays; at least one candidate stays).
* S3 draw: one uniform u in [0, 1) per token, supplied by the caller; the token is the first
  kept candidate whose cumulative mass exceeds u times the kept mass.
* S4 temperature <= 0 means greedy: the first candidate.
* S5 arithmetic: float64, sums taken left to right, e_i = exp((z_i - z_0) / T).
"""

from __future__ import annotations

import math

import numpy as np


def sample_topk(vals, idx, temperature: float, top_p: float, u: float) -> int:
    """Token drawn from the top-k candidates (vals descending, idx their token ids)."""
    vals = np.asarray(vals, dtype=np.float64)
    idx = np.asarray(idx)
    k = len(vals)
    if temperature <= 0.0:
        return int(idx[0])
    z0 = float(vals[0])
    e = [math.exp((float(v) - z0) / float(temperature)) for v in vals]
    total = 0.0
    for v in e:
        total += v
    cut, c = k - 1, 0.0
    for i in range(k):
        c += e[i]
        if c >= top_p * total:
            cut = i
            break
    kept = 0.0
    for i in range(cut + 1):
        kept += e[i]
    target = u * kept
    c = 0.0
    for i in range(cut + 1):
        c += e[i]
        if target < c:
            return int(idx[i])
    return int(idx[cut])


def decision_margin(vals, temperature: float, top_p: float, u: float) -> float:
    """Smallest relative distance of the draw's deciding comparisons from flipping: the
    nucleus test at the cut (and just before it) and the draw against each kept cumulative
    mass. A draw whose margin is below ~1e-12 could depend on the last bits of exp()."""
    vals = np.asarray(vals, dtype=np.float64)
    if temperature <= 0.0:
        return math.inf
    e = np.exp((vals - vals[0]) / temperature)
    c = np.cumsum(e)
    total = c[-1]
    reach = c >= top_p * total
    cut = int(np.argmax(reach)) if reach.any() else len(e) - 1
    m = math.inf
    if cut < len(e) - 1:                 # failing here would move the cut one later
        m = min(m, abs(c[cut] - top_p * total) / total)
    if cut > 0:                          # passing here would move the cut one earlier
        m = min(m, abs(c[cut - 1] - top_p * total) / total)
    kept = c[cut]
    m = min(m, float(np.min(np.abs(c[: cut + 1] - u * kept)) / kept))
    return m
