"""Shared builders of seeded GPU test cases (weights on the device, oracle views on the host).

Inputs come from moe_decode_weight_gb300.synth only; expected values come from oracle/ only.
Hidden states are redrawn (rejection sampling, seeded attempts) until the oracle's logits
keep every decision the comparison depends on away from a tie by more than 1e-3: the gap
between the k-th and (k+1)-th router logit of each token, and for the head the gaps among
the top entries.
"""

from __future__ import annotations

import numpy as np
import torch

from moe_decode_weight_gb300 import api, synth
from oracle import moe as OM

GAP = 1e-3


def bar_ok(gpu, ref, rtol=2e-3, atol=1e-3, extra=0.0):
    """Element-wise parity bar: relative 2e-3, or absolute 1e-3 where |ref| < 1 (plus an
    optional per-element allowance ``extra`` derived by the oracle)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(gpu - ref) - extra
    ok = np.where(np.abs(ref) < 1.0, err <= atol, err <= rtol * np.abs(ref))
    return ok


def assert_bar(gpu, ref, what, rtol=2e-3, atol=1e-3, extra=0.0):
    ok = bar_ok(gpu, ref, rtol, atol, extra)
    if not ok.all():
        bad = np.argwhere(~ok)[:5]
        g = np.asarray(gpu).reshape(ok.shape)
        r = np.asarray(ref).reshape(ok.shape)
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside the bar; first "
                             f"{[(tuple(i), float(g[tuple(i)]), float(r[tuple(i)])) for i in bad]}")


def bf16_to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().float().numpy()


class Layer:
    """One MoE layer: device weights + host regeneration of any expert for the oracle."""

    def __init__(self, seed: int, layer: int, num_experts: int = 512, top_k: int = 8,
                 shared: bool = True, device="cuda"):
        self.seed, self.layer, self.E, self.K = seed, layer, num_experts, top_k
        (w13q, w13s, w2q, w2s), sh = synth.layer_experts(seed, layer, num_experts, device=device,
                                                         with_shared=shared)
        self.wr_t = synth.router_weight(seed, layer, num_experts)
        self.wr = bf16_to_np(self.wr_t)
        self.tensors = (self.wr_t.to(device), w13q, w13s, w2q, w2s, sh)
        self.weights = api.MoeWeights(self.tensors[0], w13q, w13s, w2q, w2s,
                                      tuple(sh) if sh is not None else None, top_k)
        self.has_shared = shared
        self._cache = {}

    def expert(self, e: int):
        if e not in self._cache:
            self._cache[e] = tuple(t.numpy() for t in synth.expert_tensors(self.seed, self.layer, e))
        return self._cache[e]

    def shared(self):
        return self.expert(synth.SHARED_EXPERT) if self.has_shared else None

    def oracle_dict(self):
        return dict(wr=self.wr, experts=self.expert, shared=self.shared())


def router_gap_ok(x: np.ndarray, wr: np.ndarray, k: int, gap: float = GAP) -> bool:
    z = OM.router_logits(x, wr)
    s = -np.sort(-z, axis=1)
    return bool(np.all(s[:, k - 1] - s[:, k] > gap))


def hidden_with_gap(seed: int, m: int, wr: np.ndarray, k: int, max_attempts: int = 200) -> torch.Tensor:
    for attempt in range(max_attempts):
        x = synth.hidden_states(seed, m, attempt)
        if router_gap_ok(bf16_to_np(x), wr, k):
            return x
    raise RuntimeError("no hidden state with a clean router gap")


def topk_gap_ok(logits: np.ndarray, k: int, gap: float = GAP) -> bool:
    s = -np.sort(-logits, axis=1)[:, :k + 1]
    return bool(np.all(-np.diff(s, axis=1) > gap))


def read_ws(ws: torch.Tensor, off: int, dtype, count: int) -> np.ndarray:
    nbytes = count * np.dtype(dtype).itemsize
    return ws[off:off + nbytes].cpu().numpy().view(dtype).copy()


def norm_rounding_allowance(r, q, scale, rows=None, rel=4e-6):
    """Per (token, vocabulary row) bound on how far the head's logits may move because the
    final RMSNorm rounds to bf16 on the device from an fp32 quotient, where the oracle rounds
    the float64 one.

    The two quotients agree to about ``rel`` relative (fp32 sum of squares, reciprocal square
    root and product), so their bf16 roundings can differ only where the float64 quotient lies
    within ``rel`` of a rounding midpoint, and there by one bf16 step. Such an element moves
    logit v by at most |scale_v * e4m3(q[v, h])| * step_h. Returns float64 [M, rows].
    """
    from oracle import formats as F
    from oracle import stack as OS
    r = np.asarray(r, dtype=np.float64)
    u = r / np.sqrt(np.mean(r * r, axis=-1, keepdims=True) + OS.RMS_EPS)
    au = np.abs(u)
    _, e = np.frexp(np.where(au > 0, au, 1.0))
    step = np.ldexp(1.0, e - 1 - 7)                          # bf16 spacing at |u|
    frac = au / step - np.floor(au / step)
    amb = (np.abs(frac - 0.5) * step <= rel * au) & (au > 0)
    q = np.asarray(q) if rows is None else np.asarray(q)[np.asarray(rows)]
    sc = np.asarray(scale, dtype=np.float64) if rows is None else np.asarray(scale, dtype=np.float64)[np.asarray(rows)]
    out = np.zeros((r.shape[0], q.shape[0]))
    for t in range(r.shape[0]):
        hs = np.nonzero(amb[t])[0]
        if hs.size:
            out[t] = (np.abs(F.E4M3_LUT[q[:, hs]]) * sc[:, None]) @ step[t, hs]
    return out
