"""GPU parity of the decode-time draw (mdw_sample_topk and the draw fused into the FP8 head)
against the float64 sampler oracle: drawn token ids must match exactly. Uniforms whose draw
sits within a small margin of a decision boundary are redrawn (seeded), so that the last
bits of exp() on either side cannot decide a test."""

import numpy as np
import pytest
import torch

from moe_decode_weight_gb300 import api, synth
from oracle import lm_head as OL
from oracle import sampler as OS

from _cases import bf16_to_np, topk_gap_ok

pytestmark = pytest.mark.gpu
H = 2560


def _nucleus_margin(vals, temperature, top_p):
    """The u-independent part of the decision margin: how far the nucleus cut is from moving
    (a uniform outside [0, 1) leaves only those terms of the oracle's margin)."""
    return OS.decision_margin(vals, temperature, top_p, 2.0)


def _uniforms(vals, temperature, top_p, seed, margin):
    rng = np.random.default_rng(seed)
    out = []
    for row in vals:
        for _ in range(1000):
            u = rng.random()
            if OS.decision_margin(row, temperature, top_p, u) > margin:
                out.append(u)
                break
        else:
            raise RuntimeError("no uniform with a clean margin")
    return np.array(out, dtype=np.float64)


@pytest.mark.parametrize("temperature,top_p", [(0.6, 0.95), (1.0, 1.0), (0.0, 0.95), (0.6, 0.5), (2.0, 0.99)])
@pytest.mark.parametrize("k", [29, 1, 32])
def test_sample_topk_parity(temperature, top_p, k):
    m = 16
    rng = np.random.default_rng(k * 100 + int(temperature * 10))
    vals = -np.sort(-rng.normal(0.0, 1.5, (m, k)), axis=1).astype(np.float32)
    idx = rng.integers(0, 157184, (m, k)).astype(np.int32)
    u = _uniforms(vals, temperature, top_p, seed=k, margin=1e-9)
    out = torch.full((m,), -1, dtype=torch.int32, device="cuda")
    api.mdw_sample_topk(torch.from_numpy(vals).cuda(), torch.from_numpy(idx).cuda(), temperature, top_p,
                        torch.from_numpy(u).cuda(), out)
    want = [OS.sample_topk(vals[t], idx[t], temperature, top_p, u[t]) for t in range(m)]
    assert out.cpu().numpy().tolist() == want


def test_sample_topk_rejects_bad_settings():
    v = torch.zeros((2, 4), dtype=torch.float32, device="cuda")
    i = torch.zeros((2, 4), dtype=torch.int32, device="cuda")
    u = torch.zeros(2, dtype=torch.float64, device="cuda")
    o = torch.zeros(2, dtype=torch.int32, device="cuda")
    for tp in (0.0, 1.5):
        with pytest.raises(api.MdwError):
            api.mdw_sample_topk(v, i, 0.6, tp, u, o)


@pytest.mark.parametrize("m", [1, 4, 20])
def test_head_fused_draw(m):
    """FP8 head + draw in one launch; the oracle draws from its own float64 top-29."""
    V, k, T, P = 20011, 29, 0.6, 0.95
    w = synth.lm_head_weight(1, V)
    wd = w.cuda()
    q = torch.empty((V, H), dtype=torch.uint8, device="cuda")
    s = torch.empty(V, dtype=torch.float32, device="cuda")
    head = api.quantize_lm_head_fp8(wd, q, s)
    qo, so = OL.quantize_lm_head(bf16_to_np(w))
    rows, tops = [], []
    for t in range(m):
        for attempt in range(100):
            h = synth.hidden_states(7000 + t, 1, attempt)
            lg = OL.lm_head_fp8_logits(qo, so, bf16_to_np(h))
            if not topk_gap_ok(lg, k):
                continue
            ii = OL.topk(lg, k)
            vv = np.take_along_axis(lg, ii, axis=1)
            if _nucleus_margin(vv[0], T, P) <= 1e-3:     # no uniform could make this draw clean
                continue
            rows.append(h)
            tops.append((vv[0], ii[0]))
            break
        else:
            raise RuntimeError("no hidden state with clean gaps")
    x = torch.cat(rows, 0).cuda()
    vals = np.stack([tv for tv, _ in tops])
    u = _uniforms(vals, T, P, seed=m, margin=1e-3)
    ws = torch.zeros(api.mdw_lm_head_workspace_bytes(head, m, k), dtype=torch.uint8, device="cuda")
    out = torch.full((m,), -1, dtype=torch.int32, device="cuda")
    ti = torch.full((m, k), -1, dtype=torch.int32, device="cuda")
    api.lm_head_fp8_sample(head, x, out, ws, torch.from_numpy(u).cuda(), T, P, k, topk_idx=ti)
    assert api.mdw_device_status(ws) == 0
    assert np.array_equal(ti.cpu().numpy(), np.stack([ii for _, ii in tops]))
    want = [OS.sample_topk(vals[t], tops[t][1], T, P, u[t]) for t in range(m)]
    assert out.cpu().numpy().tolist() == want
