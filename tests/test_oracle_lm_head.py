"""Pins of the oracle's FP8 LM head: quantiser invariants, logits vs a library decode,
brute-force argmax / top-k, and the byte counts the pages print."""

import json
import os

import numpy as np
import torch

from oracle import formats as F
from oracle import lm_head as OL

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _head(v=3000, h=256, seed=0):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((v, h)) * 0.02).astype(np.float32)
    w[5] = 0.0                                   # an all-zero row
    return F.bf16_bits_to_float(F.f32_to_bf16_bits(w))


def test_quantize_rows_reach_448_and_zero_row():
    w = _head()
    q, s = OL.quantize_lm_head(w)
    mx = np.max(np.abs(F.e4m3_to_float(q)), axis=1)
    nz = np.any(w != 0, axis=1)
    assert np.all(mx[nz] == 448.0)
    assert s[5] == 1.0 and not q[5].any()


def test_logits_vs_torch_decode():
    w = _head()
    q, s = OL.quantize_lm_head(w)
    x = F.bf16_bits_to_float(F.f32_to_bf16_bits(
        np.random.default_rng(1).standard_normal((4, 256)).astype(np.float32)))
    deq = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64) * \
        torch.from_numpy(s.astype(np.float64))[:, None]
    ref = (torch.from_numpy(x.astype(np.float64)) @ deq.T).numpy()
    got = OL.lm_head_fp8_logits(q, s, x, chunk=700)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)
    rows = np.array([17, 3, 2999])
    assert np.allclose(OL.lm_head_fp8_logits(q, s, x, rows=rows), ref[:, rows], rtol=1e-12)
    # FP8 logits stay close to the unquantised head: E4M3 keeps 3 mantissa bits, so the
    # per-weight rounding error is ~2^-4/sqrt(3) relative and the logit error ~4% of spread
    b = OL.lm_head_bf16_logits(w, x, chunk=512)
    err = got - b
    assert np.std(err) < 0.06 * np.std(b) and np.max(np.abs(err)) < 0.25 * np.std(b)


def test_topk_and_argmax_brute_force():
    rng = np.random.default_rng(2)
    lg = rng.standard_normal((3, 5000))
    lg[1, 100] = lg[1, 50] = 10.0                # tie at the top: lower index first
    idx = OL.topk(lg, 29)
    for t in range(3):
        ref = sorted(range(5000), key=lambda i: (-lg[t, i], i))[:29]
        assert list(idx[t]) == ref
    assert list(OL.argmax(lg)) == [int(np.argmax(lg[t])) for t in range(3)]
    assert OL.argmax(lg)[1] == 50


def test_page_byte_counts():
    """~402M weights, ~805 MB in BF16, ~400 MB in FP8 (runbyai.xyz/posts/593 para. 3)."""
    with open(os.path.join(GOLDEN, "page_facts.json")) as f:
        facts = json.load(f)
    from moe_decode_weight_gb300 import roofline as R
    hb = facts["lm_head"]
    assert abs(R.head_weights() / 1e6 - hb["weights_millions"]) < 0.5
    assert round(R.head_bf16_bytes() / 1e6) == hb["bf16_mb_per_token"]
    assert abs(R.head_fp8_bytes(m=0) / 1e6 - hb["fp8_mb_per_token"]) / hb["fp8_mb_per_token"] < 0.01
    assert abs(R.head_bf16_bytes() / R.head_fp8_bytes(m=0) - 2.0) < 0.01
