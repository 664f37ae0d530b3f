"""GPU parity of the online-FP8 LM head (quantisation, GEMV, fused argmax / top-k) and of
the BF16 comparison head, against the float64 oracle, through the C-ABI."""

import numpy as np
import pytest
import torch

from moe_decode_weight_gb300 import api, synth
from oracle import formats as F
from oracle import lm_head as OL

from _cases import assert_bar, bf16_to_np, topk_gap_ok

pytestmark = pytest.mark.gpu
H = 2560


def _weight(V, seed=1, specials=True):
    w = synth.lm_head_weight(seed, V)
    if specials:
        w[0] = 0                                   # all-zero row: scale 1, zero codes
        w[1, :] = 1e-30                            # tiny row (bf16 subnormal range of the quotient)
        w[2, ::7] = 3.0e4                          # large entries, saturating neighbours
        w[3, :] = -2.0                             # constant row: every code is -448
    return w


def _quantize(w):
    wd = w.cuda()
    V = w.shape[0]
    q = torch.empty((V, H), dtype=torch.uint8, device="cuda")
    s = torch.empty(V, dtype=torch.float32, device="cuda")
    head = api.quantize_lm_head_fp8(wd, q, s)
    torch.cuda.synchronize()
    return head, q, s, wd


@pytest.mark.parametrize("V", [1000, 20011])
def test_quantize_bit_exact(V):
    w = _weight(V)
    head, q, s, _ = _quantize(w)
    qo, so = OL.quantize_lm_head(bf16_to_np(w))
    assert np.array_equal(s.cpu().numpy(), so)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert head.c.fmt == api.FMT_FP8 and head.c.vocab == V


def _hidden(q, s, m, k, seed=1, bf16_w=None):
    """Per token, redraw (seeded attempts) until the oracle's top-(k+1) logits are 1e-3 apart."""
    rows, logits = [], []
    for t in range(m):
        for attempt in range(100):
            h = synth.hidden_states(1000 * seed + t, 1, attempt)
            hx = bf16_to_np(h)
            lg = OL.lm_head_fp8_logits(q, s, hx) if bf16_w is None else OL.lm_head_bf16_logits(bf16_w, hx)
            if topk_gap_ok(lg, k):
                rows.append(h)
                logits.append(lg)
                break
        else:
            raise RuntimeError("no hidden state with clean top-k gaps")
    return torch.cat(rows, 0), np.concatenate(logits, 0)


def _run_head(fn, head, h, V, k, with_logits=True):
    m = h.shape[0]
    ws = torch.zeros(api.mdw_lm_head_workspace_bytes(head, m, k), dtype=torch.uint8, device="cuda")
    am = torch.full((m,), -1, dtype=torch.int32, device="cuda")
    ti = torch.full((m, k), -1, dtype=torch.int32, device="cuda")
    tv = torch.zeros((m, k), dtype=torch.float32, device="cuda")
    lg = torch.zeros((m, V), dtype=torch.float32, device="cuda") if with_logits else None
    fn(head, h.cuda(), am, ws, logits=lg, topk=k, topk_idx=ti, topk_val=tv)
    assert api.mdw_device_status(ws) == 0
    return (am.cpu().numpy(), ti.cpu().numpy(), tv.cpu().numpy(),
            lg.cpu().numpy() if lg is not None else None)


@pytest.mark.parametrize("m", [1, 4, 16, 32])
@pytest.mark.parametrize("V,k", [(20011, 29), (1000, 29), (5003, 1), (5003, 32)])
def test_lm_head_fp8_parity(m, V, k):
    w = _weight(V, specials=False)
    head, q, s, _ = _quantize(w)
    qo, so = OL.quantize_lm_head(bf16_to_np(w))      # the oracle's own codes
    h, lo = _hidden(qo, so, m, k)
    am, ti, tv, lg = _run_head(api.lm_head_fp8, head, h, V, k)
    assert_bar(lg, lo, "fp8 logits")
    ref = OL.topk(lo, k)
    assert np.array_equal(ti, ref)
    assert np.array_equal(am, ref[:, 0])
    assert_bar(tv, np.take_along_axis(lo, ref, axis=1), "top-k values")


def test_lm_head_fp8_without_logits_output():
    V, k = 20011, 29
    w = _weight(V, specials=False)
    head, q, s, _ = _quantize(w)
    qo, so = OL.quantize_lm_head(bf16_to_np(w))
    h, lo = _hidden(qo, so, 2, k, seed=5)
    am, ti, _, _ = _run_head(api.lm_head_fp8, head, h, V, k, with_logits=False)
    assert np.array_equal(ti, OL.topk(lo, k))


@pytest.mark.parametrize("m", [1, 4])
def test_lm_head_bf16_parity(m):
    V, k = 12007, 29
    w = _weight(V, specials=False)
    wd = w.cuda()
    head = api.mdw_lm_head_bf16_init(wd)
    wn = bf16_to_np(w)
    h, lo = _hidden(None, None, m, k, seed=3, bf16_w=wn)
    am, ti, tv, lg = _run_head(api.lm_head_bf16, head, h, V, k)
    assert_bar(lg, lo, "bf16 logits")
    assert np.array_equal(ti, OL.topk(lo, k))


def test_lm_head_full_vocab_sampled():
    """157,184 x 2,560 (the pages' head): codes and logits on sampled rows; the fused top-29
    equals the top-29 of the kernel's own logits; the oracle ranks those 29 rows the same."""
    V, k, m = synth.VOCAB, 29, 4
    w = synth.lm_head_weight(1, V)
    head, q, s, _ = _quantize(w)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, 1, V // 2, V - 2, V - 1], rng.integers(0, V, 3000)]))
    wn = bf16_to_np(w[torch.from_numpy(rows)])
    qo, so = OL.quantize_lm_head(wn)
    assert np.array_equal(q[torch.from_numpy(rows).cuda()].cpu().numpy(), qo)
    assert np.array_equal(s[torch.from_numpy(rows).cuda()].cpu().numpy(), so)
    h = synth.hidden_states(1, m, 0)
    am, ti, tv, lg = _run_head(api.lm_head_fp8, head, h, V, k)
    hx = bf16_to_np(h)
    assert_bar(lg[:, rows], OL.lm_head_fp8_logits(qo, so, hx), "sampled logits")
    # property: the fused selection equals a full sort of the kernel's own logits
    own = np.stack([np.lexsort((np.arange(V), -lg[t]))[:k] for t in range(m)])
    assert np.array_equal(ti, own)
    top_rows = np.unique(ti.reshape(-1))
    sel = torch.from_numpy(top_rows)
    qt, st = OL.quantize_lm_head(bf16_to_np(w[sel]))
    lt = OL.lm_head_fp8_logits(qt, st, hx)
    pos = {r: i for i, r in enumerate(top_rows)}
    for t in range(m):
        ov = lt[t, [pos[r] for r in ti[t]]]
        gaps = -np.diff(ov)
        assert np.all(gaps > -1e-3)                          # the oracle agrees on the order
