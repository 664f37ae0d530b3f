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


@pytest.mark.parametrize("m", [1, 4, 16, 21, 32])
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


@pytest.mark.parametrize("m", [2, 32])
def test_lm_head_fp8_without_logits_output(m):
    """Without a logits output: above 16 tokens the head selects from logits it writes to
    the workspace."""
    V, k = 20011, 29
    w = _weight(V, specials=False)
    head, q, s, _ = _quantize(w)
    qo, so = OL.quantize_lm_head(bf16_to_np(w))
    h, lo = _hidden(qo, so, m, k, seed=5)
    am, ti, _, _ = _run_head(api.lm_head_fp8, head, h, V, k, with_logits=False)
    assert np.array_equal(ti, OL.topk(lo, k))
    assert np.array_equal(am, ti[:, 0])


@pytest.mark.parametrize("m", [1, 4, 32])
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


@pytest.fixture(scope="module")
def full_head():
    """The pages' head (157,184 x 2,560, seed 1), quantised on the device, and the oracle's
    own codes and scales of every row (float32 steps, in row chunks)."""
    V = synth.VOCAB
    w = synth.lm_head_weight(1, V)
    head, q, s, wd = _quantize(w)
    del wd
    qo = np.empty((V, H), dtype=np.uint8)
    so = np.empty(V, dtype=np.float32)
    for r0 in range(0, V, 16384):
        r1 = min(V, r0 + 16384)
        qo[r0:r1], so[r0:r1] = OL.quantize_lm_head(bf16_to_np(w[r0:r1]))
    return head, q, s, qo, so


def test_lm_head_full_vocab_codes_bit_exact(full_head):
    """Every code and row scale of the full head equals the oracle's."""
    _, q, s, qo, so = full_head
    assert np.array_equal(s.cpu().numpy(), so)
    assert np.array_equal(q.cpu().numpy(), qo)


@pytest.mark.parametrize("m", [1, 4, 32])
def test_lm_head_full_vocab_exact(full_head, m):
    """At the real head size: hidden states are gap-sampled by the oracle over all 157,184
    logits (its top-30 entries pairwise more than 1e-3 apart), then the fused argmax and
    top-29 must equal the oracle's indices exactly and every logit must meet the bar."""
    head, _, _, qo, so = full_head
    V, k = synth.VOCAB, 29
    rows, los = [], []
    for batch in range(12):
        cand = torch.cat([synth.hidden_states(4000 + m, 1, 16 * batch + a) for a in range(16)], 0)
        lc = OL.lm_head_fp8_logits(qo, so, bf16_to_np(cand))
        for a in range(16):
            if len(rows) < m and topk_gap_ok(lc[a:a + 1], k):
                rows.append(cand[a:a + 1])
                los.append(lc[a:a + 1])
        if len(rows) == m:
            break
    assert len(rows) == m, "no hidden states with clean top-30 gaps"
    h, lo = torch.cat(rows, 0), np.concatenate(los, 0)
    am, ti, tv, lg = _run_head(api.lm_head_fp8, head, h, V, k)
    assert_bar(lg, lo, "full-vocabulary logits")
    ref = OL.topk(lo, k)
    assert np.array_equal(ti, ref)
    assert np.array_equal(am, ref[:, 0])
    assert_bar(tv, np.take_along_axis(lo, ref, axis=1), "top-29 values")
