"""GPU parity of one MoE decode layer (moe_decode_layer through the C-ABI) against the
float64 oracle, step by step:

* xq / sx (per-token E4M3 quantisation): bit-exact (both sides do the same IEEE fp32 steps);
* router logits: parity bar; selected experts: exact (inputs keep a 1e-3 router gap);
* gates: parity bar; the expert union and the (token, expert) pairs: exact;
* SwiGLU output h per pair: parity bar against the oracle fed the same xq;
* hq / s_h: bit-exact against the oracle's quantiser applied to the device's fp32 h;
* y: parity bar against the oracle's down projection fed the device's hq / s_h (the
  device computes h in fp32, the oracle in float64, so an hq code may legitimately differ
  at an E4M3 rounding boundary; the end-to-end y is also checked against a looser bound).
"""

import numpy as np
import pytest
import torch

from moe_decode_weight_gb300 import api, synth
from oracle import formats as F
from oracle import moe as OM

from _cases import Layer, assert_bar, bar_ok, bf16_to_np, hidden_with_gap, read_ws, router_gap_ok

pytestmark = pytest.mark.gpu
H, I = 2560, 768


@pytest.fixture(scope="module")
def layer512():
    return Layer(seed=0, layer=0, num_experts=512, top_k=8, shared=True)


@pytest.fixture(scope="module")
def layer64():
    return Layer(seed=7, layer=3, num_experts=64, top_k=4, shared=False)


def run_layer(layer, x, y_fp32=True, residual=None, override=None):
    m = x.shape[0]
    ws = torch.zeros(api.mdw_moe_workspace_bytes(layer.weights, m), dtype=torch.uint8, device="cuda")
    y = torch.full((m, H), float("nan"), dtype=torch.float32 if y_fp32 else torch.bfloat16, device="cuda")
    ids = torch.full((m, layer.K), -1, dtype=torch.int32, device="cuda")
    gw = torch.zeros((m, layer.K), dtype=torch.float32, device="cuda")
    api.moe_decode_layer(layer.weights, x.cuda(), y, ws,
                         residual=residual.cuda() if residual is not None else None,
                         topk_override=override.cuda() if override is not None else None,
                         topk_ids_out=ids, topk_w_out=gw)
    status = api.mdw_device_status(ws)
    return dict(y=y, ws=ws, ids=ids.cpu().numpy(), gates=gw.cpu().numpy(), status=status)


def check_layer(layer, x, out, override=None, tokens=None):
    """Full step-by-step parity of one call; returns the teacher-forced y. Codes, routing, union
    and pairs are checked for every token; h, hq and y for the given tokens (default: all)."""
    m = x.shape[0]
    tokens = set(range(m)) if tokens is None else set(tokens)
    K = layer.K
    assert out["status"] == 0
    ws = out["ws"]
    lay = api.mdw_moe_workspace_layout(layer.weights, m)
    hdr = read_ws(ws, lay["header"], np.uint32, 64)
    S, P, R = int(hdr[2]), int(hdr[3]), int(hdr[4])
    xn = bf16_to_np(x)
    # a1 activation quantisation
    xq_o, sx_o = OM.act_quant(xn)
    assert np.array_equal(read_ws(ws, lay["xq"], np.uint8, m * H).reshape(m, H), xq_o)
    assert np.array_equal(read_ws(ws, lay["sx"], np.float32, m), sx_o)
    # a2 router logits
    z_o = OM.router_logits(xn, layer.wr)
    z = read_ws(ws, lay["logits"], np.float32, m * layer.E).reshape(m, layer.E)
    assert_bar(z, z_o, "router logits", rtol=1e-4, atol=1e-5)
    # a3 selection and gates
    if override is None:
        ids_o, g_o = OM.route(z_o, K)
    else:
        ids_o = np.asarray(override, dtype=np.int64)
        g_o = OM.gates_for(z_o, ids_o)
    assert np.array_equal(out["ids"], ids_o)
    assert np.array_equal(read_ws(ws, lay["ids"], np.int32, m * K).reshape(m, K), ids_o)
    assert_bar(out["gates"], g_o, "gates", rtol=1e-5, atol=1e-6)
    # a4 union and pairs
    union = OM.expert_union(ids_o)
    first = 1 if layer.has_shared else 0
    slots = read_ws(ws, lay["slot_expert"], np.int32, S)
    assert R == len(union) and S == R + first
    assert list(slots[first:]) == list(union) and (first == 0 or slots[0] == -1)
    ptok = read_ws(ws, lay["pair_token"], np.int32, P)
    pslot = read_ws(ws, lay["pair_slot"], np.int32, P)
    pgate = read_ws(ws, lay["pair_gate"], np.float32, P)
    expect_pairs = [(s, t) for s in range(S) for t in range(m)
                    if (slots[s] < 0) or (slots[s] in set(ids_o[t].tolist()))]
    assert P == len(expect_pairs) == m * K + first * m
    assert list(zip(pslot.tolist(), ptok.tolist())) == expect_pairs
    # a5 / a6 per pair
    h = read_ws(ws, lay["h"], np.float32, P * I).reshape(P, I)
    hq = read_ws(ws, lay["hq"], np.uint8, P * I).reshape(P, I)
    sh = read_ws(ws, lay["sh"], np.float32, P)
    y_tf = np.zeros((m, H))
    for q in range(P):
        t, e = int(ptok[q]), int(slots[pslot[q]])
        if t not in tokens:
            continue
        w13q, w13s, w2q, w2s = layer.expert(e) if e >= 0 else layer.shared()
        gate, up = OM.expert_gate_up(w13q, w13s, xq_o[t], sx_o[t])
        h_o = OM.swiglu(gate, up)
        assert_bar(h[q], h_o, f"h of pair {q} (token {t}, expert {e})")
        hq_o, sh_o = F.quantize_fp8_lastdim(h[q][None, :])     # same fp32 input: bit-exact
        assert np.array_equal(hq[q], hq_o[0]) and sh[q] == sh_o[0]
        gw = 1.0 if e < 0 else g_o[t][list(ids_o[t]).index(e)]
        assert abs(pgate[q] - gw) <= 1e-6 * max(1.0, abs(gw))
        y_tf[t] += gw * OM.expert_down(w2q, w2s, hq[q], sh[q])
    return y_tf


def _e2e(layer, x, override=None, residual=None):
    return OM.moe_layer(bf16_to_np(x), layer.wr, layer.expert, layer.shared(), layer.K,
                        topk_override=override, residual=residual)["y"]


@pytest.mark.parametrize("m", [1, 2, 4, 8, 16])
def test_layer_parity_512(layer512, m):
    x = hidden_with_gap(10 + m, m, layer512.wr, layer512.K)
    out = run_layer(layer512, x)
    y = out["y"].cpu().numpy()
    y_tf = check_layer(layer512, x, out)
    assert_bar(y, y_tf, "y (teacher-forced hq)")
    y_e2e = _e2e(layer512, x)
    frac_ok = bar_ok(y, y_e2e).mean()
    assert frac_ok > 0.99, f"end-to-end y within the bar for only {frac_ok:.4f} of outputs"
    assert np.max(np.abs(y - y_e2e)) < 2e-2 * np.sqrt(np.mean(y_e2e ** 2))


def test_layer_parity_512_m32(layer512):
    """A 32-token window: the x-hat is kept as E4M3 codes in shared memory (converted in place
    from the router's bf16 rows in groups of 6 tokens) and each block's gate/up share runs in
    pieces. Codes, routing, union and pairs are checked for all 32 tokens; h and the teacher-
    forced y for tokens on both sides of conversion-group edges (5 | 6, 17 | 18) and in the
    short last group (30, 31)."""
    m = 32
    x = hidden_with_gap(42, m, layer512.wr, layer512.K)
    out = run_layer(layer512, x)
    toks = [0, 5, 6, 17, 18, 30, 31]
    y_tf = check_layer(layer512, x, out, tokens=toks)
    y = out["y"].cpu().numpy()
    assert np.isfinite(y).all()
    assert_bar(y[toks], y_tf[toks], "y (teacher-forced hq), M=32")


def test_layer_m32_zipf_override(layer512):
    """32 tokens under Zipf(1.1) popularity: popular experts carry many tokens, so their tiles
    have up to four 8-token column groups."""
    m = 32
    x = hidden_with_gap(43, m, layer512.wr, layer512.K)
    ov = synth.zipf_topk(44, m, num_experts=512, top_k=8)
    out = run_layer(layer512, x, override=torch.from_numpy(ov))
    toks = [0, 11, 31]
    y_tf = check_layer(layer512, x, out, override=ov, tokens=toks)
    y = out["y"].cpu().numpy()
    assert np.isfinite(y).all()
    assert_bar(y[toks], y_tf[toks], "y (teacher-forced hq), M=32 Zipf")


def test_layer_small_no_shared_topk4(layer64):
    for m in (1, 3):
        x = hidden_with_gap(40 + m, m, layer64.wr, layer64.K)
        out = run_layer(layer64, x)
        y_tf = check_layer(layer64, x, out)
        assert_bar(out["y"].cpu().numpy(), y_tf, "y (E=64, top-4, no shared expert)")


def test_bf16_output_and_residual(layer512):
    """bf16 output = RNE(fp32 output + residual) bit for bit on the same device run (the
    kernel is deterministic), and within one bf16 step of the oracle."""
    m = 4
    x = hidden_with_gap(21, m, layer512.wr, layer512.K)
    res = synth.hidden_states(22, m, 0)
    o32 = run_layer(layer512, x, y_fp32=True)
    o16 = run_layer(layer512, x, y_fp32=False, residual=res)
    y32 = o32["y"].cpu().numpy().astype(np.float32)
    want = F.f32_to_bf16_bits(y32 + bf16_to_np(res).astype(np.float32))
    got = o16["y"].cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_determinism(layer512):
    x = hidden_with_gap(30, 4, layer512.wr, layer512.K)
    a = run_layer(layer512, x)["y"].cpu().numpy()
    b = run_layer(layer512, x)["y"].cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("union", [8, 16, 24, 32])
def test_verify_window_union(layer512, union):
    """Four tokens whose selections overlap so the window's union has 8/16/24/32 experts:
    tokens share base vectors (+0.01 N(0,1)); the bases have disjoint top-8 sets."""
    groups = {8: [0, 0, 0, 0], 16: [0, 0, 1, 1], 24: [0, 0, 1, 2], 32: [0, 1, 2, 3]}[union]
    wr, K = layer512.wr, layer512.K
    bases, sets = [], []
    attempt = 0
    while len(bases) < 4:
        b = synth.hidden_states(2, 1, attempt)
        attempt += 1
        bn = bf16_to_np(b)
        if not router_gap_ok(bn, wr, K, gap=0.05):
            continue
        s = set(OM.route(OM.router_logits(bn, wr), K)[0][0].tolist())
        if all(not (s & o) for o in sets):
            bases.append(b)
            sets.append(s)
    toks = []
    for t, g in enumerate(groups):
        for a in range(100):
            xt = synth.perturbed_states(2, bases[g], 1000 * t + a)
            xn = bf16_to_np(xt)
            if router_gap_ok(xn, wr, K) and set(OM.route(OM.router_logits(xn, wr), K)[0][0].tolist()) == sets[g]:
                toks.append(xt)
                break
    x = torch.cat(toks, 0)
    out = run_layer(layer512, x)
    y_tf = check_layer(layer512, x, out)
    lay = api.mdw_moe_workspace_layout(layer512.weights, 4)
    hdr = read_ws(out["ws"], lay["header"], np.uint32, 64)
    assert int(hdr[4]) == union
    assert_bar(out["y"].cpu().numpy(), y_tf, f"y (union {union})")


def test_topk_override(layer512):
    m = 3
    x = synth.hidden_states(50, m, 0)
    ov = synth.zipf_topk(4, m)
    out = run_layer(layer512, x, override=torch.from_numpy(ov))
    y_tf = check_layer(layer512, x, out, override=ov)
    assert_bar(out["y"].cpu().numpy(), y_tf, "y (imposed routing)")


def test_override_out_of_range_sets_device_status(layer512):
    x = synth.hidden_states(51, 2, 0)
    ov = torch.tensor([[0, 1, 2, 3, 4, 5, 6, 512], [0, 1, 2, 3, 4, 5, 6, 7]], dtype=torch.int32)
    out = run_layer(layer512, x, override=ov)
    assert out["status"] == 7            # MDW_ERR_DEVICE_BOUNDS, nothing written
    assert torch.isnan(out["y"]).all()
    ov = torch.tensor([[0, 1, 2, 3, 4, 5, 6, 6], [0, 1, 2, 3, 4, 5, 6, 7]], dtype=torch.int32)
    assert run_layer(layer512, x, override=ov)["status"] == 7


def test_device_weights_match_host_regeneration(layer512):
    """The generator gives the same expert bytes on the device and on the host."""
    _, w13q, w13s, w2q, w2s, sh = layer512.tensors
    for e in (0, 137, 511):
        host = layer512.expert(e)
        for dev, hst in zip((w13q[e], w13s[e], w2q[e], w2s[e]), host):
            assert np.array_equal(dev.cpu().numpy(), hst)
    for dev, hst in zip(sh, layer512.shared()):
        assert np.array_equal(dev.cpu().numpy(), hst)


def _widen_scales(s: torch.Tensor) -> torch.Tensor:
    """Move two thirds of the rows' E8M0 scales outside [113, 140] (the range in which the
    kernels fold the scale into their f16 weights): rows with row % 3 == 0 get 105..112
    (2^-22 .. 2^-15), row % 3 == 1 get 141..145 (2^14 .. 2^18), the rest keep theirs, and
    block 0 of every seventh row gets code 0 (2^-127). A row
    stays within one regime, so its dot products keep an fp32-friendly dynamic range (gate
    row j and up row 768 + j share a regime). Works on [.., rows, blocks] tensors."""
    rows, blocks = s.shape[-2], s.shape[-1]
    r = torch.arange(rows, device=s.device).view(rows, 1)
    b = torch.arange(blocks, device=s.device).view(1, blocks)
    k = (r % 3).expand(rows, blocks)
    lo = (105 + (r + b) % 8).to(torch.uint8)
    hi = (141 + (r + b) % 5).to(torch.uint8)
    out = torch.where(k == 0, lo, torch.where(k == 1, hi, s))
    # code 0 (2^-127, no normal float) in block 0 of every seventh row
    zero = ((r % 7 == 3) & (b == 0)).expand(rows, blocks)
    return torch.where(zero, torch.zeros_like(out), out)


class WideScaleLayer(Layer):
    """A layer whose E8M0 scales leave the f16-exact range: the kernels must take their
    fp32-scaling path for those blocks and still match the oracle."""

    def __init__(self):
        super().__init__(seed=11, layer=2, num_experts=64, top_k=8, shared=True)
        wr, w13q, w13s, w2q, w2s, sh = self.tensors
        w13s.copy_(_widen_scales(w13s))
        w2s.copy_(_widen_scales(w2s))
        sh[1].copy_(_widen_scales(sh[1]))
        sh[3].copy_(_widen_scales(sh[3]))

    def expert(self, e: int):
        if e not in self._cache:
            q13, s13, q2, s2 = synth.expert_tensors(self.seed, self.layer, e)
            self._cache[e] = (q13.numpy(), _widen_scales(s13).numpy(), q2.numpy(), _widen_scales(s2).numpy())
        return self._cache[e]


def test_scales_outside_f16_exact_range():
    layer = WideScaleLayer()
    _, w13q, w13s, w2q, w2s, sh = layer.tensors
    host = layer.expert(5)
    assert np.array_equal(w13s[5].cpu().numpy(), host[1]) and np.array_equal(w2s[5].cpu().numpy(), host[3])
    assert (host[1] < 113).any() and (host[1] > 140).any()
    for m in (1, 4):
        x = hidden_with_gap(60 + m, m, layer.wr, layer.K)
        out = run_layer(layer, x)
        y_tf = check_layer(layer, x, out)
        assert_bar(out["y"].cpu().numpy(), y_tf, f"y (scales outside the f16-exact range, M={m})")
