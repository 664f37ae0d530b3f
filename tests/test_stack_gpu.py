"""GPU parity of the decode-step weight stream (moe_decode_stack): L MoE layers on a bf16
pre-norm residual stream, then the FP8 head with argmax / top-29.

Teacher-forced per layer: the oracle's layer l is fed the device's r_l and must give the
device's r_{l+1} to within one bf16 step (both round r_l + y once to bf16; the device's y is
fp32, the oracle's float64, so a value on a rounding boundary may land on either side).
The head is checked on the oracle's logits of bf16(RMSNorm(r_L)); argmax / top-k are
compared where the oracle's margins exceed 1e-3.
"""

import numpy as np
import pytest
import torch

from moe_decode_weight_gb300 import api, synth
from oracle import lm_head as OL
from oracle import stack as OS

from _cases import Layer, assert_bar, bf16_to_np, norm_rounding_allowance

pytestmark = pytest.mark.gpu
H = 2560


def _bf16_step(v):
    _, e = np.frexp(np.abs(v))
    return np.ldexp(1.0, e - 1 - 7)


def _check_residual(r_gpu, r_next, y_oracle, what):
    """r_{l+1} = bf16(r_l + y): the device's y may differ from the oracle's by the parity bar
    (rel 2e-3, abs 1e-3 below 1) and each side rounds once, so an element may differ by the
    bar of y plus one bf16 step of the result (where r + y cancels, the bar dominates);
    almost every element must agree exactly."""
    diff = np.abs(r_gpu - r_next)
    ay = np.abs(y_oracle)
    bar = np.where(ay < 1.0, 1e-3, 2e-3 * ay)
    assert np.all(diff <= _bf16_step(r_next) * 1.0001 + bar + 1e-30), what
    assert (diff > 0).mean() < 0.01, f"{what}: {(diff > 0).mean():.4f} of r differ"


@pytest.fixture(scope="module")
def model():
    layers = [Layer(seed=3, layer=l, num_experts=64, top_k=8, shared=True) for l in range(3)]
    V = 20011
    w = synth.lm_head_weight(1, V)
    wd = w.cuda()
    q = torch.empty((V, H), dtype=torch.uint8, device="cuda")
    s = torch.empty(V, dtype=torch.float32, device="cuda")
    head = api.quantize_lm_head_fp8(wd, q, s)
    qo, so = OL.quantize_lm_head(bf16_to_np(w))
    return layers, head, (qo, so), V


@pytest.mark.parametrize("m", [1, 4])
def test_stack_teacher_forced(model, m):
    layers, head, (qo, so), V = model
    L, k = len(layers), 29
    r0 = synth.hidden_states(3, m, 0)
    ws = torch.zeros(api.mdw_stack_workspace_bytes([l.weights for l in layers], head, m, k),
                     dtype=torch.uint8, device="cuda")
    resid = torch.zeros((L + 1, m, H), dtype=torch.bfloat16, device="cuda")
    am = torch.full((m,), -1, dtype=torch.int32, device="cuda")
    ti = torch.full((m, k), -1, dtype=torch.int32, device="cuda")
    lg = torch.zeros((m, V), dtype=torch.float32, device="cuda")
    api.moe_decode_stack([l.weights for l in layers], head, r0.cuda(), am, ws, resid_out=resid,
                         logits=lg, topk=k, topk_idx=ti)
    assert api.mdw_device_status(ws) == 0
    rs = resid.float().cpu().numpy()
    assert np.array_equal(rs[0], bf16_to_np(r0))
    for l, layer in enumerate(layers):
        r_next, _, res = OS.layer_step(rs[l], layer.oracle_dict(), layer.K)
        _check_residual(rs[l + 1], r_next, res["y"], f"layer {l}")
    xf = OS.rmsnorm_bf16(rs[L])
    lo = OL.lm_head_fp8_logits(qo, so, xf)
    lgn = lg.cpu().numpy()
    allow = norm_rounding_allowance(rs[L], qo, so)
    assert_bar(lgn, lo, "stack head logits", extra=allow)
    order = np.stack([np.lexsort((np.arange(V), -lo[t])) for t in range(m)])
    tin = ti.cpu().numpy()
    for t in range(m):
        vals = lo[t, order[t, :k + 1]]
        clean = -np.diff(vals) > 1e-3 + 2 * allow[t].max()
        # compare the prefix of the ranking whose margins are all clean
        n = k if clean.all() else int(np.argmin(clean))
        assert np.array_equal(tin[t, :n], order[t, :n]), f"token {t}"
        if clean[0]:
            assert am.cpu().numpy()[t] == order[t, 0]


@pytest.mark.parametrize("m", [1, 4])
def test_stack_imposed_routing(model, m):
    """moe_decode_stack_routed: Zipf-popular routing imposed per layer (layer l uses seed 4 + l),
    teacher-forced against the oracle layer given the same ids."""
    layers, head, _, _ = model
    L = len(layers)
    ov = np.stack([synth.zipf_topk(4 + l, m, num_experts=64, top_k=8) for l in range(L)])
    r0 = synth.hidden_states(4, m, 0)
    ws = torch.zeros(api.mdw_stack_workspace_bytes([l.weights for l in layers], None, m, 1),
                     dtype=torch.uint8, device="cuda")
    resid = torch.zeros((L + 1, m, H), dtype=torch.bfloat16, device="cuda")
    api.moe_decode_stack_routed([l.weights for l in layers], None, r0.cuda(), None, ws,
                                torch.from_numpy(ov).cuda(), resid_out=resid)
    assert api.mdw_device_status(ws) == 0
    hdr = ws[:1024].cpu().numpy().view(np.uint32)
    rs = resid.float().cpu().numpy()
    for l, layer in enumerate(layers):
        assert int(hdr[64 + l]) == len(set(ov[l].reshape(-1).tolist()))
        r_next, _, res = OS.layer_step(rs[l], layer.oracle_dict(), layer.K, topk_override=ov[l])
        _check_residual(rs[l + 1], r_next, res["y"], f"layer {l}")


def test_stack_imposed_routing_bounds(model):
    layers, _, _, _ = model
    m, L = 2, len(layers)
    ov = np.stack([synth.zipf_topk(4 + l, m, num_experts=64, top_k=8) for l in range(L)])
    ov[1, 1, 3] = 64                      # out of range in layer 1: the launch stops there
    ws = torch.zeros(api.mdw_stack_workspace_bytes([l.weights for l in layers], None, m, 1),
                     dtype=torch.uint8, device="cuda")
    resid = torch.zeros((L + 1, m, H), dtype=torch.bfloat16, device="cuda")
    api.moe_decode_stack_routed([l.weights for l in layers], None, synth.hidden_states(5, m, 0).cuda(), None,
                                ws, torch.from_numpy(ov).cuda(), resid_out=resid)
    assert api.mdw_device_status(ws) == 7


def test_stack_m32_imposed_routing_with_head(model):
    """A 32-token window through the stack and the FP8 head (which runs as two 16-token
    launches): every layer teacher-forced on tokens 0, 6 and 31 (tokens are independent), the
    head's logits and top-k checked for all 32 tokens."""
    layers, head, (qo, so), V = model
    L, m, k = len(layers), 32, 29
    ov = np.stack([synth.zipf_topk(40 + l, m, num_experts=64, top_k=8) for l in range(L)])
    r0 = synth.hidden_states(6, m, 0)
    ws = torch.zeros(api.mdw_stack_workspace_bytes([l.weights for l in layers], head, m, k),
                     dtype=torch.uint8, device="cuda")
    resid = torch.zeros((L + 1, m, H), dtype=torch.bfloat16, device="cuda")
    am = torch.full((m,), -1, dtype=torch.int32, device="cuda")
    ti = torch.full((m, k), -1, dtype=torch.int32, device="cuda")
    lg = torch.zeros((m, V), dtype=torch.float32, device="cuda")
    api.moe_decode_stack_routed([l.weights for l in layers], head, r0.cuda(), am, ws,
                                torch.from_numpy(ov).cuda(), resid_out=resid, logits=lg, topk=k, topk_idx=ti)
    assert api.mdw_device_status(ws) == 0
    hdr = ws[:1024].cpu().numpy().view(np.uint32)
    rs = resid.float().cpu().numpy()
    toks = [0, 6, 31]
    for l, layer in enumerate(layers):
        assert int(hdr[64 + l]) == len(set(ov[l].reshape(-1).tolist()))
        r_next, _, res = OS.layer_step(rs[l][toks], layer.oracle_dict(), layer.K, topk_override=ov[l][toks])
        _check_residual(rs[l + 1][toks], r_next, res["y"], f"layer {l}")
    lo = OL.lm_head_fp8_logits(qo, so, OS.rmsnorm_bf16(rs[L]))
    allow = norm_rounding_allowance(rs[L], qo, so)
    assert_bar(lg.cpu().numpy(), lo, "stack head logits (32 tokens)", extra=allow)
    tin, amn = ti.cpu().numpy(), am.cpu().numpy()
    for t in range(m):
        order = np.lexsort((np.arange(V), -lo[t]))
        clean = -np.diff(lo[t, order[:k + 1]]) > 1e-3 + 2 * allow[t].max()
        n = k if clean.all() else int(np.argmin(clean))
        assert np.array_equal(tin[t, :n], order[:n]), f"token {t}"
        if clean[0]:
            assert amn[t] == order[0]
