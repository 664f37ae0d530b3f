"""The full decode step in the launch configuration the bench times.

The configuration is 42 layers of 512 routed experts plus the shared expert, in one
moe_decode_stack launch, followed by the FP8 head over all 157,184 rows. The checks use
samples the oracle computes in seconds:

* teacher-forced layers 0, 20 and 41: the oracle's layer fed the device's r_l must give the
  device's r_{l+1};
* the head's logits of bf16(RMSNorm(r_42)) on 20,000 sampled vocabulary rows, at the bar;
* the fused top-29 and argmax against a full sort of the kernel's own logits (a property
  that holds at any size).
"""

import numpy as np
import pytest
import torch

from moe_decode_weight_gb300 import api, synth
from oracle import lm_head as OL
from oracle import stack as OS

from _cases import Layer, assert_bar, bf16_to_np, norm_rounding_allowance
from test_stack_gpu import _check_residual

pytestmark = pytest.mark.gpu
H, L, E, K, TOPK = 2560, 42, 512, 8, 29


@pytest.fixture(scope="module")
def full_model():
    layers = [Layer(seed=3, layer=l, num_experts=E, top_k=K, shared=True) for l in range(L)]
    w = synth.lm_head_weight(1, synth.VOCAB)
    wd = w.cuda()
    q = torch.empty((synth.VOCAB, H), dtype=torch.uint8, device="cuda")
    s = torch.empty(synth.VOCAB, dtype=torch.float32, device="cuda")
    head = api.quantize_lm_head_fp8(wd, q, s)
    torch.cuda.synchronize()
    del wd
    return layers, head, w


@pytest.mark.parametrize("m", [1, 4])
def test_full_step_sampled(full_model, m):
    layers, head, w = full_model
    V = synth.VOCAB
    r0 = synth.hidden_states(3, m, 100)                 # the bench's first step input
    ws = torch.zeros(api.mdw_stack_workspace_bytes([l.weights for l in layers], head, m, TOPK),
                     dtype=torch.uint8, device="cuda")
    resid = torch.zeros((L + 1, m, H), dtype=torch.bfloat16, device="cuda")
    am = torch.full((m,), -1, dtype=torch.int32, device="cuda")
    ti = torch.full((m, TOPK), -1, dtype=torch.int32, device="cuda")
    lg = torch.zeros((m, V), dtype=torch.float32, device="cuda")
    api.moe_decode_stack([l.weights for l in layers], head, r0.cuda(), am, ws, resid_out=resid,
                         logits=lg, topk=TOPK, topk_idx=ti)
    assert api.mdw_device_status(ws) == 0
    rs = resid.float().cpu().numpy()
    assert np.array_equal(rs[0], bf16_to_np(r0))
    assert np.isfinite(rs).all()
    for l in (0, 20, L - 1):
        r_next, _, res = OS.layer_step(rs[l], layers[l].oracle_dict(), K)
        _check_residual(rs[l + 1], r_next, res["y"], f"layer {l}")
    # the head on sampled rows of the final residual, at the bar (the device normalises in
    # fp32, the oracle in float64: an input element whose bf16 rounding sits at a tie may land
    # one step apart, which the oracle-derived allowance bounds)
    xf = OS.rmsnorm_bf16(rs[L])
    rows = np.unique(np.concatenate([[0, V - 1], np.random.default_rng(1).integers(0, V, 20000)]))
    qo, so = OL.quantize_lm_head(bf16_to_np(w[torch.from_numpy(rows)]))
    lgn = lg.cpu().numpy()
    allow = norm_rounding_allowance(rs[L], qo, so)
    assert_bar(lgn[:, rows], OL.lm_head_fp8_logits(qo, so, xf), "sampled head logits", extra=allow)
    own = np.stack([np.lexsort((np.arange(V), -lgn[t]))[:TOPK] for t in range(m)])
    assert np.array_equal(ti.cpu().numpy(), own)
    assert np.array_equal(am.cpu().numpy(), own[:, 0])
