"""Bounded inter-block waits: a wait that runs out ends the launch with MDW_ERR_TIMEOUT in
the status word, and the device context stays usable.

The MoE kernels' waits (the grid barrier and the tagged-word polls) give up after a budget of
clock64 cycles, record the status and leave; every other block leaves at its next wait once
the status is set, so the launch completes. The test shrinks the budget to one cycle through
the library's test hook, so the first block to wait gives up on its first poll: no GPU fault,
trap or hang is involved. The same call with the default budget then succeeds.
"""

import numpy as np
import pytest
import torch

from moe_decode_weight_gb300 import api, synth

from _cases import Layer

pytestmark = pytest.mark.gpu
H = 2560


@pytest.fixture(scope="module")
def layers():
    return [Layer(seed=21, layer=l, num_experts=64, top_k=8, shared=True) for l in range(2)]


def _layer_call(layer, x):
    m = x.shape[0]
    ws = torch.zeros(api.mdw_moe_workspace_bytes(layer.weights, m), dtype=torch.uint8, device="cuda")
    y = torch.zeros((m, H), dtype=torch.float32, device="cuda")
    api.moe_decode_layer(layer.weights, x, y, ws)
    return api.mdw_device_status(ws), y


def _stack_call(layers, x):
    m = x.shape[0]
    ws = torch.zeros(api.mdw_stack_workspace_bytes([l.weights for l in layers], None, m, 1),
                     dtype=torch.uint8, device="cuda")
    resid = torch.zeros((len(layers) + 1, m, H), dtype=torch.bfloat16, device="cuda")
    api.moe_decode_stack([l.weights for l in layers], None, x, None, ws, resid_out=resid)
    return api.mdw_device_status(ws), resid


@pytest.mark.parametrize("m", [1, 4, 16])
@pytest.mark.parametrize("mode", ["layer", "stack"])
def test_wait_runs_out_and_context_survives(layers, m, mode):
    x = synth.hidden_states(22, m, 0).cuda()
    call = (lambda: _layer_call(layers[0], x)) if mode == "layer" else (lambda: _stack_call(layers, x))
    prev = api.mdw_debug_set_spin_budget(1)
    try:
        status, _ = call()
    finally:
        api.mdw_debug_set_spin_budget(prev)
    torch.cuda.synchronize()
    assert status == 6, api.STATUS.get(status, status)         # MDW_ERR_TIMEOUT
    # the context is intact: the same call with the default budget completes cleanly
    status, out = call()
    assert status == 0
    assert np.isfinite(out.float().cpu().numpy()).all()
