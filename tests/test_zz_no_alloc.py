"""The allocation-free entry point (moe_decode_layer_noalloc) gives the same results as
moe_decode_layer on two calls in a row.

It exists for callers that cannot allocate device memory (a host framework that owns the
device-memory budget, C callers without an allocator, loops where cudaMalloc would
synchronise the device). This file is named to be collected last, so a run that stops at
the first failure has already run every other test.
"""

import numpy as np
import pytest
import torch

from moe_decode_weight_gb300 import api, synth

from _cases import Layer, assert_bar, hidden_with_gap

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def layer():
    return Layer(seed=12, layer=1, num_experts=512, top_k=8, shared=True)


def _reference(layer, x):
    m = x.shape[0]
    ws = torch.zeros(api.mdw_moe_workspace_bytes(layer.weights, m), dtype=torch.uint8, device="cuda")
    y = torch.empty((m, 2560), dtype=torch.float32, device="cuda")
    ids = torch.empty((m, layer.K), dtype=torch.int32, device="cuda")
    api.moe_decode_layer(layer.weights, x, y, ws, topk_ids_out=ids)
    assert api.mdw_device_status(ws) == 0
    return y.cpu().numpy(), ids.cpu().numpy()


def test_noalloc_matches_workspace_entry_point_twice(layer):
    # the largest window first (it fills the most of the shared array), then smaller ones: the
    # leftovers of an earlier, larger call must not leak into a later one
    xs = [hidden_with_gap(73, 32, layer.wr, layer.K).cuda(), hidden_with_gap(74, 16, layer.wr, layer.K).cuda(),
          hidden_with_gap(70, 1, layer.wr, layer.K).cuda(), hidden_with_gap(71, 4, layer.wr, layer.K).cuda()]
    refs = [_reference(layer, x) for x in xs]
    for x, (y_ref, ids_ref) in zip(xs, refs):             # two calls in a row
        m = x.shape[0]
        y = torch.full((m, 2560), float("nan"), dtype=torch.float32, device="cuda")
        ids = torch.full((m, layer.K), -1, dtype=torch.int32, device="cuda")
        status = torch.full((1,), 0xFFFF, dtype=torch.int32, device="cuda")
        api.moe_decode_layer_noalloc(layer.weights, x, y, topk_ids_out=ids, device_status_out=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert np.array_equal(ids.cpu().numpy(), ids_ref)
        assert_bar(y.cpu().numpy(), y_ref, f"noalloc y (M={m})")


def test_noalloc_rejects_bad_arguments(layer):
    x = synth.hidden_states(72, 1, 0).cuda()
    y = torch.empty((1, 2560), dtype=torch.float32, device="cuda")
    lw = layer.weights
    bad = api.MoeWeights(lw.router_w, lw.w13_q, lw.w13_s, lw.w2_q, lw.w2_s, lw.shared, lw.top_k)
    bad.c.magic = 0                                  # not a weight handle of this library
    with pytest.raises(api.MdwError) as e:
        api.moe_decode_layer_noalloc(bad, x, y)
    assert e.value.code == 3
    with pytest.raises(api.MdwError) as e:
        api.moe_decode_layer_noalloc(layer.weights, torch.empty((0, 2560), dtype=torch.bfloat16, device="cuda"), y)
    assert e.value.code == 1
