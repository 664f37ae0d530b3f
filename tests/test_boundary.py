"""The C-ABI boundary on the host: the library loads, exports every entry point that
include/moe_decode_weight.h declares, and rejects bad arguments before enqueuing anything.

These tests never give a fully valid call: every call here fails a host-side check that
runs before any CUDA call, so the fake (aligned, never dereferenced) addresses used for
device pointers are never touched.
"""

import ctypes as C
import os
import re

import pytest

from moe_decode_weight_gb300 import api

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "moe_decode_weight.h")
FAKE = 0x7F0000000000          # 16-byte aligned placeholder address


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)) - {"defined"})


def _weights(**kw):
    w = api.MoeWeightsC(api.MDW_MAGIC, api.FMT_MXFP4, 512, 8, 2560, 768,
                        FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)
    for k, v in kw.items():
        setattr(w, k, v)
    return w


def test_header_declarations_match_exports():
    lib = api.lib()
    declared = _declared()
    assert set(declared) == set(api.SYMBOLS)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings_and_version():
    for code, name in api.STATUS.items():
        assert api.mdw_status_string(code) == name
    assert api.mdw_status_string(99) == "MDW_ERR_UNKNOWN"
    assert api.mdw_version() >= 100


def test_workspace_queries_validate():
    lib = api.lib()
    w = _weights()
    assert lib.mdw_moe_workspace_bytes(C.byref(w), 1) > 0
    assert lib.mdw_moe_workspace_bytes(C.byref(w), 4) > lib.mdw_moe_workspace_bytes(C.byref(w), 1)
    assert lib.mdw_moe_workspace_bytes(C.byref(w), 0) == 0
    assert lib.mdw_moe_workspace_bytes(C.byref(w), api.MAX_M + 1) == 0
    assert lib.mdw_moe_workspace_bytes(C.byref(_weights(magic=1)), 1) == 0
    lay = api.MoeWsLayoutC()
    assert lib.mdw_moe_workspace_layout(C.byref(w), 4, C.byref(lay)) == 0
    offs = [getattr(lay, n) for n, _ in api.MoeWsLayoutC._fields_]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert lay.total == lib.mdw_moe_workspace_bytes(C.byref(w), 4)


@pytest.mark.parametrize("field,value,code", [
    ("magic", 0, 3), ("fmt", api.FMT_FP8, 3), ("hidden", 4096, 2), ("inter", 512, 2),
    ("num_experts", 0, 2), ("num_experts", 513, 2), ("top_k", 0, 1), ("top_k", 9, 1),
    ("w13_q", FAKE + 8, 1), ("router_w", None, 1), ("sh_w2_s", None, 1),
])
def test_moe_decode_layer_rejects(field, value, code):
    lib = api.lib()
    w = _weights(**{field: value})
    r = lib.moe_decode_layer(C.byref(w), 1, FAKE, FAKE, 1, None, None, None, None, FAKE, 1 << 30, None)
    assert r == code


def test_moe_decode_layer_rejects_args():
    lib = api.lib()
    w = _weights()
    call = lambda m, x, y, ws, nbytes: lib.moe_decode_layer(C.byref(w), m, x, y, 1, None, None, None,
                                                           None, ws, nbytes, None)
    assert call(0, FAKE, FAKE, FAKE, 1 << 30) == 1
    assert call(api.MAX_M + 1, FAKE, FAKE, FAKE, 1 << 30) == 1
    assert call(1, FAKE + 4, FAKE, FAKE, 1 << 30) == 1
    assert call(1, FAKE, None, FAKE, 1 << 30) == 1
    assert call(1, FAKE, FAKE, FAKE, 1024) == 4            # workspace too small


def test_head_format_tag_is_checked():
    """An FP8 head handed to the BF16 entry point (or the reverse) is an error at the call,
    never a silent reinterpretation of the bytes (the pages' FP8/BF16 integration trap)."""
    lib = api.lib()
    fp8 = api.LMHeadC(api.MDW_MAGIC, api.FMT_FP8, 157184, 2560, 0, FAKE, FAKE)
    bf16 = api.LMHeadC(api.MDW_MAGIC, api.FMT_BF16, 157184, 2560, 0, FAKE, None)
    args = lambda h: (C.byref(h), 1, FAKE, None, FAKE, 1, None, None, FAKE, 1 << 30, None)
    assert lib.lm_head_bf16(*args(fp8)) == 3
    assert lib.lm_head_fp8(*args(bf16)) == 3
    bad = api.LMHeadC(0, api.FMT_FP8, 157184, 2560, 0, FAKE, FAKE)
    assert lib.lm_head_fp8(*args(bad)) == 3
    stack_layers = (api.MoeWeightsC * 1)(_weights())
    assert lib.moe_decode_stack(stack_layers, 1, C.byref(bf16), 1, FAKE, None, None, FAKE, 1, None,
                                None, FAKE, 1 << 30, None) == 3


def test_quantize_and_bf16_init_validate():
    lib = api.lib()
    head = api.LMHeadC()
    assert lib.quantize_lm_head_fp8(FAKE, 157184, 4096, FAKE, FAKE, C.byref(head), None) == 2
    assert lib.quantize_lm_head_fp8(FAKE, 0, 2560, FAKE, FAKE, C.byref(head), None) == 2
    assert lib.quantize_lm_head_fp8(FAKE + 2, 10, 2560, FAKE, FAKE, C.byref(head), None) == 1
    assert lib.mdw_lm_head_bf16_init(FAKE, 157184, 2560, C.byref(head)) == 0
    assert head.magic == api.MDW_MAGIC and head.fmt == api.FMT_BF16 and head.vocab == 157184
    assert lib.mdw_lm_head_bf16_init(None, 10, 2560, C.byref(head)) == 1


def test_stack_rejects_mixed_layers():
    lib = api.lib()
    head = api.LMHeadC(api.MDW_MAGIC, api.FMT_FP8, 157184, 2560, 0, FAKE, FAKE)
    layers = (api.MoeWeightsC * 2)(_weights(), _weights(top_k=4))
    assert lib.moe_decode_stack(layers, 2, C.byref(head), 1, FAKE, None, None, FAKE, 1, None, None,
                                FAKE, 1 << 30, None) == 1
    layers = (api.MoeWeightsC * 2)(_weights(), _weights(fmt=api.FMT_BF16))
    assert lib.moe_decode_stack(layers, 2, C.byref(head), 1, FAKE, None, None, FAKE, 1, None, None,
                                FAKE, 1 << 30, None) == 3
    assert lib.moe_decode_stack(layers, 0, C.byref(head), 1, FAKE, None, None, FAKE, 1, None, None,
                                FAKE, 1 << 30, None) == 1


def _define(name):
    m = re.search(r"#define\s+" + name + r"\s+\(?(\d+)u?(?:\s*<<\s*(\d+))?\)?", open(HEADER).read())
    assert m, name
    return int(m.group(1)) << int(m.group(2) or 0)


def test_binding_limits_match_the_header():
    assert api.MAX_M == _define("MDW_MAX_M")
    assert api.MAX_TOPK == _define("MDW_MAX_TOPK")
    assert api.MAX_VOCAB_TOPK == _define("MDW_MAX_VOCAB_TOPK")
    assert api.MAX_EXPERTS == _define("MDW_MAX_EXPERTS")


def test_noalloc_scratch_holds_the_largest_layer_workspace():
    """moe_decode_layer_noalloc must accept every shape moe_decode_layer accepts: the workspace
    of the largest window (M = MDW_MAX_M, 512 experts, top-8) fits the compiled-in scratch."""
    lib = api.lib()
    w = _weights()
    biggest = lib.mdw_moe_workspace_bytes(C.byref(w), api.MAX_M)
    assert 0 < biggest <= _define("MDW_NOALLOC_SCRATCH_BYTES")


@pytest.mark.parametrize("m", [1, 2, 3, 4, 8, 16, 17, 31, 32])
def test_workspace_regions_hold_their_arrays(m):
    """Every region of the moe_decode_layer workspace holds the array the header documents
    for M tokens (P = M (top_k + 1) pairs, S = M top_k + 1 slots), for every window size."""
    lib = api.lib()
    w = _weights()
    lay = api.MoeWsLayoutC()
    assert lib.mdw_moe_workspace_layout(C.byref(w), m, C.byref(lay)) == 0
    E, K, H, I = 512, 8, 2560, 768
    P, S = m * (K + 1), m * K + 1
    need = {"header": 256 * 4, "xq": m * H, "sx": m * 4, "logits": m * E * 4, "ids": m * K * 4,
            "gates": m * K * 4, "slot_expert": S * 4, "pair_token": P * 4, "pair_slot": P * 4,
            "pair_gate": P * 4, "h": P * I * 4, "hq": P * I, "sh": P * 4}
    names = [n for n, _ in api.MoeWsLayoutC._fields_]
    for a, b in zip(names, names[1:]):
        assert getattr(lay, b) - getattr(lay, a) >= need[a], a


@pytest.mark.parametrize("m", [1, 2, 3, 32])
def test_stack_workspace_holds_the_head_logits_above_two_tokens(m):
    """Above two tokens the head selects from fp32 logits it writes to the workspace, so the
    stack's workspace grows by at least M * V * 4 bytes when a head is given; up to two tokens
    the head keeps its lists in registers and needs only the candidate lists."""
    lib = api.lib()
    V = 157184
    head = api.LMHeadC(api.MDW_MAGIC, api.FMT_FP8, V, 2560, 0, FAKE, FAKE)
    layers = (api.MoeWeightsC * 1)(_weights())
    with_head = lib.mdw_stack_workspace_bytes(layers, 1, C.byref(head), m, 29)
    without = lib.mdw_stack_workspace_bytes(layers, 1, None, m, 29)
    assert with_head > without > 0
    if m > 2:
        assert with_head - without >= m * V * 4
    else:
        assert with_head - without < m * V * 4
