"""Pins of the oracle's MoE layer: brute-force routing, closed-form experts, dense MLP.

Each pin compares the oracle (oracle/moe.py) with an independent computation: a full
sort for the top-k, scipy's softmax for the gates, dense float64 matmuls on matrices
packed by a test-side encoder for the expert GEMVs, and closed forms for one-hot
experts and the weighted combine. ``test_planted_*`` patch a plausible mistake into the
oracle and check that a pin catches it.
"""

import numpy as np
from scipy.special import expit, softmax

import oracle.moe as OM
from oracle import formats as F

from _mx_helpers import pack, random_mx_matrix

H, I, E = 256, 64, 16


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(0)
    for _ in range(200):
        n = int(rng.integers(2, 40))
        k = int(rng.integers(1, n + 1))
        v = rng.integers(-4, 5, size=(3, n)).astype(np.float64)   # many ties
        got = OM.topk_desc(v, k)
        for r in range(3):
            ref = sorted(range(n), key=lambda i: (-v[r, i], i))[:k]
            assert list(got[r]) == ref


def test_route_gates_are_renormalised_softmax():
    rng = np.random.default_rng(1)
    z = rng.standard_normal((5, 512))
    for k in (1, 2, 8):
        ids, g = OM.route(z, k)
        full = softmax(z, axis=1)
        sel = np.take_along_axis(full, ids, axis=1)
        assert np.allclose(g, sel / sel.sum(axis=1, keepdims=True), rtol=1e-12, atol=0)
        assert np.allclose(g.sum(axis=1), 1.0, rtol=0, atol=1e-12)
        assert np.all(np.diff(np.take_along_axis(z, ids, axis=1), axis=1) <= 0)
    ids1, g1 = OM.route(z, 1)
    assert np.all(g1 == 1.0) and np.array_equal(ids1[:, 0], np.argmax(z, axis=1))


def test_union_is_set_of_selected():
    rng = np.random.default_rng(2)
    ids = rng.integers(0, 512, size=(4, 8))
    assert list(OM.expert_union(ids)) == sorted(set(ids.reshape(-1).tolist()))


def test_mxfp4_dequant_matches_dense_construction():
    rng = np.random.default_rng(3)
    w, codes, exps = random_mx_matrix(rng, 48, 256)
    q, s = pack(codes, exps)
    assert np.array_equal(OM.mxfp4_dequant(q, s), w)


def _dense_mlp_case(seed=4, m=3):
    rng = np.random.default_rng(seed)
    w1, c1, e1 = random_mx_matrix(rng, I, H)
    w3, c3, e3 = random_mx_matrix(rng, I, H)
    w2, c2, e2 = random_mx_matrix(rng, H, I)
    q13, s13 = pack(np.concatenate([c1, c3]), np.concatenate([e1, e3]))
    q2, s2 = pack(c2, e2)
    x = F.bf16_bits_to_float(F.f32_to_bf16_bits(rng.standard_normal((m, H)).astype(np.float32)))
    return (w1, w3, w2), (q13, s13, q2, s2), x


def _dense_expected(w1, w3, w2, x):
    """Dense float64 MLP with the W4A8 activation quantisation of reading R4."""
    xq, sx = F.quantize_fp8_lastdim(x)
    xt = F.e4m3_to_float(xq) * sx[:, None]
    gate, up = xt @ w1.T, xt @ w3.T
    h = gate * expit(gate) * up
    hq, sh = F.quantize_fp8_lastdim(h.astype(np.float32))
    return (F.e4m3_to_float(hq) * sh[:, None]) @ w2.T


def dense_pin_holds():
    (w1, w3, w2), packed, x = _dense_mlp_case()
    expected = _dense_expected(w1, w3, w2, x)
    wr = np.zeros((1, H), np.float32)          # one expert, top-1: gate weight 1
    res = OM.moe_layer(x, wr, lambda e: packed, None, top_k=1)
    return np.allclose(res["y"], expected, rtol=1e-10, atol=1e-10)


def test_top1_single_expert_is_dense_mlp():
    assert dense_pin_holds()


def test_identity_expert_closed_form():
    """W1 = W3 = [I | 0] (code 0b0010 = 1.0, scale 2^0), W2 = one-hot back-map:
    y_r = s_h * e4m3(hq_r) for r < I with h_j = silu(x~_j) * x~_j, and 0 for r >= I."""
    codes13 = np.zeros((2 * I, H), np.uint8)
    codes13[np.arange(I), np.arange(I)] = 0b0010
    codes13[I + np.arange(I), np.arange(I)] = 0b0010
    codes2 = np.zeros((H, I), np.uint8)
    codes2[np.arange(I), np.arange(I)] = 0b0010
    q13, s13 = pack(codes13, np.zeros((2 * I, H // 32), int))
    q2, s2 = pack(codes2, np.zeros((H, I // 32), int))
    rng = np.random.default_rng(6)
    x = F.bf16_bits_to_float(F.f32_to_bf16_bits(rng.standard_normal((2, H)).astype(np.float32)))
    res = OM.moe_layer(x, np.zeros((1, H), np.float32), lambda e: (q13, s13, q2, s2), None, 1)
    xq, sx = F.quantize_fp8_lastdim(x)
    xt = F.e4m3_to_float(xq) * sx[:, None]
    for t in range(2):
        h = xt[t, :I] * expit(xt[t, :I]) * xt[t, :I]
        hq, sh = F.quantize_fp8_lastdim(h.astype(np.float32))
        assert np.allclose(res["y"][t, :I], F.e4m3_to_float(hq) * sh, rtol=1e-12, atol=0)
        assert not res["y"][t, I:].any()


def test_combine_closed_form_with_shared():
    """Experts that differ only by a power-of-two W2 scale c_e: y = base * (sum_i g_i c_i
    + c_shared), where base is the output of the scale-1 expert."""
    (w1, w3, w2), (q13, s13, q2, s2), x = _dense_mlp_case(seed=8, m=4)
    rng = np.random.default_rng(9)
    wr = F.bf16_bits_to_float(F.f32_to_bf16_bits(
        (rng.standard_normal((E, H)) * 0.02).astype(np.float32)))
    cexp = {e: int(e % 3) for e in range(E)}
    experts = lambda e: (q13, s13, q2, (s2.astype(int) + cexp[e]).astype(np.uint8))
    shared = (q13, s13, q2, (s2.astype(int) + 2).astype(np.uint8))
    res = OM.moe_layer(x, wr, experts, shared, top_k=4)
    base = _dense_expected(w1, w3, w2, x)
    z = x.astype(np.float64) @ wr.astype(np.float64).T
    for t in range(4):
        ids = sorted(range(E), key=lambda e: (-z[t, e], e))[:4]
        g = softmax(z[t, ids])
        c = sum(gi * 2.0 ** cexp[e] for gi, e in zip(g, ids)) + 4.0
        assert list(res["ids"][t]) == ids
        assert np.allclose(res["y"][t], base[t] * c, rtol=1e-10, atol=1e-9)


def test_zero_routed_experts_leave_the_shared_expert():
    """Routed experts whose codes are all zero (E2M1 0 = +0, any scale) contribute exactly
    nothing, so y is the shared expert's dense MLP alone (gate 1), whatever the routing."""
    (w1, w3, w2), packed, x = _dense_mlp_case(seed=12, m=3)
    q13, s13, q2, s2 = packed
    zero = (np.zeros_like(q13), s13, np.zeros_like(q2), s2)
    wr = np.random.default_rng(13).standard_normal((E, H)).astype(np.float32) * 0.02
    res = OM.moe_layer(x, wr, lambda e: zero, packed, top_k=4)
    assert np.allclose(res["y"], _dense_expected(w1, w3, w2, x), rtol=1e-10, atol=1e-9)
    assert len(res["union"]) >= 4


def test_topk_override_uses_given_ids():
    (w1, w3, w2), packed, x = _dense_mlp_case(seed=10, m=2)
    wr = np.random.default_rng(1).standard_normal((E, H)).astype(np.float32) * 0.02
    ov = np.array([[3, 1], [7, 3]])
    res = OM.moe_layer(x, wr, lambda e: packed, None, top_k=2, topk_override=ov)
    z = x.astype(np.float64) @ wr.astype(np.float64).T
    assert np.array_equal(res["ids"], ov)
    assert np.allclose(res["gates"], softmax(np.take_along_axis(z, ov, 1), axis=1))
    assert list(res["union"]) == [1, 3, 7]


# ----------------------------------------------------------------- planted mistakes


def test_planted_nibble_order_is_caught(monkeypatch):
    real = OM.mxfp4_dequant

    def swapped(q, s):
        q = np.asarray(q, np.uint8)
        return real(((q >> 4) | (q << 4)).astype(np.uint8), s)
    monkeypatch.setattr(OM, "mxfp4_dequant", swapped)
    assert not dense_pin_holds()


def test_planted_gate_up_swap_is_caught(monkeypatch):
    real = OM.expert_gate_up
    monkeypatch.setattr(OM, "expert_gate_up", lambda *a: real(*a)[::-1])
    assert not dense_pin_holds()


def test_planted_scale_bias_is_caught(monkeypatch):
    real = OM.e8m0_to_float
    monkeypatch.setattr(OM, "e8m0_to_float", lambda b: real(np.asarray(b).astype(int) + 1))
    assert not dense_pin_holds()


def test_planted_sign_drop_is_caught(monkeypatch):
    monkeypatch.setattr(OM, "E2M1_LUT", np.abs(OM.E2M1_LUT))
    assert not dense_pin_holds()


def test_planted_missing_activation_scale_is_caught(monkeypatch):
    real = OM.mx_gemv
    monkeypatch.setattr(OM, "mx_gemv", lambda q, s, a, sa: real(q, s, a, 1.0))
    assert not dense_pin_holds()
