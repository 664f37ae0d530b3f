"""Pins of the oracle's stack glue: RMSNorm invariants, bf16 residual rounding, and a
tiny end-to-end decode step that is consistent with its own layers."""

import numpy as np

from oracle import formats as F
from oracle import stack as OS
from oracle import moe as OM

from _mx_helpers import pack, random_mx_matrix


def _bf16_half_step(v):
    """Half the bf16 spacing at |v|: bf16 keeps 8 significant bits."""
    _, e = np.frexp(np.abs(v))
    return np.ldexp(1.0, e - 1 - 8)


def test_rmsnorm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(0)
    r = F.round_f64_to_bf16(rng.standard_normal((4, 2560)) * 37.0)
    x = OS.rmsnorm_bf16(r).astype(np.float64)
    assert np.allclose(np.sqrt(np.mean(x * x, axis=1)), 1.0, atol=4e-3)
    assert np.array_equal(OS.rmsnorm_bf16(r * 8.0), OS.rmsnorm_bf16(r))   # power-of-two scale
    # each output is the nearest bf16 of the float64 normalised value
    exact = r / np.sqrt(np.mean(r.astype(np.float64) ** 2, axis=1, keepdims=True) + 1e-6)
    assert np.all(np.abs(x - exact) <= _bf16_half_step(exact))


def test_residual_add_is_one_rounding():
    rng = np.random.default_rng(1)
    r = F.round_f64_to_bf16(rng.standard_normal(1000) * 10)
    y = rng.standard_normal(1000) * 40
    out = OS.residual_add_bf16(r, y).astype(np.float64)
    exact = r.astype(np.float64) + y
    assert np.all(np.abs(out - exact) <= _bf16_half_step(exact))


def test_tiny_decode_step_consistent():
    H, I, E, V = 128, 64, 8, 300
    rng = np.random.default_rng(2)
    layers = []
    for l in range(3):
        ex = {}
        for e in range(E + 1):
            _, c13, e13 = random_mx_matrix(rng, 2 * I, H)
            _, c2, e2 = random_mx_matrix(rng, H, I)
            ex[e] = pack(c13, e13) + pack(c2, e2)
        wr = F.round_f64_to_bf16(rng.standard_normal((E, H)) * 0.02)
        layers.append(dict(wr=wr, experts=lambda e, ex=ex: ex[e], shared=ex[E]))
    w = F.round_f64_to_bf16(rng.standard_normal((V, H)) * 0.02)
    from oracle import lm_head as OL
    q, s = OL.quantize_lm_head(w)
    r0 = F.round_f64_to_bf16(rng.standard_normal((2, H)))
    out = OS.decode_step(r0, layers, q, s, top_k=2, k_vocab=5)
    assert len(out["r"]) == 4 and out["logits"].shape == (2, V)
    assert np.array_equal(out["argmax"], np.argmax(out["logits"], axis=1))
    # layer-by-layer replay equals the chained result (teacher-forced form of the stack)
    r1, x0, res0 = OS.layer_step(out["r"][0], layers[0], 2)
    assert np.array_equal(r1, out["r"][1])
    assert np.array_equal(res0["ids"], OM.route(OM.router_logits(x0, layers[0]["wr"]), 2)[0])
