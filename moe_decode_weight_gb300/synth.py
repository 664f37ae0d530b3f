"""Seeded synthetic inputs shaped like the pages' model (random bytes and normals only).

This module holds no arithmetic of the method: it draws the inputs that both the CUDA
path and the float64 oracle consume. Expert weights come from a counter-based integer
hash, so any single expert of any layer can be regenerated on the host (for the oracle)
with the same bytes the device holds, without materialising the other experts. The hash
uses only integer operations that give identical results on the CPU and on a CUDA device
(all products stay below 2**63).

Shapes and distributions (the model facts are from "Three MoE Inference Optimizations
NVIDIA Measured on DGX Spark", section "Decoding was memory-bound on a 124-billion-
parameter model at batch size 1", and runbyai.xyz/posts/593, paragraphs 2-4):

* routed experts E = 512 (+1 shared), hidden H = 2560, moe_intermediate I = 768, top 8;
* MXFP4 expert bytes uniform over 0..255 (every E2M1 nibble uniform over the 16 codes);
  E8M0 block scales uniform over {119, ..., 123} (2**-8 .. 2**-4);
* router weight [E, H] bf16 ~ N(0, 0.02); hidden states bf16 ~ N(0, 1);
* LM head weight [157184, H] bf16 ~ N(0, 0.02).
"""

from __future__ import annotations

import numpy as np
import torch

HIDDEN = 2560
INTER = 768
NUM_EXPERTS = 512
TOP_K = 8
VOCAB = 157184
TOPK_VOCAB = 29
NUM_LAYERS = 42
SCALE_MIN = 119          # E8M0 code of 2**-8
SCALE_SPAN = 5           # 119..123

_M32 = 0xFFFFFFFF

# tensor ids inside one layer
T_W13Q, T_W13S, T_W2Q, T_W2S = 1, 2, 3, 4
SHARED_EXPERT = NUM_EXPERTS   # expert id of the shared expert in the generator's key space


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2**32 for int64 x in [0, 2**32) without signed overflow."""
    lo = x & 0xFFFF
    hi = x >> 16
    return (lo * c + (((hi * c) & 0xFFFF) << 16)) & _M32


def _lowbias32(x: torch.Tensor) -> torch.Tensor:
    """A 32-bit integer finaliser (xor-shift / multiply, constants 0x7feb352d, 0x846ca68b)."""
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    return x ^ (x >> 16)


def _keys(seed: int, layer: int, tensor: int, experts: torch.Tensor) -> torch.Tensor:
    """Per-expert 32-bit stream keys (int64 tensor) for (seed, layer, tensor)."""
    e = experts.to(torch.int64)
    k = (seed * 0x9E37 + layer * 0x85EB + tensor * 0xC2B2 + e * 0x27D4) & _M32
    return _lowbias32(_lowbias32(k) ^ (((seed << 8) ^ (layer << 20) ^ tensor) & _M32))


def hash_bytes(seed: int, layer: int, tensor: int, experts, nbytes: int,
               device="cpu") -> torch.Tensor:
    """Pseudo-random bytes, uint8 [len(experts), nbytes], for (seed, layer, tensor, expert).

    Row i depends only on (seed, layer, tensor, experts[i]) and the byte index.
    """
    ex = torch.as_tensor(experts, dtype=torch.int64).reshape(-1).to(device)
    nwords = (nbytes + 3) // 4
    key = _keys(seed, layer, tensor, ex)[:, None]
    n = torch.arange(nwords, dtype=torch.int64, device=device)[None, :]
    w = _lowbias32(_lowbias32(n ^ key) ^ (key >> 3))
    b = torch.stack([(w >> s) & 0xFF for s in (0, 8, 16, 24)], dim=2).reshape(ex.numel(), -1)
    return b[:, :nbytes].to(torch.uint8)


def _scale_bytes(raw: torch.Tensor) -> torch.Tensor:
    return (SCALE_MIN + ((raw.to(torch.int32) * SCALE_SPAN) >> 8)).to(torch.uint8)


def experts_tensors(seed: int, layer: int, experts, hidden: int = HIDDEN, inter: int = INTER,
                    device="cpu"):
    """(w13_q [n, 2I, H/2], w13_s [n, 2I, H/32], w2_q [n, H, I/2], w2_s [n, H, I/32]) of the
    listed experts (the shared expert is id ``SHARED_EXPERT``)."""
    ex = torch.as_tensor(experts, dtype=torch.int64).reshape(-1)
    n = ex.numel()
    w13_q = hash_bytes(seed, layer, T_W13Q, ex, 2 * inter * hidden // 2, device)
    w13_s = _scale_bytes(hash_bytes(seed, layer, T_W13S, ex, 2 * inter * hidden // 32, device))
    w2_q = hash_bytes(seed, layer, T_W2Q, ex, hidden * inter // 2, device)
    w2_s = _scale_bytes(hash_bytes(seed, layer, T_W2S, ex, hidden * inter // 32, device))
    return (w13_q.view(n, 2 * inter, hidden // 2), w13_s.view(n, 2 * inter, hidden // 32),
            w2_q.view(n, hidden, inter // 2), w2_s.view(n, hidden, inter // 32))


def expert_tensors(seed: int, layer: int, expert: int, hidden: int = HIDDEN,
                   inter: int = INTER, device="cpu"):
    """The four tensors of one expert (no leading expert axis)."""
    return tuple(t[0] for t in experts_tensors(seed, layer, [expert], hidden, inter, device))


def layer_experts(seed: int, layer: int, num_experts: int = NUM_EXPERTS, hidden: int = HIDDEN,
                  inter: int = INTER, device="cpu", with_shared: bool = True,
                  chunk: int = 32, out=None):
    """All routed experts of a layer stacked [E, ...], plus the shared expert (or None).

    The bytes of expert e equal ``expert_tensors(seed, layer, e)``; the shared expert is
    generated under expert id ``SHARED_EXPERT`` whatever ``num_experts`` is. ``out`` may
    supply the four destination tensors (e.g. views into one device allocation).
    """
    shapes = [(2 * inter, hidden // 2), (2 * inter, hidden // 32),
              (hidden, inter // 2), (hidden, inter // 32)]
    if out is None:
        out = [torch.empty((num_experts,) + s, dtype=torch.uint8, device=device) for s in shapes]
    for e0 in range(0, num_experts, chunk):
        ids = torch.arange(e0, min(num_experts, e0 + chunk))
        for dst, src in zip(out, experts_tensors(seed, layer, ids, hidden, inter, device)):
            dst[e0:e0 + ids.numel()].copy_(src)
    shared = (expert_tensors(seed, layer, SHARED_EXPERT, hidden, inter, device)
              if with_shared else None)
    return tuple(out), shared


def _normal_bf16(seed_tuple, shape, std: float) -> torch.Tensor:
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(seed_tuple))))
    v = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        v *= np.float32(std)
    return torch.from_numpy(v).to(torch.bfloat16)


def router_weight(seed: int, layer: int, num_experts: int = NUM_EXPERTS,
                  hidden: int = HIDDEN) -> torch.Tensor:
    """Router weight [E, H], bf16 ~ N(0, 0.02), on the host."""
    return _normal_bf16((seed, layer, 101), (num_experts, hidden), 0.02)


def hidden_states(seed: int, m: int, attempt: int = 0, hidden: int = HIDDEN) -> torch.Tensor:
    """Token hidden states [M, H], bf16 ~ N(0, 1), on the host; ``attempt`` indexes redraws."""
    return _normal_bf16((seed, attempt, 202), (m, hidden), 1.0)


def perturbed_states(seed: int, base: torch.Tensor, attempt: int, std: float = 0.01) -> torch.Tensor:
    """bf16(base + std * N(0, 1)): tokens close to a base vector (verify-window groups)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, attempt, 303])))
    noise = rng.standard_normal(size=tuple(base.shape), dtype=np.float32) * np.float32(std)
    return (base.float() + torch.from_numpy(noise)).to(torch.bfloat16)


def lm_head_weight(seed: int, vocab: int = VOCAB, hidden: int = HIDDEN) -> torch.Tensor:
    """LM head weight [V, H], bf16 ~ N(0, 0.02), on the host."""
    return _normal_bf16((seed, 404), (vocab, hidden), 0.02)


def zipf_topk(seed: int, m: int, num_experts: int = NUM_EXPERTS, top_k: int = TOP_K,
              s: float = 1.1) -> np.ndarray:
    """Per token, ``top_k`` distinct experts drawn without replacement from a Zipf(s)
    popularity over a seeded permutation of the experts. int32 [M, top_k]."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 505])))
    perm = rng.permutation(num_experts)
    p = 1.0 / np.arange(1, num_experts + 1) ** s
    p /= p.sum()
    out = np.empty((m, top_k), dtype=np.int32)
    for t in range(m):
        out[t] = perm[rng.choice(num_experts, size=top_k, replace=False, p=p)]
    return out
