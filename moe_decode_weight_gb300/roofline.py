"""Algorithmic byte and flop counts of the decode step (host-side arithmetic only).

"Algorithmic" bytes are the bytes the method has to move: the router weight, each
selected expert once per call (the union of the window's selections, plus the shared
expert), the FP8 head with its row scales, the token inputs and the outputs. Unselected
experts are not counted. These are the numerators of every GB/s figure the benchmark
reports.

Shapes: hidden 2,560, 512 routed experts + 1 shared, moe_intermediate 768, vocabulary
157,184 ("Three MoE Inference Optimizations NVIDIA Measured on DGX Spark", section
"Decoding was memory-bound on a 124-billion-parameter model at batch size 1").
"""

from __future__ import annotations

HIDDEN = 2560
INTER = 768
NUM_EXPERTS = 512
VOCAB = 157184


def expert_bytes(hidden: int = HIDDEN, inter: int = INTER) -> int:
    """Packed MXFP4 bytes of one expert: w13 (2I x H/2 + 2I x H/32) + w2 (H x I/2 + H x I/32)."""
    return 2 * inter * (hidden // 2 + hidden // 32) + hidden * (inter // 2 + inter // 32)


def expert_weights(hidden: int = HIDDEN, inter: int = INTER) -> int:
    return 3 * hidden * inter


def router_bytes(num_experts: int = NUM_EXPERTS, hidden: int = HIDDEN) -> int:
    return 2 * num_experts * hidden


def moe_layer_bytes(union: int, m: int, shared: bool = True, num_experts: int = NUM_EXPERTS,
                    hidden: int = HIDDEN, inter: int = INTER, out_bytes_per_elem: int = 2) -> int:
    """Router + (|U| + shared) experts + M bf16 inputs + M outputs."""
    n = union + (1 if shared else 0)
    return (router_bytes(num_experts, hidden) + n * expert_bytes(hidden, inter)
            + m * hidden * (2 + out_bytes_per_elem))


def moe_layer_flops(tokens_per_expert, hidden: int = HIDDEN, inter: int = INTER) -> int:
    """2 * m_e * 3HI per selected expert (gate, up and down GEMVs)."""
    return sum(2 * int(me) * expert_weights(hidden, inter) for me in tokens_per_expert)


def head_weights(vocab: int = VOCAB, hidden: int = HIDDEN) -> int:
    return vocab * hidden


def head_bf16_bytes(m: int = 0, vocab: int = VOCAB, hidden: int = HIDDEN) -> int:
    """BF16 head weight + M bf16 inputs + M fp32 logit rows."""
    return 2 * vocab * hidden + m * (2 * hidden + 4 * vocab)


def head_fp8_bytes(m: int = 0, vocab: int = VOCAB, hidden: int = HIDDEN) -> int:
    """E4M3 head weight + fp32 row scales + M bf16 inputs + M fp32 logit rows."""
    return vocab * hidden + 4 * vocab + m * (2 * hidden + 4 * vocab)


def head_flops(m: int, vocab: int = VOCAB, hidden: int = HIDDEN) -> int:
    return 2 * m * vocab * hidden


def stack_step_bytes(unions, m: int, vocab: int = VOCAB, hidden: int = HIDDEN,
                     inter: int = INTER, num_experts: int = NUM_EXPERTS,
                     logits: bool = True) -> int:
    """One decode step: every layer (its realised expert union) and the FP8 head."""
    layer = sum(moe_layer_bytes(u, m, True, num_experts, hidden, inter) for u in unions)
    head = head_fp8_bytes(m if logits else 0, vocab, hidden)
    if not logits:
        head += m * 2 * hidden
    return layer + head
