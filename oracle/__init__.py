"""Plain float64 CPU oracle for the batch-1 / verify-window MoE decode step.

This package is TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it. The product
path (``moe_decode_weight_gb300`` and its CUDA library) never imports, links or calls it,
and this package imports nothing from the product path: the two share no code. The only
module both sides see is the seeded input generator ``moe_decode_weight_gb300.synth``,
which holds no arithmetic of the method (random bytes and normals only); the oracle
functions here take plain numpy arrays as inputs.

What it computes, and where each step comes from (page title, then section):

* "Three MoE Inference Optimizations NVIDIA Measured on DGX Spark" (blog.neticslabs.com),
  section "Decoding was memory-bound on a 124-billion-parameter model at batch size 1":
  each MoE layer routes a token to eight of 512 routed experts alongside one shared
  expert; hidden 2,560; LM head 2,560 x 157,184.
* same page, "Humming MXFP4 kernels compile at run time for the model's real shapes":
  the MoE runs the W4A8 MXFP4 recipe (E2M1 weights with E8M0 block scales, 8-bit
  activations), moe_intermediate_size 768.
* same page, "Online FP8 quantization halves the LM head weight reads": the BF16 LM head
  is quantised to FP8 once, when it is constructed ("dynamic" quantisation).
* same page, "Multi-token prediction turns each verification into four tokens": a
  four-token verification window touches up to 32 experts instead of 8.
* same page, "GSM8K measured a 42.5% throughput gain across 1,319 questions": top_k 29.
* runbyai.xyz/posts/593, paragraphs 2-3 and 5: the same model facts and the
  ~402M-weight, ~805 MB (BF16) / ~400 MB (FP8) head.

Where the pages leave a step open (scoring function, block size, scale rules, nibble
order, the quantisation of the SwiGLU output, the stack's normalisation) the reading
taken is stated in the docstring of the function that takes it; every such reading is
also listed in the repository's design notes.

Pins. Every function is pinned by ``tests/test_oracle_*.py`` (``-m "not gpu"``) against
something other than itself: exhaustive format tables checked against library casts
(torch / ml_dtypes), closed forms (one-hot and identity experts, a top-1 MoE reducing
to a dense float64 MLP), brute-force top-k, invariants (sum of gates, max code 448),
and the byte counts the pages print. No function here is "parity unpinned".
"""

from . import formats, moe, lm_head, stack  # noqa: F401
