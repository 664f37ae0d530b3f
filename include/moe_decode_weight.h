/*
 * moe_decode_weight.h -- C-ABI of the GB300 (sm_103a) decode step of a W4A8 MXFP4
 * mixture-of-experts model: router, routed + shared experts, combine, and the online-FP8
 * LM head with a fused argmax / top-k.
 *
 * The method comes from NVIDIA's batch-size-1 study of Ling-3.0-flash on DGX Spark, as
 * reported on "Three MoE Inference Optimizations NVIDIA Measured on DGX Spark"
 * (blog.neticslabs.com) and runbyai.xyz/posts/593:
 *   - section "Decoding was memory-bound on a 124-billion-parameter model at batch
 *     size 1": each MoE layer routes a token to 8 of 512 experts plus 1 shared expert;
 *     hidden 2,560; the LM head projects 2,560 onto 157,184 tokens;
 *   - section "Humming MXFP4 kernels compile at run time for the model's real shapes":
 *     W4A8 MXFP4 experts, moe_intermediate_size 768;
 *   - section "Online FP8 quantization halves the LM head weight reads": the BF16 head
 *     is quantised to FP8 once, when it is constructed;
 *   - section "Multi-token prediction turns each verification into four tokens": a
 *     4-token window touches up to 32 experts; each is read once per window here;
 *   - section "One missing interface makes the stack slower than baseline" (and
 *     runbyai.xyz/posts/593 paragraph 9): an FP8 head read as BF16 fails silently, so every
 *     weight handle here carries a format tag that every call checks.
 *
 * Conventions (all entry points):
 *   - Device pointers: every tensor argument is a device pointer to memory the CALLER
 *     owns; the library never allocates, frees or keeps a pointer after a call returns.
 *     All device pointers must be 16-byte aligned.
 *   - Execution: work is enqueued on `stream` and runs asynchronously; no entry point
 *     synchronises except mdw_device_status().
 *   - Validation: arguments are checked on the host BEFORE anything is enqueued; on any
 *     error the call returns a non-zero mdw_status and enqueues nothing.
 *   - Device-side failures (an out-of-range imposed expert id, a bounded wait that ran
 *     out) never trap: kernels record an mdw_status in the workspace header and return;
 *     mdw_device_status() reads it.
 *   - Workspaces are caller-allocated device buffers of at least the size the matching
 *     *_workspace_bytes() query returns. Each call re-initialises the header it uses.
 *   - Thread safety: calls on different workspaces may run concurrently; calls that share
 *     a workspace must be ordered on one stream.
 *
 * Layouts (row-major, little-endian):
 *   - MXFP4 expert (format MDW_FMT_MXFP4_E2M1_E8M0_B32), per expert e:
 *       w13_q [2I][H/2] uint8  rows 0..I-1 = gate, I..2I-1 = up; byte k/2 holds K index
 *                              k in its low nibble (k even) or high nibble (k odd);
 *                              each nibble an E2M1 code (sign bit 3, exponent bits 2-1
 *                              bias 1, mantissa bit 0)
 *       w13_s [2I][H/32] uint8 E8M0 scale (2^(s-127)) of K block [32b, 32b+32)
 *       w2_q  [H][I/2]   uint8 down projection, same packing; w2_s [H][I/32] uint8
 *     The routed experts are stacked along a leading [E] axis.
 *   - Router weight [E][H] bf16. Hidden states [M][H] bf16.
 *   - FP8 head (MDW_FMT_FP8_E4M3_ROWSCALE): q [V][H] E4M3 bytes, row_scale [V] fp32.
 *   - BF16 head (MDW_FMT_BF16): w [V][H] bf16.
 */
#ifndef MOE_DECODE_WEIGHT_H
#define MOE_DECODE_WEIGHT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as the CUDA runtime's cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* mdw_stream_t;

typedef enum mdw_status {
  MDW_OK = 0,
  MDW_ERR_INVALID_ARG = 1,         /* null / misaligned pointer, M or top_k out of range */
  MDW_ERR_UNSUPPORTED_SHAPE = 2,   /* hidden / inter / experts / vocab not supported */
  MDW_ERR_FORMAT_MISMATCH = 3,     /* magic or format tag of a weight handle is wrong */
  MDW_ERR_WORKSPACE_TOO_SMALL = 4,
  MDW_ERR_CUDA = 5,                /* a CUDA runtime call failed (launch, memset, query) */
  MDW_ERR_TIMEOUT = 6,             /* device: a bounded inter-block wait ran out */
  MDW_ERR_DEVICE_BOUNDS = 7        /* device: an imposed expert id was out of range or repeated */
} mdw_status;

typedef enum mdw_format {
  MDW_FMT_BF16 = 1,
  MDW_FMT_FP8_E4M3_ROWSCALE = 2,
  MDW_FMT_MXFP4_E2M1_E8M0_B32 = 3
} mdw_format;

#define MDW_MAGIC 0x3157444Du /* "MDW1" */

/* Shapes this build is specialised for (runtime-compiled kernels in the pages' design are
 * specialised the same way: "Humming MXFP4 kernels compile at run time for the model's
 * real shapes"). Other hidden/inter values return MDW_ERR_UNSUPPORTED_SHAPE. */
#define MDW_HIDDEN 2560
#define MDW_INTER 768
#define MDW_MAX_EXPERTS 512
#define MDW_MAX_TOPK 8
#define MDW_MAX_M 32
#define MDW_MAX_VOCAB_TOPK 32

/* Weights of one MoE layer. Fill every field; set magic = MDW_MAGIC and
 * fmt = MDW_FMT_MXFP4_E2M1_E8M0_B32. The shared-expert pointers are all NULL (no shared
 * expert) or all non-NULL (one shared expert, same layout as a routed one, no [E] axis). */
typedef struct mdw_moe_weights {
  uint32_t magic;
  int32_t fmt;
  int32_t num_experts;  /* routed experts E, 1..512 */
  int32_t top_k;        /* experts per token, 1..MDW_MAX_TOPK and <= E */
  int32_t hidden;       /* H, must be MDW_HIDDEN */
  int32_t inter;        /* I, must be MDW_INTER */
  const void* router_w; /* bf16 [E][H] */
  const void* w13_q;    /* uint8 [E][2I][H/2] */
  const void* w13_s;    /* uint8 [E][2I][H/32] */
  const void* w2_q;     /* uint8 [E][H][I/2] */
  const void* w2_s;     /* uint8 [E][H][I/32] */
  const void* sh_w13_q; /* shared expert, uint8 [2I][H/2], or NULL */
  const void* sh_w13_s;
  const void* sh_w2_q;
  const void* sh_w2_s;
} mdw_moe_weights;

/* An LM head. fmt MDW_FMT_FP8_E4M3_ROWSCALE: w = E4M3 [V][H], row_scale = fp32 [V].
 * fmt MDW_FMT_BF16: w = bf16 [V][H], row_scale = NULL. */
typedef struct mdw_lm_head {
  uint32_t magic;
  int32_t fmt;
  int64_t vocab;
  int32_t hidden;
  int32_t reserved;
  const void* w;
  const float* row_scale;
} mdw_lm_head;

/* Offsets (bytes from the workspace base) of the intermediates one moe_decode_layer call
 * leaves in its workspace, for inspection. P = number of (token, expert) pairs of the
 * call, S = number of expert slots (slot 0 = the shared expert when there is one, then
 * the union of the routed selections in ascending expert id); pairs are ordered by slot,
 * then by token. In moe_decode_stack the buffers hold the last layer's values. */
typedef struct mdw_moe_ws_layout {
  size_t header;     /* uint32 [256]: [0] device status, [2] S, [3] P, [4] routed slots;
                        [64 + l] routed union size of layer l (moe_decode_stack) */
  size_t xq;         /* uint8 [M][H] E4M3 codes of the quantised expert input */
  size_t sx;         /* fp32 [M] its per-token scales */
  size_t logits;     /* fp32 [M][E] router logits */
  size_t ids;        /* int32 [M][top_k] selected experts, descending logit */
  size_t gates;      /* fp32 [M][top_k] renormalised gate weights */
  size_t slot_expert;/* int32 [S] expert id per slot (-1 = shared expert) */
  size_t pair_token; /* int32 [P] token of each pair */
  size_t pair_slot;  /* int32 [P] slot of each pair */
  size_t pair_gate;  /* fp32 [P] combine weight of each pair (1 for the shared expert) */
  size_t h;          /* fp32 [P][I] SwiGLU output per pair */
  size_t hq;         /* uint8 [P][I] E4M3 codes of h */
  size_t sh;         /* fp32 [P] per-pair scale of hq */
  size_t total;      /* workspace bytes needed */
} mdw_moe_ws_layout;

/* ---------------------------------------------------------------------------------- */

/* Human-readable name of a status code. Never NULL. */
const char* mdw_status_string(mdw_status s);

/* Library version (major*10000 + minor*100 + patch). */
int32_t mdw_version(void);

/* Test hook, not part of the decode path (the pages have no counterpart). Every inter-block
 * wait of the MoE kernels is bounded: after `cycles` clock64 cycles (default 1e9, ~0.5 s)
 * it records MDW_ERR_TIMEOUT in the workspace status word, and every block then leaves the
 * kernel at its next wait, so a launch always completes. This sets the bound for the calls
 * enqueued after it, process-wide (cycles <= 0 restores the default) and returns the
 * previous value. A test makes the bound tiny to check that a wait that runs out ends in
 * MDW_ERR_TIMEOUT with a usable device context, without faulting or hanging the GPU. */
int64_t mdw_debug_set_spin_budget(int64_t cycles);

/* Workspace bytes for moe_decode_layer with M tokens; 0 if the arguments are invalid. */
size_t mdw_moe_workspace_bytes(const mdw_moe_weights* w, int32_t M);

/* Fills *out with the workspace layout of moe_decode_layer for M tokens. */
mdw_status mdw_moe_workspace_layout(const mdw_moe_weights* w, int32_t M, mdw_moe_ws_layout* out);

/* One MoE decode layer for a window of M tokens (1 <= M <= MDW_MAX_M).
 *
 * Computes, per token t (the pages' sections cited in the file header):
 *   a1  xq_t, sx_t = E4M3 per-token quantisation of x_t (scale = amax/448, fp32 steps);
 *   a2  z_t = x_t . Wr^T on the bf16 x_t, fp32 accumulation;
 *   a3  ids_t = top_k of z_t (descending, ties -> lower id); gates = softmax of the
 *       selected logits (= the renormalised full softmax); or, if topk_override is not
 *       NULL, ids_t = topk_override[t] with the same gate rule;
 *   a4  the union of all tokens' ids (each selected expert's weights are read once per
 *       call), plus the shared expert for every token;
 *   a5  per (token, expert): gate_j, up_j = MXFP4 GEMVs of w13 with xq_t (x sx_t);
 *       h = silu(gate) * up;
 *   a6  hq, s_h = E4M3 quantisation of h (scale = amax/448, fp32 steps);
 *   a7  y_t = sum_i gates_t[i] * s_h * (W2_e . hq) + shared expert output (+ residual_t).
 *
 * x_bf16   : device bf16 [M][H], the expert input.
 * y        : device [M][H]; fp32 if y_is_fp32 != 0, else bf16 (round to nearest even of
 *            the fp32 result).
 * residual : NULL or device bf16 [M][H], added to y in fp32 before the output rounding.
 * topk_override : NULL or device int32 [M][top_k] expert ids to use instead of the
 *            router's selection (ids must be distinct per token and < E; violations set
 *            MDW_ERR_DEVICE_BOUNDS in the device status and produce no output).
 * topk_ids_out, topk_w_out : NULL or device int32 / fp32 [M][top_k] (selection, gates).
 * ws, ws_bytes : workspace (>= mdw_moe_workspace_bytes(w, M)), 16-byte aligned.
 */
mdw_status moe_decode_layer(const mdw_moe_weights* w, int32_t M, const void* x_bf16, void* y,
                            int32_t y_is_fp32, const void* residual,
                            const int32_t* topk_override, int32_t* topk_ids_out,
                            float* topk_w_out, void* ws, size_t ws_bytes, mdw_stream_t stream);

/* Bytes of the scratch array that the library holds on every GPU it runs on, for
 * moe_decode_layer_noalloc (2 MiB). */
#define MDW_NOALLOC_SCRATCH_BYTES (2u << 20)

/* moe_decode_layer without a caller workspace. The pages have no counterpart: this is an
 * integration entry point of this library.
 *
 * For callers that cannot allocate device memory: code running inside a host framework
 * that owns the whole device-memory budget and forbids further allocations, plain C callers
 * without an allocator, and latency-critical loops where cudaMalloc / cudaFree would
 * implicitly synchronise the device. The caller passes inputs and outputs exactly as for
 * moe_decode_layer (same meaning, layout and validation); the scratch is a fixed array of
 * MDW_NOALLOC_SCRATCH_BYTES compiled into the library, which every GPU that loads the
 * library holds until the process exits. Calls that moe_decode_layer accepts all fit; a
 * shape whose workspace would exceed the array returns MDW_ERR_WORKSPACE_TOO_SMALL.
 *
 * Nothing is allocated: no cudaMalloc / cudaFree, no allocating library routine, no host
 * heap. The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before any stream
 * capture. The address is kept for the life of the process: a cudaDeviceReset() after
 * the first call on that device is not supported. Every call on a device shares the one array and re-zeroes the part that must
 * start at zero; the array keeps the last call's intermediates otherwise. Calls whose work
 * overlaps on the GPU (different streams without ordering) race on the array.
 *
 * device_status_out: NULL or a device uint32 that receives the call's device status word
 * (MDW_OK, MDW_ERR_TIMEOUT or MDW_ERR_DEVICE_BOUNDS) in stream order. */
mdw_status moe_decode_layer_noalloc(const mdw_moe_weights* w, int32_t M, const void* x_bf16, void* y,
                                    int32_t y_is_fp32, const void* residual,
                                    const int32_t* topk_override, int32_t* topk_ids_out,
                                    float* topk_w_out, uint32_t* device_status_out,
                                    mdw_stream_t stream);

/* Online FP8 quantisation of a BF16 LM head ("Online FP8 quantization halves the LM head
 * weight reads": done once, when the head is constructed). Per vocabulary row v:
 * scale_v = amax_v / 448 in fp32 (1 for an all-zero row); q[v][h] = E4M3(w[v][h] / scale_v),
 * round to nearest even, saturating. w_bf16 [V][H] bf16 in, q_out [V][H] uint8 and
 * scale_out [V] fp32 out (device). On success *head_out (host struct) describes the FP8
 * head (magic, fmt = MDW_FMT_FP8_E4M3_ROWSCALE, pointers to q_out / scale_out). */
mdw_status quantize_lm_head_fp8(const void* w_bf16, int64_t V, int32_t H, void* q_out,
                                float* scale_out, mdw_lm_head* head_out, mdw_stream_t stream);

/* Fills *head_out with a descriptor of an (unquantised) BF16 head w_bf16 [V][H]. */
mdw_status mdw_lm_head_bf16_init(const void* w_bf16, int64_t V, int32_t H, mdw_lm_head* head_out);

/* Workspace bytes for lm_head_fp8 / lm_head_bf16 with M tokens and the given topk. */
size_t mdw_lm_head_workspace_bytes(const mdw_lm_head* head, int32_t M, int32_t topk);

/* FP8 LM-head GEMV with fused argmax / top-k (the pages' "output-layer projection").
 * logits[t][v] = row_scale[v] * sum_h E4M3(q[v][h]) * x[t][h], x = h_bf16 (bf16, W8A16),
 * fp32 accumulation. Outputs (device): logits (NULL = not written) fp32 [M][V];
 * argmax_out int32 [M] (required); topk_idx int32 [M][topk] and topk_val fp32 [M][topk]
 * (NULL = not written; topk in 1..MDW_MAX_VOCAB_TOPK), descending, ties -> lower index.
 * head->fmt must be MDW_FMT_FP8_E4M3_ROWSCALE, else MDW_ERR_FORMAT_MISMATCH.
 * One launch streams the head once for the whole window (1 <= M <= MDW_MAX_M); above 2
 * tokens it selects from fp32 logits written to `logits`, or to the workspace when NULL
 * (mdw_lm_head_workspace_bytes then includes M * V * 4 bytes for them). */
mdw_status lm_head_fp8(const mdw_lm_head* head, int32_t M, const void* h_bf16, float* logits,
                       int32_t* argmax_out, int32_t topk, int32_t* topk_idx, float* topk_val,
                       void* ws, size_t ws_bytes, mdw_stream_t stream);

/* The same projection on the unquantised BF16 head (head->fmt must be MDW_FMT_BF16);
 * kept for the 2x byte comparison of the pages (~805 MB vs ~400 MB per token). */
mdw_status lm_head_bf16(const mdw_lm_head* head, int32_t M, const void* h_bf16, float* logits,
                        int32_t* argmax_out, int32_t topk, int32_t* topk_idx, float* topk_val,
                        void* ws, size_t ws_bytes, mdw_stream_t stream);

/* Workspace bytes for moe_decode_stack (L layers, M tokens, vocabulary top-k). */
size_t mdw_stack_workspace_bytes(const mdw_moe_weights* layers, int32_t L, const mdw_lm_head* head,
                                 int32_t M, int32_t topk);

/* The whole decode-step weight stream: L MoE layers on a bf16 residual stream, then the
 * FP8 head. The pages omit nothing but attention here; the stack keeps the decoder's
 * pre-norm (a reading: RMSNorm with unit gain, eps 1e-6):
 *   x_l = bf16(RMSNorm(r_l));  r_{l+1} = bf16(r_l + MoE_l(x_l));
 *   logits = head(bf16(RMSNorm(r_L))), then argmax / top-k.
 * layers : HOST array of L (1..128) layer descriptors (read during the call only).
 * head   : the FP8 head (fmt MDW_FMT_FP8_E4M3_ROWSCALE), or NULL to run the L layers only
 *          (then resid_out is required, r_L is resid_out[L], and the head outputs are
 *          ignored; lm_head_fp8_rmsnorm finishes the step).
 * r0_bf16: device bf16 [M][H] initial residual.
 * resid_out : NULL or device bf16 [L+1][M][H]: every r_l, for inspection.
 * Other outputs as lm_head_fp8. The workspace header's word 64 + l holds the number of
 * distinct routed experts of layer l (the window's union). */
mdw_status moe_decode_stack(const mdw_moe_weights* layers, int32_t L, const mdw_lm_head* head,
                            int32_t M, const void* r0_bf16, void* resid_out, float* logits,
                            int32_t* argmax_out, int32_t topk, int32_t* topk_idx, float* topk_val,
                            void* ws, size_t ws_bytes, mdw_stream_t stream);

/* moe_decode_stack with imposed routing: topk_override = NULL (the router decides) or device
 * int32 [L][M][top_k], every row K distinct expert ids in [0, num_experts) (4-byte aligned);
 * the router GEMV still runs and the gates are the renormalised softmax of its logits at the
 * imposed ids. A row with an out-of-range or repeated id stops the launch at that layer
 * with MDW_ERR_DEVICE_BOUNDS in the status word. */
mdw_status moe_decode_stack_routed(const mdw_moe_weights* layers, int32_t L, const mdw_lm_head* head,
                                   int32_t M, const void* r0_bf16, void* resid_out, float* logits,
                                   int32_t* argmax_out, int32_t topk, int32_t* topk_idx, float* topk_val,
                                   const int32_t* topk_override, void* ws, size_t ws_bytes,
                                   mdw_stream_t stream);

/* The last step of moe_decode_stack on its own: lm_head_fp8 applied to bf16(RMSNorm(r)),
 * RMSNorm with unit gain and eps 1e-6 in fp32, r_bf16 = device bf16 [M][H] (the residual
 * stream after the last layer). Arguments otherwise as lm_head_fp8. */
mdw_status lm_head_fp8_rmsnorm(const mdw_lm_head* head, int32_t M, const void* r_bf16, float* logits,
                               int32_t* argmax_out, int32_t topk, int32_t* topk_idx, float* topk_val,
                               void* ws, size_t ws_bytes, mdw_stream_t stream);

/* Decode-time draw on top-k candidates ("Three MoE Inference Optimizations NVIDIA
 * Measured on DGX Spark", section "GSM8K measured a 42.5% throughput gain across 1,319 questions":
 * temperature 0.6, top_p 0.95, top_k 29). The pages give the settings only; the steps
 * (reading): per token, e_i = exp((z_i - z_0) / temperature) over the k candidates in head
 * order; keep the shortest prefix whose mass reaches top_p * total (the crossing candidate
 * stays); the token is the first kept candidate whose cumulative mass exceeds u * kept mass.
 * temperature <= 0 means greedy (the first candidate). float64 arithmetic, sums left to
 * right, one thread per token.
 * topk_val / topk_idx: device [M][k] (as lm_head_fp8 writes them: descending, ties to the
 *   lower id), k in [1, MDW_MAX_VOCAB_TOPK]; u: device float64 [M] in [0, 1), drawn by the
 *   caller (8-byte aligned); token_out: device int32 [M]. top_p in (0, 1].
 * Errors: MDW_ERR_INVALID_ARG for bad sizes, pointers or settings (nothing launched). */
mdw_status mdw_sample_topk(int32_t M, int32_t k, const float* topk_val, const int32_t* topk_idx,
                           double temperature, double top_p, const double* u, int32_t* token_out,
                           mdw_stream_t stream);

/* lm_head_fp8 (or lm_head_fp8_rmsnorm when norm_input != 0) followed by the draw of
 * mdw_sample_topk on its top-`topk` candidates, fused into the head's final merge block.
 * token_out: device int32 [M] drawn ids (required); topk_idx / topk_val nullable as in
 * lm_head_fp8; u, temperature, top_p as mdw_sample_topk; workspace as lm_head_fp8. */
mdw_status lm_head_fp8_sample(const mdw_lm_head* head, int32_t M, const void* h_bf16, int32_t norm_input,
                              int32_t topk, double temperature, double top_p, const double* u,
                              int32_t* token_out, int32_t* topk_idx, float* topk_val, void* ws,
                              size_t ws_bytes, mdw_stream_t stream);

/* Synchronises `stream`, then returns the device status word that the last call using
 * this workspace left (MDW_OK, MDW_ERR_TIMEOUT or MDW_ERR_DEVICE_BOUNDS), or MDW_ERR_CUDA
 * if the synchronisation itself failed. */
mdw_status mdw_device_status(const void* ws, mdw_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_DECODE_WEIGHT_H */
