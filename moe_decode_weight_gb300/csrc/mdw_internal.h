// Internal declarations shared by the library's translation units: kernel parameter
// blocks, the workspace layout and the launch functions. Not part of the C-ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

#include "moe_decode_weight.h"

namespace mdw {

constexpr int kThreads = 384;          // 12 warps per block, one block per SM
constexpr int kWarps = kThreads / 32;
constexpr int kMaxPairsCap = MDW_MAX_M * (MDW_MAX_TOPK + 1);
constexpr int kMaxLayers = 128;        // layer descriptors travel in the kernel parameters

// Device copy of one layer's weight pointers.
struct LayerDesc {
  const __nv_bfloat16* router_w;
  const uint8_t* w13_q;
  const uint8_t* w13_s;
  const uint8_t* w2_q;
  const uint8_t* w2_s;
  const uint8_t* sh_w13_q;
  const uint8_t* sh_w13_s;
  const uint8_t* sh_w2_q;
  const uint8_t* sh_w2_s;
};

// Everything the persistent MoE kernel reads; built by the host for one call.
struct MoeParams {
  LayerDesc layers[kMaxLayers];
  int L, M, E, K;              // layers, tokens, routed experts, experts per token
  int has_shared;
  int stack_mode;              // 1: pre-norm residual stack over L layers
  long long spin_budget;       // clock64 cycles an inter-block wait may spin (mdw_spin_budget())
  // layer mode (L == 1)
  const __nv_bfloat16* x_in;   // [M][H]
  void* y_out;                 // [M][H] fp32 or bf16
  int y_fp32;
  const __nv_bfloat16* residual;
  const int32_t* topk_override;
  int32_t* ids_out;
  float* gates_out;
  // stack mode: r_0 (input) and the residual buffers r_1..r_L: resid + ((l) or (l & 1)) * M*H
  const __nv_bfloat16* r0;
  __nv_bfloat16* resid;        // [L+1][M][H] (index l) or [2][M][H] (ping-pong, index l & 1)
  int resid_pingpong;
  // workspace
  uint32_t* hdr;
  uint8_t* xq;                 // [M][H]
  float* sx;                   // [M]
  float* logits;               // [M][E]
  int32_t* ids;                // [M][K]
  float* gates;                // [M][K]
  int32_t* slot_expert;        // [S]
  int32_t* pair_token;         // [P]
  int32_t* pair_slot;          // [P]
  float* pair_gate;            // [P]
  float* h;                    // [P][I]
  uint8_t* hq;                 // [P][I]
  float* sh;                   // [P]
  // tagged words (value in the low half, producing layer + 1 in the high half; zeroed before
  // every launch): the router logits [M][E] and (stack) the residual r_l [M][H/2], two bf16
  // per word
  uint64_t* xz;
  uint64_t* xr;
};

// The LM head's cross-block merge: blocks form groups of kHeadGroupSize; each group's last
// block merges the group's lists, the last group merges the group lists.
constexpr int kHeadGroupSize = 16;
constexpr int kHeadMaxGroups = 16;
constexpr int kMaxHeadGrid = kHeadGroupSize * kHeadMaxGroups;   // blocks of the head kernel (<= 256)
// Windows up to this many tokens keep per-warp top-k lists while the head streams; wider
// windows write their logits and select from them (still one pass over the head). Measured
// on the full 157,184-row FP8 head: lists 93 / 110 / 140 / 200 / 358 us at 1 / 2 / 4 / 8 /
// 16 tokens against 117 / 121 / 124 / 130 / 170 us for logits + selection.
#ifndef MDW_HEAD_LIST_M
#define MDW_HEAD_LIST_M 2
#endif
constexpr int kHeadListM = MDW_HEAD_LIST_M;

struct HeadParams {
  const uint8_t* w;            // [V][H] E4M3 or bf16 (as bytes)
  const float* row_scale;      // [V] or null (bf16)
  long long V;
  int M;
  int topk;                    // candidates kept per token (>= 1)
  const __nv_bfloat16* x;      // [M][H] hidden states, or the residual r_L when norm_input
  int norm_input;              // 1: x = bf16(RMSNorm(x)) first
  float* logits;               // [M][V] or null
  int32_t* argmax_out;         // [M]
  int32_t* topk_idx;           // [M][topk] or null
  float* topk_val;             // [M][topk] or null
  uint32_t* hdr;               // header (status, done counter)
  const double* sample_u;      // [M] uniforms in [0, 1), or null: no draw
  double temperature, top_p;   // draw settings (used when sample_u is set)
  int32_t* sample_out;         // [M] drawn token ids
  float* cand_val;             // [grid + kHeadMaxGroups][M][topk]: block lists, then group lists
  int32_t* cand_idx;           // [grid + kHeadMaxGroups][M][topk]
};

// Workspace layout helpers (host).
struct MoeWs {
  mdw_moe_ws_layout lay;
  size_t xz, xr;               // tagged logit / residual words (xr: stack only)
  size_t zero_end;             // [header, zero_end) is zeroed before every launch
  size_t resid;                // bf16 [2][M][H] ping-pong residual (stack mode)
  size_t cand;                 // head candidates (stack mode)
  size_t total;
};
MoeWs moe_ws_layout(int M, int E, int K, bool stack, int topk, long long V = 0);
size_t head_ws_bytes(int M, int topk, long long V);

// Spin budget of the kernels' bounded inter-block waits (the default, or the value set by
// mdw_debug_set_spin_budget).
long long mdw_spin_budget();

int device_sm_count();
int moe_grid();                // co-resident blocks of the MoE kernel (<= SM count)
int head_grid();

// Workspace pointers of one MoE launch (exchange words included).
void fill_moe_ws(MoeParams& p, const MoeWs& w, uint8_t* base);

// Launchers (return cudaSuccess or the first error).
cudaError_t launch_moe(const MoeParams& p, cudaStream_t s);
cudaError_t launch_head_fp8(const HeadParams& p, cudaStream_t s);
cudaError_t launch_head_bf16(const HeadParams& p, cudaStream_t s);
cudaError_t launch_quantize_head(const __nv_bfloat16* w, long long V, uint8_t* q, float* scale,
                                 cudaStream_t s);
size_t moe_smem_bytes(int M);

}  // namespace mdw
