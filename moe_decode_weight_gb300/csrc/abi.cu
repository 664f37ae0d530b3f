// C-ABI entry points: argument validation, workspace carving and kernel launches.
//
// The validation rules implement the lesson of "Three MoE Inference Optimizations NVIDIA
// Measured on DGX Spark", section "One missing interface makes the stack slower than
// baseline": quantisation state travels with the weight handle (magic + format tag), and
// a handle of the wrong format is an error at the call, never a silent reinterpretation.
#include <atomic>
#include <cstring>

#include "mdw_device.cuh"
#include "mdw_internal.h"

namespace mdw {

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}
int moe_grid() { return device_sm_count(); }

static std::atomic<long long> g_spin_budget{kSpinBudget};
long long mdw_spin_budget() { return g_spin_budget.load(std::memory_order_relaxed); }
int head_grid() { const int n = device_sm_count(); return n > kMaxHeadGrid ? kMaxHeadGrid : n; }

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Head workspace after the header: block + group candidate lists (values, then indices) and,
// for a window wider than kHeadListM tokens, the fp32 logits [M][V] the head selects from.
size_t head_ws_bytes(int M, int topk, long long V) {
  const size_t n = (size_t)(head_grid() + kHeadMaxGroups) * M * topk;
  return 2 * align_up(n * 4, 256) + (M > kHeadListM ? align_up((size_t)M * V * 4, 256) : 0);
}

MoeWs moe_ws_layout(int M, int E, int K, bool stack, int topk, long long V) {
  MoeWs w;
  mdw_moe_ws_layout& l = w.lay;
  const size_t P = (size_t)M * (K + 1), S = (size_t)M * K + 1;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o = align_up(o + bytes, 256); return r; };
  l.header = take(kHdrWords * 4);
  w.xz = take((size_t)M * E * 8);               // zeroed with the header before every launch
  w.xr = stack ? take((size_t)M * (kH / 2) * 8) : 0;
  w.zero_end = o;
  l.xq = take((size_t)M * kH);
  l.sx = take((size_t)M * 4);
  l.logits = take((size_t)M * E * 4);
  l.ids = take((size_t)M * K * 4);
  l.gates = take((size_t)M * K * 4);
  l.slot_expert = take(S * 4);
  l.pair_token = take(P * 4);
  l.pair_slot = take(P * 4);
  l.pair_gate = take(P * 4);
  l.h = take(P * kI * 4);
  l.hq = take(P * kI);
  l.sh = take(P * 4);
  w.resid = stack ? take((size_t)2 * M * kH * 2) : 0;
  w.cand = stack ? take(head_ws_bytes(M, topk, V)) : 0;
  l.total = o;
  w.total = o;
  return w;
}

}  // namespace mdw

using namespace mdw;

namespace {

bool al16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool al16_or_null(const void* p) { return p == nullptr || al16(p); }

mdw_status check_weights(const mdw_moe_weights* w) {
  if (!w) return MDW_ERR_INVALID_ARG;
  if (w->magic != MDW_MAGIC || w->fmt != MDW_FMT_MXFP4_E2M1_E8M0_B32) return MDW_ERR_FORMAT_MISMATCH;
  if (w->hidden != MDW_HIDDEN || w->inter != MDW_INTER) return MDW_ERR_UNSUPPORTED_SHAPE;
  if (w->num_experts < 1 || w->num_experts > MDW_MAX_EXPERTS) return MDW_ERR_UNSUPPORTED_SHAPE;
  if (w->top_k < 1 || w->top_k > MDW_MAX_TOPK || w->top_k > w->num_experts) return MDW_ERR_INVALID_ARG;
  if (!al16(w->router_w) || !al16(w->w13_q) || !al16(w->w13_s) || !al16(w->w2_q) || !al16(w->w2_s))
    return MDW_ERR_INVALID_ARG;
  const int nsh = (w->sh_w13_q != nullptr) + (w->sh_w13_s != nullptr) + (w->sh_w2_q != nullptr) +
                  (w->sh_w2_s != nullptr);
  if (nsh != 0 && nsh != 4) return MDW_ERR_INVALID_ARG;
  if (nsh == 4 && (!al16(w->sh_w13_q) || !al16(w->sh_w13_s) || !al16(w->sh_w2_q) || !al16(w->sh_w2_s)))
    return MDW_ERR_INVALID_ARG;
  return MDW_OK;
}

mdw_status check_head(const mdw_lm_head* h, int fmt) {
  if (!h) return MDW_ERR_INVALID_ARG;
  if (h->magic != MDW_MAGIC || h->fmt != fmt) return MDW_ERR_FORMAT_MISMATCH;
  if (h->hidden != MDW_HIDDEN) return MDW_ERR_UNSUPPORTED_SHAPE;
  if (h->vocab < 1 || h->vocab > 0x7fffffffLL) return MDW_ERR_UNSUPPORTED_SHAPE;
  if (!al16(h->w)) return MDW_ERR_INVALID_ARG;
  if (fmt == MDW_FMT_FP8_E4M3_ROWSCALE && !al16(h->row_scale)) return MDW_ERR_INVALID_ARG;
  return MDW_OK;
}

mdw_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MDW_OK : MDW_ERR_CUDA; }

void fill_layer(LayerDesc& d, const mdw_moe_weights* w) {
  d.router_w = static_cast<const __nv_bfloat16*>(w->router_w);
  d.w13_q = static_cast<const uint8_t*>(w->w13_q);
  d.w13_s = static_cast<const uint8_t*>(w->w13_s);
  d.w2_q = static_cast<const uint8_t*>(w->w2_q);
  d.w2_s = static_cast<const uint8_t*>(w->w2_s);
  d.sh_w13_q = static_cast<const uint8_t*>(w->sh_w13_q);
  d.sh_w13_s = static_cast<const uint8_t*>(w->sh_w13_s);
  d.sh_w2_q = static_cast<const uint8_t*>(w->sh_w2_q);
  d.sh_w2_s = static_cast<const uint8_t*>(w->sh_w2_s);
}

}  // namespace

namespace mdw {
void fill_moe_ws(MoeParams& p, const MoeWs& w, uint8_t* base) {
  const mdw_moe_ws_layout& l = w.lay;
  p.hdr = reinterpret_cast<uint32_t*>(base + l.header);
  p.xq = base + l.xq;
  p.sx = reinterpret_cast<float*>(base + l.sx);
  p.logits = reinterpret_cast<float*>(base + l.logits);
  p.ids = reinterpret_cast<int32_t*>(base + l.ids);
  p.gates = reinterpret_cast<float*>(base + l.gates);
  p.slot_expert = reinterpret_cast<int32_t*>(base + l.slot_expert);
  p.pair_token = reinterpret_cast<int32_t*>(base + l.pair_token);
  p.pair_slot = reinterpret_cast<int32_t*>(base + l.pair_slot);
  p.pair_gate = reinterpret_cast<float*>(base + l.pair_gate);
  p.h = reinterpret_cast<float*>(base + l.h);
  p.hq = base + l.hq;
  p.sh = reinterpret_cast<float*>(base + l.sh);
  p.xz = reinterpret_cast<uint64_t*>(base + w.xz);
  p.xr = w.xr ? reinterpret_cast<uint64_t*>(base + w.xr) : nullptr;
}
}  // namespace mdw

namespace {

struct Draw {                     // optional draw on the final top-k
  const double* u = nullptr;
  double temperature = 0.0, top_p = 1.0;
  int32_t* out = nullptr;
};

// One head launch for the whole window (it streams the head once): `cand` is the region
// head_ws_bytes(M, topk, V) describes; a window wider than kHeadListM tokens selects from its
// fp32 logits, written to `logits` when given, else to the workspace.
mdw_status head_call(const mdw_lm_head* head, int fmt, int32_t M, const void* h_bf16, int norm_input,
                     float* logits, int32_t* argmax_out, int32_t topk, int32_t* topk_idx,
                     float* topk_val, uint32_t* hdr, uint8_t* cand, cudaStream_t s, const Draw& draw = Draw()) {
  const size_t n = (size_t)(head_grid() + kHeadMaxGroups) * M * topk;
  HeadParams hp{};
  hp.sample_u = draw.u;
  hp.temperature = draw.temperature;
  hp.top_p = draw.top_p;
  hp.sample_out = draw.out;
  hp.w = static_cast<const uint8_t*>(head->w);
  hp.row_scale = head->row_scale;
  hp.V = head->vocab;
  hp.M = M;
  hp.topk = topk;
  hp.x = static_cast<const __nv_bfloat16*>(h_bf16);
  hp.norm_input = norm_input;
  hp.logits = logits;
  if (M > kHeadListM && !logits) hp.logits = reinterpret_cast<float*>(cand + 2 * align_up(n * 4, 256));
  hp.argmax_out = argmax_out;
  hp.topk_idx = topk_idx;
  hp.topk_val = topk_val;
  hp.hdr = hdr;
  hp.cand_val = reinterpret_cast<float*>(cand);
  hp.cand_idx = reinterpret_cast<int32_t*>(cand + align_up(n * 4, 256));
  return cuda_status(fmt == MDW_FMT_FP8_E4M3_ROWSCALE ? launch_head_fp8(hp, s) : launch_head_bf16(hp, s));
}

mdw_status head_entry(int fmt, const mdw_lm_head* head, int32_t M, const void* h_bf16, float* logits,
                      int32_t* argmax_out, int32_t topk, int32_t* topk_idx, float* topk_val, void* ws,
                      size_t ws_bytes, cudaStream_t s, int norm_input = 0, const Draw& draw = Draw()) {
  mdw_status st = check_head(head, fmt);
  if (st != MDW_OK) return st;
  if (M < 1 || M > MDW_MAX_M || topk < 1 || topk > MDW_MAX_VOCAB_TOPK || head->vocab < topk)
    return MDW_ERR_INVALID_ARG;
  if (!al16(h_bf16) || !al16_or_null(logits) || !(argmax_out || draw.out) || !al16(ws)) return MDW_ERR_INVALID_ARG;
  if (ws_bytes < mdw_lm_head_workspace_bytes(head, M, topk)) return MDW_ERR_WORKSPACE_TOO_SMALL;
  if (head_grid() <= 0) return MDW_ERR_CUDA;
  uint8_t* base = static_cast<uint8_t*>(ws);
  if (cudaMemsetAsync(base, 0, kHdrWords * 4, s) != cudaSuccess) return MDW_ERR_CUDA;
  return head_call(head, fmt, M, h_bf16, norm_input, logits, argmax_out, topk, topk_idx, topk_val,
                   reinterpret_cast<uint32_t*>(base), base + kHdrWords * 4, s, draw);
}

}  // namespace

extern "C" {

const char* mdw_status_string(mdw_status s) {
  switch (s) {
    case MDW_OK: return "MDW_OK";
    case MDW_ERR_INVALID_ARG: return "MDW_ERR_INVALID_ARG";
    case MDW_ERR_UNSUPPORTED_SHAPE: return "MDW_ERR_UNSUPPORTED_SHAPE";
    case MDW_ERR_FORMAT_MISMATCH: return "MDW_ERR_FORMAT_MISMATCH";
    case MDW_ERR_WORKSPACE_TOO_SMALL: return "MDW_ERR_WORKSPACE_TOO_SMALL";
    case MDW_ERR_CUDA: return "MDW_ERR_CUDA";
    case MDW_ERR_TIMEOUT: return "MDW_ERR_TIMEOUT";
    case MDW_ERR_DEVICE_BOUNDS: return "MDW_ERR_DEVICE_BOUNDS";
  }
  return "MDW_ERR_UNKNOWN";
}

int32_t mdw_version(void) { return 200; }

int64_t mdw_debug_set_spin_budget(int64_t cycles) {
  const long long v = cycles > 0 ? (long long)cycles : kSpinBudget;
  return (int64_t)g_spin_budget.exchange(v);
}

size_t mdw_moe_workspace_bytes(const mdw_moe_weights* w, int32_t M) {
  if (check_weights(w) != MDW_OK || M < 1 || M > MDW_MAX_M) return 0;
  return moe_ws_layout(M, w->num_experts, w->top_k, false, 1).total;
}

mdw_status mdw_moe_workspace_layout(const mdw_moe_weights* w, int32_t M, mdw_moe_ws_layout* out) {
  mdw_status st = check_weights(w);
  if (st != MDW_OK) return st;
  if (M < 1 || M > MDW_MAX_M || !out) return MDW_ERR_INVALID_ARG;
  *out = moe_ws_layout(M, w->num_experts, w->top_k, false, 1).lay;
  return MDW_OK;
}

mdw_status moe_decode_layer(const mdw_moe_weights* w, int32_t M, const void* x_bf16, void* y,
                            int32_t y_is_fp32, const void* residual, const int32_t* topk_override,
                            int32_t* topk_ids_out, float* topk_w_out, void* ws, size_t ws_bytes,
                            mdw_stream_t stream) {
  mdw_status st = check_weights(w);
  if (st != MDW_OK) return st;
  if (M < 1 || M > MDW_MAX_M) return MDW_ERR_INVALID_ARG;
  if (!al16(x_bf16) || !al16(y) || !al16_or_null(residual) || !al16_or_null(topk_override) ||
      !al16_or_null(topk_ids_out) || !al16_or_null(topk_w_out) || !al16(ws))
    return MDW_ERR_INVALID_ARG;
  const MoeWs lay = moe_ws_layout(M, w->num_experts, w->top_k, false, 1);
  if (ws_bytes < lay.total) return MDW_ERR_WORKSPACE_TOO_SMALL;
  if (moe_grid() * 16 < kH / 2) return MDW_ERR_UNSUPPORTED_SHAPE;   // rows per block bound
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  MoeParams* p = new MoeParams();
  fill_layer(p->layers[0], w);
  p->L = 1; p->M = M; p->E = w->num_experts; p->K = w->top_k;
  p->has_shared = w->sh_w13_q != nullptr;
  p->stack_mode = 0;
  p->spin_budget = mdw_spin_budget();
  p->x_in = static_cast<const __nv_bfloat16*>(x_bf16);
  p->y_out = y;
  p->y_fp32 = y_is_fp32 != 0;
  p->residual = static_cast<const __nv_bfloat16*>(residual);
  p->topk_override = topk_override;
  p->ids_out = topk_ids_out;
  p->gates_out = topk_w_out;
  uint8_t* base = static_cast<uint8_t*>(ws);
  fill_moe_ws(*p, lay, base);
  st = MDW_OK;
  if (cudaMemsetAsync(base + lay.lay.header, 0, lay.zero_end - lay.lay.header, s) != cudaSuccess) st = MDW_ERR_CUDA;
  if (st == MDW_OK) st = cuda_status(launch_moe(*p, s));
  delete p;
  return st;
}

mdw_status quantize_lm_head_fp8(const void* w_bf16, int64_t V, int32_t H, void* q_out, float* scale_out,
                                mdw_lm_head* head_out, mdw_stream_t stream) {
  if (H != MDW_HIDDEN) return MDW_ERR_UNSUPPORTED_SHAPE;
  if (V < 1 || V > 0x7fffffffLL) return MDW_ERR_UNSUPPORTED_SHAPE;
  if (!al16(w_bf16) || !al16(q_out) || !al16(scale_out) || !head_out) return MDW_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (launch_quantize_head(static_cast<const __nv_bfloat16*>(w_bf16), V, static_cast<uint8_t*>(q_out),
                           scale_out, s) != cudaSuccess)
    return MDW_ERR_CUDA;
  head_out->magic = MDW_MAGIC;
  head_out->fmt = MDW_FMT_FP8_E4M3_ROWSCALE;
  head_out->vocab = V;
  head_out->hidden = H;
  head_out->reserved = 0;
  head_out->w = q_out;
  head_out->row_scale = scale_out;
  return MDW_OK;
}

mdw_status mdw_lm_head_bf16_init(const void* w_bf16, int64_t V, int32_t H, mdw_lm_head* head_out) {
  if (H != MDW_HIDDEN) return MDW_ERR_UNSUPPORTED_SHAPE;
  if (V < 1 || V > 0x7fffffffLL) return MDW_ERR_UNSUPPORTED_SHAPE;
  if (!al16(w_bf16) || !head_out) return MDW_ERR_INVALID_ARG;
  head_out->magic = MDW_MAGIC;
  head_out->fmt = MDW_FMT_BF16;
  head_out->vocab = V;
  head_out->hidden = H;
  head_out->reserved = 0;
  head_out->w = w_bf16;
  head_out->row_scale = nullptr;
  return MDW_OK;
}

size_t mdw_lm_head_workspace_bytes(const mdw_lm_head* head, int32_t M, int32_t topk) {
  if (!head || M < 1 || M > MDW_MAX_M || topk < 1 || topk > MDW_MAX_VOCAB_TOPK) return 0;
  if (head_grid() <= 0) return 0;
  return kHdrWords * 4 + head_ws_bytes(M, topk, head->vocab);
}

mdw_status lm_head_fp8(const mdw_lm_head* head, int32_t M, const void* h_bf16, float* logits,
                       int32_t* argmax_out, int32_t topk, int32_t* topk_idx, float* topk_val, void* ws,
                       size_t ws_bytes, mdw_stream_t stream) {
  return head_entry(MDW_FMT_FP8_E4M3_ROWSCALE, head, M, h_bf16, logits, argmax_out, topk, topk_idx,
                    topk_val, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

mdw_status lm_head_bf16(const mdw_lm_head* head, int32_t M, const void* h_bf16, float* logits,
                        int32_t* argmax_out, int32_t topk, int32_t* topk_idx, float* topk_val, void* ws,
                        size_t ws_bytes, mdw_stream_t stream) {
  return head_entry(MDW_FMT_BF16, head, M, h_bf16, logits, argmax_out, topk, topk_idx, topk_val, ws,
                    ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

mdw_status lm_head_fp8_rmsnorm(const mdw_lm_head* head, int32_t M, const void* r_bf16, float* logits,
                               int32_t* argmax_out, int32_t topk, int32_t* topk_idx, float* topk_val, void* ws,
                               size_t ws_bytes, mdw_stream_t stream) {
  return head_entry(MDW_FMT_FP8_E4M3_ROWSCALE, head, M, r_bf16, logits, argmax_out, topk, topk_idx, topk_val,
                    ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream), 1);
}

mdw_status lm_head_fp8_sample(const mdw_lm_head* head, int32_t M, const void* h_bf16, int32_t norm_input,
                              int32_t topk, double temperature, double top_p, const double* u,
                              int32_t* token_out, int32_t* topk_idx, float* topk_val, void* ws,
                              size_t ws_bytes, mdw_stream_t stream) {
  if (!u || !token_out || (reinterpret_cast<uintptr_t>(u) & 7u) != 0 || (reinterpret_cast<uintptr_t>(token_out) & 3u) != 0)
    return MDW_ERR_INVALID_ARG;
  if (!(top_p > 0.0 && top_p <= 1.0) || temperature != temperature) return MDW_ERR_INVALID_ARG;
  Draw d;
  d.u = u;
  d.temperature = temperature;
  d.top_p = top_p;
  d.out = token_out;
  return head_entry(MDW_FMT_FP8_E4M3_ROWSCALE, head, M, h_bf16, nullptr, nullptr, topk, topk_idx, topk_val, ws,
                    ws_bytes, reinterpret_cast<cudaStream_t>(stream), norm_input != 0 ? 1 : 0, d);
}

size_t mdw_stack_workspace_bytes(const mdw_moe_weights* layers, int32_t L, const mdw_lm_head* head,
                                 int32_t M, int32_t topk) {
  if (!layers || L < 1 || L > kMaxLayers || M < 1 || M > MDW_MAX_M) return 0;
  if (!head) topk = 1;
  if (topk < 1 || topk > MDW_MAX_VOCAB_TOPK) return 0;
  int E = 0, K = 0;
  for (int l = 0; l < L; ++l) {
    if (check_weights(&layers[l]) != MDW_OK) return 0;
    E = E > layers[l].num_experts ? E : layers[l].num_experts;
    K = K > layers[l].top_k ? K : layers[l].top_k;
  }
  return moe_ws_layout(M, E, K, true, topk, head ? head->vocab : 0).total;
}

mdw_status moe_decode_stack(const mdw_moe_weights* layers, int32_t L, const mdw_lm_head* head, int32_t M,
                            const void* r0_bf16, void* resid_out, float* logits, int32_t* argmax_out,
                            int32_t topk, int32_t* topk_idx, float* topk_val, void* ws, size_t ws_bytes,
                            mdw_stream_t stream) {
  return moe_decode_stack_routed(layers, L, head, M, r0_bf16, resid_out, logits, argmax_out, topk, topk_idx,
                                 topk_val, nullptr, ws, ws_bytes, stream);
}

mdw_status moe_decode_stack_routed(const mdw_moe_weights* layers, int32_t L, const mdw_lm_head* head, int32_t M,
                                   const void* r0_bf16, void* resid_out, float* logits, int32_t* argmax_out,
                                   int32_t topk, int32_t* topk_idx, float* topk_val, const int32_t* topk_override,
                                   void* ws, size_t ws_bytes, mdw_stream_t stream) {
  if (!layers || L < 1 || L > kMaxLayers) return MDW_ERR_INVALID_ARG;
  mdw_status st = MDW_OK;
  if (head) {
    st = check_head(head, MDW_FMT_FP8_E4M3_ROWSCALE);
    if (st != MDW_OK) return st;
  } else if (!resid_out) {
    return MDW_ERR_INVALID_ARG;
  }
  int E = 0, K = 0;
  for (int l = 0; l < L; ++l) {
    st = check_weights(&layers[l]);
    if (st != MDW_OK) return st;
    if (l > 0 && (layers[l].num_experts != layers[0].num_experts || layers[l].top_k != layers[0].top_k ||
                  (layers[l].sh_w13_q == nullptr) != (layers[0].sh_w13_q == nullptr)))
      return MDW_ERR_INVALID_ARG;
    E = layers[l].num_experts;
    K = layers[l].top_k;
  }
  if (M < 1 || M > MDW_MAX_M) return MDW_ERR_INVALID_ARG;
  if (head && (topk < 1 || topk > MDW_MAX_VOCAB_TOPK || head->vocab < topk || !argmax_out ||
               !al16_or_null(logits)))
    return MDW_ERR_INVALID_ARG;
  if (!head) topk = 1;
  if (!al16(r0_bf16) || !al16_or_null(resid_out) || !al16(ws) ||
      (reinterpret_cast<uintptr_t>(topk_override) & 3u) != 0)
    return MDW_ERR_INVALID_ARG;
  const MoeWs lay = moe_ws_layout(M, E, K, true, topk, head ? head->vocab : 0);
  if (ws_bytes < lay.total) return MDW_ERR_WORKSPACE_TOO_SMALL;
  if (moe_grid() * 16 < kH / 2) return MDW_ERR_UNSUPPORTED_SHAPE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  MoeParams* p = new MoeParams();
  for (int l = 0; l < L; ++l) fill_layer(p->layers[l], &layers[l]);
  p->L = L; p->M = M; p->E = E; p->K = K;
  p->has_shared = layers[0].sh_w13_q != nullptr;
  p->stack_mode = 1;
  p->spin_budget = mdw_spin_budget();
  p->topk_override = topk_override;
  p->r0 = static_cast<const __nv_bfloat16*>(r0_bf16);
  if (resid_out) {
    p->resid = static_cast<__nv_bfloat16*>(resid_out);
    p->resid_pingpong = 0;
  } else {
    p->resid = reinterpret_cast<__nv_bfloat16*>(base + lay.resid);
    p->resid_pingpong = 1;
  }
  fill_moe_ws(*p, lay, base);
  st = MDW_OK;
  if (cudaMemsetAsync(base + lay.lay.header, 0, lay.zero_end - lay.lay.header, s) != cudaSuccess) st = MDW_ERR_CUDA;
  if (st == MDW_OK && resid_out &&
      cudaMemcpyAsync(resid_out, r0_bf16, (size_t)M * kH * 2, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    st = MDW_ERR_CUDA;
  if (st == MDW_OK) st = cuda_status(launch_moe(*p, s));
  const __nv_bfloat16* rL = p->resid + (size_t)(p->resid_pingpong ? (L & 1) : L) * M * kH;
  delete p;
  if (st != MDW_OK || !head) return st;
  return head_call(head, MDW_FMT_FP8_E4M3_ROWSCALE, M, rL, 1, logits, argmax_out, topk, topk_idx, topk_val,
                   reinterpret_cast<uint32_t*>(base + lay.lay.header), base + lay.cand, s);
}

mdw_status mdw_device_status(const void* ws, mdw_stream_t stream) {
  if (!al16(ws)) return MDW_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return MDW_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, ws, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return MDW_ERR_CUDA;
  return static_cast<mdw_status>(v);
}

}  // extern "C"
