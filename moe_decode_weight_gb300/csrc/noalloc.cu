// moe_decode_layer_noalloc: the same MoE decode layer as moe_decode_layer, for callers that
// cannot allocate device memory. Its scratch is a fixed array compiled into the library
// (one per GPU that loads it, held until the process exits) instead of a caller workspace.
//
// Who needs it: callers that run inside a host framework which owns the whole device-memory
// budget (an inference server that pre-reserves HBM for weights and caches and forbids
// further allocations), plain C callers without an allocator of their own, and
// latency-critical loops where a cudaMalloc / cudaFree would implicitly synchronise the
// device. Such a caller still provides its inputs and outputs; nothing else is allocated.
#include <mutex>

#include "mdw_device.cuh"
#include "mdw_internal.h"

namespace mdw {
namespace {

// The scratch of every moe_decode_layer_noalloc call on this GPU. 2 MiB hold the
// workspace of any call moe_decode_layer accepts (M <= MDW_MAX_M, E <= 512, top_k <= 8).
static __device__ __align__(256) uint8_t g_noalloc_scratch[MDW_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
uint8_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array for the current device, looked up once per device
// (in host code the array's name is only a stand-in for the device symbol).
mdw_status scratch_for_current_device(uint8_t** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MDW_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MDW_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<uint8_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  return MDW_OK;
}

bool aligned16_or_null(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace mdw

using namespace mdw;

extern "C" mdw_status moe_decode_layer_noalloc(const mdw_moe_weights* w, int32_t M, const void* x_bf16,
                                               void* y, int32_t y_is_fp32, const void* residual,
                                               const int32_t* topk_override, int32_t* topk_ids_out,
                                               float* topk_w_out, uint32_t* device_status_out,
                                               mdw_stream_t stream) {
  // shape and weight checks (format tag, M range, ...) and the scratch layout of this call
  mdw_moe_ws_layout pub;
  mdw_status st = mdw_moe_workspace_layout(w, M, &pub);
  if (st != MDW_OK) return st;
  const MoeWs ws = moe_ws_layout(M, w->num_experts, w->top_k, false, 1);
  const mdw_moe_ws_layout& lay = ws.lay;
  if (lay.total > MDW_NOALLOC_SCRATCH_BYTES) return MDW_ERR_WORKSPACE_TOO_SMALL;
  if (!x_bf16 || !y || !aligned16_or_null(x_bf16) || !aligned16_or_null(y) || !aligned16_or_null(residual) ||
      !aligned16_or_null(topk_override) || !aligned16_or_null(topk_ids_out) ||
      !aligned16_or_null(topk_w_out) || (reinterpret_cast<uintptr_t>(device_status_out) & 3u) != 0)
    return MDW_ERR_INVALID_ARG;
  if (moe_grid() * 16 < kH / 2) return MDW_ERR_UNSUPPORTED_SHAPE;
  uint8_t* base = nullptr;
  st = scratch_for_current_device(&base);
  if (st != MDW_OK) return st;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  MoeParams p{};                                   // on the host stack: no heap allocation
  LayerDesc& d = p.layers[0];
  d.router_w = static_cast<const __nv_bfloat16*>(w->router_w);
  d.w13_q = static_cast<const uint8_t*>(w->w13_q);
  d.w13_s = static_cast<const uint8_t*>(w->w13_s);
  d.w2_q = static_cast<const uint8_t*>(w->w2_q);
  d.w2_s = static_cast<const uint8_t*>(w->w2_s);
  d.sh_w13_q = static_cast<const uint8_t*>(w->sh_w13_q);
  d.sh_w13_s = static_cast<const uint8_t*>(w->sh_w13_s);
  d.sh_w2_q = static_cast<const uint8_t*>(w->sh_w2_q);
  d.sh_w2_s = static_cast<const uint8_t*>(w->sh_w2_s);
  p.L = 1; p.M = M; p.E = w->num_experts; p.K = w->top_k;
  p.has_shared = w->sh_w13_q != nullptr;
  p.stack_mode = 0;
  p.spin_budget = mdw_spin_budget();
  p.x_in = static_cast<const __nv_bfloat16*>(x_bf16);
  p.y_out = y;
  p.y_fp32 = y_is_fp32 != 0;
  p.residual = static_cast<const __nv_bfloat16*>(residual);
  p.topk_override = topk_override;
  p.ids_out = topk_ids_out;
  p.gates_out = topk_w_out;
  fill_moe_ws(p, ws, base);
  // the status word, the grid-barrier counter and the tagged exchange words must start at
  // zero on every call
  if (cudaMemsetAsync(base + lay.header, 0, ws.zero_end - lay.header, s) != cudaSuccess) return MDW_ERR_CUDA;
  if (launch_moe(p, s) != cudaSuccess) return MDW_ERR_CUDA;
  if (device_status_out &&
      cudaMemcpyAsync(device_status_out, base + lay.header, 4, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return MDW_ERR_CUDA;
  return MDW_OK;
}
