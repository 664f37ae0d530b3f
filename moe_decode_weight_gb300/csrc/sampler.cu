// mdw_sample_topk: the decode-time draw on top-k candidates already in device memory (the
// steps and their source are in mdw_sampler.cuh). One warp per token.
#include "mdw_device.cuh"
#include "mdw_internal.h"
#include "mdw_sampler.cuh"

namespace mdw {
namespace {

__global__ void __launch_bounds__(128) sample_kernel(int M, int k, const float* __restrict__ val,
                                                     const int32_t* __restrict__ idx, double temperature,
                                                     double top_p, const double* __restrict__ u,
                                                     int32_t* __restrict__ out) {
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= M) return;                               // warp-uniform
  const float* v = val + (size_t)t * k;
  const int32_t* ix = idx + (size_t)t * k;
  const int32_t tok = sample_candidates_warp([&](int i) { return v[i]; }, [&](int i) { return ix[i]; }, k,
                                             temperature, top_p, u[t], lane);
  if (lane == 0) out[t] = tok;
}

bool al4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace
}  // namespace mdw

using namespace mdw;

extern "C" mdw_status mdw_sample_topk(int32_t M, int32_t k, const float* topk_val, const int32_t* topk_idx,
                                      double temperature, double top_p, const double* u, int32_t* token_out,
                                      mdw_stream_t stream) {
  if (M < 1 || k < 1 || k > MDW_MAX_VOCAB_TOPK) return MDW_ERR_INVALID_ARG;
  if (!topk_val || !topk_idx || !u || !token_out || !al4(topk_val) || !al4(topk_idx) || !al4(token_out) ||
      (reinterpret_cast<uintptr_t>(u) & 7u) != 0)
    return MDW_ERR_INVALID_ARG;
  if (!(top_p > 0.0 && top_p <= 1.0) || temperature != temperature) return MDW_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  sample_kernel<<<(M + 3) / 4, 128, 0, s>>>(M, k, topk_val, topk_idx, temperature, top_p, u, token_out);
  return cudaGetLastError() == cudaSuccess ? MDW_OK : MDW_ERR_CUDA;
}
