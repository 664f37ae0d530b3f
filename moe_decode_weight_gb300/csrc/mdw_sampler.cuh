// The decode-time draw on the LM head's top-k candidates: temperature, nucleus (top_p) and
// one inverse-CDF draw per token.
//
// Method: "Three MoE Inference Optimizations NVIDIA Measured on DGX Spark",
// section "GSM8K measured a 42.5% throughput gain across 1,319 questions" -- the evaluation
// samples at temperature 0.6, top_p 0.95, top_k 29 (also runbyai.xyz/posts/593, paragraph
// 6). The pages give only the settings; the steps are the plain reading:
//   * candidates in head order (descending logit, ties to the lower id), softmax of z / T
//     over the k candidates, e_i = exp((z_i - z_0) / T);
//   * keep the shortest prefix whose mass reaches top_p (the crossing candidate stays);
//   * the token is the first kept candidate whose cumulative mass exceeds u * kept mass,
//     u in [0, 1) supplied by the caller;
//   * temperature <= 0: the first candidate (greedy).
// Arithmetic: float64, sums left to right (one warp per token; k <= 32).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mdw {

// One warp per token: lane i < k computes e_i (one exp per lane), lane 0 takes the sums in
// order. Every lane returns the drawn id.
template <typename LoadV, typename LoadI>
__device__ __forceinline__ int32_t sample_candidates_warp(LoadV val, LoadI id, int k, double temperature,
                                                          double top_p, double u, int lane) {
  if (!(temperature > 0.0)) return id(0);
  const double z0 = (double)val(0);
  const double e = lane < k ? exp(((double)val(lane) - z0) / temperature) : 0.0;
  int pick = 0;
  if (true) {
    double total = 0.0;
    for (int i = 0; i < k; ++i) total += __shfl_sync(0xffffffffu, e, i);
    int cut = k - 1;
    double c = 0.0;
    for (int i = 0; i < k; ++i) {
      c += __shfl_sync(0xffffffffu, e, i);
      if (c >= top_p * total) { cut = i; break; }
    }
    double kept = 0.0;
    for (int i = 0; i <= cut; ++i) kept += __shfl_sync(0xffffffffu, e, i);
    const double target = u * kept;
    c = 0.0;
    pick = cut;
    for (int i = 0; i <= cut; ++i) {
      c += __shfl_sync(0xffffffffu, e, i);
      if (target < c) { pick = i; break; }
    }
  }
  return id(pick);
}

}  // namespace mdw
