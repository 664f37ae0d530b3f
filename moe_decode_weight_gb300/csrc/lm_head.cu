// Online-FP8 LM head: one-time row-wise quantisation, and the weight-streaming GEMV with a
// fused arg-max / top-k (block-local lists, then a global merge in the last block).
//
// Method: "Three MoE Inference Optimizations NVIDIA Measured on DGX Spark", section
// "Online FP8 quantization halves the LM head weight reads" -- the BF16 head (157,184 x
// 2,560, ~402M weights, ~805 MB per token; runbyai.xyz/posts/593 paragraph 3) is quantised
// to FP8 once, when the head is built, halving the bytes every generated token reads;
// section "GSM8K measured a 42.5% throughput gain across 1,319 questions": decoding samples
// among the top_k = 29 tokens, and the synthetic run is greedy (arg-max).
//
// GB300 mapping: one block of 384 threads per SM, each block a contiguous slice of
// ~V/152 vocabulary rows; one warp per row at a time (a 2,560-byte FP8 row is exactly five
// 16-byte loads per lane), per-row scale applied after the warp reduction; each warp keeps
// its running top-k per token in registers (lane i holds the i-th best), the block merges
// its warps' lists, and the last block to finish merges all blocks' lists.
#include "mdw_device.cuh"
#include "mdw_internal.h"

namespace mdw {
namespace {

constexpr int kHeadThreads = kThreads;
constexpr int kMaxTK = 32;               // candidates per token per warp (lane-distributed)
constexpr int kMergeCap = 256;           // compacted candidates per warp during a merge

__host__ __device__ inline size_t head_smem_bytes(int M) {
  return (size_t)M * kH * 4 + (size_t)kWarps * (2 * kMaxTK + 2 * kMergeCap + 2 * kMaxTK) * 4;
}

// ------------------------------------------------------------------ quantisation

// One warp per row: amax (exact), scale = amax/448 (IEEE division; 1 for a zero row),
// q = E4M3(w / scale) rounded to nearest even, saturating.
__global__ void __launch_bounds__(256) quantize_head_kernel(const __nv_bfloat16* __restrict__ w,
                                                            long long V, uint8_t* __restrict__ q,
                                                            float* __restrict__ scale) {
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= V) return;
  const uint4* src = reinterpret_cast<const uint4*>(w + row * kH);
  uint4 v[10];
  float am = 0.f;
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    v[i] = ldg_stream16(src + 32 * i + lane);
    const uint32_t a[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
      am = fmaxf(am, fmaxf(fabsf(__uint_as_float(a[k] << 16)), fabsf(__uint_as_float(a[k] & 0xFFFF0000u))));
  }
  am = warp_max(am);
  const float s = am > 0.f ? __fdiv_rn(am, kE4M3Max) : 1.0f;
  uint2* dst = reinterpret_cast<uint2*>(q + row * kH);
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint32_t a[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    uint32_t c[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      c[k] = f32x2_to_e4m3x2(__fdiv_rn(__uint_as_float(a[k] << 16), s),
                             __fdiv_rn(__uint_as_float(a[k] & 0xFFFF0000u), s));
    dst[32 * i + lane] = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
  }
  if (lane == 0) scale[row] = s;
}

// ------------------------------------------------------------------ top-k lists

// Lane-distributed sorted list (lane i = i-th best; lanes >= tk hold -inf).
struct WarpList {
  float v;
  int i;
  float thr_v;   // warp-uniform copy of entry tk-1
  int thr_i;
};

__device__ __forceinline__ void list_init(WarpList& L) {
  L.v = -INFINITY; L.i = 0x7fffffff; L.thr_v = -INFINITY; L.thr_i = 0x7fffffff;
}

__device__ __forceinline__ void list_insert(WarpList& L, float v, int idx, int tk, int lane) {
  if (!beats(v, idx, L.thr_v, L.thr_i)) return;           // warp-uniform decision
  const unsigned better = __ballot_sync(0xffffffffu, lane < tk && beats(L.v, L.i, v, idx));
  const int pos = __popc(better);
  const float uv = __shfl_up_sync(0xffffffffu, L.v, 1);
  const int ui = __shfl_up_sync(0xffffffffu, L.i, 1);
  if (lane < tk) {
    if (lane == pos) { L.v = v; L.i = idx; }
    else if (lane > pos) { L.v = uv; L.i = ui; }
  }
  L.thr_v = __shfl_sync(0xffffffffu, L.v, tk - 1);
  L.thr_i = __shfl_sync(0xffffffffu, L.i, tk - 1);
}

// Top-tk (descending) of n candidates by one warp. Only candidates not worse than the
// threshold (tv, ti) can qualify: they are first compacted into tmp (capacity cap), then
// tk rounds of warp arg-max pick them in order. load(k) returns candidate k. If more than
// cap candidates pass, the rounds scan the candidates directly (slower, same result).
template <typename Load>
__device__ void warp_topk(Load load, int n, int tk, float tv, int ti, float* tmpv, int* tmpi, int cap,
                          float* outv, int* outi, int lane) {
  int count = 0;
  for (int k0 = 0; k0 < n; k0 += 32) {
    const int k = k0 + lane;
    float v = -INFINITY;
    int i = 0x7fffffff;
    bool keep = false;
    if (k < n) { load(k, v, i); keep = !beats(tv, ti, v, i); }
    const unsigned m = __ballot_sync(0xffffffffu, keep);
    const int pos = count + __popc(m & ((1u << lane) - 1u));
    if (keep && pos < cap) { tmpv[pos] = v; tmpi[pos] = i; }
    count += __popc(m);
  }
  __syncwarp();
  const bool compact = count <= cap;
  float pv = INFINITY;
  int pi = -1;
  for (int r = 0; r < tk; ++r) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    const int lim = compact ? count : n;
    for (int k = lane; k < lim; k += 32) {
      float v;
      int i;
      if (compact) { v = tmpv[k]; i = tmpi[k]; } else { load(k, v, i); }
      if (beats(tv, ti, v, i) || !beats(pv, pi, v, i)) continue;   // below threshold / taken
      if (beats(v, i, bv, bi)) { bv = v; bi = i; }
    }
    warp_argmax(bv, bi);
    pv = bv; pi = bi;
    if (lane == 0) { outv[r] = bv; outi[r] = bi; }
  }
  __syncwarp();
}

// ------------------------------------------------------------------ GEMV

template <bool FP8>
struct RowLoad {
  uint4 q[FP8 ? 5 : 10];
};

// Dot products of one row with the M tokens' hidden states (fp32 in shared memory, or in
// registers when M == 1), returned warp-reduced in acc[t].
template <bool FP8, int MAXM>
__device__ __forceinline__ void row_dot(const RowLoad<FP8>& ld, const float* xs, const float (&xr)[80],
                                        int M, int lane, float (&acc)[MAXM]) {
#pragma unroll
  for (int t = 0; t < MAXM; ++t) acc[t] = 0.f;
  constexpr int NC = FP8 ? 5 : 10;
  constexpr int EPC = FP8 ? 16 : 8;        // elements per 16-byte chunk
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    float w[EPC];
    const uint32_t a[4] = {ld.q[c].x, ld.q[c].y, ld.q[c].z, ld.q[c].w};
    if (FP8) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t lo = e4m3x2_to_f16x2(a[k] & 0xFFFF), hi = e4m3x2_to_f16x2(a[k] >> 16);
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&lo));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&hi));
        w[4 * k] = f0.x; w[4 * k + 1] = f0.y; w[4 * k + 2] = f1.x; w[4 * k + 3] = f1.y;
      }
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        w[2 * k] = __uint_as_float(a[k] << 16);
        w[2 * k + 1] = __uint_as_float(a[k] & 0xFFFF0000u);
      }
    }
    const int e0 = (32 * c + lane) * EPC;   // first hidden index of this chunk
#pragma unroll
    for (int t = 0; t < MAXM; ++t) {
      if (t < M) {
        float s0 = acc[t];
        if (MAXM == 1) {
#pragma unroll
          for (int k = 0; k < EPC; ++k) s0 = fmaf(w[k], xr[c * EPC + k], s0);
        } else {
          const float4* x4 = reinterpret_cast<const float4*>(xs + (size_t)t * kH + e0);
#pragma unroll
          for (int k = 0; k < EPC / 4; ++k) {
            const float4 xv = x4[k];
            s0 = fmaf(w[4 * k], xv.x, s0);
            s0 = fmaf(w[4 * k + 1], xv.y, s0);
            s0 = fmaf(w[4 * k + 2], xv.z, s0);
            s0 = fmaf(w[4 * k + 3], xv.w, s0);
          }
        }
        acc[t] = s0;
      }
    }
  }
#pragma unroll
  for (int t = 0; t < MAXM; ++t)
    if (t < M) acc[t] = warp_sum(acc[t]);
}

template <bool FP8, int MAXM>
__global__ void __launch_bounds__(kHeadThreads, 1) head_kernel(HeadParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  float* xs = reinterpret_cast<float*>(smem);                             // [M][H] fp32
  float* mv = reinterpret_cast<float*>(smem + (size_t)p.M * kH * 4);      // warp lists
  int* mi = reinterpret_cast<int*>(mv + kWarps * kMaxTK);
  float* tv_s = reinterpret_cast<float*>(mi + kWarps * kMaxTK);           // per-warp scratch
  int* ti_s = reinterpret_cast<int*>(tv_s + kWarps * kMergeCap);
  float* ov_s = reinterpret_cast<float*>(ti_s + kWarps * kMergeCap);      // per-warp results
  int* oi_s = reinterpret_cast<int*>(ov_s + kWarps * kMaxTK);
  __shared__ float th_v[kWarps];
  __shared__ int th_i[kWarps];
  __shared__ int is_last;
  const int M = p.M, tk = p.topk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long G = gridDim.x;
  const long long v0 = blockIdx.x * p.V / G, v1 = (blockIdx.x + 1) * p.V / G;
  constexpr int ROWB = FP8 ? kH : 2 * kH;

  // hidden states -> fp32 shared memory (optionally bf16(RMSNorm(.)) first)
  for (int t = warp; t < M; t += kWarps) {
    const __nv_bfloat16* src = p.x + (size_t)t * kH;
    float ss = 0.f;
    for (int e = lane; e < kH; e += 32) {
      const float a = __bfloat162float(src[e]);
      xs[(size_t)t * kH + e] = a;
      ss = fmaf(a, a, ss);
    }
    if (p.norm_input) {
      ss = warp_sum(ss);
      const float inv = rsqrtf(ss / (float)kH + 1e-6f);
      for (int e = lane; e < kH; e += 32)
        xs[(size_t)t * kH + e] = __bfloat162float(__float2bfloat16_rn(xs[(size_t)t * kH + e] * inv));
    }
  }
  __syncthreads();
  float xr[80];
  constexpr int EPC = FP8 ? 16 : 8;
  if (MAXM == 1) {
#pragma unroll
    for (int c = 0; c < (FP8 ? 5 : 10); ++c)
#pragma unroll
      for (int k = 0; k < EPC; ++k) xr[c * EPC + k] = xs[(32 * c + lane) * EPC + k];
  }

  WarpList lst[MAXM];
#pragma unroll
  for (int t = 0; t < MAXM; ++t) list_init(lst[t]);

  auto load_row = [&](long long v, RowLoad<FP8>& ld) {
    const uint4* src = reinterpret_cast<const uint4*>(p.w + v * ROWB);
#pragma unroll
    for (int c = 0; c < (FP8 ? 5 : 10); ++c) ld.q[c] = ldg_stream16(src + 32 * c + lane);
  };
  long long v = v0 + warp;
  RowLoad<FP8> cur, nxt;
  if (v < v1) load_row(v, cur);
  while (v < v1) {
    const long long vn = v + kWarps;
    if (vn < v1) load_row(vn, nxt);
    float acc[MAXM];
    row_dot<FP8, MAXM>(cur, xs, xr, M, lane, acc);
    const float sc = FP8 ? p.row_scale[v] : 1.0f;
#pragma unroll
    for (int t = 0; t < MAXM; ++t) {
      if (t < M) {
        const float logit = acc[t] * sc;
        if (p.logits && lane == 0) p.logits[(size_t)t * p.V + v] = logit;
        list_insert(lst[t], logit, (int)v, tk, lane);
      }
    }
    cur = nxt;
    v = vn;
  }

  // block merge per token: the warps' lists -> shared memory -> warp 0 selects the block's
  // top-tk among the entries not worse than the best of the warps' tk-th entries
  for (int t = 0; t < M; ++t) {
    float lv = -INFINITY, thv = -INFINITY;
    int li = 0x7fffffff, thi = 0x7fffffff;
#pragma unroll
    for (int u = 0; u < MAXM; ++u)
      if (u == t) { lv = lst[u].v; li = lst[u].i; thv = lst[u].thr_v; thi = lst[u].thr_i; }
    mv[warp * kMaxTK + lane] = lv;
    mi[warp * kMaxTK + lane] = li;
    if (lane == 0) { th_v[warp] = thv; th_i[warp] = thi; }
    __syncthreads();
    if (warp == 0) {
      float tv = lane < kWarps ? th_v[lane] : -INFINITY;
      int ti = lane < kWarps ? th_i[lane] : 0x7fffffff;
      warp_argmax(tv, ti);
      auto ld = [&](int k, float& v, int& i) { v = mv[k]; i = mi[k]; };
      warp_topk(ld, kWarps * kMaxTK, tk, tv, ti, tv_s, ti_s, kMergeCap, ov_s, oi_s, lane);
      const size_t o = ((size_t)blockIdx.x * M + t) * tk;
      for (int r = lane; r < tk; r += 32) { p.cand_val[o + r] = ov_s[r]; p.cand_idx[o + r] = oi_s[r]; }
    }
    __syncthreads();
  }

  // the last block to finish merges all blocks' candidates
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = (atomicAdd(p.hdr + kHdrDoneCtr, 1u) == (uint32_t)(G - 1));
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  for (int t = warp; t < M; t += kWarps) {
    // threshold: the best of the blocks' tk-th entries
    float tv = -INFINITY;
    int ti = 0x7fffffff;
    for (long long b = lane; b < G; b += 32) {
      const size_t o = ((size_t)b * M + t) * tk + (tk - 1);
      const float cv = ld_cg_f32(p.cand_val + o);
      const int ci = __float_as_int(ld_cg_f32(reinterpret_cast<const float*>(p.cand_idx + o)));
      if (beats(cv, ci, tv, ti)) { tv = cv; ti = ci; }
    }
    warp_argmax(tv, ti);
    auto ld = [&](int k, float& v, int& i) {
      const size_t o = ((size_t)(k / tk) * M + t) * tk + (k % tk);
      v = ld_cg_f32(p.cand_val + o);
      i = __float_as_int(ld_cg_f32(reinterpret_cast<const float*>(p.cand_idx + o)));
    };
    float* outv = ov_s + warp * kMaxTK;
    int* outi = oi_s + warp * kMaxTK;
    warp_topk(ld, (int)(G * tk), tk, tv, ti, tv_s + warp * kMergeCap, ti_s + warp * kMergeCap,
              kMergeCap, outv, outi, lane);
    for (int r = lane; r < tk; r += 32) {
      if (r == 0) p.argmax_out[t] = outi[0];
      if (p.topk_idx) p.topk_idx[(size_t)t * tk + r] = outi[r];
      if (p.topk_val) p.topk_val[(size_t)t * tk + r] = outv[r];
    }
  }
}

template <bool FP8, int MAXM>
cudaError_t launch_head_t(const HeadParams& p, cudaStream_t s) {
  const size_t smem = head_smem_bytes(p.M);
  auto kern = head_kernel<FP8, MAXM>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<head_grid(), kHeadThreads, smem, s>>>(p);
  return cudaGetLastError();
}

template <bool FP8>
cudaError_t launch_head_any(const HeadParams& p, cudaStream_t s) {
  if (p.M <= 1) return launch_head_t<FP8, 1>(p, s);
  if (p.M <= 2) return launch_head_t<FP8, 2>(p, s);
  if (p.M <= 4) return launch_head_t<FP8, 4>(p, s);
  if (p.M <= 8) return launch_head_t<FP8, 8>(p, s);
  return launch_head_t<FP8, 16>(p, s);
}

}  // namespace

size_t head_ws_bytes(int M, int topk, int grid) {
  return (size_t)grid * M * topk * 8 + 512;
}

cudaError_t launch_head_fp8(const HeadParams& p, cudaStream_t s) { return launch_head_any<true>(p, s); }
cudaError_t launch_head_bf16(const HeadParams& p, cudaStream_t s) { return launch_head_any<false>(p, s); }

cudaError_t launch_quantize_head(const __nv_bfloat16* w, long long V, uint8_t* q, float* scale,
                                 cudaStream_t s) {
  const long long blocks = (V + 7) / 8;
  quantize_head_kernel<<<(unsigned)blocks, 256, 0, s>>>(w, V, q, scale);
  return cudaGetLastError();
}

}  // namespace mdw
