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
constexpr int kMaxHeadGrid = 256;        // blocks of the head kernel (one per SM)

__host__ __device__ inline size_t head_smem_bytes(int M, int MAXM) {
  // xs [M][H] fp32 (its bytes later hold the warp lists [MAXM][warps][32] x 2 and the global
  // merge's [M][kMergeCap] x 2), thresholds / counters [MAXM] x 3, results [MAXM][32] x 2,
  // per-warp merge scratch [warps][kMergeCap] x 2
  return (size_t)M * kH * 4 + (size_t)MAXM * 12 + (size_t)MAXM * kMaxTK * 8 +
         (size_t)kWarps * kMergeCap * 8 + 64;
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

// tk-th best (value, index) among the warp's register-held candidates (PER per lane),
// by tk rounds of warp arg-max; every lane gets the result.
template <int PER>
__device__ void warp_kth(const float (&v)[PER], const int (&ix)[PER], int tk, float& kv, int& ki) {
  float pv = INFINITY;
  int pi = -1;
  for (int r = 0; r < tk; ++r) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < PER; ++j)
      if (beats(pv, pi, v[j], ix[j]) && beats(v[j], ix[j], bv, bi)) { bv = v[j]; bi = ix[j]; }
    warp_argmax(bv, bi);
    pv = bv; pi = bi;
  }
  kv = pv; ki = pi;
}

template <bool FP8, int MAXM>
__global__ void __launch_bounds__(kHeadThreads, 1) head_kernel(HeadParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  // xs [M][H] fp32 hidden states; after the row loop the same bytes hold the warps' lists
  // (mv / mi) and, in the last block, the global merge's compacted candidates
  float* xs = reinterpret_cast<float*>(smem);
  float* mv = xs;                                                         // [M][warps][32]
  int* mi = reinterpret_cast<int*>(mv + MAXM * kWarps * kMaxTK);
  float* thv = reinterpret_cast<float*>(smem + (size_t)p.M * kH * 4);     // [M] per-token thresholds
  int* thi = reinterpret_cast<int*>(thv + MAXM);
  int* cnt = thi + MAXM;                                                  // [M] compaction counters
  float* ov = reinterpret_cast<float*>(cnt + MAXM);                       // [M][32] results
  int* oi = reinterpret_cast<int*>(ov + MAXM * kMaxTK);
  float* tv_s = reinterpret_cast<float*>(oi + MAXM * kMaxTK);             // per-warp scratch (block merge)
  int* ti_s = reinterpret_cast<int*>(tv_s + kWarps * kMergeCap);
  __shared__ int is_last;
  const int M = p.M, tk = p.topk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long G = gridDim.x;
  const long long v0 = blockIdx.x * p.V / G, v1 = (blockIdx.x + 1) * p.V / G;
  constexpr int ROWB = FP8 ? kH : 2 * kH;
  constexpr int NC = FP8 ? 5 : 10;
  constexpr int EPC = FP8 ? 16 : 8;
  constexpr int kAhead = 4;                 // rows a warp prefetches into L2 ahead of use

  // prefetch this warp's first rows while the hidden states are prepared
  if (lane == 0)
    for (int a = 0; a < kAhead; ++a) {
      const long long v = v0 + warp + (long long)a * kWarps;
      if (v < v1) prefetch_l2(p.w + v * ROWB, ROWB);
    }

  // hidden states -> fp32 shared memory (optionally bf16(RMSNorm(.)) first); all threads,
  // 16-byte loads, fixed-order per-token reductions
  {
    float* part = tv_s;                      // [M][10] partial sums of squares
    for (int c = threadIdx.x; c < M * (kH / 8); c += blockDim.x) {
      const int t = c / (kH / 8), i = c % (kH / 8);
      const uint4 u = ld_cg16(reinterpret_cast<const uint4*>(p.x + (size_t)t * kH) + i);
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
      float ss = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float a = __uint_as_float(w4[k] << 16), b = __uint_as_float(w4[k] & 0xFFFF0000u);
        xs[(size_t)t * kH + 8 * i + 2 * k] = a;
        xs[(size_t)t * kH + 8 * i + 2 * k + 1] = b;
        ss = fmaf(a, a, ss);
        ss = fmaf(b, b, ss);
      }
      ss = warp_sum(ss);                    // a warp's 32 chunks belong to one token (320 % 32 == 0)
      if (lane == 0) part[t * 10 + i / 32] = ss;
    }
    __syncthreads();
    if (p.norm_input) {
      if (threadIdx.x < M) {
        float ss = 0.f;
        for (int j = 0; j < 10; ++j) ss += part[threadIdx.x * 10 + j];
        thv[threadIdx.x] = rsqrtf(ss / (float)kH + 1e-6f);
      }
      __syncthreads();
      for (int e = threadIdx.x; e < M * kH; e += blockDim.x)
        xs[e] = __bfloat162float(__float2bfloat16_rn(xs[e] * thv[e / kH]));
      __syncthreads();
    }
  }
  float xr[80];
  if (MAXM == 1) {
#pragma unroll
    for (int c = 0; c < NC; ++c)
#pragma unroll
      for (int k = 0; k < EPC; ++k) xr[c * EPC + k] = xs[(32 * c + lane) * EPC + k];
  }

  WarpList lst[MAXM];
#pragma unroll
  for (int t = 0; t < MAXM; ++t) list_init(lst[t]);

  auto load_row = [&](long long v, RowLoad<FP8>& ld) {
    const uint4* src = reinterpret_cast<const uint4*>(p.w + v * ROWB);
#pragma unroll
    for (int c = 0; c < NC; ++c) ld.q[c] = ldg_stream16(src + 32 * c + lane);
  };
  long long v = v0 + warp;
  RowLoad<FP8> cur, nxt;
  float sc_cur = 1.f, sc_nxt = 1.f;
  if (v < v1) { load_row(v, cur); if (FP8) sc_cur = p.row_scale[v]; }
  while (v < v1) {
    const long long vn = v + kWarps;
    if (lane == 0) {
      const long long vp = v + (long long)kAhead * kWarps;
      if (vp < v1) prefetch_l2(p.w + vp * ROWB, ROWB);
    }
    if (vn < v1) { load_row(vn, nxt); if (FP8) sc_nxt = p.row_scale[vn]; }
    float acc[MAXM];
    row_dot<FP8, MAXM>(cur, xs, xr, M, lane, acc);
#pragma unroll
    for (int t = 0; t < MAXM; ++t) {
      if (t < M) {
        const float logit = acc[t] * sc_cur;
        if (p.logits && lane == 0) p.logits[(size_t)t * p.V + v] = logit;
        list_insert(lst[t], logit, (int)v, tk, lane);
      }
    }
    cur = nxt;
    sc_cur = sc_nxt;
    v = vn;
  }

  // block merge: every warp writes its lists; warp t merges token t (threshold = best of
  // the warps' tk-th entries, so at least tk entries survive)
  __syncthreads();                          // xs is dead from here on: its bytes hold the lists
#pragma unroll
  for (int t = 0; t < MAXM; ++t) {
    if (t < M) {
      mv[(t * kWarps + warp) * kMaxTK + lane] = lst[t].v;
      mi[(t * kWarps + warp) * kMaxTK + lane] = lst[t].i;
    }
  }
  __syncthreads();
  for (int t = warp; t < M; t += kWarps) {
    float tv = -INFINITY;
    int ti = 0x7fffffff;
    if (lane < kWarps) {
      tv = mv[(t * kWarps + lane) * kMaxTK + tk - 1];
      ti = mi[(t * kWarps + lane) * kMaxTK + tk - 1];
    }
    warp_argmax(tv, ti);
    const float* lv = mv + t * kWarps * kMaxTK;
    const int* li = mi + t * kWarps * kMaxTK;
    auto ld = [&](int k, float& vv, int& ii) { vv = lv[k]; ii = li[k]; };
    float* outv = ov + t * kMaxTK;
    int* outi = oi + t * kMaxTK;
    warp_topk(ld, kWarps * kMaxTK, tk, tv, ti, tv_s + warp * kMergeCap, ti_s + warp * kMergeCap, kMergeCap,
              outv, outi, lane);
    const size_t o = ((size_t)blockIdx.x * M + t) * tk;
    for (int r = lane; r < tk; r += 32) { p.cand_val[o + r] = outv[r]; p.cand_idx[o + r] = outi[r]; }
  }

  // the last block to finish merges all blocks' candidates
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = (atomicAdd(p.hdr + kHdrDoneCtr, 1u) == (uint32_t)(G - 1));
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  const int n = (int)(G * tk);
  auto cand = [&](int t, int k, float& vv, int& ii) {
    const size_t o = ((size_t)(k / tk) * M + t) * tk + (k % tk);
    vv = ld_cg_f32(p.cand_val + o);
    ii = __float_as_int(ld_cg_f32(reinterpret_cast<const float*>(p.cand_idx + o)));
  };
  // A. per token, the tk-th best of the blocks' first entries: tk distinct entries are not
  //    worse than it, so it bounds the global tk-th entry from below
  for (int t = warp; t < M; t += kWarps) {
    constexpr int PER = kMaxHeadGrid / 32;
    float fv[PER];
    int fi[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) {                       // one load per block, all in flight
      const int b = lane + 32 * j;
      fv[j] = -INFINITY;
      fi[j] = 0x7fffffff;
      if (b < G) cand(t, b * tk, fv[j], fi[j]);
    }
    float kv;
    int ki;
    warp_kth<PER>(fv, fi, tk, kv, ki);
    if (lane == 0) { thv[t] = kv; thi[t] = ki; cnt[t] = 0; }
  }
  __syncthreads();
  // B. all threads: compact the candidates not worse than their token's threshold
  float* cv_s = xs;                                        // reuse (lists are dead): [M][kMergeCap]
  int* ci_s = reinterpret_cast<int*>(xs + (size_t)M * kMergeCap);
  constexpr int kScan = 8;                                 // loads in flight per thread
  for (int e0 = 0; e0 < M * n; e0 += blockDim.x * kScan) {
    float vv[kScan];
    int ii[kScan];
#pragma unroll
    for (int u = 0; u < kScan; ++u) {
      const int e = e0 + u * blockDim.x + threadIdx.x;
      vv[u] = -INFINITY;
      ii[u] = 0x7fffffff;
      if (e < M * n) cand(e / n, e % n, vv[u], ii[u]);
    }
#pragma unroll
    for (int u = 0; u < kScan; ++u) {
      const int e = e0 + u * blockDim.x + threadIdx.x;
      if (e < M * n) {
        const int t = e / n;
        if (!beats(thv[t], thi[t], vv[u], ii[u])) {
          const int pos = atomicAdd(&cnt[t], 1);
          if (pos < kMergeCap) { cv_s[t * kMergeCap + pos] = vv[u]; ci_s[t * kMergeCap + pos] = ii[u]; }
        }
      }
    }
  }
  __syncthreads();
  // C. warp t selects token t's top-tk (rescans global memory only on a compaction overflow)
  for (int t = warp; t < M; t += kWarps) {
    float* outv = ov + t * kMaxTK;
    int* outi = oi + t * kMaxTK;
    if (cnt[t] <= kMergeCap) {
      auto ld = [&](int k, float& vv, int& ii) { vv = cv_s[t * kMergeCap + k]; ii = ci_s[t * kMergeCap + k]; };
      warp_topk(ld, cnt[t], tk, thv[t], thi[t], tv_s + warp * kMergeCap, ti_s + warp * kMergeCap, kMergeCap,
                outv, outi, lane);
    } else {
      auto ld = [&](int k, float& vv, int& ii) { cand(t, k, vv, ii); };
      warp_topk(ld, n, tk, thv[t], thi[t], tv_s + warp * kMergeCap, ti_s + warp * kMergeCap, kMergeCap,
                outv, outi, lane);
    }
    for (int r = lane; r < tk; r += 32) {
      if (r == 0) p.argmax_out[t] = outi[0];
      if (p.topk_idx) p.topk_idx[(size_t)t * tk + r] = outi[r];
      if (p.topk_val) p.topk_val[(size_t)t * tk + r] = outv[r];
    }
  }
}

template <bool FP8, int MAXM>
cudaError_t launch_head_t(const HeadParams& p, cudaStream_t s) {
  const size_t smem = head_smem_bytes(p.M, MAXM);
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
