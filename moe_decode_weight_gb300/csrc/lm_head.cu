// Online-FP8 LM head: one-time row-wise quantisation, and the weight-streaming GEMV with a
// fused arg-max / top-k (block-local lists, merged per group of blocks, then globally).
//
// Method: "Three MoE Inference Optimizations NVIDIA Measured on DGX Spark", section
// "Online FP8 quantization halves the LM head weight reads" -- the BF16 head (157,184 x
// 2,560, ~402M weights, ~805 MB per token; runbyai.xyz/posts/593 paragraph 3) is quantised
// to FP8 once, when the head is built, halving the bytes every generated token reads;
// section "GSM8K measured a 42.5% throughput gain across 1,319 questions": decoding samples
// among the top_k = 29 tokens, and the synthetic run is greedy (arg-max).
//
// GB300 mapping: one block of 384 threads per SM, each block a contiguous slice of
// ~V/152 vocabulary rows, each warp walking 16-row tiles of the slice on m16n8k16 tensor-core
// MMAs (rows x tokens, fp32 accumulation; FP8 weights converted exactly to f16 in
// registers), the per-row scale applied once per logit; each warp keeps its running top-k
// per token in registers (lane i holds the i-th best), the block merges its warps' lists,
// the last block of each group of 16 to finish merges the group's lists, and the last group
// merges the group lists (and, when asked, draws the token from the final list). A window of
// more than kHeadListM tokens keeps no lists while streaming (per-token register lists cost
// more than they save there): it writes its logits, and each block then selects from its own
// rows (one warp per token), so the head is still streamed once.
#include "mdw_device.cuh"
#include "mdw_internal.h"
#include "mdw_sampler.cuh"

namespace mdw {
namespace {

constexpr int kHeadThreads = kThreads;
constexpr int kMaxTK = 32;               // list length (lane-distributed; tk <= 32)
// Built only with -DMDW_TRACE (a profiling build, never the product build): %globaltimer at
// the head kernel's phase boundaries, per block ([0] start, [1] hidden states ready, [2] all
// tiles done, [20] cut tiles finished, [21] warp lists stored, [22] block tree merged, [3]
// block list written, [4] group merge starts, [5] final merge starts, [6] end) and per warp
// ([8 + warp] its last unit done).
#ifdef MDW_TRACE
__device__ unsigned long long g_head_trace[kMaxHeadGrid * 24];
__device__ __forceinline__ void head_trace(int slot) {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  g_head_trace[blockIdx.x * 24 + slot] = t;
}
#define MDW_HEAD_TRACE(cond, slot) do { if (cond) head_trace(slot); } while (0)
#else
#define MDW_HEAD_TRACE(cond, slot) do { } while (0)
#endif
#ifndef MDW_HEAD_U
#define MDW_HEAD_U 4                     // 64-byte chunks per row whose loads a warp keeps in flight
#endif
#ifndef MDW_HEAD_PF
#define MDW_HEAD_PF 4                    // units a warp prefetches into L2 ahead of its loads
#endif

// Bytes per token row of the hidden states in shared memory (padded so the MMA B-fragment
// reads of different tokens fall in different banks).
template <bool FP8>
__host__ __device__ constexpr int head_x_stride() { return FP8 ? 2 * kH + 16 : 2 * kH + 64; }

// Region 0 holds the hidden states [M][xstride] during the tiles; afterwards the lists
// [MAXM][warps][32] (values, then indices) followed by the split tiles' partial sums
// [warps][2][NT][32 lanes][4].
__host__ __device__ inline size_t head_lists_bytes(int MAXM) { return (size_t)MAXM * kWarps * kMaxTK * 8; }
__host__ __device__ inline size_t head_region0_bytes(int M, int MAXM, int xstride) {
  const int NT = (MAXM + 7) / 8;
  size_t r = (size_t)M * xstride;
  const size_t after = head_lists_bytes(MAXM) + (size_t)kWarps * 2 * NT * 32 * 16;
  if (after > r) r = after;
  return (r + 15) & ~(size_t)15;
}
// + per-token x multipliers, 1/rms, scale exponents and partial reductions [MAXM][10]
__host__ __device__ inline size_t head_smem_bytes(int M, int MAXM, int xstride) {
  return head_region0_bytes(M, MAXM, xstride) + (size_t)MAXM * 13 * 4 + 64;
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

// Lane-distributed sorted list (lane i = i-th best under `beats`; unused lanes hold the
// pad (-inf, INT_MAX), which every real candidate beats).
struct WarpList {
  float v;
  int i;
  float thr_v;   // warp-uniform copy of entry tk-1 (the bar a new candidate must beat)
  int thr_i;
};
constexpr int kPadIdx = 0x7fffffff;

__device__ __forceinline__ void list_init(WarpList& L) {
  L.v = -INFINITY; L.i = kPadIdx; L.thr_v = -INFINITY; L.thr_i = kPadIdx;
}

// Insert one warp-uniform candidate (no-op unless it beats entry tk-1).
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

// (v, i) <- the 32 best of the union of two descending lane-distributed lists (v, i) and
// (bv, bi): pairing entry j of one with entry 31 - j of the other and keeping the better
// gives a bitonic sequence holding the 32 best; a descending bitonic merge (five
// compare-exchange stages) sorts it. The first tk lanes are then the top-tk of the union
// whenever each input holds its own top-tk.
__device__ __forceinline__ void list_merge(float& v, int& i, float bv, int bi, int lane) {
  const float rv = __shfl_sync(0xffffffffu, bv, 31 - lane);
  const int ri = __shfl_sync(0xffffffffu, bi, 31 - lane);
  if (beats(rv, ri, v, i)) { v = rv; i = ri; }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (((lane & o) == 0) == beats(ov, oi, v, i)) { v = ov; i = oi; }
  }
}

// Block-wide tree merge of the lists S[t][w] (w < warps, 32 entries each, values at sv and
// indices at si, index (t * warps + w) * 32 + lane) into S[t][0], for every token t < M.
// Level s merges list w + s into list w for w a multiple of 2s; the (token, pair) merges
// of a level are spread over the warps. Every thread of the block must call it.
__device__ void tree_merge(float* sv, int* si, int M, int warp, int lane) {
  __syncthreads();
#pragma unroll 1
  for (int s = 1; s < kWarps; s <<= 1) {
    int np = 0;
    for (int w = 0; w + s < kWarps; w += 2 * s) ++np;
    for (int job = warp; job < M * np; job += kWarps) {
      const int t = job / np, w = (job % np) * 2 * s;
      const int a = (t * kWarps + w) * kMaxTK + lane, b = (t * kWarps + w + s) * kMaxTK + lane;
      float v = sv[a];
      int i = si[a];
      list_merge(v, i, sv[b], si[b], lane);
      sv[a] = v;
      si[a] = i;
    }
    __syncthreads();
  }
}

// Loads the lists j < n of every token (list j of token t at cv / ci + ((first + j) * M + t)
// * tk, tk entries, written by other blocks of this launch), merges them into S[t][0].
// Warp w takes lists w, w + warps, ... of each token (n <= 2 * warps); the loads of up to 8
// tokens are issued before the first merge.
template <int MAXM>
__device__ void merge_global_lists(const float* cv, const int* ci, int first, int n, int M, int tk,
                                   float* sv, int* si, int warp, int lane) {
  constexpr int CH = MAXM < 8 ? MAXM : 8;
#pragma unroll 1
  for (int t0 = 0; t0 < M; t0 += CH) {
    float av[CH], bv[CH];
    int ai[CH], bi[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int t = t0 + c;
      av[c] = bv[c] = -INFINITY;
      ai[c] = bi[c] = kPadIdx;
      if (t < M && lane < tk) {
        if (warp < n) {
          const size_t o = ((size_t)(first + warp) * M + t) * tk + lane;
          av[c] = ld_cg_f32(cv + o);
          ai[c] = __float_as_int(ld_cg_f32(reinterpret_cast<const float*>(ci) + o));
        }
        if (warp + kWarps < n) {
          const size_t o = ((size_t)(first + warp + kWarps) * M + t) * tk + lane;
          bv[c] = ld_cg_f32(cv + o);
          bi[c] = __float_as_int(ld_cg_f32(reinterpret_cast<const float*>(ci) + o));
        }
      }
    }
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int t = t0 + c;
      if (t < M) {
        if (warp + kWarps < n) list_merge(av[c], ai[c], bv[c], bi[c], lane);
        sv[(t * kWarps + warp) * kMaxTK + lane] = av[c];
        si[(t * kWarps + warp) * kMaxTK + lane] = ai[c];
      }
    }
  }
  tree_merge(sv, si, M, warp, lane);
}

// ------------------------------------------------------------------ GEMV

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
               "{%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
               "{%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The head GEMV on the tensor cores. The block's vocabulary slice is cut into 16-row
// tiles, each tile's K into NG units of U 64-byte chunks, and the (tile, unit) sequence into
// 12 equal contiguous ranges, one per warp (so every warp streams the same number of
// bytes; a tile cut between warps is finished from the warps' partial sums afterwards).
// Per tile: D[16 rows][8 tokens] = W[16 rows][K] x X^T on m16n8k16 MMAs with fp32
// accumulation, then logit = D * row scale (FP8: E4M3 weights -> f16 exactly, hidden states
// as f16 under a per-token power-of-two scale that keeps them inside the f16 range; BF16:
// bf16 operands). Lane (g, q) loads bytes 16q..16q+15 of each chunk of rows g and g + 8
// (full 32-byte sectors per warp load) and the matching hidden-state values, i.e. the
// MMAs run on a permuted K order that is the same for W and X.
template <bool FP8, int MAXM>
__global__ void __launch_bounds__(kHeadThreads, 1) head_kernel(HeadParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  constexpr int XS = head_x_stride<FP8>();
  constexpr int NT = (MAXM + 7) / 8;                 // 8-token column groups
  // up to kHeadListM tokens every warp keeps its running top-k per token in registers while
  // it walks its tiles; a wider window writes its logits (p.logits is then always given) and
  // selects from the block's rows afterwards, one warp per token
  constexpr bool LISTS = MAXM <= kHeadListM;
  const int M = p.M, tk = p.topk;
  uint8_t* xsm = smem;                                // [M][XS] hidden states (MMA operand)
  float* lv = reinterpret_cast<float*>(smem);         // [MAXM][warps][32] list values
  int* li = reinterpret_cast<int*>(smem + (size_t)MAXM * kWarps * kMaxTK * 4);
  float* rec = reinterpret_cast<float*>(smem + head_lists_bytes(MAXM));   // split-tile partials
  float* tokv = reinterpret_cast<float*>(smem + head_region0_bytes(M, MAXM, XS));
  float* xmul = tokv;                                 // [MAXM] 2^k (FP8 f16 scaling)
  float* tinv = tokv + MAXM;                          // [MAXM] 1 / rms
  int* tkexp = reinterpret_cast<int*>(tokv + 2 * MAXM);   // [MAXM] k
  float* part = tokv + 3 * MAXM;                      // [MAXM][10]
  __shared__ int is_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const long long G = gridDim.x;
  const long long v0 = blockIdx.x * p.V / G, v1 = (blockIdx.x + 1) * p.V / G;
  constexpr int ROWB = FP8 ? kH : 2 * kH;
  constexpr int NCH = ROWB / 64;                      // 64-byte chunks per row
  // chunks per unit (loads in flight together); the 32-token kernel holds half as many, its
  // accumulators taking the registers
  constexpr int U = MAXM > 16 ? MDW_HEAD_U / 2 : MDW_HEAD_U;
  constexpr int NG = NCH / U;                         // units per tile
  static_assert(U % 2 == 0 && NCH % U == 0, "units must tile a row in whole 128-byte lines");
  const int ntile = (int)((v1 - v0 + 15) / 16);
  const int total = ntile * NG;
  auto ubeg = [&](int w) { return (int)((long long)w * total / kWarps); };
  const int u0 = ubeg(warp), u1 = ubeg(warp + 1);
  MDW_HEAD_TRACE(threadIdx.x == 0, 0);

  // L2 prefetch of unit u of this warp: 16 rows x 64U bytes as whole 128-byte lines
  auto prefetch_unit = [&](int u) {
    if (u >= u1) return;
    const int tl = u / NG, gi = u % NG;
    constexpr int LPR = U / 2;                         // lines per row per unit
    for (int pl = lane; pl < 16 * LPR; pl += 32) {
      const long long row = v0 + 16LL * tl + pl / LPR;
      if (row < v1) {
        const uint8_t* a = p.w + row * ROWB + 64 * U * gi + 128 * (pl % LPR);
        asm volatile("prefetch.global.L2 [%0];" :: "l"(a));
      }
    }
  };

  // hidden states -> shared memory, every chunk loaded once into registers: bf16 values
  // (optionally bf16(RMSNorm(.))), FP8 path then f16(x * 2^-k) with k = floor(log2 amax) - 14
  {
    constexpr int CPT = kH / 8;                       // 16-byte chunks per token
    constexpr int CH = (MAXM * CPT + kHeadThreads - 1) / kHeadThreads;
    uint32_t xr[CH][4];
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      const int c = threadIdx.x + j * kHeadThreads;
      uint4 u = make_uint4(0, 0, 0, 0);
      if (c < M * CPT) u = ld_cg16(reinterpret_cast<const uint4*>(p.x) + c);
      xr[j][0] = u.x; xr[j][1] = u.y; xr[j][2] = u.z; xr[j][3] = u.w;
    }
    for (int n = 0; n < MDW_HEAD_PF; ++n) prefetch_unit(u0 + n);
    // per-token reductions: a warp's 32 chunks belong to one token (320 % 32 == 0, 384 % 32 == 0)
    auto reduce = [&](bool sq) {
#pragma unroll
      for (int j = 0; j < CH; ++j) {
        const int c = threadIdx.x + j * kHeadThreads;
        if (j * kHeadThreads + warp * 32 >= M * CPT) break;      // warp-uniform
        float r = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float a = __uint_as_float(xr[j][k] << 16), b = __uint_as_float(xr[j][k] & 0xFFFF0000u);
          if (sq) { r = fmaf(a, a, r); r = fmaf(b, b, r); }
          else r = fmaxf(r, fmaxf(fabsf(a), fabsf(b)));
        }
        r = sq ? warp_sum(r) : warp_max(r);
        if (lane == 0) part[(c / CPT) * 10 + (c % CPT) / 32] = r;
      }
      __syncthreads();
    };
    if (p.norm_input) {
      reduce(true);
      if (threadIdx.x < M) {
        float ss = 0.f;
        for (int j = 0; j < 10; ++j) ss += part[threadIdx.x * 10 + j];
        tinv[threadIdx.x] = rsqrtf(ss / (float)kH + 1e-6f);
      }
      __syncthreads();
#pragma unroll
      for (int j = 0; j < CH; ++j) {
        const int c = threadIdx.x + j * kHeadThreads;
        if (c < M * CPT) {
          const float inv = tinv[c / CPT];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const __nv_bfloat162 r2 = __floats2bfloat162_rn(__uint_as_float(xr[j][k] << 16) * inv,
                                                            __uint_as_float(xr[j][k] & 0xFFFF0000u) * inv);
            xr[j][k] = *reinterpret_cast<const uint32_t*>(&r2);
          }
        }
      }
      __syncthreads();                                 // part is reused below
    }
    if (FP8) {
      reduce(false);
      if (threadIdx.x < M) {
        float am = 0.f;
        for (int j = 0; j < 10; ++j) am = fmaxf(am, part[threadIdx.x * 10 + j]);
        // scaled values lie below 2^15 (f16 max 65504) and the small ones stay clear of the
        // f16 subnormal range; every step is a power of two, so only the f16 rounding of
        // values far below amax is inexact
        int e = 0;
        frexpf(am, &e);                                // am = m * 2^e, m in [0.5, 1)
        const int k = (am > 0.f && am < INFINITY) ? max(-100, min(100, e - 15)) : 0;
        xmul[threadIdx.x] = ldexpf(1.0f, k);
        tkexp[threadIdx.x] = k;
      }
      __syncthreads();
    } else if (threadIdx.x < M) {
      xmul[threadIdx.x] = 1.0f;
    }
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      const int c = threadIdx.x + j * kHeadThreads;
      if (c < M * CPT) {
        const int t = c / CPT, i = c % CPT;
        uint32_t o[4];
        if (FP8) {
          const int k = tkexp[t];
#pragma unroll
          for (int m2 = 0; m2 < 4; ++m2) {
            const __half2 hh = __floats2half2_rn(ldexpf(__uint_as_float(xr[j][m2] << 16), -k),
                                                 ldexpf(__uint_as_float(xr[j][m2] & 0xFFFF0000u), -k));
            o[m2] = *reinterpret_cast<const uint32_t*>(&hh);
          }
        } else {
#pragma unroll
          for (int m2 = 0; m2 < 4; ++m2) o[m2] = xr[j][m2];
        }
        *reinterpret_cast<uint4*>(xsm + (size_t)t * XS + 16 * i) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    __syncthreads();
  }
  MDW_HEAD_TRACE(threadIdx.x == 0, 1);

  WarpList lst[LISTS ? MAXM : 1];
#pragma unroll
  for (int t = 0; t < (LISTS ? MAXM : 1); ++t) list_init(lst[t]);
  constexpr int STEPS = FP8 ? 4 : 2;                  // k16 steps per 64-byte chunk

  // logits of a finished tile (sums d of rows vt + g (+8), tokens 8nt + 2q (+1)) -> lists
  auto finish_tile = [&](int tl, float (&d)[NT][4]) {
    const long long vt = v0 + 16LL * tl;
    const bool va_ok = vt + g < v1, vb_ok = vt + g + 8 < v1;
    const float sa = (FP8 && va_ok) ? p.row_scale[vt + g] : 1.0f;
    const float sb = (FP8 && vb_ok) ? p.row_scale[vt + g + 8] : 1.0f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float lg[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int tok = 8 * nt + 2 * q + (j & 1);
        const bool okr = (j < 2) ? va_ok : vb_ok;
        lg[j] = d[nt][j] * ((j < 2) ? sa : sb) * (tok < M ? xmul[tok] : 1.0f);
        if (p.logits && okr && tok < M) p.logits[(size_t)tok * p.V + vt + g + ((j >> 1) << 3)] = lg[j];
        if (lg[j] != lg[j]) lg[j] = -INFINITY;         // a NaN logit ranks last in the top-k
      }
      if (!LISTS) continue;
#pragma unroll
      for (int t8 = 0; t8 < 8; ++t8) {
        const int t = 8 * nt + t8;
        if (t >= M) break;
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const bool mine = (q == (t8 >> 1)) && (hr ? vb_ok : va_ok);
          const float val = lg[2 * hr + (t8 & 1)];
          const int idx = (int)(vt + g + 8 * hr);
          WarpList& Lt = lst[LISTS ? t : 0];
          unsigned m = __ballot_sync(0xffffffffu, mine && beats(val, idx, Lt.thr_v, Lt.thr_i));
          while (m) {
            const int src = __ffs(m) - 1;
            m &= m - 1;
            const float bv = __shfl_sync(0xffffffffu, val, src);
            const int bi = __shfl_sync(0xffffffffu, idx, src);
            list_insert(Lt, bv, bi, tk, lane);
          }
        }
      }
    }
  };

  float acc[NT][STEPS][4];
  float part0[NT][4], part1[NT][4];                   // partial sums of this warp's cut first / last tile
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 4; ++j) part0[nt][j] = part1[nt][j] = 0.f;
  const uint8_t* pa = nullptr;
  const uint8_t* pb = nullptr;
  bool va_ok = false, vb_ok = false;
  for (int u = u0; u < u1; ++u) {
    const int tl = u / NG, gi = u % NG;
    if (u == u0 || gi == 0) {                          // a tile starts (or this warp's range does)
      const long long vt = v0 + 16LL * tl;
      va_ok = vt + g < v1;
      vb_ok = vt + g + 8 < v1;
      pa = p.w + (vt + g) * ROWB + 16 * q;
      pb = p.w + (vt + g + 8) * ROWB + 16 * q;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int s2 = 0; s2 < STEPS; ++s2)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[nt][s2][j] = 0.f;
    }
    if (MDW_HEAD_PF > 0) prefetch_unit(u + MDW_HEAD_PF);
    uint4 wa[U], wb[U];
#pragma unroll
    for (int c = 0; c < U; ++c) {
      const int off = 64 * (gi * U + c);
      wa[c] = va_ok ? ldg_stream16(pa + off) : make_uint4(0, 0, 0, 0);
      wb[c] = vb_ok ? ldg_stream16(pb + off) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int c = 0; c < U; ++c) {
      const int ch = gi * U + c;
      const uint32_t A[4] = {wa[c].x, wa[c].y, wa[c].z, wa[c].w};
      const uint32_t B[4] = {wb[c].x, wb[c].y, wb[c].z, wb[c].w};
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int tok = 8 * nt + g;
        const bool have = tok < M;
        const uint8_t* xt = xsm + (size_t)tok * XS;
        if (FP8) {
          uint4 x0 = make_uint4(0, 0, 0, 0), x1 = make_uint4(0, 0, 0, 0);
          if (have) {
            x0 = *reinterpret_cast<const uint4*>(xt + 2 * (64 * ch + 16 * q));
            x1 = *reinterpret_cast<const uint4*>(xt + 2 * (64 * ch + 16 * q) + 16);
          }
          const uint32_t X[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
          for (int s2 = 0; s2 < STEPS; ++s2)
            mma_f16_16816(acc[nt][s2], e4m3x2_to_f16x2(A[s2] & 0xFFFF), e4m3x2_to_f16x2(B[s2] & 0xFFFF),
                          e4m3x2_to_f16x2(A[s2] >> 16), e4m3x2_to_f16x2(B[s2] >> 16), X[2 * s2], X[2 * s2 + 1]);
        } else {
          uint4 x0 = make_uint4(0, 0, 0, 0);
          if (have) x0 = *reinterpret_cast<const uint4*>(xt + 64 * ch + 16 * q);
          const uint32_t X[4] = {x0.x, x0.y, x0.z, x0.w};
#pragma unroll
          for (int s2 = 0; s2 < STEPS; ++s2)
            mma_bf16_16816(acc[nt][s2], A[2 * s2], B[2 * s2], A[2 * s2 + 1], B[2 * s2 + 1], X[2 * s2], X[2 * s2 + 1]);
        }
      }
    }
    if (gi == NG - 1 || u == u1 - 1) {                 // a tile ends (or this warp's range does)
      float d[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float v = acc[nt][0][j];
#pragma unroll
          for (int s2 = 1; s2 < STEPS; ++s2) v += acc[nt][s2][j];
          d[nt][j] = v;
        }
      if (tl * NG >= u0 && gi == NG - 1) {
        finish_tile(tl, d);                            // the whole tile is this warp's
      } else if (tl == u0 / NG) {                      // first tile, cut at one end or both
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int j = 0; j < 4; ++j) part0[nt][j] = d[nt][j];
      } else {                                         // last tile, cut at the range's end
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int j = 0; j < 4; ++j) part1[nt][j] = d[nt][j];
      }
    }
  }
  MDW_HEAD_TRACE(lane == 0, 8 + warp);
  __syncthreads();                                     // the hidden states are dead from here on
  MDW_HEAD_TRACE(threadIdx.x == 0, 2);

  // tiles cut between warps: every warp leaves its cut first / last tile's partial sums in
  // shared memory; the warp holding a cut tile's first unit adds the later warps' parts in
  // K order and finishes the tile
  const bool nonempty = u0 < u1;
  const int tF = u0 / NG, tL = nonempty ? (u1 - 1) / NG : tF;
  auto rec_at = [&](int w, int side, int nt) {
    return reinterpret_cast<float4*>(rec + ((size_t)((w * 2 + side) * NT + nt) * 32 + lane) * 4);
  };
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    *rec_at(warp, 0, nt) = make_float4(part0[nt][0], part0[nt][1], part0[nt][2], part0[nt][3]);
    *rec_at(warp, 1, nt) = make_float4(part1[nt][0], part1[nt][1], part1[nt][2], part1[nt][3]);
  }
  __syncthreads();
  MDW_HEAD_TRACE(threadIdx.x == 0, 20);
  if (nonempty && tL * NG >= u0 && (tL + 1) * NG > u1) {
    float d[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) d[nt][j] = (tL == tF) ? part0[nt][j] : part1[nt][j];
    for (int w2 = warp + 1; w2 < kWarps && ubeg(w2) < (tL + 1) * NG; ++w2) {
      if (ubeg(w2) == ubeg(w2 + 1)) continue;          // empty range
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float4 r = *rec_at(w2, 0, nt);           // tile tL is w2's first tile
        d[nt][0] += r.x; d[nt][1] += r.y; d[nt][2] += r.z; d[nt][3] += r.w;
      }
    }
    finish_tile(tL, d);
  }

  if (LISTS) {
    // block list of every token: the warps' lists, tree-merged
#pragma unroll
    for (int t = 0; t < (LISTS ? MAXM : 1); ++t)
      if (t < M) {
        lv[(t * kWarps + warp) * kMaxTK + lane] = lst[t].v;
        li[(t * kWarps + warp) * kMaxTK + lane] = lst[t].i;
      }
#ifdef MDW_TRACE
    __syncthreads();
    MDW_HEAD_TRACE(threadIdx.x == 0, 21);
#endif
    tree_merge(lv, li, M, warp, lane);
    MDW_HEAD_TRACE(threadIdx.x == 0, 22);
    for (int t = warp; t < M; t += kWarps)
      if (lane < tk) {
        const size_t o = ((size_t)blockIdx.x * M + t) * tk + lane;
        p.cand_val[o] = lv[t * kWarps * kMaxTK + lane];
        p.cand_idx[o] = li[t * kWarps * kMaxTK + lane];
      }
  } else {
    // the block's logits are written (and visible to the block after the barrier); warp w
    // walks the block's rows of tokens w, w + warps, ..., 32 rows per step and R steps of
    // loads in flight for all its tokens at once, and its list is the block list
    __syncthreads();
    MDW_HEAD_TRACE(threadIdx.x == 0, 21);
    constexpr int TPW = (MAXM + kWarps - 1) / kWarps;  // tokens per warp
    constexpr int R = 8;
    WarpList sel[TPW];
#pragma unroll
    for (int k = 0; k < TPW; ++k) list_init(sel[k]);
    for (long long vb = v0; vb < v1; vb += 32 * R) {
      float val[TPW][R];
#pragma unroll
      for (int k = 0; k < TPW; ++k) {
        const int t = warp + k * kWarps;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const long long v = vb + 32 * r + lane;
          val[k][r] = (t < M && v < v1) ? ld_cg_f32(p.logits + (size_t)t * p.V + v) : -INFINITY;
        }
      }
#pragma unroll
      for (int k = 0; k < TPW; ++k) {
        if (warp + k * kWarps >= M) break;               // warp-uniform
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const long long v = vb + 32 * r + lane;
          const float x = val[k][r] != val[k][r] ? -INFINITY : val[k][r];
          const int idx = (int)v;
          unsigned m = __ballot_sync(0xffffffffu, v < v1 && beats(x, idx, sel[k].thr_v, sel[k].thr_i));
          while (m) {
            const int src = __ffs(m) - 1;
            m &= m - 1;
            const float bv = __shfl_sync(0xffffffffu, x, src);
            const int bi = __shfl_sync(0xffffffffu, idx, src);
            list_insert(sel[k], bv, bi, tk, lane);
          }
        }
      }
    }
    MDW_HEAD_TRACE(threadIdx.x == 0, 22);
#pragma unroll
    for (int k = 0; k < TPW; ++k) {
      const int t = warp + k * kWarps;
      if (t < M && lane < tk) {
        const size_t o = ((size_t)blockIdx.x * M + t) * tk + lane;
        p.cand_val[o] = sel[k].v;
        p.cand_idx[o] = sel[k].i;
      }
    }
  }
  MDW_HEAD_TRACE(threadIdx.x == 0, 3);

  // the last block of each group of kHeadGroupSize blocks merges the group's lists; the last
  // group to finish merges the group lists into the result
  __threadfence();
  __syncthreads();
  const int grp = blockIdx.x / kHeadGroupSize;
  const int gfirst = grp * kHeadGroupSize;
  const int gn = min((int)G - gfirst, kHeadGroupSize);
  if (threadIdx.x == 0) is_last = (atomicAdd(p.hdr + kHdrHeadGroups + grp, 1u) == (uint32_t)(gn - 1));
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  MDW_HEAD_TRACE(threadIdx.x == 0, 4);
  merge_global_lists<MAXM>(p.cand_val, p.cand_idx, gfirst, gn, M, tk, lv, li, warp, lane);
  float* gcv = p.cand_val + (size_t)G * M * tk;
  int* gci = p.cand_idx + (size_t)G * M * tk;
  for (int t = warp; t < M; t += kWarps)
    if (lane < tk) {
      const size_t o = ((size_t)grp * M + t) * tk + lane;
      gcv[o] = lv[t * kWarps * kMaxTK + lane];
      gci[o] = li[t * kWarps * kMaxTK + lane];
    }
  __threadfence();
  __syncthreads();
  const int ngroups = (int)((G + kHeadGroupSize - 1) / kHeadGroupSize);
  if (threadIdx.x == 0) is_last = (atomicAdd(p.hdr + kHdrDoneCtr, 1u) == (uint32_t)(ngroups - 1));
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  MDW_HEAD_TRACE(threadIdx.x == 0, 5);
  merge_global_lists<MAXM>(gcv, gci, 0, ngroups, M, tk, lv, li, warp, lane);
  for (int t = warp; t < M; t += kWarps)
    if (lane < tk) {
      const float v = lv[t * kWarps * kMaxTK + lane];
      const int i = li[t * kWarps * kMaxTK + lane];
      if (lane == 0 && p.argmax_out) p.argmax_out[t] = i;
      if (p.topk_idx) p.topk_idx[(size_t)t * tk + lane] = i;
      if (p.topk_val) p.topk_val[(size_t)t * tk + lane] = v;
    }
  if (p.sample_u) {
    // the draw on the final top-k (one warp per token, candidates in shared memory)
    for (int t = warp; t < M; t += kWarps) {
      const float* cv = lv + t * kWarps * kMaxTK;
      const int* ci = li + t * kWarps * kMaxTK;
      const int32_t tok = sample_candidates_warp([&](int i) { return cv[i]; }, [&](int i) { return ci[i]; }, tk,
                                                 p.temperature, p.top_p, p.sample_u[t], lane);
      if (lane == 0) p.sample_out[t] = tok;
    }
  }
  MDW_HEAD_TRACE(threadIdx.x == 0, 6);
}

template <bool FP8, int MAXM>
cudaError_t launch_head_t(const HeadParams& p, cudaStream_t s) {
  const size_t smem = head_smem_bytes(p.M, MAXM, head_x_stride<FP8>());
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
  if (p.M > kHeadListM && !p.logits) return cudaErrorInvalidValue;   // it selects from its logits
  if (p.M <= 8) return launch_head_t<FP8, 8>(p, s);
  if (p.M <= 16) return launch_head_t<FP8, 16>(p, s);
  return launch_head_t<FP8, 32>(p, s);
}

}  // namespace

cudaError_t launch_head_fp8(const HeadParams& p, cudaStream_t s) { return launch_head_any<true>(p, s); }
cudaError_t launch_head_bf16(const HeadParams& p, cudaStream_t s) { return launch_head_any<false>(p, s); }

cudaError_t launch_quantize_head(const __nv_bfloat16* w, long long V, uint8_t* q, float* scale,
                                 cudaStream_t s) {
  const long long blocks = (V + 7) / 8;
  quantize_head_kernel<<<(unsigned)blocks, 256, 0, s>>>(w, V, q, scale);
  return cudaGetLastError();
}

}  // namespace mdw

#ifdef MDW_TRACE
extern "C" int mdw_head_trace_read(void* host, size_t bytes) {
  if (bytes > sizeof(mdw::g_head_trace)) bytes = sizeof(mdw::g_head_trace);
  return cudaMemcpyFromSymbol(host, mdw::g_head_trace, bytes) == cudaSuccess ? 0 : -1;
}
#endif
