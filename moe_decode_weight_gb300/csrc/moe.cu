// Persistent W4A8 MXFP4 MoE decode kernel: router, top-k, expert dedup, gate/up + SwiGLU,
// h quantisation, down projection and weighted combine, for one layer or a stack of
// layers with a pre-norm bf16 residual stream.
//
// Method (page titles and sections):
//   "Three MoE Inference Optimizations NVIDIA Measured on DGX Spark",
//   - "Decoding was memory-bound on a 124-billion-parameter model at batch size 1": each
//     MoE layer routes a token to 8 of 512 experts alongside one shared expert; decode is
//     bound by weight reads, so every kernel here is organised around streaming each
//     needed weight byte exactly once;
//   - "Humming MXFP4 kernels compile at run time for the model's real shapes": W4A8 MXFP4
//     experts, moe_intermediate 768; this kernel is specialised ahead of time on the
//     model's shapes (H 2560, I 768) in the same spirit;
//   - "Multi-token prediction turns each verification into four tokens": a window of M
//     tokens touches the union of their experts; each union member is read once and
//     applied to every token routed to it.
//
// Execution model (GB300, one block of 384 threads per SM, cooperative launch):
//   per layer, every block
//   P0  the weights of its router row are requested first; (stack) x = bf16(RMSNorm(r_l))
//       and (all) xq = E4M3(x / sx), computed redundantly by every block from the 5 KB/token
//       input (up to two tokens r_l arrives as tagged words the previous layer's blocks
//       published, above two it is read after the residual barrier B3);
//   P1  router logits for its slice of the E router rows, published as tagged words (value
//       and layer tag in one 8-byte word), so no barrier is needed before the top-k;
//   P2  top-k + dedup redundantly from the E x M logits, which the top-k warps poll (every
//       block derives the same slot / pair tables; slot 0 is the shared expert);
//   P3  gate/up for its contiguous share of the (slot, row-pair tile) space -- of the
//       (slot, tile, 8-token column group) space above 8 tokens -> h; arrive(B2); while
//       waiting: bulk L2 prefetch of its W2 rows of every slot and (stack) of the next
//       layer's router rows and shared-expert slice; wait(B2);
//   P4  every block quantises all pairs' h (amax / 448) into shared memory, then computes
//       its slice of output rows over all slots (no atomics: a fixed summation order);
//       (stack) r_{l+1} = bf16(r_l + y), up to two tokens also published as tagged words,
//       above two followed by B3.
//   The expert GEMVs run on m16n8k16 tensor-core MMAs: with up to four tokens the MMA
//   columns carry (token, K-block) pairs (block-column form, one or two tiles, scales applied
//   per column in fp32); with more tokens they carry tokens, the E8M0 scale folded into the
//   f16 weights when that is exact (token-column form); above 16 tokens the expert input is
//   kept in shared memory as E4M3 codes and widened to f16 at the fragment loads.
// Every inter-block wait is bounded and records MDW_ERR_TIMEOUT instead of hanging.
#include "mdw_device.cuh"
#include "mdw_internal.h"
#include "mdw_mma.cuh"

namespace mdw {
namespace {

constexpr int kRows13 = 2 * kI;                 // w13 rows per expert
constexpr int kW13RowBytes = kH / 2;            // 1280
constexpr int kW2RowBytes = kI / 2;             // 384
constexpr int kXhBytes = kH * 2 + 64;           // f16 x-hat per token, padded (conflict-free B loads)
constexpr int kXh8Bytes = kH + 32;              // E4M3 x-hat per token (M > 16), padded likewise
constexpr int kTablesBytes = 18432;             // shared memory reserved for the per-block tables
constexpr int kGuRound = 4 * kWarps;            // gate/up units per round (partials in smem)
constexpr int kGuMaxTiles = 320;                // list entries per block (gate/up above 8 tokens, down units)
constexpr int kMaxSegs = 48;                    // slot segments per block list (>= kPairChunk + 1)
constexpr int kTopkCand = 128;                  // compacted top-k candidates per warp
constexpr int kHhBytes = kI * 2 + 64;           // f16 h-hat per pair, padded (conflict-free A loads)
constexpr int kPairChunk = 36;                  // pairs quantised into smem at a time (all of M = 4)
constexpr int kTaggedResidM = 2;                // windows up to this size exchange r as tagged words
// per-warp cp.async rings (16-byte asynchronous copies into padded, bank-conflict-free rows)
constexpr int kGuU = 8;                         // gate/up: 32-blocks per stage
constexpr int kGuStages = 3;
constexpr int kGuPitch = kGuU * 16 + 16;        // bytes per staged row (16 rows per stage)
constexpr int kGuStageBytes = 16 * kGuPitch + 16 * kGuU;
constexpr int kDnStages = 2;                    // down: 16 W2 rows x 12 blocks per stage
constexpr int kDnKB = kIBlocks / 2;             // blocks per K half (12)
constexpr int kDnPitch = kDnKB * 16 + 16;       // 208 bytes: conflict-free fragment reads
constexpr int kDnBcPitch = kDnKB * 16;          // 192 bytes (= 64 mod 128): conflict-free 16-byte reads
constexpr int kDnStageBytes = 16 * kDnPitch + 16 * kIBlocks;
constexpr int kWarpRing = (kGuStages * kGuStageBytes > kDnStages * kDnStageBytes)
                              ? kGuStages * kGuStageBytes : kDnStages * kDnStageBytes;
// block-column form (M <= 4): unpadded 128-byte rows (swizzled chunks); the same depth as
// the token-column ring (4 or 5 stages measured no faster at M = 1 and 2-4 % slower at
// M = 2 and 4: the phase is not limited by the bytes a warp has in flight)
constexpr int kGuBcStages = 3;
constexpr int kGuBcStageBytes = 16 * kGuU * 16 + 16 * kGuU;
constexpr int kWarpRingBc = (kGuBcStages * kGuBcStageBytes > kDnStages * kDnStageBytes)
                                ? kGuBcStages * kGuBcStageBytes : kDnStages * kDnStageBytes;
__host__ __device__ constexpr int warp_ring_bytes(int M) { return M <= 4 ? kWarpRingBc : kWarpRing; }
constexpr int kMaxRowsPerBlock = 32;            // down-projection rows per block (>= H / grid)

// ------------------------------------------------------------------ phase trace

constexpr int kTraceNone = -1;

// Built only with -DMDW_TRACE (a profiling build of the library, never the product build):
// thread 0 of every block records %globaltimer at each phase boundary of every layer.
#ifdef MDW_TRACE
constexpr int kTracePhases = 24;
constexpr int kTraceLayers = 64;
__device__ unsigned long long g_trace[kTraceLayers * kTracePhases * 256];
#define MDW_TRACE_POINT(layer, phase)                                                        \
  do {                                                                                       \
    if (threadIdx.x == 0 && (layer) >= 0 && (layer) < kTraceLayers && blockIdx.x < 256) {                    \
      unsigned long long t_;                                                                 \
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                                 \
      g_trace[((layer) * kTracePhases + (phase)) * 256 + blockIdx.x] = t_;                   \
    }                                                                                        \
  } while (0)
#else
#define MDW_TRACE_POINT(layer, phase) do { } while (0)
#endif

// Shared-memory carve-up (bytes), for M tokens.
struct Smem {
  size_t xh, xb, hh, ring, part, yacc, gured, small, total;
};
// R1 = x-hat (gate/up) or h-hat (down); R2 = bf16 x (router) or the per-warp cp.async rings.
// Up to 16 tokens the x-hat is f16; beyond, it is kept as E4M3 codes (decoded to f16 at the
// fragment loads) and the router's bf16 x spans R1 and R2 until the codes replace it.
__host__ __device__ inline Smem smem_layout(int M) {
  Smem s;
  const size_t rings = (size_t)kWarps * warp_ring_bytes(M);
  const size_t hh = (size_t)kPairChunk * kHhBytes;
  s.xh = 0;
  s.hh = 0;
  if (M > 16) {
    const size_t r1 = (size_t)M * kXh8Bytes > hh ? (size_t)M * kXh8Bytes : hh;
    s.xb = 0;
    s.ring = (r1 + 127) & ~(size_t)127;
    const size_t end = s.ring + rings > (size_t)M * kH * 2 ? s.ring + rings : (size_t)M * kH * 2;
    s.part = (end + 15) & ~(size_t)15;
  } else {
    const size_t r1 = (size_t)M * kXhBytes > hh ? (size_t)M * kXhBytes : hh;
    const size_t r2 = (size_t)M * kH * 2 > rings ? (size_t)M * kH * 2 : rings;
    s.xb = (r1 + 127) & ~(size_t)127;
    s.ring = s.xb;
    s.part = (s.xb + r2 + 15) & ~(size_t)15;                    // [kPairChunk][rows] fp32
  }
  s.yacc = s.part + (size_t)kPairChunk * kMaxRowsPerBlock * 4;     // [M][rows] fp32
  s.gured = s.yacc + (size_t)M * kMaxRowsPerBlock * 4;               // [kGuRound][32][4] fp32
  s.small = s.gured + (size_t)kGuRound * 32 * 4 * 4;   // also holds the routing candidates
  s.total = s.small + kTablesBytes;
  return s;
}

// Small per-block tables in shared memory.
struct Tables {
  int ids[MDW_MAX_M * MDW_MAX_TOPK];
  float gts[MDW_MAX_M * MDW_MAX_TOPK];
  uint32_t bitmap[MDW_MAX_EXPERTS / 32];
  int slot_expert[MDW_MAX_M * MDW_MAX_TOPK + 1];
  int slot_begin[MDW_MAX_M * MDW_MAX_TOPK + 2];
  int pair_token[kMaxPairsCap];
  int pair_slot[kMaxPairsCap];
  float pair_gate[kMaxPairsCap];
  int wpre[MDW_MAX_EXPERTS / 32];
  int cnt[MDW_MAX_M * MDW_MAX_TOPK + 1];
  float sx[MDW_MAX_M];
  float inv_rms[MDW_MAX_M];
  float part[MDW_MAX_M * (kH / 256)];          // per-(token, 32-chunk group) partials
  float cand_g[MDW_MAX_M * MDW_MAX_TOPK];      // gates before they replace the logits
  float sh[kPairChunk];
  int n_slots, n_routed, n_pairs, shared_slot, bad;
  int gu_n;                                    // entries in gu_tile
  int n_segs;                                  // slot segments of the current down pair chunk
  int seg_slot[kMaxSegs], seg_lo[kMaxSegs], seg_groups[kMaxSegs], seg_off[kMaxSegs + 1];
  int4 gu_tile[kGuMaxTiles];                   // gate/up above 8 tokens: (slot, j0, rows, first token
                                               // column); down: (slot, tile, K half, first pair)
};
static_assert(sizeof(Tables) <= kTablesBytes, "tables exceed the reserved shared memory");

// ------------------------------------------------------------------ P0: input / act quant

// r_l of the stack: r_0 is the caller's input; r_1.. live in the residual buffers.
__device__ __forceinline__ const __nv_bfloat16* resid_ptr(const MoeParams& p, int l) {
  if (l == 0) return p.r0;
  const int slot = p.resid_pingpong ? (l & 1) : l;
  return p.resid + (size_t)slot * p.M * kH;
}

// x-hat layout: token t's f16 values in natural order at byte t*kXhBytes (+64 B padding per
// token, so the 8 token rows of an MMA B fragment fall in distinct banks).
template <int MAXM>
__device__ void prepare_input(const MoeParams& p, int layer, uint8_t* smem, Tables& tb) {
  const int M = p.M;
  constexpr int CPT = kH / 8;                 // 16-byte chunks per token (320, a multiple of 32)
  __nv_bfloat16* xb = reinterpret_cast<__nv_bfloat16*>(smem + smem_layout(M).xb);
  uint4* xb4 = reinterpret_cast<uint4*>(xb);
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) tb.bad = 0;
  // windows of up to kTaggedResidM tokens take r_l from tagged words; larger ones (whose
  // staging would not fit the register budget) read the residual buffer after a barrier
  const bool poll = MAXM <= kTaggedResidM && p.stack_mode && layer > 0;
  if (poll) {
    // r_l from the other blocks' tagged words (tag l): every word of this thread's chunks is
    // requested before any is checked; the missing ones are requested again together
    constexpr int NCH = (MAXM * CPT + kThreads - 1) / kThreads;
    const uint32_t tag = (uint32_t)layer;
    uint32_t want = 0;
#pragma unroll
    for (int k = 0; k < NCH; ++k)
      if ((int)threadIdx.x + k * kThreads < M * CPT) want |= 1u << k;
    long long t0 = 0;
    for (int n = 0; want != 0; ++n) {
      uint64_t w[NCH][4];
#pragma unroll
      for (int k = 0; k < NCH; ++k) {
        const size_t c = threadIdx.x + (size_t)k * kThreads;
        if (want & (1u << k)) {
          ld_word2(p.xr + 4 * c, w[k][0], w[k][1]);
          ld_word2(p.xr + 4 * c + 2, w[k][2], w[k][3]);
        }
      }
      uint32_t got = 0;
#pragma unroll
      for (int k = 0; k < NCH; ++k) {
        if ((want & (1u << k)) && tag_of(w[k][0]) == tag && tag_of(w[k][1]) == tag && tag_of(w[k][2]) == tag &&
            tag_of(w[k][3]) == tag) {
          xb4[threadIdx.x + k * kThreads] = make_uint4((uint32_t)w[k][0], (uint32_t)w[k][1], (uint32_t)w[k][2], (uint32_t)w[k][3]);
          got |= 1u << k;
        }
      }
      want &= ~got;
      if (want == 0) break;
      if (n == 0) t0 = clock64();
      if ((n & 15) == 15 && ld_volatile_u32(p.hdr + kHdrStatus) != 0) { atomicExch(&tb.bad, 2); break; }
      if (clock64() - t0 > p.spin_budget) { set_status(p.hdr, MDW_ERR_TIMEOUT); atomicExch(&tb.bad, 2); break; }
    }
    __syncthreads();
  }
  MDW_TRACE_POINT(layer, 12);
  const uint4* src = reinterpret_cast<const uint4*>(!p.stack_mode ? p.x_in : resid_ptr(p, layer));
  // Every block must derive bit-identical x and xq: per-token reductions are taken in a fixed
  // order (a warp's 32 chunks share one token; the 10 warp partials are summed in order).
  // 1. load (all threads, one 16-byte chunk each); stack: sum of squares, else: amax
  for (int c = threadIdx.x; c < M * CPT; c += blockDim.x) {
    const uint4 v = poll ? xb4[c] : ld_cg16(src + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float r = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float a = __uint_as_float(w[k] << 16), b = __uint_as_float(w[k] & 0xFFFF0000u);
      if (p.stack_mode) { r = fmaf(a, a, r); r = fmaf(b, b, r); }
      else r = fmaxf(r, fmaxf(fabsf(a), fabsf(b)));
    }
    r = p.stack_mode ? warp_sum(r) : warp_max(r);
    if (lane == 0) tb.part[c / 32] = r;
    xb4[c] = v;
  }
  __syncthreads();
  // up to 4 tokens (at most 4 chunks per thread) every thread derives a token's 1/rms and
  // scale itself from the warps' partials, in the same order as the one thread would, instead
  // of one thread per token and a block barrier after it; the amax partials then go to a
  // second array so no partial is overwritten while another warp may still read it
  constexpr bool kSelf = MAXM <= 4;
  float* part_am = tb.part + (kSelf && p.stack_mode ? MAXM * (CPT / 32) : 0);
  auto token_inv = [&](int t) {
    float ss = 0.f;
    for (int g = 0; g < CPT / 32; ++g) ss += tb.part[t * (CPT / 32) + g];
    return rsqrtf(ss / (float)kH + 1e-6f);
  };
  auto token_scale = [&](int t) {
    float am = 0.f;
    for (int g = 0; g < CPT / 32; ++g) am = fmaxf(am, part_am[t * (CPT / 32) + g]);
    return am > 0.f ? __fdiv_rn(am, kE4M3Max) : 1.0f;
  };
  if (p.stack_mode) {
    // 2. x = bf16(r * rsqrt(mean(r^2) + eps)), then its amax
    if (!kSelf) {
      if (threadIdx.x < M) tb.inv_rms[threadIdx.x] = token_inv(threadIdx.x);
      __syncthreads();
    }
    for (int c = threadIdx.x; c < M * CPT; c += blockDim.x) {
      const float inv = kSelf ? token_inv(c / CPT) : tb.inv_rms[c / CPT];
      const uint4 v = xb4[c];
      uint32_t w[4] = {v.x, v.y, v.z, v.w};
      float am = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 r2 = __floats2bfloat162_rn(__uint_as_float(w[k] << 16) * inv,
                                                        __uint_as_float(w[k] & 0xFFFF0000u) * inv);
        w[k] = *reinterpret_cast<const uint32_t*>(&r2);
        am = fmaxf(am, fmaxf(fabsf(__uint_as_float(w[k] << 16)), fabsf(__uint_as_float(w[k] & 0xFFFF0000u))));
      }
      am = warp_max(am);
      if (lane == 0) part_am[c / 32] = am;
      xb4[c] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncthreads();
  }
  // 3. per-token scale = amax/448 (IEEE division), then codes: x/scale correctly rounded,
  //    round-to-nearest-even saturating conversion; x-hat (f16) into the planes layout
  if (!kSelf) {
    if (threadIdx.x < M) {
      const float sc = token_scale(threadIdx.x);
      tb.sx[threadIdx.x] = sc;
      if (blockIdx.x == 0) p.sx[threadIdx.x] = sc;
    }
    __syncthreads();
  }
  if (MAXM > 16) return;                          // codes written after the router (xhat_codes_in_place)
  const bool writer = (blockIdx.x == 0);
  for (int c = threadIdx.x; c < M * CPT; c += blockDim.x) {
    const int t = c / CPT, i = c % CPT;           // chunk i = elements 8i .. 8i+7 of token t
    float sc;
    if (kSelf) {
      sc = token_scale(t);
      if (i == 0) {                               // one writer per token (read after the last barrier)
        tb.sx[t] = sc;
        if (blockIdx.x == 0) p.sx[t] = sc;
      }
    } else {
      sc = tb.sx[t];
    }
    const uint4 v = xb4[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t q[4], h[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      q[k] = f32x2_to_e4m3x2(__fdiv_rn(__uint_as_float(w[k] << 16), sc),
                             __fdiv_rn(__uint_as_float(w[k] & 0xFFFF0000u), sc));
      h[k] = e4m3x2_to_f16x2(q[k]);
    }
    *reinterpret_cast<uint4*>(smem + (size_t)t * kXhBytes + (size_t)i * 16) = make_uint4(h[0], h[1], h[2], h[3]);
    if (writer)
      reinterpret_cast<uint2*>(p.xq + (size_t)t * kH)[i] = make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
  }
  __syncthreads();
}

// E4M3 x-hat of more than 16 tokens, once the router has read the bf16 x: token t's codes
// (the same quotients and rounding as above) move from its bf16 row at byte t * 2H to byte
// t * kXh8Bytes. Groups of 6 tokens, 5 chunks per thread: a group's rows are all read into
// registers before any of its codes is written, and a group's codes end below the first byte
// of the next group's rows, so no row is overwritten before it is read.
__device__ void xhat_codes_in_place(const MoeParams& p, uint8_t* smem, const Tables& tb) {
  constexpr int CPT = kH / 8;                     // 8-value chunks per token
  constexpr int GT = 6;                           // tokens per group
  constexpr int CH = GT * CPT / kThreads;         // chunks per thread per group
  static_assert(GT * CPT % kThreads == 0, "a group must give every thread the same chunk count");
  static_assert(kXh8Bytes <= 2 * kH, "codes must not pass the rows they replace");
  const int M = p.M;
  const uint4* xb4 = reinterpret_cast<const uint4*>(smem + smem_layout(M).xb);
  const bool writer = (blockIdx.x == 0);
  for (int t0 = 0; t0 < M; t0 += GT) {
    uint4 v[CH];
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      const int c = t0 * CPT + (int)threadIdx.x + j * kThreads;
      v[j] = c < M * CPT ? xb4[c] : make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      const int c = t0 * CPT + (int)threadIdx.x + j * kThreads;
      if (c >= M * CPT) continue;
      const int t = c / CPT, i = c % CPT;
      const float sc = tb.sx[t];
      const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
      uint32_t q[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        q[k] = f32x2_to_e4m3x2(__fdiv_rn(__uint_as_float(w[k] << 16), sc),
                               __fdiv_rn(__uint_as_float(w[k] & 0xFFFF0000u), sc));
      const uint2 codes = make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
      *reinterpret_cast<uint2*>(smem + smem_layout(M).xh + (size_t)t * kXh8Bytes + (size_t)i * 8) = codes;
      if (writer) reinterpret_cast<uint2*>(p.xq + (size_t)t * kH)[i] = codes;
    }
  }
  __syncthreads();
}

// ------------------------------------------------------------------ P1: router rows

// The block's router rows [e0, e1): warp w takes rows e0 + w, e0 + w + warps, ...; the first
// row's weights are loaded (into `wv`) before the input is ready, by load_router_row.
__device__ __forceinline__ void router_range(const MoeParams& p, int& e0, int& e1) {
  const int G = gridDim.x;
  e0 = (int)((long long)blockIdx.x * p.E / G);
  e1 = (int)((long long)(blockIdx.x + 1) * p.E / G);
}
__device__ __forceinline__ void load_router_row(const LayerDesc& L, int e, uint4 (&wv)[10]) {
  const uint4* wr = reinterpret_cast<const uint4*>(L.router_w + (size_t)e * kH);
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 10; ++i) wv[i] = ldg_stream16(wr + 32 * i + lane);
}
__device__ void router_rows(const MoeParams& p, const LayerDesc& L, const uint8_t* smem, uint4 (&wv)[10], int layer) {
  const int M = p.M, E = p.E;
  int e0, e1;
  router_range(p, e0, e1);
  const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(smem + smem_layout(M).xb);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = e0 + warp; e < e1; e += kWarps) {
    if (e != e0 + warp) load_router_row(L, e, wv);
    for (int t = 0; t < M; ++t) {
      const uint4* x4 = reinterpret_cast<const uint4*>(xb + (size_t)t * kH);
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 10; ++i) {
        uint4 xv = x4[32 * i + lane];
        const uint32_t a[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
        const uint32_t b[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc = fmaf(__uint_as_float(a[k] << 16), __uint_as_float(b[k] << 16), acc);
          acc = fmaf(__uint_as_float(a[k] & 0xFFFF0000u), __uint_as_float(b[k] & 0xFFFF0000u), acc);
        }
      }
      acc = warp_sum(acc);
      if (lane == 0) {
        st_word(p.xz + (size_t)t * E + e, tagged(__float_as_uint(acc), (uint32_t)layer + 1));
        p.logits[(size_t)t * E + e] = acc;          // inspection copy
      }
    }
  }
}

// ------------------------------------------------------------------ P2: top-k + dedup

// Block 0 publishes the routing of the layer (inspection and the optional outputs).
__device__ void publish_routing(const MoeParams& p, const Tables& tb, int layer) {
  const int M = p.M, K = p.K;
  for (int i = threadIdx.x; i < M * K; i += blockDim.x) {
    p.ids[i] = tb.ids[i];
    p.gates[i] = tb.gts[i];
    if (p.ids_out) p.ids_out[i] = tb.ids[i];
    if (p.gates_out) p.gates_out[i] = tb.gts[i];
  }
  for (int s = threadIdx.x; s < tb.n_slots; s += blockDim.x) p.slot_expert[s] = tb.slot_expert[s];
  for (int q = threadIdx.x; q < tb.n_pairs; q += blockDim.x) {
    p.pair_token[q] = tb.pair_token[q];
    p.pair_slot[q] = tb.pair_slot[q];
    p.pair_gate[q] = tb.pair_gate[q];
  }
  if (threadIdx.x == 0) {
    p.hdr[kHdrSlots] = tb.n_slots;
    p.hdr[kHdrPairs] = tb.n_pairs;
    p.hdr[kHdrRouted] = tb.n_routed;
    if (layer < kHdrWords - kHdrUnions) p.hdr[kHdrUnions + layer] = tb.n_routed;
  }
}

// Routing tables of one token (M == 1), by warp 0 in registers: the gates (softmax of the K
// selected logits, the same K-lane butterflies as the general tables), the union (the K
// distinct ids ascending, slots first..first+K-1) and one pair per slot.
__device__ void routing_tables_one(Tables& tb, int K, int first, int lane) {
  const bool act = lane < K;
  const int id = act ? tb.ids[lane] : 0x7fffffff;
  const float z = act ? tb.gts[lane] : 0.f;
  float gate;
  if ((K & (K - 1)) == 0) {
    float mx = z;
    for (int o = 1; o < K; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float ez = expf(z - mx);
    float sum = ez;
    for (int o = 1; o < K; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    gate = ez / sum;
  } else {
    float mx = tb.gts[0];
    for (int r = 1; r < K; ++r) mx = fmaxf(mx, tb.gts[r]);
    float sum = 0.f;
    for (int r = 0; r < K; ++r) sum += expf(tb.gts[r] - mx);
    gate = act ? expf(z - mx) / sum : 0.f;
  }
  int rank = 0;
  for (int j = 0; j < K; ++j) rank += (__shfl_sync(0xffffffffu, id, j) < id);
  __syncwarp();
  const int S = K + first;
  if (act) {
    const int slot = first + rank;
    tb.slot_expert[slot] = id;
    tb.pair_token[slot] = 0;
    tb.pair_slot[slot] = slot;
    tb.pair_gate[slot] = gate;
    tb.gts[lane] = gate;
  }
  for (int sidx = lane; sidx <= S; sidx += 32) tb.slot_begin[sidx] = sidx;
  if (lane == 0) {
    if (first) { tb.slot_expert[0] = -1; tb.pair_token[0] = 0; tb.pair_slot[0] = 0; tb.pair_gate[0] = 1.0f; }
    tb.n_routed = K;
    tb.n_slots = S;
    tb.n_pairs = S;
    tb.shared_slot = first ? 0 : -1;
  }
}

// Token t's E router logits (tag layer + 1) into v[] (v[j] = logit of expert lane + 32 j), every
// word requested before any is checked; false (MDW_ERR_TIMEOUT recorded, or another block's
// failure seen) when the bounded wait runs out. Warp-collective.
__device__ bool poll_logits(const MoeParams& p, int t, int layer, float (&v)[MDW_MAX_EXPERTS / 32]) {
  constexpr int PER = MDW_MAX_EXPERTS / 32;
  const int lane = threadIdx.x & 31, E = p.E;
  const uint32_t tag = (uint32_t)layer + 1;
  const uint64_t* z = p.xz + (size_t)t * E;
  uint32_t want = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    v[j] = -INFINITY;
    if (lane + 32 * j < E) want |= 1u << j;
  }
  long long t0 = 0;
  for (int n = 0;; ++n) {
    uint64_t w[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) w[j] = (want & (1u << j)) ? ld_word(z + lane + 32 * j) : 0;
    uint32_t got = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j)
      if ((want & (1u << j)) && tag_of(w[j]) == tag) { v[j] = __uint_as_float((uint32_t)w[j]); got |= 1u << j; }
    want &= ~got;
    if (!__any_sync(0xffffffffu, want != 0)) return true;
    if (n == 0) t0 = clock64();
    bool bad = (n & 15) == 15 && ld_volatile_u32(p.hdr + kHdrStatus) != 0;
    if (clock64() - t0 > p.spin_budget) { if (lane == 0) set_status(p.hdr, MDW_ERR_TIMEOUT); bad = true; }
    if (__any_sync(0xffffffffu, bad)) return false;
  }
}

__device__ void route_tokens(const MoeParams& p, const LayerDesc& L, Tables& tb, int layer, uint8_t* scratch) {
  const int M = p.M, E = p.E, K = p.K;
  // per-warp candidate buffers live in the gate/up partial-sum region (not live during
  // routing)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  MDW_TRACE_POINT(layer, 3);                      // (re-stamped below by the top-k warp 0)
  MDW_TRACE_POINT(layer, 4);
  if (p.topk_override) {
    // imposed routing: [M][K] for one layer, [L][M][K] for the stack
    const int32_t* ov = p.topk_override + (p.stack_mode ? (size_t)layer * M * K : 0);
    for (int t = warp; t < M; t += kWarps) {
      if (lane < K) {
        int id = ov[t * K + lane];
        bool ok = id >= 0 && id < E;
        for (int j = 0; j < K; ++j)
          if (j != lane && ov[t * K + j] == id) ok = false;
        if (!ok) { atomicExch(&tb.bad, 1); id = 0; }
        tb.ids[t * K + lane] = id;
      }
      // the imposed ids' logits: each lane polls its own word
      const uint32_t tag = (uint32_t)layer + 1;
      const uint64_t* z = p.xz + (size_t)t * E + (lane < K ? tb.ids[t * K + lane] : 0);
      bool have = lane >= K;
      uint64_t w = 0;
      const long long t0 = clock64();
      for (int n = 0; !__all_sync(0xffffffffu, have); ++n) {
        if (!have) { w = ld_word(z); have = tag_of(w) == tag; }
        bool bad = (n & 15) == 15 && ld_volatile_u32(p.hdr + kHdrStatus) != 0;
        if (clock64() - t0 > p.spin_budget) { if (lane == 0) set_status(p.hdr, MDW_ERR_TIMEOUT); bad = true; }
        if (__any_sync(0xffffffffu, bad)) { if (lane == 0) atomicExch(&tb.bad, 2); break; }
      }
      if (lane < K) tb.gts[t * K + lane] = __uint_as_float((uint32_t)w);
    }
  } else {
    // Top-K per token, one warp per token (ties -> lower expert id):
    //  1. each lane holds E/32 logits and its local best;
    //  2. a bitonic sort of the 32 lane bests across the warp; T = the K-th of them. K
    //     distinct logits are not worse than T, so T bounds the K-th largest from below;
    //  3. the logits not worse than T (typically little more than K) are compacted into
    //     shared memory and ranked among themselves; rank < K gives the result in order.
    float* cv_all = reinterpret_cast<float*>(scratch);
    int* ci_all = reinterpret_cast<int*>(cv_all + kWarps * kTopkCand);
    int* cnt_all = ci_all + kWarps * kTopkCand;
    for (int t = warp; t < M; t += kWarps) {
      constexpr int PER = MDW_MAX_EXPERTS / 32;
      float v[PER];
      if (!poll_logits(p, t, layer, v)) { if (lane == 0) atomicExch(&tb.bad, 2); break; }
      MDW_TRACE_POINT(layer, 3);
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        const int e = lane + 32 * j;
        if (v[j] != v[j]) v[j] = -INFINITY;            // a NaN logit ranks last (ids stay valid)
        if (e < E && beats(v[j], e, bv, bi)) { bv = v[j]; bi = e; }
      }
      // bitonic sort of (bv, bi), descending in `beats` order
#pragma unroll
      for (int kk = 2; kk <= 32; kk <<= 1)
#pragma unroll
        for (int jj = kk >> 1; jj > 0; jj >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, jj);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, jj);
          const bool up = ((lane & kk) == 0);              // this pair sorts descending
          const bool lower = ((lane & jj) == 0);
          const bool take_better = (up == lower);
          const bool o_better = beats(ov, oi, bv, bi);
          if (take_better ? o_better : !o_better && !(ov == bv && oi == bi)) { bv = ov; bi = oi; }
        }
      const float tv = __shfl_sync(0xffffffffu, bv, K - 1);
      const int ti = __shfl_sync(0xffffffffu, bi, K - 1);
      MDW_TRACE_POINT(layer, 4);
      float* cv = cv_all + warp * kTopkCand;
      int* ci = ci_all + warp * kTopkCand;
      int count = 0;
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        const int e = lane + 32 * j;
        const bool keep = e < E && !beats(tv, ti, v[j], e);
        const unsigned m = __ballot_sync(0xffffffffu, keep);
        const int pos = count + __popc(m & ((1u << lane) - 1u));
        if (keep && pos < kTopkCand) { cv[pos] = v[j]; ci[pos] = e; }
        count += __popc(m);
      }
      __syncwarp();
      if (lane == 0) cnt_all[warp] = count;
      if (count <= kTopkCand) {
        for (int k = lane; k < count; k += 32) {
          const float vv = cv[k];
          const int ii = ci[k];
          int rank = 0;
          for (int o = 0; o < count; ++o) rank += beats(cv[o], ci[o], vv, ii);
          if (rank < K) { tb.ids[t * K + rank] = ii; tb.gts[t * K + rank] = vv; }
        }
      } else {
        // many equal logits: K rounds of warp arg-max over the register-held logits
        float pv = INFINITY;
        int pi = -1;
        for (int r = 0; r < K; ++r) {
          float best = -INFINITY;
          int bidx = 0x7fffffff;
#pragma unroll
          for (int j = 0; j < PER; ++j) {
            const int e = lane + 32 * j;
            if (e < E && beats(pv, pi, v[j], e) && beats(v[j], e, best, bidx)) { best = v[j]; bidx = e; }
          }
          warp_argmax(best, bidx);
          pv = best; pi = bidx;
          if (lane == 0) { tb.ids[t * K + r] = bidx; tb.gts[t * K + r] = best; }
        }
      }
      __syncwarp();
    }
  }
  const int first = p.has_shared ? 1 : 0;
  if (M == 1) {
    // one token: warp 0 selected it and builds the tables in registers, no block barrier
    if (warp == 0) {
      __syncwarp();
      if (!tb.bad) routing_tables_one(tb, K, first, lane);
    }
    __syncthreads();
    MDW_TRACE_POINT(layer, 10);
    MDW_TRACE_POINT(layer, 20);
    MDW_TRACE_POINT(layer, 21);
    MDW_TRACE_POINT(layer, 11);
    MDW_TRACE_POINT(layer, 22);
    if (tb.bad) return;
    if (blockIdx.x == 0) publish_routing(p, tb, layer);
    return;
  }
  __syncthreads();
  MDW_TRACE_POINT(layer, 10);
  if (tb.bad) return;
  // Routing tables (warp 0): gates, the union of the selections and its slots (slot 0 = shared
  // expert when present, then the union ascending); then the pairs (slot-major,
  // token-minor).
  auto slot_of = [&](int e) {
    return first + tb.wpre[e >> 5] + __popc(tb.bitmap[e >> 5] & ((1u << (e & 31)) - 1u));
  };
  if (warp == 0) {
    // gates: softmax over each token's K selected logits, one (token, rank) per lane
    const bool pow2 = (K & (K - 1)) == 0;             // then a token's K entries share K aligned lanes
    for (int i0 = 0; i0 < M * K; i0 += 32) {
      const int i = i0 + lane;
      const bool act = i < M * K;
      float gate = 0.f;
      if (pow2) {
        const float z = act ? tb.gts[i] : 0.f;
        float mx = z;
        for (int o = 1; o < K; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float ez = expf(z - mx);
        float sum = ez;
        for (int o = 1; o < K; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        gate = ez / sum;
      } else if (act) {
        const float* z = tb.gts + (i / K) * K;
        float mx = z[0];
        for (int r = 1; r < K; ++r) mx = fmaxf(mx, z[r]);
        float sum = 0.f;
        for (int r = 0; r < K; ++r) sum += expf(z[r] - mx);
        gate = expf(z[i % K] - mx) / sum;
      }
      if (act) tb.cand_g[i] = gate;
    }
    MDW_TRACE_POINT(layer, 20);
    if (lane < MDW_MAX_EXPERTS / 32) tb.bitmap[lane] = 0;
    __syncwarp();
    for (int i = lane; i < M * K; i += 32) {
      tb.gts[i] = tb.cand_g[i];
      atomicOr(&tb.bitmap[tb.ids[i] >> 5], 1u << (tb.ids[i] & 31));
    }
    __syncwarp();
    const uint32_t word = lane < MDW_MAX_EXPERTS / 32 ? tb.bitmap[lane] : 0u;
    const int cnt = __popc(word);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int nb = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += nb;
    }
    if (lane < MDW_MAX_EXPERTS / 32) tb.wpre[lane] = incl - cnt;
    MDW_TRACE_POINT(layer, 21);
    int pos = first + incl - cnt;
    for (uint32_t w = word; w; w &= w - 1) {
      tb.cnt[pos] = 0;                                  // token masks of the routed slots
      tb.slot_expert[pos++] = lane * 32 + __ffs(w) - 1;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == 0) {
      tb.n_routed = total;
      tb.n_slots = total + first;
      tb.shared_slot = p.has_shared ? 0 : -1;
      if (p.has_shared) tb.slot_expert[0] = -1;
    }
  }
  MDW_TRACE_POINT(layer, 11);
  if (warp == 0) {
    __syncwarp();
    const int S = tb.n_slots;
    // token masks of the routed slots -> counts -> slot_begin (scan) -> pair positions: the
    // pairs of a slot are token-ordered, so a pair's rank is the number of the slot's earlier
    // tokens, popc(mask & ((1 << t) - 1))
    for (int i = lane; i < M * K; i += 32) atomicOr(reinterpret_cast<unsigned*>(&tb.cnt[slot_of(tb.ids[i])]), 1u << (i / K));
    __syncwarp();
    int carry = 0;
    for (int b0 = 0; b0 < S; b0 += 32) {
      const int sidx = b0 + lane;
      const int c = sidx < S ? (sidx < first ? M : __popc((unsigned)tb.cnt[sidx])) : 0;
      int in2 = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int nb = __shfl_up_sync(0xffffffffu, in2, o);
        if (lane >= o) in2 += nb;
      }
      if (sidx < S) tb.slot_begin[sidx] = carry + in2 - c;
      carry += __shfl_sync(0xffffffffu, in2, 31);
    }
    if (lane == 0) { tb.slot_begin[S] = carry; tb.n_pairs = carry; }
    __syncwarp();
    for (int i = lane; i < M * K; i += 32) {
      const int t = i / K, sidx = slot_of(tb.ids[i]);
      const int q = tb.slot_begin[sidx] + __popc((unsigned)tb.cnt[sidx] & ((1u << t) - 1u));
      tb.pair_token[q] = t;
      tb.pair_slot[q] = sidx;
      tb.pair_gate[q] = tb.gts[i];
    }
    if (p.has_shared)
      for (int t = lane; t < M; t += 32) { tb.pair_token[t] = t; tb.pair_slot[t] = 0; tb.pair_gate[t] = 1.0f; }
  }
  MDW_TRACE_POINT(layer, 22);
  __syncthreads();
  if (blockIdx.x == 0) publish_routing(p, tb, layer);
}

// ------------------------------------------------------------------ P3: gate/up + SwiGLU

// One gate/up unit: MMA rows 0..7 = gate rows j0..j0+7 and rows 8..15 = the matching up rows
// of one expert; columns = 8 tokens of the slot (xtok = this lane's token's x-hat, or null);
// K = spu stages of kGuU blocks of 32 from block kb0.
struct GuUnit {
  const uint8_t* q13;
  const uint8_t* s13;
  const uint8_t* xtok;
  const uint8_t* xtok2;       // block-column form with two tiles: the lane's token of tile 1
  int j0, nr, kb0;
};

// A warp's n gate/up units as one continuous pipeline: the weight rows of every stage stream
// through the warp's cp.async ring (STAGES stages of kGuU blocks x 16 rows, rows padded so
// the fragment reads are bank-conflict free), the next unit's stages being requested while
// the current one is computed. Each 32-block is two k16 MMAs on a permuted K order: lane
// (g, q) feeds bytes 4q..4q+3 of the block (E2M1 pairs, via cvt.e2m1x2) as its A registers
// and the matching x-hat values 8q..8q+7 (one 16-byte load of f16 values, or above 16 tokens
// one 8-byte load of E4M3 codes widened to f16) as its B registers. When every
// E8M0 scale of a stage keeps E2M1 x 2^(s-127) exact in f16, the scale is multiplied into the
// f16 weights and the MMAs accumulate straight into fp32 (even and odd blocks in two
// accumulators); otherwise each block's fresh fp32 result is scaled in fp32 and added. At the
// end of unit j, done(j, acc) receives
//   acc[0..1] = gate rows g, tokens 2q..2q+1;  acc[2..3] = up rows g, same tokens.
template <int BCN, bool X8, typename Info, typename Done>
__device__ __forceinline__ void gate_up_units(int n, int spu, Info info, Done done, uint8_t* ring, int lane) {
  constexpr bool BC = BCN > 0;                 // block-column form with BCN tiles, else token columns
  constexpr int NT = BC ? BCN : 1;
  constexpr int STAGES = BC ? kGuBcStages : kGuStages;
  constexpr int SBYTES = BC ? kGuBcStageBytes : kGuStageBytes;
  const int g = lane >> 2, q = lane & 3;
  const int total = n * spu;
  // unit descriptors held in registers: the one being requested and the one being computed
  GuUnit Ui, Uc;
  int ji = -1, jc = -1;
  // stage counters instead of divisions by spu: the issue side is at stage `is` of unit ji,
  // the compute side at stage `cs` of unit jc
  int is = 0, cs = 0;
  auto issue = [&](int st) {
    if (is == 0) { ++ji; Ui = info(ji); }
    const GuUnit& U = Ui;
    uint8_t* dst = ring + (st % STAGES) * SBYTES;
    const int bb = U.kb0 + is * kGuU;
    if (++is == spu) is = 0;
    // token-column layout: rows of kGuPitch bytes (padded for the 4-byte fragment reads);
    // block-column layout: rows of 128 bytes, chunk b of row r at b ^ 4 (r & 1), so the
    // 16-byte reads of lanes (g, q) (rows g, chunks sb + q) hit distinct banks
    constexpr int pitch = BC ? kGuU * 16 : kGuPitch;
#pragma unroll
    for (int k = 0; k < 16 * kGuU / 32; ++k) {        // 16 rows x kGuU chunks of 16 bytes
      const int c = lane + 32 * k, row = c / kGuU, blk = c % kGuU, rr = row & 7;
      if (rr < U.nr) {
        const size_t grow = (size_t)(row < 8 ? U.j0 + rr : kI + U.j0 + rr);
        const int pos = BC ? (blk ^ ((row & 1) << 2)) : blk;
        cp_async16(dst + row * pitch + pos * 16, U.q13 + grow * kW13RowBytes + (bb + blk) * 16);
      }
    }
    if (lane < 16 && (lane & 7) < U.nr) {              // 16 rows x kGuU scale bytes
      const size_t grow = (size_t)(lane < 8 ? U.j0 + lane : kI + U.j0 + (lane & 7));
      cp_async8(dst + 16 * pitch + lane * 8, U.s13 + grow * kHBlocks + bb);
    }
  };
#pragma unroll
  for (int st = 0; st < STAGES - 1; ++st) {
    if (st < total) issue(st);
    cp_async_commit();
  }
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};   // even / odd blocks
  float bcacc[NT][2] = {};                                           // block columns: tiles x rows g, g + 8
  for (int st = 0; st < total; ++st) {
    if (st + STAGES - 1 < total) issue(st + STAGES - 1);
    cp_async_commit();
    cp_async_wait<STAGES - 1>();
    __syncwarp();
    if (cs == 0) { ++jc; Uc = (jc == ji) ? Ui : info(jc); }
    const GuUnit& U = Uc;
    const bool rv = g < U.nr;
    const uint8_t* buf = ring + (st % STAGES) * SBYTES;
    const int bb = U.kb0 + cs * kGuU;
    const bool unit_end = ++cs == spu;
    if (unit_end) cs = 0;
    if (BC) {
      constexpr int pitch = kGuU * 16;
      const uint8_t* scp = buf + 16 * pitch;
      // two token tiles: the super-steps as a loop (less code; measured 3.6 % faster at 4
      // tokens, 2 % slower at one token)
#pragma unroll (NT > 1 ? 1 : 2)
      for (int sb = 0; sb < kGuU; sb += 4) {
        const int pos = (sb + q) ^ ((g & 1) << 2);
        uint4 w0 = make_uint4(0, 0, 0, 0), w1 = w0;
        uint32_t s0 = 0x7F7Fu, s1 = 0x7F7Fu;             // 1.0 for absent rows
        if (rv) {
          w0 = *reinterpret_cast<const uint4*>(buf + g * pitch + pos * 16);
          w1 = *reinterpret_cast<const uint4*>(buf + (g + 8) * pitch + pos * 16);
          s0 = *reinterpret_cast<const uint16_t*>(scp + g * 8 + sb + 2 * (q & 1));
          s1 = *reinterpret_cast<const uint16_t*>(scp + (g + 8) * 8 + sb + 2 * (q & 1));
        }
        float d[NT][4] = {};
        const uint8_t* xb[NT];
        xb[0] = U.xtok ? U.xtok + 64 * (bb + sb + q) : nullptr;
        if (NT > 1) xb[NT - 1] = U.xtok2 ? U.xtok2 + 64 * (bb + sb + q) : nullptr;
        bc_step<NT>(w0, w1, xb, d);
#pragma unroll
        for (int j = 0; j < NT; ++j) bc_scale_add(d[j], s0 & 0xFF, s0 >> 8, s1 & 0xFF, s1 >> 8, bcacc[j]);
      }
      __syncwarp();
      if (unit_end) {
        float r[4];
        bc_finish<NT>(bcacc, q, r);
        done(jc, r);
#pragma unroll
        for (int j = 0; j < NT; ++j) bcacc[j][0] = bcacc[j][1] = 0.f;
      }
      continue;
    }
    uint2 scg = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu), scu = scg;
    if (rv) {
      scg = *reinterpret_cast<const uint2*>(buf + 16 * kGuPitch + g * 8);
      scu = *reinterpret_cast<const uint2*>(buf + 16 * kGuPitch + (g + 8) * 8);
    }
    // fast path (every scale of the stage in the f16-exact range): the scale is folded into
    // the f16 weights (an exact power-of-two multiply) and the MMAs accumulate directly
    const bool fast = __all_sync(0xffffffffu, e8m0x4_f16_exact(scg.x) && e8m0x4_f16_exact(scg.y) &&
                                                  e8m0x4_f16_exact(scu.x) && e8m0x4_f16_exact(scu.y));
#pragma unroll
    for (int u = 0; u < kGuU; ++u) {
      uint32_t wg = 0, wu = 0;
      if (rv) {
        wg = *reinterpret_cast<const uint32_t*>(buf + g * kGuPitch + u * 16 + 4 * q);
        wu = *reinterpret_cast<const uint32_t*>(buf + (g + 8) * kGuPitch + u * 16 + 4 * q);
      }
      uint4 xv = make_uint4(0, 0, 0, 0);
      if (U.xtok) {
        if (X8) {                                      // E4M3 codes 8q..8q+7 of the block -> f16
          const uint2 c = *reinterpret_cast<const uint2*>(U.xtok + 32 * (bb + u) + 8 * q);
          xv = make_uint4(e4m3x2_to_f16x2(c.x & 0xFFFFu), e4m3x2_to_f16x2(c.x >> 16), e4m3x2_to_f16x2(c.y & 0xFFFFu),
                          e4m3x2_to_f16x2(c.y >> 16));
        } else {
          xv = *reinterpret_cast<const uint4*>(U.xtok + 64 * (bb + u) + 16 * q);
        }
      }
      const uint32_t sgb = ((u < 4 ? scg.x : scg.y) >> (8 * (u & 3))) & 0xFF;
      const uint32_t sub = ((u < 4 ? scu.x : scu.y) >> (8 * (u & 3))) & 0xFF;
      uint32_t hg[4], hu[4];
      e2m1x8_to_f16x2x4(wg, hg);
      e2m1x8_to_f16x2x4(wu, hu);
      if (fast) {
        const uint32_t fg = e8m0_to_f16x2_pow2(sgb), fu = e8m0_to_f16x2_pow2(sub);
        float (&a)[4] = acc[u & 1];
        mma_16816(a, hmul2_u32(hg[0], fg), hmul2_u32(hu[0], fu), hmul2_u32(hg[1], fg), hmul2_u32(hu[1], fu), xv.x, xv.y);
        mma_16816(a, hmul2_u32(hg[2], fg), hmul2_u32(hu[2], fu), hmul2_u32(hg[3], fg), hmul2_u32(hu[3], fu), xv.z, xv.w);
      } else {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        mma_16816(d, hg[0], hu[0], hg[1], hu[1], xv.x, xv.y);
        mma_16816(d, hg[2], hu[2], hg[3], hu[3], xv.z, xv.w);
        const float fg = e8m0_to_f32(sgb), fu = e8m0_to_f32(sub);
        float (&a)[4] = acc[u & 1];
        a[0] = fmaf(fg, d[0], a[0]);
        a[1] = fmaf(fg, d[1], a[1]);
        a[2] = fmaf(fu, d[2], a[2]);
        a[3] = fmaf(fu, d[3], a[3]);
      }
    }
    __syncwarp();
    if (unit_end) {
      const float r[4] = {acc[0][0] + acc[1][0], acc[0][1] + acc[1][1], acc[0][2] + acc[1][2], acc[0][3] + acc[1][3]};
      done(jc, r);
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[0][i] = acc[1][i] = 0.f;
    }
  }
}

// Tile list of the kernels for more than 8 tokens, where a slot can have several 8-token
// column groups: the work space is every (slot, tile of 8 row pairs, column group) entry,
// slot-major, then tile, then group (slot s has 96 ceil(m_s / 8) entries), and the block takes
// entries [E b / G, E (b + 1) / G) of the E in all. Shares of whole tiles would give the
// blocks holding the shared expert's tiles (M tokens: ceil(M / 8) groups per tile) several
// times the work of the others. A share holds at most (257 slots x 96 + 36 x 96) / 152 < 190
// entries. `scratch` (n_slots + 1 ints) holds the slots' entry offsets. Every thread of the
// block must call it.
__device__ void build_gate_up_entries(Tables& tb, int* scratch) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = tb.n_slots, G = gridDim.x;
  constexpr int kTilesPerSlot = kI / 8;
  if (warp == 0) {
    int carry = 0;
    for (int b0 = 0; b0 < S; b0 += 32) {
      const int sidx = b0 + lane;
      const int c = sidx < S ? kTilesPerSlot * ((tb.slot_begin[sidx + 1] - tb.slot_begin[sidx] + 7) / 8) : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int nb = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += nb;
      }
      if (sidx < S) scratch[sidx] = carry + incl - c;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) scratch[S] = carry;
  }
  __syncthreads();
  const long long E = scratch[S];
  const int e0 = (int)(E * blockIdx.x / G), e1 = (int)(E * (blockIdx.x + 1) / G);
  const int n = e1 - e0 < kGuMaxTiles ? e1 - e0 : kGuMaxTiles;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int e = e0 + i;
    int lo = 0, hi = S - 1;                 // the slot with scratch[s] <= e < scratch[s + 1]
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (scratch[mid] <= e) lo = mid; else hi = mid - 1;
    }
    const int gq = (tb.slot_begin[lo + 1] - tb.slot_begin[lo] + 7) / 8, local = e - scratch[lo];
    tb.gu_tile[i] = make_int4(lo, 8 * (local / gq), 8, 8 * (local % gq));
  }
  if (threadIdx.x == 0) tb.gu_n = e1 - e0 > kGuMaxTiles ? -1 : e1 - e0;   // -1: does not fit
  __syncthreads();
}

// All gate/up tiles of the block's list: units (tile, K half) in rounds of kGuRound; the two
// halves' partials are summed in a fixed order, then SwiGLU, then h per (pair, row).
// Up to 8 tokens the list is implicit: the block's whole tiles are the virtual tiles
// [vt0, vt0 + ntiles) (slot vt / 96, rows 8 (vt mod 96)), none cut by a slot boundary since
// the shares are whole tiles; above, the tiles come from tb.gu_tile (tb.gu_n entries).
template <int MAXM>
__device__ void gate_up_tiles(const MoeParams& p, const LayerDesc& L, const uint8_t* smem, Tables& tb,
                              int vt0, int ntiles, int trace_layer = kTraceNone) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  float4* red = reinterpret_cast<float4*>(const_cast<uint8_t*>(smem) + smem_layout(p.M).gured);
  constexpr int kTilesPerSlot = kI / 8;
  auto tile_at = [&](int i) {
    if (MAXM <= 8) {
      const int vt = vt0 + i;
      return make_int4(vt / kTilesPerSlot, 8 * (vt % kTilesPerSlot), 8, 0);
    }
    return tb.gu_tile[i];
  };
  const int nt = MAXM <= 8 ? ntiles : tb.gu_n;
  // K split per tile: ks parts of 10 / ks stages (8 blocks each), chosen to minimise the
  // busiest warp's stages, ceil(tiles * ks / warps) * 10 / ks, plus about three stages of
  // latency and epilogue per round of kGuRound units (ties: the smaller ks)
  int ks = 1, best = 1 << 30;
  constexpr int kParts[4] = {1, 2, 5, 10};     // the divisors of the 10 stages (constant divisions)
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = kParts[i], per_round = kGuRound / c * c;
    const int rounds = (nt * c + per_round - 1) / per_round;
    const int cost = (nt * c + kWarps - 1) / kWarps * (10 / c) + 3 * rounds;
    if (cost < best) { best = cost; ks = c; }
  }
  const int units = nt * ks;
  const int kpart = kHBlocks / ks;
  // MMA form, fixed per kernel instantiation (each carries only its own loop, which keeps the
  // register allocation of the small-M kernels free of the other forms): block columns with
  // one tile for up to two tokens, two tiles for up to four, token columns beyond
  constexpr int BCN = MAXM <= 2 ? 1 : MAXM <= 4 ? 2 : 0;
  const bool bc = BCN > 0;
  const int round = kGuRound / ks * ks;            // a whole number of tiles per round
  uint8_t* ring = const_cast<uint8_t*>(smem) + smem_layout(p.M).ring + (size_t)warp * warp_ring_bytes(p.M);
  for (int u0 = 0; u0 < units; u0 += round) {
    const int un = min(round, units - u0);
    MDW_TRACE_POINT(trace_layer, 15);
    const int mine = un > warp ? (un - warp + kWarps - 1) / kWarps : 0;
    auto info = [&](int j) {
      const int u = u0 + warp + j * kWarps;
      const int4 t = tile_at(u / ks);
      const int kp = u % ks, slot = t.x, e = tb.slot_expert[slot];
      const int pb = tb.slot_begin[slot], m = tb.slot_begin[slot + 1] - pb;
      GuUnit U;
      U.q13 = e < 0 ? L.sh_w13_q : L.w13_q + (size_t)e * kRows13 * kW13RowBytes;
      U.s13 = e < 0 ? L.sh_w13_s : L.w13_s + (size_t)e * kRows13 * kHBlocks;
      U.xtok2 = nullptr;
      if (bc) {       // lane (g, q) feeds token 2j + (g >> 2) of tile j, on its own block q == g & 3
        const int tt = g >> 2;
        U.xtok = (q == (g & 3) && t.w + tt < m) ? smem + (size_t)tb.pair_token[pb + t.w + tt] * kXhBytes : nullptr;
        U.xtok2 = (q == (g & 3) && t.w + 2 + tt < m) ? smem + (size_t)tb.pair_token[pb + t.w + 2 + tt] * kXhBytes
                                                     : nullptr;
      } else {
        constexpr size_t xs = MAXM > 16 ? kXh8Bytes : kXhBytes;
        U.xtok = (t.w + g < m) ? smem + (size_t)tb.pair_token[pb + t.w + g] * xs : nullptr;
      }
      U.j0 = t.y;
      U.nr = t.z;
      U.kb0 = kp * kpart;
      return U;
    };
    auto done = [&](int j, const float (&acc)[4]) {
      red[(warp + j * kWarps) * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    };
    gate_up_units<BCN, (MAXM > 16)>(mine, 10 / ks, info, done, ring, lane);
    __syncthreads();
    MDW_TRACE_POINT(trace_layer, 16);
    for (int u = warp; u < un; u += kWarps) {
      if ((u0 + u) % ks != 0) continue;
      const int4 t = tile_at((u0 + u) / ks);
      float4 r = red[u * 32 + lane];
      for (int k = 1; k < ks; ++k) {
        const float4 o = red[(u + k) * 32 + lane];
        r.x += o.x; r.y += o.y; r.z += o.z; r.w += o.w;
      }
      const int slot = t.x, pb = tb.slot_begin[slot], m = tb.slot_begin[slot + 1] - pb;
      if (g < t.z) {
        const float gv[2] = {r.x, r.y}, uv[2] = {r.z, r.w};
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int col = t.w + 2 * q + c;
          if (col < m) {
            const float sx = tb.sx[tb.pair_token[pb + col]];
            const float gs = gv[c] * sx, us = uv[c] * sx;
            p.h[(size_t)(pb + col) * kI + t.y + g] = gs / (1.0f + expf(-gs)) * us;
          }
        }
      }
    }
    // the partial sums are reused by the next round; after the last one the caller's barrier
    // arrival (a block barrier first) follows
    if (u0 + round < units) __syncthreads();
  }
}

// ------------------------------------------------------------------ P4: h quant + down

// Quantise pairs [q0, q0 + n) into the h-hat planes of shared memory (and, from block 0,
// into the workspace for inspection).
__device__ void quantise_pairs(const MoeParams& p, uint8_t* smem, Tables& tb, int q0, int n) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int J = kI / 128;                     // 16-byte loads per lane per pair (6)
  // one pair per warp at a time, 16-byte loads
  for (int k0 = warp; k0 < n; k0 += kWarps) {
    uint4 v[1][J];
#pragma unroll
    for (int r = 0; r < 1; ++r) {
      const int k = k0 + r * kWarps;
      if (k < n) {
        const uint4* hv = reinterpret_cast<const uint4*>(p.h + (size_t)(q0 + k) * kI);
#pragma unroll
        for (int j = 0; j < J; ++j) v[r][j] = ld_cg16(hv + lane + 32 * j);
      }
    }
#pragma unroll
    for (int r = 0; r < 1; ++r) {
      const int k = k0 + r * kWarps;
      if (k >= n) break;                            // warp-uniform
      const int q = q0 + k;
      float am = 0.f;
#pragma unroll
      for (int j = 0; j < J; ++j)
        am = fmaxf(am, fmaxf(fmaxf(fabsf(__uint_as_float(v[r][j].x)), fabsf(__uint_as_float(v[r][j].y))),
                             fmaxf(fabsf(__uint_as_float(v[r][j].z)), fabsf(__uint_as_float(v[r][j].w)))));
      am = warp_max(am);
      const float s = am > 0.f ? __fdiv_rn(am, kE4M3Max) : 1.0f;
      if (lane == 0) tb.sh[k] = s;
      uint8_t* hh = smem + smem_layout(p.M).hh + (size_t)k * kHhBytes;
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int e = 4 * (lane + 32 * j);          // elements e .. e + 3
        const uint32_t c01 = f32x2_to_e4m3x2(__fdiv_rn(__uint_as_float(v[r][j].x), s),
                                             __fdiv_rn(__uint_as_float(v[r][j].y), s));
        const uint32_t c23 = f32x2_to_e4m3x2(__fdiv_rn(__uint_as_float(v[r][j].z), s),
                                             __fdiv_rn(__uint_as_float(v[r][j].w), s));
        *reinterpret_cast<uint2*>(hh + (size_t)e * 2) = make_uint2(e4m3x2_to_f16x2(c01), e4m3x2_to_f16x2(c23));
        if (blockIdx.x == 0) *reinterpret_cast<uint32_t*>(p.hq + (size_t)q * kI + e) = c01 | (c23 << 16);
      }
      if (blockIdx.x == 0 && lane == 0) p.sh[q] = s;
    }
  }
}

// Down projection + combine for the block's output rows [r0, r0 + nrows), in chunks of
// kPairChunk pairs (their h quantised into shared memory first).
//  * Full 16-row tiles on the tensor cores: m16n8k16 with A = 16 W2 rows (E2M1 -> f16),
//    B = h-hat of up to 8 of the slot's tokens (f16), K = 768 split in two halves of 12
//    blocks (one unit each, staged through the warp's cp.async ring); each block's fresh
//    result is scaled by the row's E8M0 scale in fp32; the halves are added in a fixed order.
//  * Leftover rows (nrows mod 16) on the CUDA cores, one warp per (pair, row).
// Every (pair, row) result is multiplied by the pair's gate and h scale into `part`, and the
// per-token sums are taken in pair order, so the output does not depend on scheduling.
// One down-projection unit in block-column form (NT tiles): 16 W2 rows x 12 blocks staged in
// buf (rows of kDnBcPitch bytes, then the rows' 24 scale bytes); h0 / h1 = the lane's h-hat
// of tile 0 / 1 (or null). Result in the token-column layout (see bc_finish).
template <int NT>
__device__ __forceinline__ void down_bc_unit(const uint8_t* buf, int g, int qd, int kb0, const uint8_t* h0,
                                             const uint8_t* h1, float (&r)[4]) {
  const uint8_t* scp = buf + 16 * kDnBcPitch;
  float bcacc[NT][2] = {};
#pragma unroll (NT > 1 ? 1 : 3)
  for (int sb = 0; sb < kDnKB; sb += 4) {
    const uint4 w0 = *reinterpret_cast<const uint4*>(buf + g * kDnBcPitch + (sb + qd) * 16);
    const uint4 w1 = *reinterpret_cast<const uint4*>(buf + (g + 8) * kDnBcPitch + (sb + qd) * 16);
    const uint32_t s0 = *reinterpret_cast<const uint16_t*>(scp + g * kIBlocks + kb0 + sb + 2 * (qd & 1));
    const uint32_t s1 = *reinterpret_cast<const uint16_t*>(scp + (g + 8) * kIBlocks + kb0 + sb + 2 * (qd & 1));
    float d[NT][4] = {};
    const uint8_t* xb[NT];
    xb[0] = h0 ? h0 + 64 * (kb0 + sb + qd) : nullptr;
    if (NT > 1) xb[NT - 1] = h1 ? h1 + 64 * (kb0 + sb + qd) : nullptr;
    bc_step<NT>(w0, w1, xb, d);
#pragma unroll
    for (int j = 0; j < NT; ++j) bc_scale_add(d[j], s0 & 0xFF, s0 >> 8, s1 & 0xFF, s1 >> 8, bcacc[j]);
  }
  bc_finish<NT>(bcacc, qd, r);
}

// Down-projection unit list of pairs [q0, q0 + n): (slot, full 16-row tile, K half, 8-pair
// group). The slots of the chunk (at most kPairChunk + 1, 32 per round of warp 0) and their
// unit counts (tiles x 8-pair groups x 2 K halves) are scanned; then every thread writes
// units. Every thread of the block must call it.
__device__ void build_down_units(Tables& tb, int q0, int n, int nfull) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  static_assert(kMaxSegs >= kPairChunk + 1, "segment tables too small for a pair chunk");
  if (warp == 0) {
    const int s_lo = tb.pair_slot[q0], s_hi = tb.pair_slot[q0 + n - 1];
    int carry = 0;
    for (int b0 = 0; s_lo + b0 <= s_hi; b0 += 32) {
      const int sidx = s_lo + b0 + lane;
      int c = 0, pa = 0;
      if (sidx <= s_hi) {
        pa = max(tb.slot_begin[sidx], q0);
        const int pz = min(tb.slot_begin[sidx + 1], q0 + n);
        c = nfull * ((pz - pa + 7) / 8) * 2;
      }
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int nb = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += nb;
      }
      if (sidx <= s_hi) {
        tb.seg_slot[b0 + lane] = sidx;
        tb.seg_lo[b0 + lane] = pa;
        tb.seg_groups[b0 + lane] = c / (2 * max(1, nfull));
        tb.seg_off[b0 + lane] = carry + incl - c;
      }
      if (sidx == s_hi) { tb.seg_off[b0 + lane + 1] = carry + incl; tb.gu_n = carry + incl; }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) tb.n_segs = s_hi - s_lo + 1;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < tb.gu_n; i += blockDim.x) {
    int k = 0;
    while (i >= tb.seg_off[k + 1]) ++k;
    const int r = i - tb.seg_off[k], gq = tb.seg_groups[k];
    const int kp = r & 1, tg = r >> 1;
    tb.gu_tile[i] = make_int4(tb.seg_slot[k], tg / gq, kp, tb.seg_lo[k] + 8 * (tg % gq));
  }
  __syncthreads();
}

// The block's output rows [r0, r1): an equal share of the H rows; for the windows that publish
// the residual as tagged words (two bf16 each) in whole row pairs (16 or 18 rows on 152
// blocks), so that every word it publishes is its own; else 16 or 17 rows.
template <int MAXM>
__device__ __forceinline__ void out_rows(int G, int& r0, int& r1) {
  if (MAXM <= kTaggedResidM) {
    r0 = 2 * (int)((long long)blockIdx.x * (kH / 2) / G);
    r1 = 2 * (int)((long long)(blockIdx.x + 1) * (kH / 2) / G);
  } else {
    r0 = (int)((long long)blockIdx.x * kH / G);
    r1 = (int)((long long)(blockIdx.x + 1) * kH / G);
  }
}

// Output rows [r0, r1) of this block: 16-row tiles + a remainder.
template <int MAXM>
__device__ __forceinline__ int down_full_tiles(int G) {
  int r0, r1;
  out_rows<MAXM>(G, r0, r1);
  return (r1 - r0) / 16;
}

template <int MAXM>
__device__ void down_combine(const MoeParams& p, const LayerDesc& L, uint8_t* smem, Tables& tb,
                             int layer, bool first_list_ready) {
  const int M = p.M, G = gridDim.x;
  int r0, r1;
  out_rows<MAXM>(G, r0, r1);
  const int nrows = r1 - r0, nfull = nrows / 16, nrem = nrows - 16 * nfull;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, qd = lane & 3;
  const Smem sl = smem_layout(M);
  float* part = reinterpret_cast<float*>(smem + sl.part);
  float* yacc = reinterpret_cast<float*>(smem + sl.yacc);
  float4* red = reinterpret_cast<float4*>(smem + sl.gured);
  uint8_t* ring = smem + sl.ring + (size_t)warp * warp_ring_bytes(M);
  for (int i = threadIdx.x; i < M * kMaxRowsPerBlock; i += blockDim.x) yacc[i] = 0.f;
  // the residual of this thread's first output element, requested now (its load overlaps
  // the whole projection instead of following it)
  const __nv_bfloat16* res_in = p.stack_mode ? resid_ptr(p, layer) : p.residual;
  float res0 = 0.f;
  if (res_in && threadIdx.x < M * nrows) {
    const int t = threadIdx.x / nrows, rr = threadIdx.x % nrows;
    res0 = __bfloat162float(res_in[(size_t)t * kH + r0 + rr]);
  }
  auto w2_of = [&](int slot, const uint8_t*& q2, const uint8_t*& s2) {
    const int e = tb.slot_expert[slot];
    q2 = e < 0 ? L.sh_w2_q : L.w2_q + (size_t)e * kH * kW2RowBytes;
    s2 = e < 0 ? L.sh_w2_s : L.w2_s + (size_t)e * kH * kIBlocks;
  };
  const int NP = tb.n_pairs;
  constexpr int BCN = MAXM <= 2 ? 1 : MAXM <= 4 ? 2 : 0;   // as in gate_up_tiles
  const bool bc = BCN > 0;
  // 2 to 4 tokens: the pairs (at most 36) are one chunk and every slot is one pair group, so
  // the unit list is implicit: unit i = (slot i / (2 nfull), tile (i / 2) mod nfull, K half
  // i mod 2, first pair slot_begin[slot]) -- the order build_down_units lays out (measured
  // 2.6 / 4.3 % faster at 2 / 4 tokens; one token keeps the list built during the h barrier,
  // 1 % faster there)
  constexpr bool kImplicit = MAXM > 1 && MAXM <= 4;
  static_assert(!kImplicit || 4 * (MDW_MAX_TOPK + 1) <= kPairChunk, "one chunk up to 4 tokens");
  auto unit_at = [&](int i) {
    if (kImplicit) {
      const int s = i / (2 * nfull), r = i - s * 2 * nfull;
      return make_int4(s, r >> 1, r & 1, tb.slot_begin[s]);
    }
    return tb.gu_tile[i];
  };
  for (int q0 = 0; q0 < NP; q0 += kPairChunk) {
    const int n = min(kPairChunk, NP - q0);
    // a later chunk overwrites the h-hat, partials and list of the previous one (the first
    // follows the h barrier's block barrier, after which nothing here is still being read)
    if (q0 > 0) __syncthreads();
    MDW_TRACE_POINT(layer, 17);
    quantise_pairs(p, smem, tb, q0, n);
    MDW_TRACE_POINT(layer, 18);
    // unit list (the first chunk's was built during the h barrier); either way a block-wide
    // barrier follows, so every warp sees the whole chunk's h-hat before the tiles
    if (!kImplicit && (q0 > 0 || !first_list_ready)) build_down_units(tb, q0, n, nfull);
    else __syncthreads();
    MDW_TRACE_POINT(layer, 13);
    // leftover rows (nrows mod 16, CUDA cores, one warp per (pair, row)): the weights of
    // this warp's first item are requested now, so they arrive while the tiles run
    const int rem_items = n * nrem;
    const int rem_first = kWarps - 1 - warp;         // the last warps (fewest tiles) start
    uint4 rem_w = make_uint4(0, 0, 0, 0);
    uint32_t rem_s = 0;
    if (rem_first < rem_items && lane < kIBlocks) {
      const int k2 = rem_first / nrem, rr = 16 * nfull + rem_first % nrem;
      const uint8_t *q2, *s2;
      w2_of(tb.pair_slot[q0 + k2], q2, s2);
      rem_w = ldg_stream16(q2 + (size_t)(r0 + rr) * kW2RowBytes + lane * 16);
      rem_s = ldg_stream_u8(s2 + (size_t)(r0 + rr) * kIBlocks + lane);
    }
    // leftover rows: lanes 0..23 one block each; run by each warp right after its tiles
    auto do_rem = [&]() {
    for (int it = rem_first; it < rem_items; it += kWarps) {
      const int k2 = it / nrem, rr = 16 * nfull + it % nrem, q = q0 + k2;
      float dsum = 0.f;
      if (lane < kIBlocks) {
        if (it != rem_first) {
          const uint8_t *q2, *s2;
          w2_of(tb.pair_slot[q], q2, s2);
          rem_w = ldg_stream16(q2 + (size_t)(r0 + rr) * kW2RowBytes + lane * 16);
          rem_s = ldg_stream_u8(s2 + (size_t)(r0 + rr) * kIBlocks + lane);
        }
        const uint8_t* hh = smem + sl.hh + (size_t)k2 * kHhBytes + 64 * lane;
        uint32_t x2[16];
#pragma unroll
        for (int pl = 0; pl < 4; ++pl) {
          const uint4 xv = *reinterpret_cast<const uint4*>(hh + 16 * pl);
          x2[4 * pl] = xv.x; x2[4 * pl + 1] = xv.y; x2[4 * pl + 2] = xv.z; x2[4 * pl + 3] = xv.w;
        }
        dsum = mx_block_dot(rem_w, x2) * e8m0_to_f32(rem_s);
      }
      dsum = warp_sum(dsum);
      if (lane == 0) part[k2 * kMaxRowsPerBlock + rr] = dsum * tb.sh[k2] * tb.pair_gate[q];
    }
    };
    const int units = kImplicit ? tb.n_slots * 2 * nfull : tb.gu_n;
    for (int u0 = 0; u0 < units; u0 += kGuRound) {
      const int un = min(kGuRound, units - u0);
      const int mine = un > warp ? (un - warp + kWarps - 1) / kWarps : 0;
      auto issue = [&](int k) {
        const int4 t = unit_at(u0 + warp + k * kWarps);
        const uint8_t *q2, *s2;
        w2_of(t.x, q2, s2);
        uint8_t* dst = ring + (k % kDnStages) * kDnStageBytes;
        const int rb = r0 + 16 * t.y, kb0 = t.z * kDnKB;
        const int pitch = bc ? kDnBcPitch : kDnPitch;
#pragma unroll
        for (int j = 0; j < 16 * kDnKB / 32; ++j) {     // 16 rows x 12 chunks of 16 bytes
          const int c = lane + 32 * j, row = c / kDnKB, blk = c % kDnKB;
          cp_async16(dst + row * pitch + blk * 16, q2 + (size_t)(rb + row) * kW2RowBytes + (kb0 + blk) * 16);
        }
        if (lane < 16 * 3 / 2) {                         // 16 rows x 24 scale bytes, 8 at a time
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int c = lane + 24 * j, row = c / 3, part8 = c % 3;
            cp_async8(dst + 16 * pitch + row * kIBlocks + part8 * 8,
                      s2 + (size_t)(rb + row) * kIBlocks + part8 * 8);
          }
        }
      };
      if (mine > 0) issue(0);
      cp_async_commit();
      for (int k = 0; k < mine; ++k) {
        if (k + 1 < mine) issue(k + 1);
        cp_async_commit();
        cp_async_wait<kDnStages - 1>();
        __syncwarp();
        const uint8_t* buf = ring + (k % kDnStages) * kDnStageBytes;
        const int4 t = unit_at(u0 + warp + k * kWarps);
        const int pz = min(tb.slot_begin[t.x + 1], q0 + n);
        const int kb0 = t.z * kDnKB;
        if (bc) {
          // block columns: lane (g, q) feeds pair t.w + 2j + (g >> 2) of tile j on its own block
          // q == g & 3
          const int tt = g >> 2;
          const uint8_t* h0 = (qd == (g & 3) && t.w + tt < pz) ? smem + sl.hh + (size_t)(t.w + tt - q0) * kHhBytes : nullptr;
          const uint8_t* h1 = (qd == (g & 3) && t.w + 2 + tt < pz) ? smem + sl.hh + (size_t)(t.w + 2 + tt - q0) * kHhBytes
                                                                   : nullptr;
          float r[4];
          down_bc_unit<BCN ? BCN : 1>(buf, g, qd, kb0, h0, h1, r);
          __syncwarp();
          red[(warp + k * kWarps) * 32 + lane] = make_float4(r[0], r[1], r[2], r[3]);
          continue;
        }
        // B column g = token pair t.w + g of the slot (if it exists in this chunk)
        const uint8_t* hb = (t.w + g < pz) ? smem + sl.hh + (size_t)(t.w + g - q0) * kHhBytes : nullptr;
        const uint8_t* sc_g = buf + 16 * kDnPitch + g * kIBlocks + kb0;
        const uint8_t* sc_g8 = buf + 16 * kDnPitch + (g + 8) * kIBlocks + kb0;
        // scales of the unit (12 blocks of rows g and g + 8): fast path as in the gate/up units
        uint32_t sa3[3], sb3[3];
#pragma unroll
        for (int i = 0; i < 3; ++i) {
          sa3[i] = reinterpret_cast<const uint32_t*>(sc_g)[i];      // 4-byte aligned: 3328 + 24 g + 12 kp
          sb3[i] = reinterpret_cast<const uint32_t*>(sc_g8)[i];
        }
        const bool fast = __all_sync(0xffffffffu, e8m0x4_f16_exact(sa3[0]) && e8m0x4_f16_exact(sa3[1]) &&
                                                      e8m0x4_f16_exact(sa3[2]) && e8m0x4_f16_exact(sb3[0]) &&
                                                      e8m0x4_f16_exact(sb3[1]) && e8m0x4_f16_exact(sb3[2]));
        float acc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int b = 0; b < kDnKB; ++b) {
          const uint32_t wa = *reinterpret_cast<const uint32_t*>(buf + g * kDnPitch + b * 16 + 4 * qd);
          const uint32_t wb = *reinterpret_cast<const uint32_t*>(buf + (g + 8) * kDnPitch + b * 16 + 4 * qd);
          uint4 xv = make_uint4(0, 0, 0, 0);
          if (hb) xv = *reinterpret_cast<const uint4*>(hb + 64 * (kb0 + b) + 16 * qd);
          uint32_t ha[4], hc[4];
          e2m1x8_to_f16x2x4(wa, ha);
          e2m1x8_to_f16x2x4(wb, hc);
          const uint32_t sab = (sa3[b >> 2] >> (8 * (b & 3))) & 0xFF, sbb = (sb3[b >> 2] >> (8 * (b & 3))) & 0xFF;
          float (&a)[4] = acc2[b & 1];
          if (fast) {
            const uint32_t fa = e8m0_to_f16x2_pow2(sab), fb = e8m0_to_f16x2_pow2(sbb);
            mma_16816(a, hmul2_u32(ha[0], fa), hmul2_u32(hc[0], fb), hmul2_u32(ha[1], fa), hmul2_u32(hc[1], fb), xv.x, xv.y);
            mma_16816(a, hmul2_u32(ha[2], fa), hmul2_u32(hc[2], fb), hmul2_u32(ha[3], fa), hmul2_u32(hc[3], fb), xv.z, xv.w);
          } else {
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            mma_16816(d, ha[0], hc[0], ha[1], hc[1], xv.x, xv.y);
            mma_16816(d, ha[2], hc[2], ha[3], hc[3], xv.z, xv.w);
            const float fa = e8m0_to_f32(sab), fb = e8m0_to_f32(sbb);
            a[0] = fmaf(fa, d[0], a[0]);
            a[1] = fmaf(fa, d[1], a[1]);
            a[2] = fmaf(fb, d[2], a[2]);
            a[3] = fmaf(fb, d[3], a[3]);
          }
        }
        const float acc[4] = {acc2[0][0] + acc2[1][0], acc2[0][1] + acc2[1][1], acc2[0][2] + acc2[1][2],
                              acc2[0][3] + acc2[1][3]};
        __syncwarp();
        red[(warp + k * kWarps) * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      }
      if (u0 + kGuRound >= units) do_rem();          // the last round: leftover rows next
      __syncthreads();
      MDW_TRACE_POINT(layer, 19);
      // K halves added in order (unit kp = 0 owns the pair); D rows = W2 rows g, g + 8;
      // D columns 2qd, 2qd + 1 = pairs t.w + 2qd (+1)
      for (int u = warp; u < un; u += kWarps) {
        const int4 t = unit_at(u0 + u);
        if (t.z != 0) continue;
        const float4 a0 = red[u * 32 + lane], a1 = red[(u + 1) * 32 + lane];
        const float v[4] = {a0.x + a1.x, a0.y + a1.y, a0.z + a1.z, a0.w + a1.w};
        const int pz = min(tb.slot_begin[t.x + 1], q0 + n);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int q = t.w + 2 * qd + c;
          if (q >= pz) continue;
          const int k2 = q - q0;
          const float f = tb.sh[k2] * tb.pair_gate[q];
          part[k2 * kMaxRowsPerBlock + 16 * t.y + g] = v[c] * f;
          part[k2 * kMaxRowsPerBlock + 16 * t.y + g + 8] = v[2 + c] * f;
        }
      }
    }
    if (units == 0) do_rem();
    __syncthreads();
    MDW_TRACE_POINT(layer, 14);
    // fixed-order accumulation over the chunk's pairs (ascending)
    for (int i = threadIdx.x; i < M * nrows; i += blockDim.x) {
      const int t = i / nrows, rr = i % nrows;
      float a = yacc[t * kMaxRowsPerBlock + rr];
      for (int k = 0; k < n; ++k)
        if (tb.pair_token[q0 + k] == t) a += part[k * kMaxRowsPerBlock + rr];
      yacc[t * kMaxRowsPerBlock + rr] = a;
    }
  }
  __syncthreads();
  if (p.stack_mode) {
    // r_{l+1} = bf16(r_l + y) for the block's rows, row pairs: into the residual buffer and,
    // for the next layer, as tagged words (two bf16 each, tag l + 1)
    __nv_bfloat16* rout = const_cast<__nv_bfloat16*>(resid_ptr(p, layer + 1));
    if (MAXM > kTaggedResidM) {
      for (int i = threadIdx.x; i < M * nrows; i += blockDim.x) {
        const int t = i / nrows, rr = i % nrows;
        const size_t o = (size_t)t * kH + r0 + rr;
        rout[o] = __float2bfloat16_rn(__bfloat162float(res_in[o]) + yacc[t * kMaxRowsPerBlock + rr]);
      }
      return;
    }
    const int np = nrows / 2;
    for (int i = threadIdx.x; i < M * np; i += blockDim.x) {
      const int t = i / np, rr = 2 * (i % np);
      const size_t o = (size_t)t * kH + r0 + rr;
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(__bfloat162float(res_in[o]) + yacc[t * kMaxRowsPerBlock + rr],
                                                      __bfloat162float(res_in[o + 1]) + yacc[t * kMaxRowsPerBlock + rr + 1]);
      const uint32_t bits = *reinterpret_cast<const uint32_t*>(&b2);
      *reinterpret_cast<uint32_t*>(rout + o) = bits;
      if (layer + 1 < p.L) st_word(p.xr + o / 2, tagged(bits, (uint32_t)layer + 1));
    }
    return;
  }
  for (int i = threadIdx.x; i < M * nrows; i += blockDim.x) {
    const int t = i / nrows, rr = i % nrows;
    const float y = yacc[t * kMaxRowsPerBlock + rr];
    const size_t o = (size_t)t * kH + r0 + rr;
    const float rv = (i == (int)threadIdx.x) ? res0 : (res_in ? __bfloat162float(res_in[o]) : 0.f);
    {
      float v = y;
      if (p.residual) v += rv;
      if (p.y_fp32) reinterpret_cast<float*>(p.y_out)[o] = v;
      else reinterpret_cast<__nv_bfloat16*>(p.y_out)[o] = __float2bfloat16_rn(v);
    }
  }
}

// Bulk L2 prefetch of [base + lo, base + hi) shrunk to 16-byte boundaries (the TMA unit
// handles it, so the SM's load path stays free).
__device__ __forceinline__ void prefetch_bulk(const uint8_t* base, size_t lo, size_t hi) {
  lo = (lo + 15) & ~(size_t)15;
  hi &= ~(size_t)15;
  if (hi > lo) prefetch_l2(base + lo, (uint32_t)(hi - lo));
}

// Bulk L2 prefetches are accepted by the TMA unit only as fast as the memory system takes
// their requests, so the issuing thread (and its warp) blocks for about (bytes in flight
// GPU-wide) / (DRAM bandwidth). The W2 rows are therefore requested after the block has
// arrived at the h barrier, where the blocking overlaps the wait; the gate/up rows are not
// prefetched at all (measured: requesting them right after routing delayed the warps that
// issued them by more than the cp.async pipeline gained).
// The block's W2 rows [r0, r1) (and scales) of every slot, dealt to every warp's lane 0.
template <int MAXM>
__device__ void prefetch_down_rows(const LayerDesc& L, const Tables& tb) {
  const int G = gridDim.x;
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) != 0) return;
  int r0, r1;
  out_rows<MAXM>(G, r0, r1);
  for (int s = warp; s < tb.n_slots; s += kWarps) {
    const int e = tb.slot_expert[s];
    const uint8_t* q2 = e < 0 ? L.sh_w2_q : L.w2_q + (size_t)e * kH * kW2RowBytes;
    const uint8_t* s2 = e < 0 ? L.sh_w2_s : L.w2_s + (size_t)e * kH * kIBlocks;
    prefetch_bulk(q2, (size_t)r0 * kW2RowBytes, (size_t)r1 * kW2RowBytes);
    prefetch_bulk(s2, (size_t)r0 * kIBlocks, (size_t)r1 * kIBlocks);
  }
}

// This block's router rows and shared-expert slice of a layer (routing-independent): five
// bulk L2 prefetches, from lane 0 of warps 0..4.
__device__ void prefetch_static(const MoeParams& p, const LayerDesc& L) {
  const int G = gridDim.x, E = p.E;
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) != 0 || warp > 4) return;
  if (warp == 0) {
    const int e0 = (int)((long long)blockIdx.x * E / G), e1 = (int)((long long)(blockIdx.x + 1) * E / G);
    prefetch_l2(L.router_w + (size_t)e0 * kH, (uint32_t)((e1 - e0) * kH * 2));
  } else if (p.has_shared) {
    const int j0 = (int)((long long)blockIdx.x * kI / G), j1 = (int)((long long)(blockIdx.x + 1) * kI / G);
    const size_t row = (size_t)((warp - 1) & 1) * kI + j0;
    if (warp <= 2) prefetch_l2(L.sh_w13_q + row * kW13RowBytes, (uint32_t)((j1 - j0) * kW13RowBytes));
    else prefetch_l2(L.sh_w13_s + row * kHBlocks, (uint32_t)((j1 - j0) * kHBlocks));
  }
}

// ------------------------------------------------------------------ the kernel

template <int MAXM>
__global__ void __launch_bounds__(kThreads, 1) moe_persistent_kernel(const __grid_constant__ MoeParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  Tables& tb = *reinterpret_cast<Tables*>(smem + smem_layout(p.M).small);
  GridBarrier bar{p.hdr, 0, p.spin_budget};
  const int G = gridDim.x;
  for (int layer = 0; layer < p.L; ++layer) {
    const LayerDesc& L = p.layers[layer];
    MDW_TRACE_POINT(layer, 0);
    {
      // the router row's weights are requested before the input, so the two loads overlap
      uint4 wv[10];
      int e0, e1;
      router_range(p, e0, e1);
      if (e0 + (int)(threadIdx.x >> 5) < e1) load_router_row(L, e0 + (threadIdx.x >> 5), wv);
      prepare_input<MAXM>(p, layer, smem, tb);
      MDW_TRACE_POINT(layer, 1);
      if (tb.bad) return;                                           // the residual wait ran out
      router_rows(p, L, smem, wv, layer);
    }
    // the logits travel as tagged words (route_tokens polls them): no barrier
    if (MAXM > 16) xhat_codes_in_place(p, smem, tb);                 // the router is done with x
    MDW_TRACE_POINT(layer, 2);
    route_tokens(p, L, tb, layer, smem + smem_layout(p.M).gured);
    __syncthreads();
    // tb.bad: 1 = an imposed id out of range or repeated, 2 = a wait ran out (status recorded)
    if (tb.bad) { if (threadIdx.x == 0 && tb.bad == 1) set_status(p.hdr, MDW_ERR_DEVICE_BOUNDS); return; }
    {
      // gate/up tiles of 8 row pairs of every slot (the shared expert is slot 0; 96 whole
      // tiles per slot), dealt to the blocks in equal contiguous shares of whole tiles (up to
      // 8 tokens) or of (tile, column group) entries (more tokens), so no block pays for a
      // tile cut at a share boundary
      const long long T = (long long)tb.n_slots * (kI / 8);
      const int a = 8 * (int)((long long)blockIdx.x * T / G), b = 8 * (int)((long long)(blockIdx.x + 1) * T / G);
      MDW_TRACE_POINT(layer, 5);
      if (MAXM > 8) {
        // (up to 8 tokens every slot has one column group and the block's share is the whole
        // tiles [a / 8, b / 8), walked without a list)
        build_gate_up_entries(tb, reinterpret_cast<int*>(smem + smem_layout(p.M).gured));
        if (tb.gu_n < 0) { if (threadIdx.x == 0) set_status(p.hdr, MDW_ERR_UNSUPPORTED_SHAPE); return; }
      }
      gate_up_tiles<MAXM>(p, L, smem, tb, a / 8, (b - a) / 8, layer);
    }
    bar.arrive();                                                   // B2 (h)
    MDW_TRACE_POINT(layer, 6);
    // during the h barrier: W2 rows into L2, the first chunk's down unit list (the gate/up
    // tile list it overwrites is finished), and the next layer's static weights
    prefetch_down_rows<MAXM>(L, tb);
    if (MAXM == 1 || MAXM > 4) build_down_units(tb, 0, min(kPairChunk, tb.n_pairs), down_full_tiles<MAXM>(G));
    if (p.stack_mode && layer + 1 < p.L) prefetch_static(p, p.layers[layer + 1]);
    if (!bar.wait()) return;
    MDW_TRACE_POINT(layer, 7);
    down_combine<MAXM>(p, L, smem, tb, layer, true);
    MDW_TRACE_POINT(layer, 8);
    // r_{l+1}: up to kTaggedResidM tokens it travels as tagged words (the next layer's input
    // polls them) and no barrier is needed -- a block can only overwrite this layer's h,
    // logits or tables after every block has published its next-layer logits, i.e. after
    // every block has finished this layer's down phase; larger windows meet at a barrier
    if (MAXM > kTaggedResidM && p.stack_mode && layer + 1 < p.L) {
      if (!bar.sync()) return;                                      // B3 (r_{l+1})
    }
    MDW_TRACE_POINT(layer, 9);
  }
}

template <int MAXM>
cudaError_t launch_t(const MoeParams& p, cudaStream_t s) {
  const size_t smem = smem_layout(p.M).total;
  auto kern = moe_persistent_kernel<MAXM>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  void* args[] = {const_cast<MoeParams*>(&p)};
  return cudaLaunchCooperativeKernel((const void*)kern, dim3(moe_grid()), dim3(kThreads), args, smem, s);
}

}  // namespace

size_t moe_smem_bytes(int M) { return smem_layout(M).total; }

#ifdef MDW_TRACE
extern "C" int mdw_trace_read(void* dst, size_t bytes) {
  return (int)cudaMemcpyFromSymbol(dst, g_trace, bytes < sizeof(g_trace) ? bytes : sizeof(g_trace));
}
#endif

cudaError_t launch_moe(const MoeParams& p, cudaStream_t s) {
  if (p.M <= 1) return launch_t<1>(p, s);
  if (p.M <= 2) return launch_t<2>(p, s);
  if (p.M <= 4) return launch_t<4>(p, s);
  if (p.M <= 8) return launch_t<8>(p, s);
  if (p.M <= 16) return launch_t<16>(p, s);
  return launch_t<32>(p, s);
}

}  // namespace mdw
