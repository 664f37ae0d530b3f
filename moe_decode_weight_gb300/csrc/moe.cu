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
//   P0  (stack) x = bf16(RMSNorm(r_l)) and (all) xq = E4M3(x / sx): computed redundantly
//       by every block from the 5 KB/token input, so no exchange is needed;
//   P1  router logits for its slice of the E router rows -> global; arrive(B1);
//       while B1 completes: the shared expert's gate/up for its static slice of rows;
//   P2  wait(B1); top-k + dedup redundantly from the E x M logits (every block derives
//       the same slot / pair tables); L2 prefetch of its down-projection rows;
//   P3  routed gate/up for its contiguous slice of the (slot, row-pair) space -> h;
//       arrive(B2); (stack) L2 prefetch of the next layer's static weights; wait(B2);
//   P4  every block quantises all pairs' h (amax / 448) into shared memory, then computes
//       its slice of output rows over all slots (no atomics: a fixed summation order);
//       (stack) r_{l+1} = bf16(r_l + y); B3.
// Every inter-block wait is bounded and records MDW_ERR_TIMEOUT instead of hanging.
#include "mdw_device.cuh"
#include "mdw_internal.h"

namespace mdw {
namespace {

constexpr int kRows13 = 2 * kI;                 // w13 rows per expert
constexpr int kW13RowBytes = kH / 2;            // 1280
constexpr int kW2RowBytes = kI / 2;             // 384
constexpr int kXhBytes = kH * 2;                // f16 x-hat per token (planes layout)
constexpr int kHhBytes = kI * 2;                // f16 h-hat per pair (planes layout)
constexpr int kPairChunk = 48;                  // pairs quantised into smem at a time
constexpr int kMaxRowsPerBlock = 32;            // down-projection rows per block (>= H / grid)

// Shared-memory carve-up (bytes), for M tokens.
struct Smem {
  size_t xh, xb, hh, part, yacc, small, total;
};
__host__ __device__ inline Smem smem_layout(int M) {
  Smem s;
  s.xh = 0;
  s.xb = s.xh + (size_t)M * kXhBytes;
  size_t region = s.xb + (size_t)M * kH * 2;                   // x-hat + bf16 x
  size_t hh_bytes = (size_t)kPairChunk * kHhBytes;             // reuses the x region
  s.hh = 0;
  size_t big = region > hh_bytes ? region : hh_bytes;
  s.part = (big + 15) & ~(size_t)15;                            // [kPairChunk][rows] fp32
  s.yacc = s.part + (size_t)kPairChunk * kMaxRowsPerBlock * 4;     // [M][rows] fp32
  s.small = s.yacc + (size_t)M * kMaxRowsPerBlock * 4;
  s.total = s.small + 12288;
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
  float sh[kPairChunk];
  int n_slots, n_routed, n_pairs, shared_slot, bad;
};
static_assert(sizeof(Tables) <= 12288, "tables exceed the reserved shared memory");

// ------------------------------------------------------------------ P0: input / act quant

// r_l of the stack: r_0 is the caller's input; r_1.. live in the residual buffers.
__device__ __forceinline__ const __nv_bfloat16* resid_ptr(const MoeParams& p, int l) {
  if (l == 0) return p.r0;
  const int slot = p.resid_pingpong ? (l & 1) : l;
  return p.resid + (size_t)slot * p.M * kH;
}

// x-hat planes layout: token t, block b, plane c (elements 8c..8c+7 of the block) at
// byte t*kXhBytes + (c*kHBlocks + b)*16.
template <int MAXM>
__device__ void prepare_input(const MoeParams& p, int layer, uint8_t* smem, Tables& tb) {
  const int M = p.M;
  __nv_bfloat16* xb = reinterpret_cast<__nv_bfloat16*>(smem + smem_layout(M).xb);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const __nv_bfloat16* src = !p.stack_mode ? p.x_in : resid_ptr(p, layer);
  // 1. copy (stack: then normalise) into xb; one warp per token
  for (int t = warp; t < M; t += kWarps) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src + (size_t)t * kH);
    uint4* d4 = reinterpret_cast<uint4*>(xb + (size_t)t * kH);
    if (!p.stack_mode) {
      for (int i = lane; i < kH / 8; i += 32) d4[i] = ld_cg16(s4 + i);
    } else {
      float ss = 0.f;
      for (int i = lane; i < kH / 8; i += 32) {
        uint4 v = ld_cg16(s4 + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float a = __uint_as_float(w[k] << 16), b = __uint_as_float(w[k] & 0xFFFF0000u);
          ss = fmaf(a, a, ss);
          ss = fmaf(b, b, ss);
        }
        d4[i] = v;
      }
      ss = warp_sum(ss);
      const float inv = rsqrtf(ss / (float)kH + 1e-6f);
      for (int i = lane; i < kH / 8; i += 32) {
        uint4 v = d4[i];
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float a = __uint_as_float(w[k] << 16) * inv, b = __uint_as_float(w[k] & 0xFFFF0000u) * inv;
          __nv_bfloat162 r = __floats2bfloat162_rn(a, b);
          w[k] = *reinterpret_cast<uint32_t*>(&r);
        }
        d4[i] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
  __syncthreads();
  // 2. per-token E4M3 quantisation: amax exact, scale = amax/448 and x/scale correctly
  //    rounded (IEEE division), round-to-nearest-even saturating conversion
  for (int t = warp; t < M; t += kWarps) {
    const uint32_t* x32 = reinterpret_cast<const uint32_t*>(xb + (size_t)t * kH);
    float am = 0.f;
    for (int i = lane; i < kH / 2; i += 32) {
      uint32_t w = x32[i];
      am = fmaxf(am, fmaxf(fabsf(__uint_as_float(w << 16)), fabsf(__uint_as_float(w & 0xFFFF0000u))));
    }
    am = warp_max(am);
    const float s = am > 0.f ? __fdiv_rn(am, kE4M3Max) : 1.0f;
    if (lane == 0) tb.sx[t] = s;
    uint8_t* xh = smem + (size_t)t * kXhBytes;
    const bool writer = (blockIdx.x == 0);
    for (int i = lane; i < kH / 2; i += 32) {      // element pair (2i, 2i+1)
      uint32_t w = x32[i];
      uint32_t q = f32x2_to_e4m3x2(__fdiv_rn(__uint_as_float(w << 16), s),
                                   __fdiv_rn(__uint_as_float(w & 0xFFFF0000u), s));
      const int e = 2 * i, b = e >> 5, c = (e & 31) >> 3, o = e & 7;
      *reinterpret_cast<uint32_t*>(xh + (size_t)(c * kHBlocks + b) * 16 + o * 2) = e4m3x2_to_f16x2(q);
      if (writer) reinterpret_cast<uint16_t*>(p.xq + (size_t)t * kH)[i] = (uint16_t)q;
    }
    if (writer && lane == 0) p.sx[t] = s;
  }
  __syncthreads();
}

// ------------------------------------------------------------------ P1: router rows

__device__ void router_rows(const MoeParams& p, const LayerDesc& L, const uint8_t* smem) {
  const int M = p.M, E = p.E, G = gridDim.x;
  const int e0 = (int)((long long)blockIdx.x * E / G), e1 = (int)((long long)(blockIdx.x + 1) * E / G);
  const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(smem + smem_layout(M).xb);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = e0 + warp; e < e1; e += kWarps) {
    const uint4* wr = reinterpret_cast<const uint4*>(L.router_w + (size_t)e * kH);
    uint4 wv[10];
#pragma unroll
    for (int i = 0; i < 10; ++i) wv[i] = ldg_stream16(wr + 32 * i + lane);
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
      if (lane == 0) p.logits[(size_t)t * E + e] = acc;
    }
  }
}

// ------------------------------------------------------------------ P2: top-k + dedup

__device__ void route_tokens(const MoeParams& p, Tables& tb, int layer) {
  const int M = p.M, E = p.E, K = p.K;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < MDW_MAX_EXPERTS / 32) tb.bitmap[threadIdx.x] = 0;
  if (threadIdx.x == 0) tb.bad = 0;
  __syncthreads();
  for (int t = warp; t < M; t += kWarps) {
    const float* z = p.logits + (size_t)t * E;
    if (p.topk_override) {
      if (lane < K) {
        int id = p.topk_override[t * K + lane];
        bool ok = id >= 0 && id < E;
        for (int j = 0; j < K; ++j)
          if (j != lane && p.topk_override[t * K + j] == id) ok = false;
        if (!ok) { atomicExch(&tb.bad, 1); id = 0; }
        tb.ids[t * K + lane] = id;
        tb.gts[t * K + lane] = ld_cg_f32(z + id);
      }
      __syncwarp();
    } else {
      // k rounds of warp arg-max over E logits (16 per lane), ties -> lower index
      float v[MDW_MAX_EXPERTS / 32];
      const int per = (E + 31) / 32;
#pragma unroll
      for (int i = 0; i < MDW_MAX_EXPERTS / 32; ++i) {
        const int e = lane + 32 * i;
        v[i] = (i < per && e < E) ? ld_cg_f32(z + e) : -INFINITY;
      }
      for (int r = 0; r < K; ++r) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < MDW_MAX_EXPERTS / 32; ++i) {
          const int e = lane + 32 * i;
          if (e < E && beats(v[i], e, bv, bi)) { bv = v[i]; bi = e; }
        }
        warp_argmax(bv, bi);
        if ((bi & 31) == lane) {
#pragma unroll
          for (int i = 0; i < MDW_MAX_EXPERTS / 32; ++i)
            if (lane + 32 * i == bi) v[i] = -INFINITY;
        }
        if (lane == 0) { tb.ids[t * K + r] = bi; tb.gts[t * K + r] = bv; }
      }
      __syncwarp();
    }
    // gates: softmax over the selected logits
    if (lane == 0) {
      float mx = -INFINITY;
      for (int r = 0; r < K; ++r) mx = fmaxf(mx, tb.gts[t * K + r]);
      float sum = 0.f;
      float ex[MDW_MAX_TOPK];
      for (int r = 0; r < K; ++r) { ex[r] = expf(tb.gts[t * K + r] - mx); sum += ex[r]; }
      for (int r = 0; r < K; ++r) tb.gts[t * K + r] = ex[r] / sum;
    }
  }
  __syncthreads();
  if (tb.bad) return;
  // union bitmap
  for (int i = threadIdx.x; i < M * K; i += blockDim.x) {
    const int id = tb.ids[i];
    atomicOr(&tb.bitmap[id >> 5], 1u << (id & 31));
  }
  __syncthreads();
  const int first = p.has_shared ? 1 : 0;
  if (warp == 0) {
    // slot 0 = shared expert (if any), then the routed union ascending
    const uint32_t word = lane < MDW_MAX_EXPERTS / 32 ? tb.bitmap[lane] : 0u;
    int cnt = __popc(word), incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane < MDW_MAX_EXPERTS / 32) tb.wpre[lane] = incl - cnt;
    int pos = first + incl - cnt;
    uint32_t w = word;
    while (w) {
      const int b = __ffs(w) - 1;
      w &= w - 1;
      tb.cnt[pos] = 0;
      tb.slot_expert[pos++] = lane * 32 + b;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == 0) {
      tb.n_routed = total;
      tb.n_slots = total + first;
      if (p.has_shared) { tb.slot_expert[0] = -1; tb.cnt[0] = M; }
      tb.shared_slot = p.has_shared ? 0 : -1;
    }
  }
  __syncthreads();
  auto slot_of = [&](int e) {
    return first + tb.wpre[e >> 5] + __popc(tb.bitmap[e >> 5] & ((1u << (e & 31)) - 1u));
  };
  for (int i = threadIdx.x; i < M * K; i += blockDim.x) atomicAdd(&tb.cnt[slot_of(tb.ids[i])], 1);
  __syncthreads();
  if (warp == 0) {
    // exclusive scan of the per-slot pair counts (S <= 257)
    const int S = tb.n_slots;
    int carry = 0;
    for (int b0 = 0; b0 < S; b0 += 32) {
      const int s = b0 + lane;
      const int c = s < S ? tb.cnt[s] : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (s < S) tb.slot_begin[s] = carry + incl - c;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) { tb.slot_begin[S] = carry; tb.n_pairs = carry; }
  }
  __syncthreads();
  // pair of (t, r): slot-major, token-minor
  for (int i = threadIdx.x; i < M * K; i += blockDim.x) {
    const int t = i / K, e = tb.ids[i];
    int rank = 0;
    for (int t2 = 0; t2 < t; ++t2)
      for (int r2 = 0; r2 < K; ++r2) rank += (tb.ids[t2 * K + r2] == e);
    const int s = slot_of(e);
    const int q = tb.slot_begin[s] + rank;
    tb.pair_token[q] = t;
    tb.pair_slot[q] = s;
    tb.pair_gate[q] = tb.gts[i];
  }
  if (p.has_shared)
    for (int t = threadIdx.x; t < M; t += blockDim.x) {
      tb.pair_token[t] = t;
      tb.pair_slot[t] = 0;
      tb.pair_gate[t] = 1.0f;
    }
  __syncthreads();
  if (blockIdx.x == 0) {
    // publish the routing (inspection + optional outputs)
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
}

// ------------------------------------------------------------------ P3: gate/up + SwiGLU

// One warp computes gate_j and up_j of one expert for the tokens of one slot and writes
// h = silu(gate) * up. Lane l reads (16-byte chunks = one MX block each): gate blocks l,
// l+32; up blocks l, l+32; and block 64 + (l & 15) of gate (l < 16) or up (l >= 16).
template <int MAXM>
struct RowPairLoad {
  uint4 q[5];
  uint32_t s[5];
};

__device__ __forceinline__ int rp_block(int c, int lane) {
  return c < 4 ? (lane + 32 * (c & 1)) : 64 + (lane & 15);
}
__device__ __forceinline__ bool rp_is_up(int c, int lane) {
  return c < 4 ? (c >= 2) : (lane >= 16);
}

template <int MAXM>
__device__ __forceinline__ void rp_load(RowPairLoad<MAXM>& ld, const uint8_t* q13, const uint8_t* s13,
                                        int j, int lane) {
#pragma unroll
  for (int c = 0; c < 5; ++c) {
    const int row = j + (rp_is_up(c, lane) ? kI : 0);
    const int b = rp_block(c, lane);
    ld.q[c] = ldg_stream16(q13 + (size_t)row * kW13RowBytes + b * 16);
    ld.s[c] = ldg_stream_u8(s13 + (size_t)row * kHBlocks + b);
  }
}

template <int MAXM>
__device__ __forceinline__ void rp_compute(const RowPairLoad<MAXM>& ld, const uint8_t* smem,
                                           const uint32_t (&xr)[3][16], const int* toks, int m,
                                           const float* sx, float* hout /* h[pair0][j], stride kI */,
                                           int lane) {
  float g[MAXM], u[MAXM];
#pragma unroll
  for (int i = 0; i < MAXM; ++i) { g[i] = 0.f; u[i] = 0.f; }
#pragma unroll
  for (int c = 0; c < 5; ++c) {
    uint32_t w2[16];
    mx_block_decode(ld.q[c], w2);
    const float sc = e8m0_to_f32(ld.s[c]);
    const int b = rp_block(c, lane);
    const bool up = rp_is_up(c, lane);
    const int xi = c < 4 ? (c & 1) : 2;
#pragma unroll
    for (int i = 0; i < MAXM; ++i) {
      if (i < m) {
        float d;
        if (MAXM == 1) {
          d = dot32_f16(w2, xr[xi]);
        } else {
          const uint8_t* xh = smem + (size_t)toks[i] * kXhBytes;
          uint32_t x2[16];
#pragma unroll
          for (int pl = 0; pl < 4; ++pl) {
            uint4 v = *reinterpret_cast<const uint4*>(xh + (size_t)(pl * kHBlocks + b) * 16);
            x2[4 * pl] = v.x; x2[4 * pl + 1] = v.y; x2[4 * pl + 2] = v.z; x2[4 * pl + 3] = v.w;
          }
          d = dot32_f16(w2, x2);
        }
        if (up) u[i] = fmaf(d, sc, u[i]); else g[i] = fmaf(d, sc, g[i]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < MAXM; ++i) {
    if (i < m) {
      const float gs = warp_sum(g[i]) * sx[toks[i]];
      const float us = warp_sum(u[i]) * sx[toks[i]];
      if (lane == 0) hout[(size_t)i * kI] = gs / (1.0f + expf(-gs)) * us;
    }
  }
}

// Row pairs [r0, r1) of the virtual space; slot s covers [s*kI, (s+1)*kI).
template <int MAXM>
__device__ void gate_up_range(const MoeParams& p, const LayerDesc& L, const uint8_t* smem,
                              const Tables& tb, int r0, int r1, int slot_offset) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t xr[3][16];
  if (MAXM == 1) {
    const int blocks[3] = {lane, lane + 32, 64 + (lane & 15)};
#pragma unroll
    for (int k = 0; k < 3; ++k)
#pragma unroll
      for (int pl = 0; pl < 4; ++pl) {
        uint4 v = *reinterpret_cast<const uint4*>(smem + (size_t)(pl * kHBlocks + blocks[k]) * 16);
        xr[k][4 * pl] = v.x; xr[k][4 * pl + 1] = v.y; xr[k][4 * pl + 2] = v.z; xr[k][4 * pl + 3] = v.w;
      }
  }
  int rp = r0 + warp;
  if (rp >= r1) return;
  RowPairLoad<MAXM> cur, nxt;
  auto expert_ptrs = [&](int vrp, const uint8_t*& q13, const uint8_t*& s13, int& j, int& slot) {
    slot = vrp / kI + slot_offset;
    j = vrp % kI;
    const int e = tb.slot_expert[slot];
    if (e < 0) { q13 = L.sh_w13_q; s13 = L.sh_w13_s; }
    else {
      q13 = L.w13_q + (size_t)e * kRows13 * kW13RowBytes;
      s13 = L.w13_s + (size_t)e * kRows13 * kHBlocks;
    }
  };
  const uint8_t *q13, *s13;
  int j, slot;
  expert_ptrs(rp, q13, s13, j, slot);
  rp_load<MAXM>(cur, q13, s13, j, lane);
  while (true) {
    const int nrp = rp + kWarps;
    const uint8_t *nq13 = nullptr, *ns13 = nullptr;
    int nj = 0, nslot = 0;
    if (nrp < r1) {
      expert_ptrs(nrp, nq13, ns13, nj, nslot);
      rp_load<MAXM>(nxt, nq13, ns13, nj, lane);
    }
    const int pb = tb.slot_begin[slot], m = tb.slot_begin[slot + 1] - pb;
    rp_compute<MAXM>(cur, smem, xr, tb.pair_token + pb, m, tb.sx, p.h + (size_t)pb * kI + j, lane);
    if (nrp >= r1) break;
    cur = nxt;
    rp = nrp; j = nj; slot = nslot;
  }
}

// ------------------------------------------------------------------ P4: h quant + down

// Quantise pairs [q0, q0 + n) into the h-hat planes of shared memory (and, from block 0,
// into the workspace for inspection).
__device__ void quantise_pairs(const MoeParams& p, uint8_t* smem, Tables& tb, int q0, int n) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int k = warp; k < n; k += kWarps) {
    const int q = q0 + k;
    const float* hv = p.h + (size_t)q * kI;
    float v[kI / 32];
    float am = 0.f;
#pragma unroll
    for (int i = 0; i < kI / 32; ++i) { v[i] = ld_cg_f32(hv + lane + 32 * i); am = fmaxf(am, fabsf(v[i])); }
    am = warp_max(am);
    const float s = am > 0.f ? __fdiv_rn(am, kE4M3Max) : 1.0f;
    if (lane == 0) tb.sh[k] = s;
    uint8_t* hh = smem + smem_layout(p.M).hh + (size_t)k * kHhBytes;
#pragma unroll
    for (int i = 0; i < kI / 32; ++i) {
      const int e = lane + 32 * i, b = e >> 5, c = (e & 31) >> 3, o = e & 7;
      const uint32_t code = f32x2_to_e4m3x2(__fdiv_rn(v[i], s), 0.f) & 0xFF;
      const uint32_t f = e4m3x2_to_f16x2(code);
      *reinterpret_cast<uint16_t*>(hh + (size_t)(c * kIBlocks + b) * 16 + o * 2) = (uint16_t)f;
      if (blockIdx.x == 0) p.hq[(size_t)q * kI + e] = (uint8_t)code;
    }
    if (blockIdx.x == 0 && lane == 0) p.sh[q] = s;
  }
}

constexpr int kDownBatch = 8;   // (row, pair) items whose loads a warp keeps in flight

__device__ void down_combine(const MoeParams& p, const LayerDesc& L, uint8_t* smem, Tables& tb,
                             int layer) {
  const int M = p.M, G = gridDim.x;
  const int r0 = (int)((long long)blockIdx.x * kH / G), r1 = (int)((long long)(blockIdx.x + 1) * kH / G);
  const int nrows = r1 - r0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Smem sl = smem_layout(M);
  float* part = reinterpret_cast<float*>(smem + sl.part);
  float* yacc = reinterpret_cast<float*>(smem + sl.yacc);
  for (int i = threadIdx.x; i < M * kMaxRowsPerBlock; i += blockDim.x) yacc[i] = 0.f;
  const int NP = tb.n_pairs;
  for (int q0 = 0; q0 < NP; q0 += kPairChunk) {
    const int n = min(kPairChunk, NP - q0);
    __syncthreads();
    quantise_pairs(p, smem, tb, q0, n);
    __syncthreads();
    // items (row, pair) of this chunk; a warp takes kDownBatch consecutive items, issues
    // all their loads, then reduces each: lanes 0..23 hold one MX block of the row each
    const int items = nrows * n;
    for (int base = warp * kDownBatch; base < items; base += kWarps * kDownBatch) {
      uint4 w[kDownBatch];
      uint32_t sc[kDownBatch];
#pragma unroll
      for (int u = 0; u < kDownBatch; ++u) {
        const int it = base + u;
        w[u] = make_uint4(0, 0, 0, 0);
        sc[u] = 0;
        if (it < items && lane < kIBlocks) {
          const int k = it % n, r = r0 + it / n;
          const int e = tb.slot_expert[tb.pair_slot[q0 + k]];
          const uint8_t* q2 = e < 0 ? L.sh_w2_q : L.w2_q + (size_t)e * kH * kW2RowBytes;
          const uint8_t* s2 = e < 0 ? L.sh_w2_s : L.w2_s + (size_t)e * kH * kIBlocks;
          w[u] = ldg_stream16(q2 + (size_t)r * kW2RowBytes + lane * 16);
          sc[u] = ldg_stream_u8(s2 + (size_t)r * kIBlocks + lane);
        }
      }
#pragma unroll
      for (int u = 0; u < kDownBatch; ++u) {
        const int it = base + u;
        if (it >= items) break;
        const int k = it % n, rr = it / n;
        float d = 0.f;
        if (lane < kIBlocks) {
          const uint8_t* hh = smem + sl.hh + (size_t)k * kHhBytes;
          uint32_t x2[16];
#pragma unroll
          for (int pl = 0; pl < 4; ++pl) {
            uint4 v = *reinterpret_cast<const uint4*>(hh + (size_t)(pl * kIBlocks + lane) * 16);
            x2[4 * pl] = v.x; x2[4 * pl + 1] = v.y; x2[4 * pl + 2] = v.z; x2[4 * pl + 3] = v.w;
          }
          d = mx_block_dot(w[u], x2) * e8m0_to_f32(sc[u]);
        }
        d = warp_sum(d);
        if (lane == 0) part[k * kMaxRowsPerBlock + rr] = d * tb.sh[k] * tb.pair_gate[q0 + k];
      }
    }
    __syncthreads();
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
  for (int i = threadIdx.x; i < M * nrows; i += blockDim.x) {
    const int t = i / nrows, rr = i % nrows;
    const float y = yacc[t * kMaxRowsPerBlock + rr];
    const size_t o = (size_t)t * kH + r0 + rr;
    if (p.stack_mode) {
      const __nv_bfloat16* rin = resid_ptr(p, layer);
      __nv_bfloat16* rout = const_cast<__nv_bfloat16*>(resid_ptr(p, layer + 1));
      rout[o] = __float2bfloat16_rn(__bfloat162float(rin[o]) + y);
    } else {
      float v = y;
      if (p.residual) v += __bfloat162float(p.residual[o]);
      if (p.y_fp32) reinterpret_cast<float*>(p.y_out)[o] = v;
      else reinterpret_cast<__nv_bfloat16*>(p.y_out)[o] = __float2bfloat16_rn(v);
    }
  }
}

// ------------------------------------------------------------------ prefetch helpers

__device__ void prefetch_static(const MoeParams& p, const LayerDesc& L) {
  // this block's router rows and shared-expert slice of a layer (issued by one thread)
  if (threadIdx.x != 0) return;
  const int G = gridDim.x, E = p.E;
  const int e0 = (int)((long long)blockIdx.x * E / G), e1 = (int)((long long)(blockIdx.x + 1) * E / G);
  prefetch_l2(L.router_w + (size_t)e0 * kH, (uint32_t)((e1 - e0) * kH * 2));
  if (p.has_shared) {
    const int j0 = (int)((long long)blockIdx.x * kI / G), j1 = (int)((long long)(blockIdx.x + 1) * kI / G);
    for (int half = 0; half < 2; ++half) {
      const size_t row = (size_t)half * kI + j0;
      prefetch_l2(L.sh_w13_q + row * kW13RowBytes, (uint32_t)((j1 - j0) * kW13RowBytes));
      prefetch_l2(L.sh_w13_s + row * kHBlocks, (uint32_t)(((j1 - j0) * kHBlocks + 15) & ~15));
    }
  }
}

// L2 prefetch of the w13 rows (and scales) of virtual row pairs [a, b).
__device__ void prefetch_gate_up(const LayerDesc& L, const Tables& tb, int a, int b, int slot_offset) {
  if (threadIdx.x != 0) return;
  while (a < b) {
    const int slot = a / kI + slot_offset, j0 = a % kI;
    const int j1 = min(kI, j0 + (b - a));
    const int e = tb.slot_expert[slot];
    const uint8_t* q13 = e < 0 ? L.sh_w13_q : L.w13_q + (size_t)e * kRows13 * kW13RowBytes;
    const uint8_t* s13 = e < 0 ? L.sh_w13_s : L.w13_s + (size_t)e * kRows13 * kHBlocks;
    for (int half = 0; half < 2; ++half) {
      const size_t row = (size_t)half * kI + j0;
      prefetch_l2(q13 + row * kW13RowBytes, (uint32_t)((j1 - j0) * kW13RowBytes));
      const size_t sb = (row * kHBlocks) & ~(size_t)15;
      const size_t se = (((row + (j1 - j0)) * kHBlocks) + 15) & ~(size_t)15;
      prefetch_l2(s13 + sb, (uint32_t)(se - sb));
    }
    a += j1 - j0;
  }
}

__device__ void prefetch_down(const MoeParams& p, const LayerDesc& L, const Tables& tb) {
  const int G = gridDim.x;
  const int r0 = (int)((long long)blockIdx.x * kH / G), r1 = (int)((long long)(blockIdx.x + 1) * kH / G);
  for (int s = threadIdx.x; s < tb.n_slots; s += blockDim.x) {
    const int e = tb.slot_expert[s];
    const uint8_t* q2 = e < 0 ? L.sh_w2_q : L.w2_q + (size_t)e * kH * kW2RowBytes;
    const uint8_t* s2 = e < 0 ? L.sh_w2_s : L.w2_s + (size_t)e * kH * kIBlocks;
    prefetch_l2(q2 + (size_t)r0 * kW2RowBytes, (uint32_t)((r1 - r0) * kW2RowBytes));
    const size_t sb = (size_t)r0 * kIBlocks & ~(size_t)15;
    const size_t se = ((size_t)r1 * kIBlocks + 15) & ~(size_t)15;
    prefetch_l2(s2 + sb, (uint32_t)(se - sb));
  }
}

// ------------------------------------------------------------------ the kernel

template <int MAXM>
__global__ void __launch_bounds__(kThreads, 1) moe_persistent_kernel(const __grid_constant__ MoeParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  Tables& tb = *reinterpret_cast<Tables*>(smem + smem_layout(p.M).small);
  GridBarrier bar{p.hdr, 0};
  const int G = gridDim.x;
  for (int layer = 0; layer < p.L; ++layer) {
    const LayerDesc& L = p.layers[layer];
    prepare_input<MAXM>(p, layer, smem, tb);
    router_rows(p, L, smem);
    bar.arrive();                                                   // B1 (logits)
    if (p.has_shared) {
      // shared expert: static slice of its row pairs, needs only x-hat
      if (threadIdx.x == 0) { tb.slot_expert[0] = -1; tb.slot_begin[0] = 0; tb.slot_begin[1] = p.M; }
      if (threadIdx.x < p.M) tb.pair_token[threadIdx.x] = threadIdx.x;
      __syncthreads();
      const int j0 = (int)((long long)blockIdx.x * kI / G), j1 = (int)((long long)(blockIdx.x + 1) * kI / G);
      gate_up_range<MAXM>(p, L, smem, tb, j0, j1, 0);
    }
    if (!bar.wait()) return;
    route_tokens(p, tb, layer);
    __syncthreads();
    if (tb.bad) { if (threadIdx.x == 0) set_status(p.hdr, MDW_ERR_DEVICE_BOUNDS); return; }
    {
      const int first = p.has_shared ? 1 : 0;
      const long long PR = (long long)tb.n_routed * kI;
      const int a = (int)((long long)blockIdx.x * PR / G), b = (int)((long long)(blockIdx.x + 1) * PR / G);
      prefetch_gate_up(L, tb, a, b, first);
      prefetch_down(p, L, tb);
      gate_up_range<MAXM>(p, L, smem, tb, a, b, first);
    }
    bar.arrive();                                                   // B2 (h)
    if (p.stack_mode && layer + 1 < p.L) prefetch_static(p, p.layers[layer + 1]);
    if (!bar.wait()) return;
    down_combine(p, L, smem, tb, layer);
    if (p.stack_mode && layer + 1 < p.L) {
      if (!bar.sync()) return;                                      // B3 (r_{l+1})
    }
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

cudaError_t launch_moe(const MoeParams& p, cudaStream_t s) {
  if (p.M <= 1) return launch_t<1>(p, s);
  if (p.M <= 2) return launch_t<2>(p, s);
  if (p.M <= 4) return launch_t<4>(p, s);
  if (p.M <= 8) return launch_t<8>(p, s);
  return launch_t<16>(p, s);
}

}  // namespace mdw
