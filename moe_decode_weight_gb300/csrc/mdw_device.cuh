// Device helpers shared by the decode kernels: number formats, streaming loads, L2
// prefetch, warp reductions, the bounded grid barrier and the device status word.
//
// Formats (the pages name them only: "Humming MXFP4 kernels compile at run time for the
// model's real shapes" -- W4A8 MXFP4; "Online FP8 quantization halves the LM head weight
// reads" -- FP8): E2M1 elements with an E8M0 scale per 32 K elements, E4M3 activations
// and head weights, bf16 hidden states. Conversions use the sm_100-family hardware
// instructions (cvt ... e2m1x2 / e4m3x2 / satfinite), which round to nearest even.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "moe_decode_weight.h"

namespace mdw {

constexpr int kH = MDW_HIDDEN;          // 2560
constexpr int kI = MDW_INTER;           // 768
constexpr int kBlk = 32;                // MX block (K elements per E8M0 scale)
constexpr int kHBlocks = kH / kBlk;     // 80
constexpr int kIBlocks = kI / kBlk;     // 24
constexpr float kE4M3Max = 448.0f;

// Workspace header words (uint32), zeroed by the host at the start of every call.
enum HeaderWord : int {
  kHdrStatus = 0,     // mdw_status recorded by kernels (first error wins)
  kHdrBarrier = 1,    // grid-barrier arrival counter
  kHdrSlots = 2,      // S: expert slots of the last layer
  kHdrPairs = 3,      // P: (token, expert) pairs of the last layer
  kHdrRouted = 4,     // routed slots of the last layer
  kHdrDoneCtr = 5,    // last-group-done counter of the LM head
  kHdrHeadGroups = 16,  // [16 + g]: blocks of LM-head group g done (16 words)
  kHdrUnions = 64,    // [64 + l]: routed union size of layer l (stack)
  kHdrWords = 256
};

// ------------------------------------------------------------------ status

__device__ __forceinline__ void set_status(uint32_t* hdr, mdw_status s) {
  atomicCAS(hdr + kHdrStatus, 0u, (uint32_t)s);
}

// ------------------------------------------------------------------ loads

// 16-byte streaming load that bypasses L1 (weights are read once per call).
__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg_stream_u8(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
// Coherent loads of data written earlier in the same kernel by other blocks (after a
// grid barrier): must not use the non-coherent path.
__device__ __forceinline__ float ld_cg_f32(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 ld_cg16(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// Fire-and-forget prefetch of [p, p + bytes) into L2 (bytes multiple of 16, p 16-aligned).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  if (bytes == 0) return;
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(bytes) : "memory");
}

// ------------------------------------------------------------------ formats

// Two E2M1 codes (one byte: low nibble = element 0) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(r) : "r"(byte));
  return r;
}
// Two E4M3 codes (16 bits: low byte = element 0) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)two));
  return r;
}
// fp32 pair -> two E4M3 codes (low byte = a), round to nearest even, saturating.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}
// Four E2M1 code pairs (the four bytes of w, byte 0 first) -> four f16x2 (exact).
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&h)[4]) {
  asm("{ .reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %4;"
      " cvt.rn.f16x2.e2m1x2 %0, b0; cvt.rn.f16x2.e2m1x2 %1, b1;"
      " cvt.rn.f16x2.e2m1x2 %2, b2; cvt.rn.f16x2.e2m1x2 %3, b3; }"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]) : "r"(w));
}
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// E8M0 scales whose power of two, applied to any E2M1 value in f16, stays exact: s in
// [113, 140] gives 2^-14 .. 2^13 (a normal f16), and every product E2M1 x 2^(s-127) lies in
// [2^-15, 6 * 2^13], a multiple of 2^-24 below 65504. All four bytes of `four` checked.
__device__ __forceinline__ bool e8m0x4_f16_exact(uint32_t four) {
  return __vcmpleu4(__vsub4(four, 0x71717171u), 0x1B1B1B1Bu) == 0xFFFFFFFFu;
}
// f16x2 with 2^(s-127) in both halves, for s in [113, 140] (exponent field s - 112).
__device__ __forceinline__ uint32_t e8m0_to_f16x2_pow2(uint32_t s) { return (s - 112u) * 0x04000400u; }

// E8M0 scale byte -> fp32 2^(s-127) (s = 0 gives 2^-127, a subnormal; 255 gives NaN).
__device__ __forceinline__ float e8m0_to_f32(uint32_t s) {
  return s == 0 ? __uint_as_float(0x00400000u) : (s == 255 ? __uint_as_float(0x7FC00000u)
                                                           : __uint_as_float(s << 23));
}

// acc + w.lo * x.lo + w.hi * x.hi with f16 operands, exact products, fp32 accumulation.
__device__ __forceinline__ float fma2_f16_f32(uint32_t w2, uint32_t x2, float acc) {
  float d;
  asm("{ .reg .f16 wl, wh, xl, xh; .reg .f32 t;"
      " mov.b32 {wl, wh}, %1; mov.b32 {xl, xh}, %2;"
      " fma.rn.f32.f16 t, wl, xl, %3; fma.rn.f32.f16 %0, wh, xh, t; }"
      : "=f"(d) : "r"(w2), "r"(x2), "f"(acc));
  return d;
}

// Dot product of one MX block (16 bytes = 32 E2M1 codes) with 32 f16 activations
// (16 f16x2 words), unscaled, fp32 accumulation in two chains.
__device__ __forceinline__ float mx_block_dot(uint4 q, const uint32_t* x2) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int b = 0; b < 4; b += 2) {
      a0 = fma2_f16_f32(e2m1x2_to_f16x2((w[i] >> (8 * b)) & 0xFF), x2[4 * i + b], a0);
      a1 = fma2_f16_f32(e2m1x2_to_f16x2((w[i] >> (8 * b + 8)) & 0xFF), x2[4 * i + b + 1], a1);
    }
  }
  return a0 + a1;
}

// The same block decoded once into 16 f16x2 words (for reuse across several tokens).
__device__ __forceinline__ void mx_block_decode(uint4 q, uint32_t* w2) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int b = 0; b < 4; ++b) w2[4 * i + b] = e2m1x2_to_f16x2((w[i] >> (8 * b)) & 0xFF);
}
__device__ __forceinline__ float dot32_f16(const uint32_t* w2, const uint32_t* x2) {
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    a0 = fma2_f16_f32(w2[i], x2[i], a0);
    a1 = fma2_f16_f32(w2[i + 1], x2[i + 1], a1);
  }
  return a0 + a1;
}

// ------------------------------------------------------------------ warp helpers

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Ordering of (value, index) candidates: larger value first, then lower index.
__device__ __forceinline__ bool beats(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Warp-wide arg-max of one candidate per lane under `beats`; every lane gets the winner.
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, v, o);
    int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (beats(ov, oi, v, i)) { v = ov; i = oi; }
  }
}

// ------------------------------------------------------------------ tagged words

// A value published for other blocks travels in an 8-byte word with the producing layer's tag
// in the high half (an aligned 64-bit access is single-copy atomic), so the consumer's poll of
// the word is also its read of the value: no barrier, no second round trip. The words are
// zeroed before every launch and tags start at 1. A poll requests every word it waits for
// before it checks any (a load whose predicate depended on the previous word's check would
// cost one L2 round trip per word).
__device__ __forceinline__ uint64_t tagged(uint32_t payload, uint32_t tag) { return ((uint64_t)tag << 32) | payload; }
__device__ __forceinline__ uint32_t tag_of(uint64_t w) { return (uint32_t)(w >> 32); }
__device__ __forceinline__ void st_word(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_word(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ void ld_word2(const uint64_t* p, uint64_t& a, uint64_t& b) {
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p));
}

// ------------------------------------------------------------------ grid barrier

__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_volatile_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.volatile.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Default spin budget of one inter-block wait, in clock64 cycles (~0.5 s at 2 GHz).
constexpr long long kSpinBudget = 1000000000LL;

// Grid-wide barrier over a monotonically increasing arrival counter (zeroed by the host
// before each launch). `seq` counts the barriers this launch has passed. Split into
// arrive (release) and wait (acquire) so a block can do independent work in between.
// A wait that exceeds the budget records MDW_ERR_TIMEOUT and reports failure; callers
// then leave the kernel. All blocks must be co-resident (cooperative launch).
struct GridBarrier {
  uint32_t* hdr;
  uint32_t seq;
  long long budget;             // clock64 cycles one wait may spin before it gives up
  __device__ void arrive() {
    __syncthreads();
    if (threadIdx.x == 0) red_release_add(hdr + kHdrBarrier, 1u);
    ++seq;
  }
  // returns false on timeout or if another block already recorded a failure
  __device__ bool wait() {
    __shared__ int ok;
    if (threadIdx.x == 0) {
      const uint32_t target = seq * gridDim.x;
      int good = 1;
      long long t0 = clock64();
      while ((int)(ld_acquire(hdr + kHdrBarrier) - target) < 0) {
        if (ld_volatile_u32(hdr + kHdrStatus) != 0) { good = 0; break; }
        if (clock64() - t0 > budget) { set_status(hdr, MDW_ERR_TIMEOUT); good = 0; break; }
      }
      ok = good;
    }
    __syncthreads();
    return ok != 0;
  }
  __device__ bool sync() { arrive(); return wait(); }
};

}  // namespace mdw
