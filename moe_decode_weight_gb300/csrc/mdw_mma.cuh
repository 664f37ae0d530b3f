// Tensor-core and asynchronous-copy helpers shared by the MoE kernels: the m16n8k16 MMA,
// cp.async copies, and the block-column MMA steps that serve windows of up to four tokens.
#pragma once

#include "mdw_device.cuh"

namespace mdw {

// D += A x B on the tensor cores: m16n8k16, f16 operands (exact for E2M1 and E4M3 values),
// fp32 accumulation.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
               "{%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" :: "r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }
// ---- block-column MMA steps (at most two tokens per MMA tile) ----
// With one or two tokens, most of an m16n8 tile's eight columns would be idle. Instead the
// columns carry (token, block) pairs: column c = token c >> 2, block c & 3 of a four-block
// super-step. Lane (g, q) holds the whole 16-byte block sb + q of rows g and g + 8, so its
// k positions of every MMA come from that block; the B operand of column c is the token's
// x-hat on block sb + (c & 3) and zero elsewhere, so column c collects the (unscaled) dot
// product of each row with one block, and each lane scales its own columns by the rows'
// E8M0 scales in fp32. The MMAs need no per-block fresh accumulator and the weights no
// scaling, so the step costs about half the instructions of the token-column form.
//
// With three or four tokens a second m16n8 tile (NT = 2) carries tokens 2 and 3 the same way:
// tile j's column c = token 2j + (c >> 2), block c & 3; both tiles share the converted
// weights.
//
// bc_step: wr0 / wr1 = block sb + q of rows g and g + 8; xb[j] = the x-hat (f16, natural
// order) of token 2j + (g >> 2) on block sb + q when q == (g & 3), else null. Adds the partial
// dots of the lane's columns 2q, 2q + 1 of each tile (token 2j + (q >> 1), blocks
// sb + 2 (q & 1) + {0, 1}) into d[j].
template <int NT>
__device__ __forceinline__ void bc_step(uint4 wr0, uint4 wr1, const uint8_t* const (&xb)[NT], float (&d)[NT][4]) {
  const uint32_t A[4] = {wr0.x, wr0.y, wr0.z, wr0.w}, B[4] = {wr1.x, wr1.y, wr1.z, wr1.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t ha[4], hb[4];
    e2m1x8_to_f16x2x4(A[w], ha);
    e2m1x8_to_f16x2x4(B[w], hb);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      uint4 xv = make_uint4(0, 0, 0, 0);
      if (xb[j]) xv = *reinterpret_cast<const uint4*>(xb[j] + 16 * w);
      mma_16816(d[j], ha[0], hb[0], ha[1], hb[1], xv.x, xv.y);
      mma_16816(d[j], ha[2], hb[2], ha[3], hb[3], xv.z, xv.w);
    }
  }
}
// acc[0] (row g) and acc[1] (row g + 8) += the lane's two columns scaled by the rows' E8M0
// scales of those blocks (sa0/sa1: row g, blocks 2 (q & 1) + {0, 1} of the super-step; sb0 /
// sb1: row g + 8).
__device__ __forceinline__ void bc_scale_add(const float (&d)[4], uint32_t sa0, uint32_t sa1, uint32_t sb0,
                                             uint32_t sb1, float (&acc)[2]) {
  acc[0] = fmaf(e8m0_to_f32(sa0), d[0], acc[0]);
  acc[0] = fmaf(e8m0_to_f32(sa1), d[1], acc[0]);
  acc[1] = fmaf(e8m0_to_f32(sb0), d[2], acc[1]);
  acc[1] = fmaf(e8m0_to_f32(sb1), d[3], acc[1]);
}
// End of a block-column unit: per tile, the lane pairs (q, q ^ 1) add their blocks and lane
// q == 0 collects the tile's second token from lane 2; tile j's pair of tokens then moves to
// lane q == j, giving the token-column layout of an m16n8 result:
// r = {row g token 2q, row g token 2q+1, row g+8 token 2q, row g+8 token 2q+1} on lanes
// q < NT, zeros on the others.
template <int NT>
__device__ __forceinline__ void bc_finish(const float (&acc)[NT][2], int q, float (&r)[4]) {
  float rr[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const float a0 = acc[j][0] + __shfl_xor_sync(0xffffffffu, acc[j][0], 1);
    const float a1 = acc[j][1] + __shfl_xor_sync(0xffffffffu, acc[j][1], 1);
    rr[j][0] = a0;
    rr[j][1] = __shfl_xor_sync(0xffffffffu, a0, 2);
    rr[j][2] = a1;
    rr[j][3] = __shfl_xor_sync(0xffffffffu, a1, 2);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float v = (q == 0) ? rr[0][i] : 0.f;
    if (NT > 1) {
      const float t = __shfl_up_sync(0xffffffffu, rr[NT > 1 ? 1 : 0][i], 1);
      if (q == 1) v = t;
    }
    r[i] = v;
  }
}

}  // namespace mdw
