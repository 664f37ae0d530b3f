// Streaming W4A8 MXFP4 MoE decode kernel for windows of up to four tokens: router, top-k,
// expert dedup, gate/up + SwiGLU, h quantisation, down projection and weighted combine, for
// one layer or a stack of layers with a pre-norm bf16 residual stream.
//
// Method (page titles and sections):
//   "Three MoE Inference Optimizations NVIDIA Measured on DGX Spark",
//   - "Decoding was memory-bound on a 124-billion-parameter model at batch size 1": each MoE
//     layer routes a token to 8 of 512 experts plus one shared expert, and decode time is
//     weight reads: the design goal is to keep HBM streaming the selected experts' bytes;
//   - "Humming MXFP4 kernels compile at run time for the model's real shapes": W4A8 MXFP4
//     experts, hidden 2560, moe_intermediate 768, compiled in for these shapes;
//   - "Multi-token prediction turns each verification into four tokens": a window of M
//     tokens touches the union of their experts, each read once for all of them.
//
// Execution model (GB300: one block of 384 threads per SM, co-resident by a cooperative
// launch). Blocks never meet at a grid barrier. Every value one block produces for the
// others is published as 8-byte words that carry the producing layer's tag next to the
// payload (the aligned 64-bit access is single-copy atomic), so a consumer's poll of the
// words is also its read of the data, with one L2 round trip:
//   xr  the residual r_l, two bf16 per word (stack, layers >= 1);
//   xz  the router logits, one fp32 per word;
//   xh  the SwiGLU output h of every (token, expert) pair, one fp32 per word.
// The exchange buffers are zeroed by the host before every launch and tags start at 1, so
// stale words never match. One buffer of each suffices: a block can only produce layer
// l + 1's words after every block has consumed layer l's (each exchange depends on the one
// before it through every block).
//
// Per layer, every block:
//   P0  reads r_l (tagged poll) or the input x; RMSNorm (stack); per-token E4M3 x-hat in f16;
//       the router weights of its rows were loaded into registers before the poll;
//   P1  its router rows -> xz;
//   P2  polls xz; top-k and dedup per token, redundantly in every block (slot 0 = the shared
//       expert, then the union ascending; pairs slot-major, token-minor);
//   P3  its contiguous share of the (slot, 8-row-pair tile) space, then its output rows of
//       every slot's W2, stream through a ring of shared-memory slots filled by bulk async
//       copies (cp.async.bulk, completion counted on an mbarrier per slot): the whole ring is
//       requested at once and a slot is refilled by the warp that finishes its last unit, so
//       the block keeps up to the ring's size of weight bytes in flight. A gate/up tile is
//       cut into 10 K parts run by different warps on the tensor cores (block-column m16n8k16
//       MMAs); the last warp of a tile sums the parts in order, applies SwiGLU and publishes
//       h -> xh;
//   P4  polls xh of every pair; quantises each pair's h (amax / 448) into f16 h-hat; bulk L2
//       prefetch of the next layer's router rows and shared-expert slice meanwhile;
//   P5  down projection of its output rows for every slot from the ring (MMA for 16 rows,
//       CUDA cores for the rest), combine in a fixed pair order (+ residual); stack: r_{l+1}
//       = bf16(r_l + y) -> xr.
// Every wait (tag polls and mbarrier waits) is bounded: when it runs out the block records
// MDW_ERR_TIMEOUT, waits (bounded) for its own copies in flight and leaves; every block
// leaves at its next wait once the status word is set.
#include "mdw_device.cuh"
#include "mdw_internal.h"
#include "mdw_mma.cuh"

namespace mdw {
namespace {

constexpr int kW13RowBytes = kH / 2;            // 1280
constexpr int kW2RowBytes = kI / 2;             // 384
constexpr int kXhBytes = kH * 2 + 64;           // f16 x-hat per token (natural order, padded)
constexpr int kHhBytes = kI * 2 + 64;           // f16 h-hat per pair
constexpr int kTileRP = 8;                      // row pairs (gate row j + up row j) per tile
constexpr int kTilesPerSlot = kI / kTileRP;     // 96
constexpr int kGuParts = 10;                    // K parts of a tile (8 MX blocks each)
constexpr int kDnParts = 3;                     // K parts of a down slot (8 of the 24 blocks)
constexpr int kTileW = kTileRP * kW13RowBytes;  // 10240: the gate (or up) rows of a tile
constexpr int kTileS = kTileRP * kHBlocks;      // 640: their scales
constexpr int kSlotBytes = 22528;               // ring slot: one tile or up to 3 down chunks
constexpr int kMaxRows = 32;                    // output rows per block (H / grid, even)
constexpr int kMaxSlots = 4 * MDW_MAX_TOPK + 1; // slots of a window of <= 4 tokens
constexpr int kMaxPairs = 4 * (MDW_MAX_TOPK + 1);
static_assert(2 * kTileW + 2 * kTileS <= kSlotBytes, "a tile must fit a ring slot");

__host__ __device__ constexpr int ring_slots(int maxm) { return maxm <= 2 ? 6 : 5; }

// ------------------------------------------------------------------ phase trace

// Built only with -DMDW_TRACE (the profiling library, never the product build): thread 0 of
// every block records %globaltimer at each phase boundary of every layer.
#ifdef MDW_TRACE
// clock64 at each phase boundary of each layer (thread 0), kept in shared memory during the
// launch and written out at its end, so the stamps add no global traffic
constexpr int kSTraceLayers = 64, kSTracePoints = 20, kSTraceBlocks = 256;
__device__ unsigned long long g_strace[kSTraceLayers * kSTracePoints * kSTraceBlocks];
__shared__ unsigned long long s_strace[kSTraceLayers * kSTracePoints];
#define STRACE(layer, point)                                                                   \
  do {                                                                                         \
    if (threadIdx.x == 0 && (layer) < kSTraceLayers) s_strace[(layer) * kSTracePoints + (point)] = clock64(); \
  } while (0)
#define STRACE_FLUSH(nl)                                                                       \
  do {                                                                                         \
    __syncthreads();                                                                           \
    if (blockIdx.x < kSTraceBlocks)                                                            \
      for (int i_ = threadIdx.x; i_ < (nl) * kSTracePoints && i_ < kSTraceLayers * kSTracePoints; i_ += blockDim.x) \
        g_strace[(i_ / kSTracePoints * kSTracePoints + i_ % kSTracePoints) * kSTraceBlocks + blockIdx.x] = s_strace[i_]; \
  } while (0)
#else
#define STRACE(layer, point) do { } while (0)
#define STRACE_FLUSH(nl) do { } while (0)
#endif

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
               : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
// Orders this thread's (and, after a barrier, the block's) earlier generic accesses to shared
// memory before later asynchronous-proxy (bulk copy) writes to it.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// [dst, dst + bytes) <- [src, src + bytes): one bulk asynchronous copy (16-byte aligned, a
// multiple of 16 bytes), its bytes counted on `bar`
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void st_word(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}
// Poll loads. A poll issues all of its loads before it looks at any of them: a load whose
// predicate depended on the previous word's check would wait a full L2 round trip per word.
__device__ __forceinline__ uint64_t ld_word(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ void ld_word2(const uint64_t* p, uint64_t& a, uint64_t& b) {
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p));
}
__device__ __forceinline__ uint64_t tagged(uint32_t payload, uint32_t tag) {
  return ((uint64_t)tag << 32) | payload;
}
__device__ __forceinline__ uint32_t tag_of(uint64_t w) { return (uint32_t)(w >> 32); }

// ------------------------------------------------------------------ shared memory

template <int MAXM>
struct SLayout {
  static constexpr int NS = ring_slots(MAXM);
  static constexpr int NT = MAXM <= 2 ? 1 : 2;                      // block-column tiles
  static constexpr size_t ring = 0;                                 // [NS][kSlotBytes]
  static constexpr size_t xb = ring + (size_t)NS * kSlotBytes;     // bf16 x [M][H] (router)
  static constexpr size_t xh = xb + (size_t)MAXM * kH * 2;          // f16 x-hat [M][kXhBytes]
  static constexpr size_t r1_end = xh + (size_t)MAXM * kXhBytes;
  static constexpr size_t hh = xb;                                  // f16 h-hat [P][kHhBytes] (down phase)
  static constexpr size_t hh_end = hh + (size_t)(MAXM * (MDW_MAX_TOPK + 1)) * kHhBytes;
  static constexpr size_t part = ((r1_end > hh_end ? r1_end : hh_end) + 15) & ~(size_t)15;
  // gate/up K-part results: [NS][kGuParts][8 g][NT q] float4
  static constexpr size_t dres = part + (size_t)NS * kGuParts * 8 * NT * 16;
  // down results: [P][kDnParts][16] fp32 (MMA rows), then leftover rows [P][kMaxRows - 16]
  static constexpr size_t dleft = dres + (size_t)kMaxPairs * kDnParts * 16 * 4;
  static constexpr size_t rres = dleft + (size_t)kMaxPairs * (kMaxRows - 16) * 4;   // [M][kMaxRows] fp32
  static constexpr size_t cand = rres + (size_t)MAXM * kMaxRows * 4;               // top-k scratch
  static constexpr size_t zrow = cand + (size_t)MAXM * 128 * 8;                    // polled logits [M][E] fp32
  static constexpr size_t tabs = zrow + (size_t)MAXM * MDW_MAX_EXPERTS * 4;
  static constexpr size_t bars = tabs + 4096;                                      // mbarriers, counters
  static constexpr size_t total = bars + (size_t)NS * 16 + 16 + 16;   // + the router barrier
};

struct STables {
  int ids[4 * MDW_MAX_TOPK];
  float gts[4 * MDW_MAX_TOPK];
  uint32_t bitmap[MDW_MAX_EXPERTS / 32];
  int wpre[MDW_MAX_EXPERTS / 32];
  int slot_expert[kMaxSlots];
  int slot_begin[kMaxSlots + 1];
  int cnt[kMaxSlots];
  int pair_token[kMaxPairs];
  float pair_gate[kMaxPairs];
  float sh[kMaxPairs];
  float sx[4];
  float inv_rms[4];
  float red[4 * (kH / 256)];                    // per-(token, 256-element chunk group) partials
  int n_slots, n_routed, n_pairs, bad, fail;
};
static_assert(sizeof(STables) <= 4096, "tables exceed their shared-memory region");

// Per-block pipeline state (the pointers and `seq` are identical in all threads).
struct Ring {
  uint64_t* full;        // [NS] mbarriers: one phase per item requested into the slot
  uint64_t* rbar;        // mbarrier of the router rows' copy (one phase per layer)
  int* done;             // [NS] finished units of the item in the slot
  uint32_t* item;        // [NS] ring sequence number of the item last requested into the slot
  uint32_t seq;          // items of all layers so far
};
constexpr uint32_t kNoItem = 0xFFFFFFFFu;

__device__ __forceinline__ uint32_t ld_volatile_shared(const uint32_t* p) {
  return *reinterpret_cast<const volatile uint32_t*>(p);
}

// ------------------------------------------------------------------ bounded waits

// Spin on `bar` until phase `parity` completes; false (status recorded) on timeout or when
// another block failed.
__device__ __forceinline__ bool wait_full(uint64_t* bar, uint32_t parity, const MoeParams& p) {
  if (mbar_test(bar, parity)) return true;
  const long long t0 = clock64();
  int n = 0;
  while (!mbar_test(bar, parity)) {
    if ((++n & 63) == 0 && ld_volatile_u32(p.hdr + kHdrStatus) != 0) return false;
    if (clock64() - t0 > p.spin_budget) { set_status(p.hdr, MDW_ERR_TIMEOUT); return false; }
  }
  return true;
}

// Waits until item g (ring sequence number) has landed in its slot. A slot's mbarrier
// completes one phase per item and a parity wait only tells phases two apart, so the wait
// first makes sure the slot already holds item g: then the previous item of the slot has
// completed (it was consumed before the slot was refilled) and the item after it cannot be
// requested before this warp's unit of item g is done, so the parity is unambiguous.
template <int NS>
__device__ __forceinline__ bool wait_item(const Ring& rg, uint32_t g, const MoeParams& p) {
  const int s = g % NS;
  if (ld_volatile_shared(rg.item + s) != g) {
    const long long t0 = clock64();
    int n = 0;
    while (ld_volatile_shared(rg.item + s) != g) {
      if ((++n & 63) == 0 && ld_volatile_u32(p.hdr + kHdrStatus) != 0) return false;
      if (clock64() - t0 > p.spin_budget) { set_status(p.hdr, MDW_ERR_TIMEOUT); return false; }
    }
  }
  return wait_full(rg.full + s, (g / NS) & 1, p);
}

// ------------------------------------------------------------------ items of the ring

// The block's gate/up tiles are tiles [t0, t0 + n_gu) of the slot-major tile space
// (slot = t / 96, row pairs 8 (t % 96) .. +8); then its down chunks, `dps` slots per item.
struct Plan {
  int t0, n_gu;          // gate/up tiles
  int dps, n_dn;         // down slots per item, down items
  int r0, nrows;         // output rows
  int n_items;
  uint32_t base;         // ring sequence number of item 0 of this layer
};

__device__ __forceinline__ int item_units(const Plan& pl, int it, int n_slots) {
  if (it < pl.n_gu) return kGuParts;
  const int s0 = (it - pl.n_gu) * pl.dps;
  const int ns = min(pl.dps, n_slots - s0);
  return ns * (kDnParts + (pl.nrows > 16 ? 1 : 0));
}

// Requests item `it` into its ring slot (one thread).
template <int MAXM>
__device__ void issue_item(const MoeParams& p, const LayerDesc& L, const STables& tb, const Plan& pl, Ring& rg,
                           uint8_t* smem, int it) {
  using SL = SLayout<MAXM>;
  const uint32_t g = pl.base + it;
  const int s = g % SL::NS;
  uint8_t* dst = smem + SL::ring + (size_t)s * kSlotBytes;
  uint64_t* bar = rg.full + s;
  *reinterpret_cast<volatile uint32_t*>(rg.item + s) = g;
  fence_proxy_async();
  if (it < pl.n_gu) {
    const int t = pl.t0 + it, slot = t / kTilesPerSlot, j0 = (t % kTilesPerSlot) * kTileRP;
    const int e = tb.slot_expert[slot];
    const uint8_t* q13 = e < 0 ? L.sh_w13_q : L.w13_q + (size_t)e * (2 * kI) * kW13RowBytes;
    const uint8_t* s13 = e < 0 ? L.sh_w13_s : L.w13_s + (size_t)e * (2 * kI) * kHBlocks;
    mbar_arrive_expect_tx(bar, 2 * kTileW + 2 * kTileS);
    bulk_copy(dst, q13 + (size_t)j0 * kW13RowBytes, kTileW, bar);
    bulk_copy(dst + kTileW, q13 + (size_t)(kI + j0) * kW13RowBytes, kTileW, bar);
    bulk_copy(dst + 2 * kTileW, s13 + (size_t)j0 * kHBlocks, kTileS, bar);
    bulk_copy(dst + 2 * kTileW + kTileS, s13 + (size_t)(kI + j0) * kHBlocks, kTileS, bar);
  } else {
    const int s0 = (it - pl.n_gu) * pl.dps, ns = min(pl.dps, tb.n_slots - s0);
    const uint32_t qb = pl.nrows * kW2RowBytes, sb = pl.nrows * kIBlocks;
    mbar_arrive_expect_tx(bar, ns * (qb + sb));
    for (int c = 0; c < ns; ++c) {
      const int e = tb.slot_expert[s0 + c];
      const uint8_t* q2 = e < 0 ? L.sh_w2_q : L.w2_q + (size_t)e * kH * kW2RowBytes;
      const uint8_t* s2 = e < 0 ? L.sh_w2_s : L.w2_s + (size_t)e * kH * kIBlocks;
      uint8_t* d = dst + (size_t)c * (qb + sb);
      bulk_copy(d, q2 + (size_t)pl.r0 * kW2RowBytes, qb, bar);
      bulk_copy(d + qb, s2 + (size_t)pl.r0 * kIBlocks, sb, bar);
    }
  }
}

// After a failure: wait (bounded by the default budget, not the caller's) until the last
// item requested into every slot has landed (the slot's earlier items have), and the layer's
// router-row copy, so no copy writes shared memory after the block exits. Every thread of the
// block calls it after the same block barrier.
template <int MAXM>
__device__ void drain_ring(const Ring& rg, int layer, bool router_copy) {
  using SL = SLayout<MAXM>;
  __syncthreads();
  if (threadIdx.x != 0) return;
  for (int s = 0; s < SL::NS; ++s) {
    const uint32_t g = ld_volatile_shared(rg.item + s);
    if (g == kNoItem) continue;
    const long long t0 = clock64();
    while (!mbar_test(rg.full + s, (g / SL::NS) & 1))
      if (clock64() - t0 > kSpinBudget) break;
  }
  if (!router_copy) return;
  const long long t0 = clock64();
  while (!mbar_test(rg.rbar, layer & 1))
    if (clock64() - t0 > kSpinBudget) break;
}

// ------------------------------------------------------------------ P0: input

// Token rows of r_l (or x) -> bf16 x in shared memory: layer mode or the stack's first layer
// read the caller's buffer; later layers poll xr (tag l). Then RMSNorm (stack), amax, scale,
// x-hat. `rres` keeps the block's output rows of r_l for the residual add.
template <int MAXM>
__device__ bool prepare_input(const MoeParams& p, int layer, uint8_t* smem, STables& tb, const Plan& pl) {
  using SL = SLayout<MAXM>;
  const int M = p.M, lane = threadIdx.x & 31;
  constexpr int CPT = kH / 8;                     // 8-element chunks per token (320)
  uint4* xb4 = reinterpret_cast<uint4*>(smem + SL::xb);
  float* rres = reinterpret_cast<float*>(smem + SL::rres);
  const bool poll = p.stack_mode && layer > 0;
  const uint4* src = reinterpret_cast<const uint4*>(p.stack_mode ? p.r0 : p.x_in);
  // 1. rows into shared memory (a chunk = 8 bf16 = 4 tagged words when polled)
  if (poll) {
    // every chunk of this thread is requested before any is checked; missing chunks are
    // requested again together
    constexpr int NCH = (MAXM * CPT + kThreads - 1) / kThreads;
    const uint64_t* xr = p.xr;
    const uint32_t tag = (uint32_t)layer;
    uint32_t want = 0;
#pragma unroll
    for (int k = 0; k < NCH; ++k)
      if ((int)threadIdx.x + k * kThreads < M * CPT) want |= 1u << k;
    long long t0 = 0;
    bool ok = true;
    for (int n = 0; want != 0; ++n) {
      uint64_t w[NCH][4];
#pragma unroll
      for (int k = 0; k < NCH; ++k) {
        const size_t c = threadIdx.x + (size_t)k * kThreads;
        if (want & (1u << k)) {
          ld_word2(xr + 4 * c, w[k][0], w[k][1]);
          ld_word2(xr + 4 * c + 2, w[k][2], w[k][3]);
        }
      }
      uint32_t got = 0;
#pragma unroll
      for (int k = 0; k < NCH; ++k) {
        const int c = threadIdx.x + k * kThreads;
        if ((want & (1u << k)) && tag_of(w[k][0]) == tag && tag_of(w[k][1]) == tag && tag_of(w[k][2]) == tag &&
            tag_of(w[k][3]) == tag) {
          xb4[c] = make_uint4((uint32_t)w[k][0], (uint32_t)w[k][1], (uint32_t)w[k][2], (uint32_t)w[k][3]);
          got |= 1u << k;
        }
      }
      want &= ~got;
      if (want == 0) break;
      if (n == 0) t0 = clock64();
      if ((n & 15) == 15 && ld_volatile_u32(p.hdr + kHdrStatus) != 0) { ok = false; break; }
      if (clock64() - t0 > p.spin_budget) { set_status(p.hdr, MDW_ERR_TIMEOUT); ok = false; break; }
    }
    if (!ok) atomicExch(&tb.fail, 1);
  } else {
    for (int c = threadIdx.x; c < M * CPT; c += blockDim.x) xb4[c] = ld_cg16(src + c);
  }
  __syncthreads();
  if (tb.fail) return false;
  // the block's output rows of r_l (stack) or of the residual input (layer mode), fp32
  if (p.stack_mode) {
    const __nv_bfloat16* xbh = reinterpret_cast<const __nv_bfloat16*>(smem + SL::xb);
    for (int i = threadIdx.x; i < M * pl.nrows; i += blockDim.x) {
      const int t = i / pl.nrows, rr = i % pl.nrows;
      rres[t * kMaxRows + rr] = __bfloat162float(xbh[(size_t)t * kH + pl.r0 + rr]);
    }
  } else if (p.residual) {
    for (int i = threadIdx.x; i < M * pl.nrows; i += blockDim.x) {
      const int t = i / pl.nrows, rr = i % pl.nrows;
      rres[t * kMaxRows + rr] = __bfloat162float(p.residual[(size_t)t * kH + pl.r0 + rr]);
    }
  }
  // 2. per-token reductions in a fixed order (every block derives bit-identical x and x-hat):
  //    a warp's 32 chunks share one token; the 10 warp partials are combined in order
  auto reduce = [&](bool sq) {
    for (int c = threadIdx.x; c < M * CPT; c += blockDim.x) {
      const uint4 v = xb4[c];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      float r = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float a = __uint_as_float(w[k] << 16), b = __uint_as_float(w[k] & 0xFFFF0000u);
        if (sq) { r = fmaf(a, a, r); r = fmaf(b, b, r); }
        else r = fmaxf(r, fmaxf(fabsf(a), fabsf(b)));
      }
      r = sq ? warp_sum(r) : warp_max(r);
      if (lane == 0) tb.red[c / 32] = r;
    }
    __syncthreads();
  };
  if (p.stack_mode) {
    reduce(true);
    if (threadIdx.x < M) {
      float ss = 0.f;
      for (int g = 0; g < CPT / 32; ++g) ss += tb.red[threadIdx.x * (CPT / 32) + g];
      tb.inv_rms[threadIdx.x] = rsqrtf(ss / (float)kH + 1e-6f);
    }
    __syncthreads();
    for (int c = threadIdx.x; c < M * CPT; c += blockDim.x) {
      const float inv = tb.inv_rms[c / CPT];
      const uint4 v = xb4[c];
      uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 r2 = __floats2bfloat162_rn(__uint_as_float(w[k] << 16) * inv,
                                                        __uint_as_float(w[k] & 0xFFFF0000u) * inv);
        w[k] = *reinterpret_cast<const uint32_t*>(&r2);
      }
      xb4[c] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncthreads();
  }
  reduce(false);
  // 3. scale = amax / 448 (IEEE division), codes = RNE-saturating E4M3 of x / scale
  if (threadIdx.x < M) {
    float am = 0.f;
    for (int g = 0; g < CPT / 32; ++g) am = fmaxf(am, tb.red[threadIdx.x * (CPT / 32) + g]);
    const float sc = am > 0.f ? __fdiv_rn(am, kE4M3Max) : 1.0f;
    tb.sx[threadIdx.x] = sc;
    if (blockIdx.x == 0) p.sx[threadIdx.x] = sc;
  }
  __syncthreads();
  const bool writer = (blockIdx.x == 0);
  for (int c = threadIdx.x; c < M * CPT; c += blockDim.x) {
    const int t = c / CPT, i = c % CPT;
    const float sc = tb.sx[t];
    const uint4 v = xb4[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t q[4], h[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      q[k] = f32x2_to_e4m3x2(__fdiv_rn(__uint_as_float(w[k] << 16), sc),
                             __fdiv_rn(__uint_as_float(w[k] & 0xFFFF0000u), sc));
      h[k] = e4m3x2_to_f16x2(q[k]);
    }
    *reinterpret_cast<uint4*>(smem + SL::xh + (size_t)t * kXhBytes + (size_t)i * 16) = make_uint4(h[0], h[1], h[2], h[3]);
    if (writer) reinterpret_cast<uint2*>(p.xq + (size_t)t * kH)[i] = make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
  }
  __syncthreads();
  return true;
}

// ------------------------------------------------------------------ P1: router rows

__device__ __forceinline__ void router_range(int E, int& e0, int& e1) {
  e0 = (int)((long long)blockIdx.x * E / gridDim.x);
  e1 = (int)((long long)(blockIdx.x + 1) * E / gridDim.x);
}
// The block's router rows [e0, e1) (at most 4 x 5 KB) are bulk-copied into ring slot 0 at the
// start of the layer (the ring is idle until the routing is known) and read from there.
template <int MAXM>
__device__ bool router_rows(const MoeParams& p, const uint8_t* smem, const Ring& rg, int layer) {
  using SL = SLayout<MAXM>;
  const int M = p.M, E = p.E;
  int e0, e1;
  router_range(E, e0, e1);
  const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(smem + SL::xb);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t tag = (uint32_t)layer + 1;
  if (e0 + warp < e1 && !wait_full(rg.rbar, layer & 1, p)) return false;
  for (int e = e0 + warp; e < e1; e += kWarps) {
    const uint4* w4 = reinterpret_cast<const uint4*>(smem + SL::ring + (size_t)(e - e0) * kH * 2);
    for (int t = 0; t < M; ++t) {
      const uint4* x4 = reinterpret_cast<const uint4*>(xb + (size_t)t * kH);
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 10; ++i) {
        const uint4 wv = w4[32 * i + lane];
        const uint4 xv = x4[32 * i + lane];
        const uint32_t a[4] = {wv.x, wv.y, wv.z, wv.w};
        const uint32_t b[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc = fmaf(__uint_as_float(a[k] << 16), __uint_as_float(b[k] << 16), acc);
          acc = fmaf(__uint_as_float(a[k] & 0xFFFF0000u), __uint_as_float(b[k] & 0xFFFF0000u), acc);
        }
      }
      acc = warp_sum(acc);
      if (lane == 0) {
        st_word(p.xz + (size_t)t * E + e, tagged(__float_as_uint(acc), tag));
        p.logits[(size_t)t * E + e] = acc;                 // inspection copy
      }
    }
  }
  return true;
}

// ------------------------------------------------------------------ P2: routing

// Every thread of the block polls its share of the M x E logit words (tag layer + 1), all
// of them requested before any is checked, into zrow (fp32); false (tb.fail set) on timeout or
// when another block failed. Every thread of the block must call it.
template <int MAXM>
__device__ bool poll_logits(const MoeParams& p, int layer, float* zrow, STables& tb) {
  constexpr int NW = (MAXM * MDW_MAX_EXPERTS + kThreads - 1) / kThreads;
  const int n_words = p.M * p.E;
  const uint32_t tag = (uint32_t)layer + 1;
  uint32_t want = 0;
#pragma unroll
  for (int k = 0; k < NW; ++k)
    if ((int)threadIdx.x + k * kThreads < n_words) want |= 1u << k;
  long long t0 = 0;
  for (int n = 0; want != 0; ++n) {
    uint64_t w[NW];
#pragma unroll
    for (int k = 0; k < NW; ++k) w[k] = (want & (1u << k)) ? ld_word(p.xz + threadIdx.x + k * kThreads) : 0;
    uint32_t got = 0;
#pragma unroll
    for (int k = 0; k < NW; ++k)
      if ((want & (1u << k)) && tag_of(w[k]) == tag) {
        zrow[threadIdx.x + k * kThreads] = __uint_as_float((uint32_t)w[k]);
        got |= 1u << k;
      }
    want &= ~got;
    if (want == 0) break;
    if (n == 0) t0 = clock64();
    if (((n & 15) == 15 && ld_volatile_u32(p.hdr + kHdrStatus) != 0) || *reinterpret_cast<volatile int*>(&tb.fail)) {
      atomicExch(&tb.fail, 1);
      break;
    }
    if (clock64() - t0 > p.spin_budget) { set_status(p.hdr, MDW_ERR_TIMEOUT); atomicExch(&tb.fail, 1); break; }
  }
  __syncthreads();
  return tb.fail == 0;
}

// Top-K of one token's logits held by the warp (v[j] = logit lane + 32 j), ties -> lower id:
// a bitonic sort of the 32 lane bests gives a threshold T (the K-th best of them; K distinct
// logits reach T, so the K-th largest logit does too); the logits not worse than T (usually
// little more than K) are compacted into shared memory and ranked among themselves. Writes
// the ids and raw logits of ranks 0..K-1 to tb.ids / tb.gts [t * K + r].
__device__ __forceinline__ void topk_token(float (&v)[MDW_MAX_EXPERTS / 32], int E, int K, int t, STables& tb, float* cv, int* ci,
                           int layer = 0) {
  constexpr int PER = MDW_MAX_EXPERTS / 32;
  constexpr int kCand = 128;
  const int lane = threadIdx.x & 31;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int e = lane + 32 * j;
    if (v[j] != v[j]) v[j] = -INFINITY;                // a NaN logit ranks last
    if (e < E && beats(v[j], e, bv, bi)) { bv = v[j]; bi = e; }
  }
#pragma unroll
  for (int kk = 2; kk <= 32; kk <<= 1)
#pragma unroll
    for (int jj = kk >> 1; jj > 0; jj >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, jj);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, jj);
      const bool up = ((lane & kk) == 0);
      const bool lower = ((lane & jj) == 0);
      const bool o_better = beats(ov, oi, bv, bi);
      if ((up == lower) ? o_better : !o_better && !(ov == bv && oi == bi)) { bv = ov; bi = oi; }
    }
  const float tv = __shfl_sync(0xffffffffu, bv, K - 1);
  const int ti = __shfl_sync(0xffffffffu, bi, K - 1);
  int count = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int e = lane + 32 * j;
    const bool keep = e < E && !beats(tv, ti, v[j], e);
    const unsigned m = __ballot_sync(0xffffffffu, keep);
    const int pos = count + __popc(m & ((1u << lane) - 1u));
    if (keep && pos < kCand) { cv[pos] = v[j]; ci[pos] = e; }
    count += __popc(m);
  }
  __syncwarp();
  if (count <= kCand) {
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

// Routing of the window: warp t < M polls token t's logits and selects its experts (or takes
// the imposed ids); warp 0 then builds the gates (softmax of each token's selected logits),
// the union slots (slot 0 = shared expert), the per-slot token lists and the pairs.
template <int MAXM>
__device__ bool route_window(const MoeParams& p, STables& tb, int layer, uint8_t* smem) {
  using SL = SLayout<MAXM>;
  const int M = p.M, E = p.E, K = p.K;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) tb.bad = 0;
  __syncthreads();
  float* zrow = reinterpret_cast<float*>(smem + SL::zrow);
  if (!poll_logits<MAXM>(p, layer, zrow, tb)) return false;
  STRACE(layer, 3);
  if (warp < M) {
    const int t = warp;
    if (p.topk_override) {
      const int32_t* ov = p.topk_override + (p.stack_mode ? (size_t)layer * M * K : 0);
      if (lane < K) {
        int id = ov[t * K + lane];
        bool ok = id >= 0 && id < E;
        for (int j = 0; j < K; ++j)
          if (j != lane && ov[t * K + j] == id) ok = false;
        if (!ok) { atomicExch(&tb.bad, 1); id = 0; }
        tb.ids[t * K + lane] = id;
        tb.gts[t * K + lane] = zrow[t * E + id];
      }
      __syncwarp();
    } else {
      float v[MDW_MAX_EXPERTS / 32];
#pragma unroll
      for (int j = 0; j < MDW_MAX_EXPERTS / 32; ++j) v[j] = lane + 32 * j < E ? zrow[t * E + lane + 32 * j] : -INFINITY;
      float* cv = reinterpret_cast<float*>(smem + SL::cand) + t * 256;
      topk_token(v, E, K, t, tb, cv, reinterpret_cast<int*>(cv + 128), layer);
    }
    STRACE(layer, 15);
  }
  __syncthreads();
  if (tb.fail) return false;
  if (tb.bad) { if (threadIdx.x == 0) set_status(p.hdr, MDW_ERR_DEVICE_BOUNDS); return false; }
  const int first = p.has_shared ? 1 : 0;
  if (warp == 0) {
    // gates: softmax over each token's K selected logits (lanes of one token are contiguous)
    for (int i0 = 0; i0 < M * K; i0 += 32) {
      const int i = i0 + lane;
      float gate = 0.f;
      if (i < M * K) {
        const float* z = tb.gts + (i / K) * K;
        float mx = z[0];
        for (int r = 1; r < K; ++r) mx = fmaxf(mx, z[r]);
        float sum = 0.f;
        for (int r = 0; r < K; ++r) sum += expf(z[r] - mx);
        gate = expf(z[i % K] - mx) / sum;
      }
      __syncwarp();
      if (i < M * K) tb.gts[i] = gate;
      __syncwarp();
    }
    // union bitmap -> slots (ascending expert id after the shared slot)
    if (lane < MDW_MAX_EXPERTS / 32) tb.bitmap[lane] = 0;
    __syncwarp();
    for (int i = lane; i < M * K; i += 32) atomicOr(&tb.bitmap[tb.ids[i] >> 5], 1u << (tb.ids[i] & 31));
    __syncwarp();
    const uint32_t word = lane < MDW_MAX_EXPERTS / 32 ? tb.bitmap[lane] : 0u;
    const int c = __popc(word);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int nb = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += nb;
    }
    if (lane < MDW_MAX_EXPERTS / 32) tb.wpre[lane] = incl - c;
    int pos = first + incl - c;
    for (uint32_t w = word; w; w &= w - 1) {
      tb.cnt[pos] = 0;
      tb.slot_expert[pos++] = lane * 32 + __ffs(w) - 1;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    const int S = total + first;
    if (first && lane == 0) { tb.slot_expert[0] = -1; tb.cnt[0] = (1 << M) - 1; }
    __syncwarp();
    // token masks per slot -> pair counts -> slot_begin -> pairs (slot-major, token-minor)
    auto slot_of = [&](int e) {
      return first + tb.wpre[e >> 5] + __popc(tb.bitmap[e >> 5] & ((1u << (e & 31)) - 1u));
    };
    for (int i = lane; i < M * K; i += 32) atomicOr(reinterpret_cast<unsigned*>(&tb.cnt[slot_of(tb.ids[i])]), 1u << (i / K));
    __syncwarp();
    const int cs = lane < S ? __popc((unsigned)tb.cnt[lane]) : 0;   // S <= 33: two rounds at most
    int in2 = cs;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int nb = __shfl_up_sync(0xffffffffu, in2, o);
      if (lane >= o) in2 += nb;
    }
    if (lane < S) tb.slot_begin[lane] = in2 - cs;
    int carry = __shfl_sync(0xffffffffu, in2, 31);
    if (S > 32 && lane == 0) {
      tb.slot_begin[32] = carry;
      carry += __popc((unsigned)tb.cnt[32]);
    }
    if (lane == 0) { tb.slot_begin[S] = carry; tb.n_pairs = carry; tb.n_slots = S; tb.n_routed = total; }
    __syncwarp();
    for (int i = lane; i < M * K; i += 32) {
      const int t = i / K, sidx = slot_of(tb.ids[i]);
      const int q = tb.slot_begin[sidx] + __popc((unsigned)tb.cnt[sidx] & ((1u << t) - 1u));
      tb.pair_token[q] = t;
      tb.pair_gate[q] = tb.gts[i];
    }
    if (first && lane < M) { tb.pair_token[lane] = lane; tb.pair_gate[lane] = 1.0f; }
    STRACE(layer, 16);
  }
  __syncthreads();
  STRACE(layer, 17);
  if (blockIdx.x == 0) {
    // publish the routing (inspection and the optional outputs)
    for (int i = threadIdx.x; i < M * K; i += blockDim.x) {
      p.ids[i] = tb.ids[i];
      p.gates[i] = tb.gts[i];
      if (p.ids_out) p.ids_out[i] = tb.ids[i];
      if (p.gates_out) p.gates_out[i] = tb.gts[i];
    }
    const int S = tb.n_slots;
    for (int s = threadIdx.x; s < S; s += blockDim.x) {
      p.slot_expert[s] = tb.slot_expert[s];
      for (int q = tb.slot_begin[s]; q < tb.slot_begin[s + 1]; ++q) p.pair_slot[q] = s;
    }
    for (int q = threadIdx.x; q < tb.n_pairs; q += blockDim.x) {
      p.pair_token[q] = tb.pair_token[q];
      p.pair_gate[q] = tb.pair_gate[q];
    }
    if (threadIdx.x == 0) {
      p.hdr[kHdrSlots] = S;
      p.hdr[kHdrPairs] = tb.n_pairs;
      p.hdr[kHdrRouted] = tb.n_routed;
      if (layer < kHdrWords - kHdrUnions) p.hdr[kHdrUnions + layer] = tb.n_routed;
    }
  }
  return true;
}

// ------------------------------------------------------------------ P3: gate/up units

// One gate/up unit: tile in ring slot `buf`, K part kp (blocks 8 kp .. 8 kp + 7), block-column
// MMAs (NT tiles of up to two tokens each). Result in the token-column layout of bc_finish.
template <int NT>
__device__ __forceinline__ void gu_unit(const uint8_t* buf, int kp, const uint8_t* xt0, const uint8_t* xt1,
                                        int g, int q, float (&r)[4]) {
  const uint8_t* sg = buf + 2 * kTileW;            // gate scales [8][80], then up scales
  float bcacc[NT][2] = {};
#pragma unroll
  for (int sb = 0; sb < 8; sb += 4) {
    const int blk = 8 * kp + sb;                   // first block of the super-step
    const uint4 w0 = *reinterpret_cast<const uint4*>(buf + g * kW13RowBytes + (blk + q) * 16);
    const uint4 w1 = *reinterpret_cast<const uint4*>(buf + kTileW + g * kW13RowBytes + (blk + q) * 16);
    const uint32_t s0 = *reinterpret_cast<const uint16_t*>(sg + g * kHBlocks + blk + 2 * (q & 1));
    const uint32_t s1 = *reinterpret_cast<const uint16_t*>(sg + kTileS + g * kHBlocks + blk + 2 * (q & 1));
    float d[NT][4] = {};
    const uint8_t* xb[NT];
    xb[0] = xt0 ? xt0 + 64 * (blk + q) : nullptr;
    if (NT > 1) xb[NT - 1] = xt1 ? xt1 + 64 * (blk + q) : nullptr;
    bc_step<NT>(w0, w1, xb, d);
#pragma unroll
    for (int j = 0; j < NT; ++j) bc_scale_add(d[j], s0 & 0xFF, s0 >> 8, s1 & 0xFF, s1 >> 8, bcacc[j]);
  }
  bc_finish<NT>(bcacc, q, r);
}

// One down unit: W2 rows 0..15 of the block's rows of one slot (chunk `ch`: [nrows][384] then
// [nrows][24] scales), K part kp (blocks 8 kp .. +7); h0 / h1 = the lane's h-hat of tile 0 / 1.
template <int NT>
__device__ __forceinline__ void dn_unit(const uint8_t* ch, int nrows, int kp, const uint8_t* h0, const uint8_t* h1,
                                        int g, int q, float (&r)[4]) {
  const uint8_t* sc = ch + nrows * kW2RowBytes;
  float bcacc[NT][2] = {};
#pragma unroll
  for (int sb = 0; sb < 8; sb += 4) {
    const int blk = 8 * kp + sb;
    const uint4 w0 = *reinterpret_cast<const uint4*>(ch + g * kW2RowBytes + (blk + q) * 16);
    const uint4 w1 = *reinterpret_cast<const uint4*>(ch + (g + 8) * kW2RowBytes + (blk + q) * 16);
    const uint32_t s0 = *reinterpret_cast<const uint16_t*>(sc + g * kIBlocks + blk + 2 * (q & 1));
    const uint32_t s1 = *reinterpret_cast<const uint16_t*>(sc + (g + 8) * kIBlocks + blk + 2 * (q & 1));
    float d[NT][4] = {};
    const uint8_t* xb[NT];
    xb[0] = h0 ? h0 + 64 * (blk + q) : nullptr;
    if (NT > 1) xb[NT - 1] = h1 ? h1 + 64 * (blk + q) : nullptr;
    bc_step<NT>(w0, w1, xb, d);
#pragma unroll
    for (int j = 0; j < NT; ++j) bc_scale_add(d[j], s0 & 0xFF, s0 >> 8, s1 & 0xFF, s1 >> 8, bcacc[j]);
  }
  bc_finish<NT>(bcacc, q, r);
}

// A warp finished a unit of the item in ring slot s: count it; the warp that completes the
// item (returns true) may read every unit's results and refills the slot.
__device__ __forceinline__ bool finish_unit(Ring& rg, int s, int units) {
  __syncwarp();
  int last = 0;
  if ((threadIdx.x & 31) == 0) {
    __threadfence_block();
    const int old = atomicAdd(rg.done + s, 1);
    last = (old == units - 1);
    if (last) { rg.done[s] = 0; __threadfence_block(); }
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  __syncwarp();
  return last != 0;
}

// ------------------------------------------------------------------ the kernel

template <int MAXM>
__global__ void __launch_bounds__(kThreads, 1) moe_stream_kernel(const __grid_constant__ MoeParams p) {
  using SL = SLayout<MAXM>;
  constexpr int NT = SL::NT;
  extern __shared__ __align__(128) uint8_t smem[];
  STables& tb = *reinterpret_cast<STables*>(smem + SL::tabs);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const int M = p.M, G = gridDim.x;
  Ring rg;
  rg.full = reinterpret_cast<uint64_t*>(smem + SL::bars);
  rg.done = reinterpret_cast<int*>(smem + SL::bars + SL::NS * 8);
  rg.item = reinterpret_cast<uint32_t*>(smem + SL::bars + SL::NS * 12);
  rg.rbar = reinterpret_cast<uint64_t*>(smem + SL::bars + SL::NS * 16 + 16);
  rg.seq = 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < SL::NS; ++s) { mbar_init(rg.full + s, 1); rg.done[s] = 0; rg.item[s] = kNoItem; }
    mbar_init(rg.rbar, 1);
    tb.fail = 0;
    fence_mbar_init();
  }
  __syncthreads();
  Plan pl;
  bool has_router_rows;
  {
    int e0, e1;
    router_range(p.E, e0, e1);
    has_router_rows = e1 > e0;
  }
  pl.r0 = 2 * (int)((long long)blockIdx.x * (kH / 2) / G);
  pl.nrows = 2 * (int)((long long)(blockIdx.x + 1) * (kH / 2) / G) - pl.r0;
  float* part = reinterpret_cast<float*>(smem + SL::part);
  float* dres = reinterpret_cast<float*>(smem + SL::dres);
  float* dleft = reinterpret_cast<float*>(smem + SL::dleft);
  const float* rres = reinterpret_cast<const float*>(smem + SL::rres);

  for (int layer = 0; layer < p.L; ++layer) {
    const LayerDesc& L = p.layers[layer];
    if (threadIdx.x == 0) {
      // this layer's router rows into ring slot 0 (idle until the routing is known)
      int e0, e1;
      router_range(p.E, e0, e1);
      if (e1 > e0) {
        fence_proxy_async();
        mbar_arrive_expect_tx(rg.rbar, (uint32_t)(e1 - e0) * kH * 2);
        bulk_copy(smem + SL::ring, L.router_w + (size_t)e0 * kH, (uint32_t)(e1 - e0) * kH * 2, rg.rbar);
      }
    }
    pl.base = rg.seq;
    STRACE(layer, 0);
    if (!prepare_input<MAXM>(p, layer, smem, tb, pl)) { drain_ring<MAXM>(rg, layer, has_router_rows); break; }
    STRACE(layer, 1);
    if (!router_rows<MAXM>(p, smem, rg, layer)) atomicExch(&tb.fail, 1);
    STRACE(layer, 2);
    if (!route_window<MAXM>(p, tb, layer, smem)) { drain_ring<MAXM>(rg, layer, has_router_rows); break; }
    STRACE(layer, 4);
    // the block's work: tiles [t0, t0 + n_gu) of S * 96, then its rows of every slot's W2
    const int S = tb.n_slots;
    {
      const long long T = (long long)S * kTilesPerSlot;
      pl.t0 = (int)((long long)blockIdx.x * T / G);
      pl.n_gu = (int)((long long)(blockIdx.x + 1) * T / G) - pl.t0;
      const int chunk = pl.nrows * (kW2RowBytes + kIBlocks);
      pl.dps = kSlotBytes / chunk;
      pl.n_dn = (S + pl.dps - 1) / pl.dps;
      pl.n_items = pl.n_gu + pl.n_dn;
    }
    // the first NS items, requested by lanes of warp 0 (the ring is empty here)
    if (warp == 0) {
      const int n0 = min(SL::NS, pl.n_items);
      if (lane < n0) issue_item<MAXM>(p, L, tb, pl, rg, smem, lane);
    }
    rg.seq = pl.base + pl.n_items;
    STRACE(layer, 5);
    bool ok = true;
    // P3: gate/up units u = warp, warp + 12, ...: tile u / 10, K part u % 10
    const int n_gu_units = pl.n_gu * kGuParts;
    for (int u = warp; u < n_gu_units && ok; u += kWarps) {
      const int it = u / kGuParts, kp = u % kGuParts;
      const uint32_t gs = pl.base + it;
      const int s = gs % SL::NS;
      const int t = pl.t0 + it, slot = t / kTilesPerSlot, j0 = (t % kTilesPerSlot) * kTileRP;
      const int pb = tb.slot_begin[slot], m = tb.slot_begin[slot + 1] - pb;
      const uint8_t* xt0 = nullptr;
      const uint8_t* xt1 = nullptr;
      if (q == (g & 3)) {
        const int tt = g >> 2;
        if (tt < m) xt0 = smem + SL::xh + (size_t)tb.pair_token[pb + tt] * kXhBytes;
        if (NT > 1 && 2 + tt < m) xt1 = smem + SL::xh + (size_t)tb.pair_token[pb + 2 + tt] * kXhBytes;
      }
      if (!wait_item<SL::NS>(rg, gs, p)) { ok = false; break; }
      STRACE(layer, 11);
      const uint8_t* buf = smem + SL::ring + (size_t)s * kSlotBytes;
      float r[4];
      gu_unit<NT>(buf, kp, xt0, xt1, g, q, r);
      float4* pp = reinterpret_cast<float4*>(part) + ((size_t)s * kGuParts + kp) * 8 * NT;
      if (q < NT) pp[g * NT + q] = make_float4(r[0], r[1], r[2], r[3]);
      if (finish_unit(rg, s, kGuParts)) {
        // last unit of the tile: K parts summed in order, SwiGLU, h -> xh
        if (q < NT) {
          const float4* pq = reinterpret_cast<const float4*>(part) + (size_t)s * kGuParts * 8 * NT;
          float4 a = pq[g * NT + q];
          for (int k = 1; k < kGuParts; ++k) {
            const float4 b = pq[k * 8 * NT + g * NT + q];
            a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
          }
          const float gv[2] = {a.x, a.y}, uv[2] = {a.z, a.w};
          const uint32_t tag = (uint32_t)layer + 1;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int col = 2 * q + c;
            if (col < m) {
              const float sx = tb.sx[tb.pair_token[pb + col]];
              const float gsx = gv[c] * sx, usx = uv[c] * sx;
              const float h = gsx / (1.0f + expf(-gsx)) * usx;
              st_word(p.xh + (size_t)(pb + col) * kI + j0 + g, tagged(__float_as_uint(h), tag));
            }
          }
        }
        __syncwarp();
        if (lane == 0 && it + SL::NS < pl.n_items) issue_item<MAXM>(p, L, tb, pl, rg, smem, it + SL::NS);
      }
    }
    STRACE(layer, 12);
    if (!ok) { atomicExch(&tb.fail, 1); }
    __syncthreads();
    STRACE(layer, 6);
    if (tb.fail) { drain_ring<MAXM>(rg, layer, has_router_rows); break; }
    // during the h exchange: the next layer's router rows and shared-expert slice into L2
    if (p.stack_mode && layer + 1 < p.L && lane == 0 && warp < 5) {
      const LayerDesc& Ln = p.layers[layer + 1];
      if (warp == 0) {
        int e0, e1;
        router_range(p.E, e0, e1);
        prefetch_l2(Ln.router_w + (size_t)e0 * kH, (uint32_t)((e1 - e0) * kH * 2));
      } else if (p.has_shared) {
        const int j0 = (int)((long long)blockIdx.x * kI / G), j1 = (int)((long long)(blockIdx.x + 1) * kI / G);
        const size_t row = (size_t)((warp - 1) & 1) * kI + j0;
        if (warp <= 2) prefetch_l2(Ln.sh_w13_q + row * kW13RowBytes, (uint32_t)((j1 - j0) * kW13RowBytes));
        else prefetch_l2(Ln.sh_w13_s + row * kHBlocks, (uint32_t)((j1 - j0) * kHBlocks));
      }
    }
    // P4: poll every pair's h (tag layer + 1), quantise into f16 h-hat (warp per pair)
    const int P = tb.n_pairs;
    {
      const uint32_t tag = (uint32_t)layer + 1;
      constexpr int J = kI / 64;                   // 12 word pairs per lane
      for (int pr = warp; pr < P && ok; pr += kWarps) {
        const uint64_t* hw = p.xh + (size_t)pr * kI;
        float hv[2 * J];
        // two halves of six word pairs per lane, each requested in full before it is checked
        // (all twelve at once would not fit the register budget)
        constexpr int JH = J / 2;
#pragma unroll
        for (int half = 0; half < 2 && ok; ++half) {
          uint32_t want = (1u << JH) - 1;
          long long t0 = 0;
          for (int n = 0;; ++n) {
            uint64_t w[JH][2];
#pragma unroll
            for (int j = 0; j < JH; ++j)
              if (want & (1u << j)) ld_word2(hw + 2 * (lane + 32 * (half * JH + j)), w[j][0], w[j][1]);
            uint32_t got = 0;
#pragma unroll
            for (int j = 0; j < JH; ++j) {
              if ((want & (1u << j)) && tag_of(w[j][0]) == tag && tag_of(w[j][1]) == tag) {
                hv[2 * (half * JH + j)] = __uint_as_float((uint32_t)w[j][0]);
                hv[2 * (half * JH + j) + 1] = __uint_as_float((uint32_t)w[j][1]);
                got |= 1u << j;
              }
            }
            want &= ~got;
            if (!__any_sync(0xffffffffu, want != 0)) break;
            if (n == 0) t0 = clock64();
            bool bad = false;
            if ((n & 15) == 15 && ld_volatile_u32(p.hdr + kHdrStatus) != 0) bad = true;
            if (clock64() - t0 > p.spin_budget) { if (lane == 0) set_status(p.hdr, MDW_ERR_TIMEOUT); bad = true; }
            if (__any_sync(0xffffffffu, bad)) { ok = false; break; }
          }
        }
        if (!ok) break;
        float am = 0.f;
#pragma unroll
        for (int j = 0; j < 2 * J; ++j) am = fmaxf(am, fabsf(hv[j]));
        am = warp_max(am);
        const float sc = am > 0.f ? __fdiv_rn(am, kE4M3Max) : 1.0f;
        if (lane == 0) tb.sh[pr] = sc;
        uint8_t* hh = smem + SL::hh + (size_t)pr * kHhBytes;
        const bool writer = blockIdx.x == 0;
#pragma unroll
        for (int j = 0; j < J; ++j) {
          const int e = 2 * (lane + 32 * j);       // elements e, e + 1
          const uint32_t c01 = f32x2_to_e4m3x2(__fdiv_rn(hv[2 * j], sc), __fdiv_rn(hv[2 * j + 1], sc));
          *reinterpret_cast<uint32_t*>(hh + (size_t)e * 2) = e4m3x2_to_f16x2(c01);
          if (writer) {
            *reinterpret_cast<uint16_t*>(p.hq + (size_t)pr * kI + e) = (uint16_t)c01;
            *reinterpret_cast<float2*>(p.h + (size_t)pr * kI + e) = make_float2(hv[2 * j], hv[2 * j + 1]);
          }
        }
        if (writer && lane == 0) p.sh[pr] = sc;
      }
    }
    STRACE(layer, 13);
    if (!ok) atomicExch(&tb.fail, 1);
    __syncthreads();
    STRACE(layer, 7);
    if (tb.fail) { drain_ring<MAXM>(rg, layer, has_router_rows); break; }
    // P5: down units v = warp, warp + 12, ...: slot v / U, part v % U (part 3: rows 16..)
    const int U = kDnParts + (pl.nrows > 16 ? 1 : 0);
    const int n_dn_units = S * U;
    const int chunk = pl.nrows * (kW2RowBytes + kIBlocks);
    for (int v = warp; v < n_dn_units && ok; v += kWarps) {
      const int slot = v / U, kp = v % U;
      const int it = pl.n_gu + slot / pl.dps;
      const uint32_t gs = pl.base + it;
      const int s = gs % SL::NS;
      const int pb = tb.slot_begin[slot], m = tb.slot_begin[slot + 1] - pb;
      if (!wait_item<SL::NS>(rg, gs, p)) { ok = false; break; }
      const uint8_t* ch = smem + SL::ring + (size_t)s * kSlotBytes + (size_t)(slot % pl.dps) * chunk;
      if (kp < kDnParts) {
        const uint8_t* h0 = nullptr;
        const uint8_t* h1 = nullptr;
        if (q == (g & 3)) {
          const int tt = g >> 2;
          if (tt < m) h0 = smem + SL::hh + (size_t)(pb + tt) * kHhBytes;
          if (NT > 1 && 2 + tt < m) h1 = smem + SL::hh + (size_t)(pb + 2 + tt) * kHhBytes;
        }
        float r[4];
        dn_unit<NT>(ch, pl.nrows, kp, h0, h1, g, q, r);
        if (q < NT) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int col = 2 * q + c;
            if (col < m) {
              float* d = dres + ((size_t)(pb + col) * kDnParts + kp) * 16;
              d[g] = r[c];
              d[g + 8] = r[2 + c];
            }
          }
        }
      } else {
        // rows 16 .. nrows - 1 on the CUDA cores: lanes 0..23 one block each, every pair
        const uint8_t* sc = ch + pl.nrows * kW2RowBytes;
        for (int rr = 16; rr < pl.nrows; ++rr) {
          uint32_t w2[16];
          float fs = 0.f;
          if (lane < kIBlocks) {
            mx_block_decode(*reinterpret_cast<const uint4*>(ch + rr * kW2RowBytes + lane * 16), w2);
            fs = e8m0_to_f32(sc[rr * kIBlocks + lane]);
          }
          for (int c = 0; c < m; ++c) {
            float dsum = 0.f;
            if (lane < kIBlocks) {
              const uint4* hx = reinterpret_cast<const uint4*>(smem + SL::hh + (size_t)(pb + c) * kHhBytes + 64 * lane);
              uint32_t x2[16];
#pragma unroll
              for (int pl4 = 0; pl4 < 4; ++pl4) {
                const uint4 xv = hx[pl4];
                x2[4 * pl4] = xv.x; x2[4 * pl4 + 1] = xv.y; x2[4 * pl4 + 2] = xv.z; x2[4 * pl4 + 3] = xv.w;
              }
              dsum = dot32_f16(w2, x2) * fs;
            }
            dsum = warp_sum(dsum);
            if (lane == 0) dleft[(size_t)(pb + c) * (kMaxRows - 16) + rr - 16] = dsum;
          }
        }
      }
      if (finish_unit(rg, s, item_units(pl, it, S))) {
        if (lane == 0 && it + SL::NS < pl.n_items) issue_item<MAXM>(p, L, tb, pl, rg, smem, it + SL::NS);
      }
    }
    STRACE(layer, 14);
    if (!ok) atomicExch(&tb.fail, 1);
    __syncthreads();
    STRACE(layer, 8);
    if (tb.fail) { drain_ring<MAXM>(rg, layer, has_router_rows); break; }
    // combine: y[t][row] = sum over the token's pairs (ascending) of gate * s_h * dot, + residual
    {
      const uint32_t tag = (uint32_t)layer + 1;
      for (int i = threadIdx.x; i < M * (pl.nrows / 2); i += blockDim.x) {
        const int t = i / (pl.nrows / 2), rr = 2 * (i % (pl.nrows / 2));
        float y[2] = {0.f, 0.f};
        for (int k = 0; k < P; ++k) {
          if (tb.pair_token[k] != t) continue;
          const float f = tb.sh[k] * tb.pair_gate[k];
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int row = rr + c;
            float v;
            if (row < 16) {
              const float* d = dres + (size_t)k * kDnParts * 16 + row;
              v = (d[0] + d[16]) + d[32];
            } else {
              v = dleft[(size_t)k * (kMaxRows - 16) + row - 16];
            }
            y[c] += v * f;
          }
        }
        const size_t o = (size_t)t * kH + pl.r0 + rr;
        if (p.stack_mode) {
          const float a0 = rres[t * kMaxRows + rr] + y[0], a1 = rres[t * kMaxRows + rr + 1] + y[1];
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(a0, a1);
          const uint32_t bits = *reinterpret_cast<const uint32_t*>(&b2);
          __nv_bfloat16* rout = p.resid + (size_t)(p.resid_pingpong ? ((layer + 1) & 1) : (layer + 1)) * M * kH;
          *reinterpret_cast<uint32_t*>(rout + o) = bits;
          if (layer + 1 < p.L) st_word(p.xr + o / 2, tagged(bits, tag));
        } else {
          float v0 = y[0], v1 = y[1];
          if (p.residual) { v0 += rres[t * kMaxRows + rr]; v1 += rres[t * kMaxRows + rr + 1]; }
          if (p.y_fp32) {
            *reinterpret_cast<float2*>(reinterpret_cast<float*>(p.y_out) + o) = make_float2(v0, v1);
          } else {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(v0, v1);
            *reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(p.y_out) + o) = b2;
          }
        }
      }
    }
    __syncthreads();
    STRACE(layer, 9);
  }
  STRACE_FLUSH(p.L);
}

template <int MAXM>
cudaError_t launch_t(const MoeParams& p, cudaStream_t s) {
  const size_t smem = SLayout<MAXM>::total;
  auto kern = moe_stream_kernel<MAXM>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  void* args[] = {const_cast<MoeParams*>(&p)};
  return cudaLaunchCooperativeKernel((const void*)kern, dim3(moe_grid()), dim3(kThreads), args, smem, s);
}

}  // namespace

cudaError_t launch_moe_stream(const MoeParams& p, cudaStream_t s) {
  // each block owns at most kMaxRows output rows: 2 * ceil(H / 2 / grid) <= 32
  if (moe_grid() < kH / kMaxRows) return cudaErrorInvalidConfiguration;
  if (p.M <= 1) return launch_t<1>(p, s);
  if (p.M <= 2) return launch_t<2>(p, s);
  return launch_t<4>(p, s);
}

}  // namespace mdw

#ifdef MDW_TRACE
extern "C" int mdw_stream_trace_read(void* dst, size_t bytes) {
  return (int)cudaMemcpyFromSymbol(dst, mdw::g_strace, bytes < sizeof(mdw::g_strace) ? bytes : sizeof(mdw::g_strace));
}
#endif
