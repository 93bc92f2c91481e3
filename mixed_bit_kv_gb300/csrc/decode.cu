// Decode attention over the TriZone cache of RDKV
// (gist.science/ko/paper/2605.08317, section 2.3): the logits and the output
// are computed with the dequantisation fused into the two products, reading
// zones A (packed K rows and 2/4/8-bit V rows), B (fp16 V rows of 16-bit
// tokens) and C (fp16 K and V rows of the window and of decoded tokens) in one
// pass.
//
// Work: one block per SM, dealt to the (sequence, KV head) pairs in proportion
// to their estimated cost (on the host when the plan's costs are there, else by
// the kernel).  A head's work items are its zone-A tiles (32 tokens, in class
// order) followed by zone-C blocks of 16 rows; split s of n takes items s,
// s + n, s + 2n, ...  One producer warp streams the items into a shared-memory
// ring per consumer warp with bulk asynchronous copies (its lane w serves
// consumer warp w, taking the block's next item whenever that ring has room);
// every stage has a full and an empty mbarrier, and every wait is bounded
// (RDKV_ERR_TIMEOUT).  The fifteen consumer warps only compute.  The last block
// of a head to finish (an atomic ticket) merges the splits' partial softmax
// states into the output (and, when asked, the log-sum-exp).  One launch may
// attend several caches sharing the query (segments moved out of zone C and the
// live cache): each block reads one cache, the blocks of a head over all caches
// share its merge; a ragged launch attends several sequences, each head with its own merge.  The
// zones may be paged: zone A in 64 KB pages, zones B and C in 16-row pages, through tables.
//
// Products: mma.sync m16n8k16 (fp16 in, fp32 accumulate), tokens on M:
//   S^T[16 tok x 8 heads]  += K^[16 tok x 16 slots] * B[16 slots x 8 heads]
//   O^T[16 ch  x 8 heads]  += V^T[16 ch x 16 tok]   * P^T[16 tok x 8 heads]
// K is quantised per (channel, head): k^ = zero_c + scale_c * code, so the
// logit of head h is sum_c q_hc zero_c (a per-head constant, added once) plus
// sum_c code * (q_hc scale_c).  The B operand q_hc * scale_c is built once per
// block, as an fp16 high part and remainder (~22 bits).  A 32-bit A-fragment
// register holds two codes of one token (K) or of one channel (V); the layout
// puts them in the two half-words of one 32-bit word, at a bit position below
// 10, so ONE mask (a shift first for the upper positions) turns them into fp16
// subnormals code * 2^(pos - 24) exactly; the 2^pos goes into B (K) or into a
// per-channel power of two undone once (V).  The softmax runs in fp32 on the S^T
// accumulators (base-2 exponent); P^T is moved into B-fragment order by
// movmatrix.  The G query heads of a group share every loaded tile.
#include <atomic>

#include "common.cuh"

namespace rdkv {

// Consumer warps of a block: 15 with one block per SM (with the producer, four warps per
// scheduler), or 7 with two blocks per SM for launches over many (head, cache) units, whose blocks
// then share their SM as they finish.
constexpr int kConsumersWide = 15;
constexpr int kConsumersNarrow = 7;
constexpr int kManyUnits = 32;  // launches over this many units or more take the two-block layout
constexpr int kStages = 8;                 // stages in flight per consumer warp (the ring's bytes permitting)
constexpr int kPrologueItems = 4;          // stages per consumer issued before the wait for the previous kernel
constexpr int kMaxDealtBlocks = 512;       // grids up to this size may be dealt to heads on the host
constexpr uint8_t kNoHead = 0xff;
constexpr int kMaxParts = 8;               // caches one launch may attend
constexpr int kCRows = 16;                 // zone-C rows per work item
constexpr int kMaxKB = 16;                 // k-blocks of a K row (D = 128: at most 12)
constexpr int kItemEnd = -1;               // stage record: no more items for this consumer
constexpr long long kWaitCycles = 4000000000ll;  // limit of every wait on a tile copy: ~2 s at GB300 clocks
constexpr long long kMinWaitCycles = 100000;     // shortest limit the timeout self-test may ask for

// Bytes of the fixed part of the decode kernel's shared memory (before the rings): the K B-fragments
// (16 bytes per k-block and lane), zone-C query fragments, slot table, k-block offsets, stage
// barriers and records, the fused step's new row, the head's K metadata and the group's query rows.
__host__ __device__ constexpr int64_t decode_fixed_smem(int D, int NC) {
  return ((int64_t)kMaxKB * 32 * 16 + (int64_t)(D / 16) * 32 * 16 + (int64_t)(D + kSlotPad) * 2 + kMaxKB * 8 +
          (int64_t)NC * kStages * 24 + (int64_t)2 * D * 2 + (int64_t)(D + kSlotPad) * 4 +
          (int64_t)8 * D * 4 + 127) /
         128 * 128;
}
// Floats of one block's partial result (m, l, o for G heads), rounded up to a multiple of 4.
__host__ __device__ constexpr int partial_stride(int G, int D) { return decode_partial_stride(G, D); }

// The consumer warps' partial results are combined in the ring area once every ring is drained.
__host__ __device__ constexpr int64_t decode_reduce_bytes(int D, int NC) { return (int64_t)NC * 8 * (D + 2) * 4; }

// One cache attended by a launch: its zones, its zone-C length and capacity and its plan's head
// records and slot tables.  A launch attends one cache, or several sharing the query (segments
// moved out of zone C and the live cache): the softmax then runs over the union of their keys.
struct DecodePart {
  const uint8_t* zone_a;
  const uint16_t* zone_b;
  const uint16_t* zone_c_k;
  const uint16_t* zone_c_v;
  int32_t* len_dev;
  const rdkv_head_plan* heads;
  const int16_t* slots;
  const int32_t* zc_pages;  // zone-C page table, or NULL (contiguous)
  int zc_page_stride;
  int cap_c;
  const int32_t* a_pages;   // zone-A page table, or NULL (contiguous)
  const int32_t* b_pages;   // zone-B page table, or NULL (contiguous)
};

struct DecodeParams {
  const void* plan;
  const uint8_t* zone_a;
  const uint16_t* zone_b;
  const uint16_t* zone_c_k;
  const uint16_t* zone_c_v;
  const void* q;
  float* partial;   // [n_heads][splits][G][D + 2]
  int32_t* error;   // device status word
  int32_t* tickets; // [n_heads] blocks finished per head (zeroed before the launch)
  float* out;       // [batch][h_q][D]
  float* lse;       // [batch][h_q] natural-log softmax denominators, or NULL
  int32_t* len_dev;        // zone-C rows in use (advanced by the fused step)
  const void* k_new;       // fused step: the new token's K and V [batch][h_kv][D] (dtype), else NULL
  const void* v_new;
  int32_t* gticket;        // fused step: heads merged so far (zero between launches)
  const rdkv_head_plan* heads;  // the plan's head records (offset fixed by the shape)
  const int16_t* slots;         // the plan's slot tables, slot_stride entries per head
  int dtype, h_q, h_kv, cap_c, ring_bytes, ring_warps, ctas, n_heads, slot_stride;
  int dealt;                    // 1: blocks dealt to heads on the host (below); 0: by the kernel
  int ragged;                   // 1: part p is sequence p of a ragged batch (batch 1 each); the dealt head
                                //    index h means sequence h / h_kv, head h % h_kv of that cache
  long long wait_cycles;        // limit of each wait on a stage's barrier (clock64 cycles)
  int arm_only;                 // timeout self-test: stages are armed for bytes that no copy delivers
  uint8_t block_head[kMaxDealtBlocks];       // head of each block, kNoHead for a block without work
  int16_t head_first[RDKV_COST_HEADS + 1];   // first block of each head; [n_heads] = end
  // host dealing over several caches: each block reads one cache (block_part) and takes items
  // block_split, block_split + block_nsplit, ... of that cache's head; the blocks of a head over all
  // caches share its partials, ticket and merge.  One cache: part 0, the block's split of the head.
  uint8_t block_part[kMaxDealtBlocks], block_split[kMaxDealtBlocks], block_nsplit[kMaxDealtBlocks];
  DecodePart parts[kMaxParts];  // parts[0] is the cache of the fields above
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking probe of a phase (the producer polls its consumers' empty barriers with it).
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait; false when the limit (clock64 cycles) ran out.  The clock is read only when the
// first probe finds the phase still open.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}
// L2 policy of the staged zone data: evicted first, so that the small data every call re-reads
// (plan records, slot tables, queries, the split partials) stays in L2 across the layers.
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void bulk_copy_once(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                               uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// the consumer warps alone (named barrier 1)
template <int NC>
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(NC * 32) : "memory"); }
// atomic add of 1 with acquire-release semantics at GPU scope; returns the old value
__device__ __forceinline__ int ticket_acq_rel(int32_t* p) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(old) : "l"(p) : "memory");
  return old;
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
// Shared-memory loads through typed pointers into the block's shared window, so
// the compiler folds constant offsets into the address ([reg + imm]).
// Loads from a 32-bit shared-memory address (no generic-address arithmetic per access).  Volatile:
// they keep their place among the mbarrier waits and arrivals that guard the staged data.
__device__ __forceinline__ uint4 lds128_s(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64_s(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t pick4(const uint4& v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }
// (x >> 8) & 0x00ff00ff in one byte permute: bytes 1 and 3 to bytes 0 and 2, zeros above
__device__ __forceinline__ uint32_t high_bytes(uint32_t x) { return __byte_perm(x, 0u, 0x4341u); }

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// (x0, x1) and (x2, x3) as fp16 pairs: high parts {x, y}, remainders {z, w}; hi + lo keeps ~22 bits.
__device__ __forceinline__ uint4 split_hi_lo(float x0, float x1, float x2, float x3) {
  const __half2 h01 = __floats2half2_rn(x0, x1), h23 = __floats2half2_rn(x2, x3);
  const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
  uint4 r;
  r.x = *reinterpret_cast<const uint32_t*>(&h01);
  r.y = *reinterpret_cast<const uint32_t*>(&h23);
  r.z = pack_half2(x0 - f01.x, x1 - f01.y);
  r.w = pack_half2(x2 - f23.x, x3 - f23.y);
  return r;
}

// 2^x by the SFU's approximate base-2 exponential (relative error about 2^-22; results below
// the normal range flush to zero, which the softmax weights can afford)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------- per-warp state
template <int D>
struct WarpAcc {
  float o[D / 16][4];   // O^T fragments: (ch 16cm+g, heads 2q, 2q+1), (ch 16cm+g+8, ...)
  float z[4];           // zero-point products of packed V: row g = channel group g, heads 2q, 2q+1
  float m[2];           // running max (base 2) of heads 2q, 2q+1
  float l[2];           // this lane's share of the running sum
};

// Softmax update for NTB token blocks of S^T accumulators; returns P^T B-fragments.  The
// reference max m of a head is raised only when a tile's max exceeds it by more than kLazy
// (base 2), and then for every head of the warp at once (a warp-uniform branch), so most tiles
// skip the rescale of the accumulators; p = 2^(s - m) <= 2^kLazy stays well inside fp16.
constexpr float kLazy = 8.f;
template <int D, int NTB>
__device__ __forceinline__ void softmax_update(WarpAcc<D>& acc, float (&s)[NTB][4], uint32_t (&pb)[NTB][2]) {
  float mt0 = -INFINITY, mt1 = -INFINITY;
#pragma unroll
  for (int tb = 0; tb < NTB; ++tb) {
    mt0 = fmaxf(mt0, fmaxf(s[tb][0], s[tb][2]));
    mt1 = fmaxf(mt1, fmaxf(s[tb][1], s[tb][3]));
  }
  // a rescale is due when some head's tile max passes its reference by kLazy (a -inf reference:
  // no token seen yet, passes as soon as a finite logit comes)
  const bool due = mt0 > acc.m[0] + kLazy || mt1 > acc.m[1] + kLazy;
  if (__any_sync(0xffffffffu, due)) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mt0 = fmaxf(mt0, __shfl_xor_sync(0xffffffffu, mt0, o));
      mt1 = fmaxf(mt1, __shfl_xor_sync(0xffffffffu, mt1, o));
    }
    const float mn0 = fmaxf(acc.m[0], mt0), mn1 = fmaxf(acc.m[1], mt1);
    const float al0 = acc.m[0] == -INFINITY ? 0.f : ex2(acc.m[0] - mn0);
    const float al1 = acc.m[1] == -INFINITY ? 0.f : ex2(acc.m[1] - mn1);
    acc.m[0] = mn0;
    acc.m[1] = mn1;
    acc.l[0] *= al0;
    acc.l[1] *= al1;
    acc.z[0] *= al0;
    acc.z[1] *= al1;
#pragma unroll
    for (int cm = 0; cm < D / 16; ++cm) {
      acc.o[cm][0] *= al0;
      acc.o[cm][1] *= al1;
      acc.o[cm][2] *= al0;
      acc.o[cm][3] *= al1;
    }
  }
  // all tokens so far masked: keep everything at zero
  const float ref0 = acc.m[0] == -INFINITY ? 0.f : acc.m[0], ref1 = acc.m[1] == -INFINITY ? 0.f : acc.m[1];
  float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
  for (int tb = 0; tb < NTB; ++tb) {
    const float p0 = ex2(s[tb][0] - ref0), p1 = ex2(s[tb][1] - ref1);
    const float p2 = ex2(s[tb][2] - ref0), p3 = ex2(s[tb][3] - ref1);
    ps0 += p0 + p2;
    ps1 += p1 + p3;
    pb[tb][0] = movmatrix_trans(pack_half2(p0, p1));
    pb[tb][1] = movmatrix_trans(pack_half2(p2, p3));
  }
  acc.l[0] += ps0;
  acc.l[1] += ps1;
}

// K logits of one width segment W of a zone-A tile, k-blocks [kb0, kb1) (the segment's blocks are
// consecutive: 64 W bytes of words apart, the first at wb0).  Lane (g, q) reads tokens g, g+8, g+16,
// g+24 of its word of each block (one 16-byte load) and makes its two A registers per token with
// one mask each (W = 2: bits 2q and, after a shift by 8, 2q + 8; W = 4: bits 0 and 4 after a shift
// by 8 (q & 1); W = 8: bytes 0, 2 and 1, 3); B (built once per block) carries the 2^-pos of those
// positions.  PK: hi and lo share one MMA (B columns 0-3 hi, 4-7 lo); else hi products go to shi and
// lo products to slo.
template <int W, bool PK>
__device__ __forceinline__ void k_segment(uint32_t kw, uint32_t wb0, int kb0, int kb1, uint32_t bfr, int lane,
                                          float (&shi)[2][4], float (&slo)[2][4], int nrem16) {
  if (kb0 >= kb1) return;
  const int g = lane >> 2, q = lane & 3;
  // this lane's byte offset from a block's first word: its word index times 128, its tokens 16 g
  // (a partial 8- or 4-bit block's lanes past its last word read the next words of the tile: codes
  // of other slots or V bytes, always in the staged item, met by B = 0)
  const uint32_t c0 = 128u * (W == 16 ? q : W == 8 ? q : W == 4 ? (q >> 1) : 0) + 16u * g;
  const uint32_t c1 = 128u * (q + 4) + 16u * g;  // W = 16: the word of slots 2q + 8, 2q + 9
  const uint32_t m2 = 0x00030003u << (2 * q);
  const int sh4 = 8 * (q & 1);
  uint32_t wb = kw + wb0;                            // shared address of the block's first word
  uint32_t bp = bfr + 16u * (uint32_t)(kb0 * 32 + lane);  // this lane's B entry of the block
#pragma unroll 2
  for (int kb = kb0; kb < kb1; ++kb, wb += 64u * W, bp += 512u) {
    const uint4 bq = lds128_s(bp);
    const uint4 y0 = lds128_s(wb + c0);
    uint4 y1 = y0;
    uint32_t k0 = ~0u, k1 = ~0u;
    if (W == 16) {
      // raw fp16 words past the segment's last real word (the next segment's, or past the staged
      // tile) are not read: such a lane reads its first word again and masks both to zero
      const int nrem = kb == kb1 - 1 ? nrem16 : kKB;
      k0 = 2 * q < nrem ? ~0u : 0u;
      k1 = 2 * q + 8 < nrem ? ~0u : 0u;
      y1 = lds128_s(wb + (k1 ? c1 : c0));
    }
#pragma unroll
    for (int tb = 0; tb < 2; ++tb) {
      const uint32_t x0 = pick4(y0, 2 * tb), x1 = pick4(y0, 2 * tb + 1);  // tokens g + 16 tb, g + 8 + 16 tb
      uint32_t a0, a1, a2, a3;
      if (W == 16) {
        a0 = x0 & k0;
        a1 = x1 & k0;
        a2 = pick4(y1, 2 * tb) & k1;
        a3 = pick4(y1, 2 * tb + 1) & k1;
      } else if (W == 8) {
        a0 = x0 & 0x00ff00ffu;
        a1 = x1 & 0x00ff00ffu;
        a2 = high_bytes(x0);
        a3 = high_bytes(x1);
      } else if (W == 4) {
        const uint32_t t0 = x0 >> sh4, t1 = x1 >> sh4;
        a0 = t0 & 0x000f000fu;
        a1 = t1 & 0x000f000fu;
        a2 = t0 & 0x00f000f0u;
        a3 = t1 & 0x00f000f0u;
      } else {
        a0 = x0 & m2;
        a1 = x1 & m2;
        a2 = (x0 >> 8) & m2;
        a3 = (x1 >> 8) & m2;
      }
      mma16816(shi[tb], a0, a1, a2, a3, bq.x, bq.y);
      if (!PK) mma16816(slo[tb], a0, a1, a2, a3, bq.z, bq.w);
    }
  }
}

// Logits (base 2, with the per-head zero-point term) of the 32 tokens of a zone-A tile:
// raw 16-bit channels first at scale 1, then the accumulators move to 2^-24 and take the
// quantised segments' products (codes as fp16 subnormals), then back, times log2(e)/sqrt(D).
template <bool PK>
__device__ __forceinline__ void tile_logits(uint32_t kw, const int (&seg_kb)[5], const uint32_t (&seg_wb)[4],
                                            int nrem16, uint32_t bfr, int lane, float c24, float b0, float b1,
                                            float (&s)[2][4]) {
  float slo[2][4];
#pragma unroll
  for (int tb = 0; tb < 2; ++tb)
#pragma unroll
    for (int e = 0; e < 4; ++e) s[tb][e] = slo[tb][e] = 0.f;
  if (seg_kb[1] > seg_kb[0]) {
    k_segment<16, PK>(kw, seg_wb[0], seg_kb[0], seg_kb[1], bfr, lane, s, slo, nrem16);
#pragma unroll
    for (int tb = 0; tb < 2; ++tb)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s[tb][e] *= 5.9604644775390625e-8f;
        slo[tb][e] *= 5.9604644775390625e-8f;
      }
  }
  k_segment<8, PK>(kw, seg_wb[1], seg_kb[1], seg_kb[2], bfr, lane, s, slo, kKB);
  k_segment<4, PK>(kw, seg_wb[2], seg_kb[2], seg_kb[3], bfr, lane, s, slo, kKB);
  k_segment<2, PK>(kw, seg_wb[3], seg_kb[3], seg_kb[4], bfr, lane, s, slo, kKB);
  // PK: the lo columns (2q + 4, 2q + 5) are held by lane q ^ 2
#pragma unroll
  for (int tb = 0; tb < 2; ++tb) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float t = s[tb][e] + (PK ? __shfl_xor_sync(0xffffffffu, s[tb][e], 2) : slo[tb][e]);
      s[tb][e] = fmaf(t, c24, (e & 1) ? b1 : b0);
    }
  }
}

// Exponent of the power of two the products of V class `vb` (2, 4, 8; 16 = fp16 rows) carry in
// the accumulators of channel block cm: 2^-24 for the subnormal codes times 2^pos of the code's
// bit position inside its half-word (below 8 after the optional shift by 8).
__device__ __forceinline__ int v_scale_exp(int vb, int cm) {
  return vb == 16 ? 0 : vb == 2 ? -24 + 2 * (cm & 3) : vb == 4 ? -24 + 4 * (cm & 1) : -24;
}

// Moves the O^T accumulators from the scale of V class `from` to that of class `to` (powers of
// two per channel block: exact).
template <int D>
__device__ __forceinline__ void rescale_o(WarpAcc<D>& acc, int from, int to) {
#pragma unroll
  for (int cm = 0; cm < D / 16; ++cm) {
    const float f = __int_as_float((127 + v_scale_exp(to, cm) - v_scale_exp(from, cm)) << 23);
    acc.o[cm][0] *= f;
    acc.o[cm][1] *= f;
    acc.o[cm][2] *= f;
    acc.o[cm][3] *= f;
  }
}

// One code field of a V word: element e of the word (bit VB e of each half), as an fp16 subnormal
// pair at bit position (VB e) mod 8 -- positions 8 and up are shifted down by 8 first.
template <int VB>
__device__ __forceinline__ uint32_t v_field(uint32_t x, int e) {
  constexpr uint32_t m = VB == 8 ? 0x00ff00ffu : VB == 4 ? 0x000f000fu : 0x00030003u;
  const int pos = VB * e;
  if (VB == 8) return pos == 0 ? (x & m) : high_bytes(x);
  return pos < 8 ? (x & (m << pos)) : ((x >> 8) & (m << (pos - 8)));
}

// PV of a zone-A tile with packed V of width VB.  A dequantised V element is
// zero + scale * code per (token, 32-channel group), so per head h and channel c
//   O[h][c] += sum_t (p_ht scale_t) code_tc + sum_t p_ht zero_t.
// Lane (g, q) of 16-token block tb owns 2 nw consecutive code words (its two token pairs): entry k
// of its channel list (channel 16 (k mod D/16) + 8 (k div D/16) + g) sits in word k / per at
// element k mod per.  B = p * scale of the channel group (one half2 multiply per fragment); the
// zero-point sums go to acc.z through one MMA per 16 tokens whose A row g holds the zeros of
// channel group g.
template <int D, int VB>
__device__ __forceinline__ void tile_pv_packed(WarpAcc<D>& acc, uint32_t vcodes, uint32_t vmeta, int lane,
                                               const uint32_t (*pb)[2]) {
  const int g = lane >> 2, q = lane & 3;
  constexpr int CM = D / 16, NG = D / 32, NW = D * VB / 128, PER = 16 / VB;
#pragma unroll
  for (int tb = 0; tb < 2; ++tb) {
    // scales of the lane's two pairs for every group (h = 0, then h = 1), 2 NG words
    uint32_t sc[2 * NG];
    const uint32_t sp = vmeta + 4u * ((tb * 4 + q) * 2 * NG);
#pragma unroll
    for (int i = 0; i < 2 * NG; i += 4) {
      const uint4 t = lds128_s(sp + 4u * i);
      sc[i] = t.x; sc[i + 1] = t.y; sc[i + 2] = t.z; sc[i + 3] = t.w;
    }
    uint2 za = make_uint2(0u, 0u);
    if (g < NG) za = lds64_s(vmeta + 4u * (16 * NG + ((tb * NG + g) * 4 + q) * 2));
    mma16816(acc.z, za.x, 0u, za.y, 0u, pb[tb][0], pb[tb][1]);
    uint32_t bb[2][NG];
#pragma unroll
    for (int grp = 0; grp < NG; ++grp) {
      const __half2 h0 = __hmul2(*reinterpret_cast<const __half2*>(&pb[tb][0]), *reinterpret_cast<const __half2*>(&sc[grp]));
      const __half2 h1 = __hmul2(*reinterpret_cast<const __half2*>(&pb[tb][1]), *reinterpret_cast<const __half2*>(&sc[NG + grp]));
      bb[0][grp] = *reinterpret_cast<const uint32_t*>(&h0);
      bb[1][grp] = *reinterpret_cast<const uint32_t*>(&h1);
    }
    // the lane's code words: pair h = 0 then h = 1, NW words each
    uint32_t wd[2 * NW];
    const uint32_t cp = vcodes + 4u * (((tb * 8 + g) * 4 + q) * 2 * NW);
#pragma unroll
    for (int i = 0; i < 2 * NW; i += 4) {
      if (2 * NW >= 4) {
        const uint4 t = lds128_s(cp + 4u * i);
        wd[i] = t.x; wd[i + 1] = t.y; wd[i + 2] = t.z; wd[i + 3] = t.w;
      }
    }
    if (2 * NW == 2) {
      const uint2 t = lds64_s(cp);
      wd[0] = t.x; wd[1] = t.y;
    }
#pragma unroll
    for (int cm = 0; cm < CM; ++cm) {
      const int k0 = cm, k1 = CM + cm;  // the lane's entries for rows g and g + 8
      const uint32_t a0 = v_field<VB>(wd[k0 / PER], k0 % PER);
      const uint32_t a1 = v_field<VB>(wd[k1 / PER], k1 % PER);
      const uint32_t a2 = v_field<VB>(wd[NW + k0 / PER], k0 % PER);
      const uint32_t a3 = v_field<VB>(wd[NW + k1 / PER], k1 % PER);
      mma16816(acc.o[cm], a0, a1, a2, a3, bb[0][cm / 2], bb[1][cm / 2]);
    }
  }
}

// PV over fp16 V rows [rows][D] in shared memory (zone B tile or zone C block).
template <int D, int NTB>
__device__ __forceinline__ void pv_fp16(WarpAcc<D>& acc, uint32_t vrows, int lane, const uint32_t (&pb)[NTB][2]) {
  const int mi = lane >> 3, r = lane & 7;
#pragma unroll
  for (int tb = 0; tb < NTB; ++tb) {
#pragma unroll
    for (int cm = 0; cm < D / 16; ++cm) {
      const int row = 16 * tb + (mi >> 1) * 8 + r;
      const int col = 16 * cm + (mi & 1) * 8;
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(vrows + 2u * (row * D + col), a0, a1, a2, a3);
      mma16816(acc.o[cm], a0, a1, a2, a3, pb[tb][0], pb[tb][1]);
    }
  }
}

// One zone-A tile of class cls (class 3: its zone-B rows follow the tile's tb bytes): logits, the
// tokens past the kept ones masked (the last tile of a class), the softmax update, the accumulators
// moved to the class's scale, PV.
template <int D, bool PK>
__device__ __forceinline__ void consume_tile(WarpAcc<D>& acc, int& o_mode, uint32_t stp, uint32_t tb_bytes,
                                             int cls, int n_real, int RW, const int (&seg_kb)[5],
                                             const uint32_t (&seg_wb)[4], int nrem16, uint32_t bfr, int lane,
                                             float c24, float bias0, float bias1) {
  const int g = lane >> 2;
  float s[2][4];
  tile_logits<PK>(stp, seg_kb, seg_wb, nrem16, bfr, lane, c24, bias0, bias1, s);
  if (n_real < kTile) {
#pragma unroll
    for (int tb = 0; tb < 2; ++tb) {
      const bool va = 16 * tb + g < n_real, vb = 16 * tb + g + 8 < n_real;
      s[tb][0] = va ? s[tb][0] : -INFINITY;
      s[tb][1] = va ? s[tb][1] : -INFINITY;
      s[tb][2] = vb ? s[tb][2] : -INFINITY;
      s[tb][3] = vb ? s[tb][3] : -INFINITY;
    }
  }
  uint32_t pb[2][2];
  softmax_update<D, 2>(acc, s, pb);
  const int vb_cls = 2 << cls;
  if (vb_cls != o_mode) {
    rescale_o<D>(acc, o_mode, vb_cls);
    o_mode = vb_cls;
  }
  const uint32_t vcodes = stp + 4u * kTile * RW;
  if (cls == 0) tile_pv_packed<D, 2>(acc, vcodes, vcodes + kTile * D * 2 / 8, lane, pb);
  else if (cls == 1) tile_pv_packed<D, 4>(acc, vcodes, vcodes + kTile * D * 4 / 8, lane, pb);
  else if (cls == 2) tile_pv_packed<D, 8>(acc, vcodes, vcodes + kTile * D * 8 / 8, lane, pb);
  else pv_fp16<D, 2>(acc, stp + tb_bytes, lane, pb);
}

// Estimated decode cost of a head: its zone-A tiles and its zone-C blocks.
__host__ __device__ __forceinline__ int64_t head_cost(const rdkv_head_plan& hp, int zc_blocks) {
  return head_cost_a(hp) + (int64_t)zc_blocks * kZoneCBlockCost;
}

// Per-class values of a head, read with a class index without dynamic array indexing.
struct ClassVals {
  int64_t v[4];
  __device__ __forceinline__ int64_t operator()(int c) const { return c == 0 ? v[0] : c == 1 ? v[1] : c == 2 ? v[2] : v[3]; }
};

template <int D, bool PK, int NC>
__global__ void __launch_bounds__((NC + 1) * 32, NC == kConsumersWide ? 1 : 2)
    decode_kernel(const __grid_constant__ DecodeParams P) {
  constexpr int kConsumers = NC;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = P.h_q / P.h_kv;
  // the next kernel on the stream may start its own static setup once every block of this one runs
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ int asg[3];  // head, first block of the head, blocks of the head
  __shared__ __align__(16) rdkv_head_plan hp_s;  // this block's head record
  __shared__ float bias_s[8];                    // zero-point term of each query head (base 2)
  __shared__ int next_k;                         // the block's next item (producer warp)
  __shared__ int abort_s;                        // a bounded wait ran out somewhere in the block
  __shared__ int is_last;
  int16_t slot_pre = -1;  // dealt on the host: this thread's slot-table entry, loaded with the record
  // the cache this block reads (part 0 unless the host dealt blocks over several caches)
  const DecodePart& PP = P.parts[P.dealt ? P.block_part[blockIdx.x] : 0];
  if (P.dealt) {
    // dealt on the host: this block's head and split range are kernel arguments
    const int hb = P.block_head[blockIdx.x];
    const int hbc = P.ragged ? hb % P.h_kv : hb;  // the head within its cache
    if (hb != kNoHead && tid < P.slot_stride) slot_pre = PP.slots[(int64_t)hbc * P.slot_stride + tid];
    if (warp == 0) {
      if (lane == 0) {
        asg[0] = hb == kNoHead ? -1 : hb;
        asg[1] = hb == kNoHead ? 0 : P.head_first[hb];
        asg[2] = hb == kNoHead ? 0 : P.head_first[hb + 1] - P.head_first[hb];
      }
      if (hb != kNoHead)  // the head record into shared memory, one word per lane
        reinterpret_cast<int32_t*>(&hp_s)[lane] = reinterpret_cast<const int32_t*>(PP.heads + hbc)[lane];
    }
  } else if (warp == 0) {
    // Blocks are dealt to heads in proportion to their estimated cost (cumulative rounding), at least
    // one per head, over a nominal P.ctas blocks; the grid has P.ctas + n_heads blocks and the blocks
    // past the last head's range leave at once.  Warp 0: one lane per head, one round trip for the
    // plan records, then a scan.  Static inputs only (plan and capacity): the dealing is the same in
    // every launch, also before the previous kernel on the stream has finished.
    const int zc = ceil_div(P.cap_c, kCRows);
    int64_t total = 0;
    for (int h = lane; h < P.n_heads; h += 32) total += head_cost(P.heads[h], zc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
    int start = 0, found = -1;
    int64_t wbase = 0;  // cost of the heads before this round of 32
    for (int h0 = 0; h0 < P.n_heads; h0 += 32) {
      const int h = h0 + lane;
      const int64_t w = h < P.n_heads ? head_cost(P.heads[h], zc) : 0;
      // the head's share of the nominal blocks by cumulative rounding (the shares add up to P.ctas),
      // at least one
      int64_t wincl = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t v = __shfl_up_sync(0xffffffffu, wincl, o);
        if (lane >= o) wincl += v;
      }
      const int64_t lo = total > 0 ? (wbase + wincl - w) * P.ctas / total : 0;
      const int64_t hi = total > 0 ? (wbase + wincl) * P.ctas / total : 0;
      wbase += __shfl_sync(0xffffffffu, wincl, 31);
      const int c = h < P.n_heads ? max(1, (int)(hi - lo)) : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const int first = start + incl - c;
      if (c > 0 && (int)blockIdx.x >= first && (int)blockIdx.x < first + c) {
        asg[0] = h;
        asg[1] = first;
        asg[2] = c;
        found = h;
      }
      start += __shfl_sync(0xffffffffu, incl, 31);
    }
    const unsigned any = __ballot_sync(0xffffffffu, found >= 0);
    const int head_found = any ? __shfl_sync(0xffffffffu, found, __ffs(any) - 1) : -1;
    if (lane == 0 && !any) asg[0] = -1;
    if (head_found >= 0)  // the head record into shared memory, one word per lane
      reinterpret_cast<int32_t*>(&hp_s)[lane] = reinterpret_cast<const int32_t*>(P.heads + head_found)[lane];
  }
  __syncthreads();
  if (asg[0] < 0) return;
  const int head = asg[0], split = (int)blockIdx.x - asg[1], n_split = asg[2], first_block = asg[1];
  // items of this block's cache: isplit, isplit + in_split, ...
  const int isplit = P.dealt ? (int)P.block_split[blockIdx.x] : split;
  const int in_split = P.dealt ? (int)P.block_nsplit[blockIdx.x] : n_split;
  const int b = head / P.h_kv, j = head % P.h_kv;     // sequence (the part, when ragged) and KV head
  const int hc = P.ragged ? j : head;                 // the head within its cache: record, slots, zone C
  const rdkv_head_plan* hpp = &hp_s;
  const bool fused = P.k_new != nullptr;
  const int qbase = b * P.h_q + j * G;
  const int16_t* slot_ch = PP.slots + (int64_t)hc * P.slot_stride;
  const int k_slots = hpp->k_slots;  // <= D + kSlotPad <= the block's threads
  const int16_t sr = tid < k_slots ? (P.dealt ? slot_pre : slot_ch[tid]) : (int16_t)-1;

  // shared memory map
  uint4* bfr = reinterpret_cast<uint4*>(smem);                                     // [kMaxKB][32]
  uint4* qfragc = bfr + kMaxKB * 32;                                               // [D/16][32] hi, lo
  int16_t* slot_s = reinterpret_cast<int16_t*>(qfragc + (D / 16) * 32);            // [D + kSlotPad]
  uint32_t* kb_wb = reinterpret_cast<uint32_t*>(slot_s + D + kSlotPad);            // [kMaxKB] (unused entries 0)
  int* seg_kb_s = reinterpret_cast<int*>(kb_wb + kMaxKB);                          // [kMaxKB]: [0..4] block ranges
  uint64_t* full = reinterpret_cast<uint64_t*>(seg_kb_s + kMaxKB);                 // [consumers][stages]
  uint64_t* empty = full + kConsumers * kStages;                                   // [consumers][stages]
  int* st_pos = reinterpret_cast<int*>(empty + kConsumers * kStages);              // [consumers][stages]
  int* st_item = st_pos + kConsumers * kStages;                                    // [consumers][stages]
  uint16_t* newrow = reinterpret_cast<uint16_t*>(st_item + kConsumers * kStages);  // [2][D] fused step: k, v
  uint32_t* kmeta_s = reinterpret_cast<uint32_t*>(newrow + 2 * D);                 // [D + kSlotPad] {scale, zero}
  float* q_s = reinterpret_cast<float*>(kmeta_s + D + kSlotPad);                   // [8][D] the group's queries
  unsigned char* ring = smem + decode_fixed_smem(D, NC);
  float* red = reinterpret_cast<float*>(ring);                                     // [consumers][8][D + 2], after the loop

  // items of this head: its tiles in class order, then its zone-C blocks
  ClassVals cstart, coff, ctb, cnv;  // first item, first byte in zone A, tile bytes, kept tokens per class
  int zc_start;
  {
    int t = 0;
    int64_t off = hpp->a_off + head_meta_bytes(hpp->meta_slots);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      cstart.v[c] = t;
      coff.v[c] = off;
      ctb.v[c] = hpp->tile_bytes[c];
      cnv.v[c] = hpp->n_v[c];
      t += hpp->tiles[c];
      off += (int64_t)hpp->tiles[c] * hpp->tile_bytes[c];
    }
    zc_start = t;
  }
  const int64_t b_row = hpp->b_row;
  const int RW = hpp->row_words;
  if (tid == 0) {
    next_k = 0;
    abort_s = 0;
  }
  // k-block ranges of the width segments (16, 8, 4, 2 bits) and each block's first K word (bytes)
  if (warp == 1 && lane < kMaxKB) {
    int nb[4], wfirst[4];
    int nkb = 0, wsum = 0;
#pragma unroll
    for (int seg = 0; seg < 4; ++seg) {
      const int w = 16 >> seg;
      nb[seg] = nkb;
      wfirst[seg] = wsum;
      nkb += ceil_div(hpp->k_words[seg] * (32 / w), kKB);
      wsum += hpp->k_words[seg];
    }
    auto pick = [](const int (&a)[4], int i) { return i == 0 ? a[0] : i == 1 ? a[1] : i == 2 ? a[2] : a[3]; };
    if (lane < 4) seg_kb_s[lane] = pick(nb, lane);
    if (lane == 4) seg_kb_s[4] = nkb;
    uint32_t wb = 0;
    if (lane < nkb) {
      const int seg = (lane >= nb[1]) + (lane >= nb[2]) + (lane >= nb[3]);
      const int w = 16 >> seg;
      wb = 128u * (uint32_t)(pick(wfirst, seg) + (lane - pick(nb, seg)) * (w / 2));
    }
    kb_wb[lane] = wb;
  }
  if (tid < kConsumers * kStages) {
    mbar_init(&full[tid], 1);
    mbar_init(&empty[tid], 1);
  }
  if (tid == 0) asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  if (tid < k_slots) slot_s[tid] = sr;
  // the head's K metadata (zone A: static, may be read before the wait for the previous kernel)
  if (tid < hpp->meta_slots)
    kmeta_s[tid] = __ldg(reinterpret_cast<const uint32_t*>(PP.zone_a + zone_a_offset(PP.a_pages, hpp->a_off + 4 * tid)));
  __syncthreads();  // next_k, the barriers, the k-block ranges, the slot table and K metadata are set

  auto item_cls = [&](int it) {
    return it < (int)cstart.v[1] ? 0 : it < (int)cstart.v[2] ? 1 : it < (int)cstart.v[3] ? 2 : it < zc_start ? 3 : -1;
  };
  // a consumer warp's softmax state and output accumulators (unused in the producer warp)
  WarpAcc<D> acc;
#pragma unroll
  for (int cm = 0; cm < D / 16; ++cm) acc.o[cm][0] = acc.o[cm][1] = acc.o[cm][2] = acc.o[cm][3] = 0.f;
  acc.z[0] = acc.z[1] = acc.z[2] = acc.z[3] = 0.f;
  acc.m[0] = acc.m[1] = -INFINITY;
  acc.l[0] = acc.l[1] = 0.f;

  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer warp
    // lane w serves consumer warp w: its ring [ring_bytes] holds up to kStages items; an item is
    // taken from the block's counter when the ring has room for it, copied in with bulk copies that
    // complete on the stage's full barrier, and its bytes come back when the consumer arrives on the
    // stage's empty barrier.  After the last item, a stage with the record kItemEnd ends the consumer.
    const bool serve = lane < kConsumers;
    const bool has_ring = lane < P.ring_warps;
    unsigned char* wring = ring + (int64_t)lane * P.ring_bytes;
    int issued = 0, released = 0, pending = -1;
    uint32_t head_p = 0, used = 0, need[kStages] = {};
    bool drained = !has_ring, ended = !serve, items_final = false;
    int n_items = zc_start, len_c = 0;
    int cap = kPrologueItems;
    long long idle0 = clock64();
    bool timed_out = false;
    auto step = [&]() -> bool {  // one round of this lane's work; true if anything moved
      bool moved = false;
      if (ended) return false;
      // stages the consumer has released
      while (issued > released && mbar_test(&empty[lane * kStages + released % kStages], (uint32_t)(released / kStages) & 1u)) {
        used -= need[released % kStages];
        ++released;
        moved = true;
      }
      if (issued == released) head_p = used = 0;  // empty ring: start at its beginning
      while (!drained && issued - released < cap) {
        int it = pending;
        if (it < 0) it = isplit + in_split * atomicAdd(&next_k, 1);
        if (it >= n_items) {
          if (items_final) drained = true;
          else pending = it;
          break;
        }
        const int cls = item_cls(it);
        uint32_t sz, a_bytes = 0;
        int c_row = 0;
        if (cls >= 0) {
          a_bytes = (uint32_t)ctb(cls);
          sz = (uint32_t)align_up(a_bytes + (cls == 3 ? kTile * D * 2 : 0), 128);
        } else {
          c_row = (it - zc_start) * kCRows;
          sz = 2u * kCRows * D * 2;
        }
        // the held bytes end at head_p (circularly); a copy that does not fit before the end of the
        // ring starts at its beginning and also holds the skipped tail until it is released
        uint32_t phys = head_p, nd = sz;
        if (phys + sz > (uint32_t)P.ring_bytes) { nd += (uint32_t)P.ring_bytes - phys; phys = 0; }
        if (used + nd > (uint32_t)P.ring_bytes) {
          pending = it;
          break;
        }
        pending = -1;
        head_p = phys + sz;
        used += nd;
        const int slot = issued % kStages;
        need[slot] = nd;
        const int sidx = lane * kStages + slot;
        st_pos[sidx] = (int)phys;
        st_item[sidx] = ((cls + 1) << 24) | (cls >= 0 ? it - (int)cstart(cls) : it - zc_start);
        unsigned char* dst = wring + phys;
        uint64_t* bar = &full[sidx];
        if (P.arm_only) {
          // timeout self-test: the stage waits for 16 bytes and no copy is issued, so its wait runs out
          mbar_arrive_expect_tx(bar, 16u);
        } else if (cls >= 0) {
          const int ti = it - (int)cstart(cls);
          const uint32_t zb = cls == 3 ? (uint32_t)kTile * D * 2 : 0u;
          mbar_arrive_expect_tx(bar, a_bytes + zb);
          const uint64_t pol = evict_first_policy();
          // zone A through its page table: a tile that crosses a page boundary comes in two copies
          const int64_t la = coff(cls) + (int64_t)ti * a_bytes;
          const uint32_t run = (uint32_t)min((int64_t)a_bytes, zone_a_run(PP.a_pages, la));
          bulk_copy_once(dst, PP.zone_a + zone_a_offset(PP.a_pages, la), run, bar, pol);
          if (run < a_bytes) bulk_copy_once(dst + run, PP.zone_a + zone_a_offset(PP.a_pages, la + run), a_bytes - run, bar, pol);
          if (zb) {  // 32 zone-B rows: two pages of 16 rows when zone B is paged (b_row is a multiple of 32)
            const int64_t r0 = b_row + (int64_t)kTile * ti;
            if (PP.b_pages) {
              bulk_copy_once(dst + a_bytes, PP.zone_b + zone_b_offset(PP.b_pages, r0, D), zb / 2, bar, pol);
              bulk_copy_once(dst + a_bytes + zb / 2, PP.zone_b + zone_b_offset(PP.b_pages, r0 + kZoneBPageRows, D), zb / 2,
                             bar, pol);
            } else {
              bulk_copy_once(dst + a_bytes, PP.zone_b + r0 * D, zb, bar, pol);
            }
          }
        } else {
          // rows of zone C (the fused step's new row, past them, is written by the consumer)
          const int rows = max(0, min(kCRows, len_c - c_row));
          const uint32_t bytes = (uint32_t)rows * D * 2;
          // a zone-C item is 16 rows: one page when zone C is paged
          const int64_t src = zone_c_offset(PP.zc_pages, PP.zc_page_stride, PP.cap_c, hc, c_row, D);
          mbar_arrive_expect_tx(bar, 2 * bytes);
          if (bytes) {
            const uint64_t pol = evict_first_policy();
            bulk_copy_once(dst, PP.zone_c_k + src, bytes, bar, pol);
            bulk_copy_once(dst + kCRows * D * 2, PP.zone_c_v + src, bytes, bar, pol);
          }
        }
        ++issued;
        moved = true;
      }
      if (drained && issued - released < kStages) {
        const int sidx = lane * kStages + issued % kStages;
        st_item[sidx] = kItemEnd;
        mbar_arrive(&full[sidx]);
        ended = true;
        moved = true;
      }
      return moved;
    };
    // zone-A items of the prologue: static data only, before the wait for the previous kernel
    if (serve) step();
    // The query, the new token and the zone-C length may come from the kernel launched just before
    // this one on the stream: wait for it here (a no-op without programmatic dependent launch).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    len_c = min(*PP.len_dev, PP.cap_c);
    n_items = zc_start + ceil_div(len_c + (fused ? 1 : 0), kCRows);
    items_final = true;
    cap = kStages;
    idle0 = clock64();
    // a consumer takes microseconds per tile and holds up to kStages of them: the producer polls its
    // empty barriers at a growing interval while nothing moves (reset by every move)
    unsigned nap = 32;
    while (true) {
      const bool moved = serve && step();
      if (__all_sync(0xffffffffu, ended)) break;
      if (__any_sync(0xffffffffu, moved)) {
        idle0 = clock64();
        nap = 32;
      } else {
        if (clock64() - idle0 > P.wait_cycles || *(volatile int*)&abort_s) {
          timed_out = true;
          break;
        }
        __nanosleep(nap);
        nap = min(nap * 2, 512u);
      }
    }
    if (timed_out) {
      if (lane == 0) {
        atomicExch(&abort_s, 1);
        atomicExch(P.error, (int)RDKV_ERR_TIMEOUT);
      }
    }
    __syncwarp();
    // before the ring area is reused: every issued stage's copies have landed (bounded, as a whole)
    if (serve && *(volatile int*)&abort_s) {
      const long long t0 = clock64();
      for (int k = released; k < issued; ++k) {
        const uint64_t* bar = &full[lane * kStages + k % kStages];
        while (!mbar_try_wait(const_cast<uint64_t*>(bar), (uint32_t)(k / kStages) & 1u))
          if (clock64() - t0 > P.wait_cycles) break;
        if (clock64() - t0 > P.wait_cycles) break;
      }
    }
  } else {
    // ------------------------------------------------------------ consumer warps
    // Everything above read only the plan and zone A, which the kernel launched just before this one
    // on the stream does not write.  The query, the new token and the zone-C length may come from
    // it: wait for it here (a no-op without programmatic dependent launch).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int len_c = min(*PP.len_dev, PP.cap_c);
    const int n_rows = len_c + (fused ? 1 : 0);
    const int nkb = seg_kb_s[4];
    const float sl2 = 1.4426950408889634f / sqrtf((float)D);
    // K B-fragments, built once: entry (k-block kb, lane (g, q)) holds B[slot][column g] for slots
    // 2q, 2q+1 (.x) and 2q+8, 2q+9 (.y) of the block (and the remainders in .z, .w without PK);
    // column g is query head g, or with PK head g & 3, hi for g < 4 and lo for g >= 4.  A quantised
    // slot's value is q * scale * 2^-pos (pos: the bit position its lane's mask leaves the code at).
    const int s_q0 = k_slots - hpp->meta_slots;   // first quantised slot
    // the group's query rows, widened to fp32 (one load per element, all in flight together)
    for (int i = tid; i < G * D; i += kConsumers * 32) q_s[i] = load_as_float(P.q, (int64_t)qbase * D + i, P.dtype);
    consumers_sync<NC>();
    for (int i = tid; i < nkb * 32; i += kConsumers * 32) {
      const int kb = i >> 5, ln = i & 31, qq = ln & 3, gg = ln >> 2;
      const int seg = (kb >= seg_kb_s[1]) + (kb >= seg_kb_s[2]) + (kb >= seg_kb_s[3]);
      const int w = 16 >> seg;
      const int hd = PK ? (gg & 3) : gg;
      const bool lo_col = PK && gg >= 4;
      float x[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int off = 2 * qq + (e & 1) + 8 * (e >> 1);
        const int slot = kKB * kb + off;
        const int ch = slot_s[slot];
        float v = 0.f;
        if (ch >= 0 && hd < G) {
          v = q_s[hd * D + ch];
          if (w < 16) {
            const uint32_t m = kmeta_s[slot - s_q0];
            const int pos = w == 2 ? 2 * qq : (w == 4 && (e >> 1)) ? 4 : 0;
            v *= __half2float(__ushort_as_half((uint16_t)(m & 0xffffu))) * __int_as_float((127 - pos) << 23);
          }
        }
        x[e] = v;
      }
      const uint4 t = split_hi_lo(x[0], x[1], x[2], x[3]);
      bfr[i] = PK ? make_uint4(lo_col ? t.z : t.x, lo_col ? t.w : t.y, 0u, 0u) : t;
    }
    // zone-C query fragments: B[k = channel pair][n = head g] in channel order, hi and lo
    for (int i = tid; i < (D / 16) * 32; i += kConsumers * 32) {
      const int kb = i >> 5, ln = i & 31, qq = ln & 3, gg = ln >> 2;
      float x[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int ch = 16 * kb + 2 * qq + (e & 1) + 8 * (e >> 1);
        x[e] = gg < G ? q_s[gg * D + ch] : 0.f;
      }
      qfragc[i] = split_hi_lo(x[0], x[1], x[2], x[3]);
    }
    // zero-point term of the quantised K channels per query head (warp h): sum_c q_hc zero_c, base 2
    for (int hq = warp; hq < 8; hq += kConsumers) {  // query head hq (0 past the group)
      float acc0 = 0.f;
      if (hq < G)
        for (int m = lane; m < hpp->meta_slots; m += 32) {
          const int ch = slot_s[s_q0 + m];
          if (ch >= 0) acc0 = fmaf(q_s[hq * D + ch], __half2float(__ushort_as_half((uint16_t)(kmeta_s[m] >> 16))), acc0);
        }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc0 += __shfl_xor_sync(0xffffffffu, acc0, o);
      if (lane == 0) bias_s[hq] = acc0 * sl2;
    }
    if (fused)
      for (int i = tid; i < 2 * D; i += kConsumers * 32) {
        const int64_t src = (int64_t)head * D + (i % D);
        newrow[i] = half_bits(load_as_float(i < D ? P.k_new : P.v_new, src, P.dtype));
      }
    consumers_sync<NC>();

    // the V class whose scale acc.o carries (2, 4, 8; 16 for fp16 rows); a warp meets the classes
    // in increasing order (items ascend), so it switches at most four times
    int o_mode = 2;
    const int g = lane >> 2, q = lane & 3;
    const float c24 = 16777216.f * sl2;
    const bool qlo = P.dtype == RDKV_F32;
    const float bias0 = bias_s[(2 * q) & 7], bias1 = bias_s[(2 * q + 1) & 7];
    int seg_kb[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) seg_kb[i] = seg_kb_s[i];
    uint32_t seg_wb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) seg_wb[i] = kb_wb[min(seg_kb[i], kMaxKB - 1)];
    const int nrem16 = 2 * hpp->k_words[0] - kKB * (seg_kb[1] - 1);  // real slots of the last raw block
    unsigned char* wring = ring + (int64_t)warp * P.ring_bytes;
    bool ok = true;
    for (int k = 0;; ++k) {
      const int sidx = warp * kStages + k % kStages;
      if (!mbar_wait(&full[sidx], (uint32_t)(k / kStages) & 1u, P.wait_cycles)) {
        ok = false;
        break;
      }
      const int rec = st_item[sidx];
      if (rec == kItemEnd) break;
      const unsigned char* stp = wring + st_pos[sidx];
      const int cls = (rec >> 24) - 1, ti = rec & 0xffffff;  // ti: tile of the class, or zone-C block
      if (cls >= 0) {
        consume_tile<D, PK>(acc, o_mode, smem_u32(stp), (uint32_t)ctb(cls), cls, min(kTile, (int)cnv(cls) - kTile * ti),
                            RW, seg_kb, seg_wb, nrem16, smem_u32(bfr), lane, c24, bias0, bias1);
      } else {
        if (o_mode != 16) {
          rescale_o<D>(acc, o_mode, 16);
          o_mode = 16;
        }
        const uint32_t st = smem_u32(stp);
        const int c_row = ti * kCRows;
        const int rows = min(kCRows, n_rows - c_row);  // rows attended (the fused step's new row last)
        const int copied = max(0, min(kCRows, len_c - c_row));
        if (rows < kCRows || copied < rows) {
          uint32_t* kz = reinterpret_cast<uint32_t*>(const_cast<unsigned char*>(stp));
          // clear the rows past the attended ones (they meet p = 0 in the products)
          for (int i = rows * D / 2 + lane; i < kCRows * D / 2; i += 32) {
            kz[i] = 0u;
            kz[kCRows * D / 2 + i] = 0u;
          }
          if (copied < rows) {  // the new row, from the staged copy of the caller's k_new, v_new
            const uint32_t* nr = reinterpret_cast<const uint32_t*>(newrow);
            for (int i = lane; i < D / 2; i += 32) {
              kz[copied * D / 2 + i] = nr[i];
              kz[kCRows * D / 2 + copied * D / 2 + i] = nr[D / 2 + i];
            }
          }
          __syncwarp();
        }
        float s[1][4] = {{0.f, 0.f, 0.f, 0.f}};
        const int mi = lane >> 3, r = lane & 7;
#pragma unroll
        for (int kb = 0; kb < D / 16; ++kb) {
          uint32_t a0, a1, a2, a3;
          const int row = (mi & 1) * 8 + r, col = 16 * kb + (mi >> 1) * 8;
          ldsm_x4(st + 2u * (row * D + col), a0, a1, a2, a3);
          const uint4 qf = qfragc[kb * 32 + lane];
          mma16816(s[0], a0, a1, a2, a3, qf.x, qf.y);
          if (qlo) mma16816(s[0], a0, a1, a2, a3, qf.z, qf.w);  // fp16 queries have no remainder
        }
        const bool va = g < rows, vb = g + 8 < rows;
        s[0][0] = va ? s[0][0] * sl2 : -INFINITY;
        s[0][1] = va ? s[0][1] * sl2 : -INFINITY;
        s[0][2] = vb ? s[0][2] * sl2 : -INFINITY;
        s[0][3] = vb ? s[0][3] * sl2 : -INFINITY;
        uint32_t pb[1][2];
        softmax_update<D, 1>(acc, s, pb);
        pv_fp16<D, 1>(acc, st + kCRows * D * 2, lane, pb);
      }
      // release the stage: order this warp's reads before later bulk writes into it
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[sidx]);
    }
    if (!ok && lane == 0) {
      atomicExch(&abort_s, 1);
      atomicExch(P.error, (int)RDKV_ERR_TIMEOUT);
    }
    if (o_mode != 16) rescale_o<D>(acc, o_mode, 16);
    // zero-point sums of packed V: channel 16 cm + g (+8) is in group cm / 2, held by lane (cm / 2, q)
#pragma unroll
    for (int cm = 0; cm < D / 16; ++cm) {
      const float z0 = __shfl_sync(0xffffffffu, acc.z[0], (cm / 2) * 4 + q);
      const float z1 = __shfl_sync(0xffffffffu, acc.z[1], (cm / 2) * 4 + q);
      acc.o[cm][0] += z0;
      acc.o[cm][1] += z1;
      acc.o[cm][2] += z0;
      acc.o[cm][3] += z1;
    }
    // the warp's row sums, kept in registers until the rings are free (block barrier below)
    float l0 = acc.l[0], l1 = acc.l[1];
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    acc.l[0] = l0;
    acc.l[1] = l1;
  }
  __syncthreads();  // every ring drained: the ring area now holds the consumer warps' results
  if (warp < kConsumers) {
    const int g = lane >> 2, q = lane & 3;
    float* rw = red + (int64_t)warp * 8 * (D + 2);
#pragma unroll
    for (int cm = 0; cm < D / 16; ++cm) {
      rw[(2 * q) * (D + 2) + 16 * cm + g] = acc.o[cm][0];
      rw[(2 * q + 1) * (D + 2) + 16 * cm + g] = acc.o[cm][1];
      rw[(2 * q) * (D + 2) + 16 * cm + g + 8] = acc.o[cm][2];
      rw[(2 * q + 1) * (D + 2) + 16 * cm + g + 8] = acc.o[cm][3];
    }
    if (g == 0) {
      rw[(2 * q) * (D + 2) + D] = acc.m[0];
      rw[(2 * q + 1) * (D + 2) + D] = acc.m[1];
      rw[(2 * q) * (D + 2) + D + 1] = acc.l[0];
      rw[(2 * q + 1) * (D + 2) + D + 1] = acc.l[1];
    }
  }
  __syncthreads();
  // combine the consumer warps; write this block's partial result (m, l, unnormalised o) for the G
  // heads; one block's partial takes pstride floats
  const int pstride = partial_stride(G, D);
  float* part = P.partial + (int64_t)first_block * pstride;
  float* mine = part + (int64_t)split * pstride;
  // per head: the block's running max M over the warps and each warp's weight 2^(m_w - M) (0 for
  // a warp that saw no token), computed once; then each element sums the warps' results with those
  // weights (the m (c = D) entry holds M)
  __shared__ float wgt_s[8][kConsumers + 1];
  if (tid < G * kConsumers) {
    const int h = tid / kConsumers, w = tid % kConsumers;
    float M = -INFINITY;
#pragma unroll
    for (int u = 0; u < kConsumers; ++u) M = fmaxf(M, red[((int64_t)u * 8 + h) * (D + 2) + D]);
    const float mw = red[((int64_t)w * 8 + h) * (D + 2) + D];
    wgt_s[h][w] = M == -INFINITY ? 0.f : ex2(mw - M);
    if (w == 0) wgt_s[h][kConsumers] = M;
  }
  __syncthreads();
  for (int i = tid; i < G * (D + 2); i += blockDim.x) {
    const int h = i / (D + 2), c = i % (D + 2);
    float val = wgt_s[h][kConsumers];
    if (c != D) {
      val = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) val = fmaf(wgt_s[h][w], red[((int64_t)w * 8 + h) * (D + 2) + c], val);
    }
    mine[i] = val;
  }
  // the last block of this head merges every split: out = sum 2^(M_s - M) O_s / sum 2^(M_s - M) L_s.
  // One acquire-release ticket by thread 0 after the block barrier: the release covers every
  // thread's partial writes (ordered before it by the barrier), the acquire makes the other
  // blocks' released partials visible to the merging block (ordered after it by the next barrier).
  __syncthreads();
  if (tid == 0) is_last = ticket_acq_rel(&P.tickets[head]) == n_split - 1;
  __syncthreads();
  if (!is_last) return;
  if (tid == 0) P.tickets[head] = 0;  // every block of this head has counted: ready for the next call
  if (fused) {
    // every block of this head has read zone C: store the new row of this head; the last head to
    // get here advances the length (every block of every head has read it by then)
    const int len_c = min(*PP.len_dev, PP.cap_c);
    if (len_c < P.cap_c) {
      const int64_t dst = zone_c_offset(PP.zc_pages, PP.zc_page_stride, PP.cap_c, hc, len_c, D);
      for (int i = tid; i < D; i += blockDim.x) {
        const_cast<uint16_t*>(PP.zone_c_k)[dst + i] = newrow[i];
        const_cast<uint16_t*>(PP.zone_c_v)[dst + i] = newrow[D + i];
      }
    } else if (tid == 0) {
      atomicExch(P.error, (int)RDKV_ERR_CAPACITY);
    }
    if (tid == 0 && atomicAdd(P.gticket, 1) == P.n_heads - 1) {
      *P.gticket = 0;
      if (len_c < P.cap_c) *P.len_dev = len_c + 1;
    }
  }
  // Merge: out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s per query head and channel.  Each
  // thread takes two adjacent channels of one head and loads, for every split, that head's (m, l) and
  // the two o values (8-byte loads from L2; the acquire above made them visible), all in flight
  // together (kMergeBatch splits at a time), then folds each batch into its running (M, L, O).
  constexpr int kMergeBatch = 24;
  for (int i = tid; i < G * D / 2; i += blockDim.x) {
    const int h = (2 * i) / D, c = (2 * i) % D;
    const float* ph = part + h * (D + 2);
    float M = -INFINITY, L = 0.f, O0 = 0.f, O1 = 0.f;
    for (int s0 = 0; s0 < n_split; s0 += kMergeBatch) {
      float2 ml[kMergeBatch], ov[kMergeBatch];
#pragma unroll
      for (int k = 0; k < kMergeBatch; ++k) {
        const bool in = s0 + k < n_split;
        const float* ps = ph + (int64_t)(s0 + k) * pstride;
        ml[k] = in ? __ldcg(reinterpret_cast<const float2*>(ps + D)) : make_float2(-INFINITY, 0.f);
        ov[k] = in ? __ldcg(reinterpret_cast<const float2*>(ps + c)) : make_float2(0.f, 0.f);
      }
      float Mn = M;
#pragma unroll
      for (int k = 0; k < kMergeBatch; ++k) Mn = fmaxf(Mn, ml[k].x);
      if (Mn == -INFINITY) continue;  // no token seen so far
      const float so = M == -INFINITY ? 0.f : ex2(M - Mn);
      float l1 = 0.f, o0 = 0.f, o1 = 0.f;
#pragma unroll
      for (int k = 0; k < kMergeBatch; ++k) {
        const float w = ex2(ml[k].x - Mn);  // 0 for a split without tokens (m = -inf)
        l1 = fmaf(w, ml[k].y, l1);
        o0 = fmaf(w, ov[k].x, o0);
        o1 = fmaf(w, ov[k].y, o1);
      }
      L = fmaf(L, so, l1);
      O0 = fmaf(O0, so, o0);
      O1 = fmaf(O1, so, o1);
      M = Mn;
    }
    float* op = P.out + ((int64_t)b * P.h_q + j * G + h) * D + c;  // (the caller's out needs 4-byte alignment only)
    op[0] = L > 0.f ? O0 / L : 0.f;
    op[1] = L > 0.f ? O1 / L : 0.f;
    // ln of the denominator: the running sums are of 2^(s log2(e) / sqrt(D) - M)
    if (P.lse != nullptr && c == 0)
      P.lse[(int64_t)b * P.h_q + j * G + h] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
  }
}

constexpr int64_t kDecodeSmemLimit = 227 * 1024 - 1024;  // per-block limit less room for static shared memory
constexpr int64_t kDecodeSmemLimitNarrow = 112 * 1024;    // two blocks per SM (228 KB) with their static parts

struct DecodeGeom {
  int nc;       // consumer warps of a block (kConsumersWide, one block per SM, or kConsumersNarrow, two)
  int64_t max_item;
  int ctas;     // nominal number of blocks dealt to heads
  int splits;   // grid size: ctas + one spare block per head
  int ring_bytes;
  int ring_warps;  // warps with a ring (all, or fewer with larger rings when tiles are large)
  size_t smem;
  size_t partial_bytes;
  size_t ticket_off;   // tickets then the status word
  int n_heads;         // heads with their own ticket and merge: batch * h_kv, or n * h_kv for a ragged batch
};

// Geometry of a launch over the caches parts[0 .. n): one, segments and the live cache of the same
// sequences, or (ragged) the independent sequences of a ragged batch.
static DecodeGeom decode_geom(const rdkv_cache* const* parts, int n, bool ragged = false) {
  DecodeGeom g;
  const rdkv_shape& s = parts[0]->shape;
  const int D = s.head_dim, G = s.h_q / s.h_kv;
  const int n_heads = s.batch * s.h_kv;
  const int sms = num_sms();
  // (head, cache) units of the launch: many of them take two narrower blocks per SM
  const int nc = (int64_t)n_heads * n >= kManyUnits ? kConsumersNarrow : kConsumersWide;
  const int blocks_per_sm = nc == kConsumersWide ? 1 : 2;
  const int64_t smem_limit = nc == kConsumersWide ? kDecodeSmemLimit : kDecodeSmemLimitNarrow;
  const int64_t fixed = decode_fixed_smem(D, nc);
  g.nc = nc;
  int64_t max_item = 2 * kCRows * D * 2, items = 0;
  for (int p = 0; p < n; ++p) {
    max_item = std::max<int64_t>(max_item, align_up(parts[p]->sizes.max_stage_bytes, 128));
    items += ceil_div64(parts[p]->sizes.index_slots, kTile) + (int64_t)n_heads * ceil_div(parts[p]->cap_c, kCRows);
  }
  g.max_item = max_item;
  // the consumer warps with a ring share what is left equally: all of them, or half (a quarter)
  // with twice (four times) the ring when the largest staged tile needs it
  int ring_warps = nc;
  int64_t ring = ((smem_limit - fixed) / ring_warps) / 128 * 128;
  while (ring < max_item && ring_warps > std::max(1, nc / 4)) {
    ring_warps /= 2;
    ring = ((smem_limit - fixed) / ring_warps) / 128 * 128;
  }
  if ((int64_t)ring_warps * ring < decode_reduce_bytes(D, nc)) ring = 0;  // the warps' results reuse the rings
  g.ring_bytes = (int)ring;
  g.ring_warps = ring_warps;
  g.smem = (size_t)(fixed + (int64_t)ring_warps * ring);
  // blocks dealt to heads in proportion to their work: a nominal count that fills every SM once,
  // fewer when there is little work (at least one item per consumer warp on average).  Every SM
  // takes work: leaving one per head free for the merges measured slower (the next call's blocks
  // wait for this call to finish before they read the query anyway).
  g.ctas = (int)std::max<int64_t>(1, std::min<int64_t>((int64_t)blocks_per_sm * sms, ceil_div64(items, nc)));
  g.splits = g.ctas + n_heads * n;  // grid size: room for at least one block per (cache, head)
  g.partial_bytes = (size_t)align_up((int64_t)g.splits * partial_stride(G, D) * 4, 256);
  g.ticket_off = g.partial_bytes;
  g.n_heads = ragged ? n * s.h_kv : n_heads;
  return g;
}
static DecodeGeom decode_geom(const rdkv_cache* c) { return decode_geom(&c, 1); }

// ws: partials, then per-head tickets, the status word and the fused step's head counter
static size_t decode_ws_bytes(const DecodeGeom& g) { return g.ticket_off + (size_t)decode_ticket_bytes(g.n_heads); }

rdkv_status check_cache_public(const rdkv_cache* c);

// Kernel arguments of one decode call over parts[0 .. n); ws holds the partials, then the tickets and
// the status word.  The blocks are dealt on the host when every cache's plan costs reached it
// (rdkv_plan_sizes), else (one cache only) by the kernel.
static DecodeParams decode_params(const rdkv_cache* const* parts, int n, const DecodeGeom& geo, const void* q,
                                  float* out, void* ws, const void* k_new = nullptr, const void* v_new = nullptr,
                                  float* lse = nullptr, bool ragged = false) {
  const rdkv_cache* cache = parts[0];
  const rdkv_shape& s = cache->shape;
  const int n_heads = geo.n_heads;                    // heads with their own ticket and merge
  const int cache_heads = s.batch * s.h_kv;           // heads of one cache
  const PlanLayout L = plan_layout(s.batch, s.h_kv, s.head_dim);
  DecodeParams P;
  P.plan = cache->plan;
  P.zone_a = cache->zone_a;
  P.zone_b = cache->zone_b;
  P.zone_c_k = cache->zone_c_k;
  P.zone_c_v = cache->zone_c_v;
  P.q = q;
  P.partial = static_cast<float*>(ws);
  P.tickets = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + geo.ticket_off);
  P.error = P.tickets + n_heads;
  P.gticket = P.tickets + n_heads + 1;
  P.out = out;
  P.lse = lse;
  P.len_dev = cache->len_dev;
  P.k_new = k_new;
  P.v_new = v_new;
  P.heads = reinterpret_cast<const rdkv_head_plan*>(static_cast<const char*>(cache->plan) + L.heads_off);
  P.slots = reinterpret_cast<const int16_t*>(static_cast<const char*>(cache->plan) + L.slots_off);
  P.slot_stride = L.slot_stride;
  P.n_heads = n_heads;
  P.dtype = s.dtype;
  P.h_q = s.h_q;
  P.h_kv = s.h_kv;
  P.cap_c = cache->cap_c;
  P.ring_bytes = geo.ring_bytes;
  P.ring_warps = geo.ring_warps;
  P.ctas = geo.ctas;
  P.wait_cycles = kWaitCycles;
  P.arm_only = 0;
  P.ragged = ragged ? 1 : 0;
  for (int p = 0; p < kMaxParts; ++p) {
    const rdkv_cache* c = parts[p < n ? p : 0];
    DecodePart& d = P.parts[p];
    d.zone_a = c->zone_a;
    d.zone_b = c->zone_b;
    d.zone_c_k = c->zone_c_k;
    d.zone_c_v = c->zone_c_v;
    d.len_dev = c->len_dev;
    d.heads = reinterpret_cast<const rdkv_head_plan*>(static_cast<const char*>(c->plan) + L.heads_off);
    d.slots = reinterpret_cast<const int16_t*>(static_cast<const char*>(c->plan) + L.slots_off);
    d.zc_pages = c->zone_c_pages;
    d.zc_page_stride = c->zone_c_page_stride;
    d.cap_c = c->cap_c;
    d.a_pages = c->zone_a_pages;
    d.b_pages = c->zone_b_pages;
  }
  // Deal the blocks to the heads here when the plans' cost estimates reached the host: the kernel
  // then knows its head at once instead of reading every head record first.  At least one block per
  // head and cache; every other block of the nominal count goes, one at a time, to the (head, cache)
  // whose cost per block is then the largest, so the slowest block is as fast as it can be and every
  // SM takes work.  A ragged batch: head h is head h % h_kv of cache h / h_kv alone.
  P.dealt = 0;
  bool known = n_heads <= RDKV_COST_HEADS && geo.splits <= kMaxDealtBlocks;
  for (int p = 0; known && p < n; ++p) {
    known = parts[p]->sizes.n_heads == cache_heads;
    for (int h = 0; known && h < cache_heads; ++h) known = parts[p]->sizes.head_cost[h] > 0;
  }
  if (known) {
    auto cost = [&](int p, int h) {
      return parts[p]->sizes.head_cost[h] + (int64_t)ceil_div(parts[p]->cap_c, kCRows) * kZoneCBlockCost;
    };
    auto part_of = [&](int h, int p) { return ragged ? h / s.h_kv : p; };       // the cache of (head, part p)
    auto head_in = [&](int h) { return ragged ? h % s.h_kv : h; };             // the head within that cache
    const int parts_per_head = ragged ? 1 : n;
    const int n_units = n_heads * parts_per_head;  // unit u: head u / parts_per_head, part u % parts_per_head
    int64_t ucost[RDKV_COST_HEADS * kMaxParts];
    int ublocks[RDKV_COST_HEADS * kMaxParts];
    int64_t total = 0;
    for (int u = 0; u < n_units; ++u) {
      ucost[u] = std::max<int64_t>(1, cost(part_of(u / parts_per_head, u % parts_per_head), head_in(u / parts_per_head)));
      total += ucost[u];
    }
    // in proportion, rounded down (at least one), then the rest one at a time
    int dealt = 0;
    for (int u = 0; u < n_units; ++u) {
      ublocks[u] = std::max(1, (int)(ucost[u] * geo.ctas / total));
      dealt += ublocks[u];
    }
    for (int extra = geo.ctas - dealt; extra > 0; --extra) {
      int best = 0;  // the unit with the largest cost per block (cross-multiplied: exact)
      for (int u = 1; u < n_units; ++u)
        if (ucost[u] * ublocks[best] > ucost[best] * ublocks[u]) best = u;
      ++ublocks[best];
    }
    int start = 0;
    for (int h = 0; h < n_heads; ++h) {
      P.head_first[h] = (int16_t)start;
      for (int pi = 0; pi < parts_per_head; ++pi) {
        const int p = part_of(h, pi);
        const int c = ublocks[h * parts_per_head + pi];
        for (int k = 0; k < c; ++k) {
          P.block_head[start + k] = (uint8_t)h;
          P.block_part[start + k] = (uint8_t)p;
          P.block_split[start + k] = (uint8_t)k;
          P.block_nsplit[start + k] = (uint8_t)c;
        }
        start += c;
      }
    }
    P.head_first[n_heads] = (int16_t)start;
    for (int k = start; k < geo.splits; ++k) {
      P.block_head[k] = kNoHead;
      P.block_part[k] = P.block_split[k] = 0;
      P.block_nsplit[k] = 1;
    }
    P.dealt = 1;
  }
  return P;
}
static DecodeParams decode_params(const rdkv_cache* cache, const DecodeGeom& geo, const void* q, float* out, void* ws,
                                  const void* k_new = nullptr, const void* v_new = nullptr, float* lse = nullptr) {
  return decode_params(&cache, 1, geo, q, out, ws, k_new, v_new, lse);
}

// pdl: programmatic dependent launch; the kernel's static setup (plan, zone A) may then overlap
// the tail of the kernel launched before it on the stream, and it waits for that kernel before
// it reads the query, the new token or zone C.
static rdkv_status launch_decode(const DecodeParams& P, const DecodeGeom& geo, const rdkv_shape& s, cudaStream_t cs,
                                 bool pdl) {
  // the dynamic shared-memory limit is raised once per device and kernel (not while a graph is
  // captured); threads that get here together may both raise it, to the same value
  static std::atomic<size_t> smem_set[8][64];
  int dev = 0;
  RDKV_TRY_CUDA(cudaGetDevice(&dev), "device");
  // at most 4 query heads per KV head: the hi and lo parts of the K operand share one MMA per block
  const bool pk = s.h_q / s.h_kv <= 4;
  const bool wide = geo.nc == kConsumersWide;
  const int ki = (s.head_dim == 128 ? 2 : 0) + (pk ? 1 : 0) + (wide ? 4 : 0);
  void (*const fn)(DecodeParams) = ki == 7 ? decode_kernel<128, true, kConsumersWide>
                                 : ki == 6 ? decode_kernel<128, false, kConsumersWide>
                                 : ki == 5 ? decode_kernel<64, true, kConsumersWide>
                                 : ki == 4 ? decode_kernel<64, false, kConsumersWide>
                                 : ki == 3 ? decode_kernel<128, true, kConsumersNarrow>
                                 : ki == 2 ? decode_kernel<128, false, kConsumersNarrow>
                                 : ki == 1 ? decode_kernel<64, true, kConsumersNarrow>
                                           : decode_kernel<64, false, kConsumersNarrow>;
  const int64_t limit = wide ? kDecodeSmemLimit : kDecodeSmemLimitNarrow;
  if (dev < 64 && geo.smem > smem_set[ki][dev].load(std::memory_order_acquire)) {
    RDKV_TRY_CUDA(cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)limit),
                  "decode smem");
    smem_set[ki][dev].store((size_t)limit, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(geo.splits);
  cfg.blockDim = dim3((geo.nc + 1) * 32);
  cfg.dynamicSmemBytes = geo.smem;
  cfg.stream = cs;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  RDKV_TRY_CUDA(cudaLaunchKernelEx(&cfg, fn, P), "decode launch");
  RDKV_CHECK_LAUNCH("decode");
  return RDKV_OK;
}

}  // namespace rdkv

using namespace rdkv;

extern "C" size_t rdkv_decode_workspace_bytes(const rdkv_cache* cache) {
  if (check_cache_public(cache) != RDKV_OK) return 0;
  return decode_ws_bytes(decode_geom(cache));
}

// selftest_wait > 0: the timeout self-test (stages armed for bytes that no copy delivers, each wait
// limited to that many cycles)
static rdkv_status decode_attn_impl(const rdkv_cache* cache, const void* q, float* out, float* lse, void* ws,
                                    size_t ws_bytes, void* stream, long long selftest_wait = 0) {
  rdkv_status st = check_cache_public(cache);
  if (st != RDKV_OK) return st;
  RDKV_REQUIRE(q && out, RDKV_ERR_INVALID_ARG, "NULL pointer argument");
  const rdkv_shape& s = cache->shape;
  const DecodeGeom geo = decode_geom(cache);
  const size_t need = decode_ws_bytes(geo);
  RDKV_REQUIRE(ws && ws_bytes >= need, RDKV_ERR_WORKSPACE, "decode workspace too small (%zu < %zu)", ws_bytes, need);
  RDKV_REQUIRE(geo.ring_bytes >= geo.max_item, RDKV_ERR_UNSUPPORTED, "tiles too large for the decode ring (%lld B)",
               (long long)geo.max_item);
  // the tickets are zero here: the workspace starts zero-filled and every call leaves them at zero
  DecodeParams P = decode_params(cache, geo, q, out, ws, nullptr, nullptr, lse);
  if (selftest_wait > 0) {
    P.arm_only = 1;
    P.wait_cycles = std::min(kWaitCycles, std::max(kMinWaitCycles, selftest_wait));
  }
  return launch_decode(P, geo, s, (cudaStream_t)stream, selftest_wait == 0);
}

static rdkv_status decode_step_impl(rdkv_cache* cache, const void* q, const void* k_new, const void* v_new, float* out,
                                    float* lse, void* ws, size_t ws_bytes, void* stream) {
  rdkv_status st = check_cache_public(cache);
  if (st != RDKV_OK) return st;
  RDKV_REQUIRE(q && out && k_new && v_new, RDKV_ERR_INVALID_ARG, "NULL pointer argument");
  RDKV_REQUIRE(cache->len_c < cache->cap_c, RDKV_ERR_CAPACITY, "zone C is full (%d rows)", cache->cap_c);
  const rdkv_shape& s = cache->shape;
  const DecodeGeom geo = decode_geom(cache);
  const size_t need = decode_ws_bytes(geo);
  RDKV_REQUIRE(ws && ws_bytes >= need, RDKV_ERR_WORKSPACE, "decode workspace too small (%zu < %zu)", ws_bytes, need);
  RDKV_REQUIRE(geo.ring_bytes >= geo.max_item, RDKV_ERR_UNSUPPORTED, "tiles too large for the decode ring (%lld B)",
               (long long)geo.max_item);
  st = launch_decode(decode_params(cache, geo, q, out, ws, k_new, v_new, lse), geo, s, (cudaStream_t)stream, true);
  if (st == RDKV_OK) cache->len_c += 1;
  return st;
}

extern "C" rdkv_status rdkv_decode_attn(const rdkv_cache* cache, const void* q, float* out, void* ws, size_t ws_bytes,
                                        void* stream) {
  return decode_attn_impl(cache, q, out, nullptr, ws, ws_bytes, stream);
}

extern "C" rdkv_status rdkv_decode_attn_lse(const rdkv_cache* cache, const void* q, float* out, float* lse, void* ws,
                                            size_t ws_bytes, void* stream) {
  RDKV_REQUIRE(lse, RDKV_ERR_INVALID_ARG, "NULL lse");
  return decode_attn_impl(cache, q, out, lse, ws, ws_bytes, stream);
}

extern "C" rdkv_status rdkv_decode_timeout_selftest(const rdkv_cache* cache, const void* q, float* out, void* ws,
                                                    size_t ws_bytes, int64_t wait_cycles, void* stream) {
  RDKV_REQUIRE(wait_cycles > 0, RDKV_ERR_INVALID_ARG, "wait_cycles %lld must be positive", (long long)wait_cycles);
  return decode_attn_impl(cache, q, out, nullptr, ws, ws_bytes, stream, wait_cycles);
}

extern "C" rdkv_status rdkv_decode_step(rdkv_cache* cache, const void* q, const void* k_new, const void* v_new,
                                        float* out, void* ws, size_t ws_bytes, void* stream) {
  return decode_step_impl(cache, q, k_new, v_new, out, nullptr, ws, ws_bytes, stream);
}

extern "C" rdkv_status rdkv_decode_step_lse(rdkv_cache* cache, const void* q, const void* k_new, const void* v_new,
                                            float* out, float* lse, void* ws, size_t ws_bytes, void* stream) {
  RDKV_REQUIRE(lse, RDKV_ERR_INVALID_ARG, "NULL lse");
  return decode_step_impl(cache, q, k_new, v_new, out, lse, ws, ws_bytes, stream);
}

static rdkv_status decode_status_at(const void* ws, size_t status_off, void* stream) {
  int32_t v = 0;
  RDKV_TRY_CUDA(cudaMemcpyAsync(&v, static_cast<const char*>(ws) + status_off, 4, cudaMemcpyDeviceToHost,
                                (cudaStream_t)stream),
                "status read");
  RDKV_TRY_CUDA(cudaStreamSynchronize((cudaStream_t)stream), "status sync");
  if (v != RDKV_OK) {
    if (v == RDKV_ERR_TIMEOUT) set_error("decode: a bounded wait for a tile copy ran out");
    else if (v == RDKV_ERR_CAPACITY) set_error("decode step: zone C was full, the new token was not stored");
    else set_error("decode reported status %d", v);
    RDKV_TRY_CUDA(cudaMemsetAsync(static_cast<char*>(const_cast<void*>(ws)) + status_off, 0, 4, (cudaStream_t)stream),
                  "status clear");
    RDKV_TRY_CUDA(cudaStreamSynchronize((cudaStream_t)stream), "status clear sync");
  }
  return (rdkv_status)v;
}

extern "C" rdkv_status rdkv_decode_status(const rdkv_cache* cache, const void* ws, void* stream) {
  rdkv_status st = check_cache_public(cache);
  if (st != RDKV_OK) return st;
  RDKV_REQUIRE(ws, RDKV_ERR_INVALID_ARG, "NULL workspace");
  const DecodeGeom geo = decode_geom(cache);
  return decode_status_at(ws, geo.ticket_off + 4 * (size_t)geo.n_heads, stream);
}

// ---------------------------------------------------------------- one launch over several caches
static rdkv_status check_parts(const rdkv_cache* const* parts, int32_t n_parts) {
  RDKV_REQUIRE(parts && n_parts >= 1 && n_parts <= kMaxParts, RDKV_ERR_INVALID_ARG, "n_parts %d outside [1, %d]",
               n_parts, kMaxParts);
  for (int p = 0; p < n_parts; ++p) {
    rdkv_status st = check_cache_public(parts[p]);
    if (st != RDKV_OK) return st;
    const rdkv_shape &a = parts[0]->shape, &b = parts[p]->shape;
    RDKV_REQUIRE(a.batch == b.batch && a.h_q == b.h_q && a.h_kv == b.h_kv && a.head_dim == b.head_dim &&
                     a.dtype == b.dtype,
                 RDKV_ERR_INVALID_ARG, "cache %d does not share the shape of cache 0 (batch, heads, D, dtype)", p);
  }
  return RDKV_OK;
}

extern "C" size_t rdkv_decode_multi_workspace_bytes(const rdkv_cache* const* parts, int32_t n_parts) {
  if (check_parts(parts, n_parts) != RDKV_OK) return 0;
  return decode_ws_bytes(decode_geom(parts, n_parts));
}

extern "C" rdkv_status rdkv_decode_attn_multi(const rdkv_cache* const* parts, int32_t n_parts, const void* q,
                                              float* out, float* lse, void* ws, size_t ws_bytes, void* stream) {
  rdkv_status st = check_parts(parts, n_parts);
  if (st != RDKV_OK) return st;
  RDKV_REQUIRE(q && out, RDKV_ERR_INVALID_ARG, "NULL pointer argument");
  const rdkv_shape& s = parts[0]->shape;
  const DecodeGeom geo = decode_geom(parts, n_parts);
  const size_t need = decode_ws_bytes(geo);
  RDKV_REQUIRE(ws && ws_bytes >= need, RDKV_ERR_WORKSPACE, "decode workspace too small (%zu < %zu)", ws_bytes, need);
  RDKV_REQUIRE(geo.ring_bytes >= geo.max_item, RDKV_ERR_UNSUPPORTED, "tiles too large for the decode ring (%lld B)",
               (long long)geo.max_item);
  const DecodeParams P = decode_params(parts, n_parts, geo, q, out, ws, nullptr, nullptr, lse);
  RDKV_REQUIRE(P.dealt || n_parts == 1, RDKV_ERR_UNSUPPORTED,
               "several caches need their plan costs on the host (rdkv_plan_sizes), at most %d heads and %d blocks",
               RDKV_COST_HEADS, kMaxDealtBlocks);
  return launch_decode(P, geo, s, (cudaStream_t)stream, true);
}

extern "C" rdkv_status rdkv_decode_multi_status(const rdkv_cache* const* parts, int32_t n_parts, const void* ws,
                                                void* stream) {
  rdkv_status st = check_parts(parts, n_parts);
  if (st != RDKV_OK) return st;
  RDKV_REQUIRE(ws, RDKV_ERR_INVALID_ARG, "NULL workspace");
  const DecodeGeom geo = decode_geom(parts, n_parts);
  return decode_status_at(ws, geo.ticket_off + 4 * (size_t)geo.n_heads, stream);
}

// ---------------------------------------------------------------- one launch over a ragged batch
static rdkv_status check_ragged(const rdkv_cache* const* seqs, int32_t n_seq) {
  RDKV_REQUIRE(seqs && n_seq >= 1 && n_seq <= kMaxParts, RDKV_ERR_INVALID_ARG, "n_seq %d outside [1, %d]", n_seq,
               kMaxParts);
  for (int p = 0; p < n_seq; ++p) {
    rdkv_status st = check_cache_public(seqs[p]);
    if (st != RDKV_OK) return st;
    const rdkv_shape &a = seqs[0]->shape, &b = seqs[p]->shape;
    RDKV_REQUIRE(b.batch == 1, RDKV_ERR_INVALID_ARG, "sequence %d: a ragged batch takes caches of batch 1", p);
    RDKV_REQUIRE(a.h_q == b.h_q && a.h_kv == b.h_kv && a.head_dim == b.head_dim && a.dtype == b.dtype,
                 RDKV_ERR_INVALID_ARG, "sequence %d does not share the heads, D and dtype of sequence 0", p);
  }
  RDKV_REQUIRE((int64_t)n_seq * seqs[0]->shape.h_kv <= RDKV_COST_HEADS, RDKV_ERR_UNSUPPORTED,
               "a ragged batch holds at most %d (sequence, KV head) pairs", RDKV_COST_HEADS);
  return RDKV_OK;
}

extern "C" size_t rdkv_decode_ragged_workspace_bytes(const rdkv_cache* const* seqs, int32_t n_seq) {
  if (check_ragged(seqs, n_seq) != RDKV_OK) return 0;
  return decode_ws_bytes(decode_geom(seqs, n_seq, true));
}

extern "C" rdkv_status rdkv_decode_ragged(const rdkv_cache* const* seqs, int32_t n_seq, const void* q, float* out,
                                          float* lse, void* ws, size_t ws_bytes, void* stream) {
  rdkv_status st = check_ragged(seqs, n_seq);
  if (st != RDKV_OK) return st;
  RDKV_REQUIRE(q && out, RDKV_ERR_INVALID_ARG, "NULL pointer argument");
  const DecodeGeom geo = decode_geom(seqs, n_seq, true);
  const size_t need = decode_ws_bytes(geo);
  RDKV_REQUIRE(ws && ws_bytes >= need, RDKV_ERR_WORKSPACE, "decode workspace too small (%zu < %zu)", ws_bytes, need);
  RDKV_REQUIRE(geo.ring_bytes >= geo.max_item, RDKV_ERR_UNSUPPORTED, "tiles too large for the decode ring (%lld B)",
               (long long)geo.max_item);
  const DecodeParams P = decode_params(seqs, n_seq, geo, q, out, ws, nullptr, nullptr, lse, true);
  RDKV_REQUIRE(P.dealt, RDKV_ERR_UNSUPPORTED,
               "a ragged batch needs every cache's plan costs on the host (rdkv_plan_sizes) and at most %d blocks",
               kMaxDealtBlocks);
  return launch_decode(P, geo, seqs[0]->shape, (cudaStream_t)stream, true);
}

extern "C" rdkv_status rdkv_decode_ragged_status(const rdkv_cache* const* seqs, int32_t n_seq, const void* ws,
                                                 void* stream) {
  rdkv_status st = check_ragged(seqs, n_seq);
  if (st != RDKV_OK) return st;
  RDKV_REQUIRE(ws, RDKV_ERR_INVALID_ARG, "NULL workspace");
  const DecodeGeom geo = decode_geom(seqs, n_seq, true);
  return decode_status_at(ws, geo.ticket_off + 4 * (size_t)geo.n_heads, stream);
}

// ---------------------------------------------------------------- decode without a caller workspace
// Scratch of rdkv_decode_attn_noalloc: split partials, tickets and the status
// word.  Every GPU that loads this library holds it until the process exits.
namespace rdkv {
constexpr size_t kNoAllocScratchBytes = 4u << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array for the current device, looked up once per
// device (in the CUDA runtime's primary context of that device, the one every
// entry point of this library runs in).  The array's name is only a host-side
// stand-in in host code.  Threads making their first call at the same time may
// each look the address up; they store the same value into an atomic slot, so
// the cache itself never races.
static rdkv_status noalloc_scratch(void** out) {
  static std::atomic<void*> addr[64];
  int dev = 0;
  RDKV_TRY_CUDA(cudaGetDevice(&dev), "device");
  RDKV_REQUIRE(dev >= 0 && dev < 64, RDKV_ERR_UNSUPPORTED, "device index %d", dev);
  void* p = addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    RDKV_TRY_CUDA(cudaGetSymbolAddress(&p, g_noalloc_scratch), "scratch address");
    addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return RDKV_OK;
}
}  // namespace rdkv

extern "C" rdkv_status rdkv_decode_attn_noalloc(const rdkv_cache* cache, const void* q, float* out, void* stream) {
  rdkv_status st = check_cache_public(cache);
  if (st != RDKV_OK) return st;
  RDKV_REQUIRE(q && out, RDKV_ERR_INVALID_ARG, "NULL pointer argument");
  const rdkv_shape& s = cache->shape;
  const int n_heads = s.batch * s.h_kv;
  const DecodeGeom geo = decode_geom(cache);
  const size_t need = decode_ws_bytes(geo);
  RDKV_REQUIRE(need <= kNoAllocScratchBytes, RDKV_ERR_WORKSPACE,
               "this cache needs %zu bytes of decode scratch; the built-in scratch holds %zu "
               "(use rdkv_decode_attn with a workspace)",
               need, kNoAllocScratchBytes);
  RDKV_REQUIRE(geo.ring_bytes >= geo.max_item, RDKV_ERR_UNSUPPORTED, "tiles too large for the decode ring (%lld B)",
               (long long)geo.max_item);
  void* ws = nullptr;
  st = noalloc_scratch(&ws);
  if (st != RDKV_OK) return st;
  const DecodeParams P = decode_params(cache, geo, q, out, ws);
  // the previous call's tickets and status word are still in the scratch: clear them
  RDKV_TRY_CUDA(cudaMemsetAsync(P.tickets, 0, ((size_t)n_heads + 2) * 4, (cudaStream_t)stream), "decode ticket reset");
  return launch_decode(P, geo, s, (cudaStream_t)stream, false);
}
