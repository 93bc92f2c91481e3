// Decode attention over the TriZone cache of RDKV
// (gist.science/ko/paper/2605.08317, section 2.3): the logits and the output
// are computed with the dequantisation fused into the two products, reading
// zones A (packed K rows and 2/4/8-bit V rows), B (fp16 V rows of 16-bit
// tokens) and C (fp16 K and V rows of the window and of decoded tokens) in one
// pass.
//
// Work: one block of 16 warps per SM, dealt to the (sequence, KV head) pairs
// in proportion to their estimated cost (on the host when the plan's costs are
// there, else by the kernel).  A head's work items are its zone-A tiles (32
// tokens, in class order) followed by zone-C blocks of 16 rows; split s of n
// takes items s, s + n, s + 2n, ... and its warps take them in order of need.
// Every warp streams its items through its own ring of shared memory, filled
// by bulk asynchronous copies that complete on per-slot mbarriers (all waits
// are bounded and report RDKV_ERR_TIMEOUT).  The last block of a head to
// finish (an atomic ticket) merges the splits' partial softmax states into
// the output (and, when asked, the log-sum-exp).  One launch may attend
// several caches sharing the query (segments moved out of zone C and the live
// cache): each block reads one cache, the blocks of a head over all caches
// share its merge.  Zone C may be paged (16-row pages through a table).
//
// Products: mma.sync m16n8k16 (fp16 in, fp32 accumulate), tokens on M:
//   S^T[16 tok x 8 heads]  += K^[16 tok x 16 slots] * Q^T[16 slots x 8 heads]
//   O^T[16 ch  x 8 heads]  += V^T[16 ch x 16 tok]   * P^T[16 tok x 8 heads]
// A 32-bit A-fragment register holds two consecutive elements along the
// contraction axis (two K slots of one token; two tokens of one V channel);
// the word rule of the layout puts both codes of such a pair in the two
// half-words of one 32-bit word, so one shift and one mask (one byte permute
// for 8-bit codes) place them as fp16 subnormals, code * 2^-24 exactly; the
// scales enter through the other operand.  The softmax runs in fp32 on the
// S^T accumulators (base-2 exponent); P^T is moved into B-fragment order by
// movmatrix.  The G query heads of a group share every loaded tile.
#include <atomic>

#include "common.cuh"

namespace rdkv {

constexpr int kDecWarps = 16;  // one block per SM
constexpr int kMaxInflight = 4;
constexpr int kPrologueItems = 2;     // copies a warp issues before the wait for the previous kernel
constexpr int kMaxDealtBlocks = 256;  // grids up to this size may be dealt to heads on the host
constexpr uint8_t kNoHead = 0xff;
constexpr int kMaxParts = 8;          // caches one launch may attend
constexpr int kCRows = 16;        // zone-C rows per work item
constexpr int kMaxKB = 16;        // k-blocks of a K row (D = 128: at most 13)
constexpr long long kWaitCycles = 4000000000ll;  // limit of every wait on a tile copy: ~2 s at GB300 clocks
constexpr long long kMinWaitCycles = 100000;     // shortest limit the timeout self-test may ask for

// One k-block of a head's K rows (16 slots inside one width segment).  The same for every lane:
// each lane adds its own constant offsets.
struct KBDesc {
  int32_t wbyte;    // byte offset in a tile of the block's first word: 128 * word (word-major layout)
  int32_t mbyte;    // byte offset of the block's first slot pair in the K metadata: 8 * pair
  int32_t nrem;     // slots of the segment from the block start (>= 1)
  int32_t slot0;    // first slot of the block (for the query fragments)
};

// Bytes of the fixed part of the decode kernel's shared memory (before the rings): k-block
// descriptors, query fragments (float4 per lane for fp32 queries, two fp16 pairs otherwise),
// zone-C query fragments, slot table, ring bookkeeping, the fused step's new row.
__host__ __device__ constexpr int64_t decode_fixed_smem(int D, bool qlo) {
  return ((256 + (int64_t)kMaxKB * 32 * (qlo ? 16 : 8) + (int64_t)(D / 16) * 32 * 16 +
           (int64_t)(D + kSlotPad) * 2 + kDecWarps * kMaxInflight * 20 + (int64_t)2 * D * 2) + 127) /
         128 * 128;
}
// Floats of one block's partial result (m, l, o for G heads), rounded up to a multiple of 4.
__host__ __device__ constexpr int partial_stride(int G, int D) { return (G * (D + 2) + 3) / 4 * 4; }

// The warps' partial results are combined in the ring area once every ring is drained.
__host__ __device__ constexpr int64_t decode_reduce_bytes(int D) { return (int64_t)kDecWarps * 8 * (D + 2) * 4; }

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
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait; false when the limit (clock64 cycles) ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, long long limit) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}
// L2 policy of the staged zone data: evicted first, so that the small data every call re-reads
// (plan records, slot tables, queries, the split partials) stays in L2 across the layers.  Zone C
// too: keeping its rows (a few hundred KB per layer) resident measured no better.
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
__device__ __forceinline__ uint32_t lds32(const unsigned char* base, uint32_t off) {
  return *reinterpret_cast<const uint32_t*>(base + off);
}
__device__ __forceinline__ uint2 lds64(const unsigned char* base, uint32_t off) {
  return *reinterpret_cast<const uint2*>(base + off);
}
__device__ __forceinline__ uint4 lds128(const unsigned char* base, uint32_t off) {
  return *reinterpret_cast<const uint4*>(base + off);
}
__device__ __forceinline__ uint32_t pick4(const uint4& v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }

// Byte-permute selector that moves bytes (0, 2) (odd = 0) or (1, 3) (odd = 1) of a word to the
// low bytes of its two half-words and zeroes the high bytes: the two 8-bit codes of a pair at
// bit 0 and bit 16, the same as a shift by 0 or 8 and a mask, in one instruction.
__device__ __forceinline__ uint32_t byte_pair_sel(int odd) { return odd ? 0x4341u : 0x4240u; }

// Two codes of a pair (already shifted to bit 0 and bit 16) -> exact fp16 codes
// -> scale * code + zero, one rounding.
__device__ __forceinline__ uint32_t dequant_pair(uint32_t w, int shift, uint32_t mask2, uint32_t scale2,
                                                 uint32_t zero2) {
  const uint32_t x = ((w >> shift) & mask2) | 0x64006400u;
  const __half2 c = __hsub2(*reinterpret_cast<const __half2*>(&x), __half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400)));
  const __half2 r = __hfma2(c, *reinterpret_cast<const __half2*>(&scale2), *reinterpret_cast<const __half2*>(&zero2));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// Two codes of a pair -> the same codes as exact fp16 values (no scale, no zero).
__device__ __forceinline__ uint32_t exact_codes(uint32_t w, int shift, uint32_t mask2) {
  const uint32_t x = ((w >> shift) & mask2) | 0x64006400u;
  const __half2 c = __hsub2(*reinterpret_cast<const __half2*>(&x), __half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400)));
  return *reinterpret_cast<const uint32_t*>(&c);
}

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

// K logits of one width segment of a zone-A tile, k-blocks [kb0, kb1).
// A quantised K element is zero_c + scale_c * code, so per head g
//   q_g . k^ = sum_c q_gc zero_c + sum_c code * (q_gc scale_c).
// The codes are exact in fp16 and form the A operand; q_gc * scale_c (exact in
// fp32) is split into an fp16 high part and an fp16 remainder, two B operands,
// so the products keep ~22 bits; the zero term is summed in fp32.  Raw 16-bit
// channels use the stored fp16 value against q (split the same way when q
// carries more than fp16 precision).
template <int W, bool QLO>
__device__ __forceinline__ void k_segment(const unsigned char* kw, const unsigned char* kmeta, int kb0, int kb1,
                                          const KBDesc* kbd, const float4* qv, int lane, float (&s)[2][4],
                                          float& bias) {
  const int g = lane >> 2, q = lane & 3;
  // word offsets (inside the block's first word) and shifts of this lane's two slot pairs
  constexpr uint32_t mask2 = W == 8 ? 0x00ff00ffu : W == 4 ? 0x000f000fu : 0x00030003u;
  const int o0 = W == 16 ? q : W == 8 ? (q >> 1) : 0;
  const int o1 = W == 16 ? q + 4 : W == 8 ? (q >> 1) + 2 : W == 4 ? 1 : 0;
  const int sh0 = W == 8 ? 8 * (q & 1) : W == 4 ? 4 * q : W == 2 ? 2 * q : 0;
  const int sh1 = W == 2 ? 2 * q + 8 : sh0;
  for (int kb = kb0; kb < kb1; ++kb) {
    const KBDesc d = kbd[kb];
    const float4 qq = qv[kb * 32 + lane];  // q_g at slots 2q, 2q+1, 2q+8, 2q+9 (0 for pads and missing slots)
    uint32_t bh0, bh1, bl0 = 0, bl1 = 0;
    if (W == 16) {
      if (QLO) {
        const uint4 t = split_hi_lo(qq.x, qq.y, qq.z, qq.w);
        bh0 = t.x; bh1 = t.y; bl0 = t.z; bl1 = t.w;
      } else {
        bh0 = pack_half2(qq.x, qq.y);
        bh1 = pack_half2(qq.z, qq.w);
      }
    } else {
      // a pair past the segment end reads the block's first (valid) pair: its q entries are 0
      const uint32_t p0 = d.mbyte + (2 * q < d.nrem ? 8 * q : 0), p1 = d.mbyte + (2 * q + 8 < d.nrem ? 8 * (q + 4) : 0);
      const uint2 m0 = lds64(kmeta, p0), m1 = lds64(kmeta, p1);
      const float2 s0 = __half22float2(*reinterpret_cast<const __half2*>(&m0.x));
      const float2 z0 = __half22float2(*reinterpret_cast<const __half2*>(&m0.y));
      const float2 s1 = __half22float2(*reinterpret_cast<const __half2*>(&m1.x));
      const float2 z1 = __half22float2(*reinterpret_cast<const __half2*>(&m1.y));
      bias = fmaf(qq.x, z0.x, fmaf(qq.y, z0.y, fmaf(qq.z, z1.x, fmaf(qq.w, z1.y, bias))));
      const uint4 t = split_hi_lo(qq.x * s0.x, qq.y * s0.y, qq.z * s1.x, qq.w * s1.y);
      bh0 = t.x; bh1 = t.y; bl0 = t.z; bl1 = t.w;
    }
    // tokens g, g+8, g+16, g+24 of the lane's two words
    const uint4 x0 = lds128(kw, (uint32_t)d.wbyte + 128u * o0 + 16u * g);
    const uint4 x1 = W == 2 ? x0 : lds128(kw, (uint32_t)d.wbyte + 128u * o1 + 16u * g);
#pragma unroll
    for (int tb = 0; tb < 2; ++tb) {
      uint32_t a0, a1, a2, a3;
      if (W == 16) {
        // raw fp16 words past the segment end may hold anything: zero them
        const bool v0 = 2 * q < d.nrem, v1 = 2 * q + 8 < d.nrem;
        a0 = v0 ? pick4(x0, 2 * tb) : 0u; a1 = v0 ? pick4(x0, 2 * tb + 1) : 0u;
        a2 = v1 ? pick4(x1, 2 * tb) : 0u; a3 = v1 ? pick4(x1, 2 * tb + 1) : 0u;
      } else {
        // codes past the segment end are small integers met by zero query entries
        a0 = exact_codes(pick4(x0, 2 * tb), sh0, mask2);
        a1 = exact_codes(pick4(x0, 2 * tb + 1), sh0, mask2);
        a2 = exact_codes(pick4(x1, 2 * tb), sh1, mask2);
        a3 = exact_codes(pick4(x1, 2 * tb + 1), sh1, mask2);
      }
      mma16816(s[tb], a0, a1, a2, a3, bh0, bh1);
      if (W != 16 || QLO) mma16816(s[tb], a0, a1, a2, a3, bl0, bl1);
    }
  }
}

// The same for fp16 queries (q exact in fp16).  hi = fp16(q * scale) by one
// half2 multiply (the exact product rounded once) and lo = q * scale - hi by
// one half2 FMA, which is exact because that remainder fits fp16.  The codes
// enter the tensor core as fp16 subnormals: the bit pattern of a code c placed
// at bit 0 of a half-word is the value c * 2^-24 exactly, so one shift and one
// mask make the A operand and the products land at 2^-24: the hi products in
// shi, the lo products in slo (two accumulators, two independent chains).  Raw
// 16-bit channels use the stored fp16 value against q, at scale 1, into shi.
// The zero-point term sum_c q_c zero_c runs as an MMA whose A rows g + 8 hold
// the zeros, so zacc[2], zacc[3] carry it for heads (2q, 2q+1).  A segment's
// k-blocks are consecutive: 64 W bytes of words and 64 bytes of metadata
// apart, and only the last one may be partial.
// PK (at most 4 heads): the hi and lo operands share one MMA.  B columns 0-3
// take hi of heads 0-3 and columns 4-7 lo of the same heads (lanes g >= 4 of
// the query fragments hold head g - 4), so one product gives both and shi
// holds hi in its columns (2q, 2q+1) for q < 2 and lo for q >= 2; slo is unused.
template <int W, bool PK>
__device__ __forceinline__ void k_segment_h(const unsigned char* kw, const unsigned char* kmeta, int kb0, int kb1,
                                            const KBDesc* kbd, const uint2* qh, int lane, float (&shi)[2][4],
                                            float (&slo)[2][4], float (&zacc)[4]) {
  if (kb0 >= kb1) return;
  const int g = lane >> 2, q = lane & 3;
  // PK: lo lanes take q * scale - fp16(q * scale), hi lanes fp16(q * scale); raw channels only hi
  const bool lo_lane = PK && g >= 4;
  const __half2 lo_sel = lo_lane ? __half2(__float2half(-1.f), __float2half(-1.f)) : __half2(__float2half(0.f), __float2half(0.f));
  constexpr uint32_t mask2 = W == 8 ? 0x00ff00ffu : W == 4 ? 0x000f000fu : 0x00030003u;
  const int sh0 = W == 8 ? 8 * (q & 1) : W == 4 ? 4 * q : W == 2 ? 2 * q : 0;
  const int sh1 = W == 2 ? 2 * q + 8 : sh0;
  const uint32_t bsel = byte_pair_sel(q & 1);  // 8-bit codes: bytes (0, 2) or (1, 3) of a word
  // this lane's offsets from a block's first word: words o0, o1 of its two slot pairs, tokens g ..
  const uint32_t c0 = 128u * (W == 16 ? q : W == 8 ? (q >> 1) : 0) + 16u * g;
  const uint32_t c1 = 128u * (W == 16 ? q + 4 : W == 8 ? (q >> 1) + 2 : W == 4 ? 1 : 0) + 16u * g;
  const KBDesc d0 = kbd[kb0];
  const int last_nrem = kbd[kb1 - 1].nrem;
  uint32_t wb = (uint32_t)d0.wbyte, mb = (uint32_t)d0.mbyte;
  const uint2* qp = qh + kb0 * 32 + lane;
#pragma unroll 1
  for (int kb = kb0; kb < kb1; ++kb, wb += 64u * W, mb += 64u, qp += 32) {
    const int nrem = kb == kb1 - 1 ? last_nrem : 16;
    const uint2 qq = *qp;  // q_g (fp16 pairs) at slots (2q, 2q+1), (2q+8, 2q+9); 0 for pads
    const bool v0 = 2 * q < nrem, v1 = 2 * q + 8 < nrem;
    // tokens g, g+8, g+16, g+24 of the lane's two words (one word for 2-bit codes)
    const uint4 y0 = lds128(kw, wb + c0);
    const uint4 y1 = W == 2 ? y0 : lds128(kw, wb + c1);
    uint32_t bh0 = lo_lane ? 0u : qq.x, bh1 = lo_lane ? 0u : qq.y, bl0 = 0, bl1 = 0;
    if (W != 16 && PK) {
      const uint2 m0 = lds64(kmeta, mb + (v0 ? 8u * q : 0u));
      const uint2 m1 = lds64(kmeta, mb + (v1 ? 8u * (q + 4) : 0u));
      const __half2 q0 = *reinterpret_cast<const __half2*>(&qq.x), q1 = *reinterpret_cast<const __half2*>(&qq.y);
      const __half2 s0 = *reinterpret_cast<const __half2*>(&m0.x), s1 = *reinterpret_cast<const __half2*>(&m1.x);
      // hi: q * scale + 0 rounded once; lo: q * scale - hi, exact
      const __half2 h0 = __hmul2(q0, s0), h1 = __hmul2(q1, s1);
      const __half2 b0 = __hfma2(q0, s0, __hmul2(h0, lo_sel)), b1 = __hfma2(q1, s1, __hmul2(h1, lo_sel));
      bh0 = *reinterpret_cast<const uint32_t*>(&b0);
      bh1 = *reinterpret_cast<const uint32_t*>(&b1);
      mma16816(zacc, m0.x, m0.y, m1.x, m1.y, qq.x, qq.y);
    } else if (W != 16) {
      // a pair past the segment end reads the block's first pair (its q entries are 0)
      const uint2 m0 = lds64(kmeta, mb + (v0 ? 8u * q : 0u));
      const uint2 m1 = lds64(kmeta, mb + (v1 ? 8u * (q + 4) : 0u));
      const __half2 q0 = *reinterpret_cast<const __half2*>(&qq.x), q1 = *reinterpret_cast<const __half2*>(&qq.y);
      const __half2 s0 = *reinterpret_cast<const __half2*>(&m0.x), s1 = *reinterpret_cast<const __half2*>(&m1.x);
      const __half2 h0 = __hmul2(q0, s0), h1 = __hmul2(q1, s1);
      const __half2 l0 = __hfma2(q0, s0, __hneg2(h0)), l1 = __hfma2(q1, s1, __hneg2(h1));
      bh0 = *reinterpret_cast<const uint32_t*>(&h0);
      bh1 = *reinterpret_cast<const uint32_t*>(&h1);
      bl0 = *reinterpret_cast<const uint32_t*>(&l0);
      bl1 = *reinterpret_cast<const uint32_t*>(&l1);
      // A = the metadata as loaded, {scales, zeros} of the two pairs: rows g get sum scale * q
      // (unused) and rows g + 8 the zero-point term sum zero * q, with no register shuffling
      mma16816(zacc, m0.x, m0.y, m1.x, m1.y, qq.x, qq.y);
    }
#pragma unroll
    for (int tb = 0; tb < 2; ++tb) {
      const uint32_t x0 = pick4(y0, 2 * tb), x1 = pick4(y0, 2 * tb + 1);
      const uint32_t x2 = pick4(y1, 2 * tb), x3 = pick4(y1, 2 * tb + 1);
      if (W == 16) {  // raw fp16 words past the segment end may hold anything: zero them
        const uint32_t k0 = v0 ? ~0u : 0u, k1 = v1 ? ~0u : 0u;
        mma16816(shi[tb], x0 & k0, x1 & k0, x2 & k1, x3 & k1, bh0, bh1);
      } else {
        const uint32_t a0 = W == 8 ? __byte_perm(x0, 0u, bsel) : (x0 >> sh0) & mask2;
        const uint32_t a1 = W == 8 ? __byte_perm(x1, 0u, bsel) : (x1 >> sh0) & mask2;
        const uint32_t a2 = W == 8 ? __byte_perm(x2, 0u, bsel) : (x2 >> sh1) & mask2;
        const uint32_t a3 = W == 8 ? __byte_perm(x3, 0u, bsel) : (x3 >> sh1) & mask2;
        mma16816(shi[tb], a0, a1, a2, a3, bh0, bh1);
        if (!PK) mma16816(slo[tb], a0, a1, a2, a3, bl0, bl1);
      }
    }
  }
}

template <int D, bool QLO, bool PK>
__device__ __forceinline__ void tile_logits(const unsigned char* kw, const unsigned char* kmeta, const int (&seg_kb)[5],
                                            const KBDesc* kbd, const float4* qv, int lane,
                                            float (&s)[2][4]) {
  float bias = 0.f;  // sum over this lane's slots of q_g * zero (head g)
#pragma unroll
  for (int tb = 0; tb < 2; ++tb) s[tb][0] = s[tb][1] = s[tb][2] = s[tb][3] = 0.f;
  const int q = lane & 3;
  float be, bo;
  if (QLO) {
    k_segment<16, QLO>(kw, kmeta, seg_kb[0], seg_kb[1], kbd, qv, lane, s, bias);
    k_segment<8, QLO>(kw, kmeta, seg_kb[1], seg_kb[2], kbd, qv, lane, s, bias);
    k_segment<4, QLO>(kw, kmeta, seg_kb[2], seg_kb[3], kbd, qv, lane, s, bias);
    k_segment<2, QLO>(kw, kmeta, seg_kb[3], seg_kb[4], kbd, qv, lane, s, bias);
    // zero-point term: lanes (g, 0..3) hold parts of head g; S^T lane (g', q') needs heads 2q', 2q'+1
    bias += __shfl_xor_sync(0xffffffffu, bias, 1);
    bias += __shfl_xor_sync(0xffffffffu, bias, 2);
    be = __shfl_sync(0xffffffffu, bias, 8 * q);
    bo = __shfl_sync(0xffffffffu, bias, 8 * q + 4);
  } else {
    const uint2* qh = reinterpret_cast<const uint2*>(qv);
    float zacc[4] = {0.f, 0.f, 0.f, 0.f};  // [2], [3]: zero-point term of heads 2q, 2q+1
    // raw 16-bit channels first, at scale 1 in s; then s moves to 2^-24 and takes the hi products
    float slo[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    k_segment_h<16, PK>(kw, kmeta, seg_kb[0], seg_kb[1], kbd, qh, lane, s, slo, zacc);
#pragma unroll
    for (int tb = 0; tb < 2; ++tb)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[tb][e] *= 5.9604644775390625e-8f;
    k_segment_h<8, PK>(kw, kmeta, seg_kb[1], seg_kb[2], kbd, qh, lane, s, slo, zacc);
    k_segment_h<4, PK>(kw, kmeta, seg_kb[2], seg_kb[3], kbd, qh, lane, s, slo, zacc);
    k_segment_h<2, PK>(kw, kmeta, seg_kb[3], seg_kb[4], kbd, qh, lane, s, slo, zacc);
    // back to scale 1; PK: the lo columns (2q + 4, 2q + 5) are held by lane q ^ 2
#pragma unroll
    for (int tb = 0; tb < 2; ++tb)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        s[tb][e] = (s[tb][e] + (PK ? __shfl_xor_sync(0xffffffffu, s[tb][e], 2) : slo[tb][e])) * 16777216.f;
    be = zacc[2];
    bo = zacc[3];
  }
#pragma unroll
  for (int tb = 0; tb < 2; ++tb) {
    s[tb][0] += be;
    s[tb][1] += bo;
    s[tb][2] += be;
    s[tb][3] += bo;
  }
}

// PV of a zone-A tile with packed V of width VB.  A dequantised V element is
// zero + scale * code per (token, 32-channel group), so per head h and channel c
//   O[h][c] += sum_t (p_ht scale_t) code_tc + sum_t p_ht zero_t.
// The codes enter the tensor core as fp16 subnormals (code * 2^-24, one shift
// and one mask) against B = p * scale of the group (one half2 multiply per
// fragment), so the products land in acc.o scaled by 2^-24 (the caller keeps
// track of that scale); the zero-point sums go to acc.z through one MMA per
// 16 tokens whose A row g holds the zeros of channel group g.
template <int D, int VB>
__device__ __forceinline__ void tile_pv_packed(WarpAcc<D>& acc, const unsigned char* vcodes, const unsigned char* vmeta, int lane,
                                               const uint32_t (&pb)[2][2]) {
  const int g = lane >> 2, q = lane & 3;
  constexpr int wpp = D * VB / 16;  // words per token pair
  constexpr int per = 16 / VB;      // channels per half-word
  constexpr int NG = D / 32;        // channel groups
  constexpr uint32_t mask2 = VB == 8 ? 0x00ff00ffu : VB == 4 ? 0x000f000fu : 0x00030003u;
  constexpr int R = VB / 2;         // word groups inside a pair (words w = r mod R together)
  const int sh0 = VB * (g % per), sh1 = VB * ((g + 8) % per);
  const uint32_t bsel = byte_pair_sel(g & 1);  // 8-bit codes: bytes (0, 2) or (1, 3) of a word
#pragma unroll
  for (int tb = 0; tb < 2; ++tb) {
    const int p0 = 8 * tb + q, p1 = p0 + 4;
    // this lane's channels c = g + 8 i (i = 0 .. D/8-1) live in the words w = 2 i / ... of group
    // g / per, stored adjacently in order of i: word i of the group holds channel g + 8 i
    const unsigned char* base0 = vcodes + 4 * (p0 * wpp + (g / per) * (wpp / R));
    const unsigned char* base1 = vcodes + 4 * (p1 * wpp + (g / per) * (wpp / R));
    uint32_t za0 = 0u, za2 = 0u;
    if (g < NG) {
      za0 = lds32(vmeta, 8 * (p0 * NG + g) + 4);
      za2 = lds32(vmeta, 8 * (p1 * NG + g) + 4);
    }
    mma16816(acc.z, za0, 0u, za2, 0u, pb[tb][0], pb[tb][1]);
#pragma unroll
    for (int grp = 0; grp < NG; ++grp) {
      const uint32_t s0 = lds32(vmeta, 8 * (p0 * NG + grp)), s1 = lds32(vmeta, 8 * (p1 * NG + grp));
      const __half2 b0h = __hmul2(*reinterpret_cast<const __half2*>(&pb[tb][0]), *reinterpret_cast<const __half2*>(&s0));
      const __half2 b1h = __hmul2(*reinterpret_cast<const __half2*>(&pb[tb][1]), *reinterpret_cast<const __half2*>(&s1));
      const uint32_t b0 = *reinterpret_cast<const uint32_t*>(&b0h), b1 = *reinterpret_cast<const uint32_t*>(&b1h);
      // words i = 4 grp .. 4 grp + 3 of the lane's group: channels of (cm, c0), (cm, c1) for
      // cm = 2 grp, 2 grp + 1
      const uint4 v0 = lds128(base0, 16 * grp), v1 = lds128(base1, 16 * grp);
      const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w}, w1[4] = {v1.x, v1.y, v1.z, v1.w};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int cm = 2 * grp + half;
        const uint32_t a0 = VB == 8 ? __byte_perm(w0[2 * half], 0u, bsel) : (w0[2 * half] >> sh0) & mask2;
        const uint32_t a1 = VB == 8 ? __byte_perm(w0[2 * half + 1], 0u, bsel) : (w0[2 * half + 1] >> sh1) & mask2;
        const uint32_t a2 = VB == 8 ? __byte_perm(w1[2 * half], 0u, bsel) : (w1[2 * half] >> sh0) & mask2;
        const uint32_t a3 = VB == 8 ? __byte_perm(w1[2 * half + 1], 0u, bsel) : (w1[2 * half + 1] >> sh1) & mask2;
        mma16816(acc.o[cm], a0, a1, a2, a3, b0, b1);
      }
    }
  }
}

// Multiplies the O^T accumulators by f (a power of two: exact).
template <int D>
__device__ __forceinline__ void scale_o(WarpAcc<D>& acc, float f) {
#pragma unroll
  for (int cm = 0; cm < D / 16; ++cm) {
    acc.o[cm][0] *= f;
    acc.o[cm][1] *= f;
    acc.o[cm][2] *= f;
    acc.o[cm][3] *= f;
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

// Estimated decode cost of a head: its zone-A tiles and its zone-C blocks.
__host__ __device__ __forceinline__ int64_t head_cost(const rdkv_head_plan& hp, int zc_blocks) {
  return head_cost_a(hp) + (int64_t)zc_blocks * kZoneCBlockCost;
}

// Per-class values of a head, read with a class index without dynamic array indexing.
struct ClassVals {
  int64_t v[4];
  __device__ __forceinline__ int64_t operator()(int c) const { return c == 0 ? v[0] : c == 1 ? v[1] : c == 2 ? v[2] : v[3]; }
};

template <int D, bool QLO, bool PK>
__global__ void __launch_bounds__(kDecWarps * 32, 1) decode_kernel(const __grid_constant__ DecodeParams P) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = P.h_q / P.h_kv;
  // the next kernel on the stream may start its own static setup once every block of this one runs
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ int asg[3];  // head, first block of the head, blocks of the head
  __shared__ __align__(16) rdkv_head_plan hp_s;  // this block's head record
  int16_t slot_pre = -1;  // dealt on the host: this thread's slot-table entry, loaded with the record
  // the cache this block reads (part 0 unless the host dealt blocks over several caches)
  const DecodePart& PP = P.parts[P.dealt ? P.block_part[blockIdx.x] : 0];
  if (P.dealt) {
    // dealt on the host: this block's head and split range are kernel arguments
    const int hb = P.block_head[blockIdx.x];
    if (hb != kNoHead && tid < P.slot_stride) slot_pre = PP.slots[(int64_t)hb * P.slot_stride + tid];
    if (warp == 0) {
      if (lane == 0) {
        asg[0] = hb == kNoHead ? -1 : hb;
        asg[1] = hb == kNoHead ? 0 : P.head_first[hb];
        asg[2] = hb == kNoHead ? 0 : P.head_first[hb + 1] - P.head_first[hb];
      }
      if (hb != kNoHead)  // the head record into shared memory, one word per lane
        reinterpret_cast<int32_t*>(&hp_s)[lane] = reinterpret_cast<const int32_t*>(PP.heads + hb)[lane];
    }
  } else if (warp == 0) {
    // Blocks are dealt to heads in proportion to their estimated cost, at least one per head, over a
    // nominal P.ctas blocks; the grid has P.ctas + n_heads blocks and the blocks past the last head's
    // range leave at once.  Warp 0: one lane per head, one round trip for the plan records and the
    // zone-C length, then a scan.
    // static inputs only (plan and capacity): the dealing is the same in every launch, also before
    // the previous kernel on the stream has finished
    const int zc = ceil_div(P.cap_c, kCRows);
    int64_t total = 0;
    for (int h = lane; h < P.n_heads; h += 32) total += head_cost(P.heads[h], zc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
    int start = 0, found = -1;
    for (int h0 = 0; h0 < P.n_heads; h0 += 32) {
      const int h = h0 + lane;
      const int64_t w = h < P.n_heads ? head_cost(P.heads[h], zc) : 0;
      const int c = h < P.n_heads ? max(1, (int)(total > 0 ? w * P.ctas / total : 0)) : 0;
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
  const int b = head / P.h_kv, j = head % P.h_kv;
  const rdkv_head_plan* hpp = &hp_s;
  const bool fused = P.k_new != nullptr;

  // the slot table goes into registers now (static data)
  const int qbase = b * P.h_q + j * G;
  const int16_t* slot_ch = PP.slots + (int64_t)head * P.slot_stride;
  const int k_slots = hpp->k_slots;  // <= D + kSlotPad <= the block's threads
  const int16_t sr = tid < k_slots ? (P.dealt ? slot_pre : slot_ch[tid]) : (int16_t)-1;

  // shared memory map
  KBDesc* kbd = reinterpret_cast<KBDesc*>(smem);                                   // [kMaxKB]
  float4* qv = reinterpret_cast<float4*>(smem + 256);                              // [kMaxKB][32] (uint2 if !QLO)
  uint4* qfragc = reinterpret_cast<uint4*>(smem + 256 + kMaxKB * 32 * (QLO ? 16 : 8));  // [D/16][32] hi, lo
  int16_t* slot_s = reinterpret_cast<int16_t*>(qfragc + (D / 16) * 32);            // [D + kSlotPad] slot table
  uint64_t* bars = reinterpret_cast<uint64_t*>(slot_s + D + kSlotPad);             // [warps][kMaxInflight]
  int* ring_pos = reinterpret_cast<int*>(bars + kDecWarps * kMaxInflight);         // [warps][kMaxInflight]
  int* ring_item = ring_pos + kDecWarps * kMaxInflight;                            // [warps][kMaxInflight]
  uint32_t* ring_need = reinterpret_cast<uint32_t*>(ring_item + kDecWarps * kMaxInflight);  // [warps][kMaxInflight]
  uint16_t* newrow = reinterpret_cast<uint16_t*>(ring_need + kDecWarps * kMaxInflight);     // [2][D] fused step: k, v
  unsigned char* ring = smem + decode_fixed_smem(D, QLO);
  float* red = reinterpret_cast<float*>(ring);                                     // [warps][8][D + 2], after the loop
  __shared__ int seg_kb_s[5];
  __shared__ int is_last;
  __shared__ int next_k;

  // items of this head: its tiles in class order, then its zone-C blocks
  ClassVals cstart, coff, ctb, cnv;  // first item, first byte in zone A, tile bytes, kept tokens per class
  int zc_start;
  {
    int t = 0;
    int64_t off = hpp->a_off;
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
  const int RW = hpp->row_words, meta_slots = hpp->meta_slots;
  // split s of n takes items s, s + n, s + 2n, ...: every split gets its share of each class.  The
  // zone-C length is known only after the wait for the previous kernel: until then only zone-A
  // items are issued (an item past them stays pending)
  int n_items = zc_start, len_c = 0, n_rows = 0;
  bool items_final = false;
  if (tid == 0) next_k = 0;

  // k-block descriptors of this head's K rows (each block inside one width segment), one per thread
  if (warp == 1 && lane < kMaxKB) {
    int nb[4], wb[4], sb[4], mb[4], ns[4];
    int nkb = 0, wsum = 0, ssum = 0, msum = 0;
#pragma unroll
    for (int seg = 0; seg < 4; ++seg) {
      const int w = 16 >> seg, per = 32 / w;
      const int nslot = hpp->k_words[seg] * per;
      ns[seg] = nslot;
      nb[seg] = nkb;
      wb[seg] = wsum;
      sb[seg] = ssum;
      mb[seg] = msum;
      nkb += ceil_div(nslot, 16);
      wsum += hpp->k_words[seg];
      ssum += nslot;
      if (w < 16) msum += nslot;
    }
    auto pick = [](const int (&a)[4], int i) { return i == 0 ? a[0] : i == 1 ? a[1] : i == 2 ? a[2] : a[3]; };
    if (lane < 4) seg_kb_s[lane] = pick(nb, lane);
    if (lane == 4) seg_kb_s[4] = nkb;
    if (lane < nkb) {
      const int seg = (lane >= nb[1]) + (lane >= nb[2]) + (lane >= nb[3]);
      const int w = 16 >> seg, per = 32 / w;
      const int nslot = pick(ns, seg);
      const int s0 = 16 * (lane - pick(nb, seg));
      KBDesc d;
      d.wbyte = 128 * (pick(wb, seg) + s0 / per);
      d.mbyte = 8 * ((w < 16 ? pick(mb, seg) + s0 : 0) / 2);
      d.nrem = min(16, nslot - s0);
      d.slot0 = pick(sb, seg) + s0;
      kbd[lane] = d;
    }
  }

  auto item_cls = [&](int it) {
    return it < (int)cstart.v[1] ? 0 : it < (int)cstart.v[2] ? 1 : it < (int)cstart.v[3] ? 2 : it < zc_start ? 3 : -1;
  };

  // per-warp ring of shared memory filled by bulk copies (lane 0 issues)
  unsigned char* wring = ring + (int64_t)warp * P.ring_bytes;
  uint64_t* wbar = bars + warp * kMaxInflight;
  int* wpos = ring_pos + warp * kMaxInflight;
  uint32_t head_p = 0, used = 0;       // lane 0: next write offset; bytes held, wrap waste included
  int* witem = ring_item + warp * kMaxInflight;  // per slot: (class + 1) << 24 | index within the class
  uint32_t* wneed = ring_need + warp * kMaxInflight;  // bytes each slot holds, wrap waste included
  int issued = 0, done = 0;
  bool drained = warp >= P.ring_warps;  // lane 0: no item left for this warp (warps without a ring take none)
  int pending = -1;                    // lane 0: item taken but not yet issued (ring full)
  int cap = kPrologueItems;  // items in flight per warp: fewer before the loop starts
  auto issue = [&]() {
    if (issued == done) head_p = used = 0;  // empty ring: start at its beginning
    while (!drained && issued - done < cap) {
      int it = pending;
      if (it < 0) it = isplit + in_split * atomicAdd(&next_k, 1);  // taken in order of need: no warp idles early
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
      uint32_t phys = head_p, need = sz;
      if (phys + sz > (uint32_t)P.ring_bytes) { need += (uint32_t)P.ring_bytes - phys; phys = 0; }
      if (used + need > (uint32_t)P.ring_bytes) {
        pending = it;
        break;
      }
      pending = -1;
      head_p = phys + sz;
      used += need;
      const int slot = issued % kMaxInflight;
      wneed[slot] = need;
      wpos[slot] = (int)phys;
      witem[slot] = ((cls + 1) << 24) | (cls >= 0 ? it - (int)cstart(cls) : it - zc_start);
      unsigned char* dst = wring + phys;
      uint64_t* bar = &wbar[slot];
      if (P.arm_only) {
        // timeout self-test: the stage waits for 16 bytes and no copy is issued, so its wait runs out
        mbar_arrive_expect_tx(bar, 16u);
      } else if (cls >= 0) {
        const int ti = it - (int)cstart(cls);
        const uint32_t zb = cls == 3 ? (uint32_t)kTile * D * 2 : 0u;
        mbar_arrive_expect_tx(bar, a_bytes + zb);
        const uint64_t pol = evict_first_policy();
        bulk_copy_once(dst, PP.zone_a + coff(cls) + (int64_t)ti * a_bytes, a_bytes, bar, pol);
        if (zb) bulk_copy_once(dst + a_bytes, PP.zone_b + (b_row + (int64_t)kTile * ti) * D, zb, bar, pol);
      } else {
        // rows of zone C (the fused step's new row, past them, is written by the consumer)
        const int rows = max(0, min(kCRows, len_c - c_row));
        const uint32_t bytes = (uint32_t)rows * D * 2;
        // a zone-C item is 16 rows: one page when zone C is paged
        const int64_t src = zone_c_offset(PP.zc_pages, PP.zc_page_stride, PP.cap_c, head, c_row, D);
        mbar_arrive_expect_tx(bar, 2 * bytes);
        if (bytes) {
          const uint64_t pol = evict_first_policy();
          bulk_copy_once(dst, PP.zone_c_k + src, bytes, bar, pol);
          bulk_copy_once(dst + kCRows * D * 2, PP.zone_c_v + src, bytes, bar, pol);
        }
      }
      ++issued;
    }
  };
  if (lane == 0) {
    for (int k = 0; k < kMaxInflight; ++k) mbar_init(&wbar[k], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid < k_slots) slot_s[tid] = sr;
  __syncthreads();  // next_k, the barriers, the k-block descriptors and the slot table are set
  if (lane == 0) issue();  // the first zone-A copies fly while the query fragments are built
  const int nkb = seg_kb_s[4];
  int seg_kb[5];
#pragma unroll
  for (int i = 0; i < 5; ++i) seg_kb[i] = seg_kb_s[i];
  // Query fragments: B[k = slot pair][n = head g] in slot order (zone A) and channel order (zone C),
  // at most two per thread.  Which query element each entry takes is static: look it up now.
  static_assert((kMaxKB + 128 / 16) * 32 <= 2 * kDecWarps * 32, "two query fragments per thread");
  const int n_frag = (nkb + D / 16) * 32;
  int fq[2][4];  // element of the group's query rows [G][D] per fragment entry, or -1
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int i = tid + r * kDecWarps * 32;
    const int kb = i >> 5, ln = i & 31, qq = ln & 3;
    // the head of column g: zone-A fragments with PK hold heads 0-3 twice (hi and lo columns)
    const int g = (PK && kb < nkb) ? (ln >> 2) & 3 : ln >> 2;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int off = 2 * qq + (e & 1) + 8 * (e >> 1);
      int ch = -1;
      if (i < n_frag && g < G) {
        if (kb < nkb) {
          const KBDesc d = kbd[kb];
          ch = off < d.nrem ? slot_s[d.slot0 + off] : -1;
        } else {
          ch = 16 * (kb - nkb) + off;
        }
      }
      fq[r][e] = ch >= 0 ? g * D + ch : -1;
    }
  }
  // Everything so far read only the plan and zone A, which the kernel launched just before this one
  // on the stream does not write.  The query, the new token and the zone-C length may come from
  // it: wait for it here (a no-op without programmatic dependent launch).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  len_c = min(*PP.len_dev, PP.cap_c);
  n_rows = len_c + (fused ? 1 : 0);
  n_items = zc_start + ceil_div(n_rows, kCRows);
  items_final = true;
  float qf[2][4];
#pragma unroll
  for (int r = 0; r < 2; ++r)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      qf[r][e] = fq[r][e] >= 0 ? load_as_float(P.q, (int64_t)qbase * D + fq[r][e], P.dtype) : 0.f;
  if (fused && tid < 2 * D) {
    const int64_t src = (int64_t)head * D + (tid % D);
    newrow[tid] = half_bits(load_as_float(tid < D ? P.k_new : P.v_new, src, P.dtype));
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int i = tid + r * kDecWarps * 32;
    if (i < n_frag) {
      const int kb = i >> 5, ln = i & 31;
      const float* v = qf[r];
      if (kb >= nkb) qfragc[(kb - nkb) * 32 + ln] = split_hi_lo(v[0], v[1], v[2], v[3]);
      else if (QLO) qv[kb * 32 + ln] = make_float4(v[0], v[1], v[2], v[3]);
      else reinterpret_cast<uint2*>(qv)[kb * 32 + ln] = make_uint2(pack_half2(v[0], v[1]), pack_half2(v[2], v[3]));
    }
  }
  __syncthreads();

  cap = kMaxInflight;
  WarpAcc<D> acc;
#pragma unroll
  for (int cm = 0; cm < D / 16; ++cm) acc.o[cm][0] = acc.o[cm][1] = acc.o[cm][2] = acc.o[cm][3] = 0.f;
  acc.z[0] = acc.z[1] = acc.z[2] = acc.z[3] = 0.f;
  // acc.o holds packed-V products at 2^-24 while this is set; a warp meets the classes in
  // increasing order (items ascend), so it switches at most once, at its first 16-bit tile or
  // zone-C block
  bool o_sub = true;
  acc.m[0] = acc.m[1] = -INFINITY;
  acc.l[0] = acc.l[1] = 0.f;
  const float sl2 = 1.4426950408889634f / sqrtf((float)D);
  const int g = lane >> 2, q = lane & 3;
  bool ok = true;

  while (true) {
    if (lane == 0) issue();
    __syncwarp();
    if (__shfl_sync(0xffffffffu, issued, 0) == done) break;  // nothing in flight and nothing left
    const int slot = done % kMaxInflight;
    const bool arrived = mbar_wait(&wbar[slot], (uint32_t)(done / kMaxInflight) & 1u, P.wait_cycles);
    if (__any_sync(0xffffffffu, !arrived)) {
      ok = false;
      break;
    }
    const uint32_t st = smem_u32(wring + wpos[slot]);
    const int rec = witem[slot];
    const int cls = (rec >> 24) - 1, ti = rec & 0xffffff;  // ti: tile of the class, or zone-C block
    if (cls >= 0) {
      const int n_real = min(kTile, (int)cnv(cls) - kTile * ti);
      const unsigned char* stp = wring + wpos[slot];
      const unsigned char* kmeta = stp + 4 * kTile * RW;
      float s[2][4];
      tile_logits<D, QLO, PK>(stp, kmeta, seg_kb, kbd, qv, lane, s);
#pragma unroll
      for (int tb = 0; tb < 2; ++tb)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[tb][e] *= sl2;
      if (n_real < kTile) {  // the last tile of a class: tokens past the kept ones
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
      const unsigned char* vcodes = kmeta + 4 * meta_slots;
      if (cls < 3 && !o_sub) {
        scale_o(acc, 5.9604644775390625e-8f);
        o_sub = true;
      } else if (cls == 3 && o_sub) {
        scale_o(acc, 16777216.f);
        o_sub = false;
      }
      if (cls == 0) tile_pv_packed<D, 2>(acc, vcodes, vcodes + kTile * D * 2 / 8, lane, pb);
      else if (cls == 1) tile_pv_packed<D, 4>(acc, vcodes, vcodes + kTile * D * 4 / 8, lane, pb);
      else if (cls == 2) tile_pv_packed<D, 8>(acc, vcodes, vcodes + kTile * D * 8 / 8, lane, pb);
      else pv_fp16<D, 2>(acc, st + (uint32_t)ctb.v[3], lane, pb);
    } else {
      if (o_sub) {
        scale_o(acc, 16777216.f);
        o_sub = false;
      }
      const int c_row = ti * kCRows;
      const int rows = min(kCRows, n_rows - c_row);  // rows attended (the fused step's new row last)
      const int copied = max(0, min(kCRows, len_c - c_row));
      if (rows < kCRows || copied < rows) {
        uint32_t* kz = reinterpret_cast<uint32_t*>(wring + wpos[slot]);
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
        if (QLO) mma16816(s[0], a0, a1, a2, a3, qf.z, qf.w);
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
    if (lane == 0) used -= wneed[slot];
    ++done;
  }
  if (!ok) {
    if (lane == 0) {
      atomicExch(P.error, (int)RDKV_ERR_TIMEOUT);
      // wait (bounded) for this warp's copies still in flight before the ring is reused
      for (int k = done; k < issued; ++k)
        if (!mbar_wait(&wbar[k % kMaxInflight], (uint32_t)(k / kMaxInflight) & 1u, P.wait_cycles)) break;
    }
    __syncwarp();
  }
  __syncthreads();  // every ring drained: the ring area now holds the warps' results
  if (o_sub) scale_o(acc, 16777216.f);
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

  // warp result -> shared memory: m, l per head; O per head and channel
  float l0 = acc.l[0], l1 = acc.l[1];
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, o);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o);
  }
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
    rw[(2 * q) * (D + 2) + D + 1] = l0;
    rw[(2 * q + 1) * (D + 2) + D + 1] = l1;
  }
  __syncthreads();
  // combine the warps; write this block's partial result (m, l, unnormalised o) for the G heads;
  // one block's partial takes pstride floats
  const int pstride = partial_stride(G, D);
  float* part = P.partial + (int64_t)first_block * pstride;
  float* mine = part + (int64_t)split * pstride;
  // each element: the block's running max M of its head over the warps, then the warps' results
  // weighted by 2^(m_w - M) (the m (c = D) entry holds M)
  for (int i = tid; i < G * (D + 2); i += blockDim.x) {
    const int h = i / (D + 2), c = i % (D + 2);
    float mw[kDecWarps];
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) {
      mw[w] = red[((int64_t)w * 8 + h) * (D + 2) + D];
      M = fmaxf(M, mw[w]);
    }
    float val = M;
    if (c != D) {
      val = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) val = fmaf(ex2(mw[w] - M), red[((int64_t)w * 8 + h) * (D + 2) + c], val);
      }
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
    if (len_c < P.cap_c) {
      const int64_t dst = zone_c_offset(PP.zc_pages, PP.zc_page_stride, PP.cap_c, head, len_c, D);
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
  // Merge: out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s per query head and channel.  One
  // thread per output element loads what it needs straight from the splits' partials (L2; the
  // acquire above made them visible), kMergeBatch splits at a time with every load of a batch in
  // flight together, and folds each batch into its running (M, L, O).
  constexpr int kMergeBatch = 24;
  for (int i = tid; i < G * D; i += blockDim.x) {
    const int h = i / D, c = i % D;
    const float* ph = part + h * (D + 2);
    float M = -INFINITY, L = 0.f, O = 0.f;
    for (int s0 = 0; s0 < n_split; s0 += kMergeBatch) {
      float mv[kMergeBatch], lv[kMergeBatch], ov[kMergeBatch];
#pragma unroll
      for (int k = 0; k < kMergeBatch; ++k) {
        const bool in = s0 + k < n_split;
        const float* ps = ph + (int64_t)(s0 + k) * pstride;
        mv[k] = in ? __ldcg(ps + D) : -INFINITY;
        lv[k] = in ? __ldcg(ps + D + 1) : 0.f;
        ov[k] = in ? __ldcg(ps + c) : 0.f;
      }
      float Mn = M;
#pragma unroll
      for (int k = 0; k < kMergeBatch; ++k) Mn = fmaxf(Mn, mv[k]);
      if (Mn == -INFINITY) continue;  // no token seen so far
      const float so = M == -INFINITY ? 0.f : ex2(M - Mn);
      float l1 = 0.f, o1 = 0.f;
#pragma unroll
      for (int k = 0; k < kMergeBatch; ++k) {
        const float w = ex2(mv[k] - Mn);  // 0 for a split without tokens (m = -inf)
        l1 = fmaf(w, lv[k], l1);
        o1 = fmaf(w, ov[k], o1);
      }
      L = fmaf(L, so, l1);
      O = fmaf(O, so, o1);
      M = Mn;
    }
    P.out[((int64_t)b * P.h_q + j * G + h) * D + c] = L > 0.f ? O / L : 0.f;
    // ln of the denominator: the running sums are of 2^(s log2(e) / sqrt(D) - M)
    if (P.lse != nullptr && c == 0)
      P.lse[(int64_t)b * P.h_q + j * G + h] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
  }
}

constexpr int64_t kDecodeSmemLimit = 227 * 1024 - 1024;  // per-block limit less room for static shared memory

struct DecodeGeom {
  int64_t max_item;
  int ctas;     // nominal number of blocks dealt to heads
  int splits;   // grid size: ctas + one spare block per head
  int ring_bytes;
  int ring_warps;  // warps with a ring (all, or fewer with larger rings when tiles are large)
  size_t smem;
  size_t partial_bytes;
  size_t ticket_off;   // tickets then the status word
};

// Geometry of a launch over the caches parts[0 .. n) (one, or segments and the live cache).
static DecodeGeom decode_geom(const rdkv_cache* const* parts, int n) {
  DecodeGeom g;
  const rdkv_shape& s = parts[0]->shape;
  const int D = s.head_dim, G = s.h_q / s.h_kv;
  const int n_heads = s.batch * s.h_kv;
  const int sms = num_sms();
  const int64_t fixed = decode_fixed_smem(D, s.dtype == RDKV_F32);
  int64_t max_item = 2 * kCRows * D * 2, items = 0;
  for (int p = 0; p < n; ++p) {
    max_item = std::max<int64_t>(max_item, align_up(parts[p]->sizes.max_stage_bytes, 128));
    items += ceil_div64(parts[p]->sizes.index_slots, kTile) + (int64_t)n_heads * ceil_div(parts[p]->cap_c, kCRows);
  }
  g.max_item = max_item;
  // one block of kDecWarps warps per SM; the warps with a ring share what is left equally: all of
  // them, or half (a quarter) with twice (four times) the ring when the largest staged tile needs it
  int ring_warps = kDecWarps;
  int64_t ring = ((kDecodeSmemLimit - fixed) / ring_warps) / 128 * 128;
  while (ring < max_item && ring_warps > kDecWarps / 4) {
    ring_warps /= 2;
    ring = ((kDecodeSmemLimit - fixed) / ring_warps) / 128 * 128;
  }
  const int blocks_per_sm = 1;
  if ((int64_t)ring_warps * ring < decode_reduce_bytes(D)) ring = 0;  // the warps' results reuse the rings
  g.ring_bytes = (int)ring;
  g.ring_warps = ring_warps;
  g.smem = (size_t)(fixed + (int64_t)ring_warps * ring);
  // blocks dealt to heads in proportion to their work: a nominal count that fills every SM once,
  // fewer when there is little work (at least kDecWarps items per block on average).
  // With few heads, leave one SM per head free: the last block of each head merges after the
  // others have left, and on those SMs the next call's blocks would otherwise start only after
  // the merge, with their whole set-up still ahead of them.
  const int free_sms = n_heads <= sms / 16 ? n_heads : 0;
  g.ctas = (int)std::max<int64_t>(
      1, std::min<int64_t>((int64_t)blocks_per_sm * (sms - free_sms), ceil_div64(items, kDecWarps)));
  g.splits = g.ctas + n_heads * n;  // grid size: room for at least one block per (cache, head)
  g.partial_bytes = (size_t)align_up((int64_t)g.splits * partial_stride(G, D) * 4, 256);
  g.ticket_off = g.partial_bytes;
  return g;
}
static DecodeGeom decode_geom(const rdkv_cache* c) { return decode_geom(&c, 1); }

// ws: partials, then per-head tickets, the status word and the fused step's head counter
static size_t decode_ws_bytes(const DecodeGeom& g, int n_heads) {
  return g.ticket_off + (size_t)align_up(((int64_t)n_heads + 2) * 4, 256);
}

rdkv_status check_cache_public(const rdkv_cache* c);

// Kernel arguments of one decode call over parts[0 .. n); ws holds the partials, then the tickets and
// the status word.  The blocks are dealt on the host when every cache's plan costs reached it
// (rdkv_plan_sizes), else (one cache only) by the kernel.
static DecodeParams decode_params(const rdkv_cache* const* parts, int n, const DecodeGeom& geo, const void* q,
                                  float* out, void* ws, const void* k_new = nullptr, const void* v_new = nullptr,
                                  float* lse = nullptr) {
  const rdkv_cache* cache = parts[0];
  const rdkv_shape& s = cache->shape;
  const int n_heads = s.batch * s.h_kv;
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
  }
  // Deal the blocks to the heads here when the plans' cost estimates reached the host: the kernel
  // then knows its head at once instead of reading every head record first.  The rule is the
  // kernel's own (at least one block per head and cache, the rest in proportion to the cost).
  P.dealt = 0;
  bool known = n_heads <= RDKV_COST_HEADS && geo.splits <= kMaxDealtBlocks;
  for (int p = 0; known && p < n; ++p) {
    known = parts[p]->sizes.n_heads == n_heads;
    for (int h = 0; known && h < n_heads; ++h) known = parts[p]->sizes.head_cost[h] > 0;
  }
  if (known) {
    auto cost = [&](int p, int h) {
      return parts[p]->sizes.head_cost[h] + (int64_t)ceil_div(parts[p]->cap_c, kCRows) * kZoneCBlockCost;
    };
    int64_t total = 0;
    for (int p = 0; p < n; ++p)
      for (int h = 0; h < n_heads; ++h) total += cost(p, h);
    int start = 0;
    for (int h = 0; h < n_heads; ++h) {
      P.head_first[h] = (int16_t)start;
      for (int p = 0; p < n; ++p) {
        const int c = std::max(1, (int)(cost(p, h) * geo.ctas / total));
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
  static std::atomic<size_t> smem_set[6][64];
  int dev = 0;
  RDKV_TRY_CUDA(cudaGetDevice(&dev), "device");
  const bool qlo = s.dtype == RDKV_F32;
  // fp16 queries and at most 4 heads per KV head: hi and lo share one MMA per K block
  const bool pk = !qlo && s.h_q / s.h_kv <= 4;
  const int ki = (s.head_dim == 128 ? 3 : 0) + (qlo ? 1 : pk ? 2 : 0);
  void (*const fn)(DecodeParams) = ki == 4 ? decode_kernel<128, true, false>
                                 : ki == 5 ? decode_kernel<128, false, true>
                                 : ki == 3 ? decode_kernel<128, false, false>
                                 : ki == 1 ? decode_kernel<64, true, false>
                                 : ki == 2 ? decode_kernel<64, false, true>
                                           : decode_kernel<64, false, false>;
  if (dev < 64 && geo.smem > smem_set[ki][dev].load(std::memory_order_acquire)) {
    RDKV_TRY_CUDA(cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kDecodeSmemLimit),
                  "decode smem");
    smem_set[ki][dev].store((size_t)kDecodeSmemLimit, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(geo.splits);
  cfg.blockDim = dim3(kDecWarps * 32);
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
  return decode_ws_bytes(decode_geom(cache), cache->shape.batch * cache->shape.h_kv);
}

// selftest_wait > 0: the timeout self-test (stages armed for bytes that no copy delivers, each wait
// limited to that many cycles)
static rdkv_status decode_attn_impl(const rdkv_cache* cache, const void* q, float* out, float* lse, void* ws,
                                    size_t ws_bytes, void* stream, long long selftest_wait = 0) {
  rdkv_status st = check_cache_public(cache);
  if (st != RDKV_OK) return st;
  RDKV_REQUIRE(q && out, RDKV_ERR_INVALID_ARG, "NULL pointer argument");
  const rdkv_shape& s = cache->shape;
  const int n_heads = s.batch * s.h_kv;
  const DecodeGeom geo = decode_geom(cache);
  const size_t need = decode_ws_bytes(geo, n_heads);
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
  const int n_heads = s.batch * s.h_kv;
  const DecodeGeom geo = decode_geom(cache);
  const size_t need = decode_ws_bytes(geo, n_heads);
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
  const int n_heads = cache->shape.batch * cache->shape.h_kv;
  return decode_status_at(ws, geo.ticket_off + 4 * (size_t)n_heads, stream);
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
  return decode_ws_bytes(decode_geom(parts, n_parts), parts[0]->shape.batch * parts[0]->shape.h_kv);
}

extern "C" rdkv_status rdkv_decode_attn_multi(const rdkv_cache* const* parts, int32_t n_parts, const void* q,
                                              float* out, float* lse, void* ws, size_t ws_bytes, void* stream) {
  rdkv_status st = check_parts(parts, n_parts);
  if (st != RDKV_OK) return st;
  RDKV_REQUIRE(q && out, RDKV_ERR_INVALID_ARG, "NULL pointer argument");
  const rdkv_shape& s = parts[0]->shape;
  const int n_heads = s.batch * s.h_kv;
  const DecodeGeom geo = decode_geom(parts, n_parts);
  const size_t need = decode_ws_bytes(geo, n_heads);
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
  return decode_status_at(ws, geo.ticket_off + 4 * (size_t)(parts[0]->shape.batch * parts[0]->shape.h_kv), stream);
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
  const size_t need = decode_ws_bytes(geo, n_heads);
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
