// Decode attention over the TriZone cache of RDKV
// (gist.science/ko/paper/2605.08317, section 2.3): the logits and the output
// are computed with the dequantisation fused into the two products, reading
// zones A (packed K rows and 2/4/8-bit V rows), B (fp16 V rows of 16-bit
// tokens) and C (fp16 K and V rows of the window and of decoded tokens) in one
// pass.
//
// Work: grid = (splits, sequence x KV head).  A head's work items are its
// zone-A tiles (32 tokens, in class order) followed by zone-C blocks of 16
// rows; split s takes a contiguous range of items and its 4 warps take the
// items round-robin.  Every warp streams its items through its own ring of
// shared memory, filled by bulk asynchronous copies that complete on
// per-slot mbarriers (all waits are bounded and report RDKV_ERR_TIMEOUT).
//
// Products: mma.sync m16n8k16 (fp16 in, fp32 accumulate), tokens on M:
//   S^T[16 tok x 8 heads]  += K^[16 tok x 16 slots] * Q^T[16 slots x 8 heads]
//   O^T[16 ch  x 8 heads]  += V^T[16 ch x 16 tok]   * P^T[16 tok x 8 heads]
// A 32-bit A-fragment register holds two consecutive elements along the
// contraction axis (two K slots of one token; two tokens of one V channel);
// the word rule of the layout puts both codes of such a pair in the two
// half-words of one 32-bit word, so one shift and one mask place them, an
// OR with the fp16 pattern of 1024 and a subtraction give the exact codes,
// and one half2 FMA applies scale and zero.  The softmax runs in fp32 on the
// S^T accumulators (base-2 exponent); P^T is moved into B-fragment order by
// movmatrix.  The G query heads of a group share every loaded tile.
#include "common.cuh"

namespace rdkv {

constexpr int kDecWarps = 4;
constexpr int kMaxInflight = 8;
constexpr int kCRows = 16;        // zone-C rows per work item
constexpr int kMaxKB = 16;        // k-blocks of a K row (D = 128: at most 13)
constexpr long long kWaitCycles = 4000000000ll;  // ~2 s at GB300 clocks

struct KBDesc {
  int16_t width;    // 16, 8, 4, 2
  int16_t nrem;     // slots of the segment from the block start (>= 1)
  int32_t word0;    // word of the block's first slot inside a K row
  int32_t meta0;    // index of the block's first slot pair among the quantised pairs
  int32_t pad;
};

// Bytes of the fixed part of the decode kernel's shared memory (before the rings).
__host__ __device__ constexpr int64_t decode_fixed_smem(int D) {
  return ((256 + (int64_t)kMaxKB * 32 * 16 + (int64_t)(D / 16) * 32 * 16 + kDecWarps * kMaxInflight * 12 +
           (int64_t)kDecWarps * 8 * (D + 2) * 4) + 127) / 128 * 128;
}

struct DecodeParams {
  const void* plan;
  const uint8_t* zone_a;
  const uint16_t* zone_b;
  const uint16_t* zone_c_k;
  const uint16_t* zone_c_v;
  const void* q;
  float* partial;   // [n_heads][splits][G][D + 2]
  int32_t* error;   // device status word
  const int32_t* len_dev;  // zone-C rows in use
  int dtype, h_q, h_kv, cap_c, ring_bytes;
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
// Bounded wait; false when the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitCycles) return false;
  }
  return true;
}
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

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

// ---------------------------------------------------------------- per-warp state
template <int D>
struct WarpAcc {
  float o[D / 16][4];   // O^T fragments: (ch 16cm+g, heads 2q, 2q+1), (ch 16cm+g+8, ...)
  float m[2];           // running max (base 2) of heads 2q, 2q+1
  float l[2];           // this lane's share of the running sum
};

// Softmax update for NTB token blocks of S^T accumulators; returns P^T B-fragments.
template <int D, int NTB>
__device__ __forceinline__ void softmax_update(WarpAcc<D>& acc, float (&s)[NTB][4], uint32_t (&pb)[NTB][2]) {
  float mt0 = -INFINITY, mt1 = -INFINITY;
#pragma unroll
  for (int tb = 0; tb < NTB; ++tb) {
    mt0 = fmaxf(mt0, fmaxf(s[tb][0], s[tb][2]));
    mt1 = fmaxf(mt1, fmaxf(s[tb][1], s[tb][3]));
  }
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    mt0 = fmaxf(mt0, __shfl_xor_sync(0xffffffffu, mt0, o));
    mt1 = fmaxf(mt1, __shfl_xor_sync(0xffffffffu, mt1, o));
  }
  const float mn0 = fmaxf(acc.m[0], mt0), mn1 = fmaxf(acc.m[1], mt1);
  // all tokens so far masked: keep everything at zero
  const float ref0 = mn0 == -INFINITY ? 0.f : mn0, ref1 = mn1 == -INFINITY ? 0.f : mn1;
  const float al0 = exp2f(acc.m[0] - ref0), al1 = exp2f(acc.m[1] - ref1);
  acc.m[0] = mn0;
  acc.m[1] = mn1;
  float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
  for (int tb = 0; tb < NTB; ++tb) {
    const float p0 = exp2f(s[tb][0] - ref0), p1 = exp2f(s[tb][1] - ref1);
    const float p2 = exp2f(s[tb][2] - ref0), p3 = exp2f(s[tb][3] - ref1);
    ps0 += p0 + p2;
    ps1 += p1 + p3;
    pb[tb][0] = movmatrix_trans(pack_half2(p0, p1));
    pb[tb][1] = movmatrix_trans(pack_half2(p2, p3));
  }
  acc.l[0] = acc.l[0] * al0 + ps0;
  acc.l[1] = acc.l[1] * al1 + ps1;
#pragma unroll
  for (int cm = 0; cm < D / 16; ++cm) {
    acc.o[cm][0] *= al0;
    acc.o[cm][1] *= al1;
    acc.o[cm][2] *= al0;
    acc.o[cm][3] *= al1;
  }
}

// K logits of a zone-A tile: S^T for token blocks 0 and 1.
// A quantised K element is zero_c + scale_c * code, so per head g
//   q_g . k^ = sum_c q_gc zero_c + sum_c code * (q_gc scale_c).
// The codes are exact in fp16 and form the A operand; q_gc * scale_c (exact in
// fp32) is split into an fp16 high part and an fp16 remainder, two B operands,
// so the products keep ~22 bits; the zero term is summed in fp32.  Raw 16-bit
// channels use the stored fp16 value against q directly.
template <int D>
__device__ __forceinline__ void tile_logits(uint32_t kw, uint32_t kmeta, int RW, int nkb, const KBDesc* kbd,
                                            const float4* qv, int lane, float (&s)[2][4]) {
  const int g = lane >> 2, q = lane & 3;
  float bias = 0.f;  // sum over this lane's slots of q_g * zero (head g)
#pragma unroll
  for (int tb = 0; tb < 2; ++tb) s[tb][0] = s[tb][1] = s[tb][2] = s[tb][3] = 0.f;
  for (int kb = 0; kb < nkb; ++kb) {
    const KBDesc d = kbd[kb];
    const float4 qq = qv[kb * 32 + lane];  // q_g at slots 2q, 2q+1, 2q+8, 2q+9 (0 for pads)
    const bool v0 = 2 * q < d.nrem, v1 = 2 * q + 8 < d.nrem;
    const int b = d.width;
    if (b == 16) {
      const uint4 qs = split_hi_lo(qq.x, qq.y, qq.z, qq.w);
      const uint32_t w0 = d.word0 + q, w1 = d.word0 + q + 4;
#pragma unroll
      for (int tb = 0; tb < 2; ++tb) {
        const uint32_t r0 = kw + 4u * ((16 * tb + g) * RW), r1 = r0 + 4u * (8 * RW);
        const uint32_t a0 = v0 ? lds32(r0 + 4 * w0) : 0u, a1 = v0 ? lds32(r1 + 4 * w0) : 0u;
        const uint32_t a2 = v1 ? lds32(r0 + 4 * w1) : 0u, a3 = v1 ? lds32(r1 + 4 * w1) : 0u;
        mma16816(s[tb], a0, a1, a2, a3, qs.x, qs.y);
        mma16816(s[tb], a0, a1, a2, a3, qs.z, qs.w);
      }
      continue;
    }
    uint32_t w0, w1, mask2;
    int sh0, sh1;
    if (b == 8) {
      w0 = d.word0 + (q >> 1); w1 = w0 + 2; sh0 = sh1 = 8 * (q & 1); mask2 = 0x00ff00ffu;
    } else if (b == 4) {
      w0 = d.word0; w1 = w0 + 1; sh0 = sh1 = 4 * q; mask2 = 0x000f000fu;
    } else {
      w0 = w1 = d.word0; sh0 = 2 * q; sh1 = 2 * q + 8; mask2 = 0x00030003u;
    }
    float sc[4] = {0.f, 0.f, 0.f, 0.f}, ze[4] = {0.f, 0.f, 0.f, 0.f};
    if (v0) {
      const uint2 m = lds64(kmeta + 8 * (d.meta0 + q));
      const float2 s2 = __half22float2(*reinterpret_cast<const __half2*>(&m.x));
      const float2 z2 = __half22float2(*reinterpret_cast<const __half2*>(&m.y));
      sc[0] = s2.x; sc[1] = s2.y; ze[0] = z2.x; ze[1] = z2.y;
    }
    if (v1) {
      const uint2 m = lds64(kmeta + 8 * (d.meta0 + q + 4));
      const float2 s2 = __half22float2(*reinterpret_cast<const __half2*>(&m.x));
      const float2 z2 = __half22float2(*reinterpret_cast<const __half2*>(&m.y));
      sc[2] = s2.x; sc[3] = s2.y; ze[2] = z2.x; ze[3] = z2.y;
    }
    bias = fmaf(qq.x, ze[0], bias);
    bias = fmaf(qq.y, ze[1], bias);
    bias = fmaf(qq.z, ze[2], bias);
    bias = fmaf(qq.w, ze[3], bias);
    const uint4 qs = split_hi_lo(qq.x * sc[0], qq.y * sc[1], qq.z * sc[2], qq.w * sc[3]);
#pragma unroll
    for (int tb = 0; tb < 2; ++tb) {
      const uint32_t r0 = kw + 4u * ((16 * tb + g) * RW), r1 = r0 + 4u * (8 * RW);
      const uint32_t a0 = v0 ? exact_codes(lds32(r0 + 4 * w0), sh0, mask2) : 0u;
      const uint32_t a1 = v0 ? exact_codes(lds32(r1 + 4 * w0), sh0, mask2) : 0u;
      const uint32_t a2 = v1 ? exact_codes(lds32(r0 + 4 * w1), sh1, mask2) : 0u;
      const uint32_t a3 = v1 ? exact_codes(lds32(r1 + 4 * w1), sh1, mask2) : 0u;
      mma16816(s[tb], a0, a1, a2, a3, qs.x, qs.y);
      mma16816(s[tb], a0, a1, a2, a3, qs.z, qs.w);
    }
  }
  // zero-point term: lanes (g, 0..3) hold parts of head g; S^T lane (g', q') needs heads 2q', 2q'+1
  bias += __shfl_xor_sync(0xffffffffu, bias, 1);
  bias += __shfl_xor_sync(0xffffffffu, bias, 2);
  const float be = __shfl_sync(0xffffffffu, bias, 8 * q), bo = __shfl_sync(0xffffffffu, bias, 8 * q + 4);
#pragma unroll
  for (int tb = 0; tb < 2; ++tb) {
    s[tb][0] += be;
    s[tb][1] += bo;
    s[tb][2] += be;
    s[tb][3] += bo;
  }
}

// PV of a zone-A tile with packed V (width vb).
template <int D>
__device__ __forceinline__ void tile_pv_packed(WarpAcc<D>& acc, uint32_t vcodes, uint32_t vmeta, int vb, int lane,
                                               const uint32_t (&pb)[2][2]) {
  const int g = lane >> 2, q = lane & 3;
  const int wpp = D * vb / 16;  // words per token pair
  const int per = 16 / vb;      // channels per word
  const uint32_t mask2 = vb == 8 ? 0x00ff00ffu : vb == 4 ? 0x000f000fu : 0x00030003u;
#pragma unroll
  for (int tb = 0; tb < 2; ++tb) {
    const int p0 = 8 * tb + q, p1 = p0 + 4;
#pragma unroll
    for (int grp = 0; grp < D / 32; ++grp) {
      const uint2 m0 = lds64(vmeta + 8 * (p0 * (D / 32) + grp));
      const uint2 m1 = lds64(vmeta + 8 * (p1 * (D / 32) + grp));
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int cm = 2 * grp + half;
        const int c0 = 16 * cm + g, c1 = c0 + 8;
        const uint32_t wa = vcodes + 4u * (p0 * wpp + c0 / per), wb = vcodes + 4u * (p0 * wpp + c1 / per);
        const uint32_t wc = vcodes + 4u * (p1 * wpp + c0 / per), wd = vcodes + 4u * (p1 * wpp + c1 / per);
        const int sh0 = vb * (c0 % per), sh1 = vb * (c1 % per);
        const uint32_t a0 = dequant_pair(lds32(wa), sh0, mask2, m0.x, m0.y);
        const uint32_t a1 = dequant_pair(lds32(wb), sh1, mask2, m0.x, m0.y);
        const uint32_t a2 = dequant_pair(lds32(wc), sh0, mask2, m1.x, m1.y);
        const uint32_t a3 = dequant_pair(lds32(wd), sh1, mask2, m1.x, m1.y);
        mma16816(acc.o[cm], a0, a1, a2, a3, pb[tb][0], pb[tb][1]);
      }
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

template <int D>
__global__ void __launch_bounds__(kDecWarps * 32) decode_kernel(DecodeParams P) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int head = blockIdx.y, split = blockIdx.x, n_split = gridDim.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = P.h_q / P.h_kv;
  const int b = head / P.h_kv, j = head % P.h_kv;
  const rdkv_head_plan hp = plan_heads(P.plan)[head];
  const int16_t* slot_ch = plan_slots(P.plan) + (int64_t)head * plan_header(P.plan)->slot_stride;

  // shared memory map
  KBDesc* kbd = reinterpret_cast<KBDesc*>(smem);                                   // [kMaxKB]
  float4* qv = reinterpret_cast<float4*>(smem + 256);                              // [kMaxKB][32]
  uint4* qfragc = reinterpret_cast<uint4*>(qv + kMaxKB * 32);                      // [D/16][32] hi, lo
  uint64_t* bars = reinterpret_cast<uint64_t*>(qfragc + (D / 16) * 32);           // [warps][kMaxInflight]
  int* ring_pos = reinterpret_cast<int*>(bars + kDecWarps * kMaxInflight);         // [warps][kMaxInflight]
  float* red = reinterpret_cast<float*>(ring_pos + kDecWarps * kMaxInflight);      // [warps][8][D + 2]
  unsigned char* ring = smem + decode_fixed_smem(D);
  __shared__ int nkb_s;

  // k-block descriptors of this head's K rows (each block inside one width segment)
  if (tid == 0) {
    int nkb = 0, wbase = 0, sbase = 0, meta = 0;
    for (int seg = 0; seg < 4; ++seg) {
      const int w = 16 >> seg, per = 32 / w;
      const int nslot = hp.k_words[seg] * per;
      for (int s0 = 0; s0 < nslot; s0 += 16) {
        KBDesc d;
        d.width = (int16_t)w;
        d.nrem = (int16_t)min(16, nslot - s0);
        d.word0 = wbase + s0 / per;
        d.meta0 = (w < 16 ? meta + s0 : 0) / 2;
        d.pad = sbase + s0;  // first slot of the block (for the query fragments)
        kbd[nkb++] = d;
      }
      wbase += hp.k_words[seg];
      sbase += nslot;
      if (w < 16) meta += nslot;
    }
    nkb_s = nkb;
  }
  __syncthreads();
  const int nkb = nkb_s;
  // query fragments: B[k = slot pair][n = head g] in slot order (zone A) and channel order (zone C)
  const int qbase = b * P.h_q + j * G;
  for (int i = tid; i < (nkb + D / 16) * 32; i += blockDim.x) {
    const int kb = i >> 5, ln = i & 31, g = ln >> 2, qq = ln & 3;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    const int offs[4] = {2 * qq, 2 * qq + 1, 2 * qq + 8, 2 * qq + 9};
    if (g < G) {
      for (int e = 0; e < 4; ++e) {
        int ch;
        if (kb < nkb) {
          const KBDesc d = kbd[kb];
          ch = offs[e] < d.nrem ? slot_ch[d.pad + offs[e]] : -1;
        } else {
          ch = 16 * (kb - nkb) + offs[e];
        }
        if (ch >= 0) v[e] = load_as_float(P.q, (int64_t)(qbase + g) * D + ch, P.dtype);
      }
    }
    if (kb < nkb) qv[kb * 32 + ln] = make_float4(v[0], v[1], v[2], v[3]);
    else qfragc[(kb - nkb) * 32 + ln] = split_hi_lo(v[0], v[1], v[2], v[3]);
  }
  if (lane == 0)
    for (int k = 0; k < kMaxInflight; ++k) mbar_init(&bars[warp * kMaxInflight + k], 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();

  // items of this head and of this split
  int cls_tiles[4], n_tiles = 0;
  for (int c = 0; c < 4; ++c) { cls_tiles[c] = hp.tiles[c]; n_tiles += hp.tiles[c]; }
  const int len_c = min(*P.len_dev, P.cap_c);
  const int n_items = n_tiles + ceil_div(len_c, kCRows);
  const int i0 = (int)((int64_t)n_items * split / n_split), i1 = (int)((int64_t)n_items * (split + 1) / n_split);
  const int my_n = i1 - i0 > warp ? ceil_div(i1 - i0 - warp, kDecWarps) : 0;

  WarpAcc<D> acc;
#pragma unroll
  for (int cm = 0; cm < D / 16; ++cm) acc.o[cm][0] = acc.o[cm][1] = acc.o[cm][2] = acc.o[cm][3] = 0.f;
  acc.m[0] = acc.m[1] = -INFINITY;
  acc.l[0] = acc.l[1] = 0.f;

  const float sl2 = 1.4426950408889634f / sqrtf((float)D);
  unsigned char* wring = ring + (int64_t)warp * P.ring_bytes;
  uint64_t* wbar = bars + warp * kMaxInflight;
  int* wpos = ring_pos + warp * kMaxInflight;
  uint32_t head_v = 0, tail_v = 0;     // virtual ring offsets (bytes)
  uint32_t vend[kMaxInflight];         // lane 0 only
  int issued = 0, done = 0;
  bool ok = true;

  auto item_info = [&](int it, int& cls, int& ti, int64_t& a_src, uint32_t& a_bytes, int& c_row) {
    if (it < n_tiles) {
      int t = it, c = 0;
      int64_t off = hp.a_off;
      while (t >= cls_tiles[c]) { off += (int64_t)cls_tiles[c] * hp.tile_bytes[c]; t -= cls_tiles[c]; ++c; }
      cls = c; ti = t; a_src = off + (int64_t)t * hp.tile_bytes[c]; a_bytes = hp.tile_bytes[c]; c_row = -1;
    } else {
      cls = -1; ti = 0; a_src = 0; a_bytes = 0; c_row = (it - n_tiles) * kCRows;
    }
  };
  auto stage_bytes = [&](int cls, uint32_t a_bytes) -> uint32_t {
    if (cls < 0) return 2u * kCRows * D * 2;
    return (uint32_t)align_up(a_bytes + (cls == 3 ? kTile * D * 2 : 0), 128);
  };

  while (done < my_n && ok) {
    // issue as many items as the ring and the slots allow (lane 0)
    if (lane == 0) {
      if (issued == done) head_v = tail_v = 0;  // empty ring: start at its beginning
      while (issued < my_n && issued - done < kMaxInflight) {
        const int it = i0 + warp + issued * kDecWarps;
        int cls, ti, c_row;
        int64_t a_src;
        uint32_t a_bytes;
        item_info(it, cls, ti, a_src, a_bytes, c_row);
        const uint32_t sz = stage_bytes(cls, a_bytes);
        uint32_t phys = head_v % (uint32_t)P.ring_bytes;
        uint32_t need = sz;
        if (phys + sz > (uint32_t)P.ring_bytes) { need += (uint32_t)P.ring_bytes - phys; phys = 0; }
        if (head_v - tail_v + need > (uint32_t)P.ring_bytes) break;
        head_v += need;
        const int slot = issued % kMaxInflight;
        vend[slot] = head_v;
        wpos[slot] = (int)phys;
        unsigned char* dst = wring + phys;
        uint64_t* bar = &wbar[slot];
        if (cls >= 0) {
          const uint32_t zb = cls == 3 ? (uint32_t)kTile * D * 2 : 0u;
          mbar_arrive_expect_tx(bar, a_bytes + zb);
          bulk_copy(dst, P.zone_a + a_src, a_bytes, bar);
          if (zb) bulk_copy(dst + a_bytes, P.zone_b + (hp.b_row + (int64_t)kTile * ti) * D, zb, bar);
        } else {
          const int rows = min(kCRows, len_c - c_row);
          const uint32_t bytes = (uint32_t)rows * D * 2;
          const int64_t src = ((int64_t)head * P.cap_c + c_row) * D;
          mbar_arrive_expect_tx(bar, 2 * bytes);
          bulk_copy(dst, P.zone_c_k + src, bytes, bar);
          bulk_copy(dst + kCRows * D * 2, P.zone_c_v + src, bytes, bar);
        }
        ++issued;
      }
    }
    __syncwarp();
    const int slot = done % kMaxInflight;
    const uint32_t parity = (uint32_t)(done / kMaxInflight) & 1u;
    const bool arrived = mbar_wait(&wbar[slot], parity);
    if (__any_sync(0xffffffffu, !arrived)) {
      ok = false;
      break;
    }
    const uint32_t st = smem_u32(wring + wpos[slot]);
    const int it = i0 + warp + done * kDecWarps;
    int cls, ti, c_row;
    int64_t a_src;
    uint32_t a_bytes;
    item_info(it, cls, ti, a_src, a_bytes, c_row);
    if (cls >= 0) {
      const int n_real = min(kTile, hp.n_v[cls] - kTile * ti);
      const uint32_t kmeta = st + 4u * kTile * hp.row_words;
      float s[2][4];
      tile_logits<D>(st, kmeta, hp.row_words, nkb, kbd, qv, lane, s);
      const int g = lane >> 2;
#pragma unroll
      for (int tb = 0; tb < 2; ++tb) {
        const bool va = 16 * tb + g < n_real, vb = 16 * tb + g + 8 < n_real;
        s[tb][0] = va ? s[tb][0] * sl2 : -INFINITY;
        s[tb][1] = va ? s[tb][1] * sl2 : -INFINITY;
        s[tb][2] = vb ? s[tb][2] * sl2 : -INFINITY;
        s[tb][3] = vb ? s[tb][3] * sl2 : -INFINITY;
      }
      uint32_t pb[2][2];
      softmax_update<D, 2>(acc, s, pb);
      const uint32_t vcodes = kmeta + 4u * hp.meta_slots;
      if (cls < 3) {
        const int vb = 2 << cls;
        tile_pv_packed<D>(acc, vcodes, vcodes + (uint32_t)(kTile * D * vb / 8), vb, lane, pb);
      } else {
        pv_fp16<D, 2>(acc, st + a_bytes, lane, pb);
      }
    } else {
      const int rows = min(kCRows, len_c - c_row);
      if (rows < kCRows) {  // clear the rows the copy did not fill (they meet p = 0 in the products)
        uint32_t* kz = reinterpret_cast<uint32_t*>(wring + wpos[slot]);
        for (int i = rows * D / 2 + lane; i < kCRows * D / 2; i += 32) {
          kz[i] = 0u;
          kz[kCRows * D / 2 + i] = 0u;
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
        mma16816(s[0], a0, a1, a2, a3, qf.z, qf.w);
      }
      const int g = lane >> 2;
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
    if (lane == 0) tail_v = vend[slot];
    ++done;
  }
  if (!ok) {
    if (lane == 0) atomicExch(P.error, (int)RDKV_ERR_TIMEOUT);
    // wait (bounded) for this warp's copies still in flight before leaving
    if (lane == 0)
      for (int k = done; k < issued; ++k)
        if (!mbar_wait(&wbar[k % kMaxInflight], (uint32_t)(k / kMaxInflight) & 1u)) break;
    __syncwarp();
  }

  // warp result -> shared memory: m, l per head; O per head and channel
  const int g = lane >> 2, q = lane & 3;
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
  // combine the warps; write this split's partial result for the G heads
  float* out = P.partial + ((int64_t)head * n_split + split) * G * (D + 2);
  for (int i = tid; i < G * (D + 2); i += blockDim.x) {
    const int h = i / (D + 2), c = i % (D + 2);
    float M = -INFINITY;
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, red[((int64_t)w * 8 + h) * (D + 2) + D]);
    float val = 0.f;
    if (c == D) {
      val = M;
    } else {
      for (int w = 0; w < kDecWarps; ++w) {
        const float mw = red[((int64_t)w * 8 + h) * (D + 2) + D];
        if (mw != -INFINITY) val += exp2f(mw - M) * red[((int64_t)w * 8 + h) * (D + 2) + c];
      }
    }
    out[i] = val;
  }
}

// out[b][h][c] = sum_s 2^(M_s - M) O_s[c] / sum_s 2^(M_s - M) L_s   (0 when no token)
__global__ void decode_merge_kernel(const float* __restrict__ partial, int n_split, int h_q, int h_kv, int D,
                                    float* __restrict__ out) {
  const int bh = blockIdx.x;  // b * h_q + h
  const int G = h_q / h_kv;
  const int b = bh / h_q, h = bh % h_q;
  const int head = b * h_kv + h / G, hl = h % G;
  const int c = threadIdx.x;
  const float* p = partial + (int64_t)head * n_split * G * (D + 2) + hl * (D + 2);
  float M = -INFINITY;
  for (int s = 0; s < n_split; ++s) M = fmaxf(M, p[(int64_t)s * G * (D + 2) + D]);
  float o = 0.f, l = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < n_split; ++s) {
      const float* ps = p + (int64_t)s * G * (D + 2);
      const float ms = ps[D];
      if (ms == -INFINITY) continue;
      const float f = exp2f(ms - M);
      o += f * ps[c];
      l += f * ps[D + 1];
    }
  }
  out[(int64_t)bh * D + c] = l > 0.f ? o / l : 0.f;
}

constexpr int64_t kDecodeSmemLimit = 227 * 1024 - 1024;  // per-block limit less room for static shared memory

struct DecodeGeom {
  int64_t max_item;
  int splits;
  int ring_bytes;
  size_t smem;
  size_t partial_bytes;
};

static DecodeGeom decode_geom(const rdkv_cache* c) {
  DecodeGeom g;
  const rdkv_shape& s = c->shape;
  const int D = s.head_dim, G = s.h_q / s.h_kv;
  const int n_heads = s.batch * s.h_kv;
  const int sms = num_sms();
  const int64_t items = ceil_div64(c->sizes.index_slots, kTile) + (int64_t)n_heads * ceil_div(c->cap_c, kCRows);
  const int64_t per_head = std::max<int64_t>(1, items / std::max(1, n_heads));
  int splits = ceil_div(2 * sms, n_heads);
  splits = (int)std::max<int64_t>(1, std::min<int64_t>(splits, ceil_div64(per_head, 2 * kDecWarps)));
  g.splits = std::min(splits, 1024);
  const int64_t max_item = std::max<int64_t>(align_up(c->sizes.max_tile_bytes + kTile * D * 2, 128), 2 * kCRows * D * 2);
  const int64_t fixed = decode_fixed_smem(D);
  const int64_t ring_cap = ((kDecodeSmemLimit - fixed) / kDecWarps) / 128 * 128;
  g.max_item = max_item;
  g.ring_bytes = (int)std::min<int64_t>(std::max<int64_t>(align_up(2 * max_item, 128), 24 * 1024), ring_cap);
  g.smem = (size_t)(fixed + (int64_t)kDecWarps * g.ring_bytes);
  g.partial_bytes = (size_t)align_up((int64_t)n_heads * g.splits * G * (D + 2) * 4, 256);
  return g;
}

rdkv_status check_cache_public(const rdkv_cache* c);

}  // namespace rdkv

using namespace rdkv;

extern "C" size_t rdkv_decode_workspace_bytes(const rdkv_cache* cache) {
  if (check_cache_public(cache) != RDKV_OK) return 0;
  return decode_geom(cache).partial_bytes + 256;
}

extern "C" rdkv_status rdkv_decode_attn(const rdkv_cache* cache, const void* q, float* out, void* ws, size_t ws_bytes,
                                        void* stream) {
  rdkv_status st = check_cache_public(cache);
  if (st != RDKV_OK) return st;
  RDKV_REQUIRE(q && out, RDKV_ERR_INVALID_ARG, "NULL pointer argument");
  const DecodeGeom geo = decode_geom(cache);
  RDKV_REQUIRE(ws && ws_bytes >= geo.partial_bytes + 256, RDKV_ERR_WORKSPACE, "decode workspace too small (%zu < %zu)",
               ws_bytes, geo.partial_bytes + 256);
  RDKV_REQUIRE(geo.ring_bytes >= geo.max_item, RDKV_ERR_UNSUPPORTED, "tiles too large for the decode ring (%lld B)",
               (long long)geo.max_item);
  const rdkv_shape& s = cache->shape;
  cudaStream_t cs = (cudaStream_t)stream;
  DecodeParams P;
  P.plan = cache->plan;
  P.zone_a = cache->zone_a;
  P.zone_b = cache->zone_b;
  P.zone_c_k = cache->zone_c_k;
  P.zone_c_v = cache->zone_c_v;
  P.q = q;
  P.error = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + geo.partial_bytes);
  P.partial = static_cast<float*>(ws);
  P.dtype = s.dtype;
  P.h_q = s.h_q;
  P.h_kv = s.h_kv;
  P.cap_c = cache->cap_c;
  P.len_dev = cache->len_dev;
  P.ring_bytes = geo.ring_bytes;
  RDKV_TRY_CUDA(cudaMemsetAsync(P.error, 0, 4, cs), "decode status reset");
  const dim3 grid(geo.splits, s.batch * s.h_kv);
  // the dynamic shared-memory limit is raised once per device and kernel (not while a graph is captured)
  static size_t smem_set[2][64] = {};
  int dev = 0;
  RDKV_TRY_CUDA(cudaGetDevice(&dev), "device");
  const int ki = s.head_dim == 128 ? 1 : 0;
  if (dev < 64 && geo.smem > smem_set[ki][dev]) {
    RDKV_TRY_CUDA(cudaFuncSetAttribute(ki ? (const void*)decode_kernel<128> : (const void*)decode_kernel<64>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDecodeSmemLimit),
                  "decode smem");
    smem_set[ki][dev] = (size_t)kDecodeSmemLimit;
  }
  if (ki)
    decode_kernel<128><<<grid, kDecWarps * 32, geo.smem, cs>>>(P);
  else
    decode_kernel<64><<<grid, kDecWarps * 32, geo.smem, cs>>>(P);
  RDKV_CHECK_LAUNCH("decode");
  decode_merge_kernel<<<s.batch * s.h_q, s.head_dim, 0, cs>>>(P.partial, geo.splits, s.h_q, s.h_kv, s.head_dim, out);
  RDKV_CHECK_LAUNCH("decode merge");
  return RDKV_OK;
}

extern "C" rdkv_status rdkv_decode_status(const rdkv_cache* cache, const void* ws, void* stream) {
  rdkv_status st = check_cache_public(cache);
  if (st != RDKV_OK) return st;
  RDKV_REQUIRE(ws, RDKV_ERR_INVALID_ARG, "NULL workspace");
  const DecodeGeom geo = decode_geom(cache);
  int32_t v = 0;
  RDKV_TRY_CUDA(cudaMemcpyAsync(&v, static_cast<const char*>(ws) + geo.partial_bytes, 4, cudaMemcpyDeviceToHost,
                                (cudaStream_t)stream),
                "status read");
  RDKV_TRY_CUDA(cudaStreamSynchronize((cudaStream_t)stream), "status sync");
  if (v != RDKV_OK) set_error("decode reported status %d (a bounded wait ran out)", v);
  return (rdkv_status)v;
}
