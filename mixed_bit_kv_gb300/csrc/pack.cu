// TriZone pack and append of RDKV (gist.science/ko/paper/2605.08317,
// section 2.3): zone A holds the kept K rows and the 2/4/8-bit V rows, packed
// and grouped by width; zone B holds the fp16 V rows of 16-bit tokens; zone C
// holds fp16 K and V rows of the recent window and of every decoded token.
//
// The quantiser is the asymmetric min-max formula of "Matematika KV Cache
// Compression" (aistudio.id, "Solusi 3") with fp16 scale and zero:
//   zero = fp16(min), scale = fp16(fl32(max - min) / (2^b - 1)),
//   code = clamp(rint((x - zero) / scale), 0, 2^b - 1)   (IEEE fp32, ties to even)
// V groups are 32 consecutive channels of a token; K groups are one channel
// over every kept prefix token of its (sequence, KV head), whose scale and zero
// are stored once in front of the head's tiles.  Layout rules: include/rdkv.h.
#include "common.cuh"

namespace rdkv {

__device__ __forceinline__ float to_float(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_float(float x) { return x; }

// Quantiser parameters of one group (scale 0: every code of the group is 0).
struct QParams {
  float zero, scale;
  uint16_t zero_h, scale_h;
};
__device__ __forceinline__ QParams qparams(float mn, float mx, int bits) {
  QParams p;
  const __half zh = __float2half_rn(mn);
  const __half sh = __float2half_rn(__fdiv_rn(mx - mn, (float)((1 << bits) - 1)));
  p.zero_h = __half_as_ushort(zh);
  p.scale_h = __half_as_ushort(sh);
  p.zero = __half2float(zh);
  p.scale = __half2float(sh);
  return p;
}
// The code clamp(rint((x - zero) / scale), 0, hi) (IEEE fp32 quotient, ties to even), with the
// division replaced by a multiply with r = fp32(1/scale): |d r - d/scale| stays below 2^-15 for the
// |d/scale| < 256 of a group's own values, so rint agrees with the IEEE quotient's unless d r is
// within 2^-12 of a half-integer; there the quotient is computed exactly.
__device__ __forceinline__ uint32_t qcode_rcp(float x, float zero, float scale, float rscale, float hi) {
  if (scale == 0.0f) return 0u;
  const float d = x - zero;
  float t = d * rscale;
  if (fabsf(t - floorf(t) - 0.5f) < 0.000244140625f) t = __fdiv_rn(d, scale);
  return (uint32_t)fminf(fmaxf(rintf(t), 0.0f), hi);
}

// Bit position of element e inside a word of b-bit elements: even elements in
// the low half-word, odd ones in the high half-word, LSB-first.
__device__ __forceinline__ int bit_off(int e, int b) { return 16 * (e & 1) + b * (e >> 1); }

// ---------------------------------------------------------------- index map
// One block per (sequence, KV head): the kept prefix tokens of each V width, in
// position order, at the class's slot range; pads -1.
__global__ void __launch_bounds__(1024) index_kernel(const uint8_t* __restrict__ bits_tok, int Np,
                                                      const void* __restrict__ plan, int32_t* __restrict__ index_map) {
  __shared__ int warp_tot[4][32];
  const int head = blockIdx.x;
  const rdkv_head_plan hp = plan_heads(plan)[head];
  const uint8_t* bt = bits_tok + (int64_t)head * Np;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
  const int chunk = ceil_div(Np, blockDim.x);
  const int t0 = min(Np, tid * chunk), t1 = min(Np, t0 + chunk);
  // the widths of this thread's tokens in position order: sixteen per load where the range is
  // 16-byte aligned, the rest one at a time
  auto visit = [&](auto&& f) {
    int t = t0;
    if (((uintptr_t)(bt + t) & 15) == 0) {
      for (; t + 16 <= t1; t += 16) {
        const uint4 v = *reinterpret_cast<const uint4*>(bt + t);
        const uint32_t vs[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int e = 0; e < 4; ++e) f(t + 4 * q + e, (int)((vs[q] >> (8 * e)) & 255u));
      }
    }
    for (; t < t1; ++t) f(t, (int)bt[t]);
  };
  int cnt[4] = {0, 0, 0, 0};
  visit([&](int, int b) {  // constant indices only: the counters stay in registers
    cnt[0] += b == 2;
    cnt[1] += b == 4;
    cnt[2] += b == 8;
    cnt[3] += b == 16;
  });
  int base[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    int x = cnt[c];
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[c][wid] = x;
    base[c] = x - cnt[c];
  }
  __syncthreads();
  if (wid == 0) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      int x = lane < nw ? warp_tot[c][lane] : 0;
      const int own = x;
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane < nw) warp_tot[c][lane] = x - own;
    }
  }
  __syncthreads();
  int start[4];
  int acc = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    base[c] += warp_tot[c][wid];
    start[c] = acc;
    acc += kTile * hp.tiles[c];
  }
  int32_t* out = index_map + hp.slot_off;
  int next[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) next[c] = start[c] + base[c];
  visit([&](int t, int b) {
    if (b == 2) out[next[0]++] = t;
    else if (b == 4) out[next[1]++] = t;
    else if (b == 8) out[next[2]++] = t;
    else if (b == 16) out[next[3]++] = t;
  });
#pragma unroll
  for (int c = 0; c < 4; ++c)
    for (int r = hp.n_v[c] + tid; r < kTile * hp.tiles[c]; r += blockDim.x) out[start[c] + r] = -1;
}

// ---------------------------------------------------------------- head K metadata
// One block per (sequence, KV head): fp16 scale and zero of every quantised K slot from the channel's
// minimum and maximum over the head's kept tokens (the allocation's channel statistics in the plan),
// in slot order from the first 8-bit slot; pads and the tail up to 16 bytes are zero.
__global__ void head_meta_kernel(const void* __restrict__ plan, const float2* __restrict__ kstat, int D,
                                 uint8_t* __restrict__ zone_a, const int32_t* __restrict__ a_pages) {
  const int head = blockIdx.x;
  const rdkv_plan_header* hdr = plan_header(plan);
  const rdkv_head_plan& hp = plan_heads(plan)[head];
  const int16_t* slot_ch = plan_slots(plan) + (int64_t)head * hdr->slot_stride;
  const int QS = hp.meta_slots, s_q0 = hp.k_slots - QS;
  const int sb4 = s_q0 + kKB * ceil_div(4 * hp.k_words[1], kKB);   // first 4-bit slot
  const int sb2 = sb4 + kKB * ceil_div(8 * hp.k_words[2], kKB);    // first 2-bit slot
  const int n_words = (int)(head_meta_bytes(QS) / 4);
  for (int m = threadIdx.x; m < n_words; m += blockDim.x) {
    uint32_t v = 0;
    const int s = s_q0 + m;
    const int c = m < QS ? slot_ch[s] : -1;
    if (c >= 0) {
      const int b = s < sb4 ? 8 : s < sb2 ? 4 : 2;
      const float2 st = kstat[(int64_t)head * D + c];
      const QParams p = qparams(st.x, st.y, b);
      v = (uint32_t)p.scale_h | ((uint32_t)p.zero_h << 16);
    }
    *reinterpret_cast<uint32_t*>(zone_a + zone_a_offset(a_pages, hp.a_off + 4 * (int64_t)m)) = v;
  }
}

// ---------------------------------------------------------------- tile pack
// One block (256 threads) per zone-A tile: stage the tile's K and V rows as floats, then the
// quantiser parameters of every K slot (from the head's channel statistics) and V group, then the K
// words and the V codes, then the V words.  A K word is built by the lane of its token from the
// codes of the word's slots (warps along words, lanes along tokens; K rows are padded to D + 1
// floats so that the 32 lanes read 32 banks, and the 32 lanes store 32 adjacent words of the
// word-major layout).  V codes go through shared memory as bytes; a V word is assembled from a
// pair's two code rows.
constexpr int kPackThreads = 256;
// Four consecutive elements as floats (8-byte load for fp16, 16-byte for fp32; the address is a
// multiple of four elements).
__device__ __forceinline__ float4 load4(const __half* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// One 32-bit K word of token row kr: word wg of the width-KB segment whose first slot is sbase.
// prm[s] = {zero, scale, 1/scale, channel (as int bits, -1 for a pad)} of slot s; codes of pad slots
// and of pad tokens (real false) are 0.
template <int KB>
__device__ __forceinline__ uint32_t k_word(int wg, int sbase, const float* kr, bool real, const float4* prm) {
  constexpr int per = 32 / KB, wpk = KB / 2;
  constexpr float hmax = (float)((1 << (KB < 16 ? KB : 1)) - 1);
  const int s0 = sbase + kKB * (wg / wpk), wi = wg % wpk;
  uint32_t word = 0;
#pragma unroll
  for (int e = 0; e < per; ++e) {
    const float4 pr = prm[s0 + k_slot_in_block(KB, wi, e)];
    const int c = __float_as_int(pr.w);
    if (c >= 0 && real) {
      const float x = kr[c];
      const uint32_t code = KB == 16 ? (uint32_t)half_bits(x) : qcode_rcp(x, pr.x, pr.y, pr.z, hmax);
      word |= code << bit_off(e, KB);
    }
  }
  return word;
}

// The V words of a tile of width VB < 16, straight from the staged rows Vf [32][D + 1]: word i is
// word wk of pair h of lane (g, q) of 16-token block tb, i = ((tb * 8 + g) * 4 + q) * 2 nw + h nw + wk
// (nw = D VB / 128); it holds entries kk = wk per + e (per = 16 / VB) of the lane's channel list,
// channel 16 (kk mod D/16) + 8 (kk div D/16) + g, at bit VB e for token 2p (low half) and 16 + VB e
// for token 2p + 1, p = 8 tb + q + 4 h.  vq [32][D/32] holds {zero, scale, 1/scale} per token and
// group; pad tokens (n_real and up) get code 0.
template <int VB, int D, typename At>
__device__ __forceinline__ void v_words(const float* Vf, const float4* vq, int n_real, int64_t vcode_b, At at) {
  constexpr int VP = D + 1, CM = D / 16, NG = D / kVGroup, NW = D * VB / 128, PER = 16 / VB;
  constexpr float hmax = (float)((1 << VB) - 1);
  for (int i = threadIdx.x; i < D * VB; i += kPackThreads) {
    const int wk = i % NW, rest = i / NW;
    const int h = rest & 1, q = (rest >> 1) & 3, g = (rest >> 3) & 7, tb = rest >> 6;
    const int r0 = 2 * (8 * tb + q + 4 * h), r1 = r0 + 1;
    uint32_t word = 0;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const int kk = wk * PER + e;
      const int c = 16 * (kk % CM) + 8 * (kk / CM) + g;
      const float4 p0 = vq[r0 * NG + c / kVGroup], p1 = vq[r1 * NG + c / kVGroup];
      const uint32_t c0 = r0 < n_real ? qcode_rcp(Vf[r0 * VP + c], p0.x, p0.y, p0.z, hmax) : 0u;
      const uint32_t c1 = r1 < n_real ? qcode_rcp(Vf[r1 * VP + c], p1.x, p1.y, p1.z, hmax) : 0u;
      word |= (c0 << (VB * e)) | (c1 << (16 + VB * e));
    }
    *reinterpret_cast<uint32_t*>(at(vcode_b + 4 * (int64_t)i)) = word;
  }
}

template <int D>
__host__ __device__ constexpr size_t pack_smem_bytes_of() {
  return (size_t)2 * kTile * (D + 1) * 4 + (size_t)(D + kSlotPad) * 16 + (size_t)kTile * (D / kVGroup) * 16 +
         (size_t)(D + kSlotPad) * 2 + 16;
}

template <typename T, int D>
__global__ void __launch_bounds__(kPackThreads) pack_tile_kernel(const T* __restrict__ k, const T* __restrict__ v,
                                                                  const void* __restrict__ plan,
                                                                  const float2* __restrict__ kstat,
                                                                  const int32_t* __restrict__ index_map,
                                                                  uint8_t* __restrict__ zone_a,
                                                                  uint16_t* __restrict__ zone_b, int N, int h_kv,
                                                                  const int32_t* __restrict__ a_pages,
                                                                  const int32_t* __restrict__ b_pages) {
  constexpr int NG = D / kVGroup;  // V groups of a token
  constexpr int KP = D + 1;        // floats of a staged K row
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const rdkv_plan_header* hdr = plan_header(plan);
  const rdkv_head_plan* heads = plan_heads(plan);
  const int64_t slot0 = (int64_t)blockIdx.x * kTile;
  // a grid sized from upper bounds (rdkv_zone_bounds) has blocks past the plan's last tile
  if (slot0 >= hdr->index_slots) return;
  // head whose slot range holds this tile
  int lo = 0, hi = hdr->n_heads - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (heads[mid].slot_off <= slot0) lo = mid; else hi = mid - 1;
  }
  const int head = lo;
  // the head record in shared memory: its arrays are read with run-time indices below
  __shared__ __align__(16) rdkv_head_plan hps;
  if (threadIdx.x < sizeof(rdkv_head_plan) / 4)
    reinterpret_cast<int32_t*>(&hps)[threadIdx.x] = reinterpret_cast<const int32_t*>(heads + head)[threadIdx.x];
  __syncthreads();
  const rdkv_head_plan& hp = hps;
  const int b = head / h_kv, j = head % h_kv;
  int ti = (int)((slot0 - hp.slot_off) / kTile), cls = 0;
  int64_t tile_off = hp.a_off + head_meta_bytes(hp.meta_slots);
  int64_t brow = hp.b_row;
  while (ti >= hp.tiles[cls]) {
    ti -= hp.tiles[cls];
    tile_off += (int64_t)hp.tiles[cls] * hp.tile_bytes[cls];
    ++cls;
  }
  tile_off += (int64_t)ti * hp.tile_bytes[cls];
  brow += (int64_t)kTile * ti;
  const int vbits = 2 << cls;
  const int n_real = min(kTile, hp.n_v[cls] - ti * kTile);
  const int RW = hp.row_words, KS = hp.k_slots;
  const int16_t* slot_ch = plan_slots(plan) + (int64_t)head * hdr->slot_stride;
  // width segments of the slots (16, 8, 4, 2 bits; each spans whole k-blocks) and of the words
  const int s16 = kKB * ceil_div(2 * hp.k_words[0], kKB);    // first 8-bit slot (the raw 16-bit slots come first)
  const int sb4 = s16 + kKB * ceil_div(4 * hp.k_words[1], kKB);  // first 4-bit slot
  const int sb2 = sb4 + kKB * ceil_div(8 * hp.k_words[2], kKB);  // first 2-bit slot
  const int w8 = hp.k_words[0], w4 = w8 + hp.k_words[1], w2 = w4 + hp.k_words[2];  // first word of each

  float* Kf = reinterpret_cast<float*>(smem_raw);               // [32][KP]
  float* Vf = Kf + kTile * KP;                                  // [32][KP]
  float4* kq = reinterpret_cast<float4*>(Vf + kTile * KP);      // [KS] zero, scale, 1/scale, channel
  float4* vq = kq + KS;                                         // [32][NG] zero, scale, 1/scale
  int16_t* sch = reinterpret_cast<int16_t*>(vq + kTile * NG);   // [KS] slot channels
  __shared__ int tok[kTile];
  const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
  if (tid < kTile) tok[tid] = index_map[slot0 + tid];
  for (int s = tid; s < KS; s += kPackThreads) sch[s] = slot_ch[s];
  __syncthreads();
  // the tile's K and V rows, four elements per load (rows are D contiguous elements, D % 4 == 0)
  for (int i = tid; i < kTile * D / 4; i += kPackThreads) {
    const int r = i / (D / 4), c = 4 * (i % (D / 4));
    const int t = tok[r];
    float4 kx = make_float4(0.f, 0.f, 0.f, 0.f), vx = kx;
    if (t >= 0) {
      const int64_t src = (((int64_t)b * N + t) * h_kv + j) * D + c;
      kx = load4(k + src);
      vx = load4(v + src);
    }
    float* kd = Kf + r * KP + c;
    kd[0] = kx.x;
    kd[1] = kx.y;
    kd[2] = kx.z;
    kd[3] = kx.w;
    float* vd = Vf + r * KP + c;
    vd[0] = vx.x;
    vd[1] = vx.y;
    vd[2] = vx.z;
    vd[3] = vx.w;
  }
  __syncthreads();

  // the tile's bytes in the zone-A pool (through the page table when zone A is paged; a tile may
  // cross a page boundary, so every store translates its own offset)
  auto at = [&](int64_t byte) { return zone_a + zone_a_offset(a_pages, tile_off + byte); };
  const int64_t vcode_b = 4 * kTile * RW;                      // V codes, then V metadata
  const int64_t vmeta_b = vcode_b + kTile * D * vbits / 8;
  // quantiser parameters: K slot s (quantised slots only: the head's channel statistics), then V
  // group (r, g) of the tile
  for (int i = tid; i < KS + (vbits < 16 ? kTile * NG : 0); i += kPackThreads) {
    if (i < KS) {
      const int s = i;
      const int c = sch[s];
      float z = 0.f, sc = 0.f, rs = 0.f;
      if (c >= 0 && s >= s16) {
        const int kb = s < sb4 ? 8 : s < sb2 ? 4 : 2;
        const float2 st = kstat[(int64_t)head * D + c];
        const QParams p = qparams(st.x, st.y, kb);
        z = p.zero;
        sc = p.scale;
        rs = sc != 0.f ? __frcp_rn(sc) : 0.f;
      }
      kq[s] = make_float4(z, sc, rs, __int_as_float(c));
    } else {
      const int vi = i - KS, r = vi / NG, g = vi % NG;
      const float* x = Vf + r * KP + g * kVGroup;
      uint16_t sc_h = 0, ze_h = 0;
      float z = 0.f, sc = 0.f, rs = 0.f;
      if (r < n_real) {
        // lanes start at different elements of their groups (groups are 32 floats apart, so in step
        // they would all hit one bank); the minimum and maximum do not depend on the order
        float mn = x[tx], mx = mn;
        for (int e = 1; e < kVGroup; ++e) {
          const float y = x[(tx + e) & (kVGroup - 1)];
          mn = fminf(mn, y);
          mx = fmaxf(mx, y);
        }
        const QParams p = qparams(mn, mx, vbits);
        sc_h = p.scale_h;
        ze_h = p.zero_h;
        z = p.zero;
        sc = p.scale;
        rs = sc != 0.f ? __frcp_rn(sc) : 0.f;
      }
      vq[vi] = make_float4(z, sc, rs, 0.f);
      // token pair p = 8 tb + q + 4 h: scales ordered (tb, q, h, group), zeros (tb, group, q, h), each
      // 32-bit word the pair's even token (low half) and odd token (high half)
      const int pp = r >> 1, tb = pp >> 3, q = pp & 3, h = (pp >> 2) & 1;
      *reinterpret_cast<uint16_t*>(at(vmeta_b + 2 * (2 * (((tb * 4 + q) * 2 + h) * NG + g) + (r & 1)))) = sc_h;
      *reinterpret_cast<uint16_t*>(at(vmeta_b + 2 * (2 * (16 * NG + ((tb * NG + g) * 4 + q) * 2 + h) + (r & 1)))) = ze_h;
    }
  }
  if (vbits == 16) {
    for (int i = tid; i < kTile * D; i += kPackThreads) {
      const int r = i / D;
      zone_b[zone_b_offset(b_pages, brow + r, D) + i % D] = r < n_real ? half_bits(Vf[r * KP + i % D]) : (uint16_t)0;
    }
  }
  __syncthreads();
  // K words: word w of token r at 32 w + 4 (r mod 8) + r / 8 (word-major; tokens r, r+8, r+16, r+24
  // of one word index side by side, so one 16-byte load gives a decode lane its four token rows).
  // The lane of token r builds the word from the codes of its slots (0 for pad slots and pad tokens).
  {
    const int r = tx;
    const bool real = r < n_real;
    const float* kr = Kf + r * KP;
    for (int w = ty; w < RW; w += kPackThreads / 32) {
      // the word's segment (a warp-uniform branch), then its codes with the width known
      const uint32_t word = w < w8   ? k_word<16>(w, 0, kr, real, kq)
                            : w < w4 ? k_word<8>(w - w8, s16, kr, real, kq)
                            : w < w2 ? k_word<4>(w - w4, sb4, kr, real, kq)
                                     : k_word<2>(w - w2, sb2, kr, real, kq);
      *reinterpret_cast<uint32_t*>(at(4 * (32 * w + 4 * (r % 8) + r / 8))) = word;
    }
  }
  // V words (codes taken straight from the staged rows), the width known at compile time
  if (vbits == 2) v_words<2, D>(Vf, vq, n_real, vcode_b, at);
  else if (vbits == 4) v_words<4, D>(Vf, vq, n_real, vcode_b, at);
  else if (vbits == 8) v_words<8, D>(Vf, vq, n_real, vcode_b, at);
}

template <typename T>
__global__ void window_kernel(const T* __restrict__ x, int N, int W, int h_kv, int D, int cap, int batch,
                              uint16_t* __restrict__ zc, const int32_t* __restrict__ pages, int stride) {
  const int64_t total = (int64_t)batch * h_kv * W * D;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(i % D);
    int64_t rest = i / D;
    const int r = (int)(rest % W);
    rest /= W;
    const int j = (int)(rest % h_kv);
    const int b = (int)(rest / h_kv);
    zc[zone_c_offset(pages, stride, cap, b * h_kv + j, r, D) + c] =
        half_bits(to_float(x[(((int64_t)b * N + (N - W) + r) * h_kv + j) * D + c]));
  }
}

// One block: every thread reads the row index before thread 0 advances it.
template <typename T>
__global__ void __launch_bounds__(1024) append_kernel(const T* __restrict__ kn, const T* __restrict__ vn, int64_t n,
                                                      int D, int cap, int32_t* len_dev, uint16_t* __restrict__ zk,
                                                      uint16_t* __restrict__ zv, const int32_t* __restrict__ pages,
                                                      int stride) {
  const int row = *len_dev;
  if (row < cap) {
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
      const int64_t dst = zone_c_offset(pages, stride, cap, (int)(i / D), row, D) + (i % D);
      zk[dst] = half_bits(to_float(kn[i]));
      zv[dst] = half_bits(to_float(vn[i]));
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && row < cap) *len_dev = row + 1;
}

__global__ void set_len_kernel(int32_t* len_dev, int value) { *len_dev = value; }

template <typename T, int D>
static rdkv_status launch_pack_tiles(const void* k, const void* v, const rdkv_cache* cache, int64_t n_tiles,
                                     cudaStream_t cs) {
  const size_t smem = pack_smem_bytes_of<D>();
  RDKV_TRY_CUDA(cudaFuncSetAttribute(pack_tile_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
                "pack smem");
  const PlanLayout L = plan_layout(cache->shape.batch, cache->shape.h_kv, D);
  const float2* kstat = reinterpret_cast<const float2*>(static_cast<const char*>(cache->plan) + L.kstat_off);
  pack_tile_kernel<T, D><<<(unsigned)n_tiles, kPackThreads, smem, cs>>>(
      static_cast<const T*>(k), static_cast<const T*>(v), cache->plan, kstat, cache->index_map, cache->zone_a,
      cache->zone_b, cache->shape.n_tokens, cache->shape.h_kv, cache->zone_a_pages, cache->zone_b_pages);
  RDKV_CHECK_LAUNCH("tile pack");
  return RDKV_OK;
}

static rdkv_status check_cache(const rdkv_cache* c) {
  RDKV_REQUIRE(c != nullptr, RDKV_ERR_INVALID_ARG, "cache is NULL");
  rdkv_status st = check_shape(&c->shape);
  if (st != RDKV_OK) return st;
  RDKV_REQUIRE(c->plan && c->zone_c_k && c->zone_c_v && c->len_dev, RDKV_ERR_INVALID_ARG,
               "cache plan, zone C or len_dev is NULL");
  RDKV_REQUIRE(c->sizes.zone_a_bytes == 0 || c->zone_a, RDKV_ERR_INVALID_ARG, "zone A is NULL");
  RDKV_REQUIRE(c->sizes.zone_b_rows == 0 || c->zone_b, RDKV_ERR_INVALID_ARG, "zone B is NULL");
  RDKV_REQUIRE(c->sizes.index_slots == 0 || c->index_map, RDKV_ERR_INVALID_ARG, "index map is NULL");
  RDKV_REQUIRE(c->cap_c >= c->shape.window && c->cap_c >= 0, RDKV_ERR_INVALID_ARG, "cap_c %d < window %d", c->cap_c,
               c->shape.window);
  RDKV_REQUIRE(c->len_c >= 0 && c->len_c <= c->cap_c, RDKV_ERR_INVALID_ARG, "len_c %d outside [0, cap_c]", c->len_c);
  RDKV_REQUIRE(c->zone_c_pages == nullptr || (int64_t)c->zone_c_page_stride * kZoneCPageRows >= c->cap_c,
               RDKV_ERR_INVALID_ARG, "page table stride %d too small for cap_c %d", c->zone_c_page_stride, c->cap_c);
  RDKV_REQUIRE(c->sizes.n_heads == c->shape.batch * c->shape.h_kv, RDKV_ERR_INVALID_ARG,
               "cache sizes do not belong to this shape (call rdkv_plan_sizes)");
  return RDKV_OK;
}

rdkv_status check_cache_public(const rdkv_cache* c) { return check_cache(c); }

}  // namespace rdkv

using namespace rdkv;

extern "C" rdkv_status rdkv_pack(rdkv_cache* cache, const void* k, const void* v, const uint8_t* bits_tok,
                                 const uint8_t* bits_chan, void* stream) {
  rdkv_status st = check_cache(cache);
  if (st != RDKV_OK) return st;
  const rdkv_shape& s = cache->shape;
  const int N = s.n_tokens, D = s.head_dim, W = s.window, Np = N - W;
  RDKV_REQUIRE(k && v && (Np == 0 || bits_tok) && bits_chan, RDKV_ERR_INVALID_ARG, "NULL pointer argument");
  RDKV_REQUIRE(reinterpret_cast<uintptr_t>(k) % 16 == 0 && reinterpret_cast<uintptr_t>(v) % 16 == 0,
               RDKV_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
  (void)bits_chan;  // the channel widths reach the pack through the plan's slot table
  cudaStream_t cs = (cudaStream_t)stream;
  const int n_heads = s.batch * s.h_kv;
  if (Np > 0 && cache->sizes.zone_a_bytes > 0) {
    const PlanLayout L = plan_layout(s.batch, s.h_kv, D);
    head_meta_kernel<<<n_heads, 128, 0, cs>>>(
        cache->plan, reinterpret_cast<const float2*>(static_cast<const char*>(cache->plan) + L.kstat_off), D,
        cache->zone_a, cache->zone_a_pages);
    RDKV_CHECK_LAUNCH("head K metadata");
  }
  if (Np > 0 && cache->sizes.index_slots > 0) {
    index_kernel<<<n_heads, 1024, 0, cs>>>(bits_tok, Np, cache->plan, cache->index_map);
    RDKV_CHECK_LAUNCH("index map");
    const int64_t n_tiles = cache->sizes.index_slots / kTile;
    RDKV_REQUIRE(n_tiles <= 0x7fffffff, RDKV_ERR_UNSUPPORTED, "too many tiles");
    rdkv_status pst;
    if (s.dtype == RDKV_F16)
      pst = D == 128 ? launch_pack_tiles<__half, 128>(k, v, cache, n_tiles, cs)
                     : launch_pack_tiles<__half, 64>(k, v, cache, n_tiles, cs);
    else
      pst = D == 128 ? launch_pack_tiles<float, 128>(k, v, cache, n_tiles, cs)
                     : launch_pack_tiles<float, 64>(k, v, cache, n_tiles, cs);
    if (pst != RDKV_OK) return pst;
  }
  if (W > 0) {
    const int64_t total = (int64_t)s.batch * s.h_kv * W * D;
    const unsigned grid = (unsigned)std::min<int64_t>(ceil_div64(total, 256), 4096);
    if (s.dtype == RDKV_F16) {
      window_kernel<__half><<<grid, 256, 0, cs>>>(static_cast<const __half*>(k), N, W, s.h_kv, D, cache->cap_c, s.batch,
                                                  cache->zone_c_k, cache->zone_c_pages, cache->zone_c_page_stride);
      window_kernel<__half><<<grid, 256, 0, cs>>>(static_cast<const __half*>(v), N, W, s.h_kv, D, cache->cap_c, s.batch,
                                                  cache->zone_c_v, cache->zone_c_pages, cache->zone_c_page_stride);
    } else {
      window_kernel<float><<<grid, 256, 0, cs>>>(static_cast<const float*>(k), N, W, s.h_kv, D, cache->cap_c, s.batch,
                                                 cache->zone_c_k, cache->zone_c_pages, cache->zone_c_page_stride);
      window_kernel<float><<<grid, 256, 0, cs>>>(static_cast<const float*>(v), N, W, s.h_kv, D, cache->cap_c, s.batch,
                                                 cache->zone_c_v, cache->zone_c_pages, cache->zone_c_page_stride);
    }
    RDKV_CHECK_LAUNCH("zone C window");
  }
  set_len_kernel<<<1, 1, 0, cs>>>(cache->len_dev, W);
  RDKV_CHECK_LAUNCH("zone C length");
  cache->len_c = W;
  return RDKV_OK;
}

// Upper bounds of the plan totals (per sequence, then times the batch).  Every kept token costs at
// least 2 of the sequence's B_V bits and a 16-bit one 16; each (head, class) segment is padded to
// whole tiles; a K row holds sum_c b_c bits plus at most one padding word per width segment, and the
// K widths of a sequence sum to at most B_K; a head's K metadata covers at most D + kSlotPad slots.
extern "C" rdkv_status rdkv_zone_bounds(const rdkv_shape* s, float avg_bits_v, float avg_bits_k, rdkv_sizes* out) {
  rdkv_status st = check_shape(s);
  if (st != RDKV_OK) return st;
  RDKV_REQUIRE(out, RDKV_ERR_INVALID_ARG, "NULL pointer argument");
  RDKV_REQUIRE(std::isfinite(avg_bits_v) && avg_bits_v >= 0 && std::isfinite(avg_bits_k) && avg_bits_k >= 0,
               RDKV_ERR_INVALID_ARG, "budgets must be finite and >= 0");
  const int64_t Np = s->n_tokens - s->window, H = s->h_kv, D = s->head_dim;
  const int64_t UV = H * Np;
  const int64_t BV = (int64_t)std::floor((double)avg_bits_v * (double)UV);
  const int64_t BK = std::min<int64_t>((int64_t)std::floor((double)avg_bits_k * (double)(H * D)), 16 * H * D);
  const int64_t kept = std::min<int64_t>(UV, BV / 2), n16 = std::min<int64_t>(UV, BV / 16);
  const int64_t tiles = ceil_div64(kept, kTile) + 4 * H;                 // sum over (head, class) of ceil(n / 32)
  const int64_t t_head = ceil_div64(std::min<int64_t>(Np, kept), kTile) + 4;  // tiles of one head
  const int64_t rw_sum = ceil_div64(BK, 32) + 4 * H;                      // row words of all heads
  const int64_t k_bytes = t_head * 4 * kTile * rw_sum + H * head_meta_bytes((int)(D + kSlotPad));
  const int64_t v_bytes = D * (std::min<int64_t>(BV, 8 * UV) / 8) + H * 4 * (kTile - 1) * D + tiles * 4 * D;
  const int64_t b = s->batch;
  out->zone_a_bytes = b * (k_bytes + v_bytes);
  out->zone_b_rows = b * kTile * (ceil_div64(n16, kTile) + H);
  out->index_slots = b * kTile * tiles;
  out->kept_tokens = b * kept;
  const int rw_max = (int)(D / 2 + 4);
  out->max_tile_bytes = tile_bytes_of(rw_max, (int)D, 8);
  out->max_stage_bytes = std::max<int64_t>(out->max_tile_bytes, tile_bytes_of(rw_max, (int)D, 16) + kTile * D * 2);
  out->status = RDKV_OK;
  out->n_heads = (int32_t)(b * H);
  for (int i = 0; i < RDKV_COST_HEADS; ++i) out->head_cost[i] = 0;
  return RDKV_OK;
}

extern "C" rdkv_status rdkv_append(rdkv_cache* cache, const void* k_new, const void* v_new, void* stream) {
  rdkv_status st = check_cache(cache);
  if (st != RDKV_OK) return st;
  RDKV_REQUIRE(k_new && v_new, RDKV_ERR_INVALID_ARG, "NULL pointer argument");
  RDKV_REQUIRE(cache->len_c < cache->cap_c, RDKV_ERR_CAPACITY, "zone C is full (%d rows)", cache->cap_c);
  const rdkv_shape& s = cache->shape;
  const int64_t n = (int64_t)s.batch * s.h_kv * s.head_dim;
  cudaStream_t cs = (cudaStream_t)stream;
  if (s.dtype == RDKV_F16)
    append_kernel<__half><<<1, 1024, 0, cs>>>(static_cast<const __half*>(k_new), static_cast<const __half*>(v_new), n,
                                               s.head_dim, cache->cap_c, cache->len_dev, cache->zone_c_k,
                                               cache->zone_c_v, cache->zone_c_pages, cache->zone_c_page_stride);
  else
    append_kernel<float><<<1, 1024, 0, cs>>>(static_cast<const float*>(k_new), static_cast<const float*>(v_new), n,
                                              s.head_dim, cache->cap_c, cache->len_dev, cache->zone_c_k,
                                              cache->zone_c_v, cache->zone_c_pages, cache->zone_c_page_stride);
  RDKV_CHECK_LAUNCH("append");
  cache->len_c += 1;
  return RDKV_OK;
}
