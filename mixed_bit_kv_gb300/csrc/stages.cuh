// Device stages of the allocation and the TriZone pack of RDKV
// (gist.science/ko/paper/2605.08317, sections 2.2 and 2.3), written once and
// called both by the one-kernel-per-stage path (allocate.cu, pack.cu) and by
// the persistent kernel that runs every stage in one launch (compress.cu), so
// the two paths do the same arithmetic in the same order.
//
// Each stage takes its work item (a block's share) and the shared memory it
// needs as arguments; the calling kernel decides how items map to blocks.  Data
// that one stage writes and a later stage of the same persistent launch reads
// (widths, partial sums, statistics, the plan, the index map) is never read
// through the read-only path.  In that launch every such address is written in
// one phase and read only in later ones, past a grid barrier, and no block
// touches it (or its 32-byte sector) before the write, so no SM's L1 can hold
// a stale copy; the loads that go through L2 (ld.global.cg) do so where it
// costs nothing.
#pragma once

#include "common.cuh"

namespace rdkv {

// ---------------------------------------------------------------- water-filling (section 2.2)
// Distortion drop per bit of each upgrade 0->2, 2->4, 4->8, 8->16, exact in fp32.
constexpr float kRdkvSlopes[4] = {0.375f, 0.09375f, 0.0146484375f, 255.0f / 524288.0f};
// All four breakpoints at the gain itself: a unit goes from 0 straight to 16 bits once its gain
// passes the level (the keep-or-drop selection of the eviction baselines).
constexpr float kKeepSlopes[4] = {1.0f, 1.0f, 1.0f, 1.0f};

struct Slopes {
  float s[4];
};
static inline Slopes slopes_of(const float (&a)[4]) { return Slopes{{a[0], a[1], a[2], a[3]}}; }

// Bits of upgrade k (0->2, 2->4, 4->8, 8->16) and the width after m upgrades.
__device__ __forceinline__ uint32_t step_bits(int k) { return k == 0 ? 2u : 1u << k; }
__device__ __forceinline__ uint8_t width_after(int m) { return m == 0 ? 0 : (uint8_t)(1 << m); }

__device__ __forceinline__ bool gain_valid(float g) { return g >= 0.0f && g <= 3.402823466e38f; }

// Bisection state of one instance: the bit pattern fixed so far and the bits bought strictly above
// the range it leaves open.
struct WfPick {
  uint32_t prefix;
  unsigned long long above;
};

// Level `level` histogram of one block's share of an instance: units u = x 256 + t, stepping by
// nx 256 (t the thread, 256 threads), of the gains g[0, n_units).  Every breakpoint fl32(g s_k)
// whose bits above this level's byte match `prefix` adds its upgrade's bits to bin (pattern >> shift)
// & 255 of h (256 words of shared memory); then, unless hist is null (a block that covers the whole
// instance keeps its bins in h), the block's bins go to hist[256] with one atomic each.  Invalid
// gains (NaN, infinite, negative) set *status at level 0 and buy nothing.
__device__ __forceinline__ void wf_hist_part(const float* g, int64_t n_units, Slopes sl, int level, uint32_t prefix,
                                             int x, int nx, uint32_t* h, unsigned long long* hist,
                                             int32_t* status) {
  for (int i = threadIdx.x; i < 256; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const int shift = 24 - 8 * level;
  bool bad = false;
  // lanes that hit the same bin add once, their count times the upgrade's bits (most gains of an
  // instance share a few bins at the first levels)
  for (int64_t u = (int64_t)x * blockDim.x + threadIdx.x; u < n_units; u += (int64_t)nx * blockDim.x) {
    const float gv = g[u];
    const bool valid = gain_valid(gv);
    bad |= !valid;
    const unsigned active = __activemask();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t p = level_bits(gv * sl.s[k]);
      const bool in = valid && (level == 0 || (p >> (shift + 8)) == (prefix >> (shift + 8)));
      const uint32_t bin = in ? (p >> shift) & 255u : 256u;
      const unsigned same = __match_any_sync(active, bin);
      if (in && (threadIdx.x & 31) == __ffs(same) - 1) atomicAdd(&h[bin], step_bits(k) * __popc(same));
    }
  }
  if (bad && level == 0 && status) atomicExch(status, (int32_t)RDKV_ERR_INVALID_ARG);
  __syncthreads();
  if (hist)
    for (int i = threadIdx.x; i < 256; i += blockDim.x)
      if (h[i]) atomicAdd(&hist[i], (unsigned long long)h[i]);
}

// The digit of level `level` (256 threads, thread t holding v = the level's bin t): the smallest d
// whose upper tail (bins > d) still fits the budget with the bits already above, i.e. the level is
// prefix | d << shift | (lower bits all ones).  Every thread returns the new state.  The tails are
// integer sums (exact in any order): suffix sums inside each warp by shuffles, then the totals of
// the warps above.  s: 9 64-bit words of shared memory, best: one int.
__device__ __forceinline__ WfPick wf_pick(unsigned long long v, int level, long long budget, WfPick cur,
                                          unsigned long long* s, int* best) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  unsigned long long x = v;  // sum over this warp's bins d' >= t
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_down_sync(0xffffffffu, x, o);
    if (lane + o < 32) x += y;
  }
  if (lane == 0) s[w] = x;
  if (t == 0) *best = 255;
  __syncthreads();
  for (int w2 = w + 1; w2 < 8; ++w2) x += s[w2];
  const unsigned long long tail = x - v;  // sum over d' > t
  if (cur.above + tail <= (unsigned long long)budget) atomicMin(best, t);
  __syncthreads();
  const int d = *best;
  if (t == d) s[8] = tail;
  __syncthreads();
  WfPick nxt;
  nxt.prefix = cur.prefix | ((uint32_t)d << (24 - 8 * level));
  nxt.above = cur.above + s[8];
  __syncthreads();  // s is free again
  return nxt;
}

// Widths of one block's share of an instance (units as in wf_hist_part) at the level lam: a unit
// takes every upgrade whose breakpoint is above it; invalid gains get 0 bits.
__device__ __forceinline__ void wf_assign_part(const float* g, int64_t n_units, Slopes sl, uint32_t lam, int x,
                                               int nx, uint8_t* bits) {
  for (int64_t u = (int64_t)x * blockDim.x + threadIdx.x; u < n_units; u += (int64_t)nx * blockDim.x) {
    const float gv = g[u];
    int m = 0;
    if (gain_valid(gv)) {
#pragma unroll
      for (int k = 0; k < 4; ++k) m += level_bits(gv * sl.s[k]) > lam ? 1 : 0;
    }
    bits[u] = width_after(m);
  }
}

// ---------------------------------------------------------------- K channel spread over kept tokens
// sigma_c (population std of K[kept tokens, j, c]) in two passes: chunk sums in fp32, combined in
// fp64 in a fixed order; then sums of squared deviations.
constexpr int kChanChunk = 256;
constexpr int kChanWarps = 8;  // warps of a chunk item (256 threads)
constexpr int kChanRows = 8;   // chunk partials combined per channel: chunks r, r + 8, ... in order, then rows 0..7

// Elements [c0, c0 + n) (n = 2 or 4, c0 a multiple of n) of one row as floats, one vector load.
__device__ __forceinline__ void load_run(const void* p, int64_t i, int dtype, int n, float (&x)[4]) {
  if (dtype == RDKV_F16) {
    const __half* h = static_cast<const __half*>(p) + i;
    if (n == 4) {
      const uint2 u = *reinterpret_cast<const uint2*>(h);
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
      x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
    } else {
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(h));
      x[0] = a.x; x[1] = a.y; x[2] = x[3] = 0.f;
    }
  } else {
    const float* f = static_cast<const float*>(p) + i;
    if (n == 4) {
      const float4 a = *reinterpret_cast<const float4*>(f);
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    } else {
      const float2 a = *reinterpret_cast<const float2*>(f);
      x[0] = a.x; x[1] = a.y; x[2] = x[3] = 0.f;
    }
  }
}

// Shared memory of a chunk item: per warp, per channel (D <= 128) the sum, minimum and maximum, and
// the warp's kept-token count.
struct ChanSmem {
  float wsum[kChanWarps][128];
  float wmin[kChanWarps][128];
  float wmax[kChanWarps][128];
  int wcnt[kChanWarps];
};

// Item (chunk, head) of a channel pass, 256 threads: lane l takes channels [l D/32, (l+1) D/32) of
// every token (one vector load; a warp reads whole rows), warp w the chunk's tokens t0 + w, t0 + w + 8,
// ... in order; the eight warps' sums are added in warp order (deterministic).  The first pass (no
// mean) also takes each channel's minimum and maximum over the kept tokens (pmin, pmax): the K
// quantiser's group of a channel is its head's kept tokens.
__device__ __forceinline__ void chan_pass_item(int chunk, int nchunk, int head, const void* k, const uint8_t* bits_tok,
                                               int dtype, int N, int h_kv, int D, int Np, const float* mean,
                                               float* part, int* part_cnt, float* pmin, float* pmax, ChanSmem& sm) {
  const int b = head / h_kv, j = head % h_kv;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int cpl = D / 32, c0 = lane * cpl;
  const int t0 = chunk * kChanChunk, t1 = min(Np, t0 + kChanChunk);
  const uint8_t* bt = bits_tok + (int64_t)head * Np;
  float m[4] = {0.f, 0.f, 0.f, 0.f};
  if (mean)
    for (int i = 0; i < cpl; ++i) m[i] = __ldcg(mean + head * D + c0 + i);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  float mn[4] = {INFINITY, INFINITY, INFINITY, INFINITY}, mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  int cnt = 0;
  const int64_t row = (int64_t)h_kv * D;
  const int64_t base = (((int64_t)b * N) * h_kv + j) * D + c0;
#pragma unroll 8
  for (int t = t0 + w; t < t1; t += kChanWarps) {
    const bool keep = __ldcg(bt + t) != 0;
    float x[4];
    load_run(k, base + (int64_t)t * row, dtype, cpl, x);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float d = x[i] - m[i];
      acc[i] += keep ? (mean ? d * d : x[i]) : 0.0f;
      mn[i] = keep ? fminf(mn[i], x[i]) : mn[i];
      mx[i] = keep ? fmaxf(mx[i], x[i]) : mx[i];
    }
    cnt += keep ? 1 : 0;
  }
  for (int i = 0; i < cpl; ++i) {
    sm.wsum[w][c0 + i] = acc[i];
    sm.wmin[w][c0 + i] = mn[i];
    sm.wmax[w][c0 + i] = mx[i];
  }
  if (lane == 0) sm.wcnt[w] = cnt;
  __syncthreads();
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float s = 0.0f, lo = INFINITY, hi = -INFINITY;
#pragma unroll
    for (int q = 0; q < kChanWarps; ++q) {
      s += sm.wsum[q][c];
      lo = fminf(lo, sm.wmin[q][c]);
      hi = fmaxf(hi, sm.wmax[q][c]);
    }
    part[((int64_t)head * nchunk + chunk) * D + c] = s;
    if (pmin) {
      pmin[((int64_t)head * nchunk + chunk) * D + c] = lo;
      pmax[((int64_t)head * nchunk + chunk) * D + c] = hi;
    }
  }
  if (threadIdx.x == 0 && part_cnt) {
    int n = 0;
    for (int q = 0; q < kChanWarps; ++q) n += sm.wcnt[q];
    part_cnt[head * nchunk + chunk] = n;
  }
  __syncthreads();  // sm is free again
}

struct ChanFinishSmem {
  double ssum[kChanRows][32];
  long long scnt[kChanRows][32];
  float smin[kChanRows][32], smax[kChanRows][32];
};

// Item (head, 32-channel slice) of the chunk combine, 256 threads: thread (r, l) takes the chunks
// r, r + 8, r + 16, ... of channel 32 slice + l, eight at a time (all loads in flight together): the
// e-th of each eight goes to fp64 accumulator e mod 4 (four independent chains), and the four
// accumulators are added in order at the end; row 0 then adds rows 1..7 in order.  The first call
// (mean_out set) also combines the chunks' minima and maxima into the head's K channel statistics
// kstat[head][c] = {min, max} over the kept tokens ({0, 0} when none is kept); the second writes
// sigma and the gain fl32(w_chan * sigma).
__device__ __forceinline__ void chan_finish_item(int head, int slice, const float* part, const int* part_cnt,
                                                 int nchunk, int D, float* mean_out, const float* w_chan,
                                                 float* sigma_out, float* g_out, const float* pmin, const float* pmax,
                                                 float2* kstat, ChanFinishSmem& sm) {
  const int l = threadIdx.x & 31, r = threadIdx.x >> 5, c = 32 * slice + l;
  constexpr int kBatch = 8;
  constexpr int kAcc = 4;
  double acc[kAcc];
#pragma unroll
  for (int e = 0; e < kAcc; ++e) acc[e] = 0.0;
  long long n = 0;
  float lo = INFINITY, hi = -INFINITY;
  const int64_t hb = (int64_t)head * nchunk;
  for (int i0 = r; i0 < nchunk; i0 += kChanRows * kBatch) {
    float ps[kBatch];
    int pc[kBatch];
#pragma unroll
    for (int e = 0; e < kBatch; ++e) {
      const int i = i0 + kChanRows * e;
      ps[e] = i < nchunk ? __ldcg(part + (hb + i) * D + c) : 0.f;
      pc[e] = i < nchunk ? __ldcg(part_cnt + hb + i) : 0;
    }
#pragma unroll
    for (int e = 0; e < kBatch; ++e) {
      if (i0 + kChanRows * e < nchunk) acc[e % kAcc] += (double)ps[e];
      n += pc[e];
    }
  }
  double s = acc[0];
#pragma unroll
  for (int e = 1; e < kAcc; ++e) s += acc[e];
  if (kstat) {
    constexpr int kMB = 8;
    for (int i0 = r; i0 < nchunk; i0 += kChanRows * kMB) {
      float pl[kMB], ph[kMB];
#pragma unroll
      for (int e = 0; e < kMB; ++e) {
        const int i = i0 + kChanRows * e;
        pl[e] = i < nchunk ? __ldcg(pmin + (hb + i) * D + c) : INFINITY;
        ph[e] = i < nchunk ? __ldcg(pmax + (hb + i) * D + c) : -INFINITY;
      }
#pragma unroll
      for (int e = 0; e < kMB; ++e) {
        lo = fminf(lo, pl[e]);
        hi = fmaxf(hi, ph[e]);
      }
    }
  }
  sm.ssum[r][l] = s;
  sm.scnt[r][l] = n;
  sm.smin[r][l] = lo;
  sm.smax[r][l] = hi;
  __syncthreads();
  if (r == 0) {
    for (int rr = 1; rr < kChanRows; ++rr) {
      s += sm.ssum[rr][l];
      n += sm.scnt[rr][l];
      lo = fminf(lo, sm.smin[rr][l]);
      hi = fmaxf(hi, sm.smax[rr][l]);
    }
    if (kstat) kstat[head * D + c] = n ? make_float2(lo, hi) : make_float2(0.f, 0.f);
    if (mean_out) {
      mean_out[head * D + c] = n ? (float)(s / (double)n) : 0.0f;
    } else {
      const float sig = n ? (float)sqrt(s / (double)n) : 0.0f;
      sigma_out[head * D + c] = sig;
      g_out[head * D + c] = __ldg(w_chan + head * D + c) * sig;
    }
  }
  __syncthreads();  // sm is free again
}

// ---------------------------------------------------------------- TriZone plan (section 2.3)
__device__ __forceinline__ int k_class_of(int b) { return b == 16 ? 0 : b == 8 ? 1 : b == 4 ? 2 : b == 2 ? 3 : 4; }

// The head record from its V class counts nv (widths 2, 4, 8, 16) and K class counts nk (widths
// 16, 8, 4, 2, 0): K segments of whole words per token whose slot ranges are whole k-blocks, the
// metadata slots of the quantised segments, tiles and tile sizes; offsets left at 0.  seg_base (may
// be null) receives the first slot of each K segment.
__device__ __forceinline__ rdkv_head_plan make_head_record(const int (&nv)[4], const int (&nk)[5], int D,
                                                           int* seg_base) {
  rdkv_head_plan hp;
  int words_total = 0, slots_total = 0, meta = 0;
  for (int i = 0; i < 4; ++i) {
    const int b = 16 >> i;
    hp.k_words[i] = ceil_div(nk[i] * b, 32);
    const int blocks = ceil_div(hp.k_words[i] * (32 / b), kKB);
    if (seg_base) seg_base[i] = slots_total;
    words_total += hp.k_words[i];
    slots_total += kKB * blocks;
    if (b < 16) meta += kKB * blocks;
  }
  for (int i = 0; i < 5; ++i) hp.n_k[i] = nk[i];
  hp.row_words = words_total;
  hp.k_slots = slots_total;
  hp.meta_slots = meta;
  int64_t a = head_meta_bytes(meta);
  for (int i = 0; i < 4; ++i) {
    hp.n_v[i] = nv[i];
    hp.tiles[i] = ceil_div(nv[i], kTile);
    hp.tile_bytes[i] = tile_bytes_of(words_total, D, 2 << i);  // V widths 2, 4, 8, 16
    a += (int64_t)hp.tiles[i] * hp.tile_bytes[i];
  }
  hp.a_bytes = a;
  hp.a_off = hp.b_row = hp.slot_off = 0;
  return hp;
}

// K classes of a head's channels: bcs[D] (shared memory) the widths; nk[5] (shared, zeroed by the
// caller before a barrier) receives the counts.  Then, once the caller has synchronised and set
// seg_base, plan_slot_table fills the slot table: the channel of rank r in its segment goes to
// element r mod (32/b) of word r div (32/b), in the k-block of that word at the slot
// k_slot_in_block gives; every other slot is -1.
__device__ __forceinline__ void plan_count_k(const uint8_t* bcs, int D, int* nk) {
  for (int c = threadIdx.x; c < D; c += blockDim.x) atomicAdd(&nk[k_class_of(bcs[c])], 1);
}
__device__ __forceinline__ void plan_slot_table(const uint8_t* bcs, int D, const int* seg_base, int16_t* slots) {
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    const int cls = k_class_of(bcs[c]);
    if (cls == 4) continue;
    int rank = 0;
    for (int c2 = 0; c2 < c; ++c2) rank += k_class_of(bcs[c2]) == cls;
    const int b = 16 >> cls, per = 32 / b, wpk = b / 2;
    const int wg = rank / per, e = rank % per;
    slots[seg_base[cls] + kKB * (wg / wpk) + k_slot_in_block(b, wg % wpk, e)] = (int16_t)c;
  }
}

// Per-class counts (widths 2, 4, 8, 16) of the widths bt[t0, t1) added to cnt; sixteen per load once
// the range is 16-byte aligned, eight loads in flight at a time.
__device__ __forceinline__ void count_classes(const uint8_t* bt, int t0, int t1, int stride_threads, int tid,
                                              int (&cnt)[4]) {
  auto count = [&](uint32_t b) {
    cnt[0] += b == 2;
    cnt[1] += b == 4;
    cnt[2] += b == 8;
    cnt[3] += b == 16;
  };
  const int lead = min(t1 - t0, (int)((16 - ((uintptr_t)(bt + t0) & 15)) & 15));
  for (int t = t0 + tid; t < t0 + lead; t += stride_threads) count(__ldcg(bt + t));
  const int n16 = (t1 - t0 - lead) / 16;
  const uint4* bt16 = reinterpret_cast<const uint4*>(bt + t0 + lead);
  constexpr int kLoads = 8;
  for (int i0 = tid; i0 < n16; i0 += kLoads * stride_threads) {
    uint4 w[kLoads];
#pragma unroll
    for (int e = 0; e < kLoads; ++e) {  // words past n16 read as width 0: no class
      const int i = i0 + e * stride_threads;
      w[e] = i < n16 ? __ldcg(bt16 + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int e = 0; e < kLoads; ++e) {
      const uint32_t ws[4] = {w[e].x, w[e].y, w[e].z, w[e].w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int f = 0; f < 4; ++f) count((ws[q] >> (8 * f)) & 255u);
    }
  }
  for (int t = t0 + lead + 16 * n16 + tid; t < t1; t += stride_threads) count(__ldcg(bt + t));
}

// Zone offsets of every head (in (sequence, KV head) order) and the plan header; one thread.
// status_v, status_k: the water-filling status words (an invalid gain makes the plan's status
// RDKV_ERR_INVALID_ARG).
__device__ __forceinline__ void plan_offsets_body(char* plan, int batch, int h_kv, int D, int slot_stride,
                                                  int64_t heads_off, int64_t slots_off, int64_t lambda_off,
                                                  int32_t sv, int32_t sk) {
  auto* hdr = reinterpret_cast<rdkv_plan_header*>(plan);
  auto* heads = reinterpret_cast<rdkv_head_plan*>(plan + heads_off);
  const int n_heads = batch * h_kv;
  int64_t a = 0, brow = 0, slot = 0, kept = 0, maxt = 0, maxs = 0;
  for (int i = 0; i < n_heads; ++i) {
    rdkv_head_plan& hp = heads[i];
    hp.a_off = a;
    hp.b_row = brow;
    hp.slot_off = slot;
    a += hp.a_bytes;
    brow += (int64_t)kTile * hp.tiles[3];
    int nt = 0;
    for (int c = 0; c < 4; ++c) {
      nt += hp.tiles[c];
      kept += hp.n_v[c];
      if (hp.tiles[c] && hp.tile_bytes[c] > maxt) maxt = hp.tile_bytes[c];
      const int64_t stage = hp.tile_bytes[c] + (c == 3 ? (int64_t)kTile * D * 2 : 0);
      if (hp.tiles[c] && stage > maxs) maxs = stage;
    }
    slot += (int64_t)kTile * nt;
  }
  int32_t s = RDKV_OK;
  if (sv != RDKV_OK) s = sv;
  if (sk != RDKV_OK) s = sk;
  hdr->status = s;
  hdr->n_heads = n_heads;
  hdr->batch = batch;
  hdr->h_kv = h_kv;
  hdr->head_dim = D;
  hdr->slot_stride = slot_stride;
  hdr->heads_off = heads_off;
  hdr->slots_off = slots_off;
  hdr->lambda_off = lambda_off;
  hdr->zone_a_bytes = a;
  hdr->zone_b_rows = brow;
  hdr->index_slots = slot;
  hdr->kept_tokens = kept;
  hdr->max_tile_bytes = maxt;
  hdr->max_stage_bytes = maxs;
}

// ---------------------------------------------------------------- pack (section 2.3)
// The quantiser is the asymmetric min-max formula of "Matematika KV Cache Compression" (aistudio.id,
// "Solusi 3") with fp16 scale and zero:
//   zero = fp16(min), scale = fp16(fl32(max - min) / (2^b - 1)),
//   code = clamp(rint((x - zero) / scale), 0, 2^b - 1)   (IEEE fp32, ties to even)
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

// Head K metadata: fp16 scale and zero of every quantised K slot from the channel's minimum and
// maximum over the head's kept tokens (the allocation's channel statistics in the plan), in slot
// order from the first 8-bit slot; pads and the tail up to 16 bytes are zero.
__device__ __forceinline__ void head_meta_body(int head, const void* plan, const float2* kstat, int D,
                                               uint8_t* zone_a, const int32_t* a_pages) {
  const rdkv_plan_header* hdr = plan_header(plan);
  const rdkv_head_plan* hpp = plan_heads(plan) + head;
  const int16_t* slot_ch = plan_slots(plan) + (int64_t)head * __ldcg(&hdr->slot_stride);
  const int QS = __ldcg(&hpp->meta_slots), s_q0 = __ldcg(&hpp->k_slots) - QS;
  const int sb4 = s_q0 + kKB * ceil_div(4 * __ldcg(&hpp->k_words[1]), kKB);  // first 4-bit slot
  const int sb2 = sb4 + kKB * ceil_div(8 * __ldcg(&hpp->k_words[2]), kKB);   // first 2-bit slot
  const int64_t a_off = __ldcg(reinterpret_cast<const long long*>(&hpp->a_off));
  const int n_words = (int)(head_meta_bytes(QS) / 4);
  for (int m = threadIdx.x; m < n_words; m += blockDim.x) {
    uint32_t v = 0;
    const int s = s_q0 + m;
    const int c = m < QS ? __ldcg(slot_ch + s) : -1;
    if (c >= 0) {
      const int b = s < sb4 ? 8 : s < sb2 ? 4 : 2;
      const float2 st = __ldcg(kstat + (int64_t)head * D + c);
      const QParams p = qparams(st.x, st.y, b);
      v = (uint32_t)p.scale_h | ((uint32_t)p.zero_h << 16);
    }
    *reinterpret_cast<uint32_t*>(zone_a + zone_a_offset(a_pages, a_off + 4 * (int64_t)m)) = v;
  }
}

// ---------------------------------------------------------------- tile pack
// One 256-thread item per zone-A tile: stage the tile's K and V rows as floats, then the quantiser
// parameters of every K slot (from the head's channel statistics) and V group, then the K words and
// the V codes, then the V words.  A K word is built by the lane of its token from the codes of the
// word's slots (warps along words, lanes along tokens; K rows are padded to D + 1 floats so that the
// 32 lanes read 32 banks, and the 32 lanes store 32 adjacent words of the word-major layout).
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

// Dynamic shared memory of a tile item: staged K and V rows, K slot and V group parameters, slot
// channels, then the head record and the tile's token list.
template <int D>
__host__ __device__ constexpr size_t pack_smem_bytes_of() {
  return (size_t)2 * kTile * (D + 1) * 4 + (size_t)(D + kSlotPad) * 16 + (size_t)kTile * (D / kVGroup) * 16 +
         (size_t)(D + kSlotPad) * 2 + 16 + sizeof(rdkv_head_plan) + kTile * 4;
}

// Tile item: the plan's slot range [32 tile, 32 tile + 32) of the index map.  smem_raw: the item's
// pack_smem_bytes_of<D>() bytes (16-byte aligned).
template <typename T, int D>
__device__ __forceinline__ void pack_tile_item(int64_t tile, const T* __restrict__ k, const T* __restrict__ v,
                                               const void* plan, const float2* kstat, const int32_t* index_map,
                                               uint8_t* __restrict__ zone_a, uint16_t* __restrict__ zone_b, int N,
                                               int h_kv, const int32_t* __restrict__ a_pages,
                                               const int32_t* __restrict__ b_pages, unsigned char* smem_raw) {
  constexpr int NG = D / kVGroup;  // V groups of a token
  constexpr int KP = D + 1;        // floats of a staged K row
  const rdkv_plan_header* hdr = plan_header(plan);
  const rdkv_head_plan* heads = plan_heads(plan);
  const int64_t slot0 = tile * kTile;
  // head whose slot range holds this tile
  int lo = 0, hi = hdr->n_heads - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (heads[mid].slot_off <= slot0) lo = mid; else hi = mid - 1;
  }
  const int head = lo;
  float* Kf = reinterpret_cast<float*>(smem_raw);               // [32][KP]
  float* Vf = Kf + kTile * KP;                                  // [32][KP]
  float4* kq = reinterpret_cast<float4*>(Vf + kTile * KP);      // [D + kSlotPad] zero, scale, 1/scale, channel
  float4* vq = kq + (D + kSlotPad);                             // [32][NG] zero, scale, 1/scale
  int16_t* sch = reinterpret_cast<int16_t*>(vq + kTile * NG);   // [D + kSlotPad] slot channels
  rdkv_head_plan* hps = reinterpret_cast<rdkv_head_plan*>(smem_raw + pack_smem_bytes_of<D>() -
                                                          sizeof(rdkv_head_plan) - kTile * 4);
  int* tok = reinterpret_cast<int*>(smem_raw + pack_smem_bytes_of<D>() - kTile * 4);
  // the head record in shared memory: its arrays are read with run-time indices below
  if (threadIdx.x < sizeof(rdkv_head_plan) / 4)
    reinterpret_cast<int32_t*>(hps)[threadIdx.x] = reinterpret_cast<const int32_t*>(heads + head)[threadIdx.x];
  __syncthreads();
  const rdkv_head_plan& hp = *hps;
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
  __syncthreads();  // the shared memory is free again
}

// Zone-C window: elements [i0, total) stepping by stride of the last W rows of x [B][N][H_kv][D]
// as fp16 rows [0, W) of each head's zone C.
template <typename T>
__device__ __forceinline__ void window_part(const T* x, int N, int W, int h_kv, int D, int cap, int batch,
                                            uint16_t* zc, const int32_t* pages, int stride, int64_t i0,
                                            int64_t step) {
  const int64_t total = (int64_t)batch * h_kv * W * D;
  for (int64_t i = i0; i < total; i += step) {
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

}  // namespace rdkv
