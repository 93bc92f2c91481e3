// Bit allocation of RDKV (gist.science/ko/paper/2605.08317, section 2.2):
// discrete reverse water-filling over widths {0, 2, 4, 8, 16} by Lagrangian
// relaxation, first for V tokens (step 2), then for K channels of the kept
// tokens (step 3); and the TriZone plan (section 2.3) that the pack and the
// decode read.
//
// Water level search.  The distortion of a unit at width b is g * 2^-b
// (section 2.1 objective), so upgrade k (b_k -> b_{k+1}) is worth it while
// g * s_k > lambda with s_k the distortion drop per bit.  The bits bought,
// H(lambda) = sum over breakpoints beta = fl32(g * s_k) > lambda of the
// upgrade's bits, only changes at breakpoints.  The smallest float32
// lambda >= 0 with H(lambda) <= B is found by bisecting the float32 bit
// pattern (monotone in value for non-negative floats) eight bits per level:
// each level histograms the breakpoints that share the prefix fixed so far,
// weighted by their bits, and keeps the smallest digit whose upper tail fits.
// Four levels give the exact minimum; the counts are integers, so the result
// does not depend on the order of the additions.
#include <algorithm>
#include <cmath>

#include "common.cuh"

namespace rdkv {

// Distortion drop per bit of each upgrade 0->2, 2->4, 4->8, 8->16, exact in fp32.
constexpr float kRdkvSlopes[4] = {0.375f, 0.09375f, 0.0146484375f, 255.0f / 524288.0f};
// All four breakpoints at the gain itself: a unit goes from 0 straight to 16 bits once its gain
// passes the level (the keep-or-drop selection of the eviction baselines).
constexpr float kKeepSlopes[4] = {1.0f, 1.0f, 1.0f, 1.0f};

struct Slopes {
  float s[4];
};
static Slopes slopes_of(const float (&a)[4]) { return Slopes{{a[0], a[1], a[2], a[3]}}; }
__constant__ uint32_t kStepBits[4] = {2, 2, 4, 8};
__constant__ uint8_t kWidth[5] = {0, 2, 4, 8, 16};

struct WfState {
  unsigned long long above;  // bits bought strictly above the fixed prefix range
  uint32_t prefix;           // bit pattern fixed so far
  int32_t pad;
};

static size_t wf_ws_bytes(int n_inst) {
  return (size_t)align_up((int64_t)n_inst * (256 * 8 + (int64_t)sizeof(WfState)) + 16, 256);
}

__global__ void wf_init(WfState* st, unsigned long long* hist, int n_inst, int32_t* status) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_inst * 256; i += gridDim.x * blockDim.x) hist[i] = 0;
  if (blockIdx.x == 0 && threadIdx.x < n_inst) st[threadIdx.x] = WfState{0ull, 0u, 0};
  if (blockIdx.x == 0 && threadIdx.x == 0 && status) *status = RDKV_OK;
}

__device__ __forceinline__ bool gain_valid(float g) { return g >= 0.0f && g <= 3.402823466e38f; }

// g of instance i starts at g + i * in_stride (units contiguous).
__global__ void wf_hist(const float* __restrict__ g, int64_t n_units, int64_t in_stride, Slopes sl, int level,
                        const WfState* __restrict__ st, unsigned long long* __restrict__ hist, int32_t* status) {
  __shared__ uint32_t h[256];
  const int inst = blockIdx.y;
  for (int i = threadIdx.x; i < 256; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const uint32_t prefix = st[inst].prefix;
  const int shift = 24 - 8 * level;
  const float* gi = g + (int64_t)inst * in_stride;
  bool bad = false;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < n_units; u += (int64_t)gridDim.x * blockDim.x) {
    const float gv = gi[u];
    if (!gain_valid(gv)) {
      bad = true;
      continue;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t p = level_bits(gv * sl.s[k]);
      if (level == 0 || (p >> (shift + 8)) == (prefix >> (shift + 8))) atomicAdd(&h[(p >> shift) & 255u], kStepBits[k]);
    }
  }
  if (bad && level == 0 && status) atomicExch(status, (int32_t)RDKV_ERR_INVALID_ARG);
  __syncthreads();
  for (int i = threadIdx.x; i < 256; i += blockDim.x)
    if (h[i]) atomicAdd(&hist[inst * 256 + i], (unsigned long long)h[i]);
}

// One block of 256 threads per instance: digit d is kept if the bits bought
// above x_d = prefix | d << shift | (lower bits all ones) fit the budget.
__global__ void wf_select(int level, long long budget, WfState* st, unsigned long long* hist) {
  __shared__ unsigned long long s[256];
  __shared__ int best;
  const int inst = blockIdx.x, t = threadIdx.x;
  const unsigned long long v = hist[inst * 256 + t];
  s[255 - t] = v;  // reversed so that an inclusive scan gives sums over d' >= t
  if (t == 0) best = 255;
  __syncthreads();
  for (int off = 1; off < 256; off <<= 1) {
    unsigned long long x = (255 - t >= off) ? s[255 - t - off] : 0ull;
    __syncthreads();
    s[255 - t] += x;
    __syncthreads();
  }
  const unsigned long long tail = s[255 - t] - v;  // sum over d' > t
  const unsigned long long above = st[inst].above;
  if (above + tail <= (unsigned long long)budget) atomicMin(&best, t);
  __syncthreads();
  const int d = best;
  if (t == d) {
    st[inst].prefix |= (uint32_t)d << (24 - 8 * level);
    st[inst].above = above + tail;
  }
  hist[inst * 256 + t] = 0;
}

__global__ void wf_assign(const float* __restrict__ g, int64_t n_units, int64_t in_stride, Slopes sl,
                          const WfState* __restrict__ st, uint8_t* __restrict__ bits, float* __restrict__ lambda_out) {
  const int inst = blockIdx.y;
  const uint32_t lam = st[inst].prefix;
  if (lambda_out && blockIdx.x == 0 && threadIdx.x == 0) lambda_out[inst] = __uint_as_float(lam);
  const float* gi = g + (int64_t)inst * in_stride;
  uint8_t* bi = bits + (int64_t)inst * n_units;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < n_units; u += (int64_t)gridDim.x * blockDim.x) {
    const float gv = gi[u];
    int m = 0;
    if (gain_valid(gv)) {
#pragma unroll
      for (int k = 0; k < 4; ++k) m += level_bits(gv * sl.s[k]) > lam ? 1 : 0;
    }
    bi[u] = kWidth[m];
  }
}

// One level per instance; instance i's n_units gains start at g + i * in_stride (in_stride = n_units
// when they are packed), its widths at bits + i * n_units.
static rdkv_status launch_waterfill(int n_inst, int64_t n_units, const float* g, float avg_bits, uint8_t* bits,
                                    float* lambda_out, int32_t* status_out, void* ws, cudaStream_t st,
                                    int64_t in_stride = -1, Slopes sl = slopes_of(kRdkvSlopes)) {
  if (in_stride < 0) in_stride = n_units;
  const long long budget = (long long)std::floor((double)avg_bits * (double)n_units);
  auto* state = reinterpret_cast<WfState*>(ws);
  auto* hist = reinterpret_cast<unsigned long long*>(static_cast<char*>(ws) + align_up((int64_t)n_inst * sizeof(WfState), 16));
  int32_t* status = status_out;
  wf_init<<<4, 256, 0, st>>>(state, hist, n_inst, status);
  RDKV_CHECK_LAUNCH("waterfill init");
  const int per_inst = (int)std::min<int64_t>(std::max<int64_t>(ceil_div64(n_units, 256 * 16), 1), 512);
  for (int level = 0; level < 4; ++level) {
    wf_hist<<<dim3(per_inst, n_inst), 256, 0, st>>>(g, n_units, in_stride, sl, level, state, hist, status);
    RDKV_CHECK_LAUNCH("waterfill histogram");
    wf_select<<<n_inst, 256, 0, st>>>(level, budget, state, hist);
    RDKV_CHECK_LAUNCH("waterfill select");
  }
  wf_assign<<<dim3(per_inst, n_inst), 256, 0, st>>>(g, n_units, in_stride, sl, state, bits, lambda_out);
  RDKV_CHECK_LAUNCH("waterfill assign");
  return RDKV_OK;
}

// Keep-or-drop at a given level: 16 bits for units whose weight exceeds tau, else 0 (invalid
// weights are flagged and dropped).
__global__ void keep_above_kernel(const float* __restrict__ w, int64_t n_units, int64_t in_stride, float tau,
                                  uint8_t* __restrict__ bits, float* __restrict__ lambda_out, int32_t* status) {
  const int inst = blockIdx.y;
  if (lambda_out && blockIdx.x == 0 && threadIdx.x == 0) lambda_out[inst] = tau;
  const float* wi = w + (int64_t)inst * in_stride;
  uint8_t* bi = bits + (int64_t)inst * n_units;
  bool bad = false;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < n_units; u += (int64_t)gridDim.x * blockDim.x) {
    const float x = wi[u];
    if (!gain_valid(x)) bad = true;
    bi[u] = (gain_valid(x) && x > tau) ? 16 : 0;
  }
  if (bad && status) atomicExch(status, (int32_t)RDKV_ERR_INVALID_ARG);
}

// Widths at given water levels (one per instance): the Lagrangian choice of wf_assign with the
// level read from levels[inst] instead of found by the bisection; invalid gains are flagged.
__global__ void assign_at_level_kernel(const float* __restrict__ g, int64_t n_units, int64_t in_stride, Slopes sl,
                                       const float* __restrict__ levels, uint8_t* __restrict__ bits,
                                       float* __restrict__ lambda_out, int32_t* status) {
  const int inst = blockIdx.y;
  const float lv = levels[inst];
  const uint32_t lam = level_bits(lv);
  if (lambda_out && blockIdx.x == 0 && threadIdx.x == 0) lambda_out[inst] = lv;
  const float* gi = g + (int64_t)inst * in_stride;
  uint8_t* bi = bits + (int64_t)inst * n_units;
  bool bad = false;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < n_units; u += (int64_t)gridDim.x * blockDim.x) {
    const float gv = gi[u];
    int m = 0;
    if (gain_valid(gv)) {
#pragma unroll
      for (int k = 0; k < 4; ++k) m += level_bits(gv * sl.s[k]) > lam ? 1 : 0;
    } else {
      bad = true;
    }
    bi[u] = kWidth[m];
  }
  if (bad && status) atomicExch(status, (int32_t)RDKV_ERR_INVALID_ARG);
}

// Allocation modes beyond the public ones: widths at given levels, pooled or per head.
constexpr int kAllocLevelsPooled = 100;
constexpr int kAllocLevelsPerHead = 101;

__global__ void fill_u8_kernel(uint8_t* __restrict__ p, int64_t n, uint8_t v) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) p[i] = v;
}

// ---------------------------------------------------------------- K channel spread over kept tokens
// sigma_c (population std of K[kept tokens, j, c]) in two passes: chunk sums
// in fp32, combined in fp64 in a fixed order; then sums of squared deviations.
constexpr int kChanChunk = 256;

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

// Block (chunk, head), 256 threads: lane l takes channels [l D/32, (l+1) D/32) of every token (one
// vector load; a warp reads whole rows), warp w the chunk's tokens t0 + w, t0 + w + 8, ... in order;
// the eight warps' sums are added in warp order (deterministic).  The first pass (no mean) also
// takes each channel's minimum and maximum over the kept tokens (pmin, pmax): the K quantiser's
// group of a channel is its head's kept tokens.
constexpr int kChanWarps = 8;
__global__ void __launch_bounds__(32 * kChanWarps) chan_pass(const void* __restrict__ k,
                                                             const uint8_t* __restrict__ bits_tok, int dtype, int N,
                                                             int h_kv, int D, int Np, const float* __restrict__ mean,
                                                             float* __restrict__ part, int* __restrict__ part_cnt,
                                                             float* __restrict__ pmin, float* __restrict__ pmax) {
  __shared__ float wsum[kChanWarps][128];
  __shared__ float wmin[kChanWarps][128], wmax[kChanWarps][128];
  __shared__ int wcnt[kChanWarps];
  const int head = blockIdx.y;  // b * h_kv + j
  const int b = head / h_kv, j = head % h_kv;
  const int chunk = blockIdx.x, nchunk = gridDim.x;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int cpl = D / 32, c0 = lane * cpl;
  const int t0 = chunk * kChanChunk, t1 = min(Np, t0 + kChanChunk);
  const uint8_t* bt = bits_tok + (int64_t)head * Np;
  float m[4] = {0.f, 0.f, 0.f, 0.f};
  if (mean)
    for (int i = 0; i < cpl; ++i) m[i] = mean[head * D + c0 + i];
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  float mn[4] = {INFINITY, INFINITY, INFINITY, INFINITY}, mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  int cnt = 0;
  const int64_t row = (int64_t)h_kv * D;
  const int64_t base = (((int64_t)b * N) * h_kv + j) * D + c0;
#pragma unroll 4
  for (int t = t0 + w; t < t1; t += kChanWarps) {
    const bool keep = bt[t] != 0;
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
    wsum[w][c0 + i] = acc[i];
    wmin[w][c0 + i] = mn[i];
    wmax[w][c0 + i] = mx[i];
  }
  if (lane == 0) wcnt[w] = cnt;
  __syncthreads();
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float s = 0.0f, lo = INFINITY, hi = -INFINITY;
#pragma unroll
    for (int q = 0; q < kChanWarps; ++q) {
      s += wsum[q][c];
      lo = fminf(lo, wmin[q][c]);
      hi = fmaxf(hi, wmax[q][c]);
    }
    part[((int64_t)head * nchunk + chunk) * D + c] = s;
    if (pmin) {
      pmin[((int64_t)head * nchunk + chunk) * D + c] = lo;
      pmax[((int64_t)head * nchunk + chunk) * D + c] = hi;
    }
  }
  if (threadIdx.x == 0 && part_cnt) {
    int n = 0;
    for (int q = 0; q < kChanWarps; ++q) n += wcnt[q];
    part_cnt[head * nchunk + chunk] = n;
  }
}

// The first call (mean_out set) also combines the chunks' minima and maxima into the head's K
// channel statistics kstat [head][c] = {min, max} over the kept tokens ({0, 0} when none is kept).
__global__ void chan_finish(const float* __restrict__ part, const int* __restrict__ part_cnt, int nchunk, int D,
                            float* __restrict__ mean_out, const float* __restrict__ w_chan,
                            float* __restrict__ sigma_out, float* __restrict__ g_out, const float* __restrict__ pmin,
                            const float* __restrict__ pmax, float2* __restrict__ kstat) {
  // thread (r, c) sums the chunks r, r + R, r + 2R, ... of channel c; the R sums are combined in a
  // fixed order (deterministic)
  __shared__ double ssum[1024];
  __shared__ long long scnt[1024];
  __shared__ float smin[1024], smax[1024];
  const int head = blockIdx.x, c = threadIdx.x % D, r = threadIdx.x / D, R = blockDim.x / D;
  double s = 0.0;
  long long n = 0;
  float lo = INFINITY, hi = -INFINITY;
  for (int i = r; i < nchunk; i += R) {
    s += (double)part[((int64_t)head * nchunk + i) * D + c];
    n += part_cnt[head * nchunk + i];
    if (kstat) {
      lo = fminf(lo, pmin[((int64_t)head * nchunk + i) * D + c]);
      hi = fmaxf(hi, pmax[((int64_t)head * nchunk + i) * D + c]);
    }
  }
  ssum[threadIdx.x] = s;
  scnt[threadIdx.x] = n;
  smin[threadIdx.x] = lo;
  smax[threadIdx.x] = hi;
  __syncthreads();
  if (r != 0) return;
  for (int rr = 1; rr < R; ++rr) {
    s += ssum[rr * D + c];
    n += scnt[rr * D + c];
    lo = fminf(lo, smin[rr * D + c]);
    hi = fmaxf(hi, smax[rr * D + c]);
  }
  if (kstat) kstat[head * D + c] = n ? make_float2(lo, hi) : make_float2(0.f, 0.f);
  if (mean_out) {
    mean_out[head * D + c] = n ? (float)(s / (double)n) : 0.0f;
  } else {
    const float sig = n ? (float)sqrt(s / (double)n) : 0.0f;
    sigma_out[head * D + c] = sig;
    g_out[head * D + c] = w_chan[head * D + c] * sig;
  }
}

// ---------------------------------------------------------------- plan
__global__ void plan_heads_kernel(const uint8_t* __restrict__ bits_tok, const uint8_t* __restrict__ bits_chan, int Np,
                                  int D, char* plan, int64_t heads_off, int64_t slots_off, int slot_stride) {
  const int head = blockIdx.x;
  __shared__ int nv[4], nk[5];
  __shared__ int seg_base[4];
  __shared__ uint8_t bcs[256];  // this head's channel widths (D <= 256)
  if (threadIdx.x < 4) nv[threadIdx.x] = 0;
  if (threadIdx.x < 5) nk[threadIdx.x] = 0;
  int16_t* slots = reinterpret_cast<int16_t*>(plan + slots_off) + (int64_t)head * slot_stride;
  for (int i = threadIdx.x; i < slot_stride; i += blockDim.x) slots[i] = -1;
  const uint8_t* bc = bits_chan + (int64_t)head * D;
  for (int c = threadIdx.x; c < D; c += blockDim.x) bcs[c] = bc[c];
  __syncthreads();
  int cnt[4] = {0, 0, 0, 0};
  auto count = [&](uint32_t b) {
    cnt[0] += b == 2;
    cnt[1] += b == 4;
    cnt[2] += b == 8;
    cnt[3] += b == 16;
  };
  const uint8_t* bt = bits_tok + (int64_t)head * Np;
  // widths of the head's tokens, sixteen per load once the row is 16-byte aligned (independent loads,
  // all in flight together); the counts do not depend on the order
  const int lead = min(Np, (int)((16 - ((uintptr_t)bt & 15)) & 15));
  for (int t = threadIdx.x; t < lead; t += blockDim.x) count(bt[t]);
  const int n16 = (Np - lead) / 16;
  const uint4* bt16 = reinterpret_cast<const uint4*>(bt + lead);
  for (int i = threadIdx.x; i < n16; i += blockDim.x) {
    const uint4 w = bt16[i];
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int e = 0; e < 4; ++e) count((ws[q] >> (8 * e)) & 255u);
  }
  for (int t = lead + 16 * n16 + threadIdx.x; t < Np; t += blockDim.x) count(bt[t]);
#pragma unroll
  for (int i = 0; i < 4; ++i) atomicAdd(&nv[i], cnt[i]);
  auto kclass = [](int b) { return b == 16 ? 0 : b == 8 ? 1 : b == 4 ? 2 : b == 2 ? 3 : 4; };
  for (int c = threadIdx.x; c < D; c += blockDim.x) atomicAdd(&nk[kclass(bcs[c])], 1);
  __syncthreads();
  if (threadIdx.x == 0) {
    // K segments of widths 16, 8, 4, 2: whole words per token, slot ranges of whole k-blocks
    rdkv_head_plan hp;
    int words_total = 0, slots_total = 0, meta = 0;
    for (int i = 0; i < 4; ++i) {
      const int b = 16 >> i;
      hp.k_words[i] = ceil_div(nk[i] * b, 32);
      const int blocks = ceil_div(hp.k_words[i] * (32 / b), kKB);
      seg_base[i] = slots_total;
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
    reinterpret_cast<rdkv_head_plan*>(plan + heads_off)[head] = hp;
  }
  __syncthreads();
  // the channel of rank r in its segment: element r mod (32/b) of word r div (32/b), in the k-block
  // of that word at the slot k_slot_in_block gives
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    const int cls = kclass(bcs[c]);
    if (cls == 4) continue;
    int rank = 0;
    for (int c2 = 0; c2 < c; ++c2) rank += kclass(bcs[c2]) == cls;
    const int b = 16 >> cls, per = 32 / b, wpk = b / 2;
    const int wg = rank / per, e = rank % per;
    slots[seg_base[cls] + kKB * (wg / wpk) + k_slot_in_block(b, wg % wpk, e)] = (int16_t)c;
  }
}

__global__ void plan_offsets_kernel(char* plan, int batch, int h_kv, int D, int slot_stride, int64_t heads_off,
                                    int64_t slots_off, int64_t lambda_off, const int32_t* status_v,
                                    const int32_t* status_k) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
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
  if (*status_v != RDKV_OK) s = *status_v;
  if (*status_k != RDKV_OK) s = *status_k;
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

// ---------------------------------------------------------------- shape checks shared with the other calls
rdkv_status check_shape(const rdkv_shape* s) {
  RDKV_REQUIRE(s != nullptr, RDKV_ERR_INVALID_ARG, "shape is NULL");
  RDKV_REQUIRE(s->batch >= 1 && s->n_tokens >= 1 && s->h_q >= 1 && s->h_kv >= 1, RDKV_ERR_INVALID_ARG,
               "shape sizes must be positive (batch=%d n_tokens=%d h_q=%d h_kv=%d)", s->batch, s->n_tokens, s->h_q,
               s->h_kv);
  RDKV_REQUIRE(s->window >= 0 && s->window <= s->n_tokens, RDKV_ERR_INVALID_ARG, "window %d outside [0, n_tokens=%d]",
               s->window, s->n_tokens);
  RDKV_REQUIRE(s->h_q % s->h_kv == 0, RDKV_ERR_INVALID_ARG, "h_q=%d is not a multiple of h_kv=%d", s->h_q, s->h_kv);
  RDKV_REQUIRE(s->h_q / s->h_kv <= 8, RDKV_ERR_UNSUPPORTED, "group size %d > 8", s->h_q / s->h_kv);
  RDKV_REQUIRE(s->head_dim == 64 || s->head_dim == 128, RDKV_ERR_UNSUPPORTED, "head_dim %d not in {64, 128}",
               s->head_dim);
  RDKV_REQUIRE(s->dtype == RDKV_F16 || s->dtype == RDKV_F32, RDKV_ERR_UNSUPPORTED, "dtype %d", s->dtype);
  return RDKV_OK;
}

}  // namespace rdkv

using namespace rdkv;

extern "C" size_t rdkv_waterfill_workspace_bytes(int32_t n_inst, int64_t n_units) {
  (void)n_units;
  return n_inst > 0 ? wf_ws_bytes(n_inst) + 256 : 0;
}

extern "C" rdkv_status rdkv_waterfill(int32_t n_inst, int64_t n_units, const float* g, float avg_bits, uint8_t* bits,
                                      float* lambda_out, int32_t* status_out, void* ws, size_t ws_bytes,
                                      void* stream) {
  RDKV_REQUIRE(n_inst >= 1 && n_inst <= 65535 && n_units >= 0, RDKV_ERR_INVALID_ARG, "n_inst=%d n_units=%lld", n_inst,
               (long long)n_units);
  RDKV_REQUIRE(std::isfinite(avg_bits) && avg_bits >= 0.0f, RDKV_ERR_INVALID_ARG, "avg_bits %f", (double)avg_bits);
  RDKV_REQUIRE(n_units == 0 || (g && bits), RDKV_ERR_INVALID_ARG, "g or bits is NULL");
  RDKV_REQUIRE(ws && ws_bytes >= rdkv_waterfill_workspace_bytes(n_inst, n_units), RDKV_ERR_WORKSPACE,
               "waterfill workspace too small (%zu < %zu)", ws_bytes, rdkv_waterfill_workspace_bytes(n_inst, n_units));
  int32_t* status = status_out ? status_out
                               : reinterpret_cast<int32_t*>(static_cast<char*>(ws) + wf_ws_bytes(n_inst));
  if (n_units == 0) {
    return RDKV_OK;
  }
  return launch_waterfill(n_inst, n_units, g, avg_bits, bits, lambda_out, status, ws, (cudaStream_t)stream);
}

extern "C" size_t rdkv_plan_bytes(const rdkv_shape* s) {
  if (!s || s->batch < 1 || s->h_kv < 1) return 0;
  return (size_t)plan_layout(s->batch, s->h_kv, s->head_dim).total;
}

// Workspace of the allocation: water-filling state, channel partial sums (and, from the same chunks,
// partial minima and maxima), counts, channel means, status words.
static size_t alloc_ws_parts(const rdkv_shape* s, size_t* wf, size_t* part, size_t* cnt, size_t* mean) {
  const int64_t n_heads = (int64_t)s->batch * s->h_kv;
  const int Np = s->n_tokens - s->window;
  const int nchunk = std::max(1, ceil_div(Np, kChanChunk));
  *wf = align_up(wf_ws_bytes(s->batch * s->h_kv), 256);  // up to one instance per (sequence, KV head)
  *part = align_up(n_heads * nchunk * s->head_dim * 4, 256);
  *cnt = align_up(n_heads * nchunk * 4, 256);
  *mean = align_up(n_heads * s->head_dim * 4, 256);
  return *wf + 3 * *part + *cnt + *mean + 256;
}

extern "C" size_t rdkv_allocate_workspace_bytes(const rdkv_shape* s) {
  if (check_shape(s) != RDKV_OK) return 0;
  size_t a, b, c, d;
  return alloc_ws_parts(s, &a, &b, &c, &d);
}

static rdkv_status allocate_impl(const rdkv_shape* s, int mode, float param, const float* w_tok, const float* g_tok,
                                 const float* w_chan, const void* k, float avg_bits_v, float avg_bits_k,
                                 uint8_t* bits_tok, float* sigma_chan, float* g_chan, uint8_t* bits_chan, void* plan,
                                 void* ws, size_t ws_bytes, void* stream, const float* levels = nullptr) {
  rdkv_status st = check_shape(s);
  if (st != RDKV_OK) return st;
  const bool at_levels = mode == kAllocLevelsPooled || mode == kAllocLevelsPerHead;
  RDKV_REQUIRE((mode >= RDKV_ALLOC_POOLED && mode <= RDKV_ALLOC_THRESHOLD) || at_levels, RDKV_ERR_INVALID_ARG,
               "unknown allocation mode %d", mode);
  RDKV_REQUIRE(!at_levels || levels != nullptr, RDKV_ERR_INVALID_ARG, "NULL levels");
  RDKV_REQUIRE(std::isfinite(avg_bits_v) && avg_bits_v >= 0 && std::isfinite(avg_bits_k) && avg_bits_k >= 0,
               RDKV_ERR_INVALID_ARG, "budgets must be finite and >= 0 (v=%f k=%f)", (double)avg_bits_v,
               (double)avg_bits_k);
  RDKV_REQUIRE(mode != RDKV_ALLOC_THRESHOLD || (std::isfinite(param) && param >= 0), RDKV_ERR_INVALID_ARG,
               "threshold must be finite and >= 0 (%f)", (double)param);
  const int Np = s->n_tokens - s->window;
  const bool by_weight = mode == RDKV_ALLOC_TOPK || mode == RDKV_ALLOC_THRESHOLD;
  RDKV_REQUIRE(w_chan && k && bits_chan && sigma_chan && g_chan && plan && (Np == 0 || bits_tok) &&
                   (Np == 0 || (by_weight ? w_tok != nullptr : g_tok != nullptr)),
               RDKV_ERR_INVALID_ARG, "NULL pointer argument");
  RDKV_REQUIRE(reinterpret_cast<uintptr_t>(k) % 16 == 0, RDKV_ERR_INVALID_ARG, "k must be 16-byte aligned");
  size_t wf_b, part_b, cnt_b, mean_b;
  const size_t need = alloc_ws_parts(s, &wf_b, &part_b, &cnt_b, &mean_b);
  RDKV_REQUIRE(ws && ws_bytes >= need, RDKV_ERR_WORKSPACE, "allocate workspace too small (%zu < %zu)", ws_bytes, need);
  cudaStream_t cs = (cudaStream_t)stream;
  char* w = static_cast<char*>(ws);
  char* wf = w;
  float* part = reinterpret_cast<float*>(w + wf_b);
  float* pmin = reinterpret_cast<float*>(w + wf_b + part_b);
  float* pmax = reinterpret_cast<float*>(w + wf_b + 2 * part_b);
  int* pcnt = reinterpret_cast<int*>(w + wf_b + 3 * part_b);
  float* mean = reinterpret_cast<float*>(w + wf_b + 3 * part_b + cnt_b);
  int32_t* status = reinterpret_cast<int32_t*>(w + wf_b + 3 * part_b + cnt_b + mean_b);  // [2]
  const PlanLayout L = plan_layout(s->batch, s->h_kv, s->head_dim);
  char* pl = static_cast<char*>(plan);
  float* lam = reinterpret_cast<float*>(pl + L.lambda_off);
  float2* kstat = reinterpret_cast<float2*>(pl + L.kstat_off);
  const int D = s->head_dim;
  const int n_heads = s->batch * s->h_kv;
  // levels: pooled: V [batch] then K [batch]; the other modes: V [n_heads] then K [n_heads]
  const int n_lev = (mode == RDKV_ALLOC_POOLED || mode == kAllocLevelsPooled) ? s->batch : n_heads;
  const int per_units = (int)std::min<int64_t>(std::max<int64_t>(ceil_div64((int64_t)s->h_kv * std::max(Np, D), 256 * 16), 1), 512);

  // step 2: V tokens
  RDKV_TRY_CUDA(cudaMemsetAsync(status, 0, 8, cs), "status reset");
  if (Np > 0) {
    if (mode == RDKV_ALLOC_POOLED) {  // one water level per sequence over all its heads
      st = launch_waterfill(s->batch, (int64_t)s->h_kv * Np, g_tok, avg_bits_v, bits_tok, lam, status, wf, cs);
    } else if (mode == RDKV_ALLOC_PER_HEAD) {  // one water level per (sequence, KV head)
      st = launch_waterfill(n_heads, Np, g_tok, avg_bits_v, bits_tok, lam, status, wf, cs);
    } else if (at_levels) {  // the given levels: one per sequence or per (sequence, KV head)
      const int64_t units = mode == kAllocLevelsPooled ? (int64_t)s->h_kv * Np : Np;
      assign_at_level_kernel<<<dim3(per_units, n_lev), 256, 0, cs>>>(g_tok, units, units, slopes_of(kRdkvSlopes), levels,
                                                                    bits_tok, lam, status);
      RDKV_CHECK_LAUNCH("widths at level (V)");
    } else if (mode == RDKV_ALLOC_TOPK) {  // keep-or-drop on w_t, at most floor(B / 16) kept per head
      st = launch_waterfill(n_heads, Np, w_tok, avg_bits_v, bits_tok, lam, status, wf, cs, s->n_tokens,
                            slopes_of(kKeepSlopes));
    } else {  // keep w_t > threshold
      const int per = (int)std::min<int64_t>(std::max<int64_t>(ceil_div64(Np, 256 * 16), 1), 512);
      keep_above_kernel<<<dim3(per, n_heads), 256, 0, cs>>>(w_tok, Np, s->n_tokens, param, bits_tok, lam, status);
      RDKV_CHECK_LAUNCH("keep above threshold");
    }
    if (st != RDKV_OK) return st;
  } else {
    RDKV_TRY_CUDA(cudaMemsetAsync(lam, 0, 4 * (size_t)n_lev, cs), "lambda reset");
  }
  // step 3: K channel spread over the kept tokens, gains, widths
  const int nchunk = std::max(1, ceil_div(Np, kChanChunk));
  if (Np > 0) {
    chan_pass<<<dim3(nchunk, n_heads), 32 * kChanWarps, 0, cs>>>(k, bits_tok, s->dtype, s->n_tokens, s->h_kv, D, Np,
                                                                 nullptr, part, pcnt, pmin, pmax);
    RDKV_CHECK_LAUNCH("channel sums");
    chan_finish<<<n_heads, std::min(1024, 8 * D), 0, cs>>>(part, pcnt, nchunk, D, mean, nullptr, nullptr, nullptr,
                                                           pmin, pmax, kstat);
    RDKV_CHECK_LAUNCH("channel means");
    chan_pass<<<dim3(nchunk, n_heads), 32 * kChanWarps, 0, cs>>>(k, bits_tok, s->dtype, s->n_tokens, s->h_kv, D, Np,
                                                                 mean, part, nullptr, nullptr, nullptr);
    RDKV_CHECK_LAUNCH("channel deviations");
    chan_finish<<<n_heads, std::min(1024, 8 * D), 0, cs>>>(part, pcnt, nchunk, D, nullptr, w_chan, sigma_chan, g_chan,
                                                           nullptr, nullptr, nullptr);
    RDKV_CHECK_LAUNCH("channel spread");
  } else {
    RDKV_TRY_CUDA(cudaMemsetAsync(sigma_chan, 0, 4 * (size_t)n_heads * D, cs), "sigma reset");
    RDKV_TRY_CUDA(cudaMemsetAsync(g_chan, 0, 4 * (size_t)n_heads * D, cs), "gain reset");
    RDKV_TRY_CUDA(cudaMemsetAsync(kstat, 0, 8 * (size_t)n_heads * D, cs), "channel statistics reset");
  }
  if (mode == RDKV_ALLOC_POOLED) {
    st = launch_waterfill(s->batch, (int64_t)s->h_kv * D, g_chan, avg_bits_k, bits_chan, lam + n_lev, status + 1,
                          wf, cs);
  } else if (mode == RDKV_ALLOC_PER_HEAD) {
    st = launch_waterfill(n_heads, D, g_chan, avg_bits_k, bits_chan, lam + n_lev, status + 1, wf, cs);
  } else if (at_levels) {
    const int64_t units = mode == kAllocLevelsPooled ? (int64_t)s->h_kv * D : D;
    assign_at_level_kernel<<<dim3(per_units, n_lev), 256, 0, cs>>>(g_chan, units, units, slopes_of(kRdkvSlopes),
                                                                  levels + n_lev, bits_chan, lam + n_lev, status + 1);
    RDKV_CHECK_LAUNCH("widths at level (K)");
  } else {  // eviction baselines keep every K channel of the kept tokens at 16 bits
    fill_u8_kernel<<<ceil_div(n_heads * D, 256), 256, 0, cs>>>(bits_chan, (int64_t)n_heads * D, 16);
    RDKV_CHECK_LAUNCH("all channels 16 bits");
    RDKV_TRY_CUDA(cudaMemsetAsync(lam + n_lev, 0, 4 * (size_t)n_lev, cs), "lambda reset");
  }
  if (st != RDKV_OK) return st;
  // TriZone plan
  plan_heads_kernel<<<n_heads, 256, 0, cs>>>(bits_tok, bits_chan, Np, D, pl, L.heads_off, L.slots_off, L.slot_stride);
  RDKV_CHECK_LAUNCH("plan heads");
  plan_offsets_kernel<<<1, 32, 0, cs>>>(pl, s->batch, s->h_kv, D, L.slot_stride, L.heads_off, L.slots_off,
                                        L.lambda_off, status, status + 1);
  RDKV_CHECK_LAUNCH("plan offsets");
  return RDKV_OK;
}

extern "C" rdkv_status rdkv_allocate(const rdkv_shape* s, const float* g_tok, const float* w_chan, const void* k,
                                     float avg_bits_v, float avg_bits_k, uint8_t* bits_tok, float* sigma_chan,
                                     float* g_chan, uint8_t* bits_chan, void* plan, void* ws, size_t ws_bytes,
                                     void* stream) {
  return allocate_impl(s, RDKV_ALLOC_POOLED, 0.f, nullptr, g_tok, w_chan, k, avg_bits_v, avg_bits_k, bits_tok,
                       sigma_chan, g_chan, bits_chan, plan, ws, ws_bytes, stream);
}

extern "C" rdkv_status rdkv_allocate_mode(const rdkv_shape* s, int mode, float param, const float* w_tok,
                                          const float* g_tok, const float* w_chan, const void* k, float avg_bits_v,
                                          float avg_bits_k, uint8_t* bits_tok, float* sigma_chan, float* g_chan,
                                          uint8_t* bits_chan, void* plan, void* ws, size_t ws_bytes, void* stream) {
  RDKV_REQUIRE(mode >= RDKV_ALLOC_POOLED && mode <= RDKV_ALLOC_THRESHOLD, RDKV_ERR_INVALID_ARG,
               "unknown allocation mode %d", mode);
  return allocate_impl(s, mode, param, w_tok, g_tok, w_chan, k, avg_bits_v, avg_bits_k, bits_tok, sigma_chan, g_chan,
                       bits_chan, plan, ws, ws_bytes, stream);
}

extern "C" rdkv_status rdkv_allocate_at_levels(const rdkv_shape* s, int32_t per_head, const float* levels,
                                               const float* g_tok, const float* w_chan, const void* k,
                                               uint8_t* bits_tok, float* sigma_chan, float* g_chan,
                                               uint8_t* bits_chan, void* plan, void* ws, size_t ws_bytes,
                                               void* stream) {
  RDKV_REQUIRE(per_head == 0 || per_head == 1, RDKV_ERR_INVALID_ARG, "per_head must be 0 or 1 (%d)", per_head);
  return allocate_impl(s, per_head ? kAllocLevelsPerHead : kAllocLevelsPooled, 0.f, nullptr, g_tok, w_chan, k, 0.f,
                       0.f, bits_tok, sigma_chan, g_chan, bits_chan, plan, ws, ws_bytes, stream, levels);
}

extern "C" rdkv_status rdkv_plan_sizes(const void* plan, rdkv_sizes* out, void* stream) {
  RDKV_REQUIRE(plan && out, RDKV_ERR_INVALID_ARG, "NULL pointer argument");
  rdkv_plan_header h;
  RDKV_TRY_CUDA(cudaMemcpyAsync(&h, plan, sizeof(h), cudaMemcpyDeviceToHost, (cudaStream_t)stream), "plan read");
  RDKV_TRY_CUDA(cudaStreamSynchronize((cudaStream_t)stream), "plan read sync");
  out->zone_a_bytes = h.zone_a_bytes;
  out->zone_b_rows = h.zone_b_rows;
  out->index_slots = h.index_slots;
  out->kept_tokens = h.kept_tokens;
  out->max_tile_bytes = h.max_tile_bytes;
  out->max_stage_bytes = h.max_stage_bytes;
  out->status = h.status;
  out->n_heads = h.n_heads;
  for (int i = 0; i < RDKV_COST_HEADS; ++i) out->head_cost[i] = 0;
  if (h.status == RDKV_OK && h.n_heads > 0 && h.n_heads <= RDKV_COST_HEADS) {
    // the head records, for the decode's estimate of each head's work
    rdkv_head_plan hp[RDKV_COST_HEADS];
    RDKV_TRY_CUDA(cudaMemcpyAsync(hp, static_cast<const char*>(plan) + h.heads_off, sizeof(rdkv_head_plan) * h.n_heads,
                                  cudaMemcpyDeviceToHost, (cudaStream_t)stream),
                  "plan heads read");
    RDKV_TRY_CUDA(cudaStreamSynchronize((cudaStream_t)stream), "plan heads read sync");
    for (int i = 0; i < h.n_heads; ++i)
      out->head_cost[i] = (int32_t)std::min<int64_t>(std::max<int64_t>(1, head_cost_a(hp[i])), 0x7fffffff);
  }
  if (h.status != RDKV_OK) set_error("plan status %d: a gain was NaN, infinite or negative", h.status);
  return (rdkv_status)h.status;
}
