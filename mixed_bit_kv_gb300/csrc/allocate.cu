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

#include "stages.cuh"

namespace rdkv {

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

// g of instance i starts at g + i * in_stride (units contiguous).
__global__ void wf_hist(const float* __restrict__ g, int64_t n_units, int64_t in_stride, Slopes sl, int level,
                        const WfState* __restrict__ st, unsigned long long* __restrict__ hist, int32_t* status) {
  __shared__ uint32_t h[256];
  const int inst = blockIdx.y;
  wf_hist_part(g + (int64_t)inst * in_stride, n_units, sl, level, st[inst].prefix, blockIdx.x, gridDim.x, h,
               hist + inst * 256, status);
}

// One block of 256 threads per instance: digit d is kept if the bits bought
// above x_d = prefix | d << shift | (lower bits all ones) fit the budget.
__global__ void wf_select(int level, long long budget, WfState* st, unsigned long long* hist) {
  __shared__ unsigned long long s[9];
  __shared__ int best;
  const int inst = blockIdx.x, t = threadIdx.x;
  const WfPick cur{st[inst].prefix, st[inst].above};
  const WfPick nxt = wf_pick(hist[inst * 256 + t], level, budget, cur, s, &best);
  if (t == 0) {
    st[inst].prefix = nxt.prefix;
    st[inst].above = nxt.above;
  }
  hist[inst * 256 + t] = 0;
}

__global__ void wf_assign(const float* __restrict__ g, int64_t n_units, int64_t in_stride, Slopes sl,
                          const WfState* __restrict__ st, uint8_t* __restrict__ bits, float* __restrict__ lambda_out) {
  const int inst = blockIdx.y;
  const uint32_t lam = st[inst].prefix;
  if (lambda_out && blockIdx.x == 0 && threadIdx.x == 0) lambda_out[inst] = __uint_as_float(lam);
  wf_assign_part(g + (int64_t)inst * in_stride, n_units, sl, lam, blockIdx.x, gridDim.x, bits + (int64_t)inst * n_units);
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
    bi[u] = width_after(m);
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
// Block (chunk, head): one chunk item of a channel pass (stages.cuh).
__global__ void __launch_bounds__(32 * kChanWarps) chan_pass(const void* __restrict__ k,
                                                             const uint8_t* __restrict__ bits_tok, int dtype, int N,
                                                             int h_kv, int D, int Np, const float* __restrict__ mean,
                                                             float* __restrict__ part, int* __restrict__ part_cnt,
                                                             float* __restrict__ pmin, float* __restrict__ pmax) {
  __shared__ ChanSmem sm;
  chan_pass_item(blockIdx.x, gridDim.x, blockIdx.y, k, bits_tok, dtype, N, h_kv, D, Np, mean, part, part_cnt, pmin,
                 pmax, sm);
}

// Block (head, 32-channel slice), 256 threads: the chunk combine (stages.cuh).  The first call
// (mean_out set) also writes the head's K channel statistics kstat.
__global__ void __launch_bounds__(32 * kChanRows) chan_finish(const float* __restrict__ part,
                                                              const int* __restrict__ part_cnt, int nchunk, int D,
                                                              float* __restrict__ mean_out,
                                                              const float* __restrict__ w_chan,
                                                              float* __restrict__ sigma_out, float* __restrict__ g_out,
                                                              const float* __restrict__ pmin,
                                                              const float* __restrict__ pmax,
                                                              float2* __restrict__ kstat) {
  __shared__ ChanFinishSmem sm;
  const int slices = D / 32;
  chan_finish_item(blockIdx.x / slices, blockIdx.x % slices, part, part_cnt, nchunk, D, mean_out, w_chan, sigma_out,
                   g_out, pmin, pmax, kstat, sm);
}

// ---------------------------------------------------------------- plan
// One block (256 threads) per head: V class counts of its tokens and K class counts of its
// channels, the head record, then the slot table.
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
  count_classes(bits_tok + (int64_t)head * Np, 0, Np, blockDim.x, threadIdx.x, cnt);
#pragma unroll
  for (int i = 0; i < 4; ++i) atomicAdd(&nv[i], cnt[i]);
  plan_count_k(bcs, D, nk);
  __syncthreads();
  if (threadIdx.x == 0) {
    const int v4[4] = {nv[0], nv[1], nv[2], nv[3]}, k5[5] = {nk[0], nk[1], nk[2], nk[3], nk[4]};
    reinterpret_cast<rdkv_head_plan*>(plan + heads_off)[head] = make_head_record(v4, k5, D, seg_base);
  }
  __syncthreads();
  plan_slot_table(bcs, D, seg_base, slots);
}

__global__ void plan_offsets_kernel(char* plan, int batch, int h_kv, int D, int slot_stride, int64_t heads_off,
                                    int64_t slots_off, int64_t lambda_off, const int32_t* status_v,
                                    const int32_t* status_k) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  plan_offsets_body(plan, batch, h_kv, D, slot_stride, heads_off, slots_off, lambda_off, *status_v, *status_k);
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
    chan_finish<<<n_heads * (D / 32), 32 * kChanRows, 0, cs>>>(part, pcnt, nchunk, D, mean, nullptr, nullptr,
                                                               nullptr, pmin, pmax, kstat);
    RDKV_CHECK_LAUNCH("channel means");
    chan_pass<<<dim3(nchunk, n_heads), 32 * kChanWarps, 0, cs>>>(k, bits_tok, s->dtype, s->n_tokens, s->h_kv, D, Np,
                                                                 mean, part, nullptr, nullptr, nullptr);
    RDKV_CHECK_LAUNCH("channel deviations");
    chan_finish<<<n_heads * (D / 32), 32 * kChanRows, 0, cs>>>(part, pcnt, nchunk, D, nullptr, w_chan, sigma_chan,
                                                               g_chan, nullptr, nullptr, nullptr);
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
