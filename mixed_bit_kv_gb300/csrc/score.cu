// Distortion weights of RDKV (gist.science/ko/paper/2605.08317, section 2.1),
// computed once after prefill on the full cache (section 2.2, step 1):
//   w_t  = sum over query positions tau >= t and the G query heads of the
//          group of the causal softmax a_{tau,h,t}        (V-cache weight)
//   w_c  = |Q_:,c| |K_:,c| / sqrt(d)                      (K-cache weight)
// plus the spread sigma_t of each V row and the gain g_t = w_t * sigma_t of
// the objective's V units.
//
// w_t needs the normaliser of every softmax row before any column can be
// summed, so the scorer runs two passes over the causal pairs: pass 1 keeps
// one log-sum-exp per query row; pass 2 recomputes each logit, turns it into
// a probability with that row's normaliser and sums the columns.  This file
// holds the CUDA-core passes (exact fp32 logits, used for fp32 inputs) and
// the row/column reductions; the fp16 passes run on the tensor cores
// (score_tc.cu), whose first pass also takes the sums of squares behind w_c
// from the tiles it loads (the column passes here serve fp32 inputs).
#include <cmath>

#include "common.cuh"

namespace rdkv {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kSTile = 32;      // query rows / keys per block in the CUDA-core passes
constexpr int kColChunk = 256;  // rows per partial column sum

// ---------------------------------------------------------------- sigma of V rows: one warp per row
// sigma of V rows: a warp takes kSpreadRows rows; lane l holds the D/32 consecutive elements
// [l D/32, (l+1) D/32) of a row, loaded as one vector, so every row is one load per lane and a
// warp keeps kSpreadRows loads in flight.
constexpr int kSpreadRows = 8;
template <typename T, int PER>
__device__ __forceinline__ void load_row_part(const T* __restrict__ p, float (&x)[PER]) {
  if constexpr (sizeof(T) == 2) {
    if constexpr (PER == 4) {
      const uint2 r = *reinterpret_cast<const uint2*>(p);
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&r.x));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&r.y));
      x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
    } else {
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(p));
      x[0] = a.x; x[1] = a.y;
    }
  } else {
    if constexpr (PER == 4) {
      const float4 r = *reinterpret_cast<const float4*>(p);
      x[0] = r.x; x[1] = r.y; x[2] = r.z; x[3] = r.w;
    } else {
      const float2 r = *reinterpret_cast<const float2*>(p);
      x[0] = r.x; x[1] = r.y;
    }
  }
}
template <typename T, int PER>
__global__ void value_spread_kernel(const T* __restrict__ v, int64_t n_rows, int h_kv, int N, float* __restrict__ sigma) {
  constexpr int D = 32 * PER;
  const int lane = threadIdx.x & 31;
  const int64_t row0 = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * kSpreadRows;  // (b, t, j) flattened
  float x[kSpreadRows][PER];
#pragma unroll
  for (int r = 0; r < kSpreadRows; ++r) {
    if (row0 + r < n_rows) load_row_part<T, PER>(v + (row0 + r) * D + lane * PER, x[r]);
    else
#pragma unroll
      for (int e = 0; e < PER; ++e) x[r][e] = 0.f;
  }
#pragma unroll
  for (int r = 0; r < kSpreadRows; ++r) {
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e) s += x[r][e];
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float mean = s / (float)D;
    float m2 = 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e) m2 += (x[r][e] - mean) * (x[r][e] - mean);
    for (int o = 16; o; o >>= 1) m2 += __shfl_xor_sync(0xffffffffu, m2, o);
    const int64_t row = row0 + r;
    if (lane == 0 && row < n_rows) {
      const int j = (int)(row % h_kv);
      const int64_t bt = row / h_kv;
      const int t = (int)(bt % N);
      const int64_t b = bt / N;
      sigma[(b * h_kv + j) * N + t] = sqrtf(m2 / (float)D);
    }
  }
}

// ---------------------------------------------------------------- column sums of squares (for w_c)
// part[b][chunk][col] = sum over the chunk's rows of x[b][row][col]^2, cols = H*D.
__global__ void colsq_kernel(const void* __restrict__ x, int dtype, int N, int cols, float* __restrict__ part) {
  const int b = blockIdx.z, chunk = blockIdx.y;
  const int col = blockIdx.x * blockDim.x + threadIdx.x;
  if (col >= cols) return;
  const int r0 = chunk * kColChunk, r1 = min(N, r0 + kColChunk);
  float acc = 0.f;
  for (int r = r0; r < r1; ++r) {
    const float v = load_as_float(x, ((int64_t)b * N + r) * cols + col, dtype);
    acc += v * v;
  }
  part[((int64_t)b * gridDim.y + chunk) * cols + col] = acc;
}

// w_c = sqrt(sum q^2) sqrt(sum k^2) / sqrt(D) per (b, KV head j, channel c) from partial sums of squares:
// qpart[b][nq][H_q][D] (the group's G query heads are added), kpart[b][nk][H_kv][D].  Block: 32 channels
// x 32 partial rows; thread (r, c) adds the partials r, r + 32, ... in fp64, the 32 sums combine in a
// fixed order (deterministic).
__global__ void __launch_bounds__(1024) channel_weight_kernel(const float* __restrict__ qpart, int nq,
                                                              const float* __restrict__ kpart, int nk, int h_q,
                                                              int h_kv, int D, float* __restrict__ w_chan) {
  __shared__ double sq[32][33], sk[32][33];
  const int head = blockIdx.x;  // b * h_kv + j
  const int b = head / h_kv, j = head % h_kv;
  const int cc = threadIdx.x & 31, r = threadIdx.x >> 5;
  const int c = blockIdx.y * 32 + cc;
  const int G = h_q / h_kv;
  double qs = 0.0, ks = 0.0;
  for (int i = r; i < nq; i += 32) {
    const float* qp = qpart + ((int64_t)b * nq + i) * h_q * D;
    for (int h = j * G; h < (j + 1) * G; ++h) qs += (double)qp[h * D + c];
  }
  for (int i = r; i < nk; i += 32) ks += (double)kpart[((int64_t)b * nk + i) * h_kv * D + j * D + c];
  sq[r][cc] = qs;
  sk[r][cc] = ks;
  __syncthreads();
  if (r != 0) return;
  for (int rr = 1; rr < 32; ++rr) {
    qs += sq[rr][cc];
    ks += sk[rr][cc];
  }
  w_chan[head * D + c] = (float)(sqrt(qs) * sqrt(ks) / sqrt((double)D));
}

rdkv_status launch_channel_weights(const rdkv_shape* s, const float* qpart, int nq, const float* kpart, int nk,
                                   float* w_chan, cudaStream_t st) {
  channel_weight_kernel<<<dim3(s->batch * s->h_kv, s->head_dim / 32), 1024, 0, st>>>(qpart, nq, kpart, nk, s->h_q,
                                                                                      s->h_kv, s->head_dim, w_chan);
  RDKV_CHECK_LAUNCH("channel weights");
  return RDKV_OK;
}

// ---------------------------------------------------------------- CUDA-core pass 1: row log-sum-exp (base 2)
// Block: 32 query rows of one (b, h); 128 threads, 4 per row, each thread
// takes 8 consecutive keys of every 32-key tile.
__global__ void __launch_bounds__(128) lse_simt_kernel(const void* __restrict__ q, const void* __restrict__ k,
                                                        int dtype, int N, int h_q, int h_kv, int D,
                                                        float* __restrict__ lse2) {
  extern __shared__ float sm[];
  float* Qs = sm;                      // [32][D + 1]
  float* Kt = sm + kSTile * (D + 1);   // [D][32 + 4] (keys contiguous)
  const int b = blockIdx.z, h = blockIdx.y, r0 = blockIdx.x * kSTile;
  const int j = h / (h_q / h_kv);
  const int tid = threadIdx.x, row = tid >> 2, sub = tid & 3;
  const float sc = kLog2e / sqrtf((float)D);
  for (int i = tid; i < kSTile * D; i += blockDim.x) {
    const int r = i / D, d = i % D;
    Qs[r * (D + 1) + d] = (r0 + r < N) ? load_as_float(q, (((int64_t)b * N + r0 + r) * h_q + h) * D + d, dtype) : 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const int tau = r0 + row;
  const int n_tiles = ceil_div(min(N, r0 + kSTile), kSTile);
  for (int kt = 0; kt < n_tiles; ++kt) {
    __syncthreads();
    for (int i = tid; i < kSTile * D; i += blockDim.x) {
      const int key = i / D, d = i % D, t = kt * kSTile + key;
      Kt[d * (kSTile + 4) + key] = (t < N) ? load_as_float(k, (((int64_t)b * N + t) * h_kv + j) * D + d, dtype) : 0.f;
    }
    __syncthreads();
    float s[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int d = 0; d < D; ++d) {
      const float qv = Qs[row * (D + 1) + d];
      const float4 k0 = *reinterpret_cast<const float4*>(&Kt[d * (kSTile + 4) + 8 * sub]);
      const float4 k1 = *reinterpret_cast<const float4*>(&Kt[d * (kSTile + 4) + 8 * sub + 4]);
      s[0] += qv * k0.x; s[1] += qv * k0.y; s[2] += qv * k0.z; s[3] += qv * k0.w;
      s[4] += qv * k1.x; s[5] += qv * k1.y; s[6] += qv * k1.z; s[7] += qv * k1.w;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int t = kt * kSTile + 8 * sub + i;
      if (t <= tau && tau < N) {
        const float x = s[i] * sc;
        if (x > m) {
          l = l * exp2f(m - x) + 1.f;
          m = x;
        } else {
          l += exp2f(x - m);
        }
      }
    }
  }
#pragma unroll
  for (int o = 1; o < 4; o <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
    const float mm = fmaxf(m, m2);
    l = (m == -INFINITY ? 0.f : l * exp2f(m - mm)) + (m2 == -INFINITY ? 0.f : l2 * exp2f(m2 - mm));
    m = mm;
  }
  if (sub == 0 && tau < N) lse2[((int64_t)b * h_q + h) * N + tau] = m + log2f(l);
}

// ---------------------------------------------------------------- CUDA-core pass 2: column sums
// Block: 32 keys of one (b, j); sweeps the query rows tau >= key block start
// for the G heads of the group.  4 threads per key, 8 rows each per tile.
__global__ void __launch_bounds__(128) colsum_simt_kernel(const void* __restrict__ q, const void* __restrict__ k,
                                                           int dtype, int N, int Np, int h_q, int h_kv, int D,
                                                           const float* __restrict__ lse2,
                                                           const float* __restrict__ sigma,
                                                           float* __restrict__ w_tok, float* __restrict__ g_tok) {
  extern __shared__ float sm[];
  float* Ks = sm;                      // [32][D + 1]
  float* Qt = sm + kSTile * (D + 1);   // [D][32 + 4] (rows contiguous)
  float* L = Qt + D * (kSTile + 4);    // [32]
  const int b = blockIdx.z, j = blockIdx.y, t0 = blockIdx.x * kSTile;
  const int G = h_q / h_kv;
  const int tid = threadIdx.x, key = tid >> 2, sub = tid & 3;
  const float sc = kLog2e / sqrtf((float)D);
  for (int i = tid; i < kSTile * D; i += blockDim.x) {
    const int r = i / D, d = i % D;
    Ks[r * (D + 1) + d] = (t0 + r < N) ? load_as_float(k, (((int64_t)b * N + t0 + r) * h_kv + j) * D + d, dtype) : 0.f;
  }
  const int t = t0 + key;
  float acc = 0.f;
  for (int h = j * G; h < (j + 1) * G; ++h) {
    for (int r0 = t0; r0 < N; r0 += kSTile) {
      __syncthreads();
      for (int i = tid; i < kSTile * D; i += blockDim.x) {
        const int r = i / D, d = i % D, tau = r0 + r;
        Qt[d * (kSTile + 4) + r] = (tau < N) ? load_as_float(q, (((int64_t)b * N + tau) * h_q + h) * D + d, dtype) : 0.f;
      }
      if (tid < kSTile) L[tid] = (r0 + tid < N) ? lse2[((int64_t)b * h_q + h) * N + r0 + tid] : 0.f;
      __syncthreads();
      float s[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      for (int d = 0; d < D; ++d) {
        const float kv = Ks[key * (D + 1) + d];
        const float4 q0 = *reinterpret_cast<const float4*>(&Qt[d * (kSTile + 4) + 8 * sub]);
        const float4 q1 = *reinterpret_cast<const float4*>(&Qt[d * (kSTile + 4) + 8 * sub + 4]);
        s[0] += kv * q0.x; s[1] += kv * q0.y; s[2] += kv * q0.z; s[3] += kv * q0.w;
        s[4] += kv * q1.x; s[5] += kv * q1.y; s[6] += kv * q1.z; s[7] += kv * q1.w;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int tau = r0 + 8 * sub + i;
        if (tau >= t && tau < N) acc += exp2f(s[i] * sc - L[8 * sub + i]);
      }
    }
  }
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  if (sub == 0 && t < N) {
    const int64_t o = ((int64_t)b * h_kv + j) * N + t;
    w_tok[o] = acc;
    if (t < Np) g_tok[((int64_t)b * h_kv + j) * Np + t] = acc * sigma[o];
  }
}

// The fp16 tensor-core passes live in score_tc.cu.
rdkv_status launch_score_tc(const rdkv_shape* s, const void* q, const void* k, const float* sigma, float* lse2,
                            float* w_tok, float* g_tok, float* qsq, float* ksq, float* w_chan, cudaStream_t st);
int score_tc_lse_stride(int n_tokens);
int score_tc_q_chunks(int n_tokens);
int score_tc_k_chunks(int n_tokens);

// Workspace: row log-sum-exps, then the partial sums of squares of the channel weights (chunks of
// kColChunk rows on the CUDA-core path; 128-row blocks for q and 256-key tiles for k on the
// tensor-core path, which takes them in scorer pass 1).
static size_t score_ws_parts(const rdkv_shape* s, size_t* lse, size_t* qp, size_t* kp) {
  const int nchunk = ceil_div(s->n_tokens, kColChunk);
  const int nq = std::max(nchunk, score_tc_q_chunks(s->n_tokens)), nk = std::max(nchunk, score_tc_k_chunks(s->n_tokens));
  *lse = align_up((int64_t)s->batch * s->h_q * score_tc_lse_stride(s->n_tokens) * 4, 256);
  *qp = align_up((int64_t)s->batch * nq * s->h_q * s->head_dim * 4, 256);
  *kp = align_up((int64_t)s->batch * nk * s->h_kv * s->head_dim * 4, 256);
  return *lse + *qp + *kp;
}

}  // namespace rdkv

using namespace rdkv;

extern "C" size_t rdkv_score_workspace_bytes(const rdkv_shape* s) {
  if (check_shape(s) != RDKV_OK) return 0;
  size_t a, b, c;
  return score_ws_parts(s, &a, &b, &c);
}

extern "C" rdkv_status rdkv_score(const rdkv_shape* s, const void* q, const void* k, const void* v, float* w_tok,
                                  float* w_chan, float* sigma_tok, float* g_tok, void* ws, size_t ws_bytes,
                                  void* stream) {
  rdkv_status st = check_shape(s);
  if (st != RDKV_OK) return st;
  const int N = s->n_tokens, D = s->head_dim, Np = N - s->window;
  RDKV_REQUIRE(q && k && v && w_tok && w_chan && sigma_tok && (Np == 0 || g_tok), RDKV_ERR_INVALID_ARG,
               "NULL pointer argument");
  RDKV_REQUIRE(((uintptr_t)q | (uintptr_t)k | (uintptr_t)v) % 16 == 0, RDKV_ERR_INVALID_ARG,
               "q, k and v must be 16-byte aligned");
  size_t lse_b, qp_b, kp_b;
  const size_t need = score_ws_parts(s, &lse_b, &qp_b, &kp_b);
  RDKV_REQUIRE(ws && ws_bytes >= need, RDKV_ERR_WORKSPACE, "score workspace too small (%zu < %zu)", ws_bytes, need);
  cudaStream_t cs = (cudaStream_t)stream;
  char* w = static_cast<char*>(ws);
  float* lse2 = reinterpret_cast<float*>(w);
  float* qpart = reinterpret_cast<float*>(w + lse_b);
  float* kpart = reinterpret_cast<float*>(w + lse_b + qp_b);

  // sigma of V rows
  const int64_t rows = (int64_t)s->batch * N * s->h_kv;
  {
    const unsigned blocks = (unsigned)ceil_div64(ceil_div64(rows, kSpreadRows) * 32, 256);
    if (s->dtype == RDKV_F16) {
      if (D == 128) value_spread_kernel<__half, 4><<<blocks, 256, 0, cs>>>(static_cast<const __half*>(v), rows, s->h_kv, N, sigma_tok);
      else value_spread_kernel<__half, 2><<<blocks, 256, 0, cs>>>(static_cast<const __half*>(v), rows, s->h_kv, N, sigma_tok);
    } else {
      if (D == 128) value_spread_kernel<float, 4><<<blocks, 256, 0, cs>>>(static_cast<const float*>(v), rows, s->h_kv, N, sigma_tok);
      else value_spread_kernel<float, 2><<<blocks, 256, 0, cs>>>(static_cast<const float*>(v), rows, s->h_kv, N, sigma_tok);
    }
  }
  RDKV_CHECK_LAUNCH("value spread");
  // fp16: token weights on the tensor cores, whose first pass also takes the channel weights' sums of
  // squares from the tiles it loads; the channel weights follow it
  if (s->dtype == RDKV_F16) return launch_score_tc(s, q, k, sigma_tok, lse2, w_tok, g_tok, qpart, kpart, w_chan, cs);
  // fp32: channel weights from their own column passes, then the token weights on the CUDA cores
  const int nchunk = ceil_div(N, kColChunk);
  colsq_kernel<<<dim3(ceil_div(s->h_q * D, 256), nchunk, s->batch), 256, 0, cs>>>(q, s->dtype, N, s->h_q * D, qpart);
  RDKV_CHECK_LAUNCH("query column norms");
  colsq_kernel<<<dim3(ceil_div(s->h_kv * D, 256), nchunk, s->batch), 256, 0, cs>>>(k, s->dtype, N, s->h_kv * D,
                                                                                   kpart);
  RDKV_CHECK_LAUNCH("key column norms");
  st = launch_channel_weights(s, qpart, nchunk, kpart, nchunk, w_chan, cs);
  if (st != RDKV_OK) return st;
  const size_t smem = (size_t)(kSTile * (D + 1) + D * (kSTile + 4) + kSTile) * 4;
  lse_simt_kernel<<<dim3(ceil_div(N, kSTile), s->h_q, s->batch), 128, smem, cs>>>(q, k, s->dtype, N, s->h_q, s->h_kv,
                                                                                    D, lse2);
  RDKV_CHECK_LAUNCH("row log-sum-exp");
  colsum_simt_kernel<<<dim3(ceil_div(N, kSTile), s->h_kv, s->batch), 128, smem, cs>>>(
      q, k, s->dtype, N, Np, s->h_q, s->h_kv, D, lse2, sigma_tok, w_tok, g_tok);
  RDKV_CHECK_LAUNCH("attention column sums");
  return RDKV_OK;
}
