// Zone-C re-compression (RDKV, gist.science/ko/paper/2605.08317, section 2.3:
// new tokens start in zone C; how they later join zones A and B is left open
// by the pages).  The oldest zone-C rows become a new segment, a TriZone cache
// of their own with no window:
//   * rdkv_zone_c_take copies them out in the prefill layout and moves the
//     remaining rows to the front of zone C;
//   * rdkv_recompress_score gives each moved token the attention the recent
//     decode queries paid it (their log-sum-exp from the decode), its V-row
//     spread and gain (section 2.1 quantities for tokens after the prefill);
//   * the widths then come from rdkv_allocate_at_levels (allocate.cu) and the
//     bytes from rdkv_pack;
//   * rdkv_merge_attn combines the decode outputs of the segments and the live
//     cache into the attention over the union of their keys.
#include <cmath>

#include "common.cuh"

namespace rdkv {

// ---------------------------------------------------------------- merge of disjoint parts
// One block per row: weights e^(lse_i - M) of the parts, then the weighted mean of their outputs.
__global__ void merge_attn_kernel(int n_parts, const float* outs, const float* __restrict__ lses, int64_t rows, int D,
                                  float* out, float* __restrict__ lse_out) {
  const int64_t row = blockIdx.x;
  float M = -INFINITY;
  for (int i = 0; i < n_parts; ++i) M = fmaxf(M, lses[(int64_t)i * rows + row]);
  float tot = 0.f;
  if (M != -INFINITY)
    for (int i = 0; i < n_parts; ++i) tot += expf(lses[(int64_t)i * rows + row] - M);  // exp(-inf) = 0
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float acc = 0.f;
    if (M != -INFINITY)
      for (int i = 0; i < n_parts; ++i) {
        const float w = expf(lses[(int64_t)i * rows + row] - M);
        if (w > 0.f) acc = fmaf(w, outs[((int64_t)i * rows + row) * D + c], acc);
      }
    // a thread reads and writes only its own element of the row: out may alias outs[0]
    out[row * D + c] = tot > 0.f ? acc / tot : 0.f;
  }
  if (lse_out && threadIdx.x == 0) lse_out[row] = tot > 0.f ? M + logf(tot) : -INFINITY;
}

// ---------------------------------------------------------------- taking zone-C rows
// Rows [0, n_move) of head (b, j) -> dst [b][t][j][D] in the cache's dtype (fp16 bits, or the fp16
// values widened to fp32); one block per (head, row).
template <typename T>
__global__ void take_rows_kernel(const uint16_t* __restrict__ zk, const uint16_t* __restrict__ zv,
                                 const int32_t* __restrict__ pages, int stride, int h_kv, int cap, int D, int n_move,
                                 T* __restrict__ k_out, T* __restrict__ v_out) {
  const int head = blockIdx.y, t = blockIdx.x;
  const int b = head / h_kv, j = head % h_kv;
  const int64_t src = zone_c_offset(pages, stride, cap, head, t, D);
  const int64_t dst = (((int64_t)b * n_move + t) * h_kv + j) * D;
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    if constexpr (sizeof(T) == 2) {
      k_out[dst + c] = zk[src + c];
      v_out[dst + c] = zv[src + c];
    } else {
      k_out[dst + c] = __half2float(__ushort_as_half(zk[src + c]));
      v_out[dst + c] = __half2float(__ushort_as_half(zv[src + c]));
    }
  }
}

// Rows [n_move, len_c) -> [0, len_c - n_move); the two ranges do not overlap (checked on the host).
__global__ void shift_rows_kernel(uint16_t* __restrict__ zk, uint16_t* __restrict__ zv,
                                  const int32_t* __restrict__ pages, int stride, int cap, int D, int n_move,
                                  int32_t* len_dev, int new_len) {
  const int head = blockIdx.y, t = blockIdx.x;
  const int64_t src = zone_c_offset(pages, stride, cap, head, n_move + t, D);
  const int64_t dst = zone_c_offset(pages, stride, cap, head, t, D);
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    zk[dst + c] = zk[src + c];
    zv[dst + c] = zv[src + c];
  }
  if (head == 0 && t == 0 && threadIdx.x == 0) *len_dev = new_len;
}

__global__ void set_len_value_kernel(int32_t* len_dev, int v) { *len_dev = v; }


// ---------------------------------------------------------------- weights of moved tokens
constexpr int kScoreTok = 32;      // moved tokens per block
constexpr int kScoreThreads = 256; // eight groups of 32 threads: token = thread % 32
constexpr int kScoreQ = 8;         // recent queries staged per round

// Block (token block, KV head j, sequence b): the K and V rows of its tokens and, round by round,
// the group's recent queries with their log-sum-exps sit in shared memory (K and V rows padded to
// D + 1 floats: the 32 threads of a warp read 32 different rows without bank conflicts; every
// thread of a warp reads the same query row).  Thread (group, token) sums
// 2^(q . k log2(e) / sqrt(D) - lse log2(e)) over its share of the (query, head) pairs.
__global__ void __launch_bounds__(kScoreThreads) recent_weights_kernel(
    const void* __restrict__ k, const void* __restrict__ v, int dtype, const void* __restrict__ q, int q_dtype,
    const float* __restrict__ lse, int R, float wscale, int n, int h_q, int h_kv, int D, float* __restrict__ w_tok,
    float* __restrict__ sigma_tok, float* __restrict__ g_tok) {
  extern __shared__ float sm[];
  const int G = h_q / h_kv;
  const int b = blockIdx.z, j = blockIdx.y, t0 = blockIdx.x * kScoreTok;
  const int tid = threadIdx.x, tok = tid % kScoreTok, grp = tid / kScoreTok;
  const int ngrp = kScoreThreads / kScoreTok;
  float* ks = sm;                                  // [32][D + 1]
  float* vs = ks + kScoreTok * (D + 1);            // [32][D + 1]
  float* qs = vs + kScoreTok * (D + 1);            // [kScoreQ * G][D]
  float* ls = qs + kScoreQ * G * D;                // [kScoreQ * G]
  float* red = ls + kScoreQ * G;                   // [8][32]
  for (int i = tid; i < kScoreTok * D; i += kScoreThreads) {
    const int r = i / D, c = i % D, t = t0 + r;
    const int64_t src = (((int64_t)b * n + t) * h_kv + j) * D + c;
    ks[r * (D + 1) + c] = t < n ? load_as_float(k, src, dtype) : 0.f;
    vs[r * (D + 1) + c] = t < n ? load_as_float(v, src, dtype) : 0.f;
  }
  const float c2 = 1.4426950408889634f / sqrtf((float)D);
  float acc = 0.f;
  for (int r0 = 0; r0 < R; r0 += kScoreQ) {
    const int nr = min(kScoreQ, R - r0);
    __syncthreads();  // the previous round's queries are consumed (and the K rows are staged)
    for (int i = tid; i < nr * G * D; i += kScoreThreads) {
      const int p = i / D, c = i % D, r = r0 + p / G, h = j * G + p % G;
      qs[p * D + c] = load_as_float(q, (((int64_t)b * R + r) * h_q + h) * D + c, q_dtype);
    }
    for (int p = tid; p < nr * G; p += kScoreThreads)
      ls[p] = lse[((int64_t)b * R + r0 + p / G) * h_q + j * G + p % G] * 1.4426950408889634f;
    __syncthreads();
    const float* kr = ks + tok * (D + 1);
    for (int p = grp; p < nr * G; p += ngrp) {
      const float* qr = qs + p * D;
      float d0 = 0.f, d1 = 0.f;
      for (int c = 0; c + 1 < D; c += 2) {
        d0 = fmaf(qr[c], kr[c], d0);
        d1 = fmaf(qr[c + 1], kr[c + 1], d1);
      }
      acc += exp2f(fmaf(d0 + d1, c2, -ls[p]));
    }
  }
  red[grp * kScoreTok + tok] = acc;
  __syncthreads();
  if (tid < kScoreTok && t0 + tid < n) {
    float w = 0.f;
    for (int g = 0; g < ngrp; ++g) w += red[g * kScoreTok + tid];
    w *= wscale;
    // population std of the V row, two passes
    const float* vr = vs + tid * (D + 1);
    float mean = 0.f;
    for (int c = 0; c < D; ++c) mean += vr[c];
    mean /= (float)D;
    float var = 0.f;
    for (int c = 0; c < D; ++c) var = fmaf(vr[c] - mean, vr[c] - mean, var);
    const float sg = sqrtf(var / (float)D);
    const int64_t o = ((int64_t)b * h_kv + j) * n + t0 + tid;
    w_tok[o] = w;
    sigma_tok[o] = sg;
    g_tok[o] = w * sg;
  }
}

static size_t recent_weights_smem(int D, int G) {
  return 4 * ((size_t)2 * kScoreTok * (D + 1) + (size_t)kScoreQ * G * D + (size_t)kScoreQ * G + 8 * kScoreTok);
}

}  // namespace rdkv

using namespace rdkv;

namespace rdkv {
rdkv_status check_cache_public(const rdkv_cache* c);
}

extern "C" rdkv_status rdkv_merge_attn(int32_t n_parts, const float* outs, const float* lses, int64_t rows,
                                       int32_t head_dim, float* out, float* lse_out, void* stream) {
  RDKV_REQUIRE(n_parts >= 1 && rows >= 0 && head_dim >= 1, RDKV_ERR_INVALID_ARG,
               "merge: n_parts %d, rows %lld, head_dim %d", n_parts, (long long)rows, head_dim);
  RDKV_REQUIRE(outs && lses && out, RDKV_ERR_INVALID_ARG, "NULL pointer argument");
  RDKV_REQUIRE(rows <= 0x7fffffff, RDKV_ERR_UNSUPPORTED, "too many rows (%lld)", (long long)rows);
  if (rows == 0) return RDKV_OK;
  merge_attn_kernel<<<(unsigned)rows, std::min(256, ((head_dim + 31) / 32) * 32), 0, (cudaStream_t)stream>>>(
      n_parts, outs, lses, rows, head_dim, out, lse_out);
  RDKV_CHECK_LAUNCH("merge attention");
  return RDKV_OK;
}

extern "C" rdkv_status rdkv_zone_c_take(rdkv_cache* cache, int32_t n_move, void* k_out, void* v_out, void* stream) {
  rdkv_status st = check_cache_public(cache);
  if (st != RDKV_OK) return st;
  RDKV_REQUIRE(k_out && v_out, RDKV_ERR_INVALID_ARG, "NULL pointer argument");
  const int L = cache->len_c;
  RDKV_REQUIRE(n_move > 0 && n_move <= L, RDKV_ERR_INVALID_ARG, "n_move %d outside (0, len_c = %d]", n_move, L);
  RDKV_REQUIRE(L - n_move <= n_move, RDKV_ERR_INVALID_ARG,
               "the %d rows that stay must fit in the %d rows that leave", L - n_move, n_move);
  const rdkv_shape& s = cache->shape;
  const int n_heads = s.batch * s.h_kv, D = s.head_dim;
  cudaStream_t cs = (cudaStream_t)stream;
  if (s.dtype == RDKV_F16)
    take_rows_kernel<uint16_t><<<dim3(n_move, n_heads), std::min(D, 256), 0, cs>>>(
        cache->zone_c_k, cache->zone_c_v, cache->zone_c_pages, cache->zone_c_page_stride, s.h_kv, cache->cap_c, D,
        n_move, static_cast<uint16_t*>(k_out), static_cast<uint16_t*>(v_out));
  else
    take_rows_kernel<float><<<dim3(n_move, n_heads), std::min(D, 256), 0, cs>>>(
        cache->zone_c_k, cache->zone_c_v, cache->zone_c_pages, cache->zone_c_page_stride, s.h_kv, cache->cap_c, D,
        n_move, static_cast<float*>(k_out), static_cast<float*>(v_out));
  RDKV_CHECK_LAUNCH("zone C rows out");
  if (L - n_move > 0) {
    shift_rows_kernel<<<dim3(L - n_move, n_heads), std::min(D, 256), 0, cs>>>(
        cache->zone_c_k, cache->zone_c_v, cache->zone_c_pages, cache->zone_c_page_stride, cache->cap_c, D, n_move,
        cache->len_dev, L - n_move);
    RDKV_CHECK_LAUNCH("zone C rows to the front");
  } else {
    set_len_value_kernel<<<1, 1, 0, cs>>>(cache->len_dev, 0);
    RDKV_CHECK_LAUNCH("zone C length");
  }
  cache->len_c = L - n_move;
  return RDKV_OK;
}

extern "C" rdkv_status rdkv_recompress_score(const rdkv_shape* seg, const void* k, const void* v, const void* q_recent,
                                             int32_t q_dtype, const float* lse_recent, int32_t n_recent,
                                             float weight_scale, float* w_tok, float* sigma_tok, float* g_tok,
                                             void* stream) {
  rdkv_status st = check_shape(seg);
  if (st != RDKV_OK) return st;
  RDKV_REQUIRE(seg->window == 0, RDKV_ERR_INVALID_ARG, "a segment has no window (window %d)", seg->window);
  RDKV_REQUIRE(q_dtype == RDKV_F16 || q_dtype == RDKV_F32, RDKV_ERR_UNSUPPORTED, "query dtype %d", q_dtype);
  RDKV_REQUIRE(n_recent >= 1, RDKV_ERR_INVALID_ARG, "n_recent %d < 1", n_recent);
  RDKV_REQUIRE(std::isfinite(weight_scale) && weight_scale > 0.f, RDKV_ERR_INVALID_ARG, "weight_scale %f",
               (double)weight_scale);
  RDKV_REQUIRE(k && v && q_recent && lse_recent && w_tok && sigma_tok && g_tok, RDKV_ERR_INVALID_ARG,
               "NULL pointer argument");
  const int D = seg->head_dim, G = seg->h_q / seg->h_kv, n = seg->n_tokens;
  const size_t smem = recent_weights_smem(D, G);
  RDKV_REQUIRE(smem <= 227 * 1024, RDKV_ERR_UNSUPPORTED, "group of %d query heads too large", G);
  RDKV_TRY_CUDA(cudaFuncSetAttribute(recent_weights_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
                "recompress smem");
  const dim3 grid(ceil_div(n, kScoreTok), seg->h_kv, seg->batch);
  recent_weights_kernel<<<grid, kScoreThreads, smem, (cudaStream_t)stream>>>(
      k, v, seg->dtype, q_recent, q_dtype, lse_recent, n_recent, weight_scale, n, seg->h_q, seg->h_kv, D, w_tok,
      sigma_tok, g_tok);
  RDKV_CHECK_LAUNCH("recent token weights");
  return RDKV_OK;
}
