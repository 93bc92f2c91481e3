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
#include "stages.cuh"

namespace rdkv {

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
// One block per (sequence, KV head): the head's K metadata (stages.cuh).
__global__ void head_meta_kernel(const void* __restrict__ plan, const float2* __restrict__ kstat, int D,
                                 uint8_t* __restrict__ zone_a, const int32_t* __restrict__ a_pages) {
  head_meta_body(blockIdx.x, plan, kstat, D, zone_a, a_pages);
}

// ---------------------------------------------------------------- tile pack
// One block (256 threads) per zone-A tile (stages.cuh); a grid sized from upper bounds
// (rdkv_zone_bounds) has blocks past the plan's last tile, which leave at once.
template <typename T, int D>
__global__ void __launch_bounds__(kPackThreads) pack_tile_kernel(const T* __restrict__ k, const T* __restrict__ v,
                                                                  const void* __restrict__ plan,
                                                                  const float2* __restrict__ kstat,
                                                                  const int32_t* __restrict__ index_map,
                                                                  uint8_t* __restrict__ zone_a,
                                                                  uint16_t* __restrict__ zone_b, int N, int h_kv,
                                                                  const int32_t* __restrict__ a_pages,
                                                                  const int32_t* __restrict__ b_pages) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  if ((int64_t)blockIdx.x * kTile >= plan_header(plan)->index_slots) return;
  pack_tile_item<T, D>(blockIdx.x, k, v, plan, kstat, index_map, zone_a, zone_b, N, h_kv, a_pages, b_pages, smem_raw);
}

template <typename T>
__global__ void window_kernel(const T* __restrict__ x, int N, int W, int h_kv, int D, int cap, int batch,
                              uint16_t* __restrict__ zc, const int32_t* __restrict__ pages, int stride) {
  window_part(x, N, W, h_kv, D, cap, batch, zc, pages, stride, (int64_t)blockIdx.x * blockDim.x + threadIdx.x,
              (int64_t)gridDim.x * blockDim.x);
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
