// Shared definitions of the RDKV CUDA sources (device helpers, plan access,
// host error reporting).  Layout constants follow the TriZone rules written
// in include/rdkv.h.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>

#include "../../include/rdkv.h"

namespace rdkv {

constexpr int kTile = 32;          // tokens per zone-A tile
constexpr int kVGroup = 32;        // channels per V quantiser group
constexpr int kSlotPad = 32;       // extra K slots a head may need for word padding

__host__ __device__ inline int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ inline int64_t align_up(int64_t a, int64_t b) { return ceil_div64(a, b) * b; }

// ---------------------------------------------------------------- plan buffer
struct PlanLayout {
  int64_t heads_off, slots_off, lambda_off, total;
  int slot_stride;
};

__host__ __device__ inline PlanLayout plan_layout(int batch, int h_kv, int head_dim) {
  PlanLayout L;
  const int64_t n_heads = (int64_t)batch * h_kv;
  L.slot_stride = head_dim + kSlotPad;
  L.heads_off = align_up(sizeof(rdkv_plan_header), 128);
  L.slots_off = align_up(L.heads_off + n_heads * (int64_t)sizeof(rdkv_head_plan), 128);
  L.lambda_off = align_up(L.slots_off + n_heads * L.slot_stride * 2, 128);
  L.total = align_up(L.lambda_off + 2 * n_heads * 4, 256);  // room for one level per (sequence, KV head)
  return L;
}

// Estimated zone-A decode cost of a head (instruction units per warp) from its plan record: every
// tile pays a base (softmax, staging) plus its K k-blocks (quantised blocks cost about twice a raw
// 16-bit one) plus its V class.  Only the ratios between heads matter: they decide how many
// blocks each head gets.
__host__ __device__ inline int64_t head_cost_a(const rdkv_head_plan& hp) {
  const int nkb16 = ceil_div(hp.k_words[0] * 2, 16);
  const int nkbq = ceil_div(hp.k_words[1] * 4, 16) + ceil_div(hp.k_words[2] * 8, 16) + ceil_div(hp.k_words[3] * 16, 16);
  const int64_t per_tile = 250 + 20 * nkb16 + 40 * nkbq;
  return (int64_t)hp.tiles[0] * (per_tile + 200) + (int64_t)hp.tiles[1] * (per_tile + 215) +
         (int64_t)hp.tiles[2] * (per_tile + 250) + (int64_t)hp.tiles[3] * (per_tile + 60);
}
// ... and of one zone-C block of 16 rows
constexpr int kZoneCBlockCost = 300;

__device__ __forceinline__ const rdkv_plan_header* plan_header(const void* plan) {
  return reinterpret_cast<const rdkv_plan_header*>(plan);
}
__device__ __forceinline__ const rdkv_head_plan* plan_heads(const void* plan) {
  return reinterpret_cast<const rdkv_head_plan*>(static_cast<const char*>(plan) + plan_header(plan)->heads_off);
}
__device__ __forceinline__ const int16_t* plan_slots(const void* plan) {
  return reinterpret_cast<const int16_t*>(static_cast<const char*>(plan) + plan_header(plan)->slots_off);
}

// Tile byte size of width class c for a head (same rule as the plan kernel).
__host__ __device__ inline int tile_bytes_of(int row_words, int meta_slots, int head_dim, int vbits) {
  int b = 4 * kTile * row_words + 4 * meta_slots;
  if (vbits < 16) b += (kTile * head_dim * vbits) / 8 + 4 * head_dim;
  return b;
}

// Element offset of row `row` of head `head` in zone C: contiguous [heads][cap][D], or, with a page
// table, row row % 16 of page pages[head * stride + row / 16] of a pool [pages][16][D].
constexpr int kZoneCPageRows = RDKV_ZONE_C_PAGE_ROWS;
__host__ __device__ inline int64_t zone_c_offset(const int32_t* pages, int stride, int cap, int head, int row, int D) {
  return pages ? ((int64_t)pages[(int64_t)head * stride + row / kZoneCPageRows] * kZoneCPageRows + row % kZoneCPageRows) * D
               : ((int64_t)head * cap + row) * D;
}

// ---------------------------------------------------------------- numerics
__device__ __forceinline__ float load_as_float(const void* p, int64_t i, int dtype) {
  return dtype == RDKV_F16 ? __half2float(static_cast<const __half*>(p)[i]) : static_cast<const float*>(p)[i];
}

__device__ __forceinline__ uint16_t half_bits(float x) { return __half_as_ushort(__float2half_rn(x)); }

// Canonical bit pattern of a water level candidate: positive finite values keep
// their pattern (monotone in value for non-negative floats), everything else is 0.
__device__ __forceinline__ uint32_t level_bits(float x) { return x > 0.0f ? __float_as_uint(x) : 0u; }

// ---------------------------------------------------------------- host error state
void set_error(const char* fmt, ...);
rdkv_status cuda_status(cudaError_t e, const char* what);
rdkv_status check_shape(const rdkv_shape* s);
int num_sms();
void count_launch();

}  // namespace rdkv

#define RDKV_TRY_CUDA(expr, what)                                       \
  do {                                                                  \
    cudaError_t _e = (expr);                                            \
    if (_e != cudaSuccess) return ::rdkv::cuda_status(_e, what);        \
  } while (0)

#define RDKV_CHECK_LAUNCH(what)                 \
  do {                                          \
    ::rdkv::count_launch();                     \
    RDKV_TRY_CUDA(cudaGetLastError(), what);    \
  } while (0)

#define RDKV_REQUIRE(cond, code, ...)            \
  do {                                           \
    if (!(cond)) {                               \
      ::rdkv::set_error(__VA_ARGS__);            \
      return code;                               \
    }                                            \
  } while (0)
