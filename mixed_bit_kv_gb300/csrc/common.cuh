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
constexpr int kKB = 16;            // K slots of one k-block
constexpr int kSlotPad = 64;       // extra K slots a head may need: each width segment spans whole k-blocks

__host__ __device__ inline int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ inline int64_t align_up(int64_t a, int64_t b) { return ceil_div64(a, b) * b; }

// ---------------------------------------------------------------- plan buffer
struct PlanLayout {
  int64_t heads_off, slots_off, lambda_off, kstat_off, total;
  int slot_stride;
};

// The plan buffer: header, head records, slot tables, water levels (one per (sequence, KV head) at
// most), then the K channel statistics of each head: {min, max} over its kept prefix tokens, fp32
// [n_heads][D][2] (written by the allocation, read by the pack).
__host__ __device__ inline PlanLayout plan_layout(int batch, int h_kv, int head_dim) {
  PlanLayout L;
  const int64_t n_heads = (int64_t)batch * h_kv;
  L.slot_stride = head_dim + kSlotPad;
  L.heads_off = align_up(sizeof(rdkv_plan_header), 128);
  L.slots_off = align_up(L.heads_off + n_heads * (int64_t)sizeof(rdkv_head_plan), 128);
  L.lambda_off = align_up(L.slots_off + n_heads * L.slot_stride * 2, 128);
  L.kstat_off = align_up(L.lambda_off + 2 * n_heads * 4, 256);
  L.total = align_up(L.kstat_off + n_heads * head_dim * 8, 256);
  return L;
}

// Slot, inside its k-block, of element e of the block's word i at K width b (the layout rule of the
// K rows: lane q of a decode fragment reads slots 2q, 2q+1, 2q+8, 2q+9 of a block from one word).
__host__ __device__ inline int k_slot_in_block(int b, int i, int e) {
  if (b == 16) return 2 * i + e;
  if (b == 8) return 2 * i + (e & 1) + 8 * (e >> 1);
  if (b == 4) return 2 * (2 * i + (e >> 2)) + (e & 1) + 8 * ((e >> 1) & 1);
  return e;
}

// K metadata of a head (fp16 scale and zero per quantised slot) in front of its tiles, whole 16 bytes.
__host__ __device__ inline int64_t head_meta_bytes(int meta_slots) { return align_up(4 * (int64_t)meta_slots, 16); }

// Estimated zone-A decode cost of a head (units of about a third of a nanosecond of one block's
// loop) from its plan record: every tile pays its V class (with the staging, softmax and
// bookkeeping every tile has) plus its K k-blocks.  The constants are a least-squares fit of the
// measured per-block loop times of 112 (head, workload, budget) cases on GB300; raw 16-bit K
// blocks, absent from those cases, are costed at three quarters of a 2-bit one, as their
// instruction count suggests.  Only the ratios between heads matter: they decide how many blocks
// each head gets.
__host__ __device__ inline int64_t head_cost_a(const rdkv_head_plan& hp) {
  const int64_t nkb16 = ceil_div(hp.k_words[0] * 2, kKB);
  const int64_t nkb8 = ceil_div(hp.k_words[1] * 4, kKB), nkb4 = ceil_div(hp.k_words[2] * 8, kKB);
  const int64_t nkb2 = ceil_div(hp.k_words[3] * 16, kKB);
  const int64_t per_tile_k = 12 * nkb16 + 20 * nkb8 + 21 * nkb4 + 16 * nkb2;
  const int64_t tiles = (int64_t)hp.tiles[0] + hp.tiles[1] + hp.tiles[2] + hp.tiles[3];
  return (int64_t)hp.tiles[0] * 238 + (int64_t)hp.tiles[1] * 277 + (int64_t)hp.tiles[2] * 534 +
         (int64_t)hp.tiles[3] * 1557 + tiles * per_tile_k;
}
// ... and of one zone-C block of 16 rows (fp16 K and V: about half a class-16 tile)
constexpr int kZoneCBlockCost = 800;

__device__ __forceinline__ const rdkv_plan_header* plan_header(const void* plan) {
  return reinterpret_cast<const rdkv_plan_header*>(plan);
}
__device__ __forceinline__ const rdkv_head_plan* plan_heads(const void* plan) {
  return reinterpret_cast<const rdkv_head_plan*>(static_cast<const char*>(plan) + plan_header(plan)->heads_off);
}
__device__ __forceinline__ const int16_t* plan_slots(const void* plan) {
  return reinterpret_cast<const int16_t*>(static_cast<const char*>(plan) + plan_header(plan)->slots_off);
}

// Tile byte size of V width vbits for a head (same rule as the plan kernel): K codes, then for
// vbits < 16 the V codes and the V metadata.
__host__ __device__ inline int tile_bytes_of(int row_words, int head_dim, int vbits) {
  int b = 4 * kTile * row_words;
  if (vbits < 16) b += (kTile * head_dim * vbits) / 8 + 4 * head_dim;
  return b;
}

// Decode workspace: one partial result (m, l, o of the G query heads) per block, G (D + 2) floats
// rounded up to four, then the per-head tickets, the status word and the fused step's head counter.
__host__ __device__ constexpr int decode_partial_stride(int G, int D) { return (G * (D + 2) + 3) / 4 * 4; }
__host__ __device__ inline int64_t decode_ticket_bytes(int64_t n_heads) { return align_up((n_heads + 2) * 4, 256); }

// Element offset of row `row` of head `head` in zone C: contiguous [heads][cap][D], or, with a page
// table, row row % 16 of page pages[head * stride + row / 16] of a pool [pages][16][D].
constexpr int kZoneCPageRows = RDKV_ZONE_C_PAGE_ROWS;
__host__ __device__ inline int64_t zone_c_offset(const int32_t* pages, int stride, int cap, int head, int row, int D) {
  return pages ? ((int64_t)pages[(int64_t)head * stride + row / kZoneCPageRows] * kZoneCPageRows + row % kZoneCPageRows) * D
               : ((int64_t)head * cap + row) * D;
}

// Byte offset in the zone-A pool of byte o of a cache's zone A: o itself (contiguous), or through the
// cache's page table (pages of RDKV_ZONE_A_PAGE_BYTES).  A staged copy that crosses a page boundary
// is split there (zone_a_run gives the bytes left in o's page).
constexpr int64_t kZoneAPageBytes = RDKV_ZONE_A_PAGE_BYTES;
__host__ __device__ inline int64_t zone_a_offset(const int32_t* pages, int64_t o) {
  return pages ? (int64_t)pages[o / kZoneAPageBytes] * kZoneAPageBytes + o % kZoneAPageBytes : o;
}
__host__ __device__ inline int64_t zone_a_run(const int32_t* pages, int64_t o) {
  return pages ? kZoneAPageBytes - o % kZoneAPageBytes : INT64_MAX;
}
// Element offset (of D fp16) of zone-B row r: r * D, or through the page table (16-row pages).
constexpr int kZoneBPageRows = RDKV_ZONE_B_PAGE_ROWS;
__host__ __device__ inline int64_t zone_b_offset(const int32_t* pages, int64_t r, int D) {
  return (pages ? (int64_t)pages[r / kZoneBPageRows] * kZoneBPageRows + r % kZoneBPageRows : r) * D;
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
