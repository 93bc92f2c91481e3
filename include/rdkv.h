/*
 * rdkv.h — C ABI of the RDKV hot path on one GPU (sm_103a).
 *
 * RDKV ("RDKV - KV 캐시 공동 추방 및 양자화를 위한 왜곡-비트 할당",
 * gist.science/ko/paper/2605.08317) compresses a KV cache after prefill by
 *   section 2.1  distortion weights: w_t (attention mass a token receives) for
 *                V tokens, w_c = |Q_:,c| |K_:,c| / sqrt(d) for K channels;
 *   section 2.2  discrete reverse water-filling (Lagrangian relaxation of a
 *                multiple-choice knapsack) over widths {0,2,4,8,16}: V tokens
 *                first, then K channels of the kept tokens;
 *   section 2.3  the TriZone layout: zone A packed 2/4/8-bit rows grouped by
 *                width, zone B fp16 V rows of 16-bit tokens, zone C fp16 rows
 *                of new tokens; decode attention dequantises inside the
 *                products and reads the three zones in one pass.
 * The quantiser is the asymmetric min-max formula of "Matematika KV Cache
 * Compression" (aistudio.id), section "Solusi 3".
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     allocates no device memory.  Scratch memory is passed in as `ws` with
 *     the size the matching *_workspace_bytes() call returns.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous on that stream unless stated otherwise.
 *   - Tensors are dense, row-major, little-endian.  fp16 = IEEE binary16.
 *   - Shapes: B = batch, N = prompt tokens, H_q, H_kv query/KV heads
 *     (G = H_q / H_kv), D = head_dim (64 or 128), W = window,
 *     N_p = N - W allocatable prefix tokens.
 *   - Errors: a call that returns anything but RDKV_OK launched nothing
 *     (argument errors) or hit a CUDA error (RDKV_ERR_CUDA); the message is
 *     in rdkv_last_error_string() (thread-local).
 */
#ifndef RDKV_H
#define RDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rdkv_status {
  RDKV_OK = 0,
  RDKV_ERR_INVALID_ARG = 1,   /* bad pointer, size, budget or (device-side) gain */
  RDKV_ERR_UNSUPPORTED = 2,   /* dtype / head_dim / group size outside the supported set */
  RDKV_ERR_CAPACITY = 3,      /* zone C is full (rdkv_append) */
  RDKV_ERR_CUDA = 4,          /* a CUDA runtime error */
  RDKV_ERR_TIMEOUT = 5,       /* a bounded device-side wait ran out */
  RDKV_ERR_WORKSPACE = 6      /* ws too small */
} rdkv_status;

enum { RDKV_F16 = 0, RDKV_F32 = 1 };

/* Problem shape.  Q, K, V of the prefill are [B][N][H][D] in `dtype`. */
typedef struct rdkv_shape {
  int32_t batch, n_tokens, h_q, h_kv, head_dim, window, dtype;
} rdkv_shape;

/* One (sequence, KV head) of the plan, written by rdkv_allocate (device memory).
 * Token classes are V widths 2,4,8,16; K segments are widths 16,8,4,2. */
typedef struct rdkv_head_plan {
  int32_t n_v[4];        /* kept prefix tokens of each V width */
  int32_t tiles[4];      /* 32-token tiles of each V width: ceil(n_v / 32) */
  int32_t n_k[5];        /* channels of K width 16, 8, 4, 2, 0 */
  int32_t k_words[4];    /* 32-bit words per K row in the 16/8/4/2-bit segments */
  int32_t row_words;     /* sum of k_words */
  int32_t k_slots;       /* channel slots of a K row (kept channels + pads) */
  int32_t meta_slots;    /* slots of the 8/4/2-bit segments (those carry scale/zero) */
  int32_t tile_bytes[4]; /* zone-A bytes of one tile of each V width */
  int64_t a_off;         /* byte offset of this head's first tile in zone A */
  int64_t a_bytes;       /* zone-A bytes of this head */
  int64_t b_row;         /* first zone-B row of this head */
  int64_t slot_off;      /* first index-map slot of this head */
} rdkv_head_plan;        /* 128 bytes */

/* Head of the device plan buffer.  The buffer continues with
 *   rdkv_head_plan heads[n_heads]                 (heads in (b, j) order)
 *   int16_t slot_channel[n_heads][slot_stride]    (channel of each K slot, -1 = pad)
 *   float levels[2][batch * h_kv]                 (water levels found; see rdkv_allocate_mode)
 * at the offsets given by the fields below. */
typedef struct rdkv_plan_header {
  int32_t status;          /* RDKV_OK, or RDKV_ERR_INVALID_ARG if a gain was NaN/inf/negative */
  int32_t n_heads;         /* batch * h_kv */
  int32_t batch, h_kv, head_dim, slot_stride;
  int64_t heads_off, slots_off, lambda_off;   /* byte offsets inside the plan buffer */
  int64_t zone_a_bytes;    /* zone-A bytes of the whole batch */
  int64_t zone_b_rows;     /* zone-B rows (each D fp16) */
  int64_t index_slots;     /* index-map entries */
  int64_t kept_tokens;     /* kept prefix tokens over all heads */
  int64_t max_tile_bytes;  /* largest zone-A tile present */
  int64_t max_stage_bytes; /* largest tile plus the zone-B rows it carries (decode staging) */
} rdkv_plan_header;

/* Heads whose decode work rdkv_plan_sizes estimates for the host (see rdkv_sizes). */
#define RDKV_COST_HEADS 64

/* Host copy of the totals, from rdkv_plan_sizes.  head_cost[h], for the first
 * min(n_heads, RDKV_COST_HEADS) (sequence, KV head) pairs in plan order, is an
 * estimate (> 0, arbitrary units) of the zone-A decode work of that head; the
 * decode calls deal their blocks to the heads in proportion to it on the host.
 * When it is not filled (zeros: more than RDKV_COST_HEADS heads, or a record
 * built by hand) the decode kernel deals the blocks itself from the plan.  Only
 * the speed of the decode depends on these numbers, never its result. */
typedef struct rdkv_sizes {
  int64_t zone_a_bytes, zone_b_rows, index_slots, kept_tokens, max_tile_bytes, max_stage_bytes;
  int32_t status, n_heads;
  int32_t head_cost[RDKV_COST_HEADS];
} rdkv_sizes;

/* Rows of one zone-C page when zone C is paged (see rdkv_cache). */
#define RDKV_ZONE_C_PAGE_ROWS 16
/* Bytes of one zone-A page and rows of one zone-B page when zones A and B are
 * paged (see rdkv_cache). */
#define RDKV_ZONE_A_PAGE_BYTES 65536
#define RDKV_ZONE_B_PAGE_ROWS 16

/* A packed TriZone cache.  All pointers are caller-owned device memory.
 * zone_c_k / zone_c_v are fp16 [batch][h_kv][cap_c][D], or, when
 * zone_c_pages is not NULL, pools of pages [n_pages][RDKV_ZONE_C_PAGE_ROWS][D]
 * (the PagedAttention block table of "Matematika KV Cache Compression",
 * "Solusi 1"): row r of head h = b * h_kv + j is row
 * r % 16 of page zone_c_pages[h * zone_c_page_stride + r / 16].  The table
 * (int32, device) must name a distinct page for every 16-row block a head may
 * use (up to cap_c rows, so zone_c_page_stride >= ceil(cap_c / 16)); the
 * kernels read it when they touch zone C.  The number of zone-C
 * rows in use (same for every sequence) is kept twice: len_dev (one device
 * int32) is what the kernels read and advance, so a captured CUDA graph of
 * append + decode calls stays correct when replayed; len_c is the host mirror
 * the host-side capacity check uses.  rdkv_pack sets both to the window W;
 * rdkv_append advances both.  Replaying captured appends advances only
 * len_dev; a device-side append past cap_c writes nothing.
 *
 * Zones A and B may live in pages of pools shared by several caches (the same
 * block table idea, applied to the zones the pack writes): when zone_a_pages is
 * not NULL, byte o of the cache's zone A (the plan's offsets, a_off and up) is
 * byte o % RDKV_ZONE_A_PAGE_BYTES of page zone_a_pages[o / RDKV_ZONE_A_PAGE_BYTES]
 * of the pool at zone_a (pages of RDKV_ZONE_A_PAGE_BYTES bytes); when
 * zone_b_pages is not NULL, zone-B row r is row r % 16 of page
 * zone_b_pages[r / 16] of the pool at zone_b ([n_pages][16][D] fp16).  The
 * tables (int32, device) name a distinct page for every page the cache's sizes
 * need (ceil(zone_a_bytes / RDKV_ZONE_A_PAGE_BYTES), ceil(zone_b_rows / 16));
 * rdkv_pack writes through them and the decode calls read through them.
 * Caches of sequences with different prompt lengths can so share one pool and
 * be attended in one launch (rdkv_decode_ragged). */
typedef struct rdkv_cache {
  rdkv_shape shape;
  const void* plan;
  uint8_t* zone_a;
  uint16_t* zone_b;
  uint16_t* zone_c_k;
  uint16_t* zone_c_v;
  int32_t* index_map;
  int32_t* len_dev;
  int32_t cap_c;
  int32_t len_c;
  rdkv_sizes sizes;
  const int32_t* zone_c_pages;  /* NULL: contiguous zone C; else its page table */
  int32_t zone_c_page_stride;   /* table entries per head */
  const int32_t* zone_a_pages;  /* NULL: contiguous zone A; else its page table */
  const int32_t* zone_b_pages;  /* NULL: contiguous zone B; else its page table */
} rdkv_cache;

/* ---------------------------------------------------------------- misc */
const char* rdkv_last_error_string(void);
int32_t rdkv_version(void);
/* Number of CUDA kernels this library has launched (or recorded into a graph
 * being captured) in this process, over all threads. */
uint64_t rdkv_launch_count(void);

/* ---------------------------------------------------------------- workspace sizes
 * One workspace query for the calls that take a shape (no counterpart in the
 * paper).  which_call:
 *   RDKV_CALL_SCORE     the same value as rdkv_score_workspace_bytes(shape);
 *   RDKV_CALL_ALLOCATE  the same value as rdkv_allocate_workspace_bytes(shape)
 *                       (also enough for rdkv_allocate_mode and
 *                       rdkv_allocate_at_levels on that shape);
 *   RDKV_CALL_DECODE    an upper bound of rdkv_decode_workspace_bytes(cache)
 *                       for every single cache of this shape on the current
 *                       device (the exact value depends on the cache's plan:
 *                       query it once the plan's sizes are known).
 * Returns 0 for an invalid shape or an unknown call.  Host only. */
enum { RDKV_CALL_SCORE = 0, RDKV_CALL_ALLOCATE = 1, RDKV_CALL_DECODE = 2 };
size_t rdkv_workspace_bytes(const rdkv_shape* shape, int32_t which_call);

/* ---------------------------------------------------------------- step 1: weights
 * RDKV section 2.1 (and section 2.2 step 1: computed once after prefill on the
 * full cache).  For each sequence b and KV head j (query heads h of group j):
 *   w_tok[b][j][t]  = sum_{h in j} sum_{tau >= t} softmax_t(q_tau,h . k_t / sqrt(D))   (causal)
 *   w_chan[b][j][c] = sqrt(sum_{tau, h in j} q_tau,h,c^2) * sqrt(sum_t k_t,j,c^2) / sqrt(D)
 *   sigma_tok[b][j][t] = population std of v_t,j over its D elements
 *   g_tok[b][j][t]  = fl32(w_tok * sigma_tok) for t < N_p
 * q [B][N][H_q][D], k, v [B][N][H_kv][D] in shape->dtype.  Outputs fp32:
 * w_tok, sigma_tok [B][H_kv][N], w_chan [B][H_kv][D], g_tok [B][H_kv][N_p].
 * Supported: D in {64, 128}, 1 <= G <= 8.  fp16 inputs use tensor cores with
 * fp32 accumulation; fp32 inputs use fp32 CUDA-core arithmetic.  q, k, v must
 * be 16-byte aligned (RDKV_ERR_INVALID_ARG otherwise). */
size_t rdkv_score_workspace_bytes(const rdkv_shape* shape);
rdkv_status rdkv_score(const rdkv_shape* shape, const void* q, const void* k, const void* v,
                       float* w_tok, float* w_chan, float* sigma_tok, float* g_tok,
                       void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- step 2/3: allocation
 * Discrete reverse water-filling (RDKV section 2.2) on n_inst independent
 * instances of n_units gains each: g [n_inst][n_units] fp32 (finite, >= 0).
 * Per instance, with B = floor((double)avg_bits * n_units):
 *   beta_{u,k} = fl32(g_u * s_k), s = (0.375, 0.09375, 0.0146484375, 255/524288)
 *   lambda*    = smallest float32 >= 0 with sum_u b_u(lambda*) <= B
 *   b_u        = width after every upgrade k with beta_{u,k} > lambda*
 * bits [n_inst][n_units] uint8 in {0,2,4,8,16}; lambda_out [n_inst] fp32 (may be NULL).
 * lambda* is found by an 8-bit-per-level bisection of the float32 bit pattern.
 * status_out (device int32, may be NULL) is set to RDKV_ERR_INVALID_ARG if a
 * gain is NaN, infinite or negative (that unit gets 0 bits). */
size_t rdkv_waterfill_workspace_bytes(int32_t n_inst, int64_t n_units);
rdkv_status rdkv_waterfill(int32_t n_inst, int64_t n_units, const float* g, float avg_bits,
                           uint8_t* bits, float* lambda_out, int32_t* status_out,
                           void* ws, size_t ws_bytes, void* stream);

/* Full allocation of a batch (RDKV section 2.2 steps 2 and 3) and the TriZone plan:
 *   V: water-filling of g_tok [B][H_kv][N_p] per sequence (pooled over heads)
 *      with avg_bits_v -> bits_tok [B][H_kv][N_p];
 *   K: sigma_chan [B][H_kv][D] = population std of K over the kept prefix
 *      tokens of the head (0 if none); g_chan = fl32(w_chan * sigma_chan);
 *      water-filling per sequence with avg_bits_k -> bits_chan [B][H_kv][D];
 *   plan: counts, orders and zone offsets (layout above) in `plan`
 *      (rdkv_plan_bytes(shape) bytes of device memory).
 * k is the prefill K [B][N][H_kv][D], 16-byte aligned (RDKV_ERR_INVALID_ARG
 * otherwise; the same holds for rdkv_allocate_mode and rdkv_allocate_at_levels). */
size_t rdkv_plan_bytes(const rdkv_shape* shape);
size_t rdkv_allocate_workspace_bytes(const rdkv_shape* shape);
rdkv_status rdkv_allocate(const rdkv_shape* shape, const float* g_tok, const float* w_chan,
                          const void* k, float avg_bits_v, float avg_bits_k,
                          uint8_t* bits_tok, float* sigma_chan, float* g_chan, uint8_t* bits_chan,
                          void* plan, void* ws, size_t ws_bytes, void* stream);

/* Allocation variants on the same plan, pack and decode (the RDKV page's
 * section 2.2 is the method; the others are a different reading of its scope
 * and two eviction-only baselines the pages compare against).
 *   RDKV_ALLOC_POOLED    the method, as rdkv_allocate (one water level per
 *                        sequence for V and one for K);
 *   RDKV_ALLOC_PER_HEAD  one water level per (sequence, KV head) for V (budget
 *                        floor(avg_bits_v * N_p) per head) and for K (budget
 *                        floor(avg_bits_k * D) per head);
 *   RDKV_ALLOC_TOPK      heavy-hitter eviction (H2O-style): per (sequence, KV
 *                        head), k = floor(floor(avg_bits_v * N_p) / 16) tokens
 *                        are affordable at 16 bits; every prefix token whose
 *                        w_t exceeds lambda, the smallest non-negative level
 *                        at most k weights exceed, is kept at 16 bits (equal
 *                        weights at lambda are all dropped); every K channel
 *                        16 bits;
 *   RDKV_ALLOC_THRESHOLD eviction by a threshold on the weight (KVzap-style):
 *                        prefix tokens with w_t > param kept at 16 bits; every
 *                        K channel 16 bits.
 * w_tok [B][H_kv][N] (rdkv_score's output; used by TOPK and THRESHOLD),
 * g_tok [B][H_kv][N_p] (used by POOLED and PER_HEAD); the other arguments as
 * rdkv_allocate (sigma_chan, g_chan are computed over the kept tokens in every
 * mode).  Levels in the plan: POOLED: V [B] then K [B]; the other modes:
 * V [B*H_kv] then K [B*H_kv] (0 for the K stage of TOPK and THRESHOLD, param
 * for the V stage of THRESHOLD). */
typedef enum rdkv_alloc_mode {
  RDKV_ALLOC_POOLED = 0,
  RDKV_ALLOC_PER_HEAD = 1,
  RDKV_ALLOC_TOPK = 2,
  RDKV_ALLOC_THRESHOLD = 3
} rdkv_alloc_mode;
rdkv_status rdkv_allocate_mode(const rdkv_shape* shape, int mode, float param, const float* w_tok,
                               const float* g_tok, const float* w_chan, const void* k,
                               float avg_bits_v, float avg_bits_k, uint8_t* bits_tok,
                               float* sigma_chan, float* g_chan, uint8_t* bits_chan,
                               void* plan, void* ws, size_t ws_bytes, void* stream);

/* Copies the plan totals to the host.  SYNCHRONISES `stream`.  Returns the
 * plan's device status (RDKV_ERR_INVALID_ARG if a gain was invalid). */
rdkv_status rdkv_plan_sizes(const void* plan, rdkv_sizes* out, void* stream);

/* Upper bounds of the plan totals rdkv_allocate (pooled or per-head levels)
 * can produce for this shape and these budgets, from the budgets alone: no
 * device access, no synchronisation.  Zones sized from them let the whole
 * compression (rdkv_score, rdkv_allocate, rdkv_pack with cache->sizes = the
 * bounds) run as one stream-ordered sequence, capturable in a CUDA graph;
 * rdkv_plan_sizes afterwards gives the exact totals (and the head costs) for
 * the decode.  Not a bound for the eviction baselines of rdkv_allocate_mode
 * (top-k, threshold), nor for the levels of rdkv_allocate_at_levels. */
rdkv_status rdkv_zone_bounds(const rdkv_shape* shape, float avg_bits_v, float avg_bits_k, rdkv_sizes* out);

/* ---------------------------------------------------------------- TriZone pack
 * RDKV section 2.3.  Writes zone A (sizes.zone_a_bytes), zone B
 * (sizes.zone_b_rows x D fp16), the index map (sizes.index_slots int32) and
 * the window rows [0, W) of zone C from the prefill k, v [B][N][H_kv][D];
 * sets cache->len_c = W.  cache->plan must be the plan bits_tok/bits_chan came
 * with; cap_c >= W; cache->sizes the plan's totals or upper bounds of them
 * (rdkv_zone_bounds); k and v 16-byte aligned (else RDKV_ERR_INVALID_ARG).  Bytes are bit-exact with the layout rules:
 * asymmetric min-max codes (aistudio.id "Solusi 3") with fp16 scale/zero. */
rdkv_status rdkv_pack(rdkv_cache* cache, const void* k, const void* v,
                      const uint8_t* bits_tok, const uint8_t* bits_chan, void* stream);

/* ---------------------------------------------------------------- allocation and pack in one launch
 * RDKV section 2.2 steps 2 and 3, then section 2.3, as ONE persistent
 * (cooperative) kernel whose phases are separated by grid-wide barriers: the
 * V water level and widths, the K channel spreads over the kept tokens, the K
 * water level and widths, the plan, the index map, the head K metadata, the
 * zone-A tiles and zone-B rows, the zone-C window and *len_dev = W.  Every
 * output (bits_tok, sigma_chan, g_chan, bits_chan, the plan with its levels
 * and channel statistics, zones A and B, the index map, zone C rows [0, W))
 * is byte-identical to rdkv_allocate (per_head = 0; rdkv_allocate_mode with
 * RDKV_ALLOC_PER_HEAD for per_head = 1) followed by rdkv_pack.
 *
 * cache: as for rdkv_pack, except that cache->plan is the plan buffer this
 *   call WRITES (rdkv_plan_bytes(shape) bytes) and cache->sizes holds the
 *   zones' capacities (zone_a_bytes, zone_b_rows, index_slots; normally
 *   rdkv_zone_bounds for these budgets).  The exact totals (and the head
 *   costs the decode deals its blocks by) come afterwards from
 *   rdkv_plan_sizes; the call itself does not synchronise, so it can be
 *   captured in a CUDA graph.  Sets cache->len_c = W.
 * g_tok, w_chan: rdkv_score's outputs; k, v: the prefill [B][N][H_kv][D],
 *   16-byte aligned.  Outputs as for rdkv_allocate.
 * ws: rdkv_allocate_pack_workspace_bytes(shape, per_head) bytes of device
 *   memory (the call clears the part it needs cleared, asynchronously on
 *   `stream`).
 * Errors: the host checks of rdkv_allocate and rdkv_pack (nothing launched);
 *   RDKV_ERR_UNSUPPORTED when fewer blocks stay resident than there are
 *   water-filling instances.  Device-side outcomes land in the plan status
 *   (read by rdkv_plan_sizes): RDKV_ERR_INVALID_ARG for an invalid gain (the
 *   pack still runs, as rdkv_pack would), RDKV_ERR_CAPACITY when the plan
 *   needs more than a capacity (then nothing is packed), RDKV_ERR_TIMEOUT when
 *   a grid barrier waited past its bound (about two seconds; the outputs are
 *   then not valid). */
size_t rdkv_allocate_pack_workspace_bytes(const rdkv_shape* shape, int32_t per_head);
rdkv_status rdkv_allocate_pack(rdkv_cache* cache, int32_t per_head, const float* g_tok,
                               const float* w_chan, const void* k, const void* v,
                               float avg_bits_v, float avg_bits_k, uint8_t* bits_tok,
                               float* sigma_chan, float* g_chan, uint8_t* bits_chan,
                               void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- append
 * RDKV section 2.3 zone C: writes the new token's k_new, v_new [B][H_kv][D]
 * (shape->dtype) as fp16 rows at row *len_dev of zone C and advances *len_dev
 * and len_c.  Returns RDKV_ERR_CAPACITY (nothing launched) when the host
 * mirror len_c == cap_c. */
rdkv_status rdkv_append(rdkv_cache* cache, const void* k_new, const void* v_new, void* stream);

/* ---------------------------------------------------------------- decode attention
 * RDKV section 2.3: for every sequence b and query head h (KV head h / G),
 *   out[b][h] = sum_t softmax_t(q[b][h] . k^_t / sqrt(D)) v^_t
 * over the kept tokens of zones A (dequantised K and V) and B (fp16 V) and the
 * *len_dev rows of zone C.  q [B][H_q][D] in shape->dtype, out [B][H_q][D]
 * fp32.  Split-K over tiles with an fp32 online softmax; the partial results
 * and per-head tickets live in ws, which must be ZERO-FILLED before its first
 * use: every call leaves the tickets at zero again, so the same ws serves any
 * number of calls (and CUDA-graph replays) without a reset. */
size_t rdkv_decode_workspace_bytes(const rdkv_cache* cache);
rdkv_status rdkv_decode_attn(const rdkv_cache* cache, const void* q, float* out,
                             void* ws, size_t ws_bytes, void* stream);

/* Launch order (rdkv_decode_attn and rdkv_decode_step): the kernel is launched
 * as a programmatic dependent of the kernel before it on `stream`.  Before it
 * waits for that kernel it reads only the plan and zone A (dealing the work,
 * staging tile copies); the query, the new token, zone C and *len_dev are read
 * after the wait.  So the plan and zone A must not be written by the kernel
 * launched immediately before a decode call on the same stream (rdkv_pack ends
 * with a kernel that writes neither); anything else may be. */

/* ---------------------------------------------------------------- decode step
 * RDKV section 2.3, one decode step in one launch: rdkv_append(k_new, v_new)
 * followed by rdkv_decode_attn(q), computed together.  The new token's row
 * enters the attention straight from k_new/v_new; once every block of a head
 * has read zone C, that head's row is stored at row *len_dev, and the last
 * head to finish advances *len_dev (and the call advances the host mirror
 * len_c).  Same q/out layout and workspace (same size, same zero-filled
 * contract) as rdkv_decode_attn.  Returns RDKV_ERR_CAPACITY (nothing
 * launched) when the host mirror len_c == cap_c; a replayed step that finds
 * *len_dev == cap_c attends with the new token but stores nothing and leaves
 * RDKV_ERR_CAPACITY in the status word. */
rdkv_status rdkv_decode_step(rdkv_cache* cache, const void* q, const void* k_new, const void* v_new,
                             float* out, void* ws, size_t ws_bytes, void* stream);

/* Reads the status word the rdkv_decode_attn / rdkv_decode_step calls on this
 * cache and ws left behind since the last read, and clears it.  SYNCHRONISES
 * `stream`.  RDKV_ERR_TIMEOUT means a bounded wait for a tile copy ran out in
 * one of those calls (its output is not valid); RDKV_ERR_CAPACITY means a
 * step found zone C full and did not store its token. */
rdkv_status rdkv_decode_status(const rdkv_cache* cache, const void* ws, void* stream);

/* Failure-detection self-test of the decode (no counterpart in the paper).
 * Runs the rdkv_decode_attn kernel on `cache`, `q`, `out` and `ws` (same
 * layouts and workspace contract) with every stage's barrier armed for 16
 * bytes that no copy delivers, and no copy issued: each warp's bounded wait
 * runs out after `wait_cycles` SM clock cycles (clamped to [1e5, 4e9]; 2e6
 * is about 1 ms), the kernel records RDKV_ERR_TIMEOUT in the status word and
 * returns, as it would if a tile copy never completed.  Nothing faults or
 * hangs and the context stays usable; `out` holds no attention result.
 * rdkv_decode_status then returns RDKV_ERR_TIMEOUT and clears the word.
 * Returns RDKV_ERR_INVALID_ARG for wait_cycles <= 0, else as rdkv_decode_attn
 * for the launch itself.  Asynchronous on `stream`. */
rdkv_status rdkv_decode_timeout_selftest(const rdkv_cache* cache, const void* q, float* out, void* ws,
                                         size_t ws_bytes, int64_t wait_cycles, void* stream);

/* ---------------------------------------------------------------- decode without a workspace
 * No counterpart in the paper: a deployment variant of rdkv_decode_attn.
 * Some callers cannot allocate device memory themselves: a plugin hosted by
 * an engine that owns every device allocation, or code that must not call the
 * allocator on its serving path.  This entry point computes the same output as
 * rdkv_decode_attn, but keeps its scratch (split partials, per-head tickets and
 * the status word) in a fixed 4 MiB array built into the library, which every
 * GPU that loads the library holds until the process exits; it allocates
 * nothing.
 *   - Returns RDKV_ERR_WORKSPACE (nothing launched) when the cache needs more
 *     than 4 MiB of scratch (rdkv_decode_workspace_bytes tells how much).
 *   - The first call on a device looks up the array's device address (and
 *     raises the kernel's shared-memory limit); make that first call before
 *     any stream capture.  The lookup is cached per device for the CUDA
 *     runtime's primary context of that device (the context every call of
 *     this library runs in); host threads may make their first calls at the
 *     same time.
 *   - All calls share the one array and each clears the counters it needs, so
 *     calls that overlap on the GPU (other streams, other threads) race and
 *     must be serialised by the caller.
 *   - The status word of a call lives in that shared array and is not exposed:
 *     if a bounded wait for a tile copy runs out inside this call, nothing
 *     reports it, the call still returns RDKV_OK and its output is undefined.
 *     Callers that need the timeout report use rdkv_decode_attn. */
rdkv_status rdkv_decode_attn_noalloc(const rdkv_cache* cache, const void* q, float* out, void* stream);

/* ---------------------------------------------------------------- zone-C re-compression
 * New tokens start in zone C (RDKV section 2.3); the pages do not say how
 * they later join zones A and B.  These calls move the oldest zone-C rows into
 * a new SEGMENT: a TriZone cache of their own (window 0) packed by rdkv_pack,
 * with token weights from the attention the recent decode queries gave them
 * and widths at the prefill's water levels (section 2.2, the levels kept
 * instead of found again).  The attention over the segments and the live
 * cache is merged from each part's output and log-sum-exp. */

/* rdkv_decode_attn / rdkv_decode_step that also write lse [B][H_q] fp32: the
 * natural log of the softmax denominator, ln sum_t exp(q . k^_t / sqrt(D)),
 * over the same keys (-inf when there are none; out is then 0).  lse is
 * caller-owned device memory; everything else as in the calls without it. */
rdkv_status rdkv_decode_attn_lse(const rdkv_cache* cache, const void* q, float* out, float* lse,
                                 void* ws, size_t ws_bytes, void* stream);
rdkv_status rdkv_decode_step_lse(rdkv_cache* cache, const void* q, const void* k_new, const void* v_new,
                                 float* out, float* lse, void* ws, size_t ws_bytes, void* stream);

/* Attention over the union of disjoint key sets from its parts:
 *   out = sum_i e^(lse_i) out_i / sum_i e^(lse_i),  lse = ln sum_i e^(lse_i)
 * per row.  outs [n_parts][rows][head_dim], lses [n_parts][rows] fp32 device
 * (rows = B * H_q for decode outputs); out [rows][head_dim] and lse_out
 * [rows] (may be NULL) fp32 device.  Parts with lse = -inf weigh 0; a row with
 * no keys in any part gets out 0, lse -inf.  out may alias outs[0]; lse_out
 * must not alias lses. */
rdkv_status rdkv_merge_attn(int32_t n_parts, const float* outs, const float* lses, int64_t rows,
                            int32_t head_dim, float* out, float* lse_out, void* stream);

/* One launch over several caches sharing the query: the softmax over the union
 * of their keys (zones A and B of each, and each one's zone-C rows), the same
 * output rdkv_merge_attn gives from one call per cache, without the extra
 * launches.  parts[0 .. n_parts) (1 <= n_parts <= 8) must share batch, h_q,
 * h_kv, head_dim and dtype; typically the segments moved out of zone C and
 * then the live cache.  q, out, lse (may be NULL) and the workspace contract
 * as rdkv_decode_attn_lse, the workspace sized by
 * rdkv_decode_multi_workspace_bytes for the same list (0 if the list is
 * invalid).  With more than one cache, every cache's sizes must carry its
 * plan costs (rdkv_plan_sizes) and the batch at most RDKV_COST_HEADS heads,
 * else RDKV_ERR_UNSUPPORTED.  rdkv_decode_multi_status reads and clears the
 * status word as rdkv_decode_status does. */
size_t rdkv_decode_multi_workspace_bytes(const rdkv_cache* const* parts, int32_t n_parts);
rdkv_status rdkv_decode_attn_multi(const rdkv_cache* const* parts, int32_t n_parts, const void* q, float* out,
                                   float* lse, void* ws, size_t ws_bytes, void* stream);
rdkv_status rdkv_decode_multi_status(const rdkv_cache* const* parts, int32_t n_parts, const void* ws, void* stream);

/* ---------------------------------------------------------------- ragged batch
 * RDKV section 2.3 for a batch of independent sequences with different prompt
 * lengths (the batching of "Matematika KV Cache Compression", "Solusi 1"): each
 * sequence is its own cache (batch 1, its own n_tokens, plan and zones, often
 * in pages of shared pools), and ONE launch attends all of them:
 *   out[s][h] = sum_t softmax_t(q[s][h] . k^_t / sqrt(D)) v^_t over the keys of
 *   sequence s only (zones A and B and the *len_dev rows of its zone C).
 * seqs[0 .. n_seq) (1 <= n_seq <= 8) must share h_q, h_kv, head_dim and dtype,
 * have batch 1, carry their plan costs (rdkv_plan_sizes), and n_seq * h_kv
 * must be at most RDKV_COST_HEADS, else RDKV_ERR_INVALID_ARG or
 * RDKV_ERR_UNSUPPORTED.  q [n_seq][H_q][D] in the caches' dtype, out
 * [n_seq][H_q][D] fp32, lse [n_seq][H_q] fp32 or NULL; the workspace sized by
 * rdkv_decode_ragged_workspace_bytes for the same list (0 if it is invalid),
 * with the zero-filled contract of rdkv_decode_attn.  rdkv_decode_ragged_status
 * reads and clears the status word as rdkv_decode_status does.  (Append the new
 * tokens with rdkv_append before the call.) */
size_t rdkv_decode_ragged_workspace_bytes(const rdkv_cache* const* seqs, int32_t n_seq);
rdkv_status rdkv_decode_ragged(const rdkv_cache* const* seqs, int32_t n_seq, const void* q, float* out, float* lse,
                               void* ws, size_t ws_bytes, void* stream);
rdkv_status rdkv_decode_ragged_status(const rdkv_cache* const* seqs, int32_t n_seq, const void* ws, void* stream);

/* Takes rows [0, n_move) of every head's zone C out of the cache: copies them
 * to k_out, v_out [B][n_move][H_kv][D] in the cache's dtype (the fp16 values
 * of zone C, widened for fp32 caches; the prefill layout, ready for
 * rdkv_recompress_score, rdkv_allocate_at_levels and rdkv_pack with a shape
 * of n_move tokens, window 0 and the cache's dtype, whose queries are then
 * the model's), moves rows [n_move, len_c) to the front and
 * lowers len_c and *len_dev by n_move.  Requires 0 < n_move <= len_c and
 * len_c - n_move <= n_move (the rows that stay fit in the rows that leave, so
 * the move never overlaps itself), else RDKV_ERR_INVALID_ARG with nothing
 * launched.  Uses the host mirror len_c: do not call it while captured
 * decode steps are pending replay. */
rdkv_status rdkv_zone_c_take(rdkv_cache* cache, int32_t n_move, void* k_out, void* v_out, void* stream);

/* Token weights and gains of moved tokens (reading of section 2.1 for tokens
 * that entered after the prefill): for sequence b, KV head j and moved token t
 *   w_tok[b][j][t] = weight_scale * sum over r < n_recent and the G query heads
 *                    h of group j of
 *                    exp(q_recent[b][r][h] . k[b][t][j] / sqrt(D) - lse_recent[b][r][h])
 * i.e. the attention the recent decode steps gave the token (their lse from
 * rdkv_decode_*_lse), scaled: a prefill weight sums the attention of up to N
 * query rows, so weight_scale = N / n_recent puts the moved tokens on the scale
 * the prefill's water levels were found for.  sigma_tok = population std of
 * the token's V row and g_tok = fl32(w_tok * sigma_tok).  seg: the segment's shape (n_tokens =
 * moved rows, window 0, dtype of k, v); k, v [B][n][H_kv][D]; q_recent
 * [B][n_recent][H_q][D] in q_dtype; lse_recent [B][n_recent][H_q] fp32;
 * outputs [B][H_kv][n] fp32.  All device memory; 1 <= n_recent. */
rdkv_status rdkv_recompress_score(const rdkv_shape* seg, const void* k, const void* v, const void* q_recent,
                                  int32_t q_dtype, const float* lse_recent, int32_t n_recent, float weight_scale,
                                  float* w_tok, float* sigma_tok, float* g_tok, void* stream);

/* Section 2.2 steps 2 and 3 at given water levels: V widths are the
 * Lagrangian choice at lam_v, then sigma_c of each K channel over the kept
 * moved tokens, g_chan = fl32(w_chan * sigma_c) and K widths at lam_k; then
 * the plan, as rdkv_allocate.  levels [2][n_inst] fp32 device: lam_v of every
 * instance, then lam_k; an instance is a sequence (per_head = 0, the pooled
 * levels of rdkv_allocate) or a (sequence, KV head) pair (per_head = 1).  The
 * plan's own levels are set to these.  w_chan is the prefill's [B][H_kv][D];
 * other arguments, outputs and the workspace as rdkv_allocate for the
 * segment's shape. */
rdkv_status rdkv_allocate_at_levels(const rdkv_shape* seg, int32_t per_head, const float* levels,
                                    const float* g_tok, const float* w_chan, const void* k, uint8_t* bits_tok,
                                    float* sigma_chan, float* g_chan, uint8_t* bits_chan, void* plan, void* ws,
                                    size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* RDKV_H */
