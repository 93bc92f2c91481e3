// Tensor-core passes of the RDKV token weights (gist.science/ko/paper/2605.08317,
// section 2.1: w_t = sum over query positions of the attention a_{tau,t}) for
// fp16 inputs, on the 5th-generation tensor cores.
//
// Both passes multiply a stationary block of 128 rows (operand A) by a stream
// of 256-row tiles (operand B), tile = A . B^T into a 128 x 256 fp32 tensor
// memory accumulator:
//   pass 1  A = 128 query rows of head h, B = key tiles t <= tau.  The epilogue
//           keeps, per query row, the running max and sum of 2^(s*c) and writes
//           -lse2, lse2 = log2 sum_t 2^(s_t * c), c = log2(e)/sqrt(D).
//   pass 2  A = 128 keys of KV head j, B = query tiles tau >= t of the G heads
//           of the group.  The epilogue adds 2^(s*c - lse2[tau]) per key:
//           the column sums of the attention, i.e. w_t; then g_t = w_t * sigma_t.
// Pass 1 also takes the channel weights' sums of squares (section 2.1:
// w_c = ||Q_:,c|| ||K_:,c|| / sqrt(D)) from the tiles it already holds: once the
// producer warp has issued its last load, it sums q^2 per channel over the
// block's 128 query rows, and in one block per (KV head, 256-key tile) k^2 over
// that tile (the block's last), each into its own partial (no atomics).
// Roles (576 threads): warp 0 loads tiles with TMA into a 2-stage ring of 64 KB
// stages; warp 1 issues tcgen05.mma (one thread) into two 256-column TMEM
// accumulators; warps 2..17 read the accumulators back (four warps per TMEM
// lane quarter, one per 64-column slice, so every SM sub-partition interleaves
// four of them) and run the softmax arithmetic.  Every wait is bounded: a wait that
// runs out writes NaN into the affected outputs, which the allocation reports
// as invalid gains.
#include <cuda.h>

#include "common.cuh"

namespace rdkv {

rdkv_status launch_channel_weights(const rdkv_shape* s, const float* qpart, int nq, const float* kpart, int nk,
                                   float* w_chan, cudaStream_t st);

namespace tc {

constexpr int kRows = 128;       // rows of A (the stationary block)
constexpr int kCols = 256;       // rows of a streamed B tile = columns of a tile product (MMA N)
constexpr int kStages = 2;       // TMA ring depth (2 x 64 KB of B tiles)
constexpr int kAcc = 2;          // TMEM accumulators (2 x 256 columns: all of tensor memory)
constexpr int kEpiWarps = 16;                 // epilogue warps: 4 per TMEM lane quarter
constexpr int kSlices = kEpiWarps / 4;        // column slices of the accumulator
constexpr int kSliceCols = kCols / kSlices;   // columns per epilogue warp (multiple of 32)
constexpr int kThreads = 64 + 32 * kEpiWarps; // producer, MMA, epilogue warps
constexpr int kBlocksPerSM = 1;
static_assert(kCols % kRows == 0, "a key tile spans whole row blocks");
constexpr long long kWait = 4000000000ll;

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t c) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(c) : "memory");
}
__device__ __forceinline__ void mbar_expect(uint64_t* b, uint32_t tx) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(tx) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
// A waiting thread sleeps inside try_wait (woken when the phase completes) for up to this long
// per attempt, instead of spinning on the issue slots the epilogue needs.
constexpr uint32_t kSuspendNs = 20000;
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity) {
  const long long t0 = clock64();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity), "r"(kSuspendNs)
        : "memory");
    if (ok) return true;
    if (clock64() - t0 > kWait) return false;
  }
}
__device__ __forceinline__ void tma4(void* dst, const CUtensorMap* m, int c0, int c1, int c2, int c3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(su32(dst)),
      "l"((uint64_t)m), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(su32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   su32(dst)),
               "l"(src), "r"(bytes), "r"(su32(bar))
               : "memory");
}
// Shared-memory matrix descriptor: K-major operand written by TMA with the
// 128-byte swizzle (8-row x 128-byte atoms, 1024 bytes apart).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) |
         ((uint64_t)2 << 61);
}
// Instruction descriptor: fp32 accumulate, fp16 A and B, both K-major, M = N = 128.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kCols >> 3) << 17) | ((uint32_t)(kRows >> 4) << 24);

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 32 consecutive accumulator columns of this thread's TMEM lane.
// Paired fp32 arithmetic (two lanes of work per instruction): a * b + c and a + b, elementwise.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n .reg .b64 pa, pb, pc, pd;\n mov.b64 pa, {%2, %3};\n mov.b64 pb, {%4, %5};\n mov.b64 pc, {%6, %7};\n"
      " fma.rn.f32x2 pd, pa, pb, pc;\n mov.b64 {%0, %1}, pd;\n}\n"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 r;
  asm("{\n .reg .b64 pa, pb, pd;\n mov.b64 pa, {%2, %3};\n mov.b64 pb, {%4, %5};\n add.rn.f32x2 pd, pa, pb;\n"
      " mov.b64 {%0, %1}, pd;\n}\n"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

__device__ __forceinline__ void tmem_ld32(uint32_t ta, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(ta));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

struct Params {
  int N, n_blk, h_q, h_kv, G, Np, lse_stride;
  float c;             // log2(e) / sqrt(D)
  float* lse2;         // [B][H_q][lse_stride]: -log2 sum_t 2^(s c) per query row (negated)
  const float* sigma;  // [B][H_kv][N]
  float* w_tok;        // [B][H_kv][N]
  float* g_tok;        // [B][H_kv][Np]
  float* qsq;          // pass 1: [B][n_blk][H_q][D] sums of q^2 over each 128-row block, or NULL
  float* ksq;          // pass 1: [B][n_kt][H_kv][D] sums of k^2 over each 256-key tile
  int n_kt;            // 256-key tiles: ceil(N / kCols)
};

// Sums of x^2 per channel over `rows` rows of a K-major fp16 tile written by TMA with the 128-byte
// swizzle (64-column halves `rows` x 128 bytes apart; in a half, row r's 16-byte chunk c sits at
// chunk c ^ (r & 7)).  Lane l takes channels D/32 * l ..; rows in order.
template <int D>
__device__ __forceinline__ void channel_squares(const uint8_t* tile, int rows, int lane, float (&acc)[D / 32]) {
  constexpr int CPL = D / 32;
  const int c0 = lane * CPL;
  const uint8_t* half = tile + (c0 / 64) * rows * 128;
  const int chunk = (c0 % 64) / 8, within = (c0 % 8) * 2;
#pragma unroll
  for (int i = 0; i < CPL; ++i) acc[i] = 0.f;
  for (int r = 0; r < rows; ++r) {
    const uint8_t* p = half + r * 128 + ((chunk ^ (r & 7)) << 4) + within;
    if (CPL == 4) {
      const uint2 w = *reinterpret_cast<const uint2*>(p);
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
      const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
      acc[0] = fmaf(a.x, a.x, acc[0]);
      acc[1 % CPL] = fmaf(a.y, a.y, acc[1 % CPL]);
      acc[2 % CPL] = fmaf(c.x, c.x, acc[2 % CPL]);
      acc[3 % CPL] = fmaf(c.y, c.y, acc[3 % CPL]);
    } else {
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(p));
      acc[0] = fmaf(a.x, a.x, acc[0]);
      acc[1 % CPL] = fmaf(a.y, a.y, acc[1 % CPL]);
    }
  }
}

template <int D, int PASS>
__global__ void __launch_bounds__(kThreads, kBlocksPerSM) score_kernel(const __grid_constant__ CUtensorMap tmA,
                                                             const __grid_constant__ CUtensorMap tmB, Params P) {
  constexpr int kHalves = D / 64;                 // 64-element (128-byte) column halves of a row
  constexpr uint32_t kTileBytes = kRows * D * 2;   // the A block (128 rows)
  constexpr uint32_t kBTileBytes = kCols * D * 2;  // one streamed B tile (256 rows)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* As = sm;
  uint8_t* Bs = sm + kTileBytes;                           // [kStages][B tile]
  float* lse_s = reinterpret_cast<float*>(Bs + kStages * kBTileBytes);  // [kAcc][kCols] (pass 2)
  __shared__ uint64_t bar_a, full[kStages], empty[kStages], tfull[kAcc], tempty[kAcc], lfull[kAcc], lempty[kAcc];
  __shared__ uint32_t tmem_base;
  __shared__ int failed;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.z;
  // pass 1: A = queries of head h = blockIdx.y, block qb; pass 2: A = keys of KV head j = blockIdx.y, block kb
  const int blk = PASS == 1 ? P.n_blk - 1 - (int)blockIdx.x : (int)blockIdx.x;  // heaviest blocks first
  const int row0 = blk * kRows;
  // pass 1: key tiles [i kCols, (i+1) kCols) up to the block's last row; pass 2: per head of the
  // group, query tiles from the block's first key on
  const int nt2 = ceil_div(P.N - row0, kCols);
  const int n_tiles = PASS == 1 ? ceil_div(row0 + kRows, kCols) : P.G * nt2;
  auto tile_of = [&](int i, int& head, int& t0) {
    if (PASS == 1) {
      head = blockIdx.y / P.G;   // KV head of query head blockIdx.y
      t0 = i * kCols;
    } else {
      head = blockIdx.y * P.G + i / nt2;
      t0 = row0 + (i % nt2) * kCols;
    }
  };

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&tmem_base)), "n"(kAcc * kCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 32) {
    mbar_init(&bar_a, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int t = 0; t < kAcc; ++t) {
      mbar_init(&tfull[t], 1);
      mbar_init(&tempty[t], kEpiWarps);
      mbar_init(&lfull[t], 1);
      mbar_init(&lempty[t], kEpiWarps);
    }
    failed = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_base;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    int last_ok = 0;  // lane 0: every load up to the last one was issued
    if (lane == 0) {
      const int a_head = blockIdx.y;
      mbar_expect(&bar_a, kTileBytes);
      for (int hh = 0; hh < kHalves; ++hh) tma4(As + hh * kRows * 128, &tmA, 64 * hh, a_head, row0, b, &bar_a);
      for (int i = 0; i < n_tiles; ++i) {
        const int s = i % kStages;
        if (!mbar_wait(&empty[s], ((i / kStages) & 1) ^ 1)) { failed = 1; break; }
        int head, t0;
        tile_of(i, head, t0);
        mbar_expect(&full[s], kBTileBytes);
        for (int hh = 0; hh < kHalves; ++hh)
          tma4(Bs + s * kBTileBytes + hh * kCols * 128, &tmB, 64 * hh, head, t0, b, &full[s]);
        if (PASS == 2) {
          const int t = i % kAcc;
          if (!mbar_wait(&lempty[t], ((i / kAcc) & 1) ^ 1)) { failed = 1; break; }
          mbar_expect(&lfull[t], kCols * 4);
          bulk_g2s(lse_s + t * kCols, P.lse2 + ((int64_t)b * P.h_q + head) * P.lse_stride + t0, kCols * 4, &lfull[t]);
        }
        if (i == n_tiles - 1) last_ok = 1;
      }
    }
    if (PASS == 1 && P.qsq != nullptr) {
      // channel sums of squares from the tiles this block holds (the A tile stays until the end,
      // and the last B tile is never overwritten): the whole warp, once every load is issued
      last_ok = __shfl_sync(0xffffffffu, last_ok, 0);
      float acc[D / 32];
      const bool a_ok = last_ok && mbar_wait(&bar_a, 0);
      if (a_ok) channel_squares<D>(As, kRows, lane, acc);
      float* qo = P.qsq + (((int64_t)b * P.n_blk + blk) * P.h_q + blockIdx.y) * D + lane * (D / 32);
#pragma unroll
      for (int i = 0; i < D / 32; ++i) qo[i] = a_ok ? acc[i] : __int_as_float(0x7fc00000);
      // keys: the block whose rows start the key tile (its last tile), first query head of the group
      if (blockIdx.y % P.G == 0 && blk % (kCols / kRows) == 0) {
        const int i = n_tiles - 1, s = i % kStages;
        const bool b_ok = last_ok && mbar_wait(&full[s], (i / kStages) & 1);
        if (b_ok) channel_squares<D>(Bs + s * kBTileBytes, kCols, lane, acc);
        float* ko = P.ksq + (((int64_t)b * P.n_kt + blk / (kCols / kRows)) * P.h_kv + blockIdx.y / P.G) * D + lane * (D / 32);
#pragma unroll
        for (int i2 = 0; i2 < D / 32; ++i2) ko[i2] = b_ok ? acc[i2] : __int_as_float(0x7fc00000);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      if (!mbar_wait(&bar_a, 0)) failed = 1;
      for (int i = 0; i < n_tiles && !failed; ++i) {
        const int s = i % kStages, t = i % kAcc;
        if (!mbar_wait(&full[s], (i / kStages) & 1)) { failed = 1; break; }
        if (!mbar_wait(&tempty[t], ((i / kAcc) & 1) ^ 1)) { failed = 1; break; }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t a0 = su32(As), b0 = su32(Bs + s * kBTileBytes);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          // 64-column halves of a row are separate swizzled blocks: +16 KB (A) / +32 KB (B) per half
          const uint32_t ka = (uint32_t)((k >> 2) * kRows * 128 + (k & 3) * 32);
          const uint32_t kb = (uint32_t)((k >> 2) * kCols * 128 + (k & 3) * 32);
          const uint64_t ad = sdesc(a0 + ka), bd = sdesc(b0 + kb);
          asm volatile(
              "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::
                  "r"(tmem + (uint32_t)(t * kCols)),
              "l"(ad), "l"(bd), "r"(kIdesc), "r"(k > 0 ? 1u : 0u));
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         su32(&empty[s]))
                     : "memory");
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         su32(&tfull[t]))
                     : "memory");
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int quarter = warp & 3;            // TMEM lanes this warp may access
    const int colh = (warp - 2) >> 2;        // column slice: warps 2..5 take slice 0, 6..9 slice 1, ...
    const int r = quarter * 32 + lane;       // accumulator row = A row
    const int row = row0 + r;                // query (pass 1) or key (pass 2)
    float m = -INFINITY, l = 0.f;            // pass 1: running max and sum (base 2, scaled logits)
    float acc = 0.f;                         // pass 2: column sum of the attention
    bool ok = true;
    for (int i = 0; i < n_tiles; ++i) {
      const int t = i % kAcc;
      if (!mbar_wait(&tfull[t], (i / kAcc) & 1)) { ok = false; break; }
      if (PASS == 2 && !mbar_wait(&lfull[t], (i / kAcc) & 1)) { ok = false; break; }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      int head, t0;
      tile_of(i, head, t0);
      const uint32_t ta = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(t * kCols + colh * kSliceCols);
#pragma unroll
      for (int ch = 0; ch < kSliceCols / 32; ++ch) {
        float v[32];
        tmem_ld32(ta + 32 * ch, v);
        const int c0 = t0 + colh * kSliceCols + ch * 32;  // first key (pass 1) or query (pass 2) of the chunk
        if (PASS == 1) {
          // valid keys: c <= row (c < N follows for rows < N); only the diagonal tile needs the mask.
          // The max is taken on raw logits (c > 0) and the scale folded into one FMA per element.
          float mx = -INFINITY;
          if (t0 + kCols <= row0) {
#pragma unroll
            for (int e = 0; e < 32; ++e) mx = fmaxf(mx, v[e]);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              v[e] = (c0 + e <= row) ? v[e] : -INFINITY;
              mx = fmaxf(mx, v[e]);
            }
          }
          const float mn = fmaxf(m, mx * P.c);
          if (mn != -INFINITY) {
            // 2^(v c - mn) with the scale-and-shift and the sums on paired fp32 instructions
            const float2 cc = make_float2(P.c, P.c), sh = make_float2(-mn, -mn);
            float2 s0 = make_float2(0.f, 0.f), s1 = s0;
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const float2 x0 = ffma2(make_float2(v[e], v[e + 1]), cc, sh);
              const float2 x1 = ffma2(make_float2(v[e + 2], v[e + 3]), cc, sh);
              s0 = fadd2(s0, make_float2(ex2(x0.x), ex2(x0.y)));
              s1 = fadd2(s1, make_float2(ex2(x1.x), ex2(x1.y)));
            }
            const float2 st = fadd2(s0, s1);
            l = l * ex2(m - mn) + (st.x + st.y);
            m = mn;
          }
        } else {
          // the staged -lse2 of the chunk's 32 queries, read with explicit shared-memory loads (the
          // aligned dynamic shared-memory base is computed through an integer, so a plain dereference
          // would be a generic load)
          const uint32_t ls_a = su32(lse_s + t * kCols + colh * kSliceCols + ch * 32);
          auto ls4_at = [&](int e4) {
            float4 r;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w) : "r"(ls_a + 16 * e4));
            return r;
          };
          float a0 = 0.f, a1 = 0.f;
          if (t0 != row0 && t0 + kCols <= P.N) {  // no causal edge and no tail in this tile
            // the staged values are -lse2: 2^(v c - lse2) = 2^(fma(v, c, -lse2)), paired
            const float2 cc = make_float2(P.c, P.c);
            float2 p0 = make_float2(0.f, 0.f), p1 = p0;
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
              const float4 L = ls4_at(e4);
              const float2 x0 = ffma2(make_float2(v[4 * e4 + 0], v[4 * e4 + 1]), cc, make_float2(L.x, L.y));
              const float2 x1 = ffma2(make_float2(v[4 * e4 + 2], v[4 * e4 + 3]), cc, make_float2(L.z, L.w));
              p0 = fadd2(p0, make_float2(ex2(x0.x), ex2(x0.y)));
              p1 = fadd2(p1, make_float2(ex2(x1.x), ex2(x1.y)));
            }
            const float2 pt = fadd2(p0, p1);
            a0 = pt.x;
            a1 = pt.y;
          } else {
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
              const float4 L = ls4_at(e4);
              const float lv[4] = {L.x, L.y, L.z, L.w};
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int c = c0 + 4 * e4 + u;
                const float p = ex2(fmaf(v[4 * e4 + u], P.c, lv[u]));
                a0 += (c >= row && c < P.N) ? p : 0.f;
              }
            }
          }
          acc += a0 + a1;
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&tempty[t]);
        if (PASS == 2) mbar_arrive(&lempty[t]);
      }
    }
    if (!ok) failed = 1;
    // combine the column slices of each row through shared memory (the A tile is free now)
    float* comb = reinterpret_cast<float*>(As);  // [2][kSlices][128] partial values
    __syncwarp();
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");  // every epilogue warp is past its last TMEM read
    const bool bad = failed != 0;
    if (PASS == 1) {
      comb[colh * kRows + r] = m;
      comb[(kSlices + colh) * kRows + r] = l;
      asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
      if (colh == 0 && row < P.N) {
        float mm = -INFINITY;
#pragma unroll
        for (int sl = 0; sl < kSlices; ++sl) mm = fmaxf(mm, comb[sl * kRows + r]);
        float ll = 0.f;
#pragma unroll
        for (int sl = 0; sl < kSlices; ++sl) {
          const float ms = comb[sl * kRows + r];
          if (ms != -INFINITY) ll += comb[(kSlices + sl) * kRows + r] * ex2(ms - mm);
        }
        // stored negated: pass 2 adds it in the same FMA that scales the logit
        P.lse2[((int64_t)b * P.h_q + blockIdx.y) * P.lse_stride + row] = bad ? __int_as_float(0x7fc00000) : -(mm + __log2f(ll));
      }
    } else {
      comb[colh * kRows + r] = acc;
      asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
      if (colh == 0 && row < P.N) {
        float w = 0.f;
#pragma unroll
        for (int sl = 0; sl < kSlices; ++sl) w += comb[sl * kRows + r];
        w = bad ? __int_as_float(0x7fc00000) : w;
        const int64_t o = ((int64_t)b * P.h_kv + blockIdx.y) * P.N + row;
        P.w_tok[o] = w;
        if (row < P.Np) P.g_tok[((int64_t)b * P.h_kv + blockIdx.y) * P.Np + row] = w * P.sigma[o];
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kAcc * kCols));
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  }
  return fn;
}

// [B][N][H][D] fp16 tensor, `rows`-row x 64-column boxes with the 128-byte swizzle.
static rdkv_status make_map(CUtensorMap* m, const void* base, int B, int N, int H, int D, int rows) {
  EncodeTiledFn enc = encode_fn();
  RDKV_REQUIRE(enc != nullptr, RDKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)N * H * D * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)rows, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  RDKV_REQUIRE(r == CUDA_SUCCESS, RDKV_ERR_CUDA, "tensor map encoding failed (%d)", (int)r);
  return RDKV_OK;
}

template <int D>
static size_t smem_bytes() {
  return 1024 + (size_t)kRows * D * 2 + (size_t)kStages * kCols * D * 2 + kAcc * kCols * 4;
}

template <int D>
static rdkv_status launch(const rdkv_shape* s, const void* q, const void* k, const float* sigma, float* lse2,
                          int lse_stride, float* w_tok, float* g_tok, float* qsq, float* ksq, float* w_chan,
                          cudaStream_t st) {
  CUtensorMap mqa, mqb, mka, mkb;  // 128-row boxes (stationary A) and 256-row boxes (streamed B)
  rdkv_status e = make_map(&mqa, q, s->batch, s->n_tokens, s->h_q, D, kRows);
  if (e == RDKV_OK) e = make_map(&mqb, q, s->batch, s->n_tokens, s->h_q, D, kCols);
  if (e == RDKV_OK) e = make_map(&mka, k, s->batch, s->n_tokens, s->h_kv, D, kRows);
  if (e == RDKV_OK) e = make_map(&mkb, k, s->batch, s->n_tokens, s->h_kv, D, kCols);
  if (e != RDKV_OK) return e;
  Params P;
  P.N = s->n_tokens;
  P.n_blk = ceil_div(s->n_tokens, kRows);
  P.h_q = s->h_q;
  P.h_kv = s->h_kv;
  P.G = s->h_q / s->h_kv;
  P.Np = s->n_tokens - s->window;
  P.lse_stride = lse_stride;
  P.c = 1.4426950408889634f / sqrtf((float)D);
  P.lse2 = lse2;
  P.sigma = sigma;
  P.w_tok = w_tok;
  P.g_tok = g_tok;
  P.qsq = qsq;
  P.ksq = ksq;
  P.n_kt = ceil_div(s->n_tokens, kCols);
  const size_t smem = smem_bytes<D>();
  static bool attr_set[2] = {false, false};
  if (!attr_set[0]) {
    RDKV_TRY_CUDA(cudaFuncSetAttribute(score_kernel<D, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
                  "score smem");
    RDKV_TRY_CUDA(cudaFuncSetAttribute(score_kernel<D, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
                  "score smem");
    attr_set[0] = attr_set[1] = true;
  }
  score_kernel<D, 1><<<dim3(P.n_blk, s->h_q, s->batch), kThreads, smem, st>>>(mqa, mkb, P);
  RDKV_CHECK_LAUNCH("row log-sum-exp (tensor cores)");
  const rdkv_status cw = launch_channel_weights(s, qsq, P.n_blk, ksq, P.n_kt, w_chan, st);
  if (cw != RDKV_OK) return cw;
  score_kernel<D, 2><<<dim3(P.n_blk, s->h_kv, s->batch), kThreads, smem, st>>>(mka, mqb, P);
  RDKV_CHECK_LAUNCH("attention column sums (tensor cores)");
  return RDKV_OK;
}

}  // namespace tc

// Row stride of the lse workspace: a streamed tile starts at a multiple of 128 below N and stages
// kCols values, up to 128 past the rounded-up length.
int score_tc_lse_stride(int n_tokens) { return ceil_div(n_tokens, tc::kRows) * tc::kRows + (tc::kCols - tc::kRows); }

rdkv_status launch_score_tc(const rdkv_shape* s, const void* q, const void* k, const float* sigma, float* lse2,
                            float* w_tok, float* g_tok, float* qsq, float* ksq, float* w_chan, cudaStream_t st) {
  RDKV_REQUIRE(((uintptr_t)q % 16) == 0 && ((uintptr_t)k % 16) == 0, RDKV_ERR_INVALID_ARG,
               "q and k must be 16-byte aligned for the tensor-core scorer");
  const int ls = score_tc_lse_stride(s->n_tokens);
  if (s->head_dim == 128) return tc::launch<128>(s, q, k, sigma, lse2, ls, w_tok, g_tok, qsq, ksq, w_chan, st);
  return tc::launch<64>(s, q, k, sigma, lse2, ls, w_tok, g_tok, qsq, ksq, w_chan, st);
}

// Partial sizes of the tensor-core path's channel sums: q over 128-row blocks, k over 256-key tiles.
int score_tc_q_chunks(int n_tokens) { return ceil_div(n_tokens, tc::kRows); }
int score_tc_k_chunks(int n_tokens) { return ceil_div(n_tokens, tc::kCols); }

}  // namespace rdkv
