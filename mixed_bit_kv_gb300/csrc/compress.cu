// Allocation and TriZone pack of RDKV (gist.science/ko/paper/2605.08317,
// sections 2.2 and 2.3) in ONE persistent launch: the water levels of V tokens
// (step 2), the K channel spreads over the kept tokens and the K water levels
// (step 3), the plan, the index map, the head K metadata, every zone-A tile and
// zone-B row, and the zone-C window.  The phases are separated by grid-wide
// barriers; the launch is cooperative, so every block is resident and each
// barrier is reached by all of them.  The arithmetic is that of the
// one-kernel-per-stage path (the stages in stages.cuh), so the outputs are
// byte-identical to rdkv_allocate (or the per-head levels of
// rdkv_allocate_mode) followed by rdkv_pack.
//
// Phases (grid barriers between them, 8 on a prompt with kept tokens) and how their work is dealt:
//   V water level  instance i gets `per` blocks (the same ones at every level, so each keeps its
//                  instance's bisection state; every block holding an instance computes the
//                  level's digit itself from the level's histogram, and those blocks alone wait for
//                  one another between levels); then the V widths;
//   channel pass 1 items (chunk of 256 tokens, head), beside the plan's V class counts, items
//                  (head, chunk of 8192 tokens); then the chunk combine, items (head, 32
//                  channels); pass 2 and its combine the same way;
//   K stage        one item per head: the block runs its instance's K water-filling by itself
//                  (histograms in shared memory), writes the head's widths, its K class counts
//                  and its slot table;
//   plan records   block 0 builds the head records and the zone offsets while the other blocks
//                  copy the zone-C window;
//   index map      items (head, chunk of 8192 tokens): the chunk's tokens placed at their class's
//                  slots after the counts of the chunks before it; head K metadata, one item per
//                  head;
//   pack           one item per 32-token tile.
#include "stages.cuh"

namespace rdkv {

constexpr int kFusedThreads = 256;
constexpr int kFusedBlocksPerSm = 5;   // by the tile items' shared memory (about 42 KB a block)
constexpr int kIdxChunk = 8192;        // tokens of a counting / index item: 32 per thread

// Grid barrier state (workspace, cleared before every launch).  Each word has a 128-byte line of its
// own.  A grid barrier is two-level: block b arrives on the counter of its group (b mod 32); the
// last block of a group arrives on the top counter; the last group releases every group's flag,
// which only that group's blocks poll (so no line holds more than a group's arrivals and polls).
constexpr int kSyncGroups = 32;
struct alignas(128) SyncWord {
  unsigned int v;
};
struct GridSync {
  SyncWord grp[kSyncGroups];  // arrivals of each group so far (all barriers)
  SyncWord rel[kSyncGroups];  // barriers released, per group
  SyncWord top;               // groups complete so far
  SyncWord group;             // arrivals of the V water-filling's blocks (their own barriers)
  SyncWord abort;             // nonzero: a block gave up waiting, nobody waits any more
  SyncWord done;              // blocks finished (the last one records a timeout in the plan status)
};
static_assert(sizeof(GridSync) == (2 * kSyncGroups + 4) * 128, "one line per word");

struct FusedArgs {
  // inputs (never written by the launch)
  const float* g_tok;   // [B][H_kv][N_p]
  const float* w_chan;  // [B][H_kv][D]
  const void* k;        // [B][N][H_kv][D]
  const void* v;
  int batch, N, h_kv, W, Np;
  Slopes sl;
  // water-filling: instances, units per instance, budgets, blocks per V instance
  int n_inst_v, n_inst_k;
  int64_t units_v, units_k;
  long long budget_v, budget_k;
  int per_v;
  // allocation outputs
  uint8_t* bits_tok;
  float* sigma_chan;
  float* g_chan;
  uint8_t* bits_chan;
  // plan buffer and its layout
  char* plan;
  int64_t heads_off, slots_off, lambda_off, kstat_off;
  int slot_stride;
  // workspace
  GridSync* sync;
  int32_t* status;  // [2]: V and K water-filling status
  unsigned long long* hist_v;  // [4][n_inst_v][256]
  float *part1, *part2, *pmin, *pmax, *mean;
  int* pcnt;
  int nchunk;   // 256-token chunks of the channel passes
  int* ccnt;    // [n_heads][nidx][4] V class counts of each index chunk
  int nidx;     // 8192-token chunks of a head
  int* nk;      // [n_heads][8] K class counts
  // cache
  uint8_t* zone_a;
  uint16_t* zone_b;
  int32_t* index_map;
  uint16_t *zc_k, *zc_v;
  const int32_t *a_pages, *b_pages, *zc_pages;
  int zc_stride, cap_c;
  int32_t* len_dev;
  int64_t cap_a_bytes, cap_b_rows, cap_slots;  // the zones' capacities
  long long wait_cycles;                       // bound of one barrier wait
};

// Polls are relaxed loads; the fence after the last poll makes the acquire (one per barrier, not
// one per poll).
__device__ __forceinline__ unsigned ld_relaxed_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Barrier of a set of blocks on a counter that only grows (every thread of each of them calls it;
// thread 0's `target` is the count at which every block of the set has arrived at this barrier).
// The block's writes so far become visible to every block that returns from the same barrier: one
// arrival (after a fence), then a poll.  The wait is bounded: a block that waits longer than
// `limit` cycles sets the abort flag, and from then on no block waits; the return value is false
// once the flag is set.
__device__ __forceinline__ bool counter_barrier(GridSync* gs, unsigned* ctr, unsigned target, long long limit,
                                                int* flag_s) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    __threadfence();
    atomicAdd(ctr, 1u);
    if (ld_relaxed_gpu(ctr) < target) {
      const long long t0 = clock64();
      unsigned nap = 32;
      while (ld_relaxed_gpu(ctr) < target) {
        if (*(volatile unsigned*)&gs->abort.v || clock64() - t0 > limit) {
          atomicExch(&gs->abort.v, 1u);
          ok = 0;
          break;
        }
        __nanosleep(nap);
        if (nap < 256) nap *= 2;
      }
    }
    __threadfence();
    if (*(volatile unsigned*)&gs->abort.v) ok = 0;
    *flag_s = ok;
  }
  __syncthreads();
  return *flag_s != 0;
}
// All blocks; bar_k (shared, thread 0's) counts the block's grid barriers so far.  Same visibility
// and bound as counter_barrier; the arrival goes through the block's group (see GridSync).
__device__ __forceinline__ bool grid_barrier(GridSync* gs, long long limit, int* flag_s, unsigned* bar_k) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    const unsigned k = ++*bar_k, nb = gridDim.x;
    const unsigned ng = min(nb, (unsigned)kSyncGroups), g = blockIdx.x % ng;
    const unsigned gsize = nb / ng + (g < nb % ng ? 1u : 0u);
    __threadfence();
    if (atomicAdd(&gs->grp[g].v, 1u) == k * gsize - 1) {  // the group's last block
      __threadfence();
      if (atomicAdd(&gs->top.v, 1u) == k * ng - 1) {        // the last group: release them all
        __threadfence();
        for (unsigned q = 0; q < ng; ++q) atomicMax(&gs->rel[q].v, k);
      }
    }
    if (ld_relaxed_gpu(&gs->rel[g].v) < k) {
      const long long t0 = clock64();
      unsigned nap = 32;
      while (ld_relaxed_gpu(&gs->rel[g].v) < k) {
        if (*(volatile unsigned*)&gs->abort.v || clock64() - t0 > limit) {
          atomicExch(&gs->abort.v, 1u);
          ok = 0;
          break;
        }
        __nanosleep(nap);
        if (nap < 256) nap *= 2;
      }
    }
    __threadfence();
    if (*(volatile unsigned*)&gs->abort.v) ok = 0;
    *flag_s = ok;
  }
  __syncthreads();
  return *flag_s != 0;
}

// Small shared scratch of the non-pack phases (placed after the tile items' area).
struct FusedSmall {
  unsigned long long s[9];
  uint32_t h[256];
  int best, flag;
  unsigned bar_k;
  int nk[5], seg_base[4], cnt[4];
  int wtot[4][kFusedThreads / 32];
  int base[4];
  uint8_t bcs[256];
};

template <int D>
__host__ __device__ constexpr size_t fused_small_off() {
  return (pack_smem_bytes_of<D>() + 15) / 16 * 16;
}
template <int D>
__host__ __device__ constexpr size_t fused_smem_bytes() {
  return fused_small_off<D>() + sizeof(FusedSmall);
}

// V water-filling: 4 levels, then the widths.  Blocks [0, n_part) hold the instances' shares
// (instance `inst` of this block, its part x of `per`; inst = -1 elsewhere): after each level they
// wait for one another only (a block barrier when one block does it all); the caller ends the stage
// with a grid barrier.  g: the instances' gains; lam: the levels' output.
__device__ __forceinline__ bool fused_waterfill(const FusedArgs& a, bool ok, int inst, int x, int per, int n_inst,
                                                const float* g, int64_t units, long long budget,
                                                unsigned long long* hist, int32_t* status, uint8_t* bits,
                                                float* lam, FusedSmall& sm) {
  const unsigned n_part = (unsigned)(n_inst * per);
  if (inst >= 0) {
    WfPick st{0u, 0ull};
#pragma unroll 1
    for (int level = 0; level < 4; ++level) {
      unsigned long long* hl = hist + ((int64_t)level * n_inst + inst) * 256;
      if (ok) wf_hist_part(g + (int64_t)inst * units, units, a.sl, level, st.prefix, x, per, sm.h, hl, status);
      if (n_part == 1) __syncthreads();
      else ok = counter_barrier(a.sync, &a.sync->group.v, n_part * (level + 1), a.wait_cycles, &sm.flag) && ok;
      if (ok) st = wf_pick(__ldcg(hl + threadIdx.x), level, budget, st, sm.s, &sm.best);
    }
    if (ok) {
      if (x == 0 && threadIdx.x == 0) lam[inst] = __uint_as_float(st.prefix);
      wf_assign_part(g + (int64_t)inst * units, units, a.sl, st.prefix, x, per, bits + (int64_t)inst * units);
    }
  }
  return ok;
}

// Plan item of a head's K channels: class counts (kept for the records) and the slot table.
__device__ __forceinline__ void k_part_item(const FusedArgs& a, int head, int D, FusedSmall& sm) {
  const int tid = threadIdx.x;
  int16_t* slots = reinterpret_cast<int16_t*>(a.plan + a.slots_off) + (int64_t)head * a.slot_stride;
  for (int i = tid; i < a.slot_stride; i += blockDim.x) slots[i] = -1;
  for (int c = tid; c < D; c += blockDim.x) sm.bcs[c] = a.bits_chan[(int64_t)head * D + c];
  if (tid < 5) sm.nk[tid] = 0;
  __syncthreads();
  plan_count_k(sm.bcs, D, sm.nk);
  __syncthreads();
  if (tid == 0) {
    const int v0[4] = {0, 0, 0, 0}, k5[5] = {sm.nk[0], sm.nk[1], sm.nk[2], sm.nk[3], sm.nk[4]};
    (void)make_head_record(v0, k5, D, sm.seg_base);
    for (int i = 0; i < 5; ++i) a.nk[head * 8 + i] = k5[i];
  }
  __syncthreads();
  plan_slot_table(sm.bcs, D, sm.seg_base, slots);
  __syncthreads();
}

// K stage item of a head (see the kernel).
__device__ __forceinline__ void k_head_item(const FusedArgs& a, int head, int D, float* lam_k, FusedSmall& sm) {
  const int hpi = a.batch * a.h_kv / a.n_inst_k;  // heads of an instance
  const int inst = head / hpi, j = head % hpi;
  const float* g = a.g_chan + (int64_t)inst * a.units_k;
  WfPick st{0u, 0ull};
#pragma unroll 1
  for (int level = 0; level < 4; ++level) {
    wf_hist_part(g, a.units_k, a.sl, level, st.prefix, 0, 1, sm.h, nullptr, a.status + 1);
    st = wf_pick(sm.h[threadIdx.x], level, a.budget_k, st, sm.s, &sm.best);
  }
  if (j == 0 && threadIdx.x == 0) lam_k[inst] = __uint_as_float(st.prefix);
  // this head's D channels are units [j D, (j + 1) D) of its instance
  wf_assign_part(g + (int64_t)j * D, D, a.sl, st.prefix, 0, 1, a.bits_chan + (int64_t)head * D);
  __syncthreads();
  k_part_item(a, head, D, sm);
}

// Plan item (head, chunk c of 8192 tokens): the chunk's V class counts.
__device__ __forceinline__ void count_item(const FusedArgs& a, int head, int c, FusedSmall& sm) {
  const int tid = threadIdx.x;
  if (tid < 4) sm.cnt[tid] = 0;
  __syncthreads();
  int cnt[4] = {0, 0, 0, 0};
  const int t0 = c * kIdxChunk, t1 = min(a.Np, t0 + kIdxChunk);
  count_classes(a.bits_tok + (int64_t)head * a.Np, t0, t1, blockDim.x, tid, cnt);
#pragma unroll
  for (int q = 0; q < 4; ++q) atomicAdd(&sm.cnt[q], cnt[q]);
  __syncthreads();
  if (tid < 4) a.ccnt[((int64_t)head * a.nidx + c) * 4 + tid] = sm.cnt[tid];
  __syncthreads();
}

// Index item (head, chunk c): the chunk's kept tokens at their class's slots, in position order,
// after the class counts of the chunks before it; chunk 0 also writes the pads (-1) of the head's
// last tile of each class.
__device__ __forceinline__ void index_item(const FusedArgs& a, int head, int c, FusedSmall& sm) {
  const int n_heads = a.batch * a.h_kv;
  (void)n_heads;
  const rdkv_head_plan* hp = plan_heads(a.plan) + head;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  // counts of the chunks before this one (warp 0: lane l sums chunks l, l + 32, ...)
  if (wid == 0) {
    int s0 = 0, s1 = 0, s2 = 0, s3 = 0;
    for (int c2 = lane; c2 < c; c2 += 32) {
      const int4 q = __ldcg(reinterpret_cast<const int4*>(a.ccnt) + (int64_t)head * a.nidx + c2);
      s0 += q.x;
      s1 += q.y;
      s2 += q.z;
      s3 += q.w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      s0 += __shfl_xor_sync(0xffffffffu, s0, o);
      s1 += __shfl_xor_sync(0xffffffffu, s1, o);
      s2 += __shfl_xor_sync(0xffffffffu, s2, o);
      s3 += __shfl_xor_sync(0xffffffffu, s3, o);
    }
    if (lane == 0) {
      sm.base[0] = s0;
      sm.base[1] = s1;
      sm.base[2] = s2;
      sm.base[3] = s3;
    }
  }
  // this thread's 32 tokens, in position order
  const uint8_t* bt = a.bits_tok + (int64_t)head * a.Np;
  const int t0 = c * kIdxChunk + 32 * tid;
  int cnt[4] = {0, 0, 0, 0};
  uint32_t cls_bits[2] = {0u, 0u};  // 2-bit class code of each token (class 0..3; width 0 marked apart)
  uint32_t kept = 0;                // bit e: token t0 + e is kept
  // the 32 widths: two 16-byte loads when the run is whole and aligned, else one byte at a time
  uint32_t wv[8];
  if (t0 + 32 <= a.Np && ((uintptr_t)(bt + t0) & 15) == 0) {
    const uint4 x0 = __ldcg(reinterpret_cast<const uint4*>(bt + t0));
    const uint4 x1 = __ldcg(reinterpret_cast<const uint4*>(bt + t0) + 1);
    wv[0] = x0.x; wv[1] = x0.y; wv[2] = x0.z; wv[3] = x0.w;
    wv[4] = x1.x; wv[5] = x1.y; wv[6] = x1.z; wv[7] = x1.w;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t x = 0;
#pragma unroll
      for (int f = 0; f < 4; ++f) {
        const int t = t0 + 4 * i + f;
        x |= (t < a.Np ? (uint32_t)bt[t] : 0u) << (8 * f);
      }
      wv[i] = x;
    }
  }
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const int b = (int)((wv[e >> 2] >> (8 * (e & 3))) & 255u);
    const int cl = b == 2 ? 0 : b == 4 ? 1 : b == 8 ? 2 : b == 16 ? 3 : -1;
    if (cl >= 0) {
      kept |= 1u << e;
      cls_bits[e >> 4] |= (uint32_t)cl << (2 * (e & 15));
      cnt[0] += cl == 0;
      cnt[1] += cl == 1;
      cnt[2] += cl == 2;
      cnt[3] += cl == 3;
    }
  }
  // block-exclusive prefix of the counts, per class
  int excl[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    int x = cnt[q];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) sm.wtot[q][wid] = x;
    excl[q] = x - cnt[q];
  }
  __syncthreads();
  int start[4];
  {
    int acc = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      int before = 0;
      for (int w2 = 0; w2 < wid; ++w2) before += sm.wtot[q][w2];
      excl[q] += before + sm.base[q];
      start[q] = acc;
      acc += kTile * hp->tiles[q];
    }
  }
  int32_t* out = a.index_map + hp->slot_off;
  // each class's next slot, kept in four scalars (no indexed local array); the kept tokens in
  // position order, one loop trip each
  int n0 = start[0] + excl[0], n1 = start[1] + excl[1], n2 = start[2] + excl[2], n3 = start[3] + excl[3];
#pragma unroll 1
  while (kept) {
    const int e = __ffs(kept) - 1;
    kept &= kept - 1u;
    const uint32_t cb = e < 16 ? cls_bits[0] : cls_bits[1];
    const int cl = (int)((cb >> (2 * (e & 15))) & 3u);
    const int pos = cl == 0 ? n0++ : cl == 1 ? n1++ : cl == 2 ? n2++ : n3++;
    out[pos] = t0 + e;
  }
  if (c == 0) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      for (int r = hp->n_v[q] + tid; r < kTile * hp->tiles[q]; r += blockDim.x) out[start[q] + r] = -1;
  }
  __syncthreads();  // sm is free again
}

template <typename T, int D>
__global__ void __launch_bounds__(kFusedThreads, kFusedBlocksPerSm) compress_kernel(const FusedArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  FusedSmall& sm = *reinterpret_cast<FusedSmall*>(smem_raw + fused_small_off<D>());
  ChanSmem& csm = *reinterpret_cast<ChanSmem*>(smem_raw);
  ChanFinishSmem& fsm = *reinterpret_cast<ChanFinishSmem*>(smem_raw);
  const int nb = gridDim.x, bid = blockIdx.x, tid = threadIdx.x;
  const int n_heads = a.batch * a.h_kv;
  float* lam = reinterpret_cast<float*>(a.plan + a.lambda_off);
  float2* kstat = reinterpret_cast<float2*>(a.plan + a.kstat_off);
  const long long lim = a.wait_cycles;
  if (tid == 0) sm.bar_k = 0;
  bool ok = true;

  // ---------------------------------------------------------------- step 2: V tokens
  {
    const bool mine = bid < a.n_inst_v * a.per_v;
    ok = fused_waterfill(a, ok, mine ? bid / a.per_v : -1, mine ? bid % a.per_v : 0, a.per_v, a.n_inst_v, a.g_tok,
                         a.units_v, a.budget_v, a.hist_v, a.status, a.bits_tok, lam, sm);
    ok = grid_barrier(a.sync, lim, &sm.flag, &sm.bar_k) && ok;
  }
  // ---------------------------------------------------------------- step 3: K channel spreads, gains
  if (a.Np > 0) {
    const int dt = sizeof(T) == 2 ? RDKV_F16 : RDKV_F32;
    // the first channel pass and the plan's V class counts (both need only the V widths)
    if (ok)
      for (int it = bid; it < a.nchunk * n_heads + n_heads * a.nidx; it += nb) {
        if (it < a.nchunk * n_heads)
          chan_pass_item(it % a.nchunk, a.nchunk, it / a.nchunk, a.k, a.bits_tok, dt, a.N, a.h_kv, D, a.Np, nullptr,
                         a.part1, a.pcnt, a.pmin, a.pmax, csm);
        else
          count_item(a, (it - a.nchunk * n_heads) / a.nidx, (it - a.nchunk * n_heads) % a.nidx, sm);
      }
    ok = grid_barrier(a.sync, lim, &sm.flag, &sm.bar_k) && ok;
    if (ok)
      for (int it = bid; it < n_heads * (D / 32); it += nb)
        chan_finish_item(it / (D / 32), it % (D / 32), a.part1, a.pcnt, a.nchunk, D, a.mean, nullptr, nullptr,
                         nullptr, a.pmin, a.pmax, kstat, fsm);
    ok = grid_barrier(a.sync, lim, &sm.flag, &sm.bar_k) && ok;
    if (ok)
      for (int it = bid; it < a.nchunk * n_heads; it += nb)
        chan_pass_item(it % a.nchunk, a.nchunk, it / a.nchunk, a.k, a.bits_tok, dt, a.N, a.h_kv, D, a.Np, a.mean,
                       a.part2, nullptr, nullptr, nullptr, csm);
    ok = grid_barrier(a.sync, lim, &sm.flag, &sm.bar_k) && ok;
    if (ok)
      for (int it = bid; it < n_heads * (D / 32); it += nb)
        chan_finish_item(it / (D / 32), it % (D / 32), a.part2, a.pcnt, a.nchunk, D, nullptr, a.w_chan, a.sigma_chan,
                         a.g_chan, nullptr, nullptr, nullptr, fsm);
  } else if (ok) {
    for (int64_t i = (int64_t)bid * blockDim.x + tid; i < (int64_t)n_heads * D; i += (int64_t)nb * blockDim.x) {
      a.sigma_chan[i] = 0.f;
      a.g_chan[i] = 0.f;
      kstat[i] = make_float2(0.f, 0.f);
    }
  }
  ok = grid_barrier(a.sync, lim, &sm.flag, &sm.bar_k) && ok;
  // K water level, widths and plan items, one item per head: the item's block runs the water-filling
  // of the head's instance (at most h_kv D units) by itself, from histograms in shared memory (every
  // block of an instance finds the same level: the digits are exact integer sums), then writes its
  // head's widths (and, for the instance's first head, the level) and the head's K plan items
  if (ok)
    for (int it = bid; it < n_heads; it += nb) k_head_item(a, it, D, lam + a.n_inst_v, sm);
  ok = grid_barrier(a.sync, lim, &sm.flag, &sm.bar_k) && ok;
  // ---------------------------------------------------------------- plan: records and offsets (block 0); window
  if (ok) {
    if (bid == 0) {
      for (int head = tid; head < n_heads; head += blockDim.x) {
        int nv[4] = {0, 0, 0, 0};
        const int4* cc = reinterpret_cast<const int4*>(a.ccnt) + (int64_t)head * a.nidx;
        for (int c = 0; c < a.nidx; ++c) {
          const int4 q = __ldcg(cc + c);
          nv[0] += q.x;
          nv[1] += q.y;
          nv[2] += q.z;
          nv[3] += q.w;
        }
        int k5[5];
        for (int i = 0; i < 5; ++i) k5[i] = __ldcg(a.nk + head * 8 + i);
        reinterpret_cast<rdkv_head_plan*>(a.plan + a.heads_off)[head] = make_head_record(nv, k5, D, nullptr);
      }
      __syncthreads();
      if (tid == 0) {
        plan_offsets_body(a.plan, a.batch, a.h_kv, D, a.slot_stride, a.heads_off, a.slots_off, a.lambda_off,
                          *(volatile int32_t*)&a.status[0], *(volatile int32_t*)&a.status[1]);
        rdkv_plan_header* hdr = reinterpret_cast<rdkv_plan_header*>(a.plan);
        if (hdr->zone_a_bytes > a.cap_a_bytes || hdr->zone_b_rows > a.cap_b_rows || hdr->index_slots > a.cap_slots)
          hdr->status = RDKV_ERR_CAPACITY;
      }
    } else if (a.W > 0) {
      const int64_t i0 = (int64_t)(bid - 1) * blockDim.x + tid, step = (int64_t)(nb - 1) * blockDim.x;
      window_part(static_cast<const T*>(a.k), a.N, a.W, a.h_kv, D, a.cap_c, a.batch, a.zc_k, a.zc_pages, a.zc_stride,
                  i0, step);
      window_part(static_cast<const T*>(a.v), a.N, a.W, a.h_kv, D, a.cap_c, a.batch, a.zc_v, a.zc_pages, a.zc_stride,
                  i0, step);
    }
  }
  ok = grid_barrier(a.sync, lim, &sm.flag, &sm.bar_k) && ok;
  const rdkv_plan_header* hdr = plan_header(a.plan);
  const bool fits = ok && __ldcg(&hdr->status) != RDKV_ERR_CAPACITY;
  // ---------------------------------------------------------------- index map, head K metadata
  if (fits && a.Np > 0) {
    for (int it = bid; it < n_heads * a.nidx + n_heads; it += nb) {
      if (it < n_heads * a.nidx) index_item(a, it / a.nidx, it % a.nidx, sm);
      else head_meta_body(it - n_heads * a.nidx, a.plan, kstat, D, a.zone_a, a.a_pages);
    }
  }
  ok = grid_barrier(a.sync, lim, &sm.flag, &sm.bar_k) && ok;
  // ---------------------------------------------------------------- tiles
  if (fits && ok && a.Np > 0) {
    const int64_t n_tiles = __ldcg(reinterpret_cast<const long long*>(&hdr->index_slots)) / kTile;
    for (int64_t t = bid; t < n_tiles; t += nb)
      pack_tile_item<T, D>(t, static_cast<const T*>(a.k), static_cast<const T*>(a.v), a.plan, kstat, a.index_map,
                           a.zone_a, a.zone_b, a.N, a.h_kv, a.a_pages, a.b_pages, smem_raw);
  }
  // ---------------------------------------------------------------- zone-C length; status of a timeout
  __syncthreads();
  if (tid == 0) {
    if (bid == 0 && ok) *a.len_dev = a.W;
    __threadfence();
    if (atomicAdd(&a.sync->done.v, 1u) == (unsigned)nb - 1) {
      __threadfence();
      if (*(volatile unsigned*)&a.sync->abort.v) reinterpret_cast<rdkv_plan_header*>(a.plan)->status = RDKV_ERR_TIMEOUT;
    }
  }
}

// Workspace: barrier state and status words, the V histograms (these are cleared per call), then the
// channel partials, counts and means, the index chunks' counts and the K class counts.
struct FusedWs {
  size_t sync, hist_v, part, cnt, mean, ccnt, nk, total, clear;
  int nchunk, nidx, n_inst_v, n_inst_k;
};
static FusedWs fused_ws(const rdkv_shape* s, int per_head) {
  FusedWs w;
  const int64_t n_heads = (int64_t)s->batch * s->h_kv;
  const int Np = s->n_tokens - s->window, D = s->head_dim;
  w.n_inst_v = per_head ? (int)n_heads : s->batch;
  w.n_inst_k = w.n_inst_v;
  w.nchunk = std::max(1, ceil_div(Np, kChanChunk));
  w.nidx = ceil_div(Np, kIdxChunk);
  size_t o = 0;
  w.sync = o;
  o += sizeof(GridSync) + 256;  // then the status words, on a line of their own
  w.hist_v = o;
  o += align_up(4 * (int64_t)w.n_inst_v * 256 * 8, 256);
  w.clear = o;
  w.part = o;
  o += 4 * align_up(n_heads * w.nchunk * D * 4, 256);  // part1, part2, pmin, pmax
  w.cnt = o;
  o += align_up(n_heads * w.nchunk * 4, 256);
  w.mean = o;
  o += align_up(n_heads * D * 4, 256);
  w.ccnt = o;
  o += align_up(n_heads * std::max(w.nidx, 1) * 16, 256);
  w.nk = o;
  o += align_up(n_heads * 8 * 4, 256);
  w.total = o;
  return w;
}

template <typename T, int D>
static rdkv_status launch_fused(const FusedArgs& a, cudaStream_t cs, int nb) {
  const size_t smem = fused_smem_bytes<D>();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)nb);
  cfg.blockDim = dim3(kFusedThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = cs;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  RDKV_TRY_CUDA(cudaLaunchKernelEx(&cfg, compress_kernel<T, D>, a), "allocate+pack launch");
  RDKV_CHECK_LAUNCH("allocate+pack");
  return RDKV_OK;
}

// Blocks of the persistent launch: as many as stay resident at once (at most kFusedBlocksPerSm a
// SM, fewer if the registers or shared memory do not allow them).
template <typename T, int D>
static rdkv_status fused_grid(int* nb) {
  const size_t smem = fused_smem_bytes<D>();
  RDKV_TRY_CUDA(cudaFuncSetAttribute(compress_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
                "allocate+pack smem");
  int per_sm = 0;
  RDKV_TRY_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, compress_kernel<T, D>, kFusedThreads, smem),
                "allocate+pack occupancy");
  *nb = std::min(per_sm, kFusedBlocksPerSm) * num_sms();
  return RDKV_OK;
}

rdkv_status check_cache_public(const rdkv_cache* c);

}  // namespace rdkv

using namespace rdkv;

extern "C" size_t rdkv_allocate_pack_workspace_bytes(const rdkv_shape* s, int32_t per_head) {
  if (check_shape(s) != RDKV_OK || (per_head != 0 && per_head != 1)) return 0;
  return fused_ws(s, per_head).total;
}

extern "C" rdkv_status rdkv_allocate_pack(rdkv_cache* cache, int32_t per_head, const float* g_tok,
                                          const float* w_chan, const void* k, const void* v, float avg_bits_v,
                                          float avg_bits_k, uint8_t* bits_tok, float* sigma_chan, float* g_chan,
                                          uint8_t* bits_chan, void* ws, size_t ws_bytes, void* stream) {
  rdkv_status st = check_cache_public(cache);
  if (st != RDKV_OK) return st;
  const rdkv_shape* s = &cache->shape;
  RDKV_REQUIRE(per_head == 0 || per_head == 1, RDKV_ERR_INVALID_ARG, "per_head must be 0 or 1 (%d)", per_head);
  RDKV_REQUIRE(std::isfinite(avg_bits_v) && avg_bits_v >= 0 && std::isfinite(avg_bits_k) && avg_bits_k >= 0,
               RDKV_ERR_INVALID_ARG, "budgets must be finite and >= 0 (v=%f k=%f)", (double)avg_bits_v,
               (double)avg_bits_k);
  const int Np = s->n_tokens - s->window, D = s->head_dim;
  RDKV_REQUIRE(w_chan && k && v && bits_chan && sigma_chan && g_chan && (Np == 0 || (bits_tok && g_tok)),
               RDKV_ERR_INVALID_ARG, "NULL pointer argument");
  RDKV_REQUIRE(reinterpret_cast<uintptr_t>(k) % 16 == 0 && reinterpret_cast<uintptr_t>(v) % 16 == 0,
               RDKV_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
  const FusedWs w = fused_ws(s, per_head);
  RDKV_REQUIRE(ws && ws_bytes >= w.total, RDKV_ERR_WORKSPACE, "allocate+pack workspace too small (%zu < %zu)",
               ws_bytes, w.total);
  int nb = 0;
  rdkv_status gst = s->dtype == RDKV_F16 ? (D == 128 ? fused_grid<__half, 128>(&nb) : fused_grid<__half, 64>(&nb))
                                          : (D == 128 ? fused_grid<float, 128>(&nb) : fused_grid<float, 64>(&nb));
  if (gst != RDKV_OK) return gst;
  RDKV_REQUIRE(nb >= std::max(w.n_inst_v, 2), RDKV_ERR_UNSUPPORTED,
               "%d water-filling instances need as many resident blocks (%d)", w.n_inst_v, nb);
  const int64_t n_heads = (int64_t)s->batch * s->h_kv;
  char* wsb = static_cast<char*>(ws);
  const PlanLayout L = plan_layout(s->batch, s->h_kv, D);
  FusedArgs a;
  a.g_tok = g_tok;
  a.w_chan = w_chan;
  a.k = k;
  a.v = v;
  a.batch = s->batch;
  a.N = s->n_tokens;
  a.h_kv = s->h_kv;
  a.W = s->window;
  a.Np = Np;
  a.sl = slopes_of(kRdkvSlopes);
  a.n_inst_v = w.n_inst_v;
  a.n_inst_k = w.n_inst_k;
  a.units_v = per_head ? (int64_t)Np : (int64_t)s->h_kv * Np;
  a.units_k = per_head ? (int64_t)D : (int64_t)s->h_kv * D;
  a.budget_v = (long long)std::floor((double)avg_bits_v * (double)a.units_v);
  a.budget_k = (long long)std::floor((double)avg_bits_k * (double)a.units_k);
  // blocks per V instance: about 16 units a thread, as the stage kernels take them
  a.per_v = (int)std::min<int64_t>(std::max<int64_t>(ceil_div64(a.units_v, 256 * 16), 1), nb / a.n_inst_v);
  a.bits_tok = bits_tok;
  a.sigma_chan = sigma_chan;
  a.g_chan = g_chan;
  a.bits_chan = bits_chan;
  a.plan = static_cast<char*>(const_cast<void*>(cache->plan));
  a.heads_off = L.heads_off;
  a.slots_off = L.slots_off;
  a.lambda_off = L.lambda_off;
  a.kstat_off = L.kstat_off;
  a.slot_stride = L.slot_stride;
  a.sync = reinterpret_cast<GridSync*>(wsb + w.sync);
  a.status = reinterpret_cast<int32_t*>(wsb + w.sync + sizeof(GridSync));
  a.hist_v = reinterpret_cast<unsigned long long*>(wsb + w.hist_v);
  const size_t pb = align_up(n_heads * w.nchunk * D * 4, 256);
  a.part1 = reinterpret_cast<float*>(wsb + w.part);
  a.part2 = reinterpret_cast<float*>(wsb + w.part + pb);
  a.pmin = reinterpret_cast<float*>(wsb + w.part + 2 * pb);
  a.pmax = reinterpret_cast<float*>(wsb + w.part + 3 * pb);
  a.pcnt = reinterpret_cast<int*>(wsb + w.cnt);
  a.mean = reinterpret_cast<float*>(wsb + w.mean);
  a.nchunk = w.nchunk;
  a.ccnt = reinterpret_cast<int*>(wsb + w.ccnt);
  a.nidx = w.nidx;
  a.nk = reinterpret_cast<int*>(wsb + w.nk);
  a.zone_a = cache->zone_a;
  a.zone_b = cache->zone_b;
  a.index_map = cache->index_map;
  a.zc_k = cache->zone_c_k;
  a.zc_v = cache->zone_c_v;
  a.a_pages = cache->zone_a_pages;
  a.b_pages = cache->zone_b_pages;
  a.zc_pages = cache->zone_c_pages;
  a.zc_stride = cache->zone_c_page_stride;
  a.cap_c = cache->cap_c;
  a.len_dev = cache->len_dev;
  a.cap_a_bytes = cache->sizes.zone_a_bytes;
  a.cap_b_rows = cache->sizes.zone_b_rows;
  a.cap_slots = cache->sizes.index_slots;
  a.wait_cycles = 4000000000ll;
  cudaStream_t cs = (cudaStream_t)stream;
  RDKV_TRY_CUDA(cudaMemsetAsync(ws, 0, w.clear, cs), "allocate+pack workspace clear");
  if (s->dtype == RDKV_F16)
    st = D == 128 ? launch_fused<__half, 128>(a, cs, nb) : launch_fused<__half, 64>(a, cs, nb);
  else
    st = D == 128 ? launch_fused<float, 128>(a, cs, nb) : launch_fused<float, 64>(a, cs, nb);
  if (st != RDKV_OK) return st;
  cache->len_c = s->window;
  return RDKV_OK;
}
