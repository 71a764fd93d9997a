// Decode / verify step (T <= 16 tokens): every distinct routed expert and
// the shared expert run once for all tokens routed to them (a verify batch
// shares one fetch of each expert, page "单卡5090跑125B 大模型", §2.3),
//   g = Wg.x, u = Wu.x, h = silu(g) * u, o = Wd.h,
//   y[t] = shared_weight * o_shared[t] + sum_i w[t,i] * o_idx[t,i][t].
//
// Fused routing: the same launch first computes the router logits (CTA c
// takes rows c, c + G, ...), passes a grid-wide arrival counter, and then
// every CTA selects the experts of the call from the full logits itself (the
// same selection as the routing kernel), so no second kernel and no plan
// round trip separate routing from the expert work.  With every key resident
// CTA 0 also takes tiles and publishes the plan, stamps and counters from
// its h-loader warp.  With a cache that can miss, CTA 0 takes no tiles and
// runs the cache (LRU victims, commit, next LRU order, plan), and CTAs
// 1..G-1 pull the call's misses from the host pool into their victim slots
// before the experts.  Otherwise (host-issued miss copies) the kernel
// follows the routing kernel and reads its plan.
//
// Work is cut into tiles of contiguous bytes of the device block layout:
//   gate/up tile (expert a, 32-row block rb of f): the Wg and Wu blocks of
//     every input group (2 * d/32 blocks, 57 KB at d = 2048); it produces
//     h = silu(g) * u for 32 rows of expert a (fp16, [expert][token][f]) and
//     bumps h_ready[a];
//   down tile (expert a, R consecutive 32-row blocks of d): R * f/32 Wd blocks
//     (R = 2 at f = 768); it multiplies by h_a and writes o_a for its rows.
// One persistent CTA per SM (but CTA 0 with a cache that can miss) takes an
// even share of each phase: a contiguous range of gate/up tiles, then a
// contiguous range of down tiles.  A producer
// thread streams every tile through a ring of 16-block stages with bulk TMA
// copies (mbarrier completion); an h-loader thread bulk-copies each expert's
// h into shared memory once per CTA when it is ready.  All 8 consumer warps
// work on every gate/up stage (2 blocks each): they expand the 3-bit codes to fp16 in
// registers and multiply on the tensor cores (mma.sync m16n8k16, fp32
// accumulate, per-group scale in fp32); in a down tile each warp sums one
// row block.  They hand each tile's partial sums to a finalizer warp that
// adds them in a fixed order, writes h or o and publishes it.  The tile CTA
// of index c then combines the row blocks c, c + G, ... of y once
// every expert's output there is written, in a fixed order (shared expert,
// then routed experts in ascending id), so y is deterministic.  All waits are
// bounded.
#include "common.cuh"
#include "internal.h"
#include "select.cuh"
#include "repack.cuh"

namespace moe {

#ifdef MOE_TIMELINE
__device__ unsigned long long g_ffn_timeline[512][32];
#endif

constexpr int kCW = 8;                        // consumer warps
constexpr int kThreads = (kCW + 3) * 32;      // + producer, h-loader and finalizer warps
constexpr int kStageBlocks = 16;
constexpr int kStageBytes = kStageBlocks * kBlockBytes;   // 7,168
constexpr int kHSlots = 2;
constexpr int kTabPerThread = (kMaxE + kThreads - 1) / kThreads;   // slot-table entries per thread
constexpr int kXPerThread = 4;                // 16-byte x chunks per thread loaded up front

template <int NT>
struct FfnCfg {
  static constexpr int kStages = NT == 1 ? 20 : 10;
};

// row blocks per down tile: the smallest R with R * (f/32) a multiple of 16
__host__ __device__ __forceinline__ int down_rows_per_tile(int f) {
  const int dg = f / 32;
  int r = 1;
  while ((r * dg) % kStageBlocks) ++r;
  return r;
}

__host__ __device__ __forceinline__ int h_row_bytes(int f) { return (f + 8) * 2; }

// elements per staged x row: 32 bytes of padding put the 4 token rows that
// one fragment-building load touches on distinct banks
__host__ __device__ __forceinline__ int x_row_elems(int d) { return d + 16; }

// floats per lane of one warp's partials: gate/up 16 per token tile, down 8
// per token tile (each warp sums one row block); +4 keeps 16-byte vectors
// aligned and the 8 lanes of each 128-byte access on distinct banks
__host__ __device__ __forceinline__ int red_per_lane(int nt) { return 16 * nt + 4; }

template <int NT>
__host__ __device__ __forceinline__ size_t ffn_smem_bytes(int d, int f) {
  return (size_t)NT * d * 16 + (size_t)FfnCfg<NT>::kStages * kStageBytes +
         (size_t)kHSlots * NT * 8 * h_row_bytes(f) + (size_t)kCW * 32 * red_per_lane(NT) * 4 +
         (2 * FfnCfg<NT>::kStages + 2 * kHSlots + 2) * 8 + 64;
}

__device__ __forceinline__ uint32_t pack_half2_from_bf16(uint32_t two_bf16) {
  const __half2 h = __floats2half2_rn(bf16_bits_to_float(two_bf16 & 0xffffu), bf16_bits_to_float(two_bf16 >> 16));
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void scales4(const uint8_t* bp, int lane, float s[4]) {
  const uint2 sc = *reinterpret_cast<const uint2*>(bp + kBlockCodeBytes + (lane >> 2) * 8);
  const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&sc.x));
  const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&sc.y));
  s[0] = lo.x;   // row g
  s[1] = lo.y;   // row g+8
  s[2] = hi.x;   // row g+16
  s[3] = hi.y;   // row g+24
}

// One 32x32 block: D[nt][mt] = A_block . B_frag[nt] (fp32, unscaled) and the
// scales of the lane's rows g, g+8, g+16, g+24.
template <int NT>
__device__ __forceinline__ void block_products(const uint8_t* bp, int lane, const uint2 (&bx)[NT][2],
                                               float (&D)[NT][2][4], float (&s)[4]) {
  const uint32_t* wp = reinterpret_cast<const uint32_t*>(bp);
  const uint32_t w0 = wp[lane], w1 = wp[32 + lane], w2 = wp[64 + lane];
  scales4(bp, lane, s);
  uint32_t A[16];
  dequant_block(w0, w1, w2, A);
  const float zero[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      mma_16816(D[nt][mt], &A[mt * 8], bx[nt][0].x, bx[nt][0].y, zero);
      mma_16816(D[nt][mt], &A[mt * 8 + 4], bx[nt][1].x, bx[nt][1].y, D[nt][mt]);
    }
  }
}

// acc[nt][mt][i] += scale(row) * D[nt][mt][i]
template <int NT>
__device__ __forceinline__ void block_accum(const float (&D)[NT][2][4], const float (&s)[4], float (&acc)[NT][2][4]) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const float sa = s[2 * mt], sb = s[2 * mt + 1];
      acc[nt][mt][0] = fmaf(sa, D[nt][mt][0], acc[nt][mt][0]);
      acc[nt][mt][1] = fmaf(sa, D[nt][mt][1], acc[nt][mt][1]);
      acc[nt][mt][2] = fmaf(sb, D[nt][mt][2], acc[nt][mt][2]);
      acc[nt][mt][3] = fmaf(sb, D[nt][mt][3], acc[nt][mt][3]);
    }
  }
}

template <int NT>
__device__ __forceinline__ void block_mma(const uint8_t* bp, int lane, const uint2 (&bx)[NT][2],
                                          float (&acc)[NT][2][4]) {
  float D[NT][2][4], s[4];
  block_products<NT>(bp, lane, bx, D, s);
  block_accum<NT>(D, s, acc);
}

template <int NT>
__device__ __forceinline__ void zero_acc(float (&acc)[NT][2][4]) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[nt][mt][i] = 0.f;
}

// B fragments of the down product from h in shared memory (token rows padded)
template <int NT>
__device__ __forceinline__ void h_frags(const uint8_t* hb, int hrow, int T, int gi, int lane, uint2 (&bx)[NT][2]) {
  const int gq = lane >> 2, cq = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int tok = nt * 8 + gq;
    const uint8_t* hr = hb + (size_t)tok * hrow + (gi * 32 + 2 * cq) * 2;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      if (tok < T) {
        bx[nt][ks].x = *reinterpret_cast<const uint32_t*>(hr + ks * 32);
        bx[nt][ks].y = *reinterpret_cast<const uint32_t*>(hr + ks * 32 + 16);
      } else {
        bx[nt][ks] = make_uint2(0u, 0u);
      }
    }
  }
}

// bytes of the routing-phase scratch kept in the (not yet used) stage ring
__host__ __device__ __forceinline__ size_t route_scratch_bytes(int E) {
  return ((sizeof(SelSmem) + 15) & ~size_t(15)) + (size_t)E * 4;
}

// MODE kPlanRead: the routing plan comes from memory (routing kernel and
// host-issued miss copies before this launch).  kFusedResident: routing in
// this kernel, every key resident.  kFusedCached: routing in this kernel with
// a cache that may miss; CTA 0 manages the cache (LRU victims, the next LRU
// order, commit, plan) while CTAs 1..G-1 pull the misses from the host pool,
// re-lay them out into their victim slots and run the experts.
// exclusive prefix sum over the kThreads threads of the CTA (every thread
// calls it); s_warp holds kThreads/32 + 1 ints
__device__ __forceinline__ int cta_exclusive_scan(int v, int* s_warp, int* total) {
  constexpr int NW = kThreads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) s_warp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int wv = lane < NW ? s_warp[lane] : 0;
    int wi = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    if (lane < NW) s_warp[lane] = wi - wv;
    if (lane == NW - 1) s_warp[NW] = wi;
  }
  __syncthreads();
  const int r = s_warp[warp] + inc - v;
  *total = s_warp[NW];
  __syncthreads();   // s_warp may be reused
  return r;
}

// Cache of a layer-call with fused routing, run by every thread of CTA 0
// (which takes no tiles).  LRU by (layer, expert), ties to the lower slot id
// (page "单卡5090跑125B 大模型", §2.1 and §7.2): U = the call's distinct
// experts (ascending); resident ones are hits; the misses, in ascending
// expert id, take the least recently used slots in (stamp, slot id) order,
// which is the order of q (least recent first) with the hits skipped.  The
// call's touched slots (hits and victims) move, in slot-id order, to the
// recent end of q.  The victims are published first (xbar[0]), because CTAs
// 1..G-1 wait for them before pulling the misses; then the commit (table,
// owners, stamps), the next order, the plan and the statistics.
// `scratch` is shared memory this CTA does not otherwise use.
__device__ __forceinline__ void cache_manager(const FfnArgs& a, int n_act, int m, const int* s_act_expert,
                                              int* s_act_slot, const int* s_pick_act, const float* s_w,
                                              long long clk, uint32_t calls, uint8_t* scratch,
                                              size_t scratch_bytes, uint32_t* xbar) {
  __shared__ int s_warp[kThreads / 32 + 1];
  __shared__ int s_evict;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.T, K = a.k, C = a.C;
  const int c_words = (C + 31) / 32;
  Plan* P = a.plan;
  int32_t* table = const_cast<int32_t*>(a.table);
  // scratch: four per-pick arrays, the touched-slot bitmap, then (if it
  // fits) the staged LRU order
  int* s_miss_ai = reinterpret_cast<int*>(scratch);
  int* s_victim = s_miss_ai + kMaxPicks;
  int* s_old = s_victim + kMaxPicks;
  int* s_hitf = s_old + kMaxPicks;
  uint32_t* bits = reinterpret_cast<uint32_t*>(s_hitf + kMaxPicks);
  const size_t head = (size_t)4 * kMaxPicks * 4;
  const size_t bits_bytes = ((size_t)c_words * 4 + 15) & ~size_t(15);
  int32_t* sq = head + bits_bytes + (size_t)C * 4 <= scratch_bytes
                    ? reinterpret_cast<int32_t*>(scratch + head + bits_bytes)
                    : nullptr;
  for (int i = tid; i < c_words; i += kThreads) bits[i] = 0;
  if (sq) {   // the LRU order staged with 16-byte loads, all in flight
    const int n4 = C >> 2;
    const int4* src4 = reinterpret_cast<const int4*>(a.q_in);
#pragma unroll 4
    for (int i = tid; i < n4; i += kThreads) reinterpret_cast<int4*>(sq)[i] = __ldcg(src4 + i);
    for (int i = 4 * n4 + tid; i < C; i += kThreads) sq[i] = a.q_in[i];
  }
  for (int i = tid; i < n_act; i += kThreads) s_hitf[i] = s_act_slot[i] >= 0;
  if (warp == 0) {   // the misses in ascending expert id
    int base = 0;
    for (int i0 = 0; i0 < n_act; i0 += 32) {
      const int i = i0 + lane;
      const bool miss = i < n_act && s_act_slot[i] < 0;
      const uint32_t bal = __ballot_sync(0xffffffffu, miss);
      if (miss) s_miss_ai[base + __popc(bal & ((1u << lane) - 1u))] = i;
      base += __popc(bal);
    }
  }
  if (tid == 0) s_evict = 0;
  __syncthreads();
  for (int i = tid; i < n_act; i += kThreads) {
    const int sl = s_act_slot[i];
    if (sl >= 0) atomicOr(&bits[sl >> 5], 1u << (sl & 31));
  }
  __syncthreads();
  const int32_t* q_in = sq ? sq : a.q_in;
  // walk q skipping the hits: the first m slots are the victims, the rest
  // keep their order at the front of the next q
  const int chunk = (C + kThreads - 1) / kThreads;
  const int lo = min(C, tid * chunk), hi = min(C, lo + chunk);
  int cnt = 0;
  for (int i = lo; i < hi; ++i) {
    const int sl = q_in[i];
    cnt += !((bits[sl >> 5] >> (sl & 31)) & 1u);
  }
  int total;
  int r = cta_exclusive_scan(cnt, s_warp, &total);
  for (int i = lo; i < hi; ++i) {
    const int sl = q_in[i];
    if (!((bits[sl >> 5] >> (sl & 31)) & 1u)) {
      if (r < m) s_victim[r] = sl;
      else a.q_out[r - m] = sl;
      ++r;
    }
  }
  __syncthreads();
  for (int j = tid; j < m; j += kThreads) {
    const int v = s_victim[j];
    const int ai = s_miss_ai[j];
    const int old = a.owner[v];
    atomicOr(&bits[v >> 5], 1u << (v & 31));
    s_old[j] = old;
    s_act_slot[ai] = v;
    P->miss_expert[j] = s_act_expert[ai];
    P->miss_slot[j] = v;
    P->evicted_key[j] = old;
  }
  __syncthreads();
  for (int i = tid; i < n_act; i += kThreads) {
    P->act_slot[i] = s_act_slot[i];
    P->act_hit[i] = s_hitf[i];
    P->act_expert[i] = s_act_expert[i];
  }
  __syncthreads();
  if (m > 0 && tid == 0) {
    MOE_TL(g_ffn_timeline, 0, 28);
    red_release_add(&xbar[0], 1u);   // covers the plan's victim entries (after the barrier)
  }
  // commit: evicted keys leave the table before the misses enter it
  for (int j = tid; j < m; j += kThreads) {
    const int old = s_old[j];
    if (old >= 0) {
      table[old] = -1;
      atomicAdd(&s_evict, 1);
    }
  }
  __syncthreads();
  for (int j = tid; j < m; j += kThreads) {
    const int v = s_victim[j];
    const int key = a.layer * a.E + s_act_expert[s_miss_ai[j]];
    a.owner[v] = key;
    table[key] = v;
    a.stamp[v] = clk;
  }
  for (int i = tid; i < n_act; i += kThreads)
    if (s_hitf[i]) a.stamp[s_act_slot[i]] = clk;
  // touched slots (hits and victims) in ascending slot id to the recent end
  const int wchunk = (c_words + kThreads - 1) / kThreads;
  const int wlo = min(c_words, tid * wchunk), whi = min(c_words, wlo + wchunk);
  int tc = 0;
  for (int i = wlo; i < whi; ++i) tc += __popc(bits[i]);
  int tr = cta_exclusive_scan(tc, s_warp, &total);
  for (int i = wlo; i < whi; ++i) {
    uint32_t b = bits[i];
    while (b) {
      const int bit = __ffs(b) - 1;
      b &= b - 1;
      a.q_out[C - n_act + tr] = i * 32 + bit;
      ++tr;
    }
  }
  // the plan's routing part and the counts
  for (int i = tid; i < T * K; i += kThreads) {
    P->idx[i] = s_act_expert[s_pick_act[i]];
    P->w[i] = s_w[i];
    P->pick_act[i] = s_pick_act[i];
  }
  const int th = __syncthreads_count(tid < T * K && s_hitf[s_pick_act[tid]]);
  if (tid == 0) {
    P->n_act = n_act;
    P->n_miss = m;
    P->T = T;
    P->clock = clk;
    P->token_hits = th;
    P->token_misses = (int64_t)T * K - th;
    a.stats[ST_CALLS] += 1;
    a.stats[ST_TOK_HIT] += th;
    a.stats[ST_TOK_MISS] += (int64_t)T * K - th;
    a.stats[ST_DIST_HIT] += n_act - m;
    a.stats[ST_DIST_MISS] += m;
    a.stats[ST_EVICT] += s_evict;
    a.stats[ST_MISS_BYTES] += (int64_t)m * a.expert_bytes;
    *a.clock = clk + 1;
    *a.counters = calls + 1;   // every CTA read the count before the router barrier
  }
}

// One arrival of this CTA on a grid counter, then the wait for all GT CTAs
// (bounded); false if the wait gave up.  Every thread calls it.
__device__ __forceinline__ bool cta_grid_barrier(uint32_t* bar, uint32_t GT, uint32_t* err, int* s_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    red_release_add(bar, 1u);   // covers this CTA's writes (after the block barrier)
    const bool ok = wait_flag_geq(bar, GT);
    if (!ok) set_error(err, DEV_TIMEOUT_FLAG);
    *s_flag = ok;
  }
  __syncthreads();
  return *s_flag != 0;
}

// CTAs 1..G-1 (index ct of GT) of a call with m > 0 misses: wait for CTA 0's
// victims, pull the misses' canonical bytes from the host pool into
// staging, a grid barrier, re-lay them out into their victim slots, a grid
// barrier.  False if a wait gave up (the error word is set).
__device__ __forceinline__ bool pull_and_place_misses(const FfnArgs& a, int m, int n_act, int* s_act_slot,
                                                      uint32_t* xbar, int GT, int ct, uint8_t* scratch) {
  int* s_mslot = reinterpret_cast<int*>(scratch);   // shared memory not yet in use by the tiles
  int* s_mexp = s_mslot + kMaxPicks;
  __shared__ int s_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Plan* P = a.plan;
  if (m > a.staging_n) {   // cannot happen (m <= T*k and m <= E); never write past the staging slots
    if (tid == 0) set_error(a.err, DEV_BAD_PLAN);
    return false;
  }
  if (tid == 0) {
    const bool ok = wait_flag_geq(&xbar[0], 1u);
    if (!ok) set_error(a.err, DEV_TIMEOUT_FLAG);
    s_flag = ok;
  }
  __syncthreads();
  if (!s_flag) return false;
  if (tid == 0) MOE_TL(g_ffn_timeline, blockIdx.x, 29);
  for (int j = tid; j < m; j += kThreads) {
    s_mslot[j] = __ldcg(&P->miss_slot[j]);
    s_mexp[j] = __ldcg(&P->miss_expert[j]);
  }
  for (int i = tid; i < n_act; i += kThreads)
    if (s_act_slot[i] < 0) s_act_slot[i] = __ldcg(&P->act_slot[i]);
  __syncthreads();
  // host pool -> staging, 16 bytes per thread and step, four loads in flight
  const int64_t per = a.expert_bytes / 16;
  const int64_t nthr = (int64_t)GT * kThreads;
  for (int j = 0; j < m; ++j) {
    const int64_t entry = ((int64_t)a.layer * a.E + s_mexp[j]) % a.pool_entries;
    const uint4* src = reinterpret_cast<const uint4*>(a.host_pool + entry * a.expert_bytes);
    uint4* dst = reinterpret_cast<uint4*>(a.staging + (int64_t)j * a.expert_bytes);
    int64_t c = (int64_t)ct * kThreads + tid;
    for (; c + 3 * nthr < per; c += 4 * nthr) {
      const uint4 v0 = src[c], v1 = src[c + nthr], v2 = src[c + 2 * nthr], v3 = src[c + 3 * nthr];
      dst[c] = v0;
      dst[c + nthr] = v1;
      dst[c + 2 * nthr] = v2;
      dst[c + 3 * nthr] = v3;
    }
    for (; c < per; c += nthr) dst[c] = src[c];
  }
  if (!cta_grid_barrier(&xbar[1], (uint32_t)GT, a.err, &s_flag)) return false;
  if (tid == 0) MOE_TL(g_ffn_timeline, blockIdx.x, 30);
  // staging -> victim slots in the device block layout, one block per warp
  const int nb = (a.f / 32) * (a.d / 32) * 2 + (a.d / 32) * (a.f / 32);
  const int64_t nwarps = (int64_t)GT * (kThreads / 32);
  uint8_t* slots = const_cast<uint8_t*>(a.slots);
  for (int64_t gw = (int64_t)ct * (kThreads / 32) + warp; gw < (int64_t)nb * m; gw += nwarps) {
    const int ex = (int)(gw / nb), bi = (int)(gw % nb);
    repack_block(a.staging + (int64_t)ex * a.expert_bytes, slots + (int64_t)s_mslot[ex] * a.expert_bytes, bi, a.d,
                 a.f, lane);
  }
  const bool ok = cta_grid_barrier(&xbar[2], (uint32_t)GT, a.err, &s_flag);
  if (tid == 0) MOE_TL(g_ffn_timeline, blockIdx.x, 31);
  return ok;
}

template <int NT, int MODE>
__global__ void __launch_bounds__(kThreads, 1) decode_ffn_kernel(FfnArgs a) {
  constexpr bool FUSED = MODE != kPlanRead;
  constexpr bool CACHED = MODE == kFusedCached;
  constexpr int NS = FfnCfg<NT>::kStages;
  extern __shared__ __align__(128) uint8_t smem[];
  const int d = a.d, f = a.f, T = a.T, K = a.k;
  const int RG = f / 32;               // gate/up row blocks (= down input groups)
  const int RD = d / 32;               // down row blocks
  const int DG = f / 32;               // groups per down row block
  const int RT = down_rows_per_tile(f);
  const int nks = d / 16;
  const int hrow = h_row_bytes(f);
  const int SGU = 2 * (d / 32) / kStageBlocks;   // stages per gate/up tile
  const int SDN = RT * DG / kStageBlocks;        // stages per down tile
  uint2* xfrag = reinterpret_cast<uint2*>(smem);
  uint8_t* ring = smem + (size_t)NT * d * 16;
  uint8_t* hbuf = ring + (size_t)NS * kStageBytes;
  const int RPL = red_per_lane(NT);
  const int WPR = kCW / RT;            // consumer warps per row block of a down tile
  float* red = reinterpret_cast<float*>(hbuf + (size_t)kHSlots * NT * 8 * hrow);
  uint64_t* full = reinterpret_cast<uint64_t*>(red + (size_t)kCW * 32 * RPL);
  uint64_t* empty = full + NS;
  uint64_t* hfull = empty + NS;
  uint64_t* hempty = hfull + kHSlots;
  uint64_t& buf_full = hempty[kHSlots];       // 8 consumer warps put a tile's partials
  uint64_t& buf_free = hempty[kHSlots + 1];   // the finalizer has read them
  // routing-phase scratch, overlaid on the stage ring (free until the first copy)
  SelSmem* sel = reinterpret_cast<SelSmem*>(ring);
  int* s_tab = reinterpret_cast<int*>(ring + ((sizeof(SelSmem) + 15) & ~size_t(15)));
  __shared__ int s_act_slot[kMaxPicks];   // slot of each distinct routed expert
  __shared__ int s_pick_act[kMaxPicks];   // [T][k] index of each pick in the distinct list
  __shared__ float s_w[kMaxPicks];        // [T][k] routing weights
  __shared__ int s_act_expert[kMaxPicks]; // expert id of each distinct routed expert (fused routing)
  __shared__ int s_nexp;
  __shared__ uint32_t s_calls;
  __shared__ long long s_clock;
  __shared__ volatile int s_hexp[kHSlots];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  if (tid == 0) MOE_TL(g_ffn_timeline, cta, 0);
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kCW);
    }
    for (int i = 0; i < kHSlots; ++i) {
      mbar_init(&hfull[i], 1);
      mbar_init(&hempty[i], kCW);
      s_hexp[i] = -1;
    }
    mbar_init(&buf_full, kCW);
    mbar_init(&buf_free, 1);
    mbar_init_fence();
  }
  // Every load of the prologue is issued before any of them is used, so the
  // prologue costs about one memory round trip.  Static inputs first: with
  // fused routing the slot table row (every key is resident, so it does not
  // change) and the first block of this warp's router row.
  int tv[kTabPerThread];
  uint4 wfirst[8];
  float wbias = 0.f;
  if (FUSED) {
    if (!CACHED) {
#pragma unroll
      for (int q = 0; q < kTabPerThread; ++q) {
        const int i = tid + q * kThreads;
        tv[q] = i < a.E ? a.table[(size_t)a.layer * a.E + i] : -1;
      }
    }
    const int e = cta + G * warp;
    if (e < a.E) {
      router_load_block(a.wr + (size_t)e * d, 0, d, lane, wfirst);
      wbias = a.bias[e];
    }
    pdl_launch_dependents();
  }
  // x, the clock and the counters may be written by earlier work in the
  // stream
  pdl_wait();
  if (CACHED) {   // the slot table changes with every commit: read it after the previous call
#pragma unroll
    for (int q = 0; q < kTabPerThread; ++q) {
      const int i = tid + q * kThreads;
      tv[q] = i < a.E ? a.table[(size_t)a.layer * a.E + i] : -1;
    }
  }
  uint32_t calls = 0;
  long long clk = 0;
  if (tid == 0) {
    calls = *a.counters;
    if (FUSED && cta == 0) clk = (long long)*a.clock;
  }
  // x (bf16) staged once in shared memory, rows xs apart, in the h / partial
  // area that is free until the first tile ends (the router reads it there),
  // and as fp16 B fragments of the gate/up products, zero past T.  Fragment
  // word (nt, kstep, lane, reg), in that order, holds token nt*8 + lane/4,
  // inputs kstep*16 + 2*(lane%4) + 8*reg and the next one, so the 16-byte
  // chunk c of token n fills reg c%2 of k-step c/2 for lanes 4(n%8) + j.
  uint16_t* xraw = reinterpret_cast<uint16_t*>(hbuf);
  const int xs = x_row_elems(d);
  const int cpr = d / 8;
  uint32_t* const xfw = reinterpret_cast<uint32_t*>(xfrag);
  auto put_x = [&](int n, int c, uint4 v) {
    *reinterpret_cast<uint4*>(xraw + (size_t)n * xs + c * 8) = v;
    uint32_t* w = xfw + ((((size_t)(n >> 3) * nks + (c >> 1)) * 32 + (n & 7) * 4) << 1) + (c & 1);
    w[0] = pack_half2_from_bf16(v.x);
    w[2] = pack_half2_from_bf16(v.y);
    w[4] = pack_half2_from_bf16(v.z);
    w[6] = pack_half2_from_bf16(v.w);
  };
  uint4 xv[kXPerThread];
#pragma unroll
  for (int q = 0; q < kXPerThread; ++q) {
    const int i = tid + q * kThreads;
    if (i < T * cpr) {
      const int n = i / cpr, c = i - n * cpr;
      xv[q] = __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)n * d + c * 8));
    }
  }
  if (tid == 0) MOE_TL(g_ffn_timeline, cta, 21);
  // now the stores
  if (FUSED) {
#pragma unroll
    for (int q = 0; q < kTabPerThread; ++q)
      if (tid + q * kThreads < a.E) s_tab[tid + q * kThreads] = tv[q];
  }
  if (tid == 0) {
    s_calls = calls;
    s_clock = clk;
  }
#pragma unroll
  for (int q = 0; q < kXPerThread; ++q) {
    const int i = tid + q * kThreads;
    if (i < T * cpr) {
      const int n = i / cpr, c = i - n * cpr;
      put_x(n, c, xv[q]);
    }
  }
  for (int i = tid + kXPerThread * kThreads; i < T * cpr; i += kThreads) {   // large T*d only
    const int n = i / cpr, c = i - n * cpr;
    put_x(n, c, __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)n * d + c * 8)));
  }
  // zero fragments of the token slots T .. NT*8-1: 32 contiguous bytes per
  // (n-tile, k-step, token)
  {
    const int nz = NT * 8 - T;
    for (int i = tid; i < nz * nks * 2; i += kThreads) {
      const int h = i & 1, q = i >> 1, kstep = q % nks, n = T + q / nks;
      reinterpret_cast<uint4*>(xfw + ((((size_t)(n >> 3) * nks + kstep) * 32 + (n & 7) * 4) << 1))[h] =
          make_uint4(0u, 0u, 0u, 0u);
    }
  }
  if (tid == 0) MOE_TL(g_ffn_timeline, cta, 22);
  __syncthreads();
  if (tid == 0) MOE_TL(g_ffn_timeline, cta, 26);
  // this call's counter set; the fused kernel's CTA 0 zeroes the other one
  // (the previous call's, complete by now) for the next call
  const uint32_t call_set = FUSED ? (s_calls & 1u) : ((s_calls - 1u) & 1u);
  uint32_t* const h_ready = a.counters + 1 + (size_t)call_set * a.set_words;
  uint32_t* const gbar = h_ready + a.max_exp;    // CTAs past the router phase
  uint32_t* const d_cnt = gbar + 1;              // [d/32] experts whose outputs of a row block are written
  if (FUSED && cta == 0) {
    uint32_t* other = a.counters + 1 + (size_t)(call_set ^ 1u) * a.set_words;
    for (int i = tid; i < a.set_words; i += kThreads) other[i] = 0;
  }
  if (tid == 0) MOE_TL(g_ffn_timeline, cta, 1);

  if (FUSED) {
    // ---- router rows e = cta + G*j, one warp per row ----------------------
    const int E = a.E;
    for (int j = warp;; j += kThreads / 32) {
      const int e = cta + G * j;
      if (e >= E) break;
      const uint16_t* wrow = a.wr + (size_t)e * d;
      if (j != warp) {
        router_load_block(wrow, 0, d, lane, wfirst);
        wbias = a.bias[e];
      }
      router_row(wrow, wfirst, xraw, xs, wbias, T, d, E, e, lane, a.logits);
    }
    __syncthreads();
    if (tid == 0) MOE_TL(g_ffn_timeline, cta, 6);
    // ---- every CTA's logits are written -----------------------------------
    if (tid == 0) {
      red_release_add(gbar, 1u);
      if (!wait_flag_geq(gbar, (uint32_t)G)) set_error(a.err, DEV_TIMEOUT_FLAG);
      MOE_TL(g_ffn_timeline, cta, 7);
    }
    __syncthreads();
#ifdef MOE_TIMELINE
    select_call(a.logits, T, E, K, sel, &g_ffn_timeline[cta][16]);
#else
    select_call(a.logits, T, E, K, sel);
#endif
    const int n_act = sel->n_act;
    for (int i = tid; i < T * K; i += kThreads) {
      const int id = sel->sel_id[i / K][i % K];
      s_pick_act[i] = sel_act_index(sel, id);
      s_w[i] = sel->sel_w[i / K][i % K];
    }
    for (int i = tid; i < n_act; i += kThreads) {
      int slot = s_tab[sel->act[i]];
      if (slot < 0 && !CACHED) {
        set_error(a.err, DEV_NOT_RESIDENT);
        slot = 0;
      }
      s_act_slot[i] = slot;   // cached: -1 marks a miss until CTA 0 assigns its victim
      s_act_expert[i] = sel->act[i];
    }
    if (tid == 0) s_nexp = n_act + 1;
    if (tid == 0) MOE_TL(g_ffn_timeline, cta, 27);
    // CTA 0 publishes the plan from its h-loader warp, after the split
  } else {
    const Plan* P = a.plan;   // the routing plan is complete and visible
    for (int i = tid; i < kMaxPicks; i += kThreads) s_act_slot[i] = P->act_slot[i];
    for (int i = tid; i < T * K; i += kThreads) {
      s_pick_act[i] = P->pick_act[i];
      s_w[i] = P->w[i];
    }
    if (tid == 0) s_nexp = P->n_act + 1;
  }
  if (tid == 0) MOE_TL(g_ffn_timeline, cta, 2);
  __syncthreads();
  // ---- this CTA's share: gate/up tiles [g0, g1), down tiles [d0, d1) ------
  // Each phase is split evenly by tile count: every down tile waits for the
  // gate/up phase, so balancing the phases separately ends both sooner than
  // balancing a CTA's total bytes.  Every thread computes it.
  const int n_exp_all = s_nexp;
  // cached mode: CTA 0 manages the cache, CTAs 1..G-1 take the tiles
  const int GT = CACHED ? G - 1 : G;
  const int ct = CACHED ? cta - 1 : cta;
  const int NG = n_exp_all * RG, ND = n_exp_all * (RD / RT);
  const int g0 = ct * NG / GT, g1 = (ct + 1) * NG / GT;
  const int d0 = ct * ND / GT, d1 = (ct + 1) * ND / GT;
  if (tid == 0) MOE_TL(g_ffn_timeline, cta, 3);
  if (CACHED) {
    const int n_act_c = n_exp_all - 1;
    const int n_miss = __syncthreads_count(tid < n_act_c && s_act_slot[tid] < 0);
    uint32_t* const xbar = a.counters + 1 + (size_t)call_set * a.set_words + a.max_exp + 1 + RD;
    if (cta == 0) {
      cache_manager(a, n_act_c, n_miss, s_act_expert, s_act_slot, s_pick_act, s_w, s_clock, s_calls, ring,
                    (size_t)NS * kStageBytes, xbar);
      return;
    }
    if (n_miss > 0 && !pull_and_place_misses(a, n_miss, n_act_c, s_act_slot, xbar, G - 1, cta - 1, ring))
      return;   // the error word is set; no copy was issued
  }
  const int n_gt = g1 - g0, n_dt = d1 - d0;
  const int DPE = RD / RT;               // down tiles per expert
  auto expert_base = [&](int ai) -> const uint8_t* {
    return ai == 0 ? a.shared_expert : a.slots + (int64_t)s_act_slot[ai - 1] * a.expert_bytes;
  };
  const int a_first = n_dt > 0 ? d0 / DPE : 0;
  const int a_last = n_dt > 0 ? (d1 - 1) / DPE : -1;

  if (warp == kCW) {
    // ---------------- producer: stages of every tile, in order -------------
    if (lane == 0) {
      // the ring held generic-proxy scratch; order it before the bulk copies
      fence_proxy_async_smem();
      // slots of this call's misses were written by other CTAs' generic stores
      if (CACHED) asm volatile("fence.proxy.async.global;" ::: "memory");
      MOE_TL(g_ffn_timeline, cta, 25);
      uint32_t it = 0;
      bool ok = true;
      for (int ti = 0; ti < n_gt + n_dt && ok; ++ti) {
        const uint8_t* tbase;
        int nst;
        if (ti < n_gt) {
          const int tg = g0 + ti, ai = tg / RG, rb = tg % RG;
          tbase = expert_base(ai) + gu_block_offset(rb, 0, 0, d);
          nst = SGU;
        } else {
          const int td = d0 + ti - n_gt, ai = td / DPE, rp = td % DPE;
          tbase = expert_base(ai) + down_block_offset(rp * RT, 0, d, f);
          nst = SDN;
        }
        for (int st = 0; st < nst; ++st, ++it) {
          const int s = it % NS;
          const uint32_t use = it / NS;
          if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1)) {
            set_error(a.err, DEV_TIMEOUT_BARRIER);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], kStageBytes);
          bulk_g2s(ring + (size_t)s * kStageBytes, tbase + (size_t)st * kStageBytes, kStageBytes, &full[s]);
          if (it == 0) MOE_TL(g_ffn_timeline, cta, 15);
        }
        if (ti == 0) MOE_TL(g_ffn_timeline, cta, 4);
      }
      MOE_TL(g_ffn_timeline, cta, 5);
      // no copy may still be in flight when the CTA exits (consumers that
      // gave up on a wait skip theirs): wait, bounded, for the last ones
      for (uint32_t k = it > (uint32_t)NS ? it - NS : 0; k < it; ++k)
        if (!mbar_wait(&full[k % NS], (k / NS) & 1)) set_error(a.err, DEV_TIMEOUT_BARRIER);
    }
  } else if (warp == kCW + 1) {
    if (FUSED && cta == 0) {
      // the plan of the call (read back for traces), LRU stamps, counters;
      // this warp is idle until the first h is ready
      Plan* P = a.plan;
      const long long clk = s_clock;
      const int n_act = n_exp_all - 1;
      for (int i = lane; i < T * K; i += 32) {
        P->idx[i] = s_act_expert[s_pick_act[i]];
        P->w[i] = s_w[i];
        P->pick_act[i] = s_pick_act[i];
      }
      for (int i = lane; i < n_act; i += 32) {
        P->act_expert[i] = s_act_expert[i];
        P->act_slot[i] = s_act_slot[i];
        P->act_hit[i] = 1;
        a.stamp[s_act_slot[i]] = clk;
      }
      if (lane == 0) {
        P->n_act = n_act;
        P->n_miss = 0;
        P->T = T;
        P->clock = clk;
        P->token_hits = (int64_t)T * K;
        P->token_misses = 0;
        a.stats[ST_CALLS] += 1;
        a.stats[ST_TOK_HIT] += (int64_t)T * K;
        a.stats[ST_DIST_HIT] += n_act;
        *a.clock = clk + 1;
        *a.counters = s_calls + 1;   // every CTA read the count before the grid barrier
      }
      __syncwarp();
    }
    // ---------------- h loader: one bulk copy of h_a per expert ------------
    if (lane == 0) {
      fence_proxy_async_smem();   // the h area held x through the generic proxy
      int armed = 0;
      for (int ai = a_first, i = 0; ai <= a_last; ++ai, ++i) {
        const int hs = i % kHSlots;
        const int use = i / kHSlots;
        if (use > 0 && !mbar_wait(&hempty[hs], (uint32_t)((use - 1) & 1))) {
          set_error(a.err, DEV_TIMEOUT_BARRIER);
          break;
        }
        if (!wait_flag_geq(&h_ready[ai], (uint32_t)RG)) {
          set_error(a.err, DEV_TIMEOUT_FLAG);
          break;
        }
        if (i == 0) MOE_TL(g_ffn_timeline, cta, 8);
        // h was written through the generic proxy by other CTAs; order it
        // before the bulk copy (async proxy) reads it
        asm volatile("fence.proxy.async.global;" ::: "memory");
        uint8_t* dst = hbuf + (size_t)hs * NT * 8 * hrow;
        s_hexp[hs] = ai;   // the previous use of this slot has been released
        mbar_arrive_expect_tx(&hfull[hs], (uint32_t)(T * f * 2));
        for (int t = 0; t < T; ++t)
          bulk_g2s(dst + (size_t)t * hrow, a.hbuf + ((size_t)ai * T + t) * f, (uint32_t)(f * 2), &hfull[hs]);
        armed = i + 1;
      }
      MOE_TL(g_ffn_timeline, cta, 14);
      for (int k = armed > kHSlots ? armed - kHSlots : 0; k < armed; ++k)
        if (!mbar_wait(&hfull[k % kHSlots], (uint32_t)((k / kHSlots) & 1))) set_error(a.err, DEV_TIMEOUT_BARRIER);
    }
  } else if (warp == kCW + 2) {
    // ---------------- finalizer ----------------------------------------------
    // Takes every tile's per-warp partial sums from the reduction buffer in
    // tile order, adds them in a fixed order (warp 0..7) and writes the
    // result: h = silu(g) * u (fp16) for a gate/up tile, the expert output o
    // for a down tile.  Its own gpu-scope releases then publish them
    // (h_ready per expert, d_cnt per row block of y), so the consumer warps
    // never wait for a fence or for each other.
    const int gq = lane >> 2, cq = lane & 3;
    bool ok = true;
    for (int ti = 0; ti < n_gt + n_dt && ok; ++ti) {
      if (!mbar_wait(&buf_full, (uint32_t)(ti & 1))) {
        set_error(a.err, DEV_TIMEOUT_BARRIER);
        ok = false;
        break;
      }
      if (ti < n_gt) {
        const int tg = g0 + ti, ai = tg / RG, rb = tg % RG;
        // lane l adds its fragment elements over the 8 warps in order
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float gs[8], us[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) gs[e] = us[e] = 0.f;
#pragma unroll
          for (int w = 0; w < kCW; ++w) {
            const float4* pw = reinterpret_cast<const float4*>(red + ((size_t)w * 32 + lane) * RPL + nt * 16);
            const float4 g0 = pw[0], g1 = pw[1], u0 = pw[2], u1 = pw[3];
            gs[0] += g0.x; gs[1] += g0.y; gs[2] += g0.z; gs[3] += g0.w;
            gs[4] += g1.x; gs[5] += g1.y; gs[6] += g1.z; gs[7] += g1.w;
            us[0] += u0.x; us[1] += u0.y; us[2] += u0.z; us[3] += u0.w;
            us[4] += u1.x; us[5] += u1.y; us[6] += u1.z; us[7] += u1.w;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float g = gs[e], u = us[e];
            const int mt = e >> 2, i = e & 3;
            const int tok = nt * 8 + 2 * cq + (i & 1);
            if (tok < T) {
              const float hv = g / (1.f + expf(-g)) * u;
              const int row = rb * 32 + mt * 16 + gq + 8 * (i >> 1);
              a.hbuf[((size_t)ai * T + tok) * f + row] = __half_as_ushort(__float2half_rn(hv));
            }
          }
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&buf_free);
          red_release_add(&h_ready[ai], 1u);   // covers this warp's h stores (after the warp sync)
        }
        if (ti + 1 == n_gt && lane == 0) MOE_TL(g_ffn_timeline, cta, 9);
      } else {
        const int td = d0 + ti - n_gt, ai = td / DPE, rp = td % DPE;
        // row block r is the sum, in warp order, of the WPR warps that took it
#pragma unroll 1
        for (int r = 0; r < RT; ++r) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            float os[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) os[e] = 0.f;
#pragma unroll 4
            for (int w = r * WPR; w < (r + 1) * WPR; ++w) {
              const float4* pw = reinterpret_cast<const float4*>(red + ((size_t)w * 32 + lane) * RPL + nt * 8);
              const float4 o0 = pw[0], o1 = pw[1];
              os[0] += o0.x; os[1] += o0.y; os[2] += o0.z; os[3] += o0.w;
              os[4] += o1.x; os[5] += o1.y; os[6] += o1.z; os[7] += o1.w;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float o = os[e];
              const int mt = e >> 2, i = e & 3;
              const int tok = nt * 8 + 2 * cq + (i & 1);
              if (tok < T) {
                const int row = (rp * RT + r) * 32 + mt * 16 + gq + 8 * (i >> 1);
                a.obuf[((size_t)ai * T + tok) * d + row] = o;
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&buf_free);
        if (lane < RT) red_release_add(&d_cnt[rp * RT + lane], 1u);
      }
    }
    if (lane == 0) MOE_TL(g_ffn_timeline, cta, 11);
    // ---- combine: CTA c owns row blocks c, c + G, ... of y.  Once all n_exp
    // expert outputs of a row block are written it forms y there in a fixed
    // order (shared expert, then the picks in ascending id), all loads of
    // one output issued before the sum.
    const int n_exp = s_nexp;
    for (int rb = ct; ok && rb < RD; rb += GT) {
      uint32_t good = 1;
      if (lane == 0 && !wait_flag_geq(&d_cnt[rb], (uint32_t)n_exp)) {
        set_error(a.err, DEV_TIMEOUT_FLAG);
        good = 0;
      }
      if (!__shfl_sync(0xffffffffu, good, 0)) break;
      if (lane == 0 && rb == ct) MOE_TL(g_ffn_timeline, cta, 23);
      __syncwarp();   // the other lanes read after lane 0's acquire
      const int row = rb * 32 + lane;
#pragma unroll 1
      for (int t = 0; t < T; ++t) {
        // every load is issued before the first use; picks past K read the
        // shared expert's row and carry weight 0
        const float* prow[kMaxTopK];
#pragma unroll
        for (int k2 = 0; k2 < kMaxTopK; ++k2)
          prow[k2] = a.obuf + ((size_t)(k2 < K ? 1 + s_pick_act[t * K + k2] : 0) * T + t) * d + row;
        const float sh = __ldcg(a.obuf + (size_t)t * d + row);
        float ov[kMaxTopK];
#pragma unroll
        for (int k2 = 0; k2 < kMaxTopK; ++k2) ov[k2] = __ldcg(prow[k2]);
        float yv = a.shared_weight * sh;
#pragma unroll
        for (int k2 = 0; k2 < kMaxTopK; ++k2)
          if (k2 < K) yv = fmaf(s_w[t * K + k2], ov[k2], yv);
        if (lane == 0 && rb == ct && t == 0) MOE_TL(g_ffn_timeline, cta, 24);
        a.y[(size_t)t * d + row] = yv;
      }
    }
    if (lane == 0) MOE_TL(g_ffn_timeline, cta, 12);
  } else {
    // ---------------- consumers: 8 warps on every stage --------------------
    // After a tile each warp writes its partial sums to the reduction buffer
    // (once the finalizer has read the previous tile's) and moves on.
    uint32_t it = 0;
    bool ok = true;
    float* mine = red + ((size_t)warp * 32 + lane) * RPL;
    auto wait_buf_free = [&](int ti) {
      if (ok && ti > 0 && !mbar_wait(&buf_free, (uint32_t)((ti - 1) & 1))) {
        set_error(a.err, DEV_TIMEOUT_BARRIER);
        ok = false;
      }
    };
    auto signal_buf_full = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(&buf_full);
    };
    for (int ti = 0; ti < n_gt + n_dt; ++ti) {
      if (ti < n_gt) {
        // ===== gate/up tile: 32 rows of Wg and Wu over all inputs =====
        float ag[NT][2][4], au[NT][2][4];
        zero_acc<NT>(ag);
        zero_acc<NT>(au);
        for (int st = 0; st < SGU; ++st, ++it) {
          const int s = it % NS;
          if (ok && !mbar_wait(&full[s], (it / NS) & 1)) {
            set_error(a.err, DEV_TIMEOUT_BARRIER);
            ok = false;
          }
          if (ok) {
            const uint8_t* sp = ring + (size_t)s * kStageBytes;
            const int gi = st * (kStageBlocks / 2) + warp;     // input group of this warp
            uint2 bx[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              bx[nt][0] = xfrag[((size_t)nt * nks + gi * 2 + 0) * 32 + lane];
              bx[nt][1] = xfrag[((size_t)nt * nks + gi * 2 + 1) * 32 + lane];
            }
            block_mma<NT>(sp + (2 * warp + 0) * kBlockBytes, lane, bx, ag);
            block_mma<NT>(sp + (2 * warp + 1) * kBlockBytes, lane, bx, au);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
        }
        wait_buf_free(ti);
        if (ok) {
          float4* m4 = reinterpret_cast<float4*>(mine);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              m4[nt * 4 + mt] = make_float4(ag[nt][mt][0], ag[nt][mt][1], ag[nt][mt][2], ag[nt][mt][3]);
              m4[nt * 4 + 2 + mt] = make_float4(au[nt][mt][0], au[nt][mt][1], au[nt][mt][2], au[nt][mt][3]);
            }
        }
        signal_buf_full();
      } else {
        // ===== down tile: RT row blocks of Wd for expert ai =====
        const int td = d0 + ti - n_gt, ai = td / DPE;
        const int hi_idx = ai - a_first, hs = hi_idx % kHSlots;
        if (ok && s_hexp[hs] != ai) {
          const uint64_t t0 = globaltimer();
          while (s_hexp[hs] != ai) {
            if (globaltimer() - t0 > kWaitLimitNs) {
              set_error(a.err, DEV_TIMEOUT_BARRIER);
              ok = false;
              break;
            }
          }
        }
        if (ok && !mbar_wait(&hfull[hs], (uint32_t)((hi_idx / kHSlots) & 1))) {
          set_error(a.err, DEV_TIMEOUT_BARRIER);
          ok = false;
        }
        if (tid == 0 && ti == n_gt) MOE_TL(g_ffn_timeline, cta, 10);
        const uint8_t* hb = hbuf + (size_t)hs * NT * 8 * hrow;
        // this warp sums row block r_w of the tile: its input groups j_w,
        // j_w + WPR, ..., met in stage order, two blocks at a time
        const int r_w = warp / WPR, j_w = warp - r_w * WPR;
        const int rbase = r_w * DG;   // first block of the row block in the tile
        float acc[NT][2][4];
        zero_acc<NT>(acc);
        for (int st = 0; st < SDN; ++st, ++it) {
          const int s = it % NS;
          if (ok && !mbar_wait(&full[s], (it / NS) & 1)) {
            set_error(a.err, DEV_TIMEOUT_BARRIER);
            ok = false;
          }
          if (ok) {
            const uint8_t* sp = ring + (size_t)s * kStageBytes;
            const int b_lo = max(rbase, st * kStageBlocks), b_hi = min(rbase + DG, (st + 1) * kStageBlocks);
            for (int b = rbase + j_w + ((b_lo - rbase - j_w + WPR - 1) / WPR) * WPR; b < b_hi; b += 2 * WPR) {
              const int b1 = b + WPR;
              uint2 bx0[NT][2];
              h_frags<NT>(hb, hrow, T, b - rbase, lane, bx0);
              float D0[NT][2][4], s0[4];
              block_products<NT>(sp + (b - st * kStageBlocks) * kBlockBytes, lane, bx0, D0, s0);
              if (b1 < b_hi) {
                uint2 bx1[NT][2];
                h_frags<NT>(hb, hrow, T, b1 - rbase, lane, bx1);
                float D1[NT][2][4], s1[4];
                block_products<NT>(sp + (b1 - st * kStageBlocks) * kBlockBytes, lane, bx1, D1, s1);
                block_accum<NT>(D0, s0, acc);
                block_accum<NT>(D1, s1, acc);
              } else {
                block_accum<NT>(D0, s0, acc);
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
        }
        // this warp is done reading expert ai's h slot after its last tile of ai
        const bool last_of_expert = (ti + 1 == n_gt + n_dt) || ((d0 + ti + 1 - n_gt) / DPE != ai);
        if (last_of_expert && lane == 0) mbar_arrive(&hempty[hs]);
        wait_buf_free(ti);
        if (ok) {
          float4* m4 = reinterpret_cast<float4*>(mine);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
              m4[nt * 2 + mt] = make_float4(acc[nt][mt][0], acc[nt][mt][1], acc[nt][mt][2], acc[nt][mt][3]);
        }
        signal_buf_full();
      }
    }
    if (tid == 0) MOE_TL(g_ffn_timeline, cta, 13);
  }
}

#ifdef MOE_TIMELINE
extern "C" int moe_debug_timeline_ffn(unsigned long long* out) {
  return (int)cudaMemcpyFromSymbol(out, g_ffn_timeline, sizeof(g_ffn_timeline));
}
#endif

template <int NT, int MODE>
static cudaError_t launch_nt(const FfnArgs& a, cudaStream_t s, bool pdl, int grid) {
  constexpr bool FUSED = MODE != kPlanRead;
  const size_t smem = ffn_smem_bytes<NT>(a.d, a.f);
  if (route_scratch_bytes(FUSED ? a.E : 0) > (size_t)FfnCfg<NT>::kStages * kStageBytes ||
      (FUSED && a.E > kTabPerThread * kThreads) || kCW % down_rows_per_tile(a.f) != 0)
    return cudaErrorInvalidValue;
  // x is staged in the h + partial area
  if ((size_t)a.T * x_row_elems(a.d) * 2 >
      (size_t)kHSlots * NT * 8 * h_row_bytes(a.f) + (size_t)kCW * 32 * red_per_lane(NT) * 4)
    return cudaErrorInvalidValue;
  // the dynamic shared-memory limit, raised once per device
  cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(decode_ffn_kernel<NT, MODE>), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, decode_ffn_kernel<NT, MODE>, a);
}

cudaError_t launch_decode_ffn(const FfnArgs& a, cudaStream_t s, bool pdl) {
  if (a.grid <= 0 || (a.cached && (!a.fused || a.grid < 2))) return cudaErrorInvalidValue;
  if (a.T <= 8) {
    if (!a.fused) return launch_nt<1, kPlanRead>(a, s, pdl, a.grid);
    return a.cached ? launch_nt<1, kFusedCached>(a, s, pdl, a.grid) : launch_nt<1, kFusedResident>(a, s, pdl, a.grid);
  }
  if (!a.fused) return launch_nt<2, kPlanRead>(a, s, pdl, a.grid);
  return a.cached ? launch_nt<2, kFusedCached>(a, s, pdl, a.grid) : launch_nt<2, kFusedResident>(a, s, pdl, a.grid);
}

}  // namespace moe
