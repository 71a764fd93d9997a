// Router + top-k + cache plan for one decode layer-call (T <= 16 tokens).
//
// Router (workload definition; the pages only fix 10-of-512 routing plus a
// shared expert, page "一张 RTX 4090 跑千亿模型", §如何做到：三层存储):
//   l[t,e] = x_t . Wr[e] + b[e] in fp32 from bf16 inputs; the k largest
//   logits are chosen (ties to the lower id); w_i = softmax over the whole
//   row restricted to the chosen set and renormalised, which equals a softmax
//   over the k chosen logits alone.
//
// Cache (LRU by (layer, expert), ties to the lower slot id; misses fetched
// from pinned host RAM, page "单卡5090跑125B 大模型", §2.1 and §7.2):
//   U = distinct experts of the call (ascending).  Resident keys are hits
//   and are stamped first; the misses, in ascending expert id, take the
//   least recently used slots in (stamp, slot id) order.  The LRU order is
//   kept as an array q (least recent first); one call moves its touched slots
//   (hits and victims), in slot-id order, to the most recent end.
//
// One launch: ceil(E/8) CTAs of 8 warps, one warp per expert row.  The last
// CTA to finish its logits (arrival counter) selects, forms U and the plan.
#include <mutex>

#include "moe_gb300.h"
#include "common.cuh"
#include "internal.h"
#include "select.cuh"

namespace moe {

#ifdef MOE_TIMELINE
__device__ unsigned long long g_route_timeline[256][16];
#endif

constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = kRouteThreads / 32;
// the LRU order q is staged in shared memory (one 16-byte load per 4 slots,
// all in flight) when the cache has at most this many slots
constexpr int kRouteQSmem = 32768;
constexpr size_t kSelBytes = (sizeof(SelSmem) + 15) & ~size_t(15);

// exclusive prefix sum over the 256 threads of the CTA; returns the total
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) s_warp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int wv = lane < kRouteWarps ? s_warp[lane] : 0;
    int wi = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    if (lane < kRouteWarps) s_warp[lane] = wi - wv;
    if (lane == kRouteWarps - 1) s_warp[kRouteWarps] = wi;
  }
  __syncthreads();
  int r = s_warp[warp] + inc - v;
  *total = s_warp[kRouteWarps];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kRouteThreads) route_kernel(RouteArgs a) {
  if (threadIdx.x == 0) MOE_TL(g_route_timeline, blockIdx.x, 0);
  pdl_launch_dependents();

  extern __shared__ __align__(16) uint8_t route_dyn_smem[];
  SelSmem& sel = *reinterpret_cast<SelSmem*>(route_dyn_smem);
  __shared__ int s_slot[kMaxPicks];
  __shared__ int s_hit[kMaxPicks];
  __shared__ int s_miss_act[kMaxPicks];
  __shared__ int s_victim[kMaxPicks];
  __shared__ uint32_t s_bits[kMaxSlots / 32];
  __shared__ int s_scan[kRouteWarps + 1];
  __shared__ int s_last, s_n_miss;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = a.T, E = a.E, K = a.k;
  // the clock of this call, fetched early (only the last CTA uses it)
  const long long clock0 = (a.mode == ROUTE_PLAN && threadIdx.x == 0) ? (long long)*a.clock : 0;

  // ---- router logits: one warp per expert row, all T tokens -------------
  const int e = blockIdx.x * kRouteWarps + warp;
  if (e < E) {
    const uint16_t* wrow = a.wr + (size_t)e * a.d;
    uint4 first[8];
    router_load_block(wrow, 0, a.d, lane, first);
    float* const lg = a.logits;
    router_row(wrow, first, a.x, a.d, a.bias[e], T, a.d, lane, [&](int t, float v) { lg[(size_t)t * E + e] = v; });
  }

  // ---- last CTA to arrive does the selection -----------------------------
  __syncthreads();
  if (threadIdx.x == 0) MOE_TL(g_route_timeline, blockIdx.x, 1);
  if (threadIdx.x == 0) s_last = (atom_acq_rel_add(a.cnt, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  if (threadIdx.x == 0) {
    MOE_TL(g_route_timeline, 200, 0);
    *a.cnt = 0;   // ready for the next launch (stream-ordered)
  }
  select_call(PlainLogits{a.logits}, T, E, K, &sel);
  if (threadIdx.x == 0) MOE_TL(g_route_timeline, 200, 1);
  const int n_act = sel.n_act;
  Plan* P = a.plan;

  if (a.mode == ROUTE_ONLY) {
    for (int i = threadIdx.x; i < T * K; i += kRouteThreads) {
      a.out_idx[i] = sel.sel_id[i / K][i % K];
      a.out_w[i] = sel.sel_w[i / K][i % K];
    }
    return;
  }

  // plan: routing part
  for (int i = threadIdx.x; i < T * K; i += kRouteThreads) {
    const int id = sel.sel_id[i / K][i % K];
    P->idx[i] = id;
    P->w[i] = sel.sel_w[i / K][i % K];
    P->pick_act[i] = sel_act_index(&sel, id);
    if (a.out_idx) {
      a.out_idx[i] = id;
      a.out_w[i] = sel.sel_w[i / K][i % K];
    }
  }
  for (int i = threadIdx.x; i < n_act; i += kRouteThreads) {
    const int slot = a.table[(size_t)a.layer * E + sel.act[i]];
    s_slot[i] = slot;
    s_hit[i] = slot >= 0;
    P->act_expert[i] = sel.act[i];
  }
  __syncthreads();
  if (threadIdx.x == 0) MOE_TL(g_route_timeline, 200, 2);

  // ---- ROUTE_PLAN: LRU victims and the next LRU order (no state commit) ---
  const int C = a.C;
  const int c_words = (C + 31) / 32;
  for (int i = threadIdx.x; i < c_words; i += kRouteThreads) s_bits[i] = 0;
  int32_t* s_q = C <= kRouteQSmem ? reinterpret_cast<int32_t*>(route_dyn_smem + kSelBytes) : nullptr;
  if (s_q) {
    const int n4 = C >> 2;
    const int4* src4 = reinterpret_cast<const int4*>(a.q_in);
#pragma unroll 4
    for (int i = threadIdx.x; i < n4; i += kRouteThreads) reinterpret_cast<int4*>(s_q)[i] = __ldg(src4 + i);
    for (int i = 4 * n4 + threadIdx.x; i < C; i += kRouteThreads) s_q[i] = a.q_in[i];
  }
  const int32_t* q_in = s_q ? s_q : a.q_in;
  if (threadIdx.x == 0) {
    int m = 0;
    for (int i = 0; i < n_act; ++i)
      if (!s_hit[i]) s_miss_act[m++] = i;   // ascending expert id
    s_n_miss = m;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n_act; i += kRouteThreads)
    if (s_hit[i]) atomicOr(&s_bits[s_slot[i] >> 5], 1u << (s_slot[i] & 31));
  __syncthreads();
  const int m = s_n_miss;

  // walk q (least recent first) skipping this call's hits: the first m
  // entries are the victims, the rest keep their order at the front of q_out
  const int chunk = (C + kRouteThreads - 1) / kRouteThreads;
  const int lo = min(C, (int)threadIdx.x * chunk), hi = min(C, lo + chunk);
  int cnt = 0;
  for (int i = lo; i < hi; ++i) {
    const int s = q_in[i];
    cnt += !((s_bits[s >> 5] >> (s & 31)) & 1u);
  }
  int total;
  int r = block_exclusive_scan(cnt, s_scan, &total);
  for (int i = lo; i < hi; ++i) {
    const int s = q_in[i];
    if (!((s_bits[s >> 5] >> (s & 31)) & 1u)) {
      if (r < m) s_victim[r] = s;
      else a.q_out[r - m] = s;
      ++r;
    }
  }
  __syncthreads();
  for (int j = threadIdx.x; j < m; j += kRouteThreads)
    atomicOr(&s_bits[s_victim[j] >> 5], 1u << (s_victim[j] & 31));
  __syncthreads();
  // touched slots (hits and victims) in ascending slot id to the recent end
  const int wchunk = (c_words + kRouteThreads - 1) / kRouteThreads;
  const int wlo = min(c_words, (int)threadIdx.x * wchunk), whi = min(c_words, wlo + wchunk);
  int tc = 0;
  for (int i = wlo; i < whi; ++i) tc += __popc(s_bits[i]);
  int tr = block_exclusive_scan(tc, s_scan, &total);
  for (int i = wlo; i < whi; ++i) {
    uint32_t bits = s_bits[i];
    while (bits) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1;
      a.q_out[C - n_act + tr] = i * 32 + b;
      ++tr;
    }
  }
  for (int j = threadIdx.x; j < m; j += kRouteThreads) {
    const int ai = s_miss_act[j];
    const int v = s_victim[j];
    s_slot[ai] = v;
    P->miss_expert[j] = sel.act[ai];
    P->miss_slot[j] = v;
    P->evicted_key[j] = a.owner[v];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n_act; i += kRouteThreads) {
    P->act_slot[i] = s_slot[i];
    P->act_hit[i] = s_hit[i];
  }
  if (threadIdx.x == 0) {
    int64_t th = 0;
    for (int i = 0; i < T * K; ++i) th += s_hit[sel_act_index(&sel, sel.sel_id[i / K][i % K])];
    P->n_act = n_act;
    P->n_miss = m;
    P->T = T;
    P->clock = clock0;
    P->token_hits = th;
    P->token_misses = (int64_t)T * K - th;
  }
}

// Applies a ROUTE_PLAN plan once its miss copies are enqueued, and readies
// the decode counters of the call's expert kernel.
__global__ void __launch_bounds__(256) commit_kernel(CommitArgs a) {
  const Plan* P = a.plan;
  const int n_act = P->n_act, m = P->n_miss;
  const int64_t clk = P->clock;
  // the expert kernel reads the bumped call count and uses the counter set
  // of the count before it; the set of the call before it is zeroed here
  const uint32_t calls = *a.counters;
  __shared__ int s_evict;
  if (threadIdx.x == 0) s_evict = 0;
  __syncthreads();
  uint32_t* prev_set = a.counters + 1 + (size_t)((calls + 1) & 1) * a.set_words;
  for (int i = threadIdx.x; i < a.set_words; i += blockDim.x) prev_set[i] = 0;
  for (int i = threadIdx.x; i < n_act; i += blockDim.x)
    if (P->act_hit[i]) a.stamp[P->act_slot[i]] = clk;
  for (int j = threadIdx.x; j < m; j += blockDim.x) {
    const int old = P->evicted_key[j];
    if (old >= 0) {
      a.table[old] = -1;
      atomicAdd(&s_evict, 1);
    }
  }
  __syncthreads();
  for (int j = threadIdx.x; j < m; j += blockDim.x) {
    const int v = P->miss_slot[j];
    const int key = a.layer * a.E + P->miss_expert[j];
    a.owner[v] = key;
    a.table[key] = v;
    a.stamp[v] = clk;
  }
  if (threadIdx.x == 0) {
    *a.counters = calls + 1;
    a.stats[ST_CALLS] += 1;
    a.stats[ST_TOK_HIT] += P->token_hits;
    a.stats[ST_TOK_MISS] += P->token_misses;
    a.stats[ST_DIST_HIT] += n_act - m;
    a.stats[ST_DIST_MISS] += m;
    a.stats[ST_EVICT] += s_evict;
    a.stats[ST_MISS_BYTES] += (int64_t)m * a.expert_bytes;
    *a.clock = clk + 1;
  }
}

#ifdef MOE_TIMELINE
extern "C" int moe_debug_timeline_route(unsigned long long* out) {
  return (int)cudaMemcpyFromSymbol(out, g_route_timeline, sizeof(g_route_timeline));
}
#endif

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s) {
  // the selection scratch (and the staged LRU order) is dynamic shared
  // memory (static + dynamic > 48 KB)
  cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(route_kernel), kSelBytes + (size_t)kRouteQSmem * 4);
  if (e != cudaSuccess) return e;
  const size_t dyn = kSelBytes + (a.mode == ROUTE_PLAN && a.C <= kRouteQSmem ? (size_t)a.C * 4 : 0);
  const int grid = (a.E + kRouteWarps - 1) / kRouteWarps;
  route_kernel<<<grid, kRouteThreads, dyn, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_commit(const CommitArgs& a, cudaStream_t s) {
  commit_kernel<<<1, 256, 0, s>>>(a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Allocation-free router: moe_route_topk_noalloc.
//
// Its scratch (the logits of up to 16 tokens x 1024 experts and the CTA
// arrival counter) is a fixed array in the library image, so the call needs
// no cudaMalloc.  Every GPU that loads the library holds these 64 KiB (+8 KiB)
// until the process exits.  A zero-bias row serves callers without a bias.
static __device__ __align__(256) float g_noalloc_logits[kMaxDecodeT * kMaxE];
static __device__ __align__(256) uint32_t g_noalloc_counter[64];
static __device__ __align__(256) float g_noalloc_zero_bias[kMaxE];

namespace {
constexpr int kNoallocMaxDevices = 64;

struct NoallocScratch {
  float* logits = nullptr;
  uint32_t* counter = nullptr;
  float* zero_bias = nullptr;
};
std::mutex g_noalloc_mu;
NoallocScratch g_noalloc[kNoallocMaxDevices];

// Device addresses of the static scratch on the current device, looked up once
// per device (with that device current) and cached.
cudaError_t noalloc_scratch(NoallocScratch* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kNoallocMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoallocScratch& s = g_noalloc[dev];
  if (!s.logits) {
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_noalloc_logits)) != cudaSuccess) return e;
    void* q = nullptr;
    if ((e = cudaGetSymbolAddress(&q, g_noalloc_counter)) != cudaSuccess) return e;
    void* z = nullptr;
    if ((e = cudaGetSymbolAddress(&z, g_noalloc_zero_bias)) != cudaSuccess) return e;
    s.logits = static_cast<float*>(p);
    s.counter = static_cast<uint32_t*>(q);
    s.zero_bias = static_cast<float*>(z);
  }
  *out = s;
  return cudaSuccess;
}
}  // namespace

}  // namespace moe

extern "C" moe_status moe_route_topk_noalloc(const void* x_bf16, const void* router_w_bf16, const float* router_b,
                                             int32_t T, int32_t d, int32_t n_experts, int32_t top_k, int32_t* idx,
                                             float* w, void* stream) {
  using namespace moe;
  if (!x_bf16 || !router_w_bf16 || !idx || !w)
    return set_last_error(MOE_ERR_INVALID_ARG, "moe_route_topk_noalloc: NULL pointer");
  if (T < 1 || T > kMaxDecodeT)
    return set_last_error(MOE_ERR_INVALID_ARG, "moe_route_topk_noalloc: T=%d exceeds the static scratch (1..%d)",
                          T, kMaxDecodeT);
  if (n_experts > kMaxE || top_k < 2 || top_k > kMaxTopK || n_experts <= top_k)
    return set_last_error(MOE_ERR_INVALID_ARG,
                          "moe_route_topk_noalloc: need 2 <= top_k <= %d and top_k < n_experts <= %d", kMaxTopK,
                          kMaxE);
  if (d <= 0 || d % 256 != 0)
    return set_last_error(MOE_ERR_INVALID_ARG, "moe_route_topk_noalloc: d must be a positive multiple of 256");
  if (reinterpret_cast<uintptr_t>(x_bf16) % 16 || reinterpret_cast<uintptr_t>(router_w_bf16) % 16)
    return set_last_error(MOE_ERR_INVALID_ARG, "moe_route_topk_noalloc: x and router_w must be 16-byte aligned");
  NoallocScratch sc;
  cudaError_t e = noalloc_scratch(&sc);
  if (e != cudaSuccess)
    return set_last_error(MOE_ERR_CUDA, "moe_route_topk_noalloc: static scratch lookup failed: %s",
                          cudaGetErrorString(e));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the arrival counter must start at zero
  e = cudaMemsetAsync(sc.counter, 0, sizeof(uint32_t), s);
  if (e != cudaSuccess) return set_last_error(MOE_ERR_CUDA, "moe_route_topk_noalloc: %s", cudaGetErrorString(e));
  RouteArgs a{};
  a.x = static_cast<const uint16_t*>(x_bf16);
  a.wr = static_cast<const uint16_t*>(router_w_bf16);
  a.bias = router_b ? router_b : sc.zero_bias;
  a.T = T;
  a.d = d;
  a.E = n_experts;
  a.k = top_k;
  a.mode = ROUTE_ONLY;
  a.logits = sc.logits;
  a.cnt = sc.counter;
  a.out_idx = idx;
  a.out_w = w;
  e = launch_route(a, s);
  if (e != cudaSuccess) return set_last_error(MOE_ERR_CUDA, "moe_route_topk_noalloc: %s", cudaGetErrorString(e));
  return MOE_OK;
}
