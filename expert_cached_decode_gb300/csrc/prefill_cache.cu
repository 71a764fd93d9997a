// The expert cache step of a prefill chunk and the fetch of its misses.
//
// A chunk of T tokens at one layer is one layer-call of the cache (the pages
// prefill in chunks of 12,288 tokens on the same offloaded expert cache that
// decode uses, page "一张 RTX 4090 跑千亿模型", §加个草稿层 and
// §如何做到：三层存储): U = the chunk's distinct routed experts, ascending;
// resident ones are hits and are stamped first; the misses, in ascending
// expert id, take the least recently used slots in (stamp, slot id) order --
// the order of the LRU array q with the hits skipped -- and the touched
// slots move, in slot-id order, to the recent end of q.  The same rule as the
// decode kernel's cache manager, for up to E distinct experts.  A token pick
// is a hit iff its expert was resident when the chunk began.
//
// prefill_cache_kernel (one CTA of 1024 threads) decides and commits;
// prefill_fetch_kernel (a persistent grid) then reads every miss from the
// registered host pool into its victim slot (fetch.cuh), before the grouped
// GEMMs run.
#include "common.cuh"
#include "fetch.cuh"
#include "internal.h"

namespace moe {

constexpr int kCacheThreads = 1024;

// exclusive prefix sum over the CTA's 1024 threads; *total gets the sum
__device__ __forceinline__ int cta1024_exclusive_scan(int v, int* s_warp, int* total) {
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
    const int wv = s_warp[lane];
    int wi = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    s_warp[lane] = wi - wv;
    if (lane == 31) s_warp[32] = wi;
  }
  __syncthreads();
  const int r = s_warp[warp] + inc - v;
  *total = s_warp[32];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kCacheThreads, 1) prefill_cache_kernel(PrefillCacheArgs a) {
  extern __shared__ __align__(16) uint8_t dsm[];
  __shared__ int s_warp[33];
  __shared__ int s_act[kMaxE];      // U, ascending
  __shared__ int s_slot[kMaxE];     // slot of each key of U (-1: miss, until its victim is known)
  __shared__ int s_missi[kMaxE];    // U index of the j-th miss
  __shared__ int s_victim[kMaxE];
  __shared__ int s_old[kMaxE];
  __shared__ int s_evict;
  const int tid = threadIdx.x, E = a.E, C = a.C;
  const int c_words = (C + 31) / 32;
  uint32_t* bits = reinterpret_cast<uint32_t*>(dsm);                     // touched slots
  int32_t* sq = a.q_staged ? reinterpret_cast<int32_t*>(dsm + (((size_t)c_words * 4 + 15) & ~size_t(15))) : nullptr;
  const long long clk = *a.clock;
  // U and its misses, in ascending expert id (one expert per thread)
  const int cnt = tid < E ? a.counts[tid] : 0;
  const int slot0 = cnt > 0 ? a.table[(size_t)a.layer * E + tid] : -1;
  int n_act, n_miss;
  const int pos = cta1024_exclusive_scan(cnt > 0, s_warp, &n_act);
  const int mpos = cta1024_exclusive_scan(cnt > 0 && slot0 < 0, s_warp, &n_miss);
  if (cnt > 0) {
    s_act[pos] = tid;
    s_slot[pos] = slot0;
    if (slot0 < 0) s_missi[mpos] = pos;
  }
  for (int i = tid; i < c_words; i += kCacheThreads) bits[i] = 0;
  if (sq) {
    for (int i = tid; i < C; i += kCacheThreads) sq[i] = a.q_in[i];
  }
  if (tid == 0) s_evict = 0;
  __syncthreads();
  if (n_miss > C - (n_act - n_miss)) {   // more misses than slots left: the capacity check failed
    if (tid == 0) set_error(a.err, DEV_BAD_PLAN);
    return;
  }
  if (cnt > 0 && slot0 >= 0) atomicOr(&bits[slot0 >> 5], 1u << (slot0 & 31));
  __syncthreads();
  const int32_t* q_in = sq ? sq : a.q_in;
  // walk q skipping the hits: the first n_miss slots are the victims, the
  // rest keep their order at the front of the next q
  const int chunk = (C + kCacheThreads - 1) / kCacheThreads;
  const int lo = min(C, tid * chunk), hi = min(C, lo + chunk);
  int nh = 0;
  for (int i = lo; i < hi; ++i) {
    const int sl = q_in[i];
    nh += !((bits[sl >> 5] >> (sl & 31)) & 1u);
  }
  int total;
  int r = cta1024_exclusive_scan(nh, s_warp, &total);
  for (int i = lo; i < hi; ++i) {
    const int sl = q_in[i];
    if (!((bits[sl >> 5] >> (sl & 31)) & 1u)) {
      if (r < n_miss) s_victim[r] = sl;
      else a.q_out[r - n_miss] = sl;
      ++r;
    }
  }
  __syncthreads();
  for (int j = tid; j < n_miss; j += kCacheThreads) {
    const int v = s_victim[j];
    const int ai = s_missi[j];
    const int old = a.owner[v];
    atomicOr(&bits[v >> 5], 1u << (v & 31));
    s_old[j] = old;
    s_slot[ai] = v;
    a.miss_expert[j] = s_act[ai];
    a.miss_slot[j] = v;
    a.evicted_key[j] = old;
  }
  __syncthreads();
  // commit: evicted keys leave the table before the misses enter it
  for (int j = tid; j < n_miss; j += kCacheThreads) {
    const int old = s_old[j];
    if (old >= 0) {
      a.table[old] = -1;
      atomicAdd(&s_evict, 1);
    }
  }
  __syncthreads();
  for (int j = tid; j < n_miss; j += kCacheThreads) {
    const int v = s_victim[j];
    const int key = a.layer * E + s_act[s_missi[j]];
    a.owner[v] = key;
    a.table[key] = v;
    a.stamp[v] = clk;
  }
  // stamps of the hits, the slot of every expert of U, token-level counts
  int th = 0, tm = 0;
  if (tid < E) a.group_slot[tid] = -1;
  __syncthreads();
  for (int i = tid; i < n_act; i += kCacheThreads) a.group_slot[s_act[i]] = s_slot[i];
  if (cnt > 0) {
    if (slot0 >= 0) {
      a.stamp[slot0] = clk;
      th = cnt;
    } else {
      tm = cnt;
    }
  }
  // touched slots (hits and victims) in ascending slot id to the recent end
  const int wchunk = (c_words + kCacheThreads - 1) / kCacheThreads;
  const int wlo = min(c_words, tid * wchunk), whi = min(c_words, wlo + wchunk);
  int tc = 0;
  for (int i = wlo; i < whi; ++i) tc += __popc(bits[i]);
  int tr = cta1024_exclusive_scan(tc, s_warp, &total);
  for (int i = wlo; i < whi; ++i) {
    uint32_t b = bits[i];
    while (b) {
      const int bit = __ffs(b) - 1;
      b &= b - 1;
      a.q_out[C - n_act + tr] = i * 32 + bit;
      ++tr;
    }
  }
  int hits, misses;
  cta1024_exclusive_scan(th, s_warp, &hits);
  cta1024_exclusive_scan(tm, s_warp, &misses);
  if (tid == 0) {
    a.info[0] = n_miss;
    a.info[1] = n_act;
    a.info[2] = hits;
    a.info[3] = misses;
    a.stats[ST_CALLS] += 1;
    a.stats[ST_TOK_HIT] += hits;
    a.stats[ST_TOK_MISS] += misses;
    a.stats[ST_DIST_HIT] += n_act - n_miss;
    a.stats[ST_DIST_MISS] += n_miss;
    a.stats[ST_EVICT] += s_evict;
    a.stats[ST_MISS_BYTES] += (int64_t)n_miss * a.expert_bytes;
    *a.clock = clk + 1;
  }
}

// The chunk's misses from the host pool into their victim slots: every CTA
// takes an even, contiguous share of the n_miss * jobs-per-miss fetch jobs.
constexpr int kFetchThreads = 512;

__global__ void __launch_bounds__(kFetchThreads, 1) prefill_fetch_kernel(MissFetch f, const int32_t* n_miss) {
  extern __shared__ __align__(16) uint8_t fsm[];
  const int J = *n_miss * fetch_jobs_per_miss(f.d, f.f);
  const int G = gridDim.x, c = blockIdx.x;
  constexpr int KPC = (14 * 2048 / 16 + kFetchThreads - 1) / kFetchThreads;
  pull_jobs<kFetchThreads, KPC>(f, (int)((int64_t)c * J / G), (int)((int64_t)(c + 1) * J / G), fsm, nullptr);
}

cudaError_t launch_prefill_cache(const PrefillCacheArgs& a, cudaStream_t s) {
  const size_t bits = (((size_t)(a.C + 31) / 32) * 4 + 15) & ~size_t(15);
  const size_t dyn = bits + (a.q_staged ? (size_t)a.C * 4 : 0);
  cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(prefill_cache_kernel), dyn);
  if (e != cudaSuccess) return e;
  prefill_cache_kernel<<<1, kCacheThreads, dyn, s>>>(a);
  return cudaGetLastError();
}

// With the host pool in the device block layout a miss is a plain copy of
// its bytes: 16-byte pieces over the whole grid, four in flight per thread.
__global__ void __launch_bounds__(256) prefill_copy_kernel(MissFetch f, const int32_t* n_miss) {
  const int m = *n_miss;
  const int64_t per = f.expert_bytes / 16;
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  for (int j = 0; j < m; ++j) {
    const int64_t entry = ((int64_t)f.layer * f.E + __ldcg(&f.miss_expert[j])) % f.pool_entries;
    const uint4* src = reinterpret_cast<const uint4*>(f.host_pool + entry * f.expert_bytes);
    uint4* dst = reinterpret_cast<uint4*>(f.slots + (int64_t)__ldcg(&f.miss_slot[j]) * f.expert_bytes);
    int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; c + 3 * nthr < per; c += 4 * nthr) {
      const uint4 v0 = src[c], v1 = src[c + nthr], v2 = src[c + 2 * nthr], v3 = src[c + 3 * nthr];
      dst[c] = v0;
      dst[c + nthr] = v1;
      dst[c + 2 * nthr] = v2;
      dst[c + 3 * nthr] = v3;
    }
    for (; c < per; c += nthr) dst[c] = src[c];
  }
}

cudaError_t launch_prefill_fetch(const MissFetch& f, const int32_t* n_miss, bool device_layout, cudaStream_t s,
                                 int num_sms) {
  if (device_layout) {
    prefill_copy_kernel<<<4 * num_sms, 256, 0, s>>>(f, n_miss);
    return cudaGetLastError();
  }
  const size_t dyn = fetch_job_bytes(f.d, f.f);
  cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(prefill_fetch_kernel), dyn);
  if (e != cudaSuccess) return e;
  prefill_fetch_kernel<<<num_sms, kFetchThreads, dyn, s>>>(f, n_miss);
  return cudaGetLastError();
}

}  // namespace moe
