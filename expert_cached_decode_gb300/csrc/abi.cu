// C ABI of the routed-expert FFN step (declared in include/moe_gb300.h).
//
// Host-side orchestration of one layer-call:
//   all keys resident  : route kernel (ROUTE_RESIDENT, stamps the hits) and
//                        the expert kernel, launched back to back with
//                        programmatic dependent launch; no host wait.
//   otherwise          : route kernel (ROUTE_PLAN) -> the host reads the
//                        miss list -> one cudaMemcpyAsync per miss (host pool
//                        -> staging) on a side stream and a re-layout kernel
//                        into the victim slots -> the main stream waits on
//                        the side stream's event -> commit kernel (LRU state,
//                        counters) -> expert kernel.  Nothing of the cache
//                        state changes unless every copy was enqueued.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "moe_gb300.h"
#include "common.cuh"
#include "internal.h"

using namespace moe;

static thread_local std::string g_last_error;

static moe_status fail(moe_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

#define CUDA_TRY(call)                                                                          \
  do {                                                                                          \
    cudaError_t e_ = (call);                                                                    \
    if (e_ != cudaSuccess)                                                                      \
      return fail(e_ == cudaErrorMemoryAllocation ? MOE_ERR_OOM : MOE_ERR_CUDA, "%s: %s (%s:%d)", \
                  #call, cudaGetErrorString(e_), __FILE__, __LINE__);                           \
  } while (0)

struct moe_ctx {
  // shape
  int d = 0, f = 0, E = 0, k = 0, L = 0;
  int64_t B = 0;  // bytes per expert
  float shared_weight = 1.f;
  int device = 0, num_sms = 0;
  // weights
  uint16_t* router_w = nullptr;  // [L][E][d]
  float* router_b = nullptr;     // [L][E]
  uint8_t* shared = nullptr;     // [L] device layout
  const uint8_t* host_pool = nullptr;
  int64_t P = 0;
  bool registered = false;
  // cache
  bool configured = false, all_resident = false;
  int64_t C = 0;
  uint8_t* slots = nullptr;
  int32_t* table = nullptr;  // [L*E]
  int32_t* owner = nullptr;  // [C]
  int64_t* stamp = nullptr;  // [C]
  int32_t* lruq[2] = {nullptr, nullptr};
  int qcur = 0;
  int64_t* clock = nullptr;
  int64_t* stats = nullptr;  // [L][ST_N]
  // scratch
  float* logits = nullptr;
  uint32_t* route_cnt = nullptr;
  Plan* plan = nullptr;
  Plan* plan_host = nullptr;  // pinned
  float* gu_partial = nullptr;
  uint16_t* hfrag = nullptr;
  float* obuf = nullptr;
  uint32_t* counters = nullptr;  // gu_cnt | h_ready | d_cnt | done
  size_t counters_n = 0;
  uint32_t* gu_cnt = nullptr;
  uint32_t* h_ready = nullptr;
  uint32_t* d_cnt = nullptr;
  uint32_t* done = nullptr;
  uint32_t* err = nullptr;
  int max_exp = 0;
  // miss path
  uint8_t* staging = nullptr;
  int staging_n = 0;
  cudaStream_t side = nullptr;
  cudaEvent_t ev_route = nullptr, ev_copy = nullptr;
};

extern "C" const char* moe_last_error(void) { return g_last_error.c_str(); }

static bool is_device_ptr(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

static moe_status repack_from(moe_ctx* c, const uint8_t* src_canonical, bool src_on_device, int n,
                              uint8_t* dst_base, const int32_t* dst_slot_host, int64_t dst_stride) {
  // copies n canonical experts (host or device) through a device staging
  // buffer and re-lays them out into dst (by slot index or contiguous)
  const int chunk = 32;
  uint8_t* stage = nullptr;
  int32_t* slots_dev = nullptr;
  CUDA_TRY(cudaMalloc(&stage, (size_t)chunk * c->B));
  CUDA_TRY(cudaMalloc(&slots_dev, chunk * sizeof(int32_t)));
  for (int i0 = 0; i0 < n; i0 += chunk) {
    const int m = n - i0 < chunk ? n - i0 : chunk;
    CUDA_TRY(cudaMemcpy(stage, src_canonical + (size_t)i0 * c->B, (size_t)m * c->B,
                        src_on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice));
    RepackArgs ra{};
    ra.src = stage;
    ra.src_stride = c->B;
    ra.dst_base = dst_base;
    ra.dst_stride = dst_stride;
    ra.n_experts = m;
    ra.d = c->d;
    ra.f = c->f;
    if (dst_slot_host) {
      CUDA_TRY(cudaMemcpy(slots_dev, dst_slot_host + i0, m * sizeof(int32_t), cudaMemcpyHostToDevice));
      ra.dst_slot = slots_dev;
    } else {
      ra.dst_base = dst_base + (size_t)i0 * dst_stride;
      ra.dst_slot = nullptr;
    }
    CUDA_TRY(launch_repack(ra, 0));
    CUDA_TRY(cudaDeviceSynchronize());
  }
  cudaFree(stage);
  cudaFree(slots_dev);
  return MOE_OK;
}

extern "C" moe_status moe_layer_create(const moe_layer_desc* desc, moe_ctx** out) {
  if (!desc || !out) return fail(MOE_ERR_INVALID_ARG, "moe_layer_create: NULL argument");
  *out = nullptr;
  const moe_layer_desc& D = *desc;
  if (D.group != 32) return fail(MOE_ERR_UNIMPLEMENTED, "group must be 32 (got %d)", D.group);
  if (D.d <= 0 || D.d % 256 != 0) return fail(MOE_ERR_UNIMPLEMENTED, "d must be a positive multiple of 256");
  if (D.f <= 0 || D.f % 64 != 0 || D.f > 1024)
    return fail(MOE_ERR_UNIMPLEMENTED, "f must be a multiple of 64 in [64, 1024]");
  if (D.top_k < 2 || D.top_k > kMaxTopK || D.n_experts <= D.top_k || D.n_experts > kMaxE)
    return fail(MOE_ERR_UNIMPLEMENTED, "need 2 <= top_k <= 16 and top_k < n_experts <= 1024");
  if (D.n_layers <= 0) return fail(MOE_ERR_INVALID_ARG, "n_layers must be positive");
  if (!D.router_w || !D.shared_q || !D.host_pool)
    return fail(MOE_ERR_INVALID_ARG, "router_w, shared_q and host_pool are required");
  if (D.host_pool_entries < 0) return fail(MOE_ERR_INVALID_ARG, "host_pool_entries < 0");

  moe_ctx* c = new moe_ctx();
  c->d = D.d;
  c->f = D.f;
  c->E = D.n_experts;
  c->k = D.top_k;
  c->L = D.n_layers;
  c->B = (int64_t)3 * D.d * D.f * 3 / 8 + (int64_t)3 * D.d * D.f / 32 * 2;
  c->shared_weight = D.shared_weight;
  c->P = D.host_pool_entries ? D.host_pool_entries : (int64_t)D.n_layers * D.n_experts;
  c->host_pool = static_cast<const uint8_t*>(D.host_pool);
  moe_status st = MOE_OK;
#define CREATE_TRY(call)                      \
  do {                                        \
    cudaError_t e_ = (call);                  \
    if (e_ != cudaSuccess) {                  \
      st = fail(e_ == cudaErrorMemoryAllocation ? MOE_ERR_OOM : MOE_ERR_CUDA, "%s: %s", #call, \
                cudaGetErrorString(e_));      \
      moe_layer_destroy(c);                   \
      return st;                              \
    }                                         \
  } while (0)
  CREATE_TRY(cudaGetDevice(&c->device));
  CREATE_TRY(cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device));
  const size_t LE = (size_t)c->L * c->E;
  CREATE_TRY(cudaMalloc(&c->router_w, LE * c->d * sizeof(uint16_t)));
  CREATE_TRY(cudaMemcpy(c->router_w, D.router_w, LE * c->d * sizeof(uint16_t), cudaMemcpyDefault));
  CREATE_TRY(cudaMalloc(&c->router_b, LE * sizeof(float)));
  if (D.router_b)
    CREATE_TRY(cudaMemcpy(c->router_b, D.router_b, LE * sizeof(float), cudaMemcpyDefault));
  else
    CREATE_TRY(cudaMemset(c->router_b, 0, LE * sizeof(float)));
  CREATE_TRY(cudaMalloc(&c->shared, (size_t)c->L * c->B));
  st = repack_from(c, static_cast<const uint8_t*>(D.shared_q), is_device_ptr(D.shared_q), c->L, c->shared,
                   nullptr, c->B);
  if (st != MOE_OK) {
    moe_layer_destroy(c);
    return st;
  }
  // host pool: pinned already, or register it
  {
    cudaPointerAttributes at;
    cudaError_t e = cudaPointerGetAttributes(&at, D.host_pool);
    if (e != cudaSuccess) cudaGetLastError();
    if (e != cudaSuccess || at.type == cudaMemoryTypeUnregistered) {
      e = cudaHostRegister(const_cast<void*>(D.host_pool), (size_t)c->P * c->B, cudaHostRegisterDefault);
      if (e != cudaSuccess) {
        cudaGetLastError();
        moe_layer_destroy(c);
        return fail(MOE_ERR_HOST_PIN, "cudaHostRegister of the host pool (%lld bytes) failed: %s",
                    (long long)(c->P * c->B), cudaGetErrorString(e));
      }
      c->registered = true;
    } else if (at.type == cudaMemoryTypeDevice) {
      moe_layer_destroy(c);
      return fail(MOE_ERR_INVALID_ARG, "host_pool must be host memory");
    }
  }
  // scratch
  c->max_exp = (kMaxDecodeT * c->k < c->E ? kMaxDecodeT * c->k : c->E) + 1;
  const int RG = c->f / 32, KC = c->d / 256, RD = c->d / 32;
  CREATE_TRY(cudaMalloc(&c->logits, (size_t)kMaxDecodeT * c->E * sizeof(float)));
  CREATE_TRY(cudaMalloc(&c->route_cnt, sizeof(uint32_t)));
  CREATE_TRY(cudaMemset(c->route_cnt, 0, sizeof(uint32_t)));
  CREATE_TRY(cudaMalloc(&c->plan, sizeof(Plan)));
  CREATE_TRY(cudaMemset(c->plan, 0, sizeof(Plan)));
  CREATE_TRY(cudaHostAlloc(&c->plan_host, sizeof(Plan), cudaHostAllocDefault));
  CREATE_TRY(cudaMalloc(&c->gu_partial, (size_t)c->max_exp * RG * KC * 2 * 512 * sizeof(float)));
  CREATE_TRY(cudaMalloc(&c->hfrag, (size_t)c->max_exp * 2 * RG * 2 * 32 * 4 * sizeof(uint16_t)));
  CREATE_TRY(cudaMalloc(&c->obuf, (size_t)c->max_exp * kMaxDecodeT * c->d * sizeof(float)));
  c->counters_n = (size_t)c->max_exp * RG + c->max_exp + RD + 1;
  CREATE_TRY(cudaMalloc(&c->counters, c->counters_n * sizeof(uint32_t)));
  CREATE_TRY(cudaMemset(c->counters, 0, c->counters_n * sizeof(uint32_t)));
  c->gu_cnt = c->counters;
  c->h_ready = c->gu_cnt + (size_t)c->max_exp * RG;
  c->d_cnt = c->h_ready + c->max_exp;
  c->done = c->d_cnt + RD;
  CREATE_TRY(cudaMalloc(&c->err, sizeof(uint32_t)));
  CREATE_TRY(cudaMemset(c->err, 0, sizeof(uint32_t)));
  CREATE_TRY(cudaMalloc(&c->clock, sizeof(int64_t)));
  CREATE_TRY(cudaMemset(c->clock, 0, sizeof(int64_t)));
  CREATE_TRY(cudaMalloc(&c->stats, (size_t)c->L * ST_N * sizeof(int64_t)));
  CREATE_TRY(cudaMemset(c->stats, 0, (size_t)c->L * ST_N * sizeof(int64_t)));
  CREATE_TRY(cudaMalloc(&c->table, LE * sizeof(int32_t)));
  CREATE_TRY(cudaMemset(c->table, 0xff, LE * sizeof(int32_t)));
  CREATE_TRY(cudaStreamCreateWithFlags(&c->side, cudaStreamNonBlocking));
  CREATE_TRY(cudaEventCreateWithFlags(&c->ev_route, cudaEventDisableTiming));
  CREATE_TRY(cudaEventCreateWithFlags(&c->ev_copy, cudaEventDisableTiming));
  CREATE_TRY(cudaDeviceSynchronize());
#undef CREATE_TRY
  *out = c;
  return MOE_OK;
}

extern "C" void moe_layer_destroy(moe_ctx* c) {
  if (!c) return;
  cudaDeviceSynchronize();
  cudaFree(c->router_w);
  cudaFree(c->router_b);
  cudaFree(c->shared);
  cudaFree(c->slots);
  cudaFree(c->table);
  cudaFree(c->owner);
  cudaFree(c->stamp);
  cudaFree(c->lruq[0]);
  cudaFree(c->lruq[1]);
  cudaFree(c->clock);
  cudaFree(c->stats);
  cudaFree(c->logits);
  cudaFree(c->route_cnt);
  cudaFree(c->plan);
  if (c->plan_host) cudaFreeHost(c->plan_host);
  cudaFree(c->gu_partial);
  cudaFree(c->hfrag);
  cudaFree(c->obuf);
  cudaFree(c->counters);
  cudaFree(c->err);
  cudaFree(c->staging);
  if (c->side) cudaStreamDestroy(c->side);
  if (c->ev_route) cudaEventDestroy(c->ev_route);
  if (c->ev_copy) cudaEventDestroy(c->ev_copy);
  if (c->registered) cudaHostUnregister(const_cast<uint8_t*>(c->host_pool));
  cudaGetLastError();
  delete c;
}

extern "C" moe_status moe_cache_configure(moe_ctx* c, int64_t capacity, const int32_t* keys, int64_t n_pre) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "NULL context");
  const int64_t LE = (int64_t)c->L * c->E;
  const int64_t min_cap = (int64_t)kMaxDecodeT * c->k < c->E ? (int64_t)kMaxDecodeT * c->k : c->E;
  if (capacity < min_cap || capacity > kMaxSlots)
    return fail(MOE_ERR_INVALID_ARG, "capacity %lld outside [%lld, %d]", (long long)capacity,
                (long long)min_cap, kMaxSlots);
  if (n_pre < 0 || n_pre > capacity || n_pre > LE || (n_pre > 0 && !keys))
    return fail(MOE_ERR_INVALID_ARG, "bad preload list");
  for (int64_t i = 0; i < n_pre; ++i) {
    if (keys[i] < 0 || keys[i] >= LE || (i > 0 && keys[i] <= keys[i - 1]))
      return fail(MOE_ERR_INVALID_ARG, "preload keys must be strictly ascending in [0, L*E)");
  }
  CUDA_TRY(cudaDeviceSynchronize());
  cudaFree(c->slots);
  cudaFree(c->owner);
  cudaFree(c->stamp);
  cudaFree(c->lruq[0]);
  cudaFree(c->lruq[1]);
  cudaFree(c->staging);
  c->slots = nullptr;
  c->owner = nullptr;
  c->stamp = nullptr;
  c->lruq[0] = c->lruq[1] = nullptr;
  c->staging = nullptr;
  c->configured = false;
  CUDA_TRY(cudaMalloc(&c->slots, (size_t)capacity * c->B));
  CUDA_TRY(cudaMalloc(&c->owner, capacity * sizeof(int32_t)));
  CUDA_TRY(cudaMalloc(&c->stamp, capacity * sizeof(int64_t)));
  CUDA_TRY(cudaMalloc(&c->lruq[0], capacity * sizeof(int32_t)));
  CUDA_TRY(cudaMalloc(&c->lruq[1], capacity * sizeof(int32_t)));
  c->C = capacity;
  c->all_resident = (n_pre == LE);
  if (!c->all_resident) {
    c->staging_n = (int)min_cap;
    CUDA_TRY(cudaMalloc(&c->staging, (size_t)c->staging_n * c->B));
  }
  std::vector<int32_t> owner(capacity, -1), q(capacity), table(LE, -1);
  std::vector<int64_t> stamp(capacity, -1);
  for (int64_t s = 0; s < capacity; ++s) q[s] = (int32_t)s;
  for (int64_t i = 0; i < n_pre; ++i) {
    owner[i] = keys[i];
    table[keys[i]] = (int32_t)i;
  }
  CUDA_TRY(cudaMemcpy(c->owner, owner.data(), capacity * sizeof(int32_t), cudaMemcpyHostToDevice));
  CUDA_TRY(cudaMemcpy(c->stamp, stamp.data(), capacity * sizeof(int64_t), cudaMemcpyHostToDevice));
  CUDA_TRY(cudaMemcpy(c->lruq[0], q.data(), capacity * sizeof(int32_t), cudaMemcpyHostToDevice));
  CUDA_TRY(cudaMemcpy(c->table, table.data(), LE * sizeof(int32_t), cudaMemcpyHostToDevice));
  c->qcur = 0;
  CUDA_TRY(cudaMemset(c->clock, 0, sizeof(int64_t)));
  CUDA_TRY(cudaMemset(c->stats, 0, (size_t)c->L * ST_N * sizeof(int64_t)));
  // preload: gather the canonical experts of the keys (pool entry key mod P)
  const int chunk = 32;
  std::vector<int32_t> slot_ids(chunk);
  uint8_t* stage = nullptr;
  int32_t* slots_dev = nullptr;
  CUDA_TRY(cudaMalloc(&stage, (size_t)chunk * c->B));
  CUDA_TRY(cudaMalloc(&slots_dev, chunk * sizeof(int32_t)));
  for (int64_t i0 = 0; i0 < n_pre; i0 += chunk) {
    const int m = (int)(n_pre - i0 < chunk ? n_pre - i0 : chunk);
    for (int j = 0; j < m; ++j) {
      const int64_t entry = keys[i0 + j] % c->P;
      CUDA_TRY(cudaMemcpyAsync(stage + (size_t)j * c->B, c->host_pool + (size_t)entry * c->B, c->B,
                               cudaMemcpyHostToDevice, 0));
      slot_ids[j] = (int32_t)(i0 + j);
    }
    CUDA_TRY(cudaMemcpy(slots_dev, slot_ids.data(), m * sizeof(int32_t), cudaMemcpyHostToDevice));
    RepackArgs ra{};
    ra.src = stage;
    ra.src_stride = c->B;
    ra.dst_base = c->slots;
    ra.dst_slot = slots_dev;
    ra.dst_stride = c->B;
    ra.n_experts = m;
    ra.d = c->d;
    ra.f = c->f;
    CUDA_TRY(launch_repack(ra, 0));
    CUDA_TRY(cudaDeviceSynchronize());
  }
  cudaFree(stage);
  cudaFree(slots_dev);
  CUDA_TRY(cudaDeviceSynchronize());
  c->configured = true;
  return MOE_OK;
}

static moe_status check_common(moe_ctx* c, int layer, const void* x, int T, int maxT) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "NULL context");
  if (layer < 0 || layer >= c->L) return fail(MOE_ERR_INVALID_ARG, "layer %d out of range", layer);
  if (!x) return fail(MOE_ERR_INVALID_ARG, "NULL input");
  if (T < 1 || T > maxT) return fail(MOE_ERR_INVALID_ARG, "T=%d outside [1, %d]", T, maxT);
  return MOE_OK;
}

static RouteArgs route_args(moe_ctx* c, int layer, const void* x, int T, int mode) {
  RouteArgs ra{};
  ra.x = static_cast<const uint16_t*>(x);
  ra.wr = c->router_w + (size_t)layer * c->E * c->d;
  ra.bias = c->router_b + (size_t)layer * c->E;
  ra.T = T;
  ra.d = c->d;
  ra.E = c->E;
  ra.k = c->k;
  ra.layer = layer;
  ra.mode = mode;
  ra.logits = c->logits;
  ra.cnt = c->route_cnt;
  ra.plan = c->plan;
  ra.table = c->table;
  ra.owner = c->owner;
  ra.stamp = c->stamp;
  ra.q_in = c->lruq[c->qcur];
  ra.q_out = c->lruq[c->qcur ^ 1];
  ra.C = (int)c->C;
  ra.clock = c->clock;
  ra.stats = c->stats + (size_t)layer * ST_N;
  ra.expert_bytes = c->B;
  ra.err = c->err;
  return ra;
}

extern "C" moe_status moe_route_topk(moe_ctx* c, int32_t layer, const void* x, int32_t T, int32_t* idx,
                                     float* w, void* stream) {
  moe_status st = check_common(c, layer, x, T, kMaxDecodeT);
  if (st != MOE_OK) return st;
  if (!idx || !w) return fail(MOE_ERR_INVALID_ARG, "NULL output");
  RouteArgs ra = route_args(c, layer, x, T, ROUTE_ONLY);
  ra.out_idx = idx;
  ra.out_w = w;
  CUDA_TRY(launch_route(ra, static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

static FfnArgs ffn_args(moe_ctx* c, int layer, const void* x, int T, float* y) {
  FfnArgs fa{};
  fa.slots = c->slots;
  fa.shared_expert = c->shared + (size_t)layer * c->B;
  fa.expert_bytes = c->B;
  fa.x = static_cast<const uint16_t*>(x);
  fa.y = y;
  fa.T = T;
  fa.d = c->d;
  fa.f = c->f;
  fa.k = c->k;
  fa.shared_weight = c->shared_weight;
  fa.plan = c->plan;
  fa.gu_partial = c->gu_partial;
  fa.hfrag = c->hfrag;
  fa.obuf = c->obuf;
  fa.gu_cnt = c->gu_cnt;
  fa.h_ready = c->h_ready;
  fa.d_cnt = c->d_cnt;
  fa.done = c->done;
  fa.err = c->err;
  fa.grid = c->num_sms;
  return fa;
}

static moe_status fill_trace(moe_ctx* c, cudaStream_t s, int T, moe_trace* tr) {
  CUDA_TRY(cudaMemcpyAsync(c->plan_host, c->plan, sizeof(Plan), cudaMemcpyDeviceToHost, s));
  CUDA_TRY(cudaStreamSynchronize(s));
  const Plan& p = *c->plan_host;
  const int n = T * c->k;
  for (int i = 0; i < n; ++i) {
    if (tr->idx) tr->idx[i] = p.idx[i];
    if (tr->w) tr->w[i] = p.w[i];
    if (tr->slot) tr->slot[i] = p.act_slot[p.pick_act[i]];
  }
  for (int j = 0; j < p.n_miss; ++j) {
    if (tr->miss_expert) tr->miss_expert[j] = p.miss_expert[j];
    if (tr->miss_slot) tr->miss_slot[j] = p.miss_slot[j];
    if (tr->evicted_key) tr->evicted_key[j] = p.evicted_key[j];
  }
  tr->n_miss = p.n_miss;
  tr->n_distinct = p.n_act;
  tr->token_hits = p.token_hits;
  tr->token_misses = p.token_misses;
  return MOE_OK;
}

extern "C" moe_status moe_forward(moe_ctx* c, int32_t layer, const void* x, int32_t T, float* y, void* stream,
                                  moe_trace* trace) {
  moe_status st = check_common(c, layer, x, T, kMaxDecodeT);
  if (st != MOE_OK) {
    if (c && T > kMaxDecodeT && T <= 16384)
      return fail(MOE_ERR_UNIMPLEMENTED, "prefill path (T > %d) not available in this build", kMaxDecodeT);
    return st;
  }
  if (!c->configured) return fail(MOE_ERR_STATE, "moe_cache_configure must come first");
  if (!y) return fail(MOE_ERR_INVALID_ARG, "NULL output");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  FfnArgs fa = ffn_args(c, layer, x, T, y);
  if (c->all_resident) {
    RouteArgs ra = route_args(c, layer, x, T, ROUTE_RESIDENT);
    CUDA_TRY(launch_route(ra, s));
    CUDA_TRY(launch_decode_ffn(fa, s, true, c->num_sms));
    if (trace) return fill_trace(c, s, T, trace);
    return MOE_OK;
  }
  // miss-capable path
  RouteArgs ra = route_args(c, layer, x, T, ROUTE_PLAN);
  CUDA_TRY(launch_route(ra, s));
  CUDA_TRY(cudaMemcpyAsync(c->plan_host, c->plan, sizeof(Plan), cudaMemcpyDeviceToHost, s));
  CUDA_TRY(cudaEventRecord(c->ev_route, s));
  CUDA_TRY(cudaEventSynchronize(c->ev_route));
  const Plan& p = *c->plan_host;
  const int m = p.n_miss;
  if (m < 0 || m > c->staging_n) return fail(MOE_ERR_CUDA, "corrupt routing plan (n_miss=%d)", m);
  for (int j = 0; j < m; ++j) {
    const int64_t key = (int64_t)layer * c->E + p.miss_expert[j];
    const int64_t entry = key % c->P;
    CUDA_TRY(cudaMemcpyAsync(c->staging + (size_t)j * c->B, c->host_pool + (size_t)entry * c->B, c->B,
                             cudaMemcpyHostToDevice, c->side));
  }
  if (m > 0) {
    RepackArgs rp{};
    rp.src = c->staging;
    rp.src_stride = c->B;
    rp.dst_base = c->slots;
    rp.dst_slot = c->plan->miss_slot;
    rp.dst_stride = c->B;
    rp.n_experts = m;
    rp.d = c->d;
    rp.f = c->f;
    CUDA_TRY(launch_repack(rp, c->side));
  }
  CUDA_TRY(cudaEventRecord(c->ev_copy, c->side));
  CUDA_TRY(cudaStreamWaitEvent(s, c->ev_copy, 0));
  CommitArgs ca{};
  ca.plan = c->plan;
  ca.table = c->table;
  ca.owner = c->owner;
  ca.stamp = c->stamp;
  ca.clock = c->clock;
  ca.stats = c->stats + (size_t)layer * ST_N;
  ca.layer = layer;
  ca.E = c->E;
  ca.expert_bytes = c->B;
  CUDA_TRY(launch_commit(ca, s));
  c->qcur ^= 1;
  CUDA_TRY(launch_decode_ffn(fa, s, false, c->num_sms));
  if (trace) {
    moe_status t = fill_trace(c, s, T, trace);
    if (t != MOE_OK) return t;
    // plan_host was refreshed after the call; the miss list is that of this call
  }
  return MOE_OK;
}

static moe_status check_device_error(moe_ctx* c) {
  uint32_t e = 0;
  CUDA_TRY(cudaMemcpy(&e, c->err, sizeof(e), cudaMemcpyDeviceToHost));
  if (e != 0) {
    CUDA_TRY(cudaMemset(c->err, 0, sizeof(uint32_t)));
    CUDA_TRY(cudaMemset(c->counters, 0, c->counters_n * sizeof(uint32_t)));
    CUDA_TRY(cudaMemset(c->route_cnt, 0, sizeof(uint32_t)));
    CUDA_TRY(cudaDeviceSynchronize());
    return fail(e == DEV_NOT_RESIDENT ? MOE_ERR_STATE : MOE_ERR_TIMEOUT,
                "device error %u (1: barrier wait, 2: flag wait, 3: key not resident)", e);
  }
  return MOE_OK;
}

extern "C" moe_status moe_sync(moe_ctx* c) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "NULL context");
  CUDA_TRY(cudaDeviceSynchronize());
  return check_device_error(c);
}

extern "C" moe_status moe_cache_stats(moe_ctx* c, moe_stats* total, moe_stats* per_layer) {
  if (!c || !total) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
  CUDA_TRY(cudaDeviceSynchronize());
  std::vector<int64_t> s((size_t)c->L * ST_N);
  CUDA_TRY(cudaMemcpy(s.data(), c->stats, s.size() * sizeof(int64_t), cudaMemcpyDeviceToHost));
  memset(total, 0, sizeof(*total));
  for (int l = 0; l < c->L; ++l) {
    const int64_t* r = &s[(size_t)l * ST_N];
    moe_stats one{r[ST_CALLS], r[ST_TOK_HIT], r[ST_TOK_MISS], r[ST_DIST_HIT], r[ST_DIST_MISS], r[ST_EVICT],
                  r[ST_MISS_BYTES]};
    if (per_layer) per_layer[l] = one;
    total->layer_calls += one.layer_calls;
    total->token_hits += one.token_hits;
    total->token_misses += one.token_misses;
    total->distinct_hits += one.distinct_hits;
    total->distinct_misses += one.distinct_misses;
    total->evictions += one.evictions;
    total->miss_bytes += one.miss_bytes;
  }
  return check_device_error(c);
}

extern "C" moe_status moe_cache_export(moe_ctx* c, int32_t* owner, int64_t* stamp) {
  if (!c || !owner || !stamp) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
  if (!c->configured) return fail(MOE_ERR_STATE, "cache not configured");
  CUDA_TRY(cudaDeviceSynchronize());
  CUDA_TRY(cudaMemcpy(owner, c->owner, c->C * sizeof(int32_t), cudaMemcpyDeviceToHost));
  CUDA_TRY(cudaMemcpy(stamp, c->stamp, c->C * sizeof(int64_t), cudaMemcpyDeviceToHost));
  return MOE_OK;
}
