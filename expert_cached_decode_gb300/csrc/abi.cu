// C ABI of the routed-expert FFN step (declared in include/moe_gb300.h).
//
// Host-side orchestration of one layer-call:
//   all keys resident  : one launch of the decode kernel with fused routing
//                        (router, selection, stamps of the hits, expert
//                        work); programmatic dependent launch lets it be
//                        scheduled while the previous call drains.  No host
//                        wait.
//   misses, GPU pull   : one launch of the decode kernel in its cached mode
//   (default)            (CTA 0 plans and commits the cache, the other CTAs
//                        pull the misses from the registered host pool into
//                        their victim slots, then run the experts).  No host
//                        wait.
//   misses, host copies: route kernel (ROUTE_PLAN) -> the host reads the
//                        miss list -> one cudaMemcpyAsync per miss (host pool
//                        -> staging) on a side stream and a re-layout kernel
//                        into the victim slots -> the main stream waits on
//                        the side stream's event -> commit kernel (LRU state,
//                        counters) -> expert kernel.  Nothing of the cache
//                        state changes unless every copy was enqueued.
#include <cuda.h>
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
#include "fetch.cuh"

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

namespace moe {
moe_status set_last_error(moe_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}
}  // namespace moe

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
  const uint8_t* host_pool_dev = nullptr;   // device address of the registered pool (NULL: none)
  bool pull = false;                        // misses pulled by the GPU
  bool pool_dev_layout = false;             // host pool entries already in the device block layout
  // lookahead (moe_forward_ahead): a layer-call whose routing, cache step and
  // miss copies are done and whose experts run next; its plan is plans(ahead_pi)
  Plan* plan2 = nullptr;
  bool ahead_valid = false;
  int ahead_layer = -1, ahead_T = 0, ahead_pi = 0;
  const void* ahead_x = nullptr;
  Plan* plans(int i) { return i ? plan2 : plan; }
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
  uint64_t* ypart = nullptr;     // [num_sms][16][d] per-CTA partials of y, (call tag, value) words
  uint64_t* tlogits = nullptr;   // [16][E] router logits of the decode kernel, (call tag, value) words
  uint32_t* counters = nullptr;  // decode calls | 2 sets of kDecodeSetWords counters
  size_t counters_n = 0;
  int set_words = 0;
  uint32_t* err = nullptr;
  uint64_t wait_ns = kWaitLimitNs;   // limit of every bounded device wait
  // prefill scratch (allocated on first use, sized for kMaxPrefillT tokens)
  float* p_logits = nullptr;
  int32_t* p_idx = nullptr;
  float* p_w = nullptr;
  int32_t* p_counts = nullptr;
  uint16_t* p_xg = nullptr;      // [T*(k+1)][d] fp16, expert-sorted activations
  uint16_t* p_hg = nullptr;      // [T*(k+1)][f] fp16 (hi part of h)
  uint16_t* p_hg_lo = nullptr;   // [T*(k+1)][f] fp16 (lo part of h)
  int32_t* p_perm = nullptr;
  float* p_wsort = nullptr;
  int32_t* p_pick = nullptr;     // [T*k] pick of each routed sorted row
  int32_t* p_miss_expert = nullptr;   // [E] the chunk's misses (cache that can miss)
  int32_t* p_miss_slot = nullptr;
  int32_t* p_evicted = nullptr;
  int32_t* p_info = nullptr;          // [4] misses, distinct, token hits, token misses
  float* p_osort = nullptr;      // [T*k][d] weighted output of each routed pick
  int32_t* p_cursor = nullptr;
  int32_t* p_group_slot = nullptr;
  PrefillTile* p_tiles_gu = nullptr;
  PrefillTile* p_tiles_dn = nullptr;
  int32_t* p_ntiles = nullptr;
  int64_t p_max_tiles = 0;
  // miss path
  uint8_t* staging = nullptr;
  int staging_n = 0;
  cudaStream_t side = nullptr;
  cudaEvent_t ev_route = nullptr, ev_copy = nullptr;
};

extern "C" const char* moe_last_error(void) { return g_last_error.c_str(); }

// ---- host-side failure injection (test hook; disarmed by default) ---------
static int g_inject_kind = 0;
static int64_t g_inject_left = 0;

// true (and disarmed) when this is the armed kind's nth event
static bool injected(int kind) {
  if (g_inject_kind != kind) return false;
  if (--g_inject_left > 0) return false;
  g_inject_kind = 0;
  return true;
}

extern "C" moe_status moe_debug_inject_failure(int32_t kind, int64_t nth) {
  if (kind == 0) {
    g_inject_kind = 0;
    return MOE_OK;
  }
  if ((kind != MOE_INJECT_MISS_COPY && kind != MOE_INJECT_HOLD_ROUTER && kind != MOE_INJECT_HOST_REGISTER &&
       kind != MOE_INJECT_DEVICE_ALLOC) ||
      nth < 1)
    return fail(MOE_ERR_INVALID_ARG, "moe_debug_inject_failure: unknown kind %d or nth %lld < 1", kind,
                (long long)nth);
  g_inject_kind = kind;
  g_inject_left = nth;
  return MOE_OK;
}

extern "C" moe_status moe_debug_set_wait_limit(moe_ctx* c, int64_t ns) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "NULL context");
  if (ns <= 0) return fail(MOE_ERR_INVALID_ARG, "wait limit must be positive (got %lld ns)", (long long)ns);
  c->wait_ns = (uint64_t)ns;
  return MOE_OK;
}

// device allocation of create/configure (fails on an armed injection)
static cudaError_t dev_alloc(void* p, size_t bytes) {
  if (injected(MOE_INJECT_DEVICE_ALLOC)) return cudaErrorMemoryAllocation;
  return cudaMalloc(reinterpret_cast<void**>(p), bytes);
}

constexpr int kMaxPrefillT = 16384;

// ---- TMA tensor maps (driver entry point fetched through the runtime) -----
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D row-major [rows][cols] 16-bit tensor, box = 64 columns x box_rows rows,
// 128-byte swizzle.
static moe_status make_tmap_2d(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows,
                               bool bf16) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return MOE_OK;
}

static bool is_device_ptr(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

// frees the device buffers it holds when it goes out of scope
struct DevTemp {
  void* p[4] = {nullptr, nullptr, nullptr, nullptr};
  ~DevTemp() {
    for (void* q : p) cudaFree(q);
  }
};

static moe_status repack_from(moe_ctx* c, const uint8_t* src_canonical, bool src_on_device, int n,
                              uint8_t* dst_base, const int32_t* dst_slot_host, int64_t dst_stride) {
  // copies n canonical experts (host or device) through a device staging
  // buffer and re-lays them out into dst (by slot index or contiguous)
  const int chunk = 32;
  DevTemp tmp;
  CUDA_TRY(dev_alloc(&tmp.p[0], (size_t)chunk * c->B));
  CUDA_TRY(dev_alloc(&tmp.p[1], chunk * sizeof(int32_t)));
  uint8_t* stage = static_cast<uint8_t*>(tmp.p[0]);
  int32_t* slots_dev = static_cast<int32_t*>(tmp.p[1]);
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
  return MOE_OK;
}

extern "C" moe_status moe_layer_create(const moe_layer_desc* desc, moe_ctx** out) {
  if (!desc || !out) return fail(MOE_ERR_INVALID_ARG, "moe_layer_create: NULL argument");
  *out = nullptr;
  const moe_layer_desc& D = *desc;
  if (D.group != 32) return fail(MOE_ERR_UNIMPLEMENTED, "group must be 32 (got %d)", D.group);
  if (D.d <= 0 || D.d % 256 != 0 || D.d > 2048)
    return fail(MOE_ERR_UNIMPLEMENTED, "d must be a positive multiple of 256, at most 2048");
  if (D.f <= 0 || D.f % 64 != 0 || D.f > 1024)
    return fail(MOE_ERR_UNIMPLEMENTED, "f must be a multiple of 64 in [64, 1024]");
  if (D.top_k < 2 || D.top_k > kMaxTopK || D.n_experts <= D.top_k || D.n_experts > kMaxE)
    return fail(MOE_ERR_UNIMPLEMENTED, "need 2 <= top_k <= 16 and top_k < n_experts <= 1024");
  if (D.n_layers <= 0) return fail(MOE_ERR_INVALID_ARG, "n_layers must be positive");
  if (!D.router_w || !D.shared_q || !D.host_pool)
    return fail(MOE_ERR_INVALID_ARG, "router_w, shared_q and host_pool are required");
  if (D.host_pool_entries < 0) return fail(MOE_ERR_INVALID_ARG, "host_pool_entries < 0");
  if (D.host_pool_layout != MOE_POOL_CANONICAL && D.host_pool_layout != MOE_POOL_DEVICE)
    return fail(MOE_ERR_INVALID_ARG, "host_pool_layout must be MOE_POOL_CANONICAL or MOE_POOL_DEVICE");

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
  c->pool_dev_layout = D.host_pool_layout == MOE_POOL_DEVICE;
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
  {
    // the decode kernel runs one CTA per SM and its grid-wide counters need
    // all of them resident at once
    bool fits = false;
    CREATE_TRY(decode_ffn_fits(c->d, &fits));
    if (!fits) {
      moe_layer_destroy(c);
      return fail(MOE_ERR_UNIMPLEMENTED, "the decode kernel does not fit one CTA per SM at d=%d", D.d);
    }
  }
  const size_t LE = (size_t)c->L * c->E;
  CREATE_TRY(dev_alloc(&c->router_w, LE * c->d * sizeof(uint16_t)));
  CREATE_TRY(cudaMemcpy(c->router_w, D.router_w, LE * c->d * sizeof(uint16_t), cudaMemcpyDefault));
  CREATE_TRY(dev_alloc(&c->router_b, LE * sizeof(float)));
  if (D.router_b)
    CREATE_TRY(cudaMemcpy(c->router_b, D.router_b, LE * sizeof(float), cudaMemcpyDefault));
  else
    CREATE_TRY(cudaMemset(c->router_b, 0, LE * sizeof(float)));
  CREATE_TRY(dev_alloc(&c->shared, (size_t)c->L * c->B));
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
      e = injected(MOE_INJECT_HOST_REGISTER)
              ? cudaErrorMemoryAllocation
              : cudaHostRegister(const_cast<void*>(D.host_pool), (size_t)c->P * c->B, cudaHostRegisterDefault);
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
    // the GPU's address of the pool, for misses pulled by the GPU itself
    void* dp = nullptr;
    if (cudaHostGetDevicePointer(&dp, const_cast<void*>(D.host_pool), 0) == cudaSuccess && dp) {
      c->host_pool_dev = static_cast<const uint8_t*>(dp);
      c->pull = true;
    } else {
      cudaGetLastError();
    }
  }
  // scratch
  CREATE_TRY(dev_alloc(&c->logits, (size_t)kMaxDecodeT * c->E * sizeof(float)));
  CREATE_TRY(dev_alloc(&c->route_cnt, sizeof(uint32_t)));
  CREATE_TRY(cudaMemset(c->route_cnt, 0, sizeof(uint32_t)));
  CREATE_TRY(dev_alloc(&c->plan, sizeof(Plan)));
  CREATE_TRY(dev_alloc(&c->plan2, sizeof(Plan)));
  CREATE_TRY(cudaMemset(c->plan, 0, sizeof(Plan)));
  CREATE_TRY(cudaHostAlloc(&c->plan_host, sizeof(Plan), cudaHostAllocDefault));
  CREATE_TRY(dev_alloc(&c->ypart, (size_t)c->num_sms * kMaxDecodeT * c->d * sizeof(uint64_t)));
  CREATE_TRY(dev_alloc(&c->tlogits, (size_t)kMaxDecodeT * c->E * sizeof(uint64_t)));
  // tag 0xffffffff: no call's tag, so nothing reads as written before it is
  CREATE_TRY(cudaMemset(c->ypart, 0xff, (size_t)c->num_sms * kMaxDecodeT * c->d * sizeof(uint64_t)));
  CREATE_TRY(cudaMemset(c->tlogits, 0xff, (size_t)kMaxDecodeT * c->E * sizeof(uint64_t)));
  // router counter | partials counter | cache-mode flags: victims published,
  // misses pulled, misses placed
  c->set_words = kDecodeSetWords;
  c->counters_n = 1 + 2 * (size_t)c->set_words;
  CREATE_TRY(dev_alloc(&c->counters, c->counters_n * sizeof(uint32_t)));
  CREATE_TRY(cudaMemset(c->counters, 0, c->counters_n * sizeof(uint32_t)));
  CREATE_TRY(dev_alloc(&c->err, sizeof(uint32_t)));
  CREATE_TRY(cudaMemset(c->err, 0, sizeof(uint32_t)));
  CREATE_TRY(dev_alloc(&c->clock, sizeof(int64_t)));
  CREATE_TRY(cudaMemset(c->clock, 0, sizeof(int64_t)));
  CREATE_TRY(dev_alloc(&c->stats, (size_t)c->L * ST_N * sizeof(int64_t)));
  CREATE_TRY(cudaMemset(c->stats, 0, (size_t)c->L * ST_N * sizeof(int64_t)));
  CREATE_TRY(dev_alloc(&c->table, LE * sizeof(int32_t)));
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
  cudaFree(c->plan2);
  if (c->plan_host) cudaFreeHost(c->plan_host);
  cudaFree(c->ypart);
  cudaFree(c->tlogits);
  cudaFree(c->counters);
  cudaFree(c->err);
  cudaFree(c->staging);
  cudaFree(c->p_logits);
  cudaFree(c->p_idx);
  cudaFree(c->p_w);
  cudaFree(c->p_counts);
  cudaFree(c->p_xg);
  cudaFree(c->p_hg);
  cudaFree(c->p_hg_lo);
  cudaFree(c->p_perm);
  cudaFree(c->p_wsort);
  cudaFree(c->p_pick);
  cudaFree(c->p_miss_expert);
  cudaFree(c->p_miss_slot);
  cudaFree(c->p_evicted);
  cudaFree(c->p_info);
  cudaFree(c->p_osort);
  cudaFree(c->p_cursor);
  cudaFree(c->p_group_slot);
  cudaFree(c->p_tiles_gu);
  cudaFree(c->p_tiles_dn);
  cudaFree(c->p_ntiles);
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
  // Every buffer of the new cache is allocated before the old one is
  // released: when an allocation fails the context keeps its previous cache
  // (slots, LRU state, counters) unchanged.
  const bool all_res = (n_pre == LE);
  const int staging_n = all_res ? 0 : (int)min_cap;
  const int chunk = 32;
  struct {
    void* p[8] = {};
  } nw;
  auto free_new = [&]() {
    for (void*& q : nw.p) {
      cudaFree(q);
      q = nullptr;
    }
  };
  const size_t sizes[8] = {(size_t)capacity * c->B, capacity * sizeof(int32_t), capacity * sizeof(int64_t),
                           capacity * sizeof(int32_t), capacity * sizeof(int32_t), (size_t)staging_n * c->B,
                           (size_t)chunk * c->B, chunk * sizeof(int32_t)};
  for (int i = 0; i < 8; ++i) {
    if (sizes[i] == 0) continue;
    cudaError_t e = dev_alloc(&nw.p[i], sizes[i]);
    if (e != cudaSuccess) {
      cudaGetLastError();
      free_new();
      return fail(e == cudaErrorMemoryAllocation ? MOE_ERR_OOM : MOE_ERR_CUDA,
                  "moe_cache_configure: allocation of %zu bytes failed (%s); the previous cache is unchanged",
                  sizes[i], cudaGetErrorString(e));
    }
  }
  cudaFree(c->slots);
  cudaFree(c->owner);
  cudaFree(c->stamp);
  cudaFree(c->lruq[0]);
  cudaFree(c->lruq[1]);
  cudaFree(c->staging);
  c->slots = static_cast<uint8_t*>(nw.p[0]);
  c->owner = static_cast<int32_t*>(nw.p[1]);
  c->stamp = static_cast<int64_t*>(nw.p[2]);
  c->lruq[0] = static_cast<int32_t*>(nw.p[3]);
  c->lruq[1] = static_cast<int32_t*>(nw.p[4]);
  c->staging = static_cast<uint8_t*>(nw.p[5]);
  DevTemp tmp;   // the preload's staging buffers, freed on every return below
  tmp.p[0] = nw.p[6];
  tmp.p[1] = nw.p[7];
  c->configured = false;   // until the new cache is filled
  c->C = capacity;
  c->all_resident = all_res;
  c->staging_n = staging_n;
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
  // preload: the experts of the keys (pool entry key mod P) into slots 0, 1,
  // ...: a copy each from a device-layout pool, else gathered and re-laid out
  if (c->pool_dev_layout) {
    for (int64_t i = 0; i < n_pre; ++i)
      CUDA_TRY(cudaMemcpyAsync(c->slots + (size_t)i * c->B, c->host_pool + (size_t)(keys[i] % c->P) * c->B, c->B,
                               cudaMemcpyHostToDevice, 0));
    CUDA_TRY(cudaDeviceSynchronize());
    c->configured = true;
  c->ahead_valid = false;
    return MOE_OK;
  }
  std::vector<int32_t> slot_ids(chunk);
  uint8_t* stage = static_cast<uint8_t*>(tmp.p[0]);
  int32_t* slots_dev = static_cast<int32_t*>(tmp.p[1]);
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
  CUDA_TRY(cudaDeviceSynchronize());
  c->configured = true;
  c->ahead_valid = false;
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

// allocates every buffer of `specs` or none: on a failure the ones already
// allocated are released and the targets stay NULL
struct AllocSpec {
  void** target;
  size_t bytes;
};
static moe_status alloc_all(const AllocSpec* specs, int n) {
  for (int i = 0; i < n; ++i) {
    void* p = nullptr;
    cudaError_t e = dev_alloc(&p, specs[i].bytes);
    if (e != cudaSuccess) {
      cudaGetLastError();
      for (int j = 0; j < i; ++j) {
        cudaFree(*specs[j].target);
        *specs[j].target = nullptr;
      }
      return fail(e == cudaErrorMemoryAllocation ? MOE_ERR_OOM : MOE_ERR_CUDA, "allocation of %zu bytes failed: %s",
                  specs[i].bytes, cudaGetErrorString(e));
    }
    *specs[i].target = p;
  }
  return MOE_OK;
}

static moe_status ensure_prefill_scratch(moe_ctx* c) {
  if (c->p_logits) return MOE_OK;
  const AllocSpec specs[] = {
      {reinterpret_cast<void**>(&c->p_logits), (size_t)kMaxPrefillT * c->E * sizeof(float)},
      {reinterpret_cast<void**>(&c->p_idx), (size_t)kMaxPrefillT * c->k * sizeof(int32_t)},
      {reinterpret_cast<void**>(&c->p_w), (size_t)kMaxPrefillT * c->k * sizeof(float)},
      {reinterpret_cast<void**>(&c->p_counts), (size_t)(c->E + 1) * sizeof(int32_t)}};
  return alloc_all(specs, 4);
}

static moe_status ensure_prefill_ffn_scratch(moe_ctx* c) {
  if (c->p_xg) return MOE_OK;
  const int64_t rows = (int64_t)kMaxPrefillT * (c->k + 1);
  c->p_max_tiles = (int64_t)(c->E + 1 + (rows + kPrefillBN - 1) / kPrefillBN);
  const AllocSpec specs[] = {
      {reinterpret_cast<void**>(&c->p_xg), (size_t)rows * c->d * sizeof(uint16_t)},
      {reinterpret_cast<void**>(&c->p_hg), (size_t)rows * c->f * sizeof(uint16_t)},
      {reinterpret_cast<void**>(&c->p_hg_lo), (size_t)rows * c->f * sizeof(uint16_t)},
      {reinterpret_cast<void**>(&c->p_perm), (size_t)rows * sizeof(int32_t)},
      {reinterpret_cast<void**>(&c->p_wsort), (size_t)rows * sizeof(float)},
      {reinterpret_cast<void**>(&c->p_pick), (size_t)kMaxPrefillT * c->k * sizeof(int32_t)},
      {reinterpret_cast<void**>(&c->p_miss_expert), (size_t)c->E * sizeof(int32_t)},
      {reinterpret_cast<void**>(&c->p_miss_slot), (size_t)c->E * sizeof(int32_t)},
      {reinterpret_cast<void**>(&c->p_evicted), (size_t)c->E * sizeof(int32_t)},
      {reinterpret_cast<void**>(&c->p_info), 4 * sizeof(int32_t)},
      {reinterpret_cast<void**>(&c->p_osort), (size_t)kMaxPrefillT * c->k * c->d * sizeof(float)},
      {reinterpret_cast<void**>(&c->p_cursor), (size_t)c->E * sizeof(int32_t)},
      {reinterpret_cast<void**>(&c->p_group_slot), (size_t)(c->E + 1) * sizeof(int32_t)},
      {reinterpret_cast<void**>(&c->p_tiles_gu), (size_t)c->p_max_tiles * (c->f / 64) * sizeof(PrefillTile)},
      {reinterpret_cast<void**>(&c->p_tiles_dn), (size_t)c->p_max_tiles * (c->d / 128) * sizeof(PrefillTile)},
      {reinterpret_cast<void**>(&c->p_ntiles), 2 * sizeof(int32_t)}};
  return alloc_all(specs, sizeof(specs) / sizeof(specs[0]));
}

// Router logits (tcgen05) + top-k for T tokens; idx/w device outputs.
static moe_status prefill_route(moe_ctx* c, int layer, const void* x, int T, int32_t* idx, float* w,
                                int32_t* counts, cudaStream_t s) {
  moe_status st = ensure_prefill_scratch(c);
  if (st != MOE_OK) return st;
  CUtensorMap ta, tb;
  st = make_tmap_2d(&ta, c->router_w + (size_t)layer * c->E * c->d, c->E, c->d, 128, true);
  if (st != MOE_OK) return st;
  st = make_tmap_2d(&tb, x, T, c->d, 256, true);
  if (st != MOE_OK) return st;
  RouterGemmArgs ga{};
  ga.bias = c->router_b + (size_t)layer * c->E;
  ga.logits = c->p_logits;
  ga.T = T;
  ga.E = c->E;
  ga.d = c->d;
  ga.err = c->err;
  CUDA_TRY(launch_router_gemm(ta, tb, ga, s, c->num_sms));
  PrefillTopkArgs ka{};
  ka.logits = c->p_logits;
  ka.idx = idx;
  ka.w = w;
  ka.counts = counts;
  ka.T = T;
  ka.E = c->E;
  ka.k = c->k;
  CUDA_TRY(launch_prefill_topk(ka, s));
  return MOE_OK;
}

extern "C" moe_status moe_route_topk(moe_ctx* c, int32_t layer, const void* x, int32_t T, int32_t* idx,
                                     float* w, void* stream) {
  moe_status st = check_common(c, layer, x, T, kMaxPrefillT);
  if (st != MOE_OK) return st;
  if (!idx || !w) return fail(MOE_ERR_INVALID_ARG, "NULL output");
  if (reinterpret_cast<uintptr_t>(x) % 16) return fail(MOE_ERR_INVALID_ARG, "x must be 16-byte aligned");
  if (T > kMaxDecodeT) return prefill_route(c, layer, x, T, idx, w, nullptr, static_cast<cudaStream_t>(stream));
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
  fa.ypart = c->ypart;
  fa.counters = c->counters;
  fa.set_words = c->set_words;
  fa.wait_ns = c->wait_ns;
  fa.err = c->err;
  fa.grid = c->num_sms;
  // fused routing (every key resident, or misses pulled by the GPU)
  fa.wr = c->router_w + (size_t)layer * c->E * c->d;
  fa.bias = c->router_b + (size_t)layer * c->E;
  fa.tlogits = c->tlogits;
  fa.E = c->E;
  fa.layer = layer;
  fa.table = c->table;
  fa.stamp = c->stamp;
  fa.stats = c->stats + (size_t)layer * ST_N;
  fa.clock = c->clock;
  // fused routing with misses pulled by the GPU (cache not all resident)
  fa.owner = c->owner;
  fa.q_in = c->lruq[c->qcur];
  fa.q_out = c->lruq[c->qcur ^ 1];
  fa.C = (int)c->C;
  fa.host_pool = c->host_pool_dev;
  fa.direct = c->pool_dev_layout ? 1 : 0;
  fa.pool_entries = c->P;
  fa.staging = c->staging;
  fa.staging_n = c->staging_n;
  return fa;
}

static moe_status fill_trace(moe_ctx* c, cudaStream_t s, int T, moe_trace* tr, const Plan* plan = nullptr) {
  CUDA_TRY(cudaMemcpyAsync(c->plan_host, plan ? plan : c->plan, sizeof(Plan), cudaMemcpyDeviceToHost, s));
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

// Prefill layer-call (T > 16): routing on the tensor cores; with a cache
// that can miss, the chunk's cache step (one key per routed expert with
// tokens) and the fetch of its misses into their victim slots; counting sort
// by expert, gather, gate/up and down grouped GEMMs, fixed-order combine.
static moe_status prefill_forward(moe_ctx* c, int layer, const void* x, int T, float* y, cudaStream_t s,
                                  moe_trace* trace) {
  if (!c->all_resident) {
    if (!c->host_pool_dev)
      return fail(MOE_ERR_UNIMPLEMENTED, "prefill on a cache that can miss needs a device-mapped host pool");
    if (c->C < c->E)
      return fail(MOE_ERR_UNIMPLEMENTED, "prefill on a cache that can miss needs capacity >= n_experts (%d < %d)",
                  (int)c->C, c->E);
  }
  if (reinterpret_cast<uintptr_t>(x) % 16 || reinterpret_cast<uintptr_t>(y) % 16)
    return fail(MOE_ERR_INVALID_ARG, "x and y must be 16-byte aligned");
  if (c->f % 128 != 0)
    return fail(MOE_ERR_UNIMPLEMENTED, "prefill (T > %d) needs f %% 128 == 0 (f = %d)", kMaxDecodeT, c->f);
  moe_status st = ensure_prefill_scratch(c);
  if (st == MOE_OK) st = ensure_prefill_ffn_scratch(c);
  if (st != MOE_OK) return st;
  const int rows = T * (c->k + 1);
  CUDA_TRY(cudaMemsetAsync(c->p_counts, 0, (size_t)(c->E + 1) * sizeof(int32_t), s));
  st = prefill_route(c, layer, x, T, c->p_idx, c->p_w, c->p_counts, s);
  if (st != MOE_OK) return st;
  if (!c->all_resident) {
    // the chunk is one layer-call of the cache: decide and commit, then
    // fetch the misses into their victim slots before the GEMMs read them
    PrefillCacheArgs ca{};
    ca.counts = c->p_counts;
    ca.table = c->table;
    ca.owner = c->owner;
    ca.stamp = c->stamp;
    ca.q_in = c->lruq[c->qcur];
    ca.q_out = c->lruq[c->qcur ^ 1];
    ca.q_staged = c->C <= 32768;
    ca.C = (int)c->C;
    ca.E = c->E;
    ca.layer = layer;
    ca.clock = c->clock;
    ca.stats = c->stats + (size_t)layer * ST_N;
    ca.expert_bytes = c->B;
    ca.group_slot = c->p_group_slot;
    ca.miss_expert = c->p_miss_expert;
    ca.miss_slot = c->p_miss_slot;
    ca.evicted_key = c->p_evicted;
    ca.info = c->p_info;
    ca.err = c->err;
    CUDA_TRY(launch_prefill_cache(ca, s));
    c->qcur ^= 1;
    const MissFetch mf{c->p_miss_expert, c->p_miss_slot, c->host_pool_dev, c->P, c->slots, c->B,
                       layer, c->E, c->d, c->f};
    CUDA_TRY(launch_prefill_fetch(mf, c->p_info, c->pool_dev_layout, s, c->num_sms));
  }
  PrefillPlanArgs pa{};
  pa.counts = c->p_counts;
  pa.cursor = c->p_cursor;
  pa.group_slot = c->p_group_slot;
  pa.tiles_gu = c->p_tiles_gu;
  pa.tiles_dn = c->p_tiles_dn;
  pa.n_tiles = c->p_ntiles;
  pa.table = c->table;
  pa.stamp = c->stamp;
  pa.clock = c->clock;
  pa.stats = c->stats + (size_t)layer * ST_N;
  pa.T = T;
  pa.E = c->E;
  pa.k = c->k;
  pa.d = c->d;
  pa.f = c->f;
  pa.layer = layer;
  pa.account = c->all_resident ? 1 : 0;
  pa.err = c->err;
  CUDA_TRY(launch_prefill_plan(pa, s));
  PrefillScatterArgs sa{};
  sa.idx = c->p_idx;
  sa.w = c->p_w;
  sa.cursor = c->p_cursor;
  sa.perm = c->p_perm;
  sa.wsort = c->p_wsort;
  sa.pick = c->p_pick;
  sa.T = T;
  sa.k = c->k;
  sa.shared_weight = c->shared_weight;
  CUDA_TRY(launch_prefill_scatter(sa, s));
  CUDA_TRY(launch_prefill_gather(static_cast<const uint16_t*>(x), c->p_perm, c->p_xg, rows, c->d, s));
  CUtensorMap tx, th, thl;
  // token tiles are loaded in two halves, one by each CTA of a cluster pair
  st = make_tmap_2d(&tx, c->p_xg, rows, c->d, kPrefillBN / 2, false);
  if (st == MOE_OK) st = make_tmap_2d(&th, c->p_hg, rows, c->f, kPrefillBN / 2, false);
  if (st == MOE_OK) st = make_tmap_2d(&thl, c->p_hg_lo, rows, c->f, kPrefillBN / 2, false);
  if (st != MOE_OK) return st;
  PrefillGemmArgs ga{};
  ga.slots = c->slots;
  ga.shared_expert = c->shared + (size_t)layer * c->B;
  ga.expert_bytes = c->B;
  ga.group_slot = c->p_group_slot;
  ga.tiles_gu = c->p_tiles_gu;
  ga.tiles_dn = c->p_tiles_dn;
  ga.n_tiles = c->p_ntiles;
  ga.hg = c->p_hg;
  ga.hg_lo = c->p_hg_lo;
  ga.perm = c->p_perm;
  ga.wsort = c->p_wsort;
  ga.pick = c->p_pick;
  ga.y = y;
  ga.osort = c->p_osort;
  ga.E = c->E;
  ga.d = c->d;
  ga.f = c->f;
  ga.err = c->err;
  CUDA_TRY(launch_prefill_gate_up(tx, ga, s, c->num_sms));
  CUDA_TRY(launch_prefill_down(th, thl, ga, s, c->num_sms));
  PrefillCombineArgs cb{};
  cb.osort = c->p_osort;
  cb.y = y;
  cb.T = T;
  cb.k = c->k;
  cb.d = c->d;
  CUDA_TRY(launch_prefill_combine(cb, s));
  if (trace) {
    const int n = T * c->k;
    std::vector<int32_t> gslot(c->E + 1);
    CUDA_TRY(cudaStreamSynchronize(s));
    if (trace->idx) CUDA_TRY(cudaMemcpy(trace->idx, c->p_idx, n * sizeof(int32_t), cudaMemcpyDeviceToHost));
    if (trace->w) CUDA_TRY(cudaMemcpy(trace->w, c->p_w, n * sizeof(float), cudaMemcpyDeviceToHost));
    CUDA_TRY(cudaMemcpy(gslot.data(), c->p_group_slot, (c->E + 1) * sizeof(int32_t), cudaMemcpyDeviceToHost));
    std::vector<int32_t> idx(n);
    CUDA_TRY(cudaMemcpy(idx.data(), c->p_idx, n * sizeof(int32_t), cudaMemcpyDeviceToHost));
    int distinct = 0;
    for (int e = 0; e < c->E; ++e) distinct += gslot[e] >= 0;
    if (trace->slot)
      for (int i = 0; i < n; ++i) trace->slot[i] = gslot[idx[i]];
    trace->n_miss = 0;
    trace->n_distinct = distinct;
    trace->token_hits = n;
    trace->token_misses = 0;
    if (!c->all_resident) {
      int32_t info[4];
      CUDA_TRY(cudaMemcpy(info, c->p_info, sizeof(info), cudaMemcpyDeviceToHost));
      const int m = info[0];
      if (trace->miss_expert) CUDA_TRY(cudaMemcpy(trace->miss_expert, c->p_miss_expert, m * sizeof(int32_t),
                                                  cudaMemcpyDeviceToHost));
      if (trace->miss_slot)
        CUDA_TRY(cudaMemcpy(trace->miss_slot, c->p_miss_slot, m * sizeof(int32_t), cudaMemcpyDeviceToHost));
      if (trace->evicted_key)
        CUDA_TRY(cudaMemcpy(trace->evicted_key, c->p_evicted, m * sizeof(int32_t), cudaMemcpyDeviceToHost));
      trace->n_miss = m;
      trace->token_hits = info[2];
      trace->token_misses = info[3];
    }
  }
  return MOE_OK;
}

// One kAhead launch: the current call (layer, x) from plan `cur` when
// has_cur, and the routing, cache step and miss copies of the next call
// (next_layer, next_x) into plan `nxt` when has_next.
static moe_status launch_ahead(moe_ctx* c, bool has_cur, int layer, const void* x, float* y, int T, bool has_next,
                               int next_layer, const void* next_x, const Plan* cur, Plan* nxt, cudaStream_t s) {
  const int rl = has_next ? next_layer : layer;   // the routing fields describe the next call
  FfnArgs fa = ffn_args(c, rl, has_next ? next_x : x, T, y);
  fa.shared_expert = c->shared + (size_t)layer * c->B;
  fa.x = static_cast<const uint16_t*>(has_cur ? x : next_x);
  fa.x_route = static_cast<const uint16_t*>(has_next ? next_x : x);
  fa.y = y;
  fa.plan = nxt;
  fa.cur_plan = cur;
  fa.has_cur = has_cur ? 1 : 0;
  fa.has_next = has_next ? 1 : 0;
  fa.fused = 1;
  fa.cached = 1;
  fa.ahead = 1;
  CUDA_TRY(launch_decode_ffn(fa, s, true));
  if (has_next) c->qcur ^= 1;
  else CUDA_TRY(launch_calls_bump(c->counters, s));
  return MOE_OK;
}

extern "C" moe_status moe_forward_ahead(moe_ctx* c, int32_t layer, const void* x, int32_t T, float* y, void* stream,
                                        moe_trace* trace, int32_t next_layer, const void* next_x) {
  moe_status st = check_common(c, layer, x, T, kMaxDecodeT);
  if (st != MOE_OK) return st;
  if (!c->configured) return fail(MOE_ERR_STATE, "moe_cache_configure must come first");
  if (!y) return fail(MOE_ERR_INVALID_ARG, "NULL output");
  if (reinterpret_cast<uintptr_t>(x) % 16 || reinterpret_cast<uintptr_t>(next_x) % 16)
    return fail(MOE_ERR_INVALID_ARG, "x and next_x must be 16-byte aligned");
  if (next_x && (next_layer < 0 || next_layer >= c->L))
    return fail(MOE_ERR_INVALID_ARG, "next layer %d out of range", next_layer);
  if (!c->pull || !c->pool_dev_layout || c->num_sms < 2 || !c->host_pool_dev)
    return fail(MOE_ERR_UNIMPLEMENTED,
                "lookahead needs the GPU miss path and a host pool in the device layout (MOE_POOL_DEVICE)");
  if (c->C < (int64_t)2 * kMaxDecodeT * c->k)
    return fail(MOE_ERR_UNIMPLEMENTED, "lookahead needs capacity >= %d (two layer-calls' experts)",
                2 * kMaxDecodeT * c->k);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!(c->ahead_valid && c->ahead_layer == layer && c->ahead_x == x && c->ahead_T == T)) {
    if (c->ahead_valid)
      return fail(MOE_ERR_STATE, "the prepared layer-call (layer %d) must run before another", c->ahead_layer);
    // no call prepared: route (layer, x), run its cache step and copy its misses
    st = launch_ahead(c, false, layer, nullptr, nullptr, T, true, layer, x, nullptr, c->plans(c->ahead_pi), s);
    if (st != MOE_OK) return st;
  }
  const Plan* cur = c->plans(c->ahead_pi);
  st = launch_ahead(c, true, layer, x, y, T, next_x != nullptr, next_layer, next_x, cur, c->plans(c->ahead_pi ^ 1), s);
  if (st != MOE_OK) {
    c->ahead_valid = false;
    return st;
  }
  c->ahead_valid = next_x != nullptr;
  c->ahead_layer = next_layer;
  c->ahead_x = next_x;
  c->ahead_T = T;
  c->ahead_pi ^= 1;
  if (trace) return fill_trace(c, s, T, trace, cur);
  return MOE_OK;
}

extern "C" moe_status moe_forward(moe_ctx* c, int32_t layer, const void* x, int32_t T, float* y, void* stream,
                                  moe_trace* trace) {
  moe_status st = check_common(c, layer, x, T, kMaxPrefillT);
  if (st != MOE_OK) return st;
  if (!c->configured) return fail(MOE_ERR_STATE, "moe_cache_configure must come first");
  if (!y) return fail(MOE_ERR_INVALID_ARG, "NULL output");
  if (c->ahead_valid) {   // a layer-call prepared by moe_forward_ahead comes first
    if (layer != c->ahead_layer || x != c->ahead_x || T != c->ahead_T)
      return fail(MOE_ERR_STATE, "the prepared layer-call (layer %d) must run before another", c->ahead_layer);
    return moe_forward_ahead(c, layer, x, T, y, stream, trace, 0, nullptr);
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T > kMaxDecodeT) return prefill_forward(c, layer, x, T, y, s, trace);
  if (reinterpret_cast<uintptr_t>(x) % 16) return fail(MOE_ERR_INVALID_ARG, "x must be 16-byte aligned");
  FfnArgs fa = ffn_args(c, layer, x, T, y);
  // test hook: CTA 0 of this call holds back its router arrival (fused routing)
  fa.dbg_hold_router = injected(MOE_INJECT_HOLD_ROUTER) ? 1 : 0;
  if (c->all_resident) {
    fa.fused = 1;
    CUDA_TRY(launch_decode_ffn(fa, s, true));
    if (trace) return fill_trace(c, s, T, trace);
    return MOE_OK;
  }
  if (c->pull && c->num_sms >= 2) {
    // one launch: routing, the cache (CTA 0) and the GPU's own pull of the
    // misses, then the experts; the LRU order alternates between two arrays
    fa.fused = 1;
    fa.cached = 1;
    CUDA_TRY(launch_decode_ffn(fa, s, true));
    c->qcur ^= 1;
    if (trace) return fill_trace(c, s, T, trace);
    return MOE_OK;
  }
  // miss-capable path
  RouteArgs ra = route_args(c, layer, x, T, ROUTE_PLAN);
  CUDA_TRY(launch_route(ra, s));
  if (c->pull) {
    // every step on the caller's stream, the miss list read on the device
    MissPullArgs mp{};
    mp.plan = c->plan;
    mp.host_pool = c->host_pool_dev;
    mp.pool_entries = c->P;
    mp.expert_bytes = c->B;
    mp.staging = c->staging;
    mp.staging_n = c->staging_n;
    mp.layer = layer;
    mp.E = c->E;
    mp.err = c->err;
    mp.dst_slots = c->pool_dev_layout ? c->slots : nullptr;
    CUDA_TRY(launch_miss_pull(mp, s, c->num_sms));
    RepackArgs rp{};
    rp.src = c->staging;
    rp.src_stride = c->B;
    rp.dst_base = c->slots;
    rp.dst_stride = c->B;
    rp.d = c->d;
    rp.f = c->f;
    rp.plan = c->plan;
    if (!c->pool_dev_layout) CUDA_TRY(launch_repack_misses(rp, s, c->num_sms));
    CommitArgs ca{};
    ca.plan = c->plan;
    ca.counters = c->counters;
    ca.set_words = c->set_words;
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
    CUDA_TRY(launch_decode_ffn(fa, s, false));
    if (trace) return fill_trace(c, s, T, trace);
    return MOE_OK;
  }
  CUDA_TRY(cudaMemcpyAsync(c->plan_host, c->plan, sizeof(Plan), cudaMemcpyDeviceToHost, s));
  CUDA_TRY(cudaEventRecord(c->ev_route, s));
  CUDA_TRY(cudaEventSynchronize(c->ev_route));
  const Plan& p = *c->plan_host;
  const int m = p.n_miss;
  if (m < 0 || m > c->staging_n) return fail(MOE_ERR_CUDA, "corrupt routing plan (n_miss=%d)", m);
  for (int j = 0; j < m; ++j) {
    const int64_t key = (int64_t)layer * c->E + p.miss_expert[j];
    const int64_t entry = key % c->P;
    if (injected(MOE_INJECT_MISS_COPY))
      return fail(MOE_ERR_CUDA, "injected failure: issue of miss copy %d of the layer-call", j);
    uint8_t* dst = c->pool_dev_layout ? c->slots + (size_t)p.miss_slot[j] * c->B : c->staging + (size_t)j * c->B;
    CUDA_TRY(cudaMemcpyAsync(dst, c->host_pool + (size_t)entry * c->B, c->B, cudaMemcpyHostToDevice, c->side));
  }
  if (m > 0 && !c->pool_dev_layout) {
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
  ca.counters = c->counters;
  ca.set_words = c->set_words;
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
  CUDA_TRY(launch_decode_ffn(fa, s, false));
  if (trace) {
    moe_status t = fill_trace(c, s, T, trace);
    if (t != MOE_OK) return t;
    // plan_host was refreshed after the call; the miss list is that of this call
  }
  return MOE_OK;
}

extern "C" moe_status moe_set_miss_mode(moe_ctx* c, int32_t mode) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "NULL context");
  if (c->ahead_valid) return fail(MOE_ERR_STATE, "a layer-call prepared by moe_forward_ahead is pending");
  if (mode == MOE_MISS_HOST_COPY) {
    c->pull = false;
    return MOE_OK;
  }
  if (mode == MOE_MISS_DEVICE_PULL) {
    if (!c->host_pool_dev) return fail(MOE_ERR_UNIMPLEMENTED, "the host pool has no device address");
    c->pull = true;
    return MOE_OK;
  }
  return fail(MOE_ERR_INVALID_ARG, "unknown miss mode %d", mode);
}

static moe_status check_device_error(moe_ctx* c) {
  uint32_t e = 0;
  CUDA_TRY(cudaMemcpy(&e, c->err, sizeof(e), cudaMemcpyDeviceToHost));
  if (e != 0) {
    CUDA_TRY(cudaMemset(c->err, 0, sizeof(uint32_t)));
    CUDA_TRY(cudaMemset(c->counters, 0, c->counters_n * sizeof(uint32_t)));
    // the call count restarts: no word a call of the failed run wrote may
    // carry a tag a later call uses
    CUDA_TRY(cudaMemset(c->ypart, 0xff, (size_t)c->num_sms * kMaxDecodeT * c->d * sizeof(uint64_t)));
    CUDA_TRY(cudaMemset(c->tlogits, 0xff, (size_t)kMaxDecodeT * c->E * sizeof(uint64_t)));
    CUDA_TRY(cudaMemset(c->route_cnt, 0, sizeof(uint32_t)));
    CUDA_TRY(cudaDeviceSynchronize());
    // with a cache that can miss, a call that gave up may have committed
    // slots whose contents never arrived: the cache must be configured again
    if (!c->all_resident) c->configured = false;
    return fail(e == DEV_NOT_RESIDENT ? MOE_ERR_STATE : MOE_ERR_TIMEOUT,
                "device error %u (1: barrier wait, 2: flag wait, 3: key not resident, 4: bad plan)", e);
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

// The GPU address of a buffer the GPU can reach (device memory, or
// page-locked host memory through its mapping); NULL otherwise.
static const void* gpu_address(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return p;
  if (at.type == cudaMemoryTypeHost) return at.devicePointer;
  return nullptr;
}

extern "C" moe_status moe_pack_experts(const void* src, void* dst, int64_t n, int32_t d, int32_t f, void* stream) {
  if (!src || !dst) return fail(MOE_ERR_INVALID_ARG, "NULL src or dst");
  if (n < 0) return fail(MOE_ERR_INVALID_ARG, "n < 0");
  if (d <= 0 || d % 256 != 0 || d > 2048)
    return fail(MOE_ERR_INVALID_ARG, "d must be a positive multiple of 256, at most 2048");
  if (f <= 0 || f % 64 != 0 || f > 1024) return fail(MOE_ERR_INVALID_ARG, "f must be a multiple of 64 in [64, 1024]");
  if (n == 0) return MOE_OK;
  const int64_t B = (int64_t)3 * d * f * 3 / 8 + (int64_t)3 * d * f / 32 * 2;
  const uint8_t* s8 = static_cast<const uint8_t*>(src);
  const uint8_t* d8 = static_cast<const uint8_t*>(dst);
  if (s8 < d8 + n * B && d8 < s8 + n * B) return fail(MOE_ERR_INVALID_ARG, "src and dst overlap");
  const void* sg = gpu_address(src);
  const void* dg = gpu_address(dst);
  if (!sg || !dg) return fail(MOE_ERR_INVALID_ARG, "src and dst must be device memory or page-locked host memory");
  const int64_t chunk = 1 << 16;   // experts per launch (the grid stays far below its limit)
  for (int64_t i0 = 0; i0 < n; i0 += chunk) {
    RepackArgs ra{};
    ra.src = static_cast<const uint8_t*>(sg) + i0 * B;
    ra.src_stride = B;
    ra.dst_base = const_cast<uint8_t*>(static_cast<const uint8_t*>(dg)) + i0 * B;
    ra.dst_stride = B;
    ra.n_experts = (int)(n - i0 < chunk ? n - i0 : chunk);
    ra.d = d;
    ra.f = f;
    CUDA_TRY(launch_repack(ra, static_cast<cudaStream_t>(stream)));
  }
  return MOE_OK;
}
