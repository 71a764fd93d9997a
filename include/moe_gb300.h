/*
 * moe_gb300.h -- C ABI of the routed-expert FFN step on one GB300 (sm_103a).
 *
 * The step (one MoE layer of an offloaded-MoE serving engine, as described in
 * the blog posts "一张 RTX 4090 跑千亿模型，Strata 实测 155 tok/s",
 * §如何做到：三层存储, and "单卡5090跑125B 大模型：Strata 把服务器级 MoE 拉进普通 PC",
 * §2.1-§2.3):
 *   1. router: logits l = x.Wr^T + b, softmax over all E experts, the k largest
 *      logits chosen (ties to the lower id), weights renormalised over the k;
 *   2. expert cache: each distinct (layer, expert) of the call is looked up in
 *      a fixed-capacity VRAM slot pool; misses are copied from pinned host
 *      memory (LRU by (layer, expert), ties to the lower slot id);
 *   3. SwiGLU experts over 3-bit group-quantised weights,
 *      E(x) = Wd.(silu(Wg.x) * (Wu.x)), for every distinct expert once for all
 *      tokens routed to it (a verify batch shares one fetch, §2.3);
 *   4. combine y[t] = sum_i w[t,i] E_idx[t,i](x_t) + shared_weight * E_shared(x_t).
 * The pages give the structure (512 routed experts, top-10, one shared
 * expert, 48 layers, hits/lookups per token pick); the formulas and the
 * weight format are the workload definition's.
 *
 * Conventions for every entry point:
 *   - Every call returns a moe_status; nothing crosses the ABI as an
 *     exception.  moe_last_error() gives a thread-local message for the last
 *     failing call on the calling thread.
 *   - "device" pointers are CUDA device (or managed) memory of the current
 *     device; "host" pointers are CPU memory.
 *   - Streams are cudaStream_t passed as void* (NULL = legacy default stream).
 *   - Calls on one context must be serialised by the caller.
 *   - The library never frees caller memory.
 *
 * Canonical packed expert (host pool, shared experts), bytes in this order:
 *   Wg codes [f][d/32][12 B], Wu codes [f][d/32][12 B], Wd codes [d][f/32][12 B],
 *   Wg scales [f][d/32] fp16, Wu scales [f][d/32] fp16, Wd scales [d][f/32] fp16.
 *   In a 12-byte group, weight i (0..31 along the input dimension) is the 3-bit
 *   field u at bits [3i, 3i+3) of the 96-bit little-endian integer; the weight
 *   is (u - 4) * scale.  Size B_x = 3*d*f*3/8 + 3*d*f/32*2 bytes
 *   (2,064,384 B at d=2048, f=768).  The library keeps its own device layout
 *   in the slot pool; a miss copies B_x bytes and re-lays them out on the GPU.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_ctx moe_ctx; /* opaque, library-owned */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,   /* bad pointer, size, shape or layer index */
  MOE_ERR_OOM = -2,           /* device or host allocation failed */
  MOE_ERR_CUDA = -3,          /* a CUDA call failed (message has the CUDA error) */
  MOE_ERR_HOST_PIN = -4,      /* the host pool could not be pinned/registered */
  MOE_ERR_TIMEOUT = -5,       /* a bounded device-side wait gave up; context reset */
  MOE_ERR_STATE = -6,         /* call out of order (e.g. forward before configure) */
  MOE_ERR_UNIMPLEMENTED = -7  /* shape or mode this build does not support */
} moe_status;

/* Shapes and weights of one MoE stack (n_layers layers of one shape).
 * Supported shapes: group == 32, d % 256 == 0, d <= 2048, f % 64 == 0,
 * f <= 1024, 2 <= top_k <= 16, top_k < n_experts <= 1024. */
typedef struct {
  int32_t d;               /* hidden size */
  int32_t f;               /* expert intermediate size */
  int32_t n_experts;       /* routed experts per layer (E) */
  int32_t top_k;           /* routed experts per token (k) */
  int32_t n_layers;        /* L */
  int32_t group;           /* quantisation group, must be 32 */
  const void* router_w;    /* [L][E][d] bf16, host or device; copied at create */
  const float* router_b;   /* [L][E] fp32, host or device, or NULL (zero bias) */
  const void* shared_q;    /* [L] canonical packed shared experts, host or device; copied */
  const void* host_pool;   /* [P] canonical packed experts, HOST memory owned by the
                              caller; must stay valid until moe_layer_destroy.  If it
                              is not page-locked the library registers it
                              (cudaHostRegister) and unregisters it at destroy. */
  int64_t host_pool_entries; /* P; identity (l, e) reads entry (l*E + e) mod P;
                                0 means P = L*E (one entry per identity) */
  float shared_weight;     /* weight of the shared expert in the combine (1.0) */
  int32_t host_pool_layout; /* MOE_POOL_CANONICAL (0): host_pool entries in the
                              canonical packed format; MOE_POOL_DEVICE (1): in the
                              device block layout (moe_pack_experts), so a miss is
                              a plain copy and the decode kernel computes a missing
                              expert straight from the host pool while it writes
                              the expert into its victim slot */
} moe_layer_desc;

enum { MOE_POOL_CANONICAL = 0, MOE_POOL_DEVICE = 1 };

/* Cumulative counters since the last moe_cache_configure.  A token pick is a
 * hit iff its (layer, expert) was resident when the layer-call began ("hits /
 * lookups" per pick, page "单卡5090跑125B 大模型", §7.2); shared experts are not
 * counted, so token_hits + token_misses = k * tokens per layer-call. */
typedef struct {
  int64_t layer_calls;
  int64_t token_hits;
  int64_t token_misses;
  int64_t distinct_hits;   /* distinct (layer, expert) per layer-call */
  int64_t distinct_misses;
  int64_t evictions;       /* misses whose victim slot held a key */
  int64_t miss_bytes;      /* bytes copied host -> device for misses */
} moe_stats;

/* Optional per-call record (host buffers owned by the caller, capacity T*k
 * entries each unless noted).  Passing a trace makes moe_forward synchronise
 * with the stream before returning. */
typedef struct {
  int32_t* idx;            /* [T][k] routed expert ids, ascending per token */
  float* w;                /* [T][k] renormalised routing weights */
  int32_t* slot;           /* [T][k] cache slot used by each pick */
  int32_t* miss_expert;    /* [<=T*k] missed expert ids, ascending */
  int32_t* miss_slot;      /* [<=T*k] victim slot of each miss */
  int32_t* evicted_key;    /* [<=T*k] key (l*E+e) the victim held, -1 if empty */
  int32_t n_miss;          /* out: number of misses */
  int32_t n_distinct;      /* out: distinct routed experts of the call */
  int64_t token_hits;      /* out */
  int64_t token_misses;    /* out */
} moe_trace;

/* Create a context: copies router weights, bias and shared experts to the
 * device (re-laid out), pins or registers the host pool.  *out receives the
 * context.  On any error nothing stays allocated or registered and *out is
 * NULL.  Errors: INVALID_ARG (shapes, NULL pointers), OOM, HOST_PIN, CUDA,
 * UNIMPLEMENTED (also when one decode CTA per SM does not fit: the decode
 * kernel's grid-wide counters need all of its CTAs resident at once). */
moe_status moe_layer_create(const moe_layer_desc* desc, moe_ctx** out);

/* Size the expert cache to capacity_slots (each B_x bytes of device memory)
 * and preload the keys preload_keys[0..n_preload) (key = l*E + e, strictly
 * ascending) into slots 0, 1, ... from the host pool.  Resets the LRU state,
 * the logical clock and the counters.  When every key of the stack is
 * preloaded no miss can occur and moe_forward never waits on the host.
 * Synchronous.  Every buffer of the new cache is allocated before the old
 * one is released, so on MOE_ERR_OOM the previous cache (slots, LRU state,
 * counters) is unchanged and usable.  Errors: INVALID_ARG (capacity < k*16
 * distinct picks of one call, n_preload > capacity, unsorted keys), OOM,
 * CUDA. */
moe_status moe_cache_configure(moe_ctx* ctx, int64_t capacity_slots,
                               const int32_t* preload_keys, int64_t n_preload);

/* Router only: idx[T][k] (ascending expert id) and w[T][k] for tokens
 * x[T][d] (bf16, device, 16-byte aligned) at layer `layer`.  idx and w are
 * device buffers.  Asynchronous on `stream`; does not touch the cache.
 * 1 <= T <= 16,384 (T > 16 computes the logits on the tensor cores). */
moe_status moe_route_topk(moe_ctx* ctx, int32_t layer, const void* x_bf16, int32_t T,
                          int32_t* idx, float* w, void* stream);

/* One layer-call: route, look up / fill the cache, run the experts and write
 * y[T][d] (fp32, device).  x[T][d] bf16 (device); x and y 16-byte aligned.  1 <= T <= 16 uses the
 * decode path; larger T (up to 16,384) the prefill path, which needs
 * f % 128 == 0 and, on a cache that can miss, a device-mapped host pool and
 * capacity >= n_experts (MOE_ERR_UNIMPLEMENTED otherwise): the chunk is one
 * layer-call of the cache (its distinct experts are the keys) and its misses
 * are read by the GPU into their victim slots before the grouped GEMMs.  The
 * result does not depend on the order in which the GPU ran its work: every
 * output is summed in a fixed order (shared expert, then the token's picks
 * in ascending expert id).  Asynchronous on
 * `stream` when every key is resident (see moe_cache_configure) and, with the
 * default MOE_MISS_DEVICE_PULL, also when misses can occur (one kernel launch
 * routes, plans and commits the cache, pulls the misses and runs the
 * experts); with MOE_MISS_HOST_COPY the host waits for the routing kernel,
 * issues the miss copies on a side stream and joins it with an event before
 * the experts run.  On error the cache state is unchanged.  `trace` may be
 * NULL (with a trace the call synchronises to read the plan back). */
moe_status moe_forward(moe_ctx* ctx, int32_t layer, const void* x_bf16, int32_t T,
                       float* y, void* stream, moe_trace* trace);

/* How a layer-call with misses fetches the missing experts (the cache of
 * page "单卡5090跑125B 大模型", §2.1 and §7.2: misses come from pinned host RAM).
 *   MOE_MISS_DEVICE_PULL (default when the host pool is device-accessible):
 *     the GPU reads the registered host pool itself (NVLink-C2C or PCIe)
 *     inside the decode kernel, which takes the miss list from its own plan,
 *     and moe_forward does not wait for the GPU (nothing between routing and
 *     the copies goes through the host);
 *   MOE_MISS_HOST_COPY: the host waits for the routing plan and issues one
 *     cudaMemcpyAsync per miss on a side stream.
 * Both give the same slots, counters and outputs.  Returns
 * MOE_ERR_UNIMPLEMENTED for device pull when the pool has no device address,
 * MOE_ERR_INVALID_ARG for an unknown mode. */
typedef enum { MOE_MISS_HOST_COPY = 0, MOE_MISS_DEVICE_PULL = 1 } moe_miss_mode;
moe_status moe_set_miss_mode(moe_ctx* ctx, int32_t mode);

/* moe_forward for decode calls (T <= 16) with cross-layer lookahead, for a
 * stream of layer-calls whose inputs are known ahead (as the layers of the
 * stack workload, which take independent tokens): besides the layer-call
 * (layer, x), the launch routes the layer-call (next_layer, next_x, same T),
 * runs its cache step and copies its misses into their victim slots, all
 * while the experts of (layer, x) compute.  That next call's experts then
 * run in the following moe_forward_ahead or moe_forward on this context,
 * which must name the same layer, the same x pointer (contents unchanged)
 * and T; until it does, every other call that touches the cache returns
 * MOE_ERR_STATE.  next_x == NULL: no next call.  The first call of a
 * sequence also prepares itself (one more launch).  Cache steps run in call
 * order, so hits, misses, victims, counters and the LRU state are exactly
 * those of the same calls made with moe_forward; the trace describes (layer,
 * x).  Needs the GPU miss path (MOE_MISS_DEVICE_PULL), a host pool in the
 * device layout (MOE_POOL_DEVICE) and a capacity of at least 32 * top_k
 * slots (two layer-calls' experts, so that no victim of the next call is an
 * expert this call still reads); else MOE_ERR_UNIMPLEMENTED.  Cross-layer
 * prefetch of the scope table's NEXT-1 (no counterpart on the pages, whose
 * layer inputs depend on the previous layer). */
moe_status moe_forward_ahead(moe_ctx* ctx, int32_t layer, const void* x_bf16, int32_t T, float* y,
                             void* stream, moe_trace* trace, int32_t next_layer, const void* next_x_bf16);

/* Test hook: make the nth (>= 1) future event of `kind` fail once, then
 * disarm; kind 0 disarms.  Process-wide, not thread-safe.  Errors:
 * INVALID_ARG for an unknown kind or nth < 1.
 *   MOE_INJECT_MISS_COPY: the issue of a miss copy in the host-copy miss mode
 *     fails, so moe_forward returns MOE_ERR_CUDA before any cache state
 *     changes;
 *   MOE_INJECT_HOLD_ROUTER: in a decode layer-call with routing inside the
 *     kernel, CTA 0 never publishes its rows of the router logits, so every
 *     CTA's bounded wait for them runs out (after the limit of
 *     moe_debug_set_wait_limit); the call returns MOE_OK (it is asynchronous)
 *     and the next moe_sync reports MOE_ERR_TIMEOUT;
 *   MOE_INJECT_HOST_REGISTER: moe_layer_create's registration of a pageable
 *     host pool fails (MOE_ERR_HOST_PIN, nothing left allocated or
 *     registered);
 *   MOE_INJECT_DEVICE_ALLOC: a device allocation of moe_layer_create or
 *     moe_cache_configure fails (MOE_ERR_OOM; create leaves nothing
 *     allocated, configure leaves the previous cache unchanged). */
enum {
  MOE_INJECT_MISS_COPY = 1,
  MOE_INJECT_HOLD_ROUTER = 2,
  MOE_INJECT_HOST_REGISTER = 3,
  MOE_INJECT_DEVICE_ALLOC = 4
};
moe_status moe_debug_inject_failure(int32_t kind, int64_t nth);

/* Test hook: the limit, in nanoseconds of the GPU's global timer, of every
 * bounded device-side wait of this context's decode kernel (default 2 s).
 * A wait that runs out sets the context's error word and the kernel returns;
 * moe_sync then reports MOE_ERR_TIMEOUT.  Errors: INVALID_ARG for ns <= 0. */
moe_status moe_debug_set_wait_limit(moe_ctx* ctx, int64_t ns);

/* Wait for all work of the context and report a deferred device error
 * (MOE_ERR_TIMEOUT if a bounded device wait gave up).  After a device error
 * on a cache that can miss, the cache must be configured again
 * (moe_forward returns MOE_ERR_STATE until then): a call that gave up may
 * have committed slots whose contents never arrived. */
moe_status moe_sync(moe_ctx* ctx);

/* Counters (synchronises).  per_layer may be NULL or point to n_layers
 * entries that receive the per-layer split. */
moe_status moe_cache_stats(moe_ctx* ctx, moe_stats* total, moe_stats* per_layer);

/* Copy the LRU state to host buffers: owner[C] (key or -1) and stamp[C]
 * (logical clock of the last use, -1 never used).  Synchronises. */
moe_status moe_cache_export(moe_ctx* ctx, int32_t* owner, int64_t* stamp);

/* Free every library-owned resource.  NULL is accepted. */
void moe_layer_destroy(moe_ctx* ctx);

/* Router only, allocating nothing: the same result as moe_route_topk
 * (idx[T][k] ascending expert ids, w[T][k] renormalised weights, device
 * buffers) for tokens x[T][d] (bf16, device) and one layer's router weights
 * router_w[E][d] (bf16, device) and bias router_b[E] (fp32, device, or NULL
 * for zero), without a context.  No counterpart on the pages: it exists for
 * callers that cannot call cudaMalloc, e.g. code whose device memory is all
 * reserved up front by its own allocator, or code on a latency-critical path
 * that must not risk the device-wide synchronisation an allocation can cause.
 * Its scratch is a fixed array inside the library (logits of at most 16
 * tokens x 1024 experts plus a counter, about 72 KiB, held by every GPU that
 * loads the library until the process exits).  Limits: 1 <= T <= 16,
 * 2 <= k <= 16, k < E <= 1024, d a positive multiple of 256, x and router_w
 * 16-byte aligned; larger sizes are rejected with MOE_ERR_INVALID_ARG and a
 * message.  The first call on a device looks up the scratch's device address
 * (cudaGetSymbolAddress) and caches it; make that first call before any
 * stream capture.  Every call shares the one scratch array: calls that
 * overlap on the GPU (e.g. on two streams) race and must be serialised by the
 * caller.  Asynchronous on `stream`. */
moe_status moe_route_topk_noalloc(const void* x_bf16, const void* router_w_bf16, const float* router_b,
                                  int32_t T, int32_t d, int32_t n_experts, int32_t top_k,
                                  int32_t* idx, float* w, void* stream);

/* Message of the last failing call on this thread ("" if none). */
const char* moe_last_error(void);

/* Re-lay n experts of shape (d, f) from the canonical packed format (src) into
 * the device block layout (dst), each expert B_x bytes, on `stream` (a
 * cudaStream_t, NULL for the default stream); asynchronous.  src and dst must
 * not overlap and must be addressable by the GPU: device memory or
 * page-locked host memory.  The same bytes, permuted: the layout the slots
 * hold (32-row x 32-input blocks of codes and scales in mma fragment order).
 * No counterpart on the pages, which keep experts in their file format; it
 * prepares a host pool once, before moe_layer_create with MOE_POOL_DEVICE.
 * Errors: INVALID_ARG (shapes as for moe_layer_create, n < 0, NULL), CUDA. */
moe_status moe_pack_experts(const void* src, void* dst, int64_t n, int32_t d, int32_t f, void* stream);

/* ---- KV-streaming window (the attention side of the same engine) ---------
 * Page "单卡5090跑125B 大模型", §2.1-§2.2 and §7.2: per QSA layer the engine
 * keeps the first 32,768 of 131,072 KV cells (int8, 1,056 bytes per cell)
 * in VRAM and streams the rest from page-locked host memory block by block,
 * counting the share of block reads served from VRAM.  The window moves
 * bytes only (a cell is opaque); which blocks a step reads is the caller's
 * choice (the pages do not give the attention's block choice).
 *
 * A layer's cells 0 .. n_cells-1: cell c < resident_cells lives in the
 * library's VRAM window, cell c >= resident_cells in the caller's host
 * buffer at [layer][c - resident_cells].  Block b is cells
 * [b*block_cells, (b+1)*block_cells); it hits VRAM when b*block_cells <
 * resident_cells (resident_cells is a multiple of block_cells, so a block
 * is wholly on one side). */
typedef struct moe_kv moe_kv;   /* opaque, library-owned */

typedef struct {
  int32_t n_layers;        /* layers with a KV window (> 0) */
  int32_t cell_bytes;      /* bytes per cell, a positive multiple of 16 */
  int64_t n_cells;         /* cells per layer, a positive multiple of block_cells */
  int64_t resident_cells;  /* the first cells of each layer held in VRAM: a multiple
                              of block_cells in [0, n_cells] */
  int32_t block_cells;     /* cells per block read (> 0) */
  void* host_cells;        /* [n_layers][n_cells - resident_cells][cell_bytes] HOST
                              memory owned by the caller, 16-byte aligned, valid
                              until moe_kv_destroy; registered (cudaHostRegister)
                              by the library when it is not page-locked.  May be
                              NULL when resident_cells == n_cells. */
} moe_kv_desc;

/* Allocates the VRAM window (n_layers * resident_cells * cell_bytes) and the
 * read counters; synchronous.  Errors: INVALID_ARG (sizes as above, host
 * memory given as device memory), OOM, HOST_PIN (registration or mapping of
 * host_cells failed), CUDA.  Nothing is left allocated on error. */
moe_status moe_kv_create(const moe_kv_desc* desc, moe_kv** out);

/* Writes cells [first_cell, first_cell + n) of `layer` from `src` (n *
 * cell_bytes bytes, device or host memory): the resident part into the
 * window, the rest into the host buffer; asynchronous on `stream`.
 * Errors: INVALID_ARG (layer or cell range), CUDA. */
moe_status moe_kv_write(moe_kv* kv, int32_t layer, int64_t first_cell, int64_t n, const void* src,
                        void* stream);

/* Block reads of one layer: dst[i] (block_cells * cell_bytes bytes, device
 * memory, 16-byte aligned) <- block block_ids[i] (device int32 array of
 * n_blocks ids, repeats allowed).  Resident blocks are read from VRAM, the
 * others from the host buffer through its device mapping; one kernel launch,
 * asynchronous on `stream`.  Adds n_blocks to the read counter and the
 * resident ones to the hit counter.  An id outside [0, n_cells/block_cells)
 * reads nothing (its dst block is left as it was) and is reported by the next
 * moe_kv_stats.  Errors: INVALID_ARG (layer, n_blocks < 0, NULL or
 * misaligned pointers), CUDA. */
moe_status moe_kv_read_blocks(moe_kv* kv, int32_t layer, const int32_t* block_ids, int32_t n_blocks, void* dst,
                              void* stream);

/* Totals since create: block reads and the reads served from VRAM (either
 * pointer may be NULL).  Synchronises the device.  Returns INVALID_ARG (once)
 * if a read named a block outside the layer. */
moe_status moe_kv_stats(moe_kv* kv, int64_t* block_reads, int64_t* block_hits);

/* Frees the window and unregisters host_cells if the library registered it;
 * synchronises the device.  NULL is a no-op. */
void moe_kv_destroy(moe_kv* kv);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
