// Library-internal declarations: the routing plan, kernel argument blocks and
// host-side launchers (one per .cu file).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_gb300.h"

namespace moe {

constexpr int kMaxDecodeT = 16;   // tokens per call on the decode path
constexpr int kMaxTopK = 16;
constexpr int kMaxE = 1024;
constexpr int kMaxPicks = kMaxDecodeT * kMaxTopK;   // 256
constexpr int kMaxSlots = 1 << 17;                  // LRU scan bitmap bound
constexpr int kMaxDevices = 64;                     // per-device launch state

// Routing plan of one layer-call, written by the route kernel.
struct Plan {
  int32_t n_act;                    // distinct routed experts
  int32_t n_miss;
  int32_t T;
  int32_t pad0;
  int64_t clock;                    // logical clock of the layer-call
  int64_t token_hits;
  int64_t token_misses;
  int32_t act_expert[kMaxPicks];    // ascending expert ids
  int32_t act_slot[kMaxPicks];      // slot after the call (victim for misses)
  int32_t act_hit[kMaxPicks];
  int32_t pick_act[kMaxPicks];      // [T][k] index into act_* of each pick
  int32_t idx[kMaxPicks];           // [T][k] ascending per token
  float w[kMaxPicks];               // [T][k]
  int32_t miss_expert[kMaxPicks];   // ascending
  int32_t miss_slot[kMaxPicks];
  int32_t evicted_key[kMaxPicks];
};

enum RouteMode : int { ROUTE_ONLY = 0, ROUTE_PLAN = 1 };

// per-layer statistics block (int64 each)
enum StatIdx : int {
  ST_CALLS = 0, ST_TOK_HIT, ST_TOK_MISS, ST_DIST_HIT, ST_DIST_MISS, ST_EVICT, ST_MISS_BYTES, ST_N
};

struct RouteArgs {
  const uint16_t* x;        // [T][d] bf16
  const uint16_t* wr;       // [E][d] bf16 (this layer)
  const float* bias;        // [E] (this layer)
  int T, d, E, k, layer, mode;
  float* logits;            // scratch [T][E]
  uint32_t* cnt;            // CTA arrival counter, 0 between launches
  Plan* plan;
  int32_t* out_idx;         // ROUTE_ONLY outputs (device) or NULL
  float* out_w;
  int32_t* table;           // [L*E]
  const int32_t* owner;     // [C]
  int64_t* stamp;           // [C]
  const int32_t* q_in;      // [C] LRU order (least recent first)
  int32_t* q_out;
  int C;
  int64_t* clock;           // device logical clock
  int64_t* stats;           // [ST_N] of this layer
  int64_t expert_bytes;
  uint32_t* err;
};

struct CommitArgs {
  const Plan* plan;
  uint32_t* counters;       // decode counters (see FfnArgs)
  int set_words;
  int32_t* table;
  int32_t* owner;
  int64_t* stamp;
  int64_t* clock;
  int64_t* stats;           // [ST_N] of this layer
  int layer, E;
  int64_t expert_bytes;
};

struct RepackArgs {
  const uint8_t* src;       // canonical experts, src_stride bytes apart
  int64_t src_stride;
  uint8_t* dst_base;        // device-layout slots
  const int32_t* dst_slot;  // slot index of expert i (NULL: expert i -> dst_base + i*stride)
  int64_t dst_stride;
  int n_experts;
  int d, f;
  const Plan* plan;         // if set: n_experts = plan->n_miss, dst_slot = plan->miss_slot
};

// Miss copies pulled by the GPU from the device-mapped host pool.
struct MissPullArgs {
  const Plan* plan;          // miss list of the layer-call
  const uint8_t* host_pool;  // device address of the registered host pool
  int64_t pool_entries;      // identity (layer, e) reads entry (layer*E + e) mod pool_entries
  int64_t expert_bytes;
  uint8_t* staging;          // [staging_n][expert_bytes]
  int staging_n;
  uint8_t* dst_slots;        // if set (device-layout pool): copy into the misses' victim slots instead
  int layer, E;
  uint32_t* err;
};

struct FfnArgs {
  const uint8_t* slots;         // slot pool base
  const uint8_t* shared_expert; // this layer's shared expert (device layout)
  int64_t expert_bytes;
  const uint16_t* x;            // [T][d] bf16
  float* y;                     // [T][d]
  int T, d, f, k;
  float shared_weight;
  Plan* plan;                   // read (after the routing kernel) or written (fused routing)
  uint64_t* ypart;              // [grid][T][d] per-CTA partials of y, (call tag, value) words
  // per-call counters: word 0 counts decode calls; then two sets of
  // set_words words (router counter | partials counter | cache mode: victims
  // published | finished fetch jobs of each miss), used by alternate calls.  A call uses set (calls before it) & 1, and the set of the call
  // before it is zeroed during the call (by the fused kernel's CTA 0, or by
  // the commit kernel on the host-copy miss path).
  uint32_t* counters;
  int set_words;
  uint32_t* err;
  int grid;
  uint64_t wait_ns;             // limit of every bounded device wait
  int dbg_hold_router;          // test hook: CTA 0 never arrives on the router counter
  // fused routing (kFusedResident, kFusedCached): router, slot table, LRU stamps, counters
  int fused;
  const uint16_t* wr;           // [E][d] bf16 (this layer)
  const float* bias;            // [E] (this layer)
  uint64_t* tlogits;            // [T][E] router logits, (call tag, value) words
  int E, layer;
  const int32_t* table;         // [L*E]
  int64_t* stamp;               // [C]
  int64_t* stats;               // this layer's counters
  int64_t* clock;
  // fused routing with a cache that may miss (misses pulled by the GPU)
  int cached;
  int32_t* owner;               // [C] key held by each slot, -1 if none
  const int32_t* q_in;          // [C] slots, least recently used first
  int32_t* q_out;               // [C] the order after this call
  int C;
  const uint8_t* host_pool;     // device address of the registered host pool
  int direct;                   // the host pool holds the device block layout (kFusedCachedDirect)
  // kAhead: the routing fields above (layer, wr, bias, table row, plan,
  // stats) describe the next call; these the current one
  int ahead;
  int has_cur, has_next;        // a current call to compute / a next call to route
  const Plan* cur_plan;         // the current call's plan (written by the previous launch)
  const uint16_t* x_route;      // [T][d] bf16 tokens of the next call
  int64_t pool_entries;         // key (layer, e) reads entry (layer*E + e) mod pool_entries
  uint8_t* staging;             // [staging_n][expert_bytes] canonical copies of this call's misses
  int staging_n;
};

// words of one per-call counter set of the decode kernel: two unused words,
// victims published, finished fetch jobs of each miss
constexpr int kDecodeSetWords = 3 + kMaxPicks;

// decode kernel modes
// kFusedCachedDirect: as kFusedCached with the host pool in the device block
// layout: a missing expert's stages come straight from the host pool into
// the units (and into its victim slot), with no fetch ahead of them.
// kAhead: the current call's experts come from a plan prepared by the
// previous launch (all resident), while this launch routes the next call
// (router rows, selection, cache step in CTA 0) and copies its misses from a
// device-layout host pool into their victim slots.
enum FfnMode : int { kPlanRead = 0, kFusedResident = 1, kFusedCached = 2, kFusedCachedDirect = 3, kAhead = 4 };

struct RouterGemmArgs {
  const float* bias;   // [E]
  float* logits;       // [T][E]
  int T, E, d;
  uint32_t* err;
};

struct PrefillTopkArgs {
  const float* logits; // [T][E]
  int32_t* idx;        // [T][k]
  float* w;            // [T][k]
  int32_t* counts;     // [E] picks per expert (atomic), or NULL
  int T, E, k;
};

constexpr int kPrefillBN = 256;   // tokens per prefill GEMM tile (max)

struct PrefillTile {
  int group;   // routed expert id, or E for the shared expert
  int row0;    // first row in the expert-sorted token order
  int nlen;    // rows in this tile (<= kPrefillBN)
  int m;       // 128-row block of the weight matrix
};

struct PrefillPlanArgs {
  const int32_t* counts;   // [E] picks per expert
  int32_t* cursor;         // [E] scatter cursors (out)
  int32_t* group_slot;     // [E+1] slot of each routed expert with tokens (out)
  PrefillTile* tiles_gu;
  PrefillTile* tiles_dn;
  int32_t* n_tiles;        // [2] (out)
  const int32_t* table;
  int64_t* stamp;
  int64_t* clock;
  int64_t* stats;
  int T, E, k, d, f, layer;
  int account;             // stamp the experts and count the call (0: the cache step did)
  uint32_t* err;
};

// cache step of a prefill chunk (every routed expert with tokens is one key)
struct PrefillCacheArgs {
  const int32_t* counts;   // [E] picks per routed expert
  int32_t* table;          // [L*E]
  int32_t* owner;          // [C]
  int64_t* stamp;          // [C]
  const int32_t* q_in;     // [C] slots, least recently used first
  int32_t* q_out;          // [C] the order after this call
  int q_staged;            // q_in is staged in shared memory (C <= 32768)
  int C, E, layer;
  int64_t* clock;
  int64_t* stats;          // [ST_N] of this layer
  int64_t expert_bytes;
  int32_t* group_slot;     // [E] out: slot of each routed expert with tokens, -1 otherwise
  int32_t* miss_expert;    // [E] out: misses, ascending
  int32_t* miss_slot;      // [E] out: victim slot of each miss
  int32_t* evicted_key;    // [E] out: key the victim held (-1: empty)
  int32_t* info;           // [4] out: misses, distinct experts, token hits, token misses
  uint32_t* err;
};

struct PrefillScatterArgs {
  const int32_t* idx;
  const float* w;
  int32_t* cursor;
  int32_t* perm;           // [T*k + T] token of each sorted row
  float* wsort;            // [T*k + T] combine weight of each sorted row
  int32_t* pick;           // [T*k] pick t*k + i of each routed sorted row
  int T, k;
  float shared_weight;
};

struct PrefillGemmArgs {
  const uint8_t* slots;
  const uint8_t* shared_expert;
  int64_t expert_bytes;
  const int32_t* group_slot;
  const PrefillTile* tiles_gu;
  const PrefillTile* tiles_dn;
  const int32_t* n_tiles;
  uint16_t* hg;            // [rows][f] fp16 hi part of h (gate/up output, down input)
  uint16_t* hg_lo;         // [rows][f] fp16 lo part of h
  const int32_t* perm;
  const float* wsort;
  const int32_t* pick;     // [T*k] pick t*k + i of each routed sorted row
  float* y;                // [T][d]: the shared expert's weighted output (down GEMM)
  float* osort;            // [T*k][d]: weighted output of pick t*k + i in row t*k + i
  int E, d, f;
  uint32_t* err;
};

struct PrefillCombineArgs {
  const float* osort;      // [T*k][d], row t*k + i: pick i of token t
  float* y;                // [T][d], holds the shared expert's part on entry
  int T, k, d;
};

// Raises `func`'s dynamic shared-memory limit to at least `bytes` on the
// current device (once per device and kernel; thread-safe).
cudaError_t ensure_dyn_smem(const void* func, size_t bytes);

// Records the thread-local message returned by moe_last_error().
moe_status set_last_error(moe_status st, const char* fmt, ...);

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s);
cudaError_t launch_commit(const CommitArgs& a, cudaStream_t s);
cudaError_t launch_repack(const RepackArgs& a, cudaStream_t s);
cudaError_t launch_miss_pull(const MissPullArgs& a, cudaStream_t s, int num_sms);
cudaError_t launch_repack_misses(const RepackArgs& a, cudaStream_t s, int num_sms);
}  // namespace moe

#include <cuda.h>
namespace moe {
cudaError_t launch_router_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const RouterGemmArgs& a,
                               cudaStream_t s, int num_sms);
cudaError_t launch_prefill_topk(const PrefillTopkArgs& a, cudaStream_t s);
cudaError_t launch_prefill_plan(const PrefillPlanArgs& a, cudaStream_t s);
cudaError_t launch_prefill_scatter(const PrefillScatterArgs& a, cudaStream_t s);
cudaError_t launch_prefill_gather(const uint16_t* x, const int32_t* perm, uint16_t* xg, int rows, int d,
                                  cudaStream_t s);
cudaError_t launch_prefill_gate_up(const CUtensorMap& tmX, const PrefillGemmArgs& a, cudaStream_t s, int grid);
cudaError_t launch_prefill_down(const CUtensorMap& tmH, const CUtensorMap& tmHlo, const PrefillGemmArgs& a,
                                cudaStream_t s, int grid);
cudaError_t launch_prefill_combine(const PrefillCombineArgs& a, cudaStream_t s);
cudaError_t launch_prefill_cache(const PrefillCacheArgs& a, cudaStream_t s);
struct MissFetch;
cudaError_t launch_prefill_fetch(const MissFetch& f, const int32_t* n_miss, bool device_layout, cudaStream_t s,
                                 int num_sms);
cudaError_t launch_decode_ffn(const FfnArgs& a, cudaStream_t s, bool pdl);
// whether one CTA of every decode-kernel variant fits on an SM at hidden size d
cudaError_t decode_ffn_fits(int d, bool* fits);
cudaError_t launch_calls_bump(uint32_t* counters, cudaStream_t s);

}  // namespace moe
