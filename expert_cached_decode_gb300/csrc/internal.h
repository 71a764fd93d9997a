// Library-internal declarations: the routing plan, kernel argument blocks and
// host-side launchers (one per .cu file).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

constexpr int kMaxDecodeT = 16;   // tokens per call on the decode path
constexpr int kMaxTopK = 16;
constexpr int kMaxE = 1024;
constexpr int kMaxPicks = kMaxDecodeT * kMaxTopK;   // 256
constexpr int kMaxSlots = 1 << 17;                  // LRU scan bitmap bound

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

enum RouteMode : int { ROUTE_ONLY = 0, ROUTE_RESIDENT = 1, ROUTE_PLAN = 2 };

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
};

struct FfnArgs {
  const uint8_t* slots;         // slot pool base
  const uint8_t* shared_expert; // this layer's shared expert (device layout)
  int64_t expert_bytes;
  const uint16_t* x;            // [T][d] bf16
  float* y;                     // [T][d]
  int T, d, f, k;
  float shared_weight;
  const Plan* plan;
  float* gu_partial;
  uint16_t* hfrag;
  float* obuf;
  uint32_t* gu_cnt;
  uint32_t* h_ready;
  uint32_t* d_cnt;
  uint32_t* done;
  uint32_t* err;
  int grid;
};

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s);
cudaError_t launch_commit(const CommitArgs& a, cudaStream_t s);
cudaError_t launch_repack(const RepackArgs& a, cudaStream_t s);
cudaError_t launch_decode_ffn(const FfnArgs& a, cudaStream_t s, bool pdl, int num_sms);

}  // namespace moe
