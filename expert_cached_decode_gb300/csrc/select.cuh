// Router logits and expert selection of one decode layer-call (T <= 16
// tokens), shared by the stand-alone routing kernel and the fused decode
// kernel so that both produce the same logits and the same selection.
//
// Router (workload definition; the pages only fix 10-of-512 routing plus a
// shared expert, page "一张 RTX 4090 跑千亿模型", §如何做到：三层存储):
//   l[t,e] = x_t . Wr[e] + b[e] in fp32 from bf16 inputs; the k largest
//   logits are chosen (ties to the lower id); w_i = softmax over the whole
//   row restricted to the chosen set and renormalised, which equals a softmax
//   over the k chosen logits alone.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace moe {

// Lane chunks j = jb + lane*8 + 256*u (u < 8) of a 2048-wide block of a
// router row (zero past d).
// Router rows are read by every call of their layer: they are kept in L2
// with the evict-last policy.
__device__ __forceinline__ void router_load_block(const uint16_t* __restrict__ wrow, int jb, int d, int lane,
                                                  uint4 (&wv)[8]) {
  const uint64_t pol = l2_evict_last_policy();
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int j = jb + lane * 8 + 256 * u;
    wv[u] = j < d ? ld_nc_v4_hint(wrow + j, pol) : make_uint4(0u, 0u, 0u, 0u);
  }
}

// s += the 8 products of one 16-byte chunk of x and of a router row, in order
__device__ __forceinline__ float dot8_bf16(uint4 w4, uint4 x4, float s) {
  s = fmaf(bf16_bits_to_float(x4.x & 0xffffu), bf16_bits_to_float(w4.x & 0xffffu), s);
  s = fmaf(bf16_bits_to_float(x4.x >> 16), bf16_bits_to_float(w4.x >> 16), s);
  s = fmaf(bf16_bits_to_float(x4.y & 0xffffu), bf16_bits_to_float(w4.y & 0xffffu), s);
  s = fmaf(bf16_bits_to_float(x4.y >> 16), bf16_bits_to_float(w4.y >> 16), s);
  s = fmaf(bf16_bits_to_float(x4.z & 0xffffu), bf16_bits_to_float(w4.z & 0xffffu), s);
  s = fmaf(bf16_bits_to_float(x4.z >> 16), bf16_bits_to_float(w4.z >> 16), s);
  s = fmaf(bf16_bits_to_float(x4.w & 0xffffu), bf16_bits_to_float(w4.w & 0xffffu), s);
  s = fmaf(bf16_bits_to_float(x4.w >> 16), bf16_bits_to_float(w4.w >> 16), s);
  return s;
}

// One warp: logits of expert row `wrow` for the T tokens of x (bf16 rows
// xstride elements apart, 16-byte aligned, global or shared memory), given
// the row's first 2048-wide block in `first` (router_load_block at jb = 0).
// Per token, lane chunks accumulate in u order within each 2048-wide block,
// blocks in order, then a butterfly sum; lane 0 hands l[t, e] = dot + bias
// to store(t, value).  Tokens run in a loop (this code runs once per call,
// so it is kept short).
template <class Store>
__device__ __forceinline__ void router_row(const uint16_t* __restrict__ wrow, const uint4 (&first)[8],
                                           const uint16_t* __restrict__ x, int xstride, float bias, int T, int d,
                                           int lane, Store store) {
#pragma unroll 1
  for (int t = 0; t < T; ++t) {
    const uint16_t* xr = x + (size_t)t * xstride;
    float s = 0.f;
#pragma unroll 1
    for (int jb = 0; jb < d; jb += 2048) {
      uint4 wv[8];
      if (jb == 0) {
#pragma unroll
        for (int u = 0; u < 8; ++u) wv[u] = first[u];
      } else {
        router_load_block(wrow, jb, d, lane, wv);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int jj = jb + lane * 8 + 256 * u;
        if (jj < d) s = dot8_bf16(wv[u], *reinterpret_cast<const uint4*>(xr + jj), s);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) store(t, s + bias);
    __syncwarp();   // the next token's shuffles run on the whole warp again
  }
}

// warps of a block that take tokens in select_call (further warps only join
// its barriers)
constexpr int kSelWarps = 8;

// Selection of one call, in shared memory.
struct SelSmem {
  float row[kSelWarps][kMaxE];               // logits row of each selecting warp
  uint64_t topk[kSelWarps][kTopkScratch];   // warp_topk scratch
  uint32_t mask[kMaxE / 32];          // chosen experts of the call
  int word_base[kMaxE / 32];          // distinct experts below word i
  int sel_id[kMaxDecodeT][kMaxTopK];  // per token, ascending id
  float sel_w[kMaxDecodeT][kMaxTopK];
  int act[kMaxPicks];                 // distinct experts U, ascending
  int n_act;
};

// Index in U of chosen expert `id`.
__device__ __forceinline__ int sel_act_index(const SelSmem* s, int id) {
  return s->word_base[id >> 5] + __popc(s->mask[id >> 5] & ((1u << (id & 31)) - 1u));
}

// Every participating thread calls this: the whole block when NTH is 0,
// else the first NTH threads (warps 0 .. NTH/32-1, synchronised by named
// barrier 1); warps below kSelWarps select.
// Reads the logits rows [T][E] through the loader (`logits.row`: plain loads
// through L2 after the writers were waited for, or tagged words polled until
// they carry the call's tag); warps take
// tokens in turn: top-k (ties to the lower id), weights, ids ascending; then
// warp 0 forms U.
// `tl` (timeline builds only) receives %globaltimer stamps of the steps.
// default loader of the logits rows: plain floats through L2; row(r, t, E,
// lane) fills r[id] = l[t, id] for the lane's ids lane, lane + 32, ...
struct PlainLogits {
  const float* p;
  __device__ __forceinline__ void row(float* r, int t, int E, int lane) const {
#pragma unroll 16
    for (int id = lane; id < E; id += 32) r[id] = ld_cg_f32(p + (size_t)t * E + id);
  }
};

template <int NTH = 0, class Load = PlainLogits>
__device__ __forceinline__ void select_call(Load logits, int T, int E, int K, SelSmem* s,
                                            unsigned long long* tl = nullptr) {
  const int nthreads = NTH == 0 ? (int)blockDim.x : NTH;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#ifdef MOE_TIMELINE
#define SEL_TL(i) \
  if (tl && threadIdx.x == 0) tl[i] = globaltimer()
#else
#define SEL_TL(i) ((void)0)
#endif
  for (int i = threadIdx.x; i < kMaxE / 32; i += nthreads) s->mask[i] = 0;
  step_bar<NTH>();
  for (int t = warp; warp < kSelWarps && t < T; t += kSelWarps) {
    float* row = s->row[warp];
    logits.row(row, t, E, lane);
    __syncwarp();
    if (t == 0) SEL_TL(0);
    float my_v;
    int my_id;
    if (E <= 512) warp_topk_reg<16>(row, E, K, lane, s->topk[warp], my_v, my_id);
    else warp_topk(row, E, K, lane, s->topk[warp], my_v, my_id);
    if (t == 0) SEL_TL(1);
    const float top = __shfl_sync(0xffffffffu, my_v, 0);
    const float ex = lane < K ? expf(my_v - top) : 0.f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    int rank = 0;
    for (int j = 0; j < K; ++j) {
      const int oid = __shfl_sync(0xffffffffu, my_id, j);
      rank += (oid < my_id) ? 1 : 0;
    }
    if (lane < K) {
      s->sel_id[t][rank] = my_id;
      s->sel_w[t][rank] = ex / sum;
      atomicOr(&s->mask[my_id >> 5], 1u << (my_id & 31));
    }
    if (t == 0) SEL_TL(2);
  }
  step_bar<NTH>();
  SEL_TL(3);
  const int n_words = (E + 31) / 32;
  if (warp == 0) {
    const uint32_t m = lane < n_words ? s->mask[lane] : 0u;
    const int c = __popc(m);
    int inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += n;
    }
    const int base = inc - c;
    if (lane < n_words) s->word_base[lane] = base;
    if (lane == 31) s->n_act = inc;
    uint32_t mm = m;
    int pos = base;
    while (mm) {
      const int bit = __ffs(mm) - 1;
      mm &= mm - 1;
      s->act[pos++] = lane * 32 + bit;
    }
  }
  step_bar<NTH>();
  SEL_TL(4);
#undef SEL_TL
}

}  // namespace moe
