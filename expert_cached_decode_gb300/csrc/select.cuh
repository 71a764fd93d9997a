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

// One warp: logits of expert row `wrow` for the T tokens of x.  Lane chunk
// j = lane*8 + 256*u of every 2048-wide block, accumulated in u order, then a
// butterfly sum; lane 0 stores l[t, e] = dot + bias at logits[t*E + e].
__device__ __forceinline__ void router_row(const uint16_t* __restrict__ wrow, const uint16_t* __restrict__ x,
                                           float bias, int T, int d, int E, int e, int lane, float* logits) {
  float acc[kMaxDecodeT];
#pragma unroll
  for (int t = 0; t < kMaxDecodeT; ++t) acc[t] = 0.f;
  for (int jb = 0; jb < d; jb += 2048) {
    uint4 wv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = jb + lane * 8 + 256 * u;
      wv[u] = j < d ? __ldg(reinterpret_cast<const uint4*>(wrow + j)) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int t = 0; t < kMaxDecodeT; ++t) {
      if (t < T) {
        uint4 xv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int j = jb + lane * 8 + 256 * u;
          xv[u] = j < d ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * d + j)) : make_uint4(0u, 0u, 0u, 0u);
        }
        float s = acc[t];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 w4 = wv[u], x4 = xv[u];
          s = fmaf(bf16_bits_to_float(x4.x & 0xffffu), bf16_bits_to_float(w4.x & 0xffffu), s);
          s = fmaf(bf16_bits_to_float(x4.x >> 16), bf16_bits_to_float(w4.x >> 16), s);
          s = fmaf(bf16_bits_to_float(x4.y & 0xffffu), bf16_bits_to_float(w4.y & 0xffffu), s);
          s = fmaf(bf16_bits_to_float(x4.y >> 16), bf16_bits_to_float(w4.y >> 16), s);
          s = fmaf(bf16_bits_to_float(x4.z & 0xffffu), bf16_bits_to_float(w4.z & 0xffffu), s);
          s = fmaf(bf16_bits_to_float(x4.z >> 16), bf16_bits_to_float(w4.z >> 16), s);
          s = fmaf(bf16_bits_to_float(x4.w & 0xffffu), bf16_bits_to_float(w4.w & 0xffffu), s);
          s = fmaf(bf16_bits_to_float(x4.w >> 16), bf16_bits_to_float(w4.w >> 16), s);
        }
        acc[t] = s;
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kMaxDecodeT; ++t) {
    if (t < T) {
      float v = acc[t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) logits[(size_t)t * E + e] = v + bias;
    }
  }
}

// Selection of one call, in shared memory.
struct SelSmem {
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

// Every thread of the block calls this.  Reads the logits rows [T][E] from
// global memory through L2 (they were written by other CTAs of this kernel
// or of the same launch); warps take tokens in turn: top-k (ties to the lower
// id), weights, ids ascending; then warp 0 forms U.
__device__ __forceinline__ void select_call(const float* logits, int T, int E, int K, SelSmem* s) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int i = threadIdx.x; i < kMaxE / 32; i += blockDim.x) s->mask[i] = 0;
  __syncthreads();
  for (int t = warp; t < T; t += nw) {
    float my_v;
    int my_id;
    if (E <= 512) {
      float v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int id = lane + 32 * i;
        v[i] = id < E ? ld_cg_f32(logits + (size_t)t * E + id) : -INFINITY;
      }
      warp_topk<16>(v, E, K, lane, my_v, my_id);
    } else {
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int id = lane + 32 * i;
        v[i] = id < E ? ld_cg_f32(logits + (size_t)t * E + id) : -INFINITY;
      }
      warp_topk<32>(v, E, K, lane, my_v, my_id);
    }
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
  }
  __syncthreads();
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
  __syncthreads();
}

}  // namespace moe
