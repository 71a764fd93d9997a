// Canonical packed expert -> device block layout (see common.cuh), one
// 32-row x 32-input block per warp; used by the repack kernel and by the
// decode kernel's in-kernel miss handling.
//
// Canonical format: weight i of a 12-byte group is the 3-bit field at bits
// [3i, 3i+3) of the 96-bit little-endian integer (q = u - 4), one fp16
// scale per group.  Lane r first reads row r's 12-byte group, then every
// lane gathers, by shuffles, the codes of its mma fragment pairs and writes
// its three words.
#pragma once

#include "common.cuh"

namespace moe {

__device__ __forceinline__ uint32_t field3(uint32_t w0, uint32_t w1, uint32_t w2, int i) {
  // bits [3i, 3i+3) of the 96-bit value (w2:w1:w0)
  const int b = 3 * i;
  const uint64_t lo = ((uint64_t)w1 << 32) | w0;
  if (b + 3 <= 64) return (uint32_t)(lo >> b) & 7u;
  if (b >= 64) return (w2 >> (b - 64)) & 7u;
  return (uint32_t)((lo >> b) | ((uint64_t)w2 << (64 - b))) & 7u;
}

// One block from its 32 rows: lane r holds row r's 12-byte group (r0, r1,
// r2) and its scale; every lane gathers, by shuffles, the codes of its mma
// fragment pairs and writes its three words, lanes 0-7 the scales.  One whole
// warp calls it.
__device__ __forceinline__ void pack_block(uint32_t r0, uint32_t r1, uint32_t r2, uint16_t my_scale, int lane,
                                           uint8_t* out) {
  const int g = lane >> 2, c = lane & 3;
  uint32_t W[3] = {0u, 0u, 0u};
#pragma unroll
  for (int p = 0; p < 16; ++p) {
    const int mt = p >> 3, ks = (p >> 2) & 1, r = p & 3;
    const int prow = mt * 16 + g + 8 * (r & 1);
    const int k0 = ks * 16 + 2 * c + 8 * (r >> 1);
    const uint32_t s0 = __shfl_sync(0xffffffffu, r0, prow);
    const uint32_t s1 = __shfl_sync(0xffffffffu, r1, prow);
    const uint32_t s2 = __shfl_sync(0xffffffffu, r2, prow);
    const uint32_t ulo = field3(s0, s1, s2, k0);
    const uint32_t uhi = field3(s0, s1, s2, k0 + 1);
    if (p < 15) {
      const int j = p / 5, fld = p % 5;
      W[j] |= (ulo << (3 * fld)) | (uhi << (16 + 3 * fld));
    } else {
#pragma unroll
      for (int b = 0; b < 3; ++b) W[b] |= (((ulo >> b) & 1u) << 15) | (((uhi >> b) & 1u) << 31);
    }
  }
  uint32_t* dw = reinterpret_cast<uint32_t*>(out);
  dw[lane] = W[0];
  dw[32 + lane] = W[1];
  dw[64 + lane] = W[2];
  // scales: lane g8 < 8 writes rows g8, g8+8, g8+16, g8+24
  const uint32_t sv = my_scale;
  const uint32_t s_a = __shfl_sync(0xffffffffu, sv, lane & 7);
  const uint32_t s_b = __shfl_sync(0xffffffffu, sv, (lane & 7) + 8);
  const uint32_t s_c = __shfl_sync(0xffffffffu, sv, (lane & 7) + 16);
  const uint32_t s_d = __shfl_sync(0xffffffffu, sv, (lane & 7) + 24);
  if (lane < 8) {
    uint2 o;
    o.x = s_a | (s_b << 16);
    o.y = s_c | (s_d << 16);
    *reinterpret_cast<uint2*>(out + kBlockCodeBytes + 8 * lane) = o;
  }
  __syncwarp();   // a following block's shuffles run on the whole warp again
}

// Block bi of the expert at `src` (canonical) into the expert at `dst`
// (device layout); blocks 0 .. 2(f/32)(d/32)-1 are gate/up (row block, group,
// Wg then Wu), the rest down (row block, group).  One whole warp calls it.
// The source is read through L2 (it may have been written by other CTAs of
// the same kernel).
__device__ __forceinline__ void repack_block(const uint8_t* src, uint8_t* dst, int bi, int d, int f, int lane) {
  const int gu_blocks = (f / 32) * (d / 32) * 2;
  // canonical sections
  const int64_t gq = (int64_t)f * (d / 32) * 12, dq = (int64_t)d * (f / 32) * 12;
  const int64_t gs = (int64_t)f * (d / 32) * 2;
  const int64_t sec_q[3] = {0, gq, 2 * gq};
  const int64_t sec_s[3] = {2 * gq + dq, 2 * gq + dq + gs, 2 * gq + dq + 2 * gs};
  int mat, rb, gi, cols;
  int64_t dst_off;
  if (bi < gu_blocks) {
    rb = bi / ((d / 32) * 2);
    const int rem = bi % ((d / 32) * 2);
    gi = rem / 2;
    mat = rem % 2;
    cols = d;
    dst_off = gu_block_offset(rb, gi, mat, d);
  } else {
    const int bj = bi - gu_blocks;
    rb = bj / (f / 32);
    gi = bj % (f / 32);
    mat = 2;
    cols = f;
    dst_off = down_block_offset(rb, gi, d, f);
  }
  const int row = rb * 32 + lane;
  const int64_t g_index = (int64_t)row * (cols / 32) + gi;
  const uint32_t* gp = reinterpret_cast<const uint32_t*>(src + sec_q[mat] + g_index * 12);
  const uint32_t r0 = __ldcg(gp), r1 = __ldcg(gp + 1), r2 = __ldcg(gp + 2);
  const uint16_t my_scale = __ldcg(reinterpret_cast<const unsigned short*>(src + sec_s[mat] + g_index * 2));
  pack_block(r0, r1, r2, my_scale, lane, dst + dst_off);
}

}  // namespace moe
