// Canonical packed expert -> device block layout (see common.cuh).
//
// Canonical format: weight i of a 12-byte group is the 3-bit field at bits
// [3i, 3i+3) of the 96-bit little-endian integer (q = u - 4), one fp16
// scale per group.  One warp re-lays out one 32-row x 32-input block: lane r
// first reads row r's 12-byte group, then every lane gathers, by shuffles,
// the codes of its mma fragment pairs and writes its three words.
#include "common.cuh"
#include "internal.h"

namespace moe {

__device__ __forceinline__ uint32_t field3(uint32_t w0, uint32_t w1, uint32_t w2, int i) {
  // bits [3i, 3i+3) of the 96-bit value (w2:w1:w0)
  const int b = 3 * i;
  const uint64_t lo = ((uint64_t)w1 << 32) | w0;
  if (b + 3 <= 64) return (uint32_t)(lo >> b) & 7u;
  if (b >= 64) return (w2 >> (b - 64)) & 7u;
  return (uint32_t)((lo >> b) | ((uint64_t)w2 << (64 - b))) & 7u;
}

__global__ void __launch_bounds__(256) repack_kernel(RepackArgs a) {
  const int lane = threadIdx.x & 31;
  const int d = a.d, f = a.f;
  const int gu_blocks = (f / 32) * (d / 32) * 2;
  const int nb = gu_blocks + (d / 32) * (f / 32);
  // with a plan, the experts are the call's misses (known on the device only)
  const int n_ex = a.plan ? a.plan->n_miss : a.n_experts;
  const int32_t* dst_slot = a.plan ? a.plan->miss_slot : a.dst_slot;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x / 32);
  for (int64_t gwarp = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); gwarp < (int64_t)nb * n_ex;
       gwarp += nwarps) {
    const int ex = (int)(gwarp / nb);
    const int bi = (int)(gwarp % nb);

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
    const uint8_t* src = a.src + (int64_t)ex * a.src_stride;
    const int row = rb * 32 + lane;
    const int64_t g_index = (int64_t)row * (cols / 32) + gi;
    const uint32_t* gp = reinterpret_cast<const uint32_t*>(src + sec_q[mat] + g_index * 12);
    const uint32_t r0 = gp[0], r1 = gp[1], r2 = gp[2];
    const uint16_t my_scale = *reinterpret_cast<const uint16_t*>(src + sec_s[mat] + g_index * 2);

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
    uint8_t* dst = (dst_slot ? a.dst_base + (int64_t)dst_slot[ex] * a.dst_stride
                             : a.dst_base + (int64_t)ex * a.dst_stride) + dst_off;
    uint32_t* dw = reinterpret_cast<uint32_t*>(dst);
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
      uint2 out;
      out.x = s_a | (s_b << 16);
      out.y = s_c | (s_d << 16);
      *reinterpret_cast<uint2*>(dst + kBlockCodeBytes + 8 * lane) = out;
    }
  }
}

// The call's missing experts, read by the GPU straight from the registered
// host pool (over NVLink-C2C or PCIe) into the staging slots, 16 bytes per
// thread and step; the miss list and its length come from the plan in device
// memory, so no host round trip sits between routing and the copies.
__global__ void __launch_bounds__(256) miss_pull_kernel(MissPullArgs a) {
  const int m = a.plan->n_miss;
  if (m > a.staging_n) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_error(a.err, DEV_BAD_PLAN);
    return;
  }
  const int64_t per = a.expert_bytes / 16;
  const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
  for (int j = 0; j < m; ++j) {
    const int64_t entry = ((int64_t)a.layer * a.E + a.plan->miss_expert[j]) % a.pool_entries;
    const uint4* src = reinterpret_cast<const uint4*>(a.host_pool + entry * a.expert_bytes);
    uint4* dst = reinterpret_cast<uint4*>(a.staging + (int64_t)j * a.expert_bytes);
    int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; c + 3 * nthr < per; c += 4 * nthr) {   // four loads in flight per thread
      const uint4 v0 = src[c], v1 = src[c + nthr], v2 = src[c + 2 * nthr], v3 = src[c + 3 * nthr];
      dst[c] = v0;
      dst[c + nthr] = v1;
      dst[c + 2 * nthr] = v2;
      dst[c + 3 * nthr] = v3;
    }
    for (; c < per; c += nthr) dst[c] = src[c];
  }
}

cudaError_t launch_miss_pull(const MissPullArgs& a, cudaStream_t s, int num_sms) {
  miss_pull_kernel<<<4 * num_sms, 256, 0, s>>>(a);
  return cudaGetLastError();
}

// repack of the plan's misses: a persistent grid (their number is on the device)
cudaError_t launch_repack_misses(const RepackArgs& a, cudaStream_t s, int num_sms) {
  repack_kernel<<<8 * num_sms, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_repack(const RepackArgs& a, cudaStream_t s) {
  const int nb = (a.f / 32) * (a.d / 32) * 2 + (a.d / 32) * (a.f / 32);
  const int64_t warps = (int64_t)nb * a.n_experts;
  if (warps == 0) return cudaSuccess;
  const int64_t grid = (warps + 7) / 8;
  repack_kernel<<<(unsigned)grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
