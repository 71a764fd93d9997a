// Canonical packed expert -> device block layout: the repack kernel (cache
// configuration and host-copied misses) and the GPU's own pull of missing
// experts from the host pool.
#include "common.cuh"
#include "internal.h"
#include "repack.cuh"

namespace moe {

__global__ void __launch_bounds__(256) repack_kernel(RepackArgs a) {
  const int lane = threadIdx.x & 31;
  const int d = a.d, f = a.f;
  const int nb = (f / 32) * (d / 32) * 2 + (d / 32) * (f / 32);
  // with a plan, the experts are the call's misses (known on the device only)
  const int n_ex = a.plan ? a.plan->n_miss : a.n_experts;
  const int32_t* dst_slot = a.plan ? a.plan->miss_slot : a.dst_slot;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x / 32);
  for (int64_t gwarp = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); gwarp < (int64_t)nb * n_ex;
       gwarp += nwarps) {
    const int ex = (int)(gwarp / nb);
    const int bi = (int)(gwarp % nb);
    uint8_t* dst = dst_slot ? a.dst_base + (int64_t)dst_slot[ex] * a.dst_stride : a.dst_base + (int64_t)ex * a.dst_stride;
    repack_block(a.src + (int64_t)ex * a.src_stride, dst, bi, d, f, lane);
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
    uint4* dst = reinterpret_cast<uint4*>(a.dst_slots ? a.dst_slots + (int64_t)a.plan->miss_slot[j] * a.expert_bytes
                                                      : a.staging + (int64_t)j * a.expert_bytes);
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
