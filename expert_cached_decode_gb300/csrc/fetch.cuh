// Fetch of missing experts from the registered host pool straight into their
// victim slots, in the device block layout (misses come from pinned host RAM
// that holds every expert, page "一张 RTX 4090 跑千亿模型", §如何做到：三层存储;
// page "单卡5090跑125B 大模型", §7.2).  Shared by the decode kernel (a call's
// misses, jobs spread over its CTAs) and the prefill chunk's fetch kernel.
//
// One job: 32 consecutive rows of one matrix of one missing expert.  In the
// canonical layout the rows' codes and their scales are two contiguous runs,
// so the host pool is read in whole 16-byte chunks; the job is staged in
// shared memory and every warp re-lays out whole 32x32 blocks into the slot.
// Jobs of miss j: Wg row blocks 0..f/32-1, Wu row blocks 0..f/32-1, Wd row
// blocks 0..d/32-1 (2 f/32 + d/32 jobs, 112 at d=2048, f=768).
#pragma once

#include "common.cuh"
#include "repack.cuh"

namespace moe {

struct MissFetch {
  const int32_t* miss_expert;   // [m] expert id (of `layer`) of each miss
  const int32_t* miss_slot;     // [m] its victim slot
  const uint8_t* host_pool;     // device address of the registered host pool (canonical experts)
  int64_t pool_entries;         // key (layer, e) reads entry (layer*E + e) mod pool_entries
  uint8_t* slots;               // slot pool (device block layout)
  int64_t expert_bytes;
  int layer, E, d, f;
};

__host__ __device__ __forceinline__ int fetch_jobs_per_miss(int d, int f) { return 2 * (f / 32) + d / 32; }

// shared-memory bytes of one job: 32 rows x groups x (12 B codes + 2 B scale)
__host__ __device__ __forceinline__ size_t fetch_job_bytes(int d, int f) { return (size_t)14 * (d > f ? d : f); }

struct PullJob {
  const uint8_t* codes;    // host pool: 32 rows x G groups x 12 B
  const uint8_t* scales;   // host pool: 32 rows x G groups x 2 B
  uint8_t* slot;           // the victim slot (device layout)
  int code_bytes, G, mat, rb, miss;
};

__device__ __forceinline__ PullJob pull_job(const MissFetch& a, int q) {
  const int d = a.d, f = a.f, RG = f / 32, JPM = fetch_jobs_per_miss(d, f);
  const int j = q / JPM, r = q - j * JPM;
  const int e = __ldcg(&a.miss_expert[j]);
  const int v = __ldcg(&a.miss_slot[j]);
  const int64_t entry = ((int64_t)a.layer * a.E + e) % a.pool_entries;
  const uint8_t* src = a.host_pool + entry * a.expert_bytes;
  const int64_t gq = (int64_t)f * (d / 32) * 12, dq = (int64_t)d * (f / 32) * 12, gs = (int64_t)f * (d / 32) * 2;
  PullJob J;
  J.miss = j;
  J.slot = a.slots + (int64_t)v * a.expert_bytes;
  if (r < 2 * RG) {
    J.mat = r / RG;
    J.rb = r - J.mat * RG;
    J.G = d / 32;
    J.codes = src + J.mat * gq + (int64_t)J.rb * 32 * J.G * 12;
    J.scales = src + 2 * gq + dq + J.mat * gs + (int64_t)J.rb * 32 * J.G * 2;
  } else {
    J.mat = 2;
    J.rb = r - 2 * RG;
    J.G = f / 32;
    J.codes = src + 2 * gq + (int64_t)J.rb * 32 * J.G * 12;
    J.scales = src + 2 * gq + dq + 2 * gs + (int64_t)J.rb * 32 * J.G * 2;
  }
  J.code_bytes = 32 * J.G * 12;
  return J;
}

// Jobs [q0, q1) by the NTH threads of named barrier 1 (threads 0..NTH-1):
// the next job's 16-byte loads are in flight while this one is re-laid out
// from shared memory `sm` (fetch_job_bytes); after each job a barrier of all
// NTH threads, then thread 0 counts it on ready[miss] (release) when `ready`
// is given.  Every job fits in KPC chunks of 16 bytes per thread.
template <int NTH, int KPC>
__device__ __forceinline__ void pull_jobs(const MissFetch& a, int q0, int q1, uint8_t* sm, uint32_t* ready) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint4 rg[KPC];
  auto load = [&](const PullJob& J) {
    const int ncb = J.code_bytes / 16, n = ncb + J.G * 4;   // scales: 32 rows x G x 2 B = G * 4 chunks
#pragma unroll
    for (int i = 0; i < KPC; ++i) {
      const int c = tid + i * NTH;
      if (c < n)
        rg[i] = c < ncb ? reinterpret_cast<const uint4*>(J.codes)[c]
                        : reinterpret_cast<const uint4*>(J.scales)[c - ncb];
    }
  };
  if (q0 < q1) load(pull_job(a, q0));
  for (int q = q0; q < q1; ++q) {
    const PullJob J = pull_job(a, q);
    const int n = J.code_bytes / 16 + J.G * 4;
#pragma unroll
    for (int i = 0; i < KPC; ++i) {
      const int c = tid + i * NTH;
      if (c < n) reinterpret_cast<uint4*>(sm)[c] = rg[i];
    }
    named_bar(1, NTH);
    if (q + 1 < q1) load(pull_job(a, q + 1));
    for (int gi = warp; gi < J.G; gi += NTH / 32) {
      const uint32_t* cw = reinterpret_cast<const uint32_t*>(sm + (size_t)(lane * J.G + gi) * 12);
      const uint16_t sc = reinterpret_cast<const uint16_t*>(sm + J.code_bytes)[lane * J.G + gi];
      const int64_t off = J.mat < 2 ? gu_block_offset(J.rb, gi, J.mat, a.d) : down_block_offset(J.rb, gi, a.d, a.f);
      pack_block(cw[0], cw[1], cw[2], sc, lane, J.slot + off);
    }
    named_bar(1, NTH);
    if (ready && tid == 0) red_release_add(&ready[J.miss], 1u);   // covers every warp's blocks (after the barrier)
  }
}

}  // namespace moe
