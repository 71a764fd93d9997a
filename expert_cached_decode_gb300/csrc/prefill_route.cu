// Prefill routing (T up to 16,384 tokens): router logits on the tensor cores,
// then top-k per token and the counting sort of token picks by expert.
//
// Router: logits^T[E x T] = Wr[E x d] . X^T, bf16 operands fetched by TMA
// (128-byte swizzle), fp32 accumulation in tensor memory, tcgen05.mma issued
// by one thread.  128 experts x 256 tokens per tile, 64-wide k blocks, a
// 4-stage shared-memory pipeline and a double-buffered accumulator so the
// epilogue of one tile overlaps the main loop of the next.  The selection is
// the same as the decode path's (ties to the lower id, softmax over the chosen
// logits, ids ascending), one warp per token.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace moe {

namespace rg {
constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;        // 16 KB
constexpr int B_BYTES = BN * BK * 2;        // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_BYTES = 32 * BM * 4;      // 32 tokens x 128 experts fp32
constexpr int THREADS = 256;                // warp 0 TMA, warp 1 MMA, warps 4-7 epilogue
constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + 256;
}  // namespace rg

__global__ void __launch_bounds__(rg::THREADS, 1)
    router_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       RouterGemmArgs a) {
  using namespace rg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_base = smem;
  float* epi = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES + EPI_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_mt = (a.E + BM - 1) / BM, n_nt = (a.T + BN - 1) / BN;
  const int n_tiles = n_mt * n_nt, n_kb = a.d / BK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 4);
    }
    mbar_init_fence();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == 0 && lane == 0) {
    uint32_t it = 0;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
      const int mt = tile % n_mt, nt = tile / n_mt;
      for (int kb = 0; kb < n_kb; ++kb, ++it) {
        const int s = it % STAGES;
        const uint32_t use = it / STAGES;
        if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1)) {
          ok = false;
          set_error(a.err, DEV_TIMEOUT_BARRIER);
          break;
        }
        uint8_t* st = stage_base + s * STAGE_BYTES;
        mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
        tma_load_2d(st, &tmA, kb * BK, mt * BM, &full[s]);
        tma_load_2d(st + A_BYTES, &tmB, kb * BK, nt * BN, &full[s]);
      }
    }
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = idesc_f16(BM, BN, 1);
    uint32_t it = 0, lt = 0;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++lt) {
      const int ab = lt & 1;
      const uint32_t use_b = lt >> 1;
      if (use_b > 0 && !mbar_wait(&tempty[ab], (use_b - 1) & 1)) {
        ok = false;
        set_error(a.err, DEV_TIMEOUT_BARRIER);
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem + ab * BN;
      for (int kb = 0; kb < n_kb; ++kb, ++it) {
        const int s = it % STAGES;
        if (!mbar_wait(&full[s], (it / STAGES) & 1)) {
          ok = false;
          set_error(a.err, DEV_TIMEOUT_BARRIER);
          break;
        }
        tc_fence_after();
        uint8_t* st = stage_base + s * STAGE_BYTES;
        const uint64_t da = smem_desc_sw128(st), db = smem_desc_sw128(st + A_BYTES);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          umma_f16(d_tmem, da + 2 * kk, db + 2 * kk, idesc, (kb | kk) != 0);
        umma_commit(&empty[s]);
      }
      if (!ok) break;
      umma_commit(&tfull[ab]);
    }
  } else if (warp >= 4) {
    const int q = warp - 4;
    uint32_t lt = 0;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++lt) {
      const int mt = tile % n_mt, nt = tile / n_mt;
      const int ab = lt & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull[ab], (lt >> 1) & 1))) {
        ok = false;
        set_error(a.err, DEV_TIMEOUT_BARRIER);
        break;
      }
      tc_fence_after();
      const int e = mt * BM + q * 32 + lane;
      const float b = e < a.E ? a.bias[e] : 0.f;
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + ab * BN + c * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) epi[j * BM + q * 32 + lane] = __uint_as_float(r[j]) + b;
        named_bar(1, 128);
        const int t0 = nt * BN + c * 32;
        for (int j = 0; j < 32; ++j) {
          const int t = t0 + j;
          const int ee = mt * BM + (threadIdx.x - 128);
          if (t < a.T && ee < a.E) a.logits[(size_t)t * a.E + ee] = epi[j * BM + (threadIdx.x - 128)];
        }
        named_bar(1, 128);
      }
      tc_fence_before();
      if (lane == 0) mbar_arrive(&tempty[ab]);
      __syncwarp();   // the next tile's tcgen05.ld runs on the whole warp
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// One warp per token: top-k of the logits row, weights, per-expert counts.
__global__ void __launch_bounds__(256) prefill_topk_kernel(PrefillTopkArgs a) {
  __shared__ uint64_t scratch[8][kTopkScratch];
  __shared__ float rows[8][kMaxE];
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= a.T) return;
  const int t = warp, E = a.E, K = a.k;
  float* row = rows[threadIdx.x >> 5];
#pragma unroll 8
  for (int id = lane; id < E; id += 32) row[id] = a.logits[(size_t)t * E + id];
  __syncwarp();
  float my_v;
  int my_id;
  if (E <= 512) warp_topk_reg<16>(row, E, K, lane, scratch[threadIdx.x >> 5], my_v, my_id);
  else warp_topk(row, E, K, lane, scratch[threadIdx.x >> 5], my_v, my_id);
  const float top = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = lane < K ? expf(my_v - top) : 0.f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  int rank = 0;
  for (int j = 0; j < K; ++j) rank += (__shfl_sync(0xffffffffu, my_id, j) < my_id) ? 1 : 0;
  if (lane < K) {
    a.idx[(size_t)t * K + rank] = my_id;
    a.w[(size_t)t * K + rank] = ex / sum;
    if (a.counts) atomicAdd(&a.counts[my_id], 1);
  }
}

cudaError_t launch_router_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const RouterGemmArgs& a,
                               cudaStream_t s, int num_sms) {
  cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(router_gemm_kernel), rg::SMEM);
  if (e != cudaSuccess) return e;
  const int n_tiles = ((a.E + rg::BM - 1) / rg::BM) * ((a.T + rg::BN - 1) / rg::BN);
  const int grid = n_tiles < num_sms ? n_tiles : num_sms;
  router_gemm_kernel<<<grid, rg::THREADS, rg::SMEM, s>>>(tmA, tmB, a);
  return cudaGetLastError();
}

cudaError_t launch_prefill_topk(const PrefillTopkArgs& a, cudaStream_t s) {
  const int blocks = (a.T * 32 + 255) / 256;
  prefill_topk_kernel<<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
