// Decode / verify expert FFN (T <= 16 tokens): every distinct routed expert
// and the shared expert run once for all tokens routed to them (a verify
// batch shares one fetch of each expert, page "单卡5090跑125B 大模型", §2.3),
//   g = Wg.x, u = Wu.x, h = silu(g) * u, o = Wd.h,
//   y[t] = shared_weight * o_shared[t] + sum_i w[t,i] * o_idx[t,i][t].
//
// Work is cut into units that stream contiguous bytes of the device layout:
//   gate/up unit (expert a, 32-row block rb of f, 8 of the d/32 groups): the
//     Wg and Wu blocks of those groups (16 x 448 B); its partial g/u sums go to
//     scratch and the last of the d/256 units of (a, rb) finishes g, u, forms
//     h = silu(g) * u (fp16) and bumps h_ready[a];
//   down unit (expert a, 32-row block rb of d): f/32 Wd blocks; waits for
//     h_ready[a] == f/32, writes o_a for its rows, and the last expert to
//     finish a row block combines y for those rows in a fixed order
//     (shared expert, then routed experts in ascending id).
// One persistent CTA per SM takes a contiguous, byte-balanced range of units.
// A producer thread streams each unit into a shared-memory ring with bulk
// TMA copies (mbarrier completion); 12 consumer warps expand the 3-bit codes
// to fp16 in registers and multiply on the tensor cores (mma.sync m16n8k16,
// fp32 accumulate, per-group scale applied in fp32).  All waits are bounded.
#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kConsumerWarps = 12;
constexpr int kFfnThreads = (kConsumerWarps + 1) * 32;
constexpr int kGuGroups = 8;     // groups per gate/up unit
constexpr int kNumSlots = 12;

__host__ __device__ __forceinline__ int ffn_slot_bytes(int f) {
  const int dg = f / 32;
  return (dg > 2 * kGuGroups ? dg : 2 * kGuGroups) * kBlockBytes;
}

__host__ __device__ __forceinline__ size_t ffn_smem_bytes(int nt, int d, int f) {
  return (size_t)nt * d * 16 + (size_t)kNumSlots * ffn_slot_bytes(f) + 2 * kNumSlots * 8 + 64;
}

__device__ __forceinline__ uint32_t pack_half2_from_bf16(uint16_t lo, uint16_t hi) {
  const __half2 h = __floats2half2_rn(bf16_bits_to_float(lo), bf16_bits_to_float(hi));
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void scales4(const uint8_t* bp, int lane, float s[4]) {
  const uint2 sc = *reinterpret_cast<const uint2*>(bp + kBlockCodeBytes + (lane >> 2) * 8);
  s[0] = __half2float(__ushort_as_half((unsigned short)(sc.x & 0xffffu)));  // row g
  s[1] = __half2float(__ushort_as_half((unsigned short)(sc.x >> 16)));      // row g+8
  s[2] = __half2float(__ushort_as_half((unsigned short)(sc.y & 0xffffu)));  // row g+16
  s[3] = __half2float(__ushort_as_half((unsigned short)(sc.y >> 16)));      // row g+24
}

// One 32x32 block: acc[nt][mt][i] += scale(row) * (A_block . B_frag[nt])
template <int NT>
__device__ __forceinline__ void block_mma(const uint8_t* bp, int lane, const uint2 (&bx)[NT][2],
                                          float (&acc)[NT][2][4]) {
  const uint32_t* wp = reinterpret_cast<const uint32_t*>(bp);
  const uint32_t w0 = wp[lane], w1 = wp[32 + lane], w2 = wp[64 + lane];
  float s[4];
  scales4(bp, lane, s);
  uint32_t A[16];
  dequant_block(w0, w1, w2, A);
  const float zero[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      float D[4];
      mma_16816(D, &A[mt * 8], bx[nt][0].x, bx[nt][0].y, zero);
      mma_16816(D, &A[mt * 8 + 4], bx[nt][1].x, bx[nt][1].y, D);
      const float sa = s[2 * mt], sb = s[2 * mt + 1];
      acc[nt][mt][0] = fmaf(sa, D[0], acc[nt][mt][0]);
      acc[nt][mt][1] = fmaf(sa, D[1], acc[nt][mt][1]);
      acc[nt][mt][2] = fmaf(sb, D[2], acc[nt][mt][2]);
      acc[nt][mt][3] = fmaf(sb, D[3], acc[nt][mt][3]);
    }
  }
}

template <int NT>
__global__ void __launch_bounds__(kFfnThreads, 1) decode_ffn_kernel(FfnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int d = a.d, f = a.f, T = a.T, K = a.k;
  const int RG = f / 32;             // gate/up row blocks == down groups
  const int KC = d / (32 * kGuGroups);
  const int RD = d / 32;
  const int DG = f / 32;
  const int nks = d / 16;
  const int slot_bytes = ffn_slot_bytes(f);
  uint2* xfrag = reinterpret_cast<uint2*>(smem);
  uint8_t* ring = smem + (size_t)NT * d * 16;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)kNumSlots * slot_bytes);
  uint64_t* empty = full + kNumSlots;
  __shared__ long long s_lo, s_hi, s_ngu;
  __shared__ int s_nexp, s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < kNumSlots; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init_fence();
  }
  // x fragments (B operand of the gate/up products), fp16, zero past T
  for (int i = tid; i < NT * nks * 32; i += kFfnThreads) {
    const int ln = i & 31, kstep = (i >> 5) % nks, nt = (i >> 5) / nks;
    const int n = nt * 8 + (ln >> 2), k = kstep * 16 + 2 * (ln & 3);
    uint2 v = make_uint2(0u, 0u);
    if (n < T) {
      const uint16_t* xr = a.x + (size_t)n * d + k;
      v.x = pack_half2_from_bf16(xr[0], xr[1]);
      v.y = pack_half2_from_bf16(xr[8], xr[9]);
    }
    xfrag[i] = v;
  }
  pdl_wait();   // the routing plan is complete and visible
  if (tid == 0) {
    const int n_exp = a.plan->n_act + 1;
    const long long n_gu = (long long)n_exp * RG * KC;
    const long long n_dn = (long long)n_exp * RD;
    const long long W = n_gu * 2 * kGuGroups + n_dn * DG;
    auto unit_at = [&](long long target) -> long long {
      if (target <= 0) return 0;
      if (target <= n_gu * 2 * kGuGroups) return (target + 2 * kGuGroups - 1) / (2 * kGuGroups);
      return n_gu + (target - n_gu * 2 * kGuGroups + DG - 1) / DG;
    };
    s_lo = unit_at(W * blockIdx.x / gridDim.x);
    s_hi = (blockIdx.x + 1 == gridDim.x) ? n_gu + n_dn : unit_at(W * (blockIdx.x + 1) / gridDim.x);
    s_ngu = n_gu;
    s_nexp = n_exp;
  }
  __syncthreads();
  const long long lo = s_lo, n_units = s_hi - s_lo, n_gu = s_ngu;
  const int n_exp = s_nexp;
  const Plan* P = a.plan;

  auto expert_base = [&](int ai) -> const uint8_t* {
    return ai == 0 ? a.shared_expert : a.slots + (int64_t)P->act_slot[ai - 1] * a.expert_bytes;
  };

  if (warp == kConsumerWarps) {
    // ---------------- producer: one thread streams units into the ring ----
    if (lane == 0) {
      for (long long j = 0; j < n_units; ++j) {
        const int s = (int)(j % kNumSlots);
        const long long n = j / kNumSlots;
        if (n > 0 && !mbar_wait(&empty[s], (uint32_t)((n - 1) & 1))) {
          set_error(a.err, DEV_TIMEOUT_BARRIER);
          break;
        }
        const long long u = lo + j;
        const uint8_t* src;
        uint32_t bytes;
        if (u < n_gu) {
          const int ai = (int)(u / (RG * KC)), rb = (int)((u / KC) % RG), kc = (int)(u % KC);
          src = expert_base(ai) + gu_block_offset(rb, kc * kGuGroups, 0, d);
          bytes = 2 * kGuGroups * kBlockBytes;
        } else {
          const long long v = u - n_gu;
          const int ai = (int)(v / RD), rbd = (int)(v % RD);
          src = expert_base(ai) + down_block_offset(rbd, 0, d, f);
          bytes = DG * kBlockBytes;
        }
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_g2s(ring + (size_t)s * slot_bytes, src, bytes, &full[s]);
      }
    }
  } else {
    // ---------------- consumers ---------------------------------------------
    for (long long j = warp; j < n_units; j += kConsumerWarps) {
      const int s = (int)(j % kNumSlots);
      const long long n = j / kNumSlots;
      const uint8_t* sp = ring + (size_t)s * slot_bytes;
      const bool ok = mbar_wait(&full[s], (uint32_t)(n & 1));
      if (!ok) set_error(a.err, DEV_TIMEOUT_BARRIER);
      const long long u = lo + j;
      if (u < n_gu) {
        const int ai = (int)(u / (RG * KC)), rb = (int)((u / KC) % RG), kc = (int)(u % KC);
        float ag[NT][2][4], au[NT][2][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) ag[nt][mt][i] = au[nt][mt][i] = 0.f;
        if (ok) {
          for (int g8 = 0; g8 < kGuGroups; ++g8) {
            const int gi = kc * kGuGroups + g8;
            uint2 bx[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              bx[nt][0] = xfrag[((size_t)nt * nks + gi * 2 + 0) * 32 + lane];
              bx[nt][1] = xfrag[((size_t)nt * nks + gi * 2 + 1) * 32 + lane];
            }
            block_mma<NT>(sp + (2 * g8 + 0) * kBlockBytes, lane, bx, ag);
            block_mma<NT>(sp + (2 * g8 + 1) * kBlockBytes, lane, bx, au);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        // partial g/u of this unit
        const size_t pbase = (((size_t)(ai * RG + rb) * KC + kc) * NT) * 512;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float4* pp = reinterpret_cast<float4*>(a.gu_partial + pbase + (size_t)nt * 512 + lane * 16);
          pp[0] = make_float4(ag[nt][0][0], ag[nt][0][1], ag[nt][0][2], ag[nt][0][3]);
          pp[1] = make_float4(ag[nt][1][0], ag[nt][1][1], ag[nt][1][2], ag[nt][1][3]);
          pp[2] = make_float4(au[nt][0][0], au[nt][0][1], au[nt][0][2], au[nt][0][3]);
          pp[3] = make_float4(au[nt][1][0], au[nt][1][1], au[nt][1][2], au[nt][1][3]);
        }
        __syncwarp();
        uint32_t old = 0;
        if (lane == 0) {
          __threadfence();
          old = atomicAdd(&a.gu_cnt[ai * RG + rb], 1u);
        }
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old == (uint32_t)(KC - 1)) {
          __threadfence();
          float g[NT][8], uu[NT][8];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 8; ++i) g[nt][i] = uu[nt][i] = 0.f;
          for (int kc2 = 0; kc2 < KC; ++kc2) {
            const size_t b2 = (((size_t)(ai * RG + rb) * KC + kc2) * NT) * 512;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const float* pp = a.gu_partial + b2 + (size_t)nt * 512 + lane * 16;
              const float4 q0 = ld_cg_f4(pp), q1 = ld_cg_f4(pp + 4), q2 = ld_cg_f4(pp + 8),
                           q3 = ld_cg_f4(pp + 12);
              g[nt][0] += q0.x; g[nt][1] += q0.y; g[nt][2] += q0.z; g[nt][3] += q0.w;
              g[nt][4] += q1.x; g[nt][5] += q1.y; g[nt][6] += q1.z; g[nt][7] += q1.w;
              uu[nt][0] += q2.x; uu[nt][1] += q2.y; uu[nt][2] += q2.z; uu[nt][3] += q2.w;
              uu[nt][4] += q3.x; uu[nt][5] += q3.y; uu[nt][6] += q3.z; uu[nt][7] += q3.w;
            }
          }
          const int gq = lane >> 2, cq = lane & 3;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e8 = 0; e8 < 8; ++e8) {
              const int mt = e8 >> 2, i = e8 & 3;
              const float gv = g[nt][e8];
              const float hv = gv / (1.f + expf(-gv)) * uu[nt][e8];
              const int tok = nt * 8 + 2 * cq + (i & 1);
              const int kk = mt * 16 + gq + 8 * (i >> 1);       // row within the f block
              const int ksd = kk >> 4, kk16 = kk & 15;
              const int reg = kk16 >> 3, cp = (kk16 & 7) >> 1, half = kk16 & 1;
              const int ln2 = (tok & 7) * 4 + cp;
              const size_t hidx =
                  ((((size_t)(ai * NT + nt) * RG + rb) * 2 + ksd) * 32 + ln2) * 4 + reg * 2 + half;
              a.hfrag[hidx] = __half_as_ushort(__float2half_rn(hv));
            }
          }
          __syncwarp();
          if (lane == 0) {
            __threadfence();
            red_release_add(&a.h_ready[ai], 1u);
          }
        }
      } else {
        const long long v = u - n_gu;
        const int ai = (int)(v / RD), rbd = (int)(v % RD);
        bool hok = ok && wait_flag_geq(&a.h_ready[ai], (uint32_t)RG);
        if (ok && !hok) set_error(a.err, DEV_TIMEOUT_FLAG);
        float acc[NT][2][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[nt][mt][i] = 0.f;
        if (hok) {
          for (int gi = 0; gi < DG; ++gi) {
            uint2 bx[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
              for (int ks = 0; ks < 2; ++ks) {
                const size_t hidx = ((((size_t)(ai * NT + nt) * RG + gi) * 2 + ks) * 32 + lane) * 4;
                bx[nt][ks] = ld_cg_u2(a.hfrag + hidx);
              }
            }
            block_mma<NT>(sp + gi * kBlockBytes, lane, bx, acc);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        const int gq = lane >> 2, cq = lane & 3;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int tok = nt * 8 + 2 * cq + (i & 1);
              if (tok < T) {
                const int row = rbd * 32 + mt * 16 + gq + 8 * (i >> 1);
                a.obuf[((size_t)ai * T + tok) * d + row] = acc[nt][mt][i];
              }
            }
        __syncwarp();
        uint32_t old = 0;
        if (lane == 0) {
          __threadfence();
          old = atomicAdd(&a.d_cnt[rbd], 1u);
        }
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old == (uint32_t)(n_exp - 1)) {
          __threadfence();
          const int row = rbd * 32 + lane;
          for (int t = 0; t < T; ++t) {
            float yv = a.shared_weight * ld_cg_f32(a.obuf + (size_t)t * d + row);
            for (int i = 0; i < K; ++i) {
              const int ap = 1 + P->pick_act[t * K + i];
              yv = fmaf(P->w[t * K + i], ld_cg_f32(a.obuf + ((size_t)ap * T + t) * d + row), yv);
            }
            a.y[(size_t)t * d + row] = yv;
          }
        }
      }
    }
  }

  // ---- the last CTA to finish clears the per-call counters ---------------
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = (atomicAdd(a.done, 1u) == gridDim.x - 1);
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    for (int i = tid; i < n_exp * RG; i += kFfnThreads) a.gu_cnt[i] = 0;
    for (int i = tid; i < n_exp; i += kFfnThreads) a.h_ready[i] = 0;
    for (int i = tid; i < RD; i += kFfnThreads) a.d_cnt[i] = 0;
    if (tid == 0) *a.done = 0;
  }
}

template <int NT>
static cudaError_t launch_nt(const FfnArgs& a, cudaStream_t s, bool pdl, int grid) {
  const size_t smem = ffn_smem_bytes(NT, a.d, a.f);
  // raise the dynamic shared-memory limit once per size (not during stream capture)
  static size_t configured = 0;
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_ffn_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kFfnThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, decode_ffn_kernel<NT>, a);
}

cudaError_t launch_decode_ffn(const FfnArgs& a, cudaStream_t s, bool pdl, int num_sms) {
  const int grid = a.grid > 0 ? a.grid : num_sms;
  if (a.T <= 8) return launch_nt<1>(a, s, pdl, grid);
  return launch_nt<2>(a, s, pdl, grid);
}

}  // namespace moe
