// Decode / verify expert FFN (T <= 16 tokens): every distinct routed expert
// and the shared expert run once for all tokens routed to them (a verify
// batch shares one fetch of each expert, page "单卡5090跑125B 大模型", §2.3),
//   g = Wg.x, u = Wu.x, h = silu(g) * u, o = Wd.h,
//   y[t] = shared_weight * o_shared[t] + sum_i w[t,i] * o_idx[t,i][t].
//
// Work is cut into units that stream contiguous bytes of the device layout:
//   gate/up unit (expert a, 32-row block rb of f, 8 of the d/32 groups): the
//     Wg and Wu blocks of those groups (16 x 448 B); its partial g/u sums go to
//     scratch and the last of the d/256 units of (a, rb) finishes g, u, writes
//     h = silu(g) * u (fp16, [expert][token][f]) and bumps h_ready[a];
//   down unit (expert a, 32-row block rb of d): f/32 Wd blocks; multiplies by
//     h_a, writes o_a for its rows, and the last expert to finish a row block
//     combines y for those rows in a fixed order (shared expert, then routed
//     experts in ascending id).
// One persistent CTA per SM takes a contiguous, byte-balanced range of units.
// Warp roles: 12 consumer warps; one producer thread streaming each unit into
// a shared-memory ring with bulk copies (mbarrier completion); one h-loader
// thread that, for each expert of the CTA's down units, waits (bounded) for
// its h and bulk-copies it into a padded shared-memory slot once.  Consumers
// expand the 3-bit codes to fp16 in registers and multiply on the tensor
// cores (mma.sync m16n8k16, fp32 accumulate, per-group scale in fp32).
#include "common.cuh"
#include "internal.h"

namespace moe {

#ifdef MOE_TIMELINE
__device__ unsigned long long g_ffn_timeline[512][16];
#endif

constexpr int kGuGroups = 8;     // groups per gate/up unit
constexpr int kHSlots = 2;       // h buffers per CTA

// One consumer warp per ring slot: slot s is always consumed by warp s, so a
// warp never waits on a slot phase more than one ahead of the slot's state
// (an mbarrier parity wait cannot tell phase n from phase n-2).
template <int NT>
struct FfnCfg {
  static constexpr int kSlots = NT == 1 ? 12 : 10;
  static constexpr int kConsumers = kSlots;
  static constexpr int kThreads = (kConsumers + 2) * 32;   // + producer warp + h-loader warp
};

__host__ __device__ __forceinline__ int ffn_slot_bytes(int f) {
  const int dg = f / 32;
  return (dg > 2 * kGuGroups ? dg : 2 * kGuGroups) * kBlockBytes;
}

// one padded h row: f fp16 values + 8 (keeps the 8 token rows on distinct banks)
__host__ __device__ __forceinline__ int h_row_bytes(int f) { return (f + 8) * 2; }

template <int NT>
__host__ __device__ __forceinline__ size_t ffn_smem_bytes(int d, int f) {
  return (size_t)NT * d * 16 + (size_t)FfnCfg<NT>::kSlots * ffn_slot_bytes(f) +
         (size_t)kHSlots * NT * 8 * h_row_bytes(f) + (2 * FfnCfg<NT>::kSlots + 2 * kHSlots) * 8 + 64;
}

__device__ __forceinline__ uint32_t pack_half2_from_bf16(uint32_t two_bf16) {
  const __half2 h = __floats2half2_rn(bf16_bits_to_float(two_bf16 & 0xffffu), bf16_bits_to_float(two_bf16 >> 16));
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
__global__ void __launch_bounds__(FfnCfg<NT>::kThreads, 1) decode_ffn_kernel(FfnArgs a) {
  constexpr int NS = FfnCfg<NT>::kSlots;
  constexpr int kConsumerWarps = FfnCfg<NT>::kConsumers;
  constexpr int kFfnThreads = FfnCfg<NT>::kThreads;
  extern __shared__ __align__(128) uint8_t smem[];
  const int d = a.d, f = a.f, T = a.T, K = a.k;
  const int RG = f / 32;             // gate/up row blocks == down groups
  const int KC = d / (32 * kGuGroups);
  const int RD = d / 32;
  const int DG = f / 32;
  const int nks = d / 16;
  const int slot_bytes = ffn_slot_bytes(f);
  const int hrow = h_row_bytes(f);
  uint2* xfrag = reinterpret_cast<uint2*>(smem);
  uint8_t* ring = smem + (size_t)NT * d * 16;
  uint8_t* hbuf = ring + (size_t)NS * slot_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(hbuf + (size_t)kHSlots * NT * 8 * hrow);
  uint64_t* empty = full + NS;
  uint64_t* hfull = empty + NS;
  uint64_t* hempty = hfull + kHSlots;
  __shared__ long long s_lo, s_hi, s_ngu;
  __shared__ int s_nexp, s_last;
  __shared__ int s_huses[kHSlots];
  __shared__ volatile int s_hexp[kHSlots];   // expert whose h a slot holds or is loading

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) MOE_TL(g_ffn_timeline, blockIdx.x, 0);
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < kHSlots; ++i) {
      mbar_init(&hfull[i], 1);
      mbar_init(&hempty[i], 1);
      s_huses[i] = 0;
      s_hexp[i] = -1;
    }
    mbar_init_fence();
  }
  // x fragments (B operand of the gate/up products), fp16, zero past T.
  // Entry (nt, kstep, lane) holds tokens nt*8 + lane/4, inputs
  // kstep*16 + 2*(lane%4) + {0, 1} (reg 0) and + {8, 9} (reg 1).
  {
    uint32_t* xf = reinterpret_cast<uint32_t*>(xfrag);
    const int cpr = d / 8;                       // 8-value chunks per token row
    for (int i = tid; i < NT * 8 * cpr; i += kFfnThreads) {
      const int n = i / cpr, k8 = (i % cpr) * 8;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (n < T) v = __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)n * d + k8));
      const int nt = n >> 3, kstep = k8 >> 4, reg = (k8 >> 3) & 1;
      const uint32_t in[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int ln = (n & 7) * 4 + q;
        xf[(((size_t)nt * nks + kstep) * 32 + ln) * 2 + reg] = pack_half2_from_bf16(in[q]);
      }
    }
  }
  if (tid == 0) MOE_TL(g_ffn_timeline, blockIdx.x, 1);
  pdl_wait();   // the routing plan is complete and visible
  if (tid == 0) MOE_TL(g_ffn_timeline, blockIdx.x, 2);
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
  if (tid == 0) MOE_TL(g_ffn_timeline, blockIdx.x, 3);
  const long long lo = s_lo, hi = s_hi, n_units = s_hi - s_lo, n_gu = s_ngu;
  const int n_exp = s_nexp;
  const Plan* P = a.plan;
  // down units of this CTA: [dlo, dhi) in down-unit numbering; experts a0..a1
  const long long dlo = (lo > n_gu ? lo : n_gu) - n_gu, dhi = (hi > n_gu ? hi : n_gu) - n_gu;
  const int a0 = (int)(dlo / RD);
  const int a1 = dhi > dlo ? (int)((dhi - 1) / RD) : a0 - 1;
  auto units_of = [&](int ai) -> int {   // down units of expert ai in this CTA
    const long long b = (long long)ai * RD, e = b + RD;
    return (int)((e < dhi ? e : dhi) - (b > dlo ? b : dlo));
  };

  auto expert_base = [&](int ai) -> const uint8_t* {
    return ai == 0 ? a.shared_expert : a.slots + (int64_t)P->act_slot[ai - 1] * a.expert_bytes;
  };

  if (warp == kConsumerWarps) {
    // ---------------- producer: one thread streams units into the ring ----
    if (lane == 0) {
      for (long long j = 0; j < n_units; ++j) {
        const int s = (int)(j % NS);
        const long long n = j / NS;
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
        if (j == 0) MOE_TL(g_ffn_timeline, blockIdx.x, 4);
      }
      MOE_TL(g_ffn_timeline, blockIdx.x, 5);
    }
  } else if (warp == kConsumerWarps + 1) {
    // ---------------- h loader: one bulk copy of h_a per expert -------------
    if (lane == 0) {
      for (int ai = a0, i = 0; ai <= a1; ++ai, ++i) {
        const int hs = i % kHSlots;
        const int use = i / kHSlots;
        if (use > 0 && !mbar_wait(&hempty[hs], (uint32_t)((use - 1) & 1))) {
          set_error(a.err, DEV_TIMEOUT_BARRIER);
          break;
        }
        if (!wait_flag_geq(&a.h_ready[ai], (uint32_t)RG)) {
          set_error(a.err, DEV_TIMEOUT_FLAG);
          break;
        }
        if (i == 0) MOE_TL(g_ffn_timeline, blockIdx.x, 8);
        // h was written through the generic proxy by other CTAs; order it
        // before the bulk copy (async proxy) reads it
        asm volatile("fence.proxy.async.global;" ::: "memory");
        uint8_t* dst = hbuf + (size_t)hs * NT * 8 * hrow;
        s_hexp[hs] = ai;   // the previous use of this slot has been released
        mbar_arrive_expect_tx(&hfull[hs], (uint32_t)(T * f * 2));
        for (int t = 0; t < T; ++t)
          bulk_g2s(dst + (size_t)t * hrow, a.hbuf + ((size_t)ai * T + t) * f, (uint32_t)(f * 2), &hfull[hs]);
      }
    }
  } else {
    // ---------------- consumers ---------------------------------------------
    const int gq = lane >> 2, cq = lane & 3;
    for (long long j = warp; j < n_units; j += kConsumerWarps) {
      const int s = (int)(j % NS);
      const long long n = j / NS;
      const uint8_t* sp = ring + (size_t)s * slot_bytes;
      const bool ok = mbar_wait(&full[s], (uint32_t)(n & 1));
      if (!ok) set_error(a.err, DEV_TIMEOUT_BARRIER);
      if (warp == 0 && lane == 0 && j == 0) MOE_TL(g_ffn_timeline, blockIdx.x, 6);
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
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e8 = 0; e8 < 8; ++e8) {
              const int mt = e8 >> 2, i = e8 & 3;
              const int tok = nt * 8 + 2 * cq + (i & 1);
              if (tok < T) {
                const float gv = g[nt][e8];
                const float hv = gv / (1.f + expf(-gv)) * uu[nt][e8];
                const int row = rb * 32 + mt * 16 + gq + 8 * (i >> 1);
                a.hbuf[((size_t)ai * T + tok) * f + row] = __half_as_ushort(__float2half_rn(hv));
              }
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
        const int hi_idx = ai - a0;
        const int hs = hi_idx % kHSlots;
        // wait until the loader has moved this slot on to expert ai, then for its data
        bool hok = ok;
        if (hok && s_hexp[hs] != ai) {
          const uint64_t t0 = globaltimer();
          while (s_hexp[hs] != ai) {
            if (globaltimer() - t0 > kWaitLimitNs) {
              hok = false;
              break;
            }
          }
        }
        hok = hok && mbar_wait(&hfull[hs], (uint32_t)((hi_idx / kHSlots) & 1));
        if (ok && !hok) set_error(a.err, DEV_TIMEOUT_BARRIER);
        float acc[NT][2][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[nt][mt][i] = 0.f;
        if (hok) {
          const uint8_t* hb = hbuf + (size_t)hs * NT * 8 * hrow;
          for (int gi = 0; gi < DG; ++gi) {
            uint2 bx[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const int tok = nt * 8 + gq;
              const uint8_t* hr = hb + (size_t)tok * hrow + (gi * 32 + 2 * cq) * 2;
#pragma unroll
              for (int ks = 0; ks < 2; ++ks) {
                if (tok < T) {
                  bx[nt][ks].x = *reinterpret_cast<const uint32_t*>(hr + ks * 32);
                  bx[nt][ks].y = *reinterpret_cast<const uint32_t*>(hr + ks * 32 + 16);
                } else {
                  bx[nt][ks] = make_uint2(0u, 0u);
                }
              }
            }
            block_mma<NT>(sp + gi * kBlockBytes, lane, bx, acc);
          }
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&empty[s]);
          if (hok && atomicAdd(&s_huses[hs], 1) + 1 == units_of(ai)) {
            s_huses[hs] = 0;
            mbar_arrive(&hempty[hs]);
          }
        }
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
  if (lane == 0 && warp < kConsumerWarps) MOE_TL(g_ffn_timeline, blockIdx.x, 9 + (warp & 1));
  __syncthreads();
  if (tid == 0) MOE_TL(g_ffn_timeline, blockIdx.x, 11);
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
    if (tid == 0) MOE_TL(g_ffn_timeline, blockIdx.x, 12);
  }
}

template <int NT>
static cudaError_t launch_nt(const FfnArgs& a, cudaStream_t s, bool pdl, int grid) {
  const size_t smem = ffn_smem_bytes<NT>(a.d, a.f);
  constexpr int kFfnThreads = FfnCfg<NT>::kThreads;
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

#ifdef MOE_TIMELINE
extern "C" int moe_debug_timeline_ffn(unsigned long long* out) {
  return (int)cudaMemcpyFromSymbol(out, g_ffn_timeline, sizeof(g_ffn_timeline));
}
#endif

cudaError_t launch_decode_ffn(const FfnArgs& a, cudaStream_t s, bool pdl, int num_sms) {
  const int grid = a.grid > 0 ? a.grid : num_sms;
  if (a.T <= 8) return launch_nt<1>(a, s, pdl, grid);
  return launch_nt<2>(a, s, pdl, grid);
}

}  // namespace moe
