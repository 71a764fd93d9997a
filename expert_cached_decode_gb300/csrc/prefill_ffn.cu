// Prefill expert FFN (T up to 16,384 tokens): grouped GEMMs on tcgen05.
//
// The chunk's token picks are counting-sorted by expert (the shared expert
// takes every token, as the last group), the activations gathered to fp16 in
// that order, and two grouped GEMMs run every expert once for all its tokens
// (a 12,288-token chunk is the pages' single-GPU prefill size, page
// "一张 RTX 4090 跑千亿模型", §加个草稿层):
//   gate/up:  [g|u]^T[f x n_e] = [Wg|Wu][f x d] . X_e^T   -> h = silu(g)*u (fp16)
//   down:     o^T[d x n_e] = Wd[d x f] . H_e^T            -> w[t,e] * o[t]
// The down GEMM writes the shared expert's weighted output straight into y
// and each routed pick's into its own row of a per-pick buffer; a combine
// kernel then adds, per token, its picks in ascending expert id (the decode
// path's order), so y is the same whatever order tiles and the counting sort
// ran in.
// h is carried as an fp16 pair (hi = RN(h), lo = RN(h - hi)) and the down
// GEMM accumulates Wd.hi + Wd.lo, so h keeps ~22 bits; the fp16 weight
// RN(q * scale) is the only rounding of an operand.
// Weights sit on the MMA M side (128 rows per tile: 64 rows of Wg over the
// same 64 rows of Wu for gate/up, 128 rows of Wd for down), tokens on N
// (<= 256 per tile, rounded up to 16).  Eight producer warps expand the
// 3-bit blocks of the slot to fp16 RN(q * scale) straight into the
// 128-byte-swizzled K-major operand tile; the token tile comes by TMA; one
// thread issues tcgen05.mma into a double-buffered tensor-memory accumulator;
// four epilogue warps read it back while the next tile accumulates.
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace moe {

// ------------------------------------------------------------------ plan ---
// One CTA: expert offsets, scatter cursors, tile lists, slot lookup, stamps.
__global__ void __launch_bounds__(1024) prefill_plan_kernel(PrefillPlanArgs a) {
  __shared__ int s_off[kMaxE + 2];
  __shared__ int s_nt[kMaxE + 2];
  __shared__ int s_warp[32];
  __shared__ int s_total[2];
  const int E = a.E, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_groups = E + 1;   // routed experts, then the shared expert
  // exclusive scan of counts and of n-tiles (n_groups <= 1025 -> two rounds)
  for (int pass = 0; pass < 2; ++pass) {
    int carry = 0;
    for (int base = 0; base < n_groups; base += 1024) {
      const int g = base + tid;
      int n = 0;
      if (g < n_groups) n = (g < E) ? a.counts[g] : a.T;
      int v = pass == 0 ? n : (n + kPrefillBN - 1) / kPrefillBN;
      int inc = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
      }
      if (lane == 31) s_warp[warp] = inc;
      __syncthreads();
      if (warp == 0) {
        const int wv = s_warp[lane];
        int wi = wv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, wi, o);
          if (lane >= o) wi += t;
        }
        s_warp[lane] = wi - wv;
        if (lane == 31) s_total[pass] = wi;
      }
      __syncthreads();
      if (g < n_groups) {
        const int ex = carry + s_warp[warp] + inc - v;
        if (pass == 0) s_off[g] = ex; else s_nt[g] = ex;
      }
      carry += s_total[pass];
      __syncthreads();
    }
    if (tid == 0) {
      if (pass == 0) s_off[n_groups] = carry; else s_nt[n_groups] = carry;
    }
    __syncthreads();
  }
  const int n_ntiles = s_nt[n_groups];
  const int MG = a.f / 64, MD = a.d / 128;   // gate/up tiles cover 64 f rows (Wg and Wu)
  int act = 0;
  for (int g = tid; g < n_groups; g += 1024) {
    const int off = s_off[g];
    const int n = s_off[g + 1] - off;
    if (g < E) a.cursor[g] = off;
    int slot = -1;
    if (g < E && n > 0) {
      ++act;
      slot = a.table[(size_t)a.layer * E + g];
      if (slot < 0) set_error(a.err, DEV_NOT_RESIDENT);
      else if (a.account) a.stamp[slot] = *a.clock;
    }
    a.group_slot[g] = slot;
  }
  // tile lists: thread i writes the tiles of token tiles i, i + 1024, ...;
  // the group of token tile nt is the last g with s_nt[g] <= nt (an empty
  // group shares its s_nt with the next group, so the last match is the
  // non-empty one)
  for (int nt = tid; nt < n_ntiles; nt += 1024) {
    int lo = 0, hi = n_groups - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_nt[mid] <= nt) lo = mid; else hi = mid - 1;
    }
    const int g = lo, j = nt - s_nt[g];
    const int off = s_off[g], n = s_off[g + 1] - off;
    PrefillTile tl;
    tl.group = g;
    tl.row0 = off + j * kPrefillBN;
    tl.nlen = min(kPrefillBN, n - j * kPrefillBN);
    for (int m = 0; m < MG; ++m) {
      tl.m = m;
      a.tiles_gu[nt * MG + m] = tl;
    }
    for (int m = 0; m < MD; ++m) {
      tl.m = m;
      a.tiles_dn[nt * MD + m] = tl;
    }
  }
  // distinct routed experts of the chunk
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) act += __shfl_xor_sync(0xffffffffu, act, o);
  if (lane == 0) s_warp[warp] = act;
  __syncthreads();
  if (tid == 0) {
    int n_act = 0;
    for (int w = 0; w < 32; ++w) n_act += s_warp[w];
    a.n_tiles[0] = n_ntiles * MG;
    a.n_tiles[1] = n_ntiles * MD;
    if (a.account) {
      a.stats[ST_CALLS] += 1;
      a.stats[ST_TOK_HIT] += (int64_t)a.T * a.k;
      a.stats[ST_DIST_HIT] += n_act;
      *a.clock += 1;
    }
  }
}

__global__ void prefill_scatter_kernel(PrefillScatterArgs a) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const int picks = a.T * a.k;
  if (i < picks) {
    const int e = a.idx[i];
    const int pos = atomicAdd(&a.cursor[e], 1);
    a.perm[pos] = i / a.k;
    a.wsort[pos] = a.w[i];
    a.pick[pos] = i;
  } else if (i < picks + a.T) {
    const int t = i - picks;
    a.perm[picks + t] = t;
    a.wsort[picks + t] = a.shared_weight;
  }
}

// Xg[r] = fp16(x[perm[r]]): one warp per row at a time, 256 16-byte chunks
// of the row (8 per lane) loaded before they are converted and stored
__global__ void __launch_bounds__(256) prefill_gather_kernel(const uint16_t* x, const int32_t* perm, uint16_t* xg,
                                                             int rows, int d) {
  const int lane = threadIdx.x & 31;
  const int nw = gridDim.x * (blockDim.x >> 5);
  const int cpr = d / 8;   // 16-byte chunks per row
  for (int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += nw) {
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)perm[r] * d);
    uint4* dst = reinterpret_cast<uint4*>(xg + (size_t)r * d);
    for (int c0 = 0; c0 < cpr; c0 += 256) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (c0 + lane + 32 * u < cpr) v[u] = __ldg(src + c0 + lane + 32 * u);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (c0 + lane + 32 * u < cpr) {
          const uint32_t in[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
          uint32_t out[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const __half2 h =
                __floats2half2_rn(bf16_bits_to_float(in[q] & 0xffffu), bf16_bits_to_float(in[q] >> 16));
            out[q] = *reinterpret_cast<const uint32_t*>(&h);
          }
          dst[c0 + lane + 32 * u] = make_uint4(out[0], out[1], out[2], out[3]);
        }
      }
    }
  }
}

// ---------------------------------------------------------- grouped GEMMs ---
// Optional per-CTA wait profile (build with -DMOE_TIMELINE): clock64 cycles
// each role spent waiting or working, read back by moe_debug_prefill_profile.
// Per-k-block amounts gather in registers (PF_ACC) and are stored once
// (PF_PUT), so the profile does not add global round trips to the loops.
#ifdef MOE_TIMELINE
__device__ unsigned long long g_prefill_prof[2][256][16];
#define PF_T0() const long long pf_t0 = clock64()
#define PF_ADD(kind, field) (g_prefill_prof[(kind)][blockIdx.x][(field)] += (unsigned long long)(clock64() - pf_t0))
#define PF_VAR(v) long long v = 0
#define PF_ACC(v) (v += clock64() - pf_t0)
#define PF_PUT(kind, field, v) (g_prefill_prof[(kind)][blockIdx.x][(field)] += (unsigned long long)(v))
#else
#define PF_T0() ((void)0)
#define PF_ADD(kind, field) ((void)0)
#define PF_VAR(v) ((void)0)
#define PF_ACC(v) ((void)0)
#define PF_PUT(kind, field, v) ((void)0)
#endif

namespace pg {
constexpr int BM = 128, BN = kPrefillBN, BK = 64;
constexpr int A_BYTES = BM * BK * 2;   // 16 KB weight tile
constexpr int B_BYTES = BN * BK * 2;   // 32 KB token tile
constexpr int NGROUP = 2;              // producer groups: group q takes the k blocks kb % NGROUP == q
constexpr int NPROD = 4 * NGROUP;      // dequant warps (4 per group, 2 blocks of each k block each)
constexpr int PSTAGES = 4;             // packed-weight staging depth per producer
constexpr int PCHUNK = 2 * kBlockBytes;   // packed bytes per producer and k block
constexpr int EPI0 = 2 + NPROD;        // first epilogue warp
constexpr int NEPI = 8;                // epilogue warps: 4 TMEM quarters x 2 column halves
constexpr int THREADS = (EPI0 + NEPI) * 32;   // 0 TMA, 1 MMA, then producers, then epilogue
constexpr int GU_ROWS = BM / 2;        // f rows per gate/up tile (Wg rows, then the same Wu rows)
constexpr int MAX_CTA_TILES = 128;     // tile descriptors of a CTA kept in shared memory
constexpr int CLUSTER = 2;             // CTAs sharing each token tile (TMA multicast)
constexpr int B_HALF = B_BYTES / CLUSTER;   // token rows a CTA loads for both
}  // namespace pg

// One 32x32 block (448 B at `bp`, shared memory) expanded to RN(q * scale)
// fp16 pairs in mma A-fragment order: register (mt, ks, rh, rl) holds, for
// lane (g, c), rows mt*16 + 8rl + g and k pair 16ks + 8rh + 2c.  The
// multiplies are volatile so that the whole expansion stays where it is
// written: producers expand before they wait for a free tile stage.
__device__ __forceinline__ void expand_block(const uint8_t* bp, int lane, uint32_t (&v)[16]) {
  const uint32_t* wp = reinterpret_cast<const uint32_t*>(bp);
  const uint32_t w0 = wp[lane], w1 = wp[32 + lane], w2 = wp[64 + lane];
  const uint2 sc = *reinterpret_cast<const uint2*>(bp + kBlockCodeBytes + (lane >> 2) * 8);
  // scale of rows g, g+8, g+16, g+24, duplicated into both halves
  const uint32_t s2[4] = {__byte_perm(sc.x, 0, 0x1010), __byte_perm(sc.x, 0, 0x3232), __byte_perm(sc.y, 0, 0x1010),
                          __byte_perm(sc.y, 0, 0x3232)};
  uint32_t A[16];
  dequant_block(w0, w1, w2, A);
#pragma unroll
  for (int i = 0; i < 16; ++i)
    asm volatile("mul.rn.f16x2 %0, %1, %2;" : "=r"(v[i]) : "r"(A[i]), "r"(s2[2 * (i >> 3) + (i & 1)]));
}

// An expanded block written as 32 rows and 32 k columns of a
// 128-byte-swizzled K-major fp16 tile.  The A-fragment order is the order
// stmatrix takes, so one m8n8.x4 store per (mt, ks) writes four 8x8
// sub-tiles; lane L gives the address of row L%8 of sub-tile L/8
// (rl = (L/8)%2, rh = L/16).  `lane_base` = tile + (row offset of the block
// + 8*((L/8)%2) + L%8) * 128; sw = (L%8) << 4 (the swizzle of that row);
// KC = the first 16-byte chunk of the block's k columns (0 or 4).
template <int KC>
__device__ __forceinline__ void store_block_tile(const uint32_t (&v)[16], int lane, uint32_t lane_base, uint32_t sw) {
  const uint32_t rh = (uint32_t)(lane >> 4);
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      const int r0 = mt * 8 + ks * 4;
      const uint32_t addr = lane_base + (uint32_t)(mt * 2048) + ((((uint32_t)(KC + 2 * ks) + rh) << 4) ^ sw);
      asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[r0]),
                   "r"(v[r0 + 1]), "r"(v[r0 + 2]), "r"(v[r0 + 3])
                   : "memory");
    }
  }
}

// DOWN = false: gate/up tiles.  The 128-row weight tile holds 64 rows of Wg
// (M rows 0-63) and the same 64 rows of Wu (M rows 64-127), so one
// accumulator of 256 columns carries g and u side by side in tensor-memory
// lanes, and two accumulators (double buffer) fit the 512 columns; the SwiGLU
// epilogue writes Hg.  DOWN = true: 128 rows of Wd, weighted atomic combine
// into y.  Producer warp p expands, for every k block of parity p/4, two
// blocks that are contiguous in the slot (gate/up: the Wg and Wu blocks of
// row block 2m + p%2, input group 2kb + (p/2)%2; down: row blocks
// 4m + 2((p/2)%2) and the next one of input group 2kb + p%2; see psrc).
template <bool DOWN>
__global__ void __launch_bounds__(pg::THREADS, 1)
    prefill_gemm_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmB2,
                        PrefillGemmArgs a) {
  using namespace pg;
  constexpr int NB = DOWN ? 2 : 1;             // token tiles per stage (down: h hi and lo)
  constexpr int STAGES = DOWN ? 2 : 3;
  constexpr int STAGE_BYTES = A_BYTES + NB * B_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  constexpr int EPI_BYTES = DOWN ? 0 : 4 * 2 * 16 * 32 * 4;   // u exchange slots
  uint8_t* epi = smem + STAGES * STAGE_BYTES;
  uint8_t* pstage = epi + EPI_BYTES;                               // NPROD * PSTAGES * PCHUNK
  uint64_t* bars = reinterpret_cast<uint64_t*>(pstage + NPROD * PSTAGES * PCHUNK);
  uint64_t* full_a = bars;
  uint64_t* full_b = full_a + STAGES;
  uint64_t* empty = full_b + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* pbar = tempty + 2;                                     // NPROD * PSTAGES
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pbar + NPROD * PSTAGES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = a.n_tiles[DOWN ? 1 : 0];
  const int K = DOWN ? a.f : a.d;
  const int n_kb = K / BK;   // even (K is a multiple of 128)
  const PrefillTile* tiles = DOWN ? a.tiles_dn : a.tiles_gu;
  // this CTA's tiles are blockIdx.x + lt * gridDim.x; their descriptors are
  // read once into shared memory (beyond MAX_CTA_TILES from global memory)
  __shared__ PrefillTile s_tiles[MAX_CTA_TILES];
  for (int l = threadIdx.x; l < MAX_CTA_TILES; l += blockDim.x) {
    const int ti = blockIdx.x + l * gridDim.x;
    if (ti < n_tiles) s_tiles[l] = tiles[ti];
  }
  auto tile_at = [&](int ti) -> PrefillTile {
    const int l = (ti - (int)blockIdx.x) / (int)gridDim.x;
    return l < MAX_CTA_TILES ? s_tiles[l] : tiles[ti];
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full_a[i], 4);   // the 4 producers of the k block's group
      mbar_init(&full_b[i], 1);
      mbar_init(&empty[i], CLUSTER);   // the MMAs of both CTAs of the cluster
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], NEPI);
    }
    for (int i = 0; i < NPROD * PSTAGES; ++i) mbar_init(&pbar[i], 1);
    mbar_init_fence();
    prefetch_tmap(&tmB);
    if (DOWN) prefetch_tmap(&tmB2);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the peer CTA multicasts into this CTA's stages and arrives on its
  // barriers: both must have initialised them first
  cluster_sync();
  const uint32_t crank = blockIdx.x % CLUSTER;

  auto weights = [&](int group) -> const uint8_t* {
    return group < a.E ? a.slots + (int64_t)a.group_slot[group] * a.expert_bytes : a.shared_expert;
  };
  // packed source of producer p for (tile, kb): two blocks, contiguous
  //   down:    Wd input group 2kb + p%2, row blocks 4m + 2((p/2)%2) and the next;
  //   gate/up: row block 2m + p%2, input group 2kb + (p/2)%2, Wg then Wu.
  auto psrc = [&](const PrefillTile& tl, int p, int kb) -> const uint8_t* {
    if (DOWN) return weights(tl.group) + down_block_offset(tl.m * 4 + 2 * ((p >> 1) & 1), 2 * kb + (p & 1), a.d, a.f);
    return weights(tl.group) + gu_block_offset(tl.m * 2 + (p & 1), 2 * kb + ((p >> 1) & 1), 0, a.d);
  };

  if (warp == 0) {
    // ---- token tiles by TMA -------------------------------------------------
    if (lane == 0) {
      PF_VAR(pf_t9);
      // the token tiles of the item kPrefetch ahead are prefetched into L2, so
      // a stage's load waits for L2 rather than DRAM
      constexpr int kPrefetch = 4;
      int pf_ti = blockIdx.x, pf_kb = 0;
      auto prefetch_next = [&]() {
        if (pf_ti >= n_tiles) return;
        const int row0 = tile_at(pf_ti).row0 + (int)crank * (BN / CLUSTER);
        tma_prefetch_l2_2d(&tmB, pf_kb * BK, row0);
        if (DOWN) tma_prefetch_l2_2d(&tmB2, pf_kb * BK, row0);
        if (++pf_kb == n_kb) {
          pf_kb = 0;
          pf_ti += gridDim.x;
        }
      };
      for (int i = 0; i < kPrefetch; ++i) prefetch_next();
      uint32_t it = 0;
      for (int ti = blockIdx.x; ti < n_tiles; ti += gridDim.x) {
        const PrefillTile tl = tile_at(ti);
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          prefetch_next();
          const int s = it % STAGES;
          const uint32_t use = it / STAGES;
          {
            PF_T0();
            if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1)) {
              set_error(a.err, DEV_TIMEOUT_BARRIER);
              goto done;
            }
            PF_ACC(pf_t9);
          }
          uint8_t* st = stages + s * STAGE_BYTES;
          // this CTA loads token rows [crank * BN/2, +BN/2) of the tile for
          // both CTAs of the cluster (the other half comes from the peer)
          mbar_arrive_expect_tx(&full_b[s], NB * B_BYTES);
          const int yrow = tl.row0 + (int)crank * (BN / CLUSTER);
          tma_load_2d_multicast(st + A_BYTES + crank * B_HALF, &tmB, kb * BK, yrow, &full_b[s], 0x3);
          if (DOWN)
            tma_load_2d_multicast(st + A_BYTES + B_BYTES + crank * B_HALF, &tmB2, kb * BK, yrow, &full_b[s], 0x3);
        }
      }
      PF_PUT(DOWN, 9, pf_t9);
    }
  } else if (warp == 1) {
    // ---- MMA issue ----------------------------------------------------------
    if (lane == 0) {
      PF_T0();
      PF_VAR(pf_wa);
      PF_VAR(pf_wb);
      PF_VAR(pf_is);
      uint32_t it = 0, lt = 0;
      for (int ti = blockIdx.x; ti < n_tiles; ti += gridDim.x, ++lt) {
        const PrefillTile tl = tile_at(ti);
        const int nmma = (tl.nlen + 15) & ~15;
        const uint32_t idesc = idesc_f16(BM, nmma, 0);
        const int ab = lt & 1;
        const uint32_t use_b = lt >> 1;
        {
          PF_T0();
          if (use_b > 0 && !mbar_wait(&tempty[ab], (use_b - 1) & 1)) {
            set_error(a.err, DEV_TIMEOUT_BARRIER);
            goto done;
          }
          PF_ADD(DOWN, 2);
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + ab * BN;
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t par = (it / STAGES) & 1;
          {
            PF_T0();
            if (!mbar_wait(&full_a[s], par)) {
              set_error(a.err, DEV_TIMEOUT_BARRIER);
              goto done;
            }
            PF_ACC(pf_wa);
          }
          {
            PF_T0();
            if (!mbar_wait(&full_b[s], par)) {
              set_error(a.err, DEV_TIMEOUT_BARRIER);
              goto done;
            }
            PF_ACC(pf_wb);
          }
          PF_T0();
          tc_fence_after();
          uint8_t* st = stages + s * STAGE_BYTES;
          const uint64_t da = smem_desc_sw128(st);
          const uint64_t db = smem_desc_sw128(st + A_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            umma_f16(d_tmem, da + 2 * kk, db + 2 * kk, idesc, (kb | kk) != 0);
            if (DOWN) {
              const uint64_t db_lo = smem_desc_sw128(st + A_BYTES + B_BYTES);
              umma_f16(d_tmem, da + 2 * kk, db_lo + 2 * kk, idesc, 1u);
            }
          }
          umma_commit_multicast(&empty[s], 0x3);   // frees the stage in both CTAs
          PF_ACC(pf_is);
        }
        umma_commit(&tfull[ab]);
      }
      PF_ADD(DOWN, 3);
      PF_PUT(DOWN, 0, pf_wa);
      PF_PUT(DOWN, 1, pf_wb);
      PF_PUT(DOWN, 11, pf_is);
    }
  } else if (warp < EPI0) {
    // ---- weight producers: 3-bit blocks -> fp16 swizzled tiles -------------
    // producer p takes the k blocks kb with kb % NGROUP == p/4; per k block
    // the 4 producers of that group expand 2 blocks each (the 8 blocks of
    // the 128 x 64 tile)
    const int p = warp - 2, par = p >> 2;
    uint8_t* my_stage = pstage + p * PSTAGES * PCHUNK;
    uint64_t* my_bar = pbar + p * PSTAGES;
    // stmatrix row addresses: lane L writes row L%8 of sub-tile L/8
    const uint32_t gx = (uint32_t)(lane & 7) << 4;
    // tile rows of this producer's first block, and the k chunk of each block
    //   down:    rows ((p/2)%2)*64 and the next 32, k chunk 4*(p%2) (input group 2kb + p%2);
    //   gate/up: Wg rows (p%2)*32, Wu rows 64 + (p%2)*32, k chunk 4*((p/2)%2).
    const int row0 = DOWN ? ((p >> 1) & 1) * 64 : (p & 1) * 32;
    const uint32_t lane_off = (uint32_t)((row0 + 8 * ((lane >> 3) & 1) + (lane & 7)) * 128);
    const bool hi_group = !DOWN && ((p >> 1) & 1);
    int ti_issue = blockIdx.x, kb_issue = par;
    uint32_t n_issued = 0;
    auto issue_next = [&]() {
      if (ti_issue >= n_tiles) return;
      const PrefillTile tl = tile_at(ti_issue);
      const int ps = n_issued % PSTAGES;
      if (lane == 0) {
        mbar_arrive_expect_tx(&my_bar[ps], PCHUNK);
        bulk_g2s(my_stage + ps * PCHUNK, psrc(tl, p, kb_issue), PCHUNK, &my_bar[ps]);
      }
      ++n_issued;
      kb_issue += NGROUP;
      if (kb_issue >= n_kb) {
        kb_issue = par;
        ti_issue += gridDim.x;
      }
    };
    for (int i = 0; i < PSTAGES - 1; ++i) issue_next();
    PF_VAR(pf_p6);
    PF_VAR(pf_p7);
    PF_VAR(pf_p8);
    uint32_t j = 0, lt = 0;
    for (int ti = blockIdx.x; ti < n_tiles; ti += gridDim.x, ++lt) {
      for (int kb = par; kb < n_kb; kb += NGROUP, ++j) {
        __syncwarp();
        issue_next();   // refills the slot consumed PSTAGES-1 items ago
        const int ps = j % PSTAGES;
        {
          PF_T0();
          if (!__all_sync(0xffffffffu, mbar_wait(&my_bar[ps], (j / PSTAGES) & 1))) {
            set_error(a.err, DEV_TIMEOUT_BARRIER);
            goto done;
          }
          PF_ACC(pf_p6);
        }
        // both blocks expanded into registers first: once the tile stage is
        // free only the stores remain before the MMA can use it
        uint32_t v0[16], v1[16];
        {
          PF_T0();
          const uint8_t* src = my_stage + ps * PCHUNK;
          expand_block(src, lane, v0);
          expand_block(src + kBlockBytes, lane, v1);
          PF_ACC(pf_p8);
        }
        const uint32_t it = lt * n_kb + kb;
        const int s = it % STAGES;
        const uint32_t use = it / STAGES;
        {
          PF_T0();
          if (use > 0 && !__all_sync(0xffffffffu, mbar_wait(&empty[s], (use - 1) & 1))) {
            set_error(a.err, DEV_TIMEOUT_BARRIER);
            goto done;
          }
          PF_ACC(pf_p7);
        }
        PF_T0();
        __syncwarp();   // after lane 0's issue and the waits: stmatrix runs on the whole warp
        const uint32_t tile_lane = smem_u32(stages + s * STAGE_BYTES) + lane_off;
        if (DOWN) {
          if (p & 1) {
            store_block_tile<4>(v0, lane, tile_lane, gx);
            store_block_tile<4>(v1, lane, tile_lane + 32 * 128, gx);
          } else {
            store_block_tile<0>(v0, lane, tile_lane, gx);
            store_block_tile<0>(v1, lane, tile_lane + 32 * 128, gx);
          }
        } else if (!hi_group) {
          store_block_tile<0>(v0, lane, tile_lane, gx);                 // Wg
          store_block_tile<0>(v1, lane, tile_lane + GU_ROWS * 128, gx);  // Wu
        } else {
          store_block_tile<4>(v0, lane, tile_lane, gx);
          store_block_tile<4>(v1, lane, tile_lane + GU_ROWS * 128, gx);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full_a[s]);
        PF_ACC(pf_p8);
      }
    }
    if (p == 0 && lane == 0) {
      PF_PUT(DOWN, 6, pf_p6);
      PF_PUT(DOWN, 7, pf_p7);
      PF_PUT(DOWN, 8, pf_p8);
    }
  } else {
    // ---- epilogue: 8 warps; warp (quarter q = warp % 4, half hf) reads TMEM
    // lanes 32q..32q+31 (M rows) and, of every 32-column chunk, the 16
    // columns (tokens) 16hf..16hf+15.  No block-wide barrier: each warp
    // writes its own rows straight to global memory.
    const int quarter = warp & 3;
    const int hf = (warp - EPI0) >> 2;
    const int ew = warp - EPI0;                     // 0..7
    uint32_t lt = 0, chunk = 0;                     // chunk: running count across tiles
    PF_VAR(pf_e12);
    PF_VAR(pf_e13);
    PF_VAR(pf_e14);
    for (int ti = blockIdx.x; ti < n_tiles; ti += gridDim.x, ++lt) {
      const PrefillTile tl = tile_at(ti);
      const int ab = lt & 1;
      // down: the token and routing weight of every column this warp reads,
      // loaded before the accumulator is ready (lane j of chunk cc holds
      // column cc*32 + 16hf + j, j < 16)
      // (routed tiles: the pick index instead of the token, the row of
      // osort that the column's output goes to)
      int ctok[kPrefillBN / 32];
      float cw[kPrefillBN / 32];
      if (DOWN) {
        const bool routed = tl.group < a.E;
#pragma unroll
        for (int cc = 0; cc < kPrefillBN / 32; ++cc) {
          const int col = cc * 32 + hf * 16 + (lane & 15);
          ctok[cc] = col < tl.nlen ? (routed ? a.pick[tl.row0 + col] : a.perm[tl.row0 + col]) : 0;
          cw[cc] = col < tl.nlen ? a.wsort[tl.row0 + col] : 0.f;
        }
      }
      {
        PF_T0();
        if (!__all_sync(0xffffffffu, mbar_wait(&tfull[ab], (lt >> 1) & 1))) {
          set_error(a.err, DEV_TIMEOUT_BARRIER);
          goto done;
        }
        if (ew == 0 && lane == 0) PF_ADD(DOWN, 5);
      }
      __syncwarp();   // tcgen05.ld below runs on the whole warp
      PF_T0();
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + ab * BN + hf * 16;
#pragma unroll 1
      for (int cc = 0; cc * 32 < tl.nlen; ++cc, ++chunk) {
        const int col0 = cc * 32 + hf * 16;          // first column (token) of this warp
        uint32_t r[16];
        {
          PF_T0();
          tmem_ld16(taddr + cc * 32, r);
          tmem_ld_wait();
          PF_ACC(pf_e12);
        }
        if (!DOWN) {
          // g rows sit in quarters 0-1, the same f rows of u in quarters 2-3.
          // The two warps of a pair swap halves through a two-slot buffer and
          // a 64-thread barrier (ids 1-4, one per pair): the g warp gets u of
          // columns 0-7 and finishes them, the u warp gets g of columns 8-15
          // and finishes those.  Slots alternate by the running chunk count,
          // so a slot is written again only after both warps have passed the
          // barrier of the chunk after the one that read it.
          const int pair = (quarter & 1) + 2 * hf;
          const bool is_g = quarter < 2;
          float* slot = reinterpret_cast<float*>(epi) + ((size_t)pair * 2 + (chunk & 1)) * 16 * 32;
          float* give = slot + (is_g ? 8 * 32 : 0);        // g 8-15 or u 0-7
          const float* take = slot + (is_g ? 0 : 8 * 32);  // u 0-7 or g 8-15
          const int own0 = is_g ? 0 : 8;                    // columns this warp finishes
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) give[jj * 32 + lane] = __uint_as_float(is_g ? r[8 + jj] : r[jj]);
          {
            PF_T0();
            named_bar(1 + pair, 64);
            PF_ACC(pf_e13);
          }
          PF_T0();
          const int frow = tl.m * GU_ROWS + (quarter & 1) * 32 + lane;
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int col = col0 + own0 + jj;
            if (col < tl.nlen) {
              const float mine = __uint_as_float(is_g ? r[jj] : r[8 + jj]), other = take[jj * 32 + lane];
              const float gv = is_g ? mine : other, uv = is_g ? other : mine;
              // silu(g) * u with the fast exponential and division (relative
              // error ~2^-21, below what the fp16 pair carries)
              const float hv = __fdividef(gv, 1.f + __expf(-gv)) * uv;
              const __half hi = __float2half_rn(hv);
              const size_t o = (size_t)(tl.row0 + col) * a.f + frow;
              a.hg[o] = __half_as_ushort(hi);
              a.hg_lo[o] = __half_as_ushort(__float2half_rn(hv - __half2float(hi)));
            }
          }
          PF_ACC(pf_e14);
        } else {
          int tokc = 0;
          float wc = 0.f;
#pragma unroll
          for (int q = 0; q < kPrefillBN / 32; ++q)
            if (q == cc) {
              tokc = ctok[q];
              wc = cw[q];
            }
          // routed expert: the weighted output of pick t*k + i goes to row
          // t*k + i of osort (so a token's picks are contiguous for the
          // combine, which sums them in pick order); the shared expert
          // (every token once): straight into y
          const int drow = tl.m * BM + quarter * 32 + lane;
          if (tl.group < a.E) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int pk = __shfl_sync(0xffffffffu, tokc, jj);
              const float w = __shfl_sync(0xffffffffu, wc, jj);
              if (col0 + jj < tl.nlen) a.osort[(size_t)pk * a.d + drow] = __uint_as_float(r[jj]) * w;
            }
          } else {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int tok = __shfl_sync(0xffffffffu, tokc, jj);
              const float w = __shfl_sync(0xffffffffu, wc, jj);
              if (col0 + jj < tl.nlen) a.y[(size_t)tok * a.d + drow] = __uint_as_float(r[jj]) * w;
            }
          }
        }
      }
      tc_fence_before();
      if (lane == 0) mbar_arrive(&tempty[ab]);
      __syncwarp();
      if (ew == 0 && lane == 0) {
        PF_ADD(DOWN, 4);
#ifdef MOE_TIMELINE
        g_prefill_prof[DOWN][blockIdx.x][10] += 1;
#endif
      }
    }
    if (ew == 2 && lane == 0) {
      PF_PUT(DOWN, 12, pf_e12);
      PF_PUT(DOWN, 13, pf_e13);
      PF_PUT(DOWN, 14, pf_e14);
    }
  }
done:
  tc_fence_before();
  __syncthreads();
  // no CTA leaves while its peer may still write into it
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

#ifdef MOE_TIMELINE
extern "C" int moe_debug_prefill_profile(unsigned long long* out, int reset) {
  if (reset) {
    static unsigned long long zero[2][256][16];
    return (int)cudaMemcpyToSymbol(g_prefill_prof, zero, sizeof(zero));
  }
  return (int)cudaMemcpyFromSymbol(out, g_prefill_prof, sizeof(g_prefill_prof));
}
#endif

template <bool DOWN>
static size_t gemm_smem() {
  constexpr int NB = DOWN ? 2 : 1;
  constexpr int STAGES = DOWN ? 2 : 3;
  constexpr int STAGE_BYTES = pg::A_BYTES + NB * pg::B_BYTES;
  constexpr int EPI_BYTES = DOWN ? 0 : 4 * 2 * 16 * 32 * 4;
  return 1024 + STAGES * STAGE_BYTES + EPI_BYTES + pg::NPROD * pg::PSTAGES * pg::PCHUNK +
         (3 * STAGES + 4 + pg::NPROD * pg::PSTAGES) * 8 + 16;
}

template <bool DOWN>
static cudaError_t launch_gemm(const CUtensorMap& tmB, const CUtensorMap& tmB2, const PrefillGemmArgs& a,
                               cudaStream_t s, int num_sms) {
  // the persistent grid (as many whole clusters as can be resident at once)
  // is found once per device, after the shared-memory limit is raised there
  static std::mutex mu;
  static int grid_of[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const size_t smem = gemm_smem<DOWN>();
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pg::CLUSTER;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(pg::THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int grid;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (grid_of[dev] == 0) {
      e = ensure_dyn_smem(reinterpret_cast<const void*>(prefill_gemm_kernel<DOWN>), smem);
      if (e != cudaSuccess) return e;
      cfg.gridDim = dim3(num_sms - num_sms % pg::CLUSTER);
      int clusters = 0;
      e = cudaOccupancyMaxActiveClusters(&clusters, prefill_gemm_kernel<DOWN>, &cfg);
      if (e != cudaSuccess) return e;
      if (clusters < 1) return cudaErrorInvalidConfiguration;
      int g = clusters * pg::CLUSTER;
      if (g > num_sms) g = num_sms - num_sms % pg::CLUSTER;
      grid_of[dev] = g;
    }
    grid = grid_of[dev];
  }
  cfg.gridDim = dim3(grid);
  return cudaLaunchKernelEx(&cfg, prefill_gemm_kernel<DOWN>, tmB, tmB2, a);
}

// y[t] += the weighted outputs of token t's routed picks, added in pick
// order (ascending expert id) after the shared expert's part, so y does not
// depend on the order in which tiles or the counting sort ran.  One thread
// per 4 consecutive outputs; every pick's load is issued before the sum.
__global__ void __launch_bounds__(256) prefill_combine_kernel(PrefillCombineArgs a) {
  const int d4 = a.d / 4;
  const int64_t n = (int64_t)a.T * d4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / d4), c = (int)(i - (int64_t)t * d4);
    float4 acc = reinterpret_cast<const float4*>(a.y + (size_t)t * a.d)[c];
    float4 o[kMaxTopK];
#pragma unroll
    for (int kk = 0; kk < kMaxTopK; ++kk)
      if (kk < a.k) o[kk] = __ldcs(reinterpret_cast<const float4*>(a.osort + ((size_t)t * a.k + kk) * a.d) + c);
#pragma unroll
    for (int kk = 0; kk < kMaxTopK; ++kk) {
      if (kk < a.k) {
        acc.x += o[kk].x;
        acc.y += o[kk].y;
        acc.z += o[kk].z;
        acc.w += o[kk].w;
      }
    }
    reinterpret_cast<float4*>(a.y + (size_t)t * a.d)[c] = acc;
  }
}

cudaError_t launch_prefill_plan(const PrefillPlanArgs& a, cudaStream_t s) {
  prefill_plan_kernel<<<1, 1024, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_prefill_scatter(const PrefillScatterArgs& a, cudaStream_t s) {
  const int n = a.T * a.k + a.T;
  prefill_scatter_kernel<<<(n + 255) / 256, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_prefill_combine(const PrefillCombineArgs& a, cudaStream_t s) {
  const int64_t n = (int64_t)a.T * (a.d / 4);
  const int64_t blocks = (n + 255) / 256;
  prefill_combine_kernel<<<(unsigned)(blocks < 65536 ? blocks : 65535), 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_prefill_gather(const uint16_t* x, const int32_t* perm, uint16_t* xg, int rows, int d,
                                  cudaStream_t s) {
  int blocks = (rows + 7) / 8;
  if (blocks > 152 * 6) blocks = 152 * 6;
  prefill_gather_kernel<<<blocks, 256, 0, s>>>(x, perm, xg, rows, d);
  return cudaGetLastError();
}

cudaError_t launch_prefill_gate_up(const CUtensorMap& tmX, const PrefillGemmArgs& a, cudaStream_t s, int grid) {
  return launch_gemm<false>(tmX, tmX, a, s, grid);
}

cudaError_t launch_prefill_down(const CUtensorMap& tmH, const CUtensorMap& tmHlo, const PrefillGemmArgs& a,
                                cudaStream_t s, int grid) {
  return launch_gemm<true>(tmH, tmHlo, a, s, grid);
}

}  // namespace moe
