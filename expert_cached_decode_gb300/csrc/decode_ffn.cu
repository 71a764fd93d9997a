// Decode / verify step (T <= 16 tokens): every distinct routed expert and
// the shared expert run once for all tokens routed to them (a verify batch
// shares one fetch of each expert, page "单卡5090跑125B 大模型", §2.3),
//   g = Wg.x, u = Wu.x, h = silu(g) * u, o = Wd.h,
//   y[t] = shared_weight * o_shared[t] + sum_i w[t,i] * o_idx[t,i][t].
//
// Work unit: one 32-row slice rb of f of one expert.  It holds the gate/up
// rows of the slice (Wg and Wu blocks of every input group, 2 * d/32 blocks)
// and the down columns of the same slice (the Wd blocks of input group rb for
// every row block of d, d/32 blocks); in the device block layout both are
// contiguous.  A CTA computes g and u of the slice, h = silu(g) * u scaled by
// the routing weight of each token, and the slice's share of the output,
// Wd[:, slice] . h[slice], added into a per-CTA partial of y held in
// registers.  So h never leaves the CTA: the only exchanges between CTAs are
// the router's logits and the final sum of the per-CTA partials.
//
// One persistent CTA per SM.  Warps: CW consumer warps, a producer warp
// (one thread streams every unit through a ring of stages of 2*CW blocks with
// bulk TMA copies, mbarrier completion) and a control warp.  Per call:
//   1. the producer starts the shared expert's units of this CTA at once
//      (static weights, issued even before the previous call has finished);
//   2. consumers stage x (bf16 for the router, fp16 mma fragments for the
//      experts), compute the router logits of rows cta, cta + G, ... and
//      arrive on a grid counter;
//   3. consumers run the CTA's shared-expert units while the other CTAs'
//      logits arrive, then wait for the grid counter and select the experts
//      of the call from the full logits (every CTA, the same selection as the
//      routing kernel), look up their slots and hand the CTA's share of the
//      routed units to the producer;
//   4. routed units; then each CTA writes its partial of y, passes a second
//      grid counter and CTA c sums the partials of rows (t, rb) with
//      t * d/32 + rb = c, c + G, ... in CTA order, so y is deterministic.
// Shared-expert units sit on fixed CTAs spread over the grid; the routed
// units are split in contiguous ranges so that every CTA's total count of
// units is even.
//
// Inside a unit: every gate/up stage gives each consumer warp two blocks, the
// Wg and Wu blocks of one input group.  Codes are expanded to exact fp16 q in
// registers (one LOP3 + one HFMA2 per code pair), multiplied on the tensor
// cores (mma.sync m16n8k16, fp32 accumulate) and scaled per group in fp32.
// The warps' partial sums meet in shared memory, are added in warp order and
// give h (fp16, times the token's routing weight) as the B operand of the
// down stages, where warp w owns the row blocks 2w + j (+ 2*CW per stage) of
// y for the whole call.
//
// With a cache that can miss, CTA 0 takes no units and runs the cache (LRU
// victims, commit, next LRU order, plan).  CTAs 1..G-1 order their routed
// units resident experts first and their producers start streaming them at
// once; the consumers first share the fetch of the call's misses: jobs of 32
// rows of one matrix, read from the registered host pool (contiguous runs of
// the canonical layout) and re-laid out straight into the victim slot, each
// finished job counted per miss.  A producer waits for a missing expert's
// count before it streams that expert's units.  With host-issued miss copies
// the kernel follows the routing kernel and reads its plan.  All waits are
// bounded.
#include "common.cuh"
#include "internal.h"
#include "select.cuh"
#include "repack.cuh"
#include "fetch.cuh"

namespace moe {

#ifdef MOE_TIMELINE
// Timeline builds: each CTA stamps %clock64 into shared memory (a stamp
// that stores to global memory itself slows the warp's next collectives by
// thousands of cycles, which distorts what it measures); the consumers'
// last thread converts the stamps to %globaltimer ns at exit.
__device__ unsigned long long g_ffn_timeline[512][32];
__shared__ long long s_tl[32];
__shared__ unsigned long long s_tl_gt0;
#define MOE_TLS(slot) (s_tl[(slot)] = clock64())
// a stamp by thread 0 in code the whole warp runs: the warp reconverges
// after it (a lane-divergent branch left open makes every later warp
// collective pay a rendezvous)
#define MOE_TL0(slot)                     \
  do {                                    \
    if (threadIdx.x == 0) MOE_TLS(slot);  \
    __syncwarp();                         \
  } while (0)
__device__ __forceinline__ void dtl_begin() {
  for (int i = 0; i < 32; ++i) s_tl[i] = 0;
  s_tl_gt0 = globaltimer();
  s_tl[0] = clock64();
}
__device__ __forceinline__ void dtl_flush(int cta) {
  if (threadIdx.x != 0) return;
  const unsigned long long gt1 = globaltimer();
  const long long c1 = clock64(), c0 = s_tl[0];
  const double ns_per_cycle = c1 > c0 ? (double)(gt1 - s_tl_gt0) / (double)(c1 - c0) : 0.0;
  for (int i = 0; i < 32; ++i)
    g_ffn_timeline[cta][i] = s_tl[i] ? s_tl_gt0 + (unsigned long long)((double)(s_tl[i] - c0) * ns_per_cycle) : 0ull;
}
#define MOE_TL_FLUSH(cta) dtl_flush(cta)
#else
#define MOE_TLS(slot) ((void)0)
#define MOE_TL0(slot) ((void)0)
#define MOE_TL_FLUSH(cta) ((void)0)
#endif

constexpr int kMaxRD = 64;                                 // row blocks of d (d <= 2048)
constexpr int kHsRow = 40;                                 // fp16 per token row of a unit's h (32 + pad)

template <int NT>
struct DCfg {
  static constexpr int CW = 8;                     // consumer warps
  static constexpr int SB = 32;                    // blocks per ring stage (14 KB bulk copies)
  static constexpr int BPW = SB / CW;              // blocks of a stage per consumer warp (4)
  static constexpr int SBYTES = SB * kBlockBytes;  // bytes per ring stage
  static constexpr int THREADS = (CW + 2) * 32;    // + producer and control warps
  static constexpr int NS = NT == 1 ? 10 : 5;      // ring stages (140 KB / 70 KB)
  static constexpr int NQ = 2 * 8 * NT;            // gate/up partial floats per lane (g and u)
  static constexpr int MAXSDN = kMaxRD / SB;       // down stages of a unit at most
};

// Per mode: with the host pool in the device layout two more warps copy the
// stages of missing experts from the host pool into the ring.
template <int NT, int MODE>
struct KCfg : DCfg<NT> {
  static constexpr int HSW = MODE == kFusedCachedDirect || MODE == kAhead ? 2 : 0;   // host-stage warps
  static constexpr int THREADS = (DCfg<NT>::CW + 2 + HSW) * 32;
};

// Index in U of chosen expert `id`.
__device__ __forceinline__ int dsel_act_index(const SelSmem* s, int id) { return sel_act_index(s, id); }

// Selection of a one-token call by all CW warps of the NTH threads of named
// barrier 1 (the same result as select_call: the k largest logits, ties to
// the lower id, weights renormalised, ids ascending, then U).  Keys are
// (order-preserving value bits, ~id), all distinct.  Each half-warp takes
// the maximum of its share of the row; the k-th largest of the 2*CW maxima
// is a threshold that at least k keys reach and every one of the k largest
// reaches; the keys at or above it (a few, in general) are ranked against
// each other.  Needs k <= 2*CW.
template <int NTH, int CW>
__device__ __forceinline__ void select_one_token(const uint64_t* logits, uint32_t tag, uint64_t lim, bool* failed,
                                                 int E, int K, SelSmem* s) {
  constexpr int V = (kMaxE + 32 * CW - 1) / (32 * CW);   // keys per lane
  constexpr int NG = 2 * CW;                             // groups: half-warps
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t* wmax = &s->topk[0][0];                       // [NG] group maxima, [NG] the threshold
  uint64_t* cand = reinterpret_cast<uint64_t*>(&s->row[0][0]);   // up to E candidates
  int* ncand = reinterpret_cast<int*>(&s->topk[1][0]);
  uint64_t* top = &s->topk[2][0];                        // [K] the chosen keys, largest first
  // contiguous ids: lane l of warp w holds ids i*32*CW + w*32 + l (i < V), so
  // a warp's loads cover whole lines; a row shorter than CW*32 leaves later
  // half-warps without keys (their maximum is 0)
  const int nv = E > warp * 32 + lane ? (E - warp * 32 - lane + 32 * CW - 1) / (32 * CW) : 0;
  float lv[V];
  tagged_values<V>(logits + warp * 32 + lane, 32 * CW, nv, tag, lim, failed, lv);
#ifdef MOE_TIMELINE
  MOE_TL0(21);
#endif
  __syncwarp();   // lanes left the polling rounds at different times
  uint64_t key[V];
  uint64_t m = 0;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int id = i * 32 * CW + warp * 32 + lane;
    key[i] = i < nv ? ((uint64_t)float_key(lv[i]) << 32) | (uint32_t)(~(uint32_t)id) : 0ull;
    m = key[i] > m ? key[i] : m;
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) {
    const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)m, o);
    const uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(m >> 32), o);
    const uint64_t n = ((uint64_t)hi << 32) | lo;
    m = n > m ? n : m;
  }
  if ((lane & 15) == 0) wmax[2 * warp + (lane >> 4)] = m;
  for (int i = tid; i < kMaxE / 32; i += NTH) s->mask[i] = 0;
  if (tid == 0) *ncand = 0;
  named_bar(1, NTH);
  if (warp == 0) {   // the K-th largest group maximum (groups without keys hold 0)
    const uint64_t mine = lane < NG ? wmax[lane] : 0ull;
    int above = 0;
#pragma unroll
    for (int j = 0; j < NG; ++j) above += wmax[j] > mine ? 1 : 0;
    const uint32_t holder = __ballot_sync(0xffffffffu, lane < NG && mine != 0 && above == K - 1);
    // fewer than K warps hold keys (a row shorter than K warps' shares):
    // every key is a candidate
    const uint64_t tau = holder ? shfl_u64(mine, __ffs(holder) - 1) : 1ull;
    if (lane == 0) wmax[NG] = tau;
  }
  named_bar(1, NTH);
#ifdef MOE_TIMELINE
  MOE_TL0(22);
#endif
  const uint64_t tau = wmax[NG];
#pragma unroll
  for (int i = 0; i < V; ++i)
    if (key[i] >= tau && key[i] != 0) cand[atomicAdd(ncand, 1)] = key[i];
  named_bar(1, NTH);
  const int nc = *ncand;
  for (int c = tid; c < nc; c += NTH) {
    const uint64_t me = cand[c];
    int r = 0;
    for (int j = 0; j < nc; ++j) r += cand[j] > me ? 1 : 0;
    if (r < K) top[r] = me;
  }
  named_bar(1, NTH);
#ifdef MOE_TIMELINE
  MOE_TL0(23);
#endif
  if (warp == 0) {
    __syncwarp();
    const uint64_t kk = lane < K ? top[lane] : 0ull;
    const float v = lane < K ? key_float((uint32_t)(kk >> 32)) : -INFINITY;
    const int id = lane < K ? (int)~(uint32_t)kk : 0x7fffffff;
    const float topv = __shfl_sync(0xffffffffu, v, 0);
    const float ex = lane < K ? expf(v - topv) : 0.f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    int rank = 0;
    for (int j = 0; j < K; ++j) rank += __shfl_sync(0xffffffffu, id, j) < id ? 1 : 0;
    if (lane < K) {
      s->sel_id[0][rank] = id;
      s->sel_w[0][rank] = ex / sum;
      atomicOr(&s->mask[id >> 5], 1u << (id & 31));
    }
    __syncwarp();
    // U: the chosen experts in ascending id
    const int n_words = (E + 31) / 32;
    const uint32_t mw = lane < n_words ? s->mask[lane] : 0u;
    const int c = __popc(mw);
    int inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += n;
    }
    const int base = inc - c;
    if (lane < n_words) s->word_base[lane] = base;
    if (lane == 31) s->n_act = inc;
    uint32_t mm = mw;
    int pos = base;
    while (mm) {
      const int bit = __ffs(mm) - 1;
      mm &= mm - 1;
      s->act[pos++] = lane * 32 + bit;
    }
  }
  named_bar(1, NTH);
}

// loader of tagged logits rows for select_call: a lane's words of row t are
// read in batches of 8 (tagged_values, bounded); a time-out is recorded in
// *failed
struct TaggedLogits {
  const uint64_t* p;
  uint32_t tag;
  uint64_t lim;
  bool* failed;
  __device__ __forceinline__ void row(float* r, int t, int E, int lane) const {
    const int nper = (E - lane + 31) / 32;   // ids lane + 32 j, j < nper
#pragma unroll 1
    for (int j0 = 0; j0 < nper; j0 += 8) {
      float v[8];
      tagged_values<8>(p + (size_t)t * E + lane + 32 * j0, 32, nper - j0 < 8 ? nper - j0 : 8, tag, lim, failed, v);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j0 + j < nper) r[lane + 32 * (j0 + j)] = v[j];
    }
  }
};

// elements per staged x row (bf16, router input): 32 bytes of padding
__host__ __device__ __forceinline__ int x_row_elems(int d) { return d + 16; }

// bytes of the shared-memory region whose uses never overlap in time: x
// rows for the router, the selection scratch, the gate/up partials, a miss
// fetch job and the combine partials
template <int NT>
__host__ __device__ __forceinline__ size_t overlay_bytes(int d) {
  using C = DCfg<NT>;
  size_t b = (size_t)NT * 8 * x_row_elems(d) * 2;
  const size_t sel = (sizeof(SelSmem) + 15) & ~size_t(15);
  const size_t red = (size_t)C::CW * C::NQ * 32 * 4;
  const size_t pull = (size_t)2 * kMaxPicks * 4;
  const size_t cmb = (size_t)C::CW * 32 * 4;
  const size_t job = fetch_job_bytes(d, 1024);   // one fetch job of a miss (f <= 1024)
  b = b > job ? b : job;
  b = b > sel ? b : sel;
  b = b > red ? b : red;
  b = b > pull ? b : pull;
  b = b > cmb ? b : cmb;
  return (b + 127) & ~size_t(127);
}

template <int NT>
__host__ __device__ __forceinline__ size_t ffn_smem_bytes(int d) {
  using C = DCfg<NT>;
  return (size_t)C::NS * C::SBYTES + (size_t)NT * d * 16 + overlay_bytes<NT>(d) + (size_t)NT * 8 * kHsRow * 2 +
         (2 * C::NS + 1) * 8;
}

// first shared-expert unit of tile CTA c: the RG shared units spread evenly
// over the GT tile CTAs (CTA c takes slices [S(c), S(c+1)))
__device__ __forceinline__ int shared_first(int c, int RG, int GT) {
  const int v = (c * RG + GT - 1) / GT;
  return v < RG ? v : RG;
}

// first routed unit of tile CTA c, for NU routed units after the shared ones:
// every CTA's total (shared + routed) is the floor or the ceiling of the mean
__device__ __forceinline__ int routed_first(int c, int NU, int RG, int GT) {
  const int q = NU + RG;
  if (RG <= GT && q >= GT) {
    const int base = q / GT, rem = q % GT;
    return c * base + (c < rem ? c : rem) - shared_first(c, RG, GT);
  }
  return (int)((int64_t)c * NU / GT);
}

__device__ __forceinline__ uint32_t pack_half2_from_bf16(uint32_t two_bf16) {
  const __half2 h = __floats2half2_rn(bf16_bits_to_float(two_bf16 & 0xffffu), bf16_bits_to_float(two_bf16 >> 16));
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void scales4(const uint8_t* bp, int lane, float s[4]) {
  const uint2 sc = *reinterpret_cast<const uint2*>(bp + kBlockCodeBytes + (lane >> 2) * 8);
  const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&sc.x));
  const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&sc.y));
  s[0] = lo.x;   // row g
  s[1] = lo.y;   // row g+8
  s[2] = hi.x;   // row g+16
  s[3] = hi.y;   // row g+24
}

// Two 32x32 blocks of one warp: acc_j[nt][mt] += scale(row) * (A_j . B[nt])
// for j = 0, 1 (blocks at bp0, bp1, with the same B fragments), products in
// fp32 on the tensor cores, the scale of the lane's rows g, g+8, g+16, g+24
// applied in fp32.  Both blocks' codes are expanded before the products, and
// the first k-step of every tile is issued before the second, so eight
// independent products overlap their latency.
template <int NT>
__device__ __forceinline__ void block_pair_mma(const uint8_t* bp0, const uint8_t* bp1, int lane,
                                               const uint2 (&bx)[NT][2], float (&acc0)[NT][2][4],
                                               float (&acc1)[NT][2][4]) {
  const uint32_t* w0p = reinterpret_cast<const uint32_t*>(bp0);
  const uint32_t* w1p = reinterpret_cast<const uint32_t*>(bp1);
  const uint32_t a0 = w0p[lane], a1 = w0p[32 + lane], a2 = w0p[64 + lane];
  const uint32_t b0 = w1p[lane], b1 = w1p[32 + lane], b2 = w1p[64 + lane];
  float s0[4], s1[4];
  scales4(bp0, lane, s0);
  scales4(bp1, lane, s1);
  uint32_t A0[16], A1[16];
  dequant_block(a0, a1, a2, A0);
  dequant_block(b0, b1, b2, A1);
  const float zero[4] = {0.f, 0.f, 0.f, 0.f};
  float D0[NT][2][4], D1[NT][2][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      mma_16816(D0[nt][mt], &A0[mt * 8], bx[nt][0].x, bx[nt][0].y, zero);
      mma_16816(D1[nt][mt], &A1[mt * 8], bx[nt][0].x, bx[nt][0].y, zero);
    }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      mma_16816(D0[nt][mt], &A0[mt * 8 + 4], bx[nt][1].x, bx[nt][1].y, D0[nt][mt]);
      mma_16816(D1[nt][mt], &A1[mt * 8 + 4], bx[nt][1].x, bx[nt][1].y, D1[nt][mt]);
    }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc0[nt][mt][i] = fmaf(s0[2 * mt + (i >> 1)], D0[nt][mt][i], acc0[nt][mt][i]);
        acc1[nt][mt][i] = fmaf(s1[2 * mt + (i >> 1)], D1[nt][mt][i], acc1[nt][mt][i]);
      }
}

// exclusive prefix sum over the NTH threads of named barrier 1 (every one of
// them calls it); s_warp holds NTH/32 + 1 ints
template <int NTH>
__device__ __forceinline__ int group_exclusive_scan(int v, int* s_warp, int* total) {
  constexpr int NW = NTH / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) s_warp[warp] = inc;
  named_bar(1, NTH);
  if (warp == 0) {
    const int wv = lane < NW ? s_warp[lane] : 0;
    int wi = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    if (lane < NW) s_warp[lane] = wi - wv;
    if (lane == NW - 1) s_warp[NW] = wi;
  }
  named_bar(1, NTH);
  const int r = s_warp[warp] + inc - v;
  *total = s_warp[NW];
  named_bar(1, NTH);   // s_warp may be reused
  return r;
}

// Cache of a layer-call with fused routing, run by the NTH consumer threads
// of CTA 0 (which takes no units).  LRU by (layer, expert), ties to the lower
// slot id (page "单卡5090跑125B 大模型", §2.1 and §7.2): U = the call's
// distinct experts (ascending); resident ones are hits; the misses, in
// ascending expert id, take the least recently used slots in (stamp, slot id)
// order, which is the order of q (least recent first) with the hits skipped.
// The call's touched slots (hits and victims) move, in slot-id order, to the
// recent end of q.  The victims and the miss count are published first
// (vict[0], on every call), because CTAs 1..G-1 wait for them before pulling
// the misses; then the commit (table, owners, stamps), the next order, the
// plan and the statistics.  `scratch`
// is shared memory this CTA does not otherwise use.
template <int NTH>
__device__ __forceinline__ void cache_manager(const FfnArgs& a, int n_act, int m, const int* s_act_expert,
                                              int* s_act_slot, const int* s_pick_act, const float* s_w,
                                              long long clk, uint32_t calls, uint8_t* scratch,
                                              size_t scratch_bytes, uint32_t* vict) {
  __shared__ int s_warp[NTH / 32 + 1];
  __shared__ int s_evict;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.T, K = a.k, C = a.C;
  const int c_words = (C + 31) / 32;
  Plan* P = a.plan;
  int32_t* table = const_cast<int32_t*>(a.table);
  // scratch: four per-pick arrays, the touched-slot bitmap, then (if it
  // fits) the staged LRU order
  int* s_miss_ai = reinterpret_cast<int*>(scratch);
  int* s_victim = s_miss_ai + kMaxPicks;
  int* s_old = s_victim + kMaxPicks;
  int* s_hitf = s_old + kMaxPicks;
  uint32_t* bits = reinterpret_cast<uint32_t*>(s_hitf + kMaxPicks);
  const size_t head = (size_t)4 * kMaxPicks * 4;
  const size_t bits_bytes = ((size_t)c_words * 4 + 15) & ~size_t(15);
  int32_t* sq = head + bits_bytes + (size_t)C * 4 <= scratch_bytes
                    ? reinterpret_cast<int32_t*>(scratch + head + bits_bytes)
                    : nullptr;
  for (int i = tid; i < c_words; i += NTH) bits[i] = 0;
  if (sq) {   // the LRU order staged with 16-byte loads, all in flight
    const int n4 = C >> 2;
    const int4* src4 = reinterpret_cast<const int4*>(a.q_in);
#pragma unroll 4
    for (int i = tid; i < n4; i += NTH) reinterpret_cast<int4*>(sq)[i] = __ldcg(src4 + i);
    for (int i = 4 * n4 + tid; i < C; i += NTH) sq[i] = a.q_in[i];
  }
  for (int i = tid; i < n_act; i += NTH) s_hitf[i] = s_act_slot[i] >= 0;
  if (warp == 0) {   // the misses in ascending expert id
    int base = 0;
    for (int i0 = 0; i0 < n_act; i0 += 32) {
      const int i = i0 + lane;
      const bool miss = i < n_act && s_act_slot[i] < 0;
      const uint32_t bal = __ballot_sync(0xffffffffu, miss);
      if (miss) s_miss_ai[base + __popc(bal & ((1u << lane) - 1u))] = i;
      base += __popc(bal);
      __syncwarp();
    }
  }
  if (tid == 0) s_evict = 0;
  named_bar(1, NTH);
  for (int i = tid; i < n_act; i += NTH) {
    const int sl = s_act_slot[i];
    if (sl >= 0) atomicOr(&bits[sl >> 5], 1u << (sl & 31));
  }
  named_bar(1, NTH);
  const int32_t* q_in = sq ? sq : a.q_in;
  // walk q skipping the hits: the first m slots are the victims, the rest
  // keep their order at the front of the next q
  const int chunk = (C + NTH - 1) / NTH;
  const int lo = min(C, tid * chunk), hi = min(C, lo + chunk);
  int cnt = 0;
  for (int i = lo; i < hi; ++i) {
    const int sl = q_in[i];
    cnt += !((bits[sl >> 5] >> (sl & 31)) & 1u);
  }
  int total;
  int r = group_exclusive_scan<NTH>(cnt, s_warp, &total);
  for (int i = lo; i < hi; ++i) {
    const int sl = q_in[i];
    if (!((bits[sl >> 5] >> (sl & 31)) & 1u)) {
      if (r < m) s_victim[r] = sl;
      else a.q_out[r - m] = sl;
      ++r;
    }
  }
  named_bar(1, NTH);
  for (int j = tid; j < m; j += NTH) {
    const int v = s_victim[j];
    const int ai = s_miss_ai[j];
    const int old = a.owner[v];
    atomicOr(&bits[v >> 5], 1u << (v & 31));
    s_old[j] = old;
    s_act_slot[ai] = v;
    P->miss_expert[j] = s_act_expert[ai];
    P->miss_slot[j] = v;
    P->evicted_key[j] = old;
  }
  named_bar(1, NTH);
  for (int i = tid; i < n_act; i += NTH) {
    P->act_slot[i] = s_act_slot[i];
    P->act_hit[i] = s_hitf[i];
    P->act_expert[i] = s_act_expert[i];
  }
  if (tid == 0) P->n_miss = m;
  named_bar(1, NTH);
  if (tid == 0) {   // published on every call (lookahead copies wait for it even without misses)
    MOE_TLS(28);
    red_release_add(&vict[0], 1u);   // covers the plan's miss count and victim entries (after the barrier)
  }
  // commit: evicted keys leave the table before the misses enter it
  for (int j = tid; j < m; j += NTH) {
    const int old = s_old[j];
    if (old >= 0) {
      table[old] = -1;
      atomicAdd(&s_evict, 1);
    }
  }
  named_bar(1, NTH);
  for (int j = tid; j < m; j += NTH) {
    const int v = s_victim[j];
    const int key = a.layer * a.E + s_act_expert[s_miss_ai[j]];
    a.owner[v] = key;
    table[key] = v;
    a.stamp[v] = clk;
  }
  for (int i = tid; i < n_act; i += NTH)
    if (s_hitf[i]) a.stamp[s_act_slot[i]] = clk;
  // touched slots (hits and victims) in ascending slot id to the recent end
  const int wchunk = (c_words + NTH - 1) / NTH;
  const int wlo = min(c_words, tid * wchunk), whi = min(c_words, wlo + wchunk);
  int tc = 0;
  for (int i = wlo; i < whi; ++i) tc += __popc(bits[i]);
  int tr = group_exclusive_scan<NTH>(tc, s_warp, &total);
  for (int i = wlo; i < whi; ++i) {
    uint32_t b = bits[i];
    while (b) {
      const int bit = __ffs(b) - 1;
      b &= b - 1;
      a.q_out[C - n_act + tr] = i * 32 + bit;
      ++tr;
    }
  }
  // the plan's routing part and the counts (T * K <= NTH: one pick per thread)
  for (int i = tid; i < T * K; i += NTH) {
    P->idx[i] = s_act_expert[s_pick_act[i]];
    P->w[i] = s_w[i];
    P->pick_act[i] = s_pick_act[i];
  }
  const int th = named_bar_count(1, NTH, tid < T * K && s_hitf[s_pick_act[tid]]);
  if (tid == 0) {
    P->n_act = n_act;
    P->n_miss = m;
    P->T = T;
    P->clock = clk;
    P->token_hits = th;
    P->token_misses = (int64_t)T * K - th;
    a.stats[ST_CALLS] += 1;
    a.stats[ST_TOK_HIT] += th;
    a.stats[ST_TOK_MISS] += (int64_t)T * K - th;
    a.stats[ST_DIST_HIT] += n_act - m;
    a.stats[ST_DIST_MISS] += m;
    a.stats[ST_EVICT] += s_evict;
    a.stats[ST_MISS_BYTES] += (int64_t)m * a.expert_bytes;
    *a.clock = clk + 1;
    *a.counters = calls + 1;   // every CTA read the count before the router barrier
  }
}

// MODE kPlanRead: the routing plan comes from memory (routing kernel and
// host-issued miss copies before this launch).  kFusedResident: routing in
// this kernel, every key resident.  kFusedCached: routing in this kernel with
// a cache that may miss (CTA 0 manages the cache; the other CTAs fetch the
// misses into their victim slots, then compute).  kFusedCachedDirect: the
// same with the host pool in the device layout: a missing expert's stages
// are copied from the host pool into the ring by the host-stage warps, which
// also write them into the victim slot, so no fetch runs ahead of the units.
template <int NT, int MODE>
__global__ void __launch_bounds__(KCfg<NT, MODE>::THREADS, 1) decode_ffn_kernel(FfnArgs a) {
  using Cfg = DCfg<NT>;
  constexpr int CW = Cfg::CW, BPW = Cfg::BPW, NS = Cfg::NS, NQ = Cfg::NQ, SB = Cfg::SB, MAXSDN = Cfg::MAXSDN;
  constexpr int SBYTES = Cfg::SBYTES;
  constexpr int NCT = CW * 32;   // consumer threads (named barrier 1)
  constexpr bool FUSED = MODE != kPlanRead;
  constexpr bool DIRECT = MODE == kFusedCachedDirect;
  constexpr bool AHEAD = MODE == kAhead;
  constexpr bool CACHED = MODE == kFusedCached || DIRECT || AHEAD;
  extern __shared__ __align__(128) uint8_t smem[];
  const int d = a.d, f = a.f, T = a.T, K = a.k;
  const int RG = f / 32;            // f slices = units per expert
  const int RD = d / 32;            // row blocks of d
  const int NGU = d / 16;           // gate/up blocks per unit
  const int SGU = (NGU + SB - 1) / SB;   // gate/up stages per unit (the last may be partial)
  const int SDN = (RD + SB - 1) / SB;    // down stages per unit
  const int nks = d / 16;
  const uint64_t lim = a.wait_ns;
  uint8_t* ring = smem;
  uint2* xfrag = reinterpret_cast<uint2*>(smem + (size_t)NS * SBYTES);
  uint8_t* ovl = reinterpret_cast<uint8_t*>(xfrag) + (size_t)NT * d * 16;
  __half* hs = reinterpret_cast<__half*>(ovl + overlay_bytes<NT>(d));
  uint64_t* full = reinterpret_cast<uint64_t*>(hs + NT * 8 * kHsRow);
  uint64_t* empty = full + NS;
  uint64_t* plan_ready = empty + NS;
  uint16_t* xraw = reinterpret_cast<uint16_t*>(ovl);   // router input rows
  SelSmem* sel = reinterpret_cast<SelSmem*>(ovl);      // selection
  float* red = reinterpret_cast<float*>(ovl);          // gate/up partials [CW][NQ][32]
  float* cmb = reinterpret_cast<float*>(ovl);          // combine partials [CW][32]

  __shared__ int s_act_slot[kMaxPicks];   // slot of each distinct routed expert
  __shared__ int s_pick_act[kMaxPicks];   // [T][k] index of each pick in the distinct list
  __shared__ float s_w[kMaxPicks];        // [T][k] routing weights
  __shared__ int s_act_expert[kMaxPicks]; // expert id of each distinct routed expert
  __shared__ int s_tab[kMaxE];            // the layer's slot-table row (fused routing)
  __shared__ int s_order[kMaxPicks];      // distinct experts in unit order (resident ones first)
  __shared__ int s_mrank[kMaxPicks];      // position of each distinct expert in the miss list, -1 if resident
  __shared__ int s_n_act, s_u0, s_u1;
  __shared__ float s_wu[16];              // routing weight of each token for the current unit's expert
  __shared__ uint32_t s_calls;
  __shared__ long long s_clock;
  // s_abort: set by any warp whose bounded wait gave up (consumers then skip
  // waits and compute, the producer stops issuing).  s_cab: consumer thread
  // 0's copy of it, taken just before a named barrier, so that every branch
  // of the consumers around further barriers is the same in all of them.
  __shared__ volatile int s_abort;
  __shared__ int s_cab;
  // direct mode: ring stages the producer hands to the host-stage warps, in
  // ring order (host source, victim-slot destination, bytes (0 ends), stage)
  constexpr int NDQ = DIRECT ? NS : 1;
  __shared__ const uint8_t* s_dq_src[NDQ];
  __shared__ uint8_t* s_dq_dst[NDQ];
  __shared__ int s_dq_bytes[NDQ], s_dq_stage[NDQ];
  __shared__ uint64_t s_dq_full[NDQ], s_dq_empty[NDQ];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int GT = CACHED ? G - 1 : G;           // CTAs that take units
  const int ct = CACHED ? cta - 1 : cta;       // tile index (-1: the cache manager)
  // kAhead: whether this launch has a current call to compute and a next
  // call to route (a launch that only prepares, or only finishes, a sequence)
  const bool CUR = !AHEAD || a.has_cur != 0;
  const bool NEXT = !AHEAD || a.has_next != 0;
  const int sh0 = ct >= 0 && CUR ? shared_first(ct, RG, GT) : 0;
  const int sh1 = ct >= 0 && CUR ? shared_first(ct + 1, RG, GT) : 0;
#ifdef MOE_TIMELINE
  if (tid == 0) dtl_begin();
#endif
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], CW);
    }
    mbar_init(plan_ready, 1);
    if (DIRECT)
      for (int i = 0; i < NDQ; ++i) {
        mbar_init(&s_dq_full[i], 1);
        mbar_init(&s_dq_empty[i], 1);
      }
    s_abort = 0;
    s_cab = 0;
    mbar_init_fence();
  }
  __syncthreads();
  pdl_launch_dependents();
  auto expert_base = [&](int ai) -> const uint8_t* {   // ai < 0: the shared expert
    return ai < 0 ? a.shared_expert : a.slots + (int64_t)s_act_slot[ai] * a.expert_bytes;
  };

  if (warp == CW) {
    // ---------------- producer: every stage of the CTA's units, in order ------
    if (lane != 0 || ct < 0) return;
    uint32_t it = 0;
    bool ok = true;
    const uint64_t pol_stream = l2_evict_first_policy(), pol_keep = l2_evict_last_policy();
    auto issue_unit = [&](const uint8_t* eb, int rb) -> bool {
      const uint64_t pol = eb == a.shared_expert ? pol_keep : pol_stream;
      const uint8_t* gu = eb + gu_block_offset(rb, 0, 0, d);
      const uint8_t* dn = eb + down_block_offset(0, rb, d, f);
      for (int st = 0; st < SGU + SDN; ++st, ++it) {
        if (s_abort) return false;
        const int s = it % NS;
        const uint32_t use = it / NS;
        if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, lim)) return false;
        const uint8_t* src;
        uint32_t bytes;
        if (st < SGU) {
          const int b0 = st * SB;
          const int nb = NGU - b0 < SB ? NGU - b0 : SB;
          src = gu + (size_t)b0 * kBlockBytes;
          bytes = (uint32_t)nb * kBlockBytes;
        } else {
          const int b0 = (st - SGU) * SB;
          const int nb = RD - b0 < SB ? RD - b0 : SB;
          src = dn + (size_t)b0 * kBlockBytes;
          bytes = (uint32_t)nb * kBlockBytes;
        }
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_g2s_hint(ring + (size_t)s * SBYTES, src, bytes, &full[s], pol);
      }
      return true;
    };
    // direct mode: a missing expert's stages go to the host-stage warps
    // (source in the host pool, destination the victim slot), in ring order
    uint32_t nd = 0;   // stages handed over
    auto hand_over = [&](const uint8_t* src, uint8_t* dst, uint32_t bytes, int s) -> bool {
      const int q = nd % NDQ;
      if (nd >= (uint32_t)NDQ && !mbar_wait(&s_dq_empty[q], (nd / NDQ - 1) & 1, lim)) return false;
      s_dq_src[q] = src;
      s_dq_dst[q] = dst;
      s_dq_bytes[q] = (int)bytes;
      s_dq_stage[q] = s;
      mbar_arrive(&s_dq_full[q]);
      ++nd;
      return true;
    };
    auto issue_unit_host = [&](const uint8_t* hb, uint8_t* vb, int rb) -> bool {
      const int64_t gu = gu_block_offset(rb, 0, 0, d), dn = down_block_offset(0, rb, d, f);
      for (int st = 0; st < SGU + SDN; ++st, ++it) {
        if (s_abort) return false;
        const int s = it % NS;
        const uint32_t use = it / NS;
        if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, lim)) return false;
        int64_t off;
        uint32_t bytes;
        if (st < SGU) {
          const int b0 = st * SB;
          const int nb = NGU - b0 < SB ? NGU - b0 : SB;
          off = gu + (int64_t)b0 * kBlockBytes;
          bytes = (uint32_t)nb * kBlockBytes;
        } else {
          const int b0 = (st - SGU) * SB;
          const int nb = RD - b0 < SB ? RD - b0 : SB;
          off = dn + (int64_t)b0 * kBlockBytes;
          bytes = (uint32_t)nb * kBlockBytes;
        }
        if (!hand_over(hb + off, vb + off, bytes, s)) return false;
      }
      return true;
    };
    // the shared expert's weights never change: its units start at once
    for (int rb = sh0; rb < sh1 && ok; ++rb) ok = issue_unit(a.shared_expert, rb);
    pdl_wait();   // slots (and their contents) may have been written by earlier work
    // slots of this call's misses were written by other CTAs' generic stores
    if (CACHED) asm volatile("fence.proxy.async.global;" ::: "memory");
    if (AHEAD) {
      // the current call's plan was completed by the previous launch (visible
      // once pdl_wait returned) with every expert resident and U's order as
      // the unit order: the routed units stream at once, while the consumers
      // still route the next call
      const Plan* P = a.cur_plan;
      const int NU = CUR ? __ldcg(&P->n_act) * RG : 0;
      const int u0 = routed_first(ct, NU, RG, GT), u1 = routed_first(ct + 1, NU, RG, GT);
      for (int u = u0; u < u1 && ok; ++u)
        ok = issue_unit(a.slots + (int64_t)__ldcg(&P->act_slot[u / RG]) * a.expert_bytes, u % RG);
    } else if (ok && !mbar_wait(plan_ready, 0, lim)) {
      ok = false;
    }
    if (ok && !AHEAD) {
      MOE_TLS(4);
      const int u0 = s_u0, u1 = s_u1;
      const uint32_t jpm = (uint32_t)(2 * RG + RD);   // fetch jobs per missing expert
      const uint32_t* ready = a.counters + 1 + (size_t)(s_calls & 1u) * a.set_words + 3;
      const uint32_t* vict_w = a.counters + 1 + (size_t)(s_calls & 1u) * a.set_words + 2;
      bool have_victims = false;
      for (int u = u0; u < u1 && ok; ++u) {
        const int ai = s_order[u / RG];
        const int j = CACHED ? s_mrank[ai] : -1;
        const uint8_t* eb;
        if (j < 0) {
          eb = expert_base(ai);
        } else if (DIRECT) {
          // a missing expert: its victim slot is known once CTA 0 has
          // published the victims
          if (!have_victims) {
            if (!wait_flag_geq(vict_w, 1u, lim)) {
              ok = false;
              break;
            }
            have_victims = true;
          }
          const int64_t entry = ((int64_t)a.layer * a.E + s_act_expert[ai]) % a.pool_entries;
          uint8_t* vb = const_cast<uint8_t*>(a.slots) + (int64_t)__ldcg(&a.plan->miss_slot[j]) * a.expert_bytes;
          ok = issue_unit_host(a.host_pool + entry * a.expert_bytes, vb, u % RG);
          continue;
        } else {
          // a missing expert: every job of its fetch is done (other CTAs'
          // generic stores, ordered before the bulk copies by the proxy fence)
          if (!wait_flag_geq(&ready[j], jpm, lim)) {
            ok = false;
            break;
          }
          asm volatile("fence.proxy.async.global;" ::: "memory");
          eb = a.slots + (int64_t)__ldcg(&a.plan->miss_slot[j]) * a.expert_bytes;
        }
        ok = issue_unit(eb, u % RG);
      }
    }
    if (!ok && !s_abort) {
      set_error(a.err, DEV_TIMEOUT_BARRIER);
      s_abort = 1;
    }
    if (DIRECT && !hand_over(nullptr, nullptr, 0u, 0)) {   // no more stages: the host-stage warps stop
      set_error(a.err, DEV_TIMEOUT_BARRIER);
      s_abort = 1;
    }
    // no copy may still be in flight when the CTA exits: wait, bounded, for
    // the last ones
    for (uint32_t k = it > (uint32_t)NS ? it - NS : 0; k < it; ++k)
      if (!mbar_wait(&full[k % NS], (k / NS) & 1, lim)) set_error(a.err, DEV_TIMEOUT_BARRIER);
    MOE_TLS(5);
    return;
  }
  if (DIRECT && warp >= CW + 2) {
    // ---------------- host-stage warps (direct mode) --------------------------
    // Each stage the producer hands over is copied by these 64 threads from
    // the host pool (16-byte pieces, all of a thread's pieces in flight at
    // once) into its ring stage and into the victim slot; then one thread
    // completes the stage's full barrier (no bytes are expected on it) and
    // frees the hand-over entry.  Nothing in this call reads the victim
    // slot: every unit of a missing expert takes its stages from the host.
    if (ct < 0) return;
    const int ht = tid - (CW + 2) * 32;
    constexpr int PER = (SBYTES / 16 + 63) / 64;   // 16-byte pieces per thread of a stage
#pragma unroll 1
    for (uint32_t k = 0;; ++k) {
      const int q = k % NDQ;
      if (!__all_sync(0xffffffffu, mbar_wait(&s_dq_full[q], (k / NDQ) & 1, lim))) {
        if (lane == 0) {
          set_error(a.err, DEV_TIMEOUT_BARRIER);
          s_abort = 1;
        }
        return;
      }
      const int n = s_dq_bytes[q] / 16;
      if (n == 0) return;
      const uint4* src = reinterpret_cast<const uint4*>(s_dq_src[q]);
      uint4* dst = reinterpret_cast<uint4*>(s_dq_dst[q]);
      const int st = s_dq_stage[q];
      uint4* stg = reinterpret_cast<uint4*>(ring + (size_t)st * SBYTES);
      uint4 v[PER];
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int c = ht + 64 * i;
        if (c < n) v[i] = src[c];
      }
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int c = ht + 64 * i;
        if (c < n) {
          stg[c] = v[i];
          dst[c] = v[i];
        }
      }
      fence_proxy_async_smem();   // the stage is refilled by bulk copies later
      named_bar(3, 64);
      if (ht == 0) {
        mbar_arrive(&full[st]);
        mbar_arrive(&s_dq_empty[q]);
      }
      __syncwarp();
    }
  }
  if (AHEAD && warp >= CW + 2) {
    // ---------------- miss copies of the next call (kAhead) ------------------
    // Once CTA 0 has published the next call's victims, the two extra warps
    // of every tile CTA copy the next call's missing experts (device layout:
    // the slot's own bytes) from the host pool into their victim slots, an
    // even share of 16-byte pieces each, four in flight per thread.  The next
    // launch finds them resident; nothing in this launch reads them.
    if (ct < 0 || !NEXT) return;
    int m = 0;
    if (lane == 0) {
      // the call's tag (s_calls) is written before the consumers hand the
      // producer its units: wait for that hand-over, then for the victims
      const bool tagged = mbar_wait(plan_ready, 0, lim);
      const uint32_t* vict_w = a.counters + 1 + (size_t)(s_calls & 1u) * a.set_words + 2;
      if (!tagged || !wait_flag_geq(vict_w, 1u, lim)) {
        set_error(a.err, DEV_TIMEOUT_FLAG);
        s_abort = 1;
      } else {
        m = __ldcg(&a.plan->n_miss);
      }
    }
    __syncwarp();   // lane 0's acquire of the victims orders the other lanes' plan reads
    m = __shfl_sync(0xffffffffu, m, 0);
    const int64_t per = a.expert_bytes / 16;
    const int64_t nthr = (int64_t)GT * 64;
    const int64_t t0 = (int64_t)ct * 64 + (tid - (CW + 2) * 32);
    for (int j = 0; j < m; ++j) {
      const int64_t entry = ((int64_t)a.layer * a.E + __ldcg(&a.plan->miss_expert[j])) % a.pool_entries;
      const uint4* src = reinterpret_cast<const uint4*>(a.host_pool + entry * a.expert_bytes);
      uint4* dst = reinterpret_cast<uint4*>(const_cast<uint8_t*>(a.slots) +
                                            (int64_t)__ldcg(&a.plan->miss_slot[j]) * a.expert_bytes);
      int64_t c = t0;
      for (; c + 3 * nthr < per; c += 4 * nthr) {
        const uint4 v0 = src[c], v1 = src[c + nthr], v2 = src[c + 2 * nthr], v3 = src[c + 3 * nthr];
        dst[c] = v0;
        dst[c + nthr] = v1;
        dst[c + 2 * nthr] = v2;
        dst[c + 3 * nthr] = v3;
      }
      for (; c < per; c += nthr) dst[c] = src[c];
    }
    return;
  }
  if (warp == CW + 1) {
    // ---------------- control: the call's plan, stamps and counters ---------
    // (every key resident: CTA 0 publishes them off the units' path)
    if (MODE != kFusedResident || cta != 0) return;
    named_bar(2, NCT + 32);   // the consumers have selected
    if (s_abort) return;
    Plan* P = a.plan;
    const long long clk = s_clock;
    const int n_act = s_n_act;
    for (int i = lane; i < T * K; i += 32) {
      P->idx[i] = s_act_expert[s_pick_act[i]];
      P->w[i] = s_w[i];
      P->pick_act[i] = s_pick_act[i];
    }
    for (int i = lane; i < n_act; i += 32) {
      P->act_expert[i] = s_act_expert[i];
      P->act_slot[i] = s_act_slot[i];
      P->act_hit[i] = 1;
      a.stamp[s_act_slot[i]] = clk;
    }
    if (lane == 0) {
      P->n_act = n_act;
      P->n_miss = 0;
      P->T = T;
      P->clock = clk;
      P->token_hits = (int64_t)T * K;
      P->token_misses = 0;
      a.stats[ST_CALLS] += 1;
      a.stats[ST_TOK_HIT] += (int64_t)T * K;
      a.stats[ST_DIST_HIT] += n_act;
      *a.clock = clk + 1;
      *a.counters = s_calls + 1;   // every CTA read the count before the router barrier
    }
    return;
  }

  // =================== consumers: warps 0 .. CW-1 ===========================
  const int E = a.E;
  // Every load of the prologue is issued before any of them is used.  Static
  // inputs first: with every key resident the slot-table row, and the first
  // block of this warp's router row.
  constexpr int kTabPer = (kMaxE + NCT - 1) / NCT;
  int tv[kTabPer];
  uint4 wfirst[8];
  float wbias = 0.f;
  if (FUSED) {
    if (!CACHED) {
#pragma unroll
      for (int q = 0; q < kTabPer; ++q) {
        const int i = tid + q * NCT;
        tv[q] = i < E ? a.table[(size_t)a.layer * E + i] : -1;
      }
    }
    const int e = cta + G * warp;
    if (e < E) {
      router_load_block(a.wr + (size_t)e * d, 0, d, lane, wfirst);
      wbias = a.bias[e];
    }
  }
  // x, the clock and the counters may be written by earlier work in the stream
  pdl_wait();
  if (FUSED && CACHED) {   // the slot table changes with every commit: read it after the previous call
#pragma unroll
    for (int q = 0; q < kTabPer; ++q) {
      const int i = tid + q * NCT;
      tv[q] = i < E ? a.table[(size_t)a.layer * E + i] : -1;
    }
  }
  uint32_t calls = 0;
  long long clk = 0;
  if (tid == 0) {
    calls = *a.counters;
    if (FUSED && cta == 0) clk = (long long)*a.clock;
  }
  // x (bf16) staged for the router, rows xs apart, and as fp16 B fragments of
  // the gate/up products, zero past T.  Fragment word (nt, kstep, lane, reg)
  // holds token nt*8 + lane/4, inputs kstep*16 + 2*(lane%4) + 8*reg and the
  // next one, so the 16-byte chunk c of token n fills reg c%2 of k-step c/2
  // for lanes 4(n%8) + j.
  const int xs = x_row_elems(d);
  const int cpr = d / 8;
  uint32_t* const xfw = reinterpret_cast<uint32_t*>(xfrag);
  constexpr int kXPer = (NT * 8 * 256 + NCT - 1) / NCT;   // 16-byte chunks per thread (d <= 2048)
  uint4 xv[kXPer];
  uint4 xn[AHEAD ? kXPer : 1];   // kAhead: the next call's tokens, for the router
#pragma unroll
  for (int q = 0; q < kXPer; ++q) {
    const int i = tid + q * NCT;
    if (i < T * cpr) {
      const int n = i / cpr, c = i - n * cpr;
      if (CUR) xv[q] = __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)n * d + c * 8));
      if (AHEAD && NEXT) xn[AHEAD ? q : 0] = __ldg(reinterpret_cast<const uint4*>(a.x_route + (size_t)n * d + c * 8));
    }
  }
  if (FUSED) {
#pragma unroll
    for (int q = 0; q < kTabPer; ++q)
      if (tid + q * NCT < E) s_tab[tid + q * NCT] = tv[q];
  }
  if (tid == 0) {
    s_calls = calls;
    s_clock = clk;
  }
  auto put_x = [&](int n, int c, uint4 v, uint4 vr) {
    if (FUSED && NEXT) *reinterpret_cast<uint4*>(xraw + (size_t)n * xs + c * 8) = AHEAD ? vr : v;
    if (!CUR) return;
    uint32_t* w = xfw + ((((size_t)(n >> 3) * nks + (c >> 1)) * 32 + (n & 7) * 4) << 1) + (c & 1);
    w[0] = pack_half2_from_bf16(v.x);
    w[2] = pack_half2_from_bf16(v.y);
    w[4] = pack_half2_from_bf16(v.z);
    w[6] = pack_half2_from_bf16(v.w);
  };
#pragma unroll
  for (int q = 0; q < kXPer; ++q) {
    const int i = tid + q * NCT;
    if (i < T * cpr) {
      const int n = i / cpr, c = i - n * cpr;
      put_x(n, c, xv[q], xn[AHEAD ? q : 0]);
    }
  }
  // zero fragments of the token slots T .. NT*8-1: 32 contiguous bytes per
  // (n-tile, k-step, token)
  {
    const int nz = NT * 8 - T;
    for (int i = tid; i < nz * nks * 2; i += NCT) {
      const int h = i & 1, q = i >> 1, kstep = q % nks, n = T + q / nks;
      reinterpret_cast<uint4*>(xfw + ((((size_t)(n >> 3) * nks + kstep) * 32 + (n & 7) * 4) << 1))[h] =
          make_uint4(0u, 0u, 0u, 0u);
    }
  }
  named_bar(1, NCT);
  MOE_TL0(1);
  // this call's counter set; the fused kernel's CTA 0 zeroes the other one
  // (the previous call's, complete by now) for the next call
  const uint32_t call_set = FUSED ? (s_calls & 1u) : ((s_calls - 1u) & 1u);
  uint32_t* const cset = a.counters + 1 + (size_t)call_set * a.set_words;
  uint32_t* const vict = cset + 2;      // cache mode: the misses' victims are published
  uint32_t* const ready = cset + 3;     // cache mode: finished fetch jobs of each miss
  if (FUSED && cta == 0) {
    uint32_t* other = a.counters + 1 + (size_t)(call_set ^ 1u) * a.set_words;
    for (int i = tid; i < a.set_words; i += NCT) other[i] = 0;
  }

  if (FUSED && NEXT) {
    // ---- router rows e = cta + G*j, one warp per row -----------------------
    for (int j = warp;; j += CW) {
      const int e = cta + G * j;
      if (e >= E) break;
      const uint16_t* wrow = a.wr + (size_t)e * d;
      if (j != warp) {
        router_load_block(wrow, 0, d, lane, wfirst);
        wbias = a.bias[e];
      }
      // each logit goes out as one (call tag, value) word: readers poll the
      // word itself, so no counter and no fence separates router and
      // selection.  A test hook can hold back CTA 0's logits so that every
      // reader's bounded wait runs out.
      uint64_t* const tl = a.tlogits;
      const uint32_t tag = s_calls;
      const bool hold = a.dbg_hold_router && cta == 0;
      router_row(wrow, wfirst, xraw, xs, wbias, T, d, lane, [&](int t, float v) {
        if (!hold) st_relaxed_u64(tl + (size_t)t * E + e, tag_word(tag, v));
      });
    }
    MOE_TL0(2);
  }

  // ---- units: the CTA's shared-expert units, then (after the routing
  // result) its routed units.  Warp w owns the row blocks
  // sd*SB + w*BPW + j of y (sd < SDN, j < BPW) in every down stage.
  float yacc[MAXSDN][BPW][NT][2][4];
#pragma unroll
  for (int sd = 0; sd < MAXSDN; ++sd)
#pragma unroll
    for (int j = 0; j < BPW; ++j)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int i = 0; i < 4; ++i) yacc[sd][j][nt][mt][i] = 0.f;
  const int gq = lane >> 2, cq = lane & 3;
  uint32_t it = 0;   // ring stage counter (the producer's order)
  bool routed = false;
  int u = sh0, u_end = sh1;
  // waits for stage s (bounded); false once any warp of the CTA gave up.
  // The answer is the same for all lanes of the warp (the MMAs that follow
  // need the whole warp).
  auto stage_wait = [&](int s, uint32_t par) -> bool {
    bool got = false;
    if (!s_abort) {
      got = mbar_wait(&full[s], par, lim);
      if (!got) {
        set_error(a.err, DEV_TIMEOUT_BARRIER);
        s_abort = 1;
      }
    }
    return __all_sync(0xffffffffu, got);
  };
  for (;;) {
    if (u >= u_end) {
      if (routed) break;
      routed = true;
      // ================= the routing result ===============================
      if (AHEAD && cta == 0 && !NEXT) {   // no next call to route (the call count moves on after the launch)
        MOE_TL_FLUSH(cta);
        return;
      }
      bool planned = false;   // warp 0: the producer already has its units
      if (FUSED && !(AHEAD && cta != 0)) {
        if (tid == 0) {
          s_cab = s_abort;
          MOE_TLS(6);
        }
        named_bar(1, NCT);
        if (!s_cab) {
          bool failed = false;
          if (T == 1 && K <= 2 * CW)
            select_one_token<NCT, CW>(a.tlogits, s_calls, lim, &failed, E, K, sel);
          else
            select_call<NCT>(TaggedLogits{a.tlogits, s_calls, lim, &failed}, T, E, K, sel);
          if (failed) {   // some logits never arrived
            set_error(a.err, DEV_TIMEOUT_FLAG);
            s_abort = 1;
          }
          MOE_TL0(16);
          const int n_act = sel->n_act;
          if (MODE == kFusedResident && warp == 0) {
            // every expert resident: the producer needs only U's slots and
            // this CTA's unit range, so warp 0 hands them over at once; the
            // routing weights and the rest of the bookkeeping follow while
            // the first copies are in flight.  (A selection that timed out
            // still yields valid ids: the units run, the call reports the
            // error.)
            for (int i = lane; i < n_act; i += 32) {
              int slot = s_tab[sel->act[i]];
              if (slot < 0) {
                set_error(a.err, DEV_NOT_RESIDENT);
                slot = 0;
              }
              s_act_slot[i] = slot;
              s_act_expert[i] = sel->act[i];
              s_order[i] = i;
              s_mrank[i] = -1;
            }
            __syncwarp();
            if (lane == 0) {
              const int NU = n_act * RG;
              s_u0 = routed_first(ct, NU, RG, GT);
              s_u1 = routed_first(ct + 1, NU, RG, GT);
              mbar_arrive(plan_ready);
              MOE_TLS(8);
            }
            __syncwarp();
            planned = true;
          }
          for (int i = tid; i < T * K; i += NCT) {
            const int id = sel->sel_id[i / K][i % K];
            s_pick_act[i] = dsel_act_index(sel, id);
            s_w[i] = sel->sel_w[i / K][i % K];
          }
          if (MODE != kFusedResident) {
            for (int i = tid; i < n_act; i += NCT) {
              int slot = s_tab[sel->act[i]];
              if (slot < 0 && !CACHED) {
                set_error(a.err, DEV_NOT_RESIDENT);
                slot = 0;
              }
              s_act_slot[i] = slot;   // cached: -1 marks a miss until CTA 0 assigns its victim
              s_act_expert[i] = sel->act[i];
            }
          }
          if (tid == 0) s_n_act = n_act;
        } else if (tid == 0) {
          s_n_act = 0;
        }
        named_bar(1, NCT);
        if (tid == 0) {   // a selection that timed out counts as no selection
          s_cab = s_abort;
          if (s_cab) s_n_act = 0;
        }
        named_bar(1, NCT);
        if (MODE == kFusedResident && cta == 0) named_bar_arrive(2, NCT + 32);
      } else {
        // the routing plan is complete and visible (kAhead: the current
        // call's, written by the previous launch; all its experts resident)
        const Plan* P = AHEAD ? a.cur_plan : a.plan;
        if (CUR) {
          for (int i = tid; i < kMaxPicks; i += NCT) s_act_slot[i] = P->act_slot[i];
          for (int i = tid; i < T * K; i += NCT) {
            s_pick_act[i] = P->pick_act[i];
            s_w[i] = P->w[i];
          }
        }
        if (tid == 0) {
          s_n_act = CUR ? P->n_act : 0;
          s_cab = s_abort;
        }
        named_bar(1, NCT);
      }
      MOE_TL0(7);
      const int n_act = s_n_act;
      // unit order: resident experts first, then the misses (ascending id
      // within each), and each miss's position in the miss list
      if (warp == 0 && !planned) {
        int nh = 0, nm = 0;
        for (int i0 = 0; i0 < n_act; i0 += 32) {
          const int i = i0 + lane;
          const bool miss = CACHED && i < n_act && s_act_slot[i] < 0;
          const uint32_t bm = __ballot_sync(0xffffffffu, miss);
          const uint32_t bh = __ballot_sync(0xffffffffu, i < n_act && !miss);
          const uint32_t below = (1u << lane) - 1u;
          if (i < n_act) s_mrank[i] = miss ? nm + __popc(bm & below) : -1;
          if (i < n_act && !miss) s_order[nh + __popc(bh & below)] = i;
          nh += __popc(bh);
          nm += __popc(bm);
          __syncwarp();
        }
        for (int i0 = 0; i0 < n_act; i0 += 32) {
          const int i = i0 + lane;
          const bool miss = CACHED && i < n_act && s_act_slot[i] < 0;
          const uint32_t bm = __ballot_sync(0xffffffffu, miss);
          if (miss) s_order[nh + __popc(bm & ((1u << lane) - 1u))] = i;
          nh += __popc(bm);
          __syncwarp();
        }
      }
      const int n_miss = named_bar_count(1, NCT, CACHED && tid < n_act && s_act_slot[tid] < 0);
      if (CACHED && cta == 0) {
        if (!s_cab)
          cache_manager<NCT>(a, n_act, n_miss, s_act_expert, s_act_slot, s_pick_act, s_w, s_clock, s_calls, ring,
                             (size_t)NS * SBYTES, vict);
        MOE_TL_FLUSH(cta);
        return;   // CTA 0 takes no units
      }
      // this CTA's routed units, handed to the producer (it streams the
      // resident experts' units at once and waits per missing expert)
      if (tid == 0 && !planned) {
        const int NU = s_cab ? 0 : n_act * RG;
        s_u0 = routed_first(ct, NU, RG, GT);
        s_u1 = routed_first(ct + 1, NU, RG, GT);
        mbar_arrive(plan_ready);
        MOE_TLS(8);
      }
      if (CACHED && !DIRECT && n_miss > 0) {
        // fetch jobs of the misses, spread over the tile CTAs, once CTA 0 has
        // published the victims
        if (tid == 0) {
          if (!s_cab && !wait_flag_geq(vict, 1u, lim)) {
            set_error(a.err, DEV_TIMEOUT_FLAG);
            s_abort = 1;
          }
          s_cab = s_abort;
        }
        named_bar(1, NCT);
        if (!s_cab) {
          const int J = n_miss * (2 * RG + RD);
          constexpr int KPC = (14 * 2048 / 16 + NCT - 1) / NCT;   // 16-byte chunks per thread of a job
          const MissFetch mf{a.plan->miss_expert, a.plan->miss_slot, a.host_pool, a.pool_entries,
                             const_cast<uint8_t*>(a.slots), a.expert_bytes, a.layer, a.E, d, f};
          pull_jobs<NCT, KPC>(mf, (int)((int64_t)ct * J / GT), (int)((int64_t)(ct + 1) * J / GT), ovl, ready);
        }
        MOE_TL0(12);
      }
      named_bar(1, NCT);
      u = s_u0;
      u_end = s_u1;
      continue;
    }
    // ================= one unit: expert ai (-1: shared), slice rb ==========
    const int ai = routed ? s_order[u / RG] : -1;
#ifdef MOE_TIMELINE
    const int tlu = routed ? u - s_u0 : -1;   // stamps of the first two routed units
    if (tlu == 1) MOE_TL0(17);
#endif
    // the routing weight of each token for this expert (0 for a token not
    // routed to it); read in the h step, after the next barrier
    if (warp == 0 && lane < NT * 8) {
      float wt = 0.f;
      if (lane < T) {
        if (ai < 0) {
          wt = a.shared_weight;
        } else {
          for (int k2 = 0; k2 < K; ++k2)
            if (s_pick_act[lane * K + k2] == ai) wt = s_w[lane * K + k2];
        }
      }
      s_wu[lane] = wt;
    }
    __syncwarp();   // warp 0's MMAs below run on the whole warp again
    // gate/up: each warp sums its blocks' input groups
    float acc[2][NT][2][4];   // g and u of the slice's 32 rows
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[j][nt][mt][i] = 0.f;
#pragma unroll 1
    for (int st = 0; st < SGU; ++st, ++it) {
      const int s = it % NS;
      // this warp's blocks: Wg and Wu of input groups (st*SB + warp*BPW)/2 + p
      if (stage_wait(s, (it / NS) & 1)) {
        const uint8_t* sp = ring + (size_t)s * SBYTES;
#pragma unroll
        for (int p = 0; p < BPW / 2; ++p) {
          const int b = warp * BPW + 2 * p;   // a stage's blocks come in (Wg, Wu) pairs
          if (st * SB + b < NGU) {
            const int gi = (st * SB + b) / 2;
            uint2 bx[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              bx[nt][0] = xfrag[((size_t)nt * nks + gi * 2 + 0) * 32 + lane];
              bx[nt][1] = xfrag[((size_t)nt * nks + gi * 2 + 1) * 32 + lane];
            }
            block_pair_mma<NT>(sp + b * kBlockBytes, sp + (b + 1) * kBlockBytes, lane, bx, acc[0], acc[1]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      __syncwarp();   // the next stage's MMAs run on the whole warp
    }
#ifdef MOE_TIMELINE
    if (tlu == 0) MOE_TL0(13);
    if (tlu == 1) MOE_TL0(18);
#endif
    // partials -> shared memory, [warp][q][lane] with q = ((j*NT + nt)*2 + mt)*4 + i.
    // They overlay the staged router input: in the CTA's first shared unit
    // the warps first wait until every warp is done with its router rows.
    if (FUSED && !routed && u == sh0) named_bar(1, NCT);
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int i = 0; i < 4; ++i)
            red[((size_t)warp * NQ + ((j * NT + nt) * 2 + mt) * 4 + i) * 32 + lane] = acc[j][nt][mt][i];
    named_bar(1, NCT);
    // h of the slice for every (row, token): g and u summed over the warps in
    // warp order, times the token's routing weight for this expert (0 for a
    // token not routed to it), fp16
    for (int p = tid; p < 256 * NT; p += NCT) {
      const int ln = p & 31, r8 = p >> 5;   // r8 = (nt*2 + mt)*4 + i
      float g = 0.f, uu = 0.f;
      // every warp holds both (j = 0: Wg, j = 1: Wu)
#pragma unroll
      for (int w = 0; w < CW; ++w) {
        g += red[((size_t)w * NQ + r8) * 32 + ln];
        uu += red[((size_t)w * NQ + NT * 8 + r8) * 32 + ln];
      }
      const int i = r8 & 3, mt = (r8 >> 2) & 1, nt = r8 >> 3;
      const int row = mt * 16 + (ln >> 2) + 8 * (i >> 1);
      const int tok = nt * 8 + 2 * (ln & 3) + (i & 1);
      // silu with the fast exponential and division (relative error ~2^-21,
      // far below the fp16 rounding of h)
      const float hv = __fdividef(g, 1.f + __expf(-g)) * uu * s_wu[tok];
      hs[tok * kHsRow + row] = __float2half_rn(hv);
    }
    named_bar(1, NCT);
#ifdef MOE_TIMELINE
    if (tlu == 0) MOE_TL0(14);
    if (tlu == 1) MOE_TL0(19);
#endif
    // B fragments of the down products (k = the slice's 32 rows of f)
    uint2 hf[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const uint32_t* hr = reinterpret_cast<const uint32_t*>(hs + (nt * 8 + gq) * kHsRow);
      hf[nt][0].x = hr[cq];
      hf[nt][0].y = hr[cq + 4];
      hf[nt][1].x = hr[cq + 8];
      hf[nt][1].y = hr[cq + 12];
    }
    // down: row blocks sd*SB + b of d, b = warp*BPW + j
#pragma unroll
    for (int sd = 0; sd < MAXSDN; ++sd) {
      if (sd < SDN) {
        const int s = it % NS;
        if (stage_wait(s, (it / NS) & 1)) {
          const uint8_t* sp = ring + (size_t)s * SBYTES;
#pragma unroll
          for (int p = 0; p < BPW / 2; ++p) {
            const int b = warp * BPW + 2 * p;   // RD and the stage's blocks are even: both or neither
            if (sd * SB + b < RD)
              block_pair_mma<NT>(sp + b * kBlockBytes, sp + (b + 1) * kBlockBytes, lane, hf, yacc[sd][2 * p],
                                 yacc[sd][2 * p + 1]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        __syncwarp();   // the next stage's MMAs run on the whole warp
        ++it;
      }
    }
#ifdef MOE_TIMELINE
    if (tlu == 0) MOE_TL0(15);
    if (tlu == 1) MOE_TL0(20);
#endif
    ++u;
  }
  MOE_TL0(9);
  if (!CUR) {   // a launch that only routes the next call: no output
    MOE_TL_FLUSH(cta);
    return;
  }

  // ---- this CTA's partial of y -> ypart[ct][t][row], (call tag, value)
  // words that the combining CTAs poll: no counter and no fence
  uint64_t* const yp = a.ypart + (size_t)ct * T * d;
  const uint32_t tag = s_calls;
#pragma unroll
  for (int sd = 0; sd < MAXSDN; ++sd)
#pragma unroll
    for (int j = 0; j < BPW; ++j) {
      const int rbd = sd * SB + warp * BPW + j;
      if (sd < SDN && rbd < RD) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int tok = nt * 8 + 2 * cq + (i & 1);
              if (tok < T)
                st_relaxed_u64(yp + (size_t)tok * d + rbd * 32 + mt * 16 + gq + 8 * (i >> 1),
                               tag_word(tag, yacc[sd][j][nt][mt][i]));
            }
      }
    }
  if (tid == 0) {
    s_cab = s_abort;
    MOE_TLS(10);
  }
  named_bar(1, NCT);
  if (s_cab) {
    MOE_TL_FLUSH(cta);
    return;
  }
  // ---- combine: item (t, rb) = t * RD + rb for items ct, ct + GT, ...; warp
  // w adds the partials of CTAs [w*GT/CW, (w+1)*GT/CW) in order, then warp 0
  // adds the warps' sums in order
  const size_t cstride = (size_t)T * d;
  const int c0 = warp * GT / CW, c1 = (warp + 1) * GT / CW;
  for (int item = ct; item < T * RD; item += GT) {
    const int t = item / RD, rbd = item - t * RD;
    const uint64_t* src = a.ypart + (size_t)t * d + rbd * 32 + lane;
    float v = 0.f;
    bool failed = false;
    // the partials of a batch are read together, in rounds until each
    // carries this call's tag (one batch covers a warp's share on grids of
    // up to 160 CTAs), then added in CTA order
    constexpr int kBatch = (160 + CW - 1) / CW;
    for (int cb = c0; cb < c1; cb += kBatch) {
      float pv[kBatch];
      tagged_values<kBatch>(src + (size_t)cb * cstride, cstride, c1 - cb < kBatch ? c1 - cb : kBatch, tag, lim,
                            &failed, pv);
#pragma unroll
      for (int q = 0; q < kBatch; ++q)
        if (cb + q < c1) v += pv[q];
    }
    if (failed) {
      set_error(a.err, DEV_TIMEOUT_FLAG);
      s_abort = 1;
    }
    cmb[warp * 32 + lane] = v;
    named_bar(1, NCT);
    if (warp == 0) {
      float y = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < CW; ++w2) y += cmb[w2 * 32 + lane];
      a.y[(size_t)t * d + rbd * 32 + lane] = y;
    }
    named_bar(1, NCT);
  }
  MOE_TL0(11);
  MOE_TL_FLUSH(cta);
}

#ifdef MOE_TIMELINE
extern "C" int moe_debug_timeline_ffn(unsigned long long* out) {
  return (int)cudaMemcpyFromSymbol(out, g_ffn_timeline, sizeof(g_ffn_timeline));
}
#endif

// After a kAhead launch without a next call (no cache step ran in it) the
// call count moves on in a launch of its own, ordered after it on the
// stream, so that no CTA of that launch can read two different counts.
__global__ void calls_bump_kernel(uint32_t* counters) { *counters += 1u; }

cudaError_t launch_calls_bump(uint32_t* counters, cudaStream_t s) {
  calls_bump_kernel<<<1, 1, 0, s>>>(counters);
  return cudaGetLastError();
}

template <int NT, int MODE>
static cudaError_t launch_nt(const FfnArgs& a, cudaStream_t s, bool pdl, int grid) {
  constexpr int NCT = DCfg<NT>::CW * 32;
  const size_t smem = ffn_smem_bytes<NT>(a.d);
  if (a.d % 256 != 0 || a.d > kMaxRD * 32 || a.f % 32 != 0 || a.T > NT * 8 || a.T * a.k > NCT)
    return cudaErrorInvalidValue;
  cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(decode_ffn_kernel<NT, MODE>), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(KCfg<NT, MODE>::THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, decode_ffn_kernel<NT, MODE>, a);
}

cudaError_t launch_decode_ffn(const FfnArgs& a, cudaStream_t s, bool pdl) {
  if (a.grid <= 0 || (a.cached && (!a.fused || a.grid < 2))) return cudaErrorInvalidValue;
  if (a.T <= 8) {
    if (!a.fused) return launch_nt<1, kPlanRead>(a, s, pdl, a.grid);
    if (a.ahead) return launch_nt<1, kAhead>(a, s, pdl, a.grid);
    if (!a.cached) return launch_nt<1, kFusedResident>(a, s, pdl, a.grid);
    return a.direct ? launch_nt<1, kFusedCachedDirect>(a, s, pdl, a.grid) : launch_nt<1, kFusedCached>(a, s, pdl, a.grid);
  }
  if (!a.fused) return launch_nt<2, kPlanRead>(a, s, pdl, a.grid);
  if (a.ahead) return launch_nt<2, kAhead>(a, s, pdl, a.grid);
  if (!a.cached) return launch_nt<2, kFusedResident>(a, s, pdl, a.grid);
  return a.direct ? launch_nt<2, kFusedCachedDirect>(a, s, pdl, a.grid) : launch_nt<2, kFusedCached>(a, s, pdl, a.grid);
}

// Whether one CTA of every decode-kernel variant fits on an SM at hidden
// size d: the kernel's grid-wide counters need all of its CTAs (one per SM)
// resident at once.
cudaError_t decode_ffn_fits(int d, bool* fits) {
  *fits = true;
  int n = 0;
  cudaError_t e;
#define MOE_FIT(NTV, MODEV)                                                                                   \
  e = ensure_dyn_smem(reinterpret_cast<const void*>(decode_ffn_kernel<NTV, MODEV>), ffn_smem_bytes<NTV>(d)); \
  if (e != cudaSuccess) return e;                                                                             \
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_ffn_kernel<NTV, MODEV>, KCfg<NTV, MODEV>::THREADS, \
                                                    ffn_smem_bytes<NTV>(d));                                   \
  if (e != cudaSuccess) return e;                                                                             \
  if (n < 1) *fits = false;
  MOE_FIT(1, kPlanRead)
  MOE_FIT(1, kFusedResident)
  MOE_FIT(1, kFusedCached)
  MOE_FIT(1, kFusedCachedDirect)
  MOE_FIT(1, kAhead)
  MOE_FIT(2, kPlanRead)
  MOE_FIT(2, kFusedResident)
  MOE_FIT(2, kFusedCached)
  MOE_FIT(2, kFusedCachedDirect)
  MOE_FIT(2, kAhead)
#undef MOE_FIT
  return cudaSuccess;
}

}  // namespace moe
