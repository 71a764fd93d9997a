// Device helpers shared by the kernels: PTX wrappers (mbarrier, bulk copy,
// acquire/release, programmatic dependent launch, mma.sync), the device
// weight layout of an expert slot, and bounded waits.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace moe {

// ----------------------------------------------------------------- errors --
// Device error codes written to the context's error word.
enum DevErr : uint32_t {
  DEV_OK = 0,
  DEV_TIMEOUT_BARRIER = 1,   // smem mbarrier wait gave up
  DEV_TIMEOUT_FLAG = 2,      // global flag wait gave up
  DEV_NOT_RESIDENT = 3,      // all-resident mode found a missing key
  DEV_BAD_PLAN = 4,
};

// Bounded waits give up after this many nanoseconds of %globaltimer.
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Optional phase timeline (build with -DMOE_TIMELINE): %globaltimer stamps
// written to a per-file device array [rows][16] that a debug entry point
// (moe_debug_timeline_*, present only in such builds) copies out.
#ifdef MOE_TIMELINE
#define MOE_TL(arr, row, slot) ((arr)[(row)][(slot)] = globaltimer())
#else
#define MOE_TL(arr, row, slot) ((void)0)
#endif

__device__ __forceinline__ void set_error(uint32_t* err, uint32_t code) {
  atomicCAS(err, 0u, code);
}

// ------------------------------------------------------------ smem/mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of an mbarrier; false if the wait gave up after
// `limit_ns` of %globaltimer.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > limit_ns) return false;
  }
  return true;
}

// Bulk (non-tensor) TMA copy global -> shared, completing on an mbarrier.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// L2 eviction policies: data read once per call (routed expert weights)
// leaves first; data every call of a layer reads again (router rows, the
// shared expert) stays longest.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// bulk_g2s with an L2 cache policy
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 16-byte read-only load with an L2 cache policy
__device__ __forceinline__ uint4 ld_nc_v4_hint(const void* p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}

// ------------------------------------------------- global memory ordering --
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t atom_acq_rel_add(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// CTA-scope release store / acquire load on shared memory
__device__ __forceinline__ void st_release_cta_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_cta_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}

// Wait until *flag >= target (acquire); false if the wait gave up after
// `limit_ns` of %globaltimer.  The first polls run back to back (a grid
// barrier usually completes within a few hundred nanoseconds).
__device__ __forceinline__ bool wait_flag_geq(const uint32_t* flag, uint32_t target,
                                              uint64_t limit_ns = kWaitLimitNs) {
  if (ld_acquire_u32(flag) >= target) return true;
  const uint64_t t0 = globaltimer();
  int spins = 0;
  while (ld_acquire_u32(flag) < target) {
    if (++spins > 64) __nanosleep(32);
    if (globaltimer() - t0 > limit_ns) return false;
  }
  return true;
}

// 64-bit relaxed (gpu scope) accesses: a (tag, value) word written by one
// CTA and polled by others; the word is read and written whole, so a reader
// that sees the tag sees the value that came with it.
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t tag_word(uint32_t tag, float v) {
  return ((uint64_t)tag << 32) | __float_as_uint(v);
}
// Values of the tagged words base[j * stride], j < n (n <= N), once each
// carries `tag`.  All n are loaded together; while some still carry an older
// tag, those are reloaded together (one round per L2 round trip), bounded by
// limit_ns of %globaltimer.  Words j >= n read as 0.  On a time-out *failed
// is set and the values are meaningless.  (Polling one word at a time costs
// a round trip per word: with 10-20 words per lane that is several times
// slower than these rounds.)
template <int N>
__device__ __forceinline__ void tagged_values(const uint64_t* base, size_t stride, int n, uint32_t tag,
                                              uint64_t limit_ns, bool* failed, float (&v)[N]) {
  static_assert(N <= 32, "one bit per word");
  uint64_t w[N];
  uint32_t miss = 0;
#pragma unroll
  for (int j = 0; j < N; ++j)
    if (j < n) w[j] = ld_relaxed_u64(base + (size_t)j * stride);
#pragma unroll
  for (int j = 0; j < N; ++j)
    if (j < n && (uint32_t)(w[j] >> 32) != tag) miss |= 1u << j;
  if (miss) {
    const uint64_t t0 = globaltimer();
    do {
      if (globaltimer() - t0 > limit_ns) {
        *failed = true;
        break;
      }
#pragma unroll
      for (int j = 0; j < N; ++j)
        if (miss >> j & 1u) w[j] = ld_relaxed_u64(base + (size_t)j * stride);
      uint32_t still = 0;
#pragma unroll
      for (int j = 0; j < N; ++j)
        if ((miss >> j & 1u) && (uint32_t)(w[j] >> 32) != tag) still |= 1u << j;
      miss = still;
    } while (miss);
  }
#pragma unroll
  for (int j = 0; j < N; ++j) v[j] = j < n ? __uint_as_float((uint32_t)w[j]) : 0.f;
}

// orders this thread's earlier generic-proxy shared-memory accesses (and
// those it synchronised with) before its later async-proxy (TMA) accesses
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// named barrier among `count` threads (multiple of 32)
__device__ __forceinline__ void named_bar(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// arrival on a named barrier without waiting (the waiting side uses named_bar)
__device__ __forceinline__ void named_bar_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// named barrier that also counts the threads whose `pred` is true
__device__ __forceinline__ int named_bar_count(int id, int count, bool pred) {
  int n;
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.popc.u32 %0, %2, %3, p;\n\t}"
      : "=r"(n)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return n;
}

// Barrier of the `nth` threads that run a block-level step: the whole CTA
// (__syncthreads) when nth is 0, else named barrier 1 among nth threads.
template <int NTH>
__device__ __forceinline__ void step_bar() {
  if constexpr (NTH == 0) __syncthreads();
  else named_bar(1, NTH);
}
template <int NTH>
__device__ __forceinline__ int step_bar_count(bool pred) {
  if constexpr (NTH == 0) return __syncthreads_count(pred);
  else return named_bar_count(1, NTH, pred);
}

// --------------------------------------------- programmatic dependent launch
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------ tensor cores --
// D = A(16x16, row) * B(16x8, col) + C, fp16 inputs, fp32 accumulate.
// (not volatile: a pure register operation, so the compiler may interleave
// independent products to hide their latency)
__device__ __forceinline__ void mma_16816(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1,
                                          const float c[4]) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
        "f"(c[3]));
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  // (a & b) | c
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// ------------------------------------------------- device weight layout ----
// An expert slot holds the same B_x bytes as the canonical format, re-laid
// out in "blocks" of 32 rows x 32 inputs (one quantisation group per row),
// 448 bytes each:
//   bytes [0, 384): three planes of 32 lane words, word (j, lane) at j*128 +
//     4*lane.  The 96 bits (w0, w1, w2) of lane l = 4g + c hold the 32 codes
//     of the mma.sync m16n8k16 A fragments of that lane for the block's two
//     16-row tiles (mt) and two 16-input steps (ks): pair p = mt*8 + ks*4 + r
//     (r = fragment register 0..3) is (row mt*16 + g + 8*(r&1),
//     inputs k0 = ks*16 + 2c + 8*(r>>1) and k0+1).  Pairs 0..14 sit in word
//     p/5, field p%5: the k0 code at bits [3f, 3f+3), the k0+1 code at bits
//     [16+3f, 16+3f+3).  Pair 15 uses the spare bits: k0 code bit b is bit 15
//     of word b, k0+1 code bit b is bit 31 of word b.
//   bytes [384, 448): fp16 scales, row-group g8 (0..7) at 384 + 8*g8 holding
//     the scales of rows g8, g8+8, g8+16, g8+24.
// Section order in a slot: gate/up part, for row-block rb (f/32) and group gi
// (d/32): the Wg block then the Wu block; then the down part, for input
// group gi (f/32) and row-block rb (d/32): the Wd block.  So the gate/up
// rows of one 32-row slice of f and the down columns of the same slice are
// two contiguous runs of bytes.
constexpr int kBlockBytes = 448;
constexpr int kBlockCodeBytes = 384;

__host__ __device__ __forceinline__ int64_t gu_block_offset(int rb, int gi, int mat, int d) {
  return ((int64_t)(rb * (d / 32) + gi) * 2 + mat) * kBlockBytes;
}
__host__ __device__ __forceinline__ int64_t down_block_offset(int rb, int gi, int d, int f) {
  return (int64_t)(f / 32) * (d / 32) * 2 * kBlockBytes + (int64_t)(gi * (d / 32) + rb) * kBlockBytes;
}

// fp16 constants of the code -> value conversion (see dequant_block)
constexpr uint32_t kMagic = 0x64006400u;     // 1024.0 | 1024.0
constexpr uint32_t kOne2 = 0x3C003C00u;      // 1.0
constexpr uint32_t kNeg1028 = 0xE404E404u;   // -1028.0
constexpr uint32_t kEighth2 = 0x30003000u;   // 0.125
constexpr uint32_t kNeg132 = 0xD820D820u;    // -132.0
constexpr uint32_t kSixtyFourth2 = 0x24002400u;  // 1/64
constexpr uint32_t kNeg20 = 0xCD00CD00u;     // -20.0

// Expand one lane's 96 code bits into 16 fp16x2 A-fragment registers holding
// q = u - 4 exactly.  OR-ing a 3-bit field into the mantissa of 1024.0 gives
// 1024 + u * 2^(3f') for field offset 3f' within the mantissa; one fused
// multiply-add with exact constants maps that to u - 4.
__device__ __forceinline__ void dequant_block(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t a[16]) {
  const uint32_t ws[3] = {w0, w1, w2};
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const uint32_t w = ws[j];
    const uint32_t t = w >> 9;
    a[j * 5 + 0] = hfma2_u32(lop3_and_or(w, 0x00070007u, kMagic), kOne2, kNeg1028);
    a[j * 5 + 1] = hfma2_u32(lop3_and_or(w, 0x00380038u, kMagic), kEighth2, kNeg132);
    a[j * 5 + 2] = hfma2_u32(lop3_and_or(w, 0x01C001C0u, kMagic), kSixtyFourth2, kNeg20);
    a[j * 5 + 3] = hfma2_u32(lop3_and_or(t, 0x00070007u, kMagic), kOne2, kNeg1028);
    a[j * 5 + 4] = hfma2_u32(lop3_and_or(t, 0x00380038u, kMagic), kEighth2, kNeg132);
  }
  uint32_t v = lop3_and_or(w0 >> 15, 0x00010001u, kMagic);
  v = lop3_and_or(w1 >> 14, 0x00020002u, v);
  v = lop3_and_or(w2 >> 13, 0x00040004u, v);
  a[15] = hfma2_u32(v, kOne2, kNeg1028);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// ------------------------------------------------------------- warp top-k ---
// L2-only load of data written by other CTAs during this kernel (after the
// caller's acquire).  Kept volatile: issued in program order with the
// dependent shared-memory stores, which measured faster for the logits row
// than batching the loads.
__device__ __forceinline__ float ld_cg_f32(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

// Order-preserving 32-bit key of a float (larger float -> larger key; -inf
// maps above 0, so 0 marks "no entry").
__device__ __forceinline__ uint32_t float_key(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__device__ __forceinline__ uint64_t shfl_u64(uint64_t v, int src) {
  const uint32_t lo = __shfl_sync(0xffffffffu, (uint32_t)v, src);
  const uint32_t hi = __shfl_sync(0xffffffffu, (uint32_t)(v >> 32), src);
  return ((uint64_t)hi << 32) | lo;
}

// u64 entries of per-warp scratch that warp_topk needs
constexpr int kTopkScratch = 80;
constexpr int kTopkMaxCand = 64;

// Key of entry `id` of a logits row: (value key, ~id), so larger values and,
// among equal values, lower ids compare larger; all keys of a row differ.
__device__ __forceinline__ uint64_t topk_key(const float* row, int id) {
  return ((uint64_t)float_key(row[id]) << 32) | (uint32_t)(~(uint32_t)id);
}

// One warp selects the K largest (K <= 16, K < E <= 1024) entries of `row`
// (shared memory; ties go to the lower id).  Lane l owns entries l, l+32, ...
// The K-th largest of the 32 lane maxima is a threshold that at least K
// entries reach and that every one of the K largest reaches; the few entries
// at or above it are ranked against each other in `scratch` (kTopkScratch
// entries of this warp).  More than kTopkMaxCand candidates (possible only
// when the largest values crowd into few lanes) take the general route: K
// rounds of the warp maximum of the remaining entries (two redux.sync
// reductions: largest key, then smallest id).  Lane r < K receives the r-th
// largest value and its id.  Loops stay short: this runs once per call, so
// code size matters more than instruction count.
__device__ __forceinline__ void warp_topk(const float* row, int E, int K, int lane, uint64_t* scratch, float& out_v,
                                          int& out_id) {
  uint64_t m = 0;
#pragma unroll 4
  for (int id = lane; id < E; id += 32) {
    const uint64_t k = topk_key(row, id);
    m = k > m ? k : m;
  }
  // the K-th largest lane maximum: each lane counts the lane maxima above
  // its own (all differ unless both are 0, and at least K + 1 lanes hold an
  // entry); the lane whose count is K - 1 holds it
  int above = 0;
#pragma unroll 8
  for (int j = 0; j < 32; ++j) above += shfl_u64(m, j) > m ? 1 : 0;
  const uint32_t holder = __ballot_sync(0xffffffffu, above == K - 1 && m != 0);
  const uint64_t tau = shfl_u64(m, __ffs(holder) - 1);
  int cnt = 0;
#pragma unroll 4
  for (int id = lane; id < E; id += 32) cnt += topk_key(row, id) >= tau ? 1 : 0;
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  const int n_c = __shfl_sync(0xffffffffu, incl, 31);
  out_v = -INFINITY;
  out_id = 0x7fffffff;
  if (n_c <= kTopkMaxCand) {
    int pos = incl - cnt;
#pragma unroll 4
    for (int id = lane; id < E; id += 32) {
      const uint64_t k = topk_key(row, id);
      if (k >= tau) scratch[pos++] = k;
    }
    __syncwarp();
#pragma unroll 1
    for (int q = lane; q < n_c; q += 32) {
      const uint64_t me = scratch[q];
      int r = 0;
#pragma unroll 4
      for (int j2 = 0; j2 < n_c; ++j2) r += scratch[j2] > me ? 1 : 0;
      if (r < K) scratch[kTopkMaxCand + r] = me;
    }
    __syncwarp();
    if (lane < K) {
      const uint64_t w = scratch[kTopkMaxCand + lane];
      out_v = key_float((uint32_t)(w >> 32));
      out_id = (int)~(uint32_t)w;
    }
    __syncwarp();   // scratch is reused by the warp's next selection
    return;
  }
  // general route; `taken` marks this lane's entries already chosen
  uint32_t taken = 0;
#pragma unroll 1
  for (int r = 0; r < K; ++r) {
    uint64_t lm = 0;
    int li = 0;
#pragma unroll 1
    for (int i = 0, id = lane; id < E; ++i, id += 32) {
      const uint64_t k = topk_key(row, id);
      if (!((taken >> i) & 1u) && k > lm) {
        lm = k;
        li = i;
      }
    }
    const uint32_t hk = (uint32_t)(lm >> 32);
    const uint32_t mx = __reduce_max_sync(0xffffffffu, hk);
    const uint32_t hid = ~(uint32_t)lm;
    const uint32_t win = __reduce_min_sync(0xffffffffu, hk == mx ? hid : 0xffffffffu);
    if (lane == r) {
      out_v = key_float(mx);
      out_id = (int)win;
    }
    if (hk == mx && hid == win) taken |= 1u << li;
  }
}

// The same selection for E <= 32 * VPL with each lane's entries held in
// registers: one shared-memory read per entry, then every pass runs on
// registers (for the E <= 512 rows of the decode path, where the loop form
// above is latency-bound).
template <int VPL>
__device__ __forceinline__ void warp_topk_reg(const float* row, int E, int K, int lane, uint64_t* scratch,
                                              float& out_v, int& out_id) {
  uint64_t s[VPL];
  uint64_t m = 0;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int id = lane + 32 * i;
    s[i] = id < E ? topk_key(row, id) : 0ull;
    m = s[i] > m ? s[i] : m;
  }
  int above = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) above += shfl_u64(m, j) > m ? 1 : 0;
  const uint32_t holder = __ballot_sync(0xffffffffu, above == K - 1 && m != 0);
  const uint64_t tau = shfl_u64(m, __ffs(holder) - 1);
  int cnt = 0;
#pragma unroll
  for (int i = 0; i < VPL; ++i) cnt += s[i] >= tau ? 1 : 0;
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  const int n_c = __shfl_sync(0xffffffffu, incl, 31);
  if (n_c > kTopkMaxCand) {   // values crowded into few lanes: the general route
    warp_topk(row, E, K, lane, scratch, out_v, out_id);
    return;
  }
  out_v = -INFINITY;
  out_id = 0x7fffffff;
  int pos = incl - cnt;
#pragma unroll
  for (int i = 0; i < VPL; ++i)
    if (s[i] >= tau) scratch[pos++] = s[i];
  __syncwarp();
  if (lane < n_c) {
    const uint64_t me = scratch[lane];
    int r = 0;
#pragma unroll 8
    for (int j2 = 0; j2 < n_c; ++j2) r += scratch[j2] > me ? 1 : 0;
    if (r < K) scratch[kTopkMaxCand + r] = me;
  }
  if (lane + 32 < n_c) {
    const uint64_t me = scratch[lane + 32];
    int r = 0;
#pragma unroll 8
    for (int j2 = 0; j2 < n_c; ++j2) r += scratch[j2] > me ? 1 : 0;
    if (r < K) scratch[kTopkMaxCand + r] = me;
  }
  __syncwarp();
  if (lane < K) {
    const uint64_t w = scratch[kTopkMaxCand + lane];
    out_v = key_float((uint32_t)(w >> 32));
    out_id = (int)~(uint32_t)w;
  }
  __syncwarp();   // scratch is reused by the warp's next selection
}

}  // namespace moe
