// KV-streaming window: per layer, the first R KV cells live in VRAM and the
// rest in page-locked host memory; reads go block by block, and the share of
// block reads served from VRAM is counted (page "单卡5090跑125B 大模型",
// §2.1-§2.2: 32,768 of 131,072 int8 cells of 1,056 bytes per QSA layer in
// VRAM, the rest streamed from host memory; §7.2: the block-read hit share).
//
// The window only moves bytes: a cell is opaque.  A block read copies the
// block's cells into the caller's device buffer; resident blocks are read
// from HBM, the others straight from host memory through its device mapping
// (no staging copy).  One kernel launch per call, grid-stride over blocks.
#include <cstdint>
#include <cuda_runtime.h>

#include "moe_gb300.h"
#include "internal.h"

using namespace moe;

struct moe_kv {
  int L = 0, cell_bytes = 0, block_cells = 0;
  int64_t n_cells = 0, resident = 0;
  int device = 0, num_sms = 0;
  uint8_t* window = nullptr;            // [L][R][cell_bytes] device
  uint8_t* host = nullptr;              // caller's [L][n - R][cell_bytes] host memory
  const uint8_t* host_dev = nullptr;    // its device mapping
  bool registered = false;
  unsigned long long* counters = nullptr;   // [2] block reads, hits (device)
  uint32_t* err = nullptr;                  // device error word: a block id out of range
};

namespace {

#define KV_TRY(call)                                                                                 \
  do {                                                                                               \
    cudaError_t e_ = (call);                                                                         \
    if (e_ != cudaSuccess)                                                                           \
      return set_last_error(e_ == cudaErrorMemoryAllocation ? MOE_ERR_OOM : MOE_ERR_CUDA, "%s: %s", \
                            #call, cudaGetErrorString(e_));                                          \
  } while (0)

struct KvReadArgs {
  const uint8_t* window;
  const uint8_t* host;
  const int32_t* ids;
  uint8_t* dst;
  unsigned long long* counters;
  uint32_t* err;
  int64_t block_bytes;                            // multiple of 16
  int32_t n_blocks, resident_blocks, total_blocks;
};

// One CTA per block at a time: each thread moves 16-byte pieces, four loads
// issued before their stores.  Thread 0 counts the read and whether it hit.
__global__ void __launch_bounds__(256) kv_read_kernel(KvReadArgs a) {
  const int64_t n16 = a.block_bytes / 16;
  unsigned long long hits = 0, reads = 0;
  for (int i = blockIdx.x; i < a.n_blocks; i += gridDim.x) {
    const int b = a.ids[i];
    if (b < 0 || b >= a.total_blocks) {   // out of range: recorded, nothing read
      if (threadIdx.x == 0) atomicOr(a.err, 1u);
      continue;
    }
    const bool hit = b < a.resident_blocks;
    const uint4* src = reinterpret_cast<const uint4*>(
        hit ? a.window + (int64_t)b * a.block_bytes : a.host + (int64_t)(b - a.resident_blocks) * a.block_bytes);
    uint4* dst = reinterpret_cast<uint4*>(a.dst + (int64_t)i * a.block_bytes);
    int64_t c = threadIdx.x;
    for (; c + 3 * 256 < n16; c += 4 * 256) {
      const uint4 v0 = src[c], v1 = src[c + 256], v2 = src[c + 512], v3 = src[c + 768];
      dst[c] = v0;
      dst[c + 256] = v1;
      dst[c + 512] = v2;
      dst[c + 768] = v3;
    }
    for (; c < n16; c += 256) dst[c] = src[c];
    reads += 1;
    hits += hit ? 1 : 0;
  }
  if (threadIdx.x == 0 && reads) {
    atomicAdd(&a.counters[0], reads);
    atomicAdd(&a.counters[1], hits);
  }
}

}  // namespace

extern "C" moe_status moe_kv_create(const moe_kv_desc* D, moe_kv** out) {
  if (!D || !out) return set_last_error(MOE_ERR_INVALID_ARG, "NULL desc or out");
  *out = nullptr;
  if (D->n_layers <= 0) return set_last_error(MOE_ERR_INVALID_ARG, "n_layers must be positive");
  if (D->cell_bytes <= 0 || D->cell_bytes % 16 != 0)
    return set_last_error(MOE_ERR_INVALID_ARG, "cell_bytes must be a positive multiple of 16");
  if (D->block_cells <= 0) return set_last_error(MOE_ERR_INVALID_ARG, "block_cells must be positive");
  if (D->n_cells <= 0 || D->n_cells % D->block_cells != 0)
    return set_last_error(MOE_ERR_INVALID_ARG, "n_cells must be a positive multiple of block_cells");
  if (D->resident_cells < 0 || D->resident_cells > D->n_cells || D->resident_cells % D->block_cells != 0)
    return set_last_error(MOE_ERR_INVALID_ARG, "resident_cells must be a multiple of block_cells in [0, n_cells]");
  if (D->n_cells / D->block_cells > INT32_MAX) return set_last_error(MOE_ERR_INVALID_ARG, "too many blocks");
  const int64_t host_cells = D->n_cells - D->resident_cells;
  if (host_cells > 0 && !D->host_cells) return set_last_error(MOE_ERR_INVALID_ARG, "NULL host_cells");
  if ((reinterpret_cast<uintptr_t>(D->host_cells) & 15u) != 0)
    return set_last_error(MOE_ERR_INVALID_ARG, "host_cells not 16-byte aligned");
  moe_kv* kv = new moe_kv();
  kv->L = D->n_layers;
  kv->cell_bytes = D->cell_bytes;
  kv->block_cells = D->block_cells;
  kv->n_cells = D->n_cells;
  kv->resident = D->resident_cells;
  kv->host = static_cast<uint8_t*>(D->host_cells);
  auto fail_destroy = [&](moe_status st) {
    moe_kv_destroy(kv);
    return st;
  };
  cudaError_t e = cudaGetDevice(&kv->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&kv->num_sms, cudaDevAttrMultiProcessorCount, kv->device);
  if (e != cudaSuccess) {
    moe_status st = set_last_error(MOE_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
    return fail_destroy(st);
  }
  const size_t wbytes = (size_t)kv->L * kv->resident * kv->cell_bytes;
  if (wbytes) {
    e = cudaMalloc(&kv->window, wbytes);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail_destroy(set_last_error(MOE_ERR_OOM, "window of %zu bytes: %s", wbytes, cudaGetErrorString(e)));
    }
  }
  if (host_cells > 0) {
    const size_t hbytes = (size_t)kv->L * host_cells * kv->cell_bytes;
    cudaPointerAttributes at;
    e = cudaPointerGetAttributes(&at, kv->host);
    if (e != cudaSuccess) cudaGetLastError();
    if (e == cudaSuccess && (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged))
      return fail_destroy(set_last_error(MOE_ERR_INVALID_ARG, "host_cells must be host memory"));
    if (e != cudaSuccess || at.type == cudaMemoryTypeUnregistered) {
      e = cudaHostRegister(kv->host, hbytes, cudaHostRegisterDefault);
      if (e != cudaSuccess) {
        cudaGetLastError();
        return fail_destroy(set_last_error(MOE_ERR_HOST_PIN, "cudaHostRegister of %zu bytes: %s", hbytes,
                                           cudaGetErrorString(e)));
      }
      kv->registered = true;
    }
    void* dp = nullptr;
    e = cudaHostGetDevicePointer(&dp, kv->host, 0);
    if (e != cudaSuccess || !dp) {
      cudaGetLastError();
      return fail_destroy(set_last_error(MOE_ERR_HOST_PIN, "host_cells has no device mapping"));
    }
    kv->host_dev = static_cast<const uint8_t*>(dp);
  }
  e = cudaMalloc(&kv->counters, 2 * sizeof(unsigned long long) + sizeof(uint32_t));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail_destroy(set_last_error(MOE_ERR_OOM, "counters: %s", cudaGetErrorString(e)));
  }
  kv->err = reinterpret_cast<uint32_t*>(kv->counters + 2);
  e = cudaMemset(kv->counters, 0, 2 * sizeof(unsigned long long) + sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail_destroy(set_last_error(MOE_ERR_CUDA, "counters: %s", cudaGetErrorString(e)));
  *out = kv;
  return MOE_OK;
}

extern "C" moe_status moe_kv_write(moe_kv* kv, int32_t layer, int64_t first_cell, int64_t n, const void* src,
                                   void* stream) {
  if (!kv || !src) return set_last_error(MOE_ERR_INVALID_ARG, "NULL kv or src");
  if (layer < 0 || layer >= kv->L) return set_last_error(MOE_ERR_INVALID_ARG, "layer %d out of range", layer);
  if (first_cell < 0 || n < 0 || first_cell + n > kv->n_cells)
    return set_last_error(MOE_ERR_INVALID_ARG, "cells [%lld, %lld) outside [0, %lld)", (long long)first_cell,
                          (long long)(first_cell + n), (long long)kv->n_cells);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t cb = kv->cell_bytes, R = kv->resident;
  const uint8_t* s8 = static_cast<const uint8_t*>(src);
  const int64_t end = first_cell + n;
  if (first_cell < R) {   // the resident part
    const int64_t m = (end < R ? end : R) - first_cell;
    KV_TRY(cudaMemcpyAsync(kv->window + ((int64_t)layer * R + first_cell) * cb, s8, (size_t)(m * cb),
                           cudaMemcpyDefault, s));
  }
  if (end > R) {          // the host part
    const int64_t c0 = first_cell > R ? first_cell : R;
    KV_TRY(cudaMemcpyAsync(kv->host + ((int64_t)layer * (kv->n_cells - R) + (c0 - R)) * cb,
                           s8 + (c0 - first_cell) * cb, (size_t)((end - c0) * cb), cudaMemcpyDefault, s));
  }
  return MOE_OK;
}

extern "C" moe_status moe_kv_read_blocks(moe_kv* kv, int32_t layer, const int32_t* block_ids, int32_t n_blocks,
                                         void* dst, void* stream) {
  if (!kv) return set_last_error(MOE_ERR_INVALID_ARG, "NULL kv");
  if (layer < 0 || layer >= kv->L) return set_last_error(MOE_ERR_INVALID_ARG, "layer %d out of range", layer);
  if (n_blocks < 0) return set_last_error(MOE_ERR_INVALID_ARG, "n_blocks < 0");
  if (n_blocks == 0) return MOE_OK;
  if (!block_ids || !dst) return set_last_error(MOE_ERR_INVALID_ARG, "NULL block_ids or dst");
  if ((reinterpret_cast<uintptr_t>(dst) & 15u) != 0) return set_last_error(MOE_ERR_INVALID_ARG, "dst not 16-byte aligned");
  KvReadArgs a{};
  const int64_t R = kv->resident, H = kv->n_cells - R;
  a.block_bytes = (int64_t)kv->block_cells * kv->cell_bytes;
  a.window = kv->window ? kv->window + (int64_t)layer * R * kv->cell_bytes : nullptr;
  a.host = kv->host_dev ? kv->host_dev + (int64_t)layer * H * kv->cell_bytes : nullptr;
  a.ids = block_ids;
  a.dst = static_cast<uint8_t*>(dst);
  a.counters = kv->counters;
  a.err = kv->err;
  a.n_blocks = n_blocks;
  a.resident_blocks = (int32_t)(R / kv->block_cells);
  a.total_blocks = (int32_t)(kv->n_cells / kv->block_cells);
  const int grid = n_blocks < 4 * kv->num_sms ? n_blocks : 4 * kv->num_sms;
  kv_read_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
  KV_TRY(cudaGetLastError());
  return MOE_OK;
}

extern "C" moe_status moe_kv_stats(moe_kv* kv, int64_t* block_reads, int64_t* block_hits) {
  if (!kv) return set_last_error(MOE_ERR_INVALID_ARG, "NULL kv");
  unsigned long long c[2] = {0, 0};
  uint32_t err = 0;
  KV_TRY(cudaDeviceSynchronize());
  KV_TRY(cudaMemcpy(c, kv->counters, sizeof(c), cudaMemcpyDeviceToHost));
  KV_TRY(cudaMemcpy(&err, kv->err, sizeof(err), cudaMemcpyDeviceToHost));
  if (block_reads) *block_reads = (int64_t)c[0];
  if (block_hits) *block_hits = (int64_t)c[1];
  if (err) {
    KV_TRY(cudaMemset(kv->err, 0, sizeof(uint32_t)));
    return set_last_error(MOE_ERR_INVALID_ARG, "a block read named a block outside the layer (nothing was read for it)");
  }
  return MOE_OK;
}

extern "C" void moe_kv_destroy(moe_kv* kv) {
  if (!kv) return;
  cudaDeviceSynchronize();
  cudaGetLastError();
  if (kv->window) cudaFree(kv->window);
  if (kv->counters) cudaFree(kv->counters);
  if (kv->registered) cudaHostUnregister(kv->host);
  cudaGetLastError();
  delete kv;
}
