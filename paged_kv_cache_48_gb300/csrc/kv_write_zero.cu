// kv_write_zero.cu -- the two producers of the paged KV cache:
//
//  * paged_kv_write: the slot-mapped write of new tokens' K and V (vLLM
//    concept page, compassingai.com, "15 分钟专家深入" item 2: blocks are
//    filled on demand; its "KV 缓存打包/解包 high-bandwidth 核函数").
//  * paged_kv_zero_blocks: zeroing of freshly allocated blocks before
//    attention first reads them (vLLM v0.17.1 notes, admirer.cn,
//    "修复方案": only new blocks, every byte of their K/V segments, ids sent
//    from host memory together with the launch).
//
// Both are pure streaming kernels: 16-byte vector loads and stores, grids
// sized in multiples of the SM count, no shared memory.
#include <algorithm>
#include <cstring>
#include <utility>

#include "e4m3_encode.cuh"
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {

static __device__ ErrorWord g_err_write_zero = {0ull, 0ull};

// The slot-mapped write of work items first, first + stride, ... < total
// (see kv_write_kernel).  I is the index type: 32-bit whenever the items
// fit, so that the per-item token index is a 32-bit shift (a power-of-two
// row, vpr_shift >= 0) or a 32-bit division instead of a 64-bit division.
template <bool FP8, typename I>
__device__ __forceinline__ void write_items(const uint4 *__restrict__ k,
                                            const uint4 *__restrict__ v,
                                            const int64_t *__restrict__ slot_mapping, I total,
                                            I first, I stride, int vecs_per_row, int vpr_shift,
                                            uint8_t *__restrict__ key_cache,
                                            uint8_t *__restrict__ value_cache, int64_t num_slots,
                                            float k_scale, float v_scale) {
  const E4m3Recip kr = e4m3_recip(k_scale), vr = e4m3_recip(v_scale);
  const I vpr = (I)vecs_per_row;
  for (I idx = first; idx < total; idx += stride) {
    const I tok = vpr_shift >= 0 ? idx >> vpr_shift : idx / vpr;
    const int vec = (int)(idx - tok * vpr);
    const int64_t slot = __ldg(slot_mapping + tok);
    if (slot < 0) continue;  // padding token
    if (slot >= num_slots) {
      if (vec == 0) record_error(&g_err_write_zero, PKV_ERR_RANGE, (long long)tok);
      continue;
    }
    const uint4 kv = __ldg(k + idx);
    const uint4 vv = __ldg(v + idx);
    const int64_t dst_vec = slot * vecs_per_row + vec;  // in 8-element units
    if (!FP8) {
      reinterpret_cast<uint4 *>(key_cache)[dst_vec] = kv;
      reinterpret_cast<uint4 *>(value_cache)[dst_vec] = vv;
    } else {
      reinterpret_cast<uint2 *>(key_cache)[dst_vec] = quant8_e4m3(kv, k_scale, kr);
      reinterpret_cast<uint2 *>(value_cache)[dst_vec] = quant8_e4m3(vv, v_scale, vr);
    }
  }
}

template <bool FP8>
__device__ __forceinline__ void write_all_items(const uint4 *__restrict__ k,
                                                const uint4 *__restrict__ v,
                                                const int64_t *__restrict__ slot_mapping,
                                                int64_t num_tokens, int vecs_per_row,
                                                uint8_t *__restrict__ key_cache,
                                                uint8_t *__restrict__ value_cache,
                                                int64_t num_slots, float k_scale, float v_scale,
                                                int64_t first, int64_t stride) {
  const int64_t total = num_tokens * vecs_per_row;
  const int vpr_shift = (vecs_per_row & (vecs_per_row - 1)) ? -1 : __ffs(vecs_per_row) - 1;
  if (total + stride <= (int64_t)UINT32_MAX)
    write_items<FP8, uint32_t>(k, v, slot_mapping, (uint32_t)total, (uint32_t)first,
                               (uint32_t)stride, vecs_per_row, vpr_shift, key_cache, value_cache,
                               num_slots, k_scale, v_scale);
  else
    write_items<FP8, int64_t>(k, v, slot_mapping, total, first, stride, vecs_per_row, vpr_shift,
                              key_cache, value_cache, num_slots, k_scale, v_scale);
}

// ---------------------------------------------------------------------------
// Slot-mapped write.  Work item = one 16-byte vector of one token's K row
// (8 bf16) plus the matching V vector.  A token row is num_kv_heads *
// head_dim elements, contiguous both in the source and in the cache, so
// consecutive threads touch consecutive addresses on both sides.
// ---------------------------------------------------------------------------
template <bool FP8>
__global__ void __launch_bounds__(256)
kv_write_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                const int64_t *__restrict__ slot_mapping, int64_t num_tokens,
                int vecs_per_row, uint8_t *__restrict__ key_cache,
                uint8_t *__restrict__ value_cache, int64_t num_slots,
                float k_scale, float v_scale) {
  grid_dependency_wait();
  allow_dependent_launch();
  write_all_items<FP8>(k, v, slot_mapping, num_tokens, vecs_per_row, key_cache, value_cache,
                       num_slots, k_scale, v_scale, blockIdx.x * (int64_t)blockDim.x + threadIdx.x,
                       (int64_t)gridDim.x * blockDim.x);
}

// ---------------------------------------------------------------------------
// Zeroing.  One CTA clears one block of both caches (grid-strided over the
// id list).  Ids arrive either through a device pointer or inside the
// launch parameters (host ids: no copy, no allocation, no wait).
// ---------------------------------------------------------------------------
constexpr int kZeroIdsPerLaunch = 4096;

struct ZeroIds {
  int32_t n;
  int32_t ids[kZeroIdsPerLaunch];
};

__device__ __forceinline__ void zero_one_block(uint4 *__restrict__ key_cache,
                                               uint4 *__restrict__ value_cache,
                                               int64_t vecs_per_block,
                                               int32_t id) {
  uint4 *kb = key_cache + (int64_t)id * vecs_per_block;
  uint4 *vb = value_cache + (int64_t)id * vecs_per_block;
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int64_t j = threadIdx.x; j < vecs_per_block; j += blockDim.x) {
    kb[j] = z;
    vb[j] = z;
  }
}

// Ids in device memory.
__global__ void __launch_bounds__(256)
zero_blocks_kernel(uint4 *__restrict__ key_cache, uint4 *__restrict__ value_cache,
                   int64_t vecs_per_block, int32_t num_blocks,
                   const int32_t *__restrict__ ids, int64_t n) {
  grid_dependency_wait();
  allow_dependent_launch();
  for (int64_t i = blockIdx.x; i < n; i += gridDim.x) {
    const int32_t id = __ldg(ids + i);
    if (id < 0 || id >= num_blocks) {
      if (threadIdx.x == 0) record_error(&g_err_write_zero, PKV_ERR_RANGE, i);
      continue;
    }
    zero_one_block(key_cache, value_cache, vecs_per_block, id);
  }
}

// Ids inside the launch parameters (copied from host memory at launch).
__global__ void __launch_bounds__(256)
zero_blocks_param_kernel(uint4 *__restrict__ key_cache,
                         uint4 *__restrict__ value_cache,
                         int64_t vecs_per_block, int32_t num_blocks,
                         const __grid_constant__ ZeroIds ids, int64_t id_base) {
  grid_dependency_wait();
  allow_dependent_launch();
  for (int i = blockIdx.x; i < ids.n; i += gridDim.x) {
    const int32_t id = ids.ids[i];
    if (id < 0 || id >= num_blocks) {
      if (threadIdx.x == 0)
        record_error(&g_err_write_zero, PKV_ERR_RANGE, id_base + i);
      continue;
    }
    zero_one_block(key_cache, value_cache, vecs_per_block, id);
  }
}

// ---------------------------------------------------------------------------
// Zeroing and write in one launch (the same result as zeroing the blocks
// and then writing the tokens).  CTAs 0 .. zero_ctas - 1 take fresh blocks:
// each first collects which of its block's 16 slots this step writes
// (a scan of slot_mapping) and zeroes only the other rows; the remaining
// CTAs write every token.  The two sets of addresses are disjoint, so no
// CTA waits for another.  Ids come in the launch parameters (ids.n > 0) or
// through a device pointer.
// ---------------------------------------------------------------------------
template <bool FP8>
__global__ void __launch_bounds__(256)
kv_zero_write_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                     const int64_t *__restrict__ slot_mapping, int64_t num_tokens,
                     int vecs_per_row, uint8_t *__restrict__ key_cache,
                     uint8_t *__restrict__ value_cache, int32_t num_blocks, float k_scale,
                     float v_scale, const int32_t *__restrict__ dev_ids, int64_t n_dev_ids,
                     const __grid_constant__ ZeroIds ids, int64_t id_base, int zero_ctas,
                     int write_tokens) {
  grid_dependency_wait();
  allow_dependent_launch();
  const int64_t num_slots = (int64_t)num_blocks * 16;
  if ((int)blockIdx.x < zero_ctas) {
    __shared__ uint32_t written;  // bit r: slot r of the block is written this step
    const int64_t n = ids.n > 0 ? ids.n : n_dev_ids;
    // a row of the block in 16-byte units of the cache element type
    const int row_vecs = FP8 ? vecs_per_row / 2 : vecs_per_row;
    for (int64_t i = blockIdx.x; i < n; i += zero_ctas) {
      const int32_t id = ids.n > 0 ? ids.ids[i] : __ldg(dev_ids + i);
      if (id < 0 || id >= num_blocks) {
        if (threadIdx.x == 0) record_error(&g_err_write_zero, PKV_ERR_RANGE, id_base + i);
        continue;
      }
      if (threadIdx.x == 0) written = 0u;
      __syncthreads();
      const int64_t lo = (int64_t)id * 16;
      uint32_t mine = 0u;
      for (int64_t t = threadIdx.x; t < num_tokens; t += blockDim.x) {
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot >= lo && slot < lo + 16) mine |= 1u << (int)(slot - lo);
      }
      if (mine) atomicOr(&written, mine);
      __syncthreads();
      const uint32_t keep = written;
      uint4 *kb = reinterpret_cast<uint4 *>(key_cache) + lo * row_vecs;
      uint4 *vb = reinterpret_cast<uint4 *>(value_cache) + lo * row_vecs;
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      for (int j = threadIdx.x; j < 16 * row_vecs; j += blockDim.x) {
        if ((keep >> (j / row_vecs)) & 1u) continue;
        kb[j] = z;
        vb[j] = z;
      }
      __syncthreads();  // `written` is reused for the next block
    }
    return;
  }
  if (!write_tokens) return;
  write_all_items<FP8>(k, v, slot_mapping, num_tokens, vecs_per_row, key_cache, value_cache,
                       num_slots, k_scale, v_scale,
                       (blockIdx.x - zero_ctas) * (int64_t)blockDim.x + threadIdx.x,
                       (int64_t)(gridDim.x - zero_ctas) * blockDim.x);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
// Launch with programmatic stream serialisation (see grid_dependency_wait).
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block,
                              cudaStream_t s, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

const void *error_word_write_zero() { return &g_err_write_zero; }

}  // namespace pkv

using namespace pkv;

extern "C" pkv_status paged_kv_write(const void *k, const void *v,
                                     const int64_t *slot_mapping,
                                     int64_t num_tokens,
                                     const pkv_cache *cache, void *stream) {
  pkv_status st = validate_cache(cache);
  if (st != PKV_OK) return st;
  if (num_tokens < 0) return PKV_ERR_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping) return PKV_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15)
    return PKV_ERR_ARG;  // 16-byte vector loads
  const bool fp8 = cache->dtype == PKV_FP8_E4M3;
  if (fp8 && !(cache->k_scale > 0.f && cache->v_scale > 0.f))
    return PKV_ERR_ARG;
  const int vecs_per_row = cache->num_kv_heads * cache->head_dim / 8;
  const int64_t total = num_tokens * vecs_per_row;
  const int threads = 256;
  const int sms = device_sm_count();
  if (sms <= 0) return PKV_ERR_CUDA;
  const int64_t want = (total + threads - 1) / threads;
  const int grid = (int)std::min<int64_t>(want, (int64_t)sms * 8);
  const int64_t num_slots = (int64_t)cache->num_blocks * cache->block_size;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (fp8)
    e = launch_pdl(kv_write_kernel<true>, dim3(grid), dim3(threads), s,
                   static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping,
                   num_tokens, vecs_per_row, static_cast<uint8_t *>(cache->key_cache),
                   static_cast<uint8_t *>(cache->value_cache), num_slots, cache->k_scale,
                   cache->v_scale);
  else
    e = launch_pdl(kv_write_kernel<false>, dim3(grid), dim3(threads), s,
                   static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping,
                   num_tokens, vecs_per_row, static_cast<uint8_t *>(cache->key_cache),
                   static_cast<uint8_t *>(cache->value_cache), num_slots, 1.f, 1.f);
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" pkv_status paged_kv_zero_blocks(const pkv_cache *cache,
                                           const int32_t *block_ids, int64_t n,
                                           int ids_on_host, void *stream) {
  pkv_status st = validate_cache(cache);
  if (st != PKV_OK) return st;
  if (n < 0) return PKV_ERR_ARG;
  if (n == 0) return PKV_OK;
  if (!block_ids) return PKV_ERR_ARG;
  const int64_t block_bytes = (int64_t)cache->block_size *
                              cache->num_kv_heads * cache->head_dim *
                              (cache->dtype == PKV_FP8_E4M3 ? 1 : 2);
  const int64_t vecs_per_block = block_bytes / 16;
  const int sms = device_sm_count();
  if (sms <= 0) return PKV_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint4 *kc = static_cast<uint4 *>(cache->key_cache);
  uint4 *vc = static_cast<uint4 *>(cache->value_cache);
  const int threads = 256;
  if (!ids_on_host) {
    const int grid = (int)std::min<int64_t>(n, (int64_t)sms * 16);
    return launch_pdl(zero_blocks_kernel, dim3(grid), dim3(threads), s, kc, vc,
                      vecs_per_block, cache->num_blocks, block_ids, n) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
  }
  // Host ids travel inside the launch parameters, kZeroIdsPerLaunch at a
  // time; the parameter block is copied at launch, so the caller's buffer
  // is free again when this returns.
  ZeroIds chunk;
  for (int64_t base = 0; base < n; base += kZeroIdsPerLaunch) {
    const int m = (int)std::min<int64_t>(kZeroIdsPerLaunch, n - base);
    chunk.n = m;
    std::memcpy(chunk.ids, block_ids + base, sizeof(int32_t) * m);
    const int grid = std::min(m, sms * 16);
    if (launch_pdl(zero_blocks_param_kernel, dim3(grid), dim3(threads), s, kc, vc,
                   vecs_per_block, cache->num_blocks, chunk, base) != cudaSuccess)
      return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

extern "C" pkv_status paged_kv_zero_and_write(const void *k, const void *v,
                                              const int64_t *slot_mapping, int64_t num_tokens,
                                              const pkv_cache *cache, const int32_t *block_ids,
                                              int64_t n, int ids_on_host, void *stream) {
  pkv_status st = validate_cache(cache);
  if (st != PKV_OK) return st;
  if (num_tokens < 0 || n < 0) return PKV_ERR_ARG;
  if (num_tokens == 0 && n == 0) return PKV_OK;
  if (num_tokens > 0) {
    if (!k || !v || !slot_mapping) return PKV_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15)
      return PKV_ERR_ARG;  // 16-byte vector loads
  }
  if (n > 0 && !block_ids) return PKV_ERR_ARG;
  const bool fp8 = cache->dtype == PKV_FP8_E4M3;
  if (fp8 && !(cache->k_scale > 0.f && cache->v_scale > 0.f)) return PKV_ERR_ARG;
  const int sms = device_sm_count();
  if (sms <= 0) return PKV_ERR_CUDA;
  const int vecs_per_row = cache->num_kv_heads * cache->head_dim / 8;
  const int threads = 256;
  const int64_t want = (num_tokens * vecs_per_row + threads - 1) / threads;
  const int write_ctas = (int)std::min<int64_t>(want, (int64_t)sms * 8);
  const float ks = fp8 ? cache->k_scale : 1.f, vs = fp8 ? cache->v_scale : 1.f;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto launch = [&](const int32_t *dev_ids, int64_t n_dev, const ZeroIds &ids, int64_t base,
                    int zero_ctas, int with_write) -> bool {
    const int grid = zero_ctas + (with_write ? write_ctas : 0);
    if (grid == 0) return true;
    auto kern = fp8 ? kv_zero_write_kernel<true> : kv_zero_write_kernel<false>;
    return launch_pdl(kern, dim3(grid), dim3(threads), s, static_cast<const uint4 *>(k),
                      static_cast<const uint4 *>(v), slot_mapping, num_tokens, vecs_per_row,
                      static_cast<uint8_t *>(cache->key_cache),
                      static_cast<uint8_t *>(cache->value_cache), cache->num_blocks, ks, vs,
                      dev_ids, n_dev, ids, base, zero_ctas, with_write) == cudaSuccess;
  };
  static thread_local ZeroIds chunk;
  if (n == 0 || !ids_on_host) {
    chunk.n = 0;
    const int zero_ctas = (int)std::min<int64_t>(n, (int64_t)sms * 16);
    return launch(block_ids, n, chunk, 0, zero_ctas, num_tokens > 0) ? PKV_OK : PKV_ERR_CUDA;
  }
  // Host ids ride in the launch parameters, kZeroIdsPerLaunch at a time;
  // the first launch also writes the tokens, the later ones only zero (each
  // zeroing CTA still skips the rows this step writes).
  for (int64_t base = 0; base < n; base += kZeroIdsPerLaunch) {
    const int m = (int)std::min<int64_t>(kZeroIdsPerLaunch, n - base);
    chunk.n = m;
    std::memcpy(chunk.ids, block_ids + base, sizeof(int32_t) * m);
    if (!launch(nullptr, 0, chunk, base, std::min(m, sms * 16), base == 0 && num_tokens > 0))
      return PKV_ERR_CUDA;
  }
  return PKV_OK;
}
