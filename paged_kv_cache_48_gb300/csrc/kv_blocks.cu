// kv_blocks.cu -- whole-block movement in the paged KV cache:
//
//  * paged_kv_copy_blocks: copy-on-write of shared blocks (vLLM internals,
//    naphjohn.github.io, §1.1: requests sharing a prefix point at the same
//    blocks, which are copied when one of them must diverge);
//  * paged_kv_swap_out / paged_kv_swap_in: moving the blocks of a preempted
//    sequence to pinned host memory and back (vLLM concept page,
//    compassingai.com, "15 分钟专家深入" item 1: swap out to CPU memory,
//    swap in when memory frees up).
//
// All three are streaming kernels: one CTA per block (grid-strided over the
// list), 16-byte vector loads and stores.  Host memory is accessed directly
// through its device-mapped address (pinned memory only; the entry points
// check that the buffers are pinned before launching).
#include <algorithm>
#include <cstring>
#include <utility>

#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {

static __device__ ErrorWord g_err_blocks = {0ull, 0ull};

constexpr int kIdsPerLaunch = 2048;

struct BlockList {
  int32_t n;
  int32_t a[kIdsPerLaunch];  // source ids (copy) or block ids (swap)
  int32_t b[kIdsPerLaunch];  // destination ids (copy)
};

__device__ __forceinline__ void copy_vecs(uint4 *__restrict__ dst, const uint4 *__restrict__ src,
                                          int64_t vecs) {
  for (int64_t j = threadIdx.x; j < vecs; j += blockDim.x) dst[j] = src[j];
}

// Copies are done in list order only in the sense that every pair is
// applied once; pairs must not overlap (a destination may not be another
// pair's source or destination).
__global__ void __launch_bounds__(256)
copy_blocks_kernel(uint4 *__restrict__ key_cache, uint4 *__restrict__ value_cache,
                   int64_t vecs_per_block, int32_t num_blocks, const int32_t *__restrict__ src,
                   const int32_t *__restrict__ dst, int64_t n,
                   const __grid_constant__ BlockList list, int64_t base) {
  grid_dependency_wait();
  allow_dependent_launch();
  const int64_t count = src ? n : list.n;
  for (int64_t i = blockIdx.x; i < count; i += gridDim.x) {
    const int32_t s = src ? __ldg(src + i) : list.a[i];
    const int32_t d = src ? __ldg(dst + i) : list.b[i];
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
      if (threadIdx.x == 0) record_error(&g_err_blocks, PKV_ERR_RANGE, base + i);
      continue;
    }
    copy_vecs(key_cache + (int64_t)d * vecs_per_block, key_cache + (int64_t)s * vecs_per_block,
              vecs_per_block);
    copy_vecs(value_cache + (int64_t)d * vecs_per_block,
              value_cache + (int64_t)s * vecs_per_block, vecs_per_block);
  }
}

// out == true: host[i] = cache[ids[i]]; out == false: cache[ids[i]] = host[i].
template <bool OUT>
__global__ void __launch_bounds__(256)
swap_blocks_kernel(uint4 *__restrict__ key_cache, uint4 *__restrict__ value_cache,
                   int64_t vecs_per_block, int32_t num_blocks, const int32_t *__restrict__ ids,
                   int64_t n, const __grid_constant__ BlockList list, int64_t base,
                   uint4 *__restrict__ host_k, uint4 *__restrict__ host_v) {
  grid_dependency_wait();
  allow_dependent_launch();
  const int64_t count = ids ? n : list.n;
  for (int64_t i = blockIdx.x; i < count; i += gridDim.x) {
    const int32_t id = ids ? __ldg(ids + i) : list.a[i];
    if (id < 0 || id >= num_blocks) {
      if (threadIdx.x == 0) record_error(&g_err_blocks, PKV_ERR_RANGE, base + i);
      continue;
    }
    uint4 *hk = host_k + (base + i) * vecs_per_block;
    uint4 *hv = host_v + (base + i) * vecs_per_block;
    uint4 *ck = key_cache + (int64_t)id * vecs_per_block;
    uint4 *cv = value_cache + (int64_t)id * vecs_per_block;
    if (OUT) {
      copy_vecs(hk, ck, vecs_per_block);
      copy_vecs(hv, cv, vecs_per_block);
    } else {
      copy_vecs(ck, hk, vecs_per_block);
      copy_vecs(cv, hv, vecs_per_block);
    }
  }
}

template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t s,
                              Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

static int64_t block_vecs(const pkv_cache *c) {
  return (int64_t)c->block_size * c->num_kv_heads * c->head_dim *
         (c->dtype == PKV_FP8_E4M3 ? 1 : 2) / 16;
}

// Device view of a pinned (page-locked, registered) host buffer; nullptr
// for anything else.  Pageable memory is refused on every platform, also
// where the GPU could reach it through the host page tables.
static void *device_view(const void *p) {
  if (!p) return nullptr;
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (attr.type != cudaMemoryTypeHost || !attr.devicePointer) return nullptr;
  return attr.devicePointer;
}

const void *error_word_blocks() { return &g_err_blocks; }

}  // namespace pkv

using namespace pkv;

extern "C" pkv_status paged_kv_copy_blocks(const pkv_cache *cache, const int32_t *src_ids,
                                           const int32_t *dst_ids, int64_t n, int ids_on_host,
                                           void *stream) {
  pkv_status st = validate_cache(cache);
  if (st != PKV_OK) return st;
  if (n < 0) return PKV_ERR_ARG;
  if (n == 0) return PKV_OK;
  if (!src_ids || !dst_ids) return PKV_ERR_ARG;
  const int sms = device_sm_count();
  if (sms <= 0) return PKV_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint4 *kc = static_cast<uint4 *>(cache->key_cache);
  uint4 *vc = static_cast<uint4 *>(cache->value_cache);
  const int64_t vecs = block_vecs(cache);
  if (!ids_on_host) {
    static const BlockList none = {0, {0}, {0}};
    const int grid = (int)std::min<int64_t>(n, (int64_t)sms * 8);
    return launch_pdl(copy_blocks_kernel, dim3(grid), dim3(256), s, kc, vc, vecs,
                      cache->num_blocks, src_ids, dst_ids, n, none, (int64_t)0) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
  }
  BlockList list;
  for (int64_t base = 0; base < n; base += kIdsPerLaunch) {
    const int m = (int)std::min<int64_t>(kIdsPerLaunch, n - base);
    list.n = m;
    std::memcpy(list.a, src_ids + base, sizeof(int32_t) * m);
    std::memcpy(list.b, dst_ids + base, sizeof(int32_t) * m);
    const int grid = std::min(m, sms * 8);
    if (launch_pdl(copy_blocks_kernel, dim3(grid), dim3(256), s, kc, vc, vecs, cache->num_blocks,
                   (const int32_t *)nullptr, (const int32_t *)nullptr, (int64_t)0, list,
                   base) != cudaSuccess)
      return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

template <bool OUT>
static pkv_status swap_blocks(const pkv_cache *cache, const int32_t *block_ids, int64_t n,
                              int ids_on_host, const void *host_k, const void *host_v,
                              void *stream) {
  pkv_status st = validate_cache(cache);
  if (st != PKV_OK) return st;
  if (n < 0) return PKV_ERR_ARG;
  if (n == 0) return PKV_OK;
  if (!block_ids) return PKV_ERR_ARG;
  uint4 *hk = static_cast<uint4 *>(device_view(host_k));
  uint4 *hv = static_cast<uint4 *>(device_view(host_v));
  if (!hk || !hv) return PKV_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(hk) | reinterpret_cast<uintptr_t>(hv)) & 15)
    return PKV_ERR_ARG;
  const int sms = device_sm_count();
  if (sms <= 0) return PKV_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint4 *kc = static_cast<uint4 *>(cache->key_cache);
  uint4 *vc = static_cast<uint4 *>(cache->value_cache);
  const int64_t vecs = block_vecs(cache);
  if (!ids_on_host) {
    static const BlockList none = {0, {0}, {0}};
    const int grid = (int)std::min<int64_t>(n, (int64_t)sms * 8);
    return launch_pdl(swap_blocks_kernel<OUT>, dim3(grid), dim3(256), s, kc, vc, vecs,
                      cache->num_blocks, block_ids, n, none, (int64_t)0, hk, hv) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
  }
  BlockList list;
  for (int64_t base = 0; base < n; base += kIdsPerLaunch) {
    const int m = (int)std::min<int64_t>(kIdsPerLaunch, n - base);
    list.n = m;
    std::memcpy(list.a, block_ids + base, sizeof(int32_t) * m);
    const int grid = std::min(m, sms * 8);
    if (launch_pdl(swap_blocks_kernel<OUT>, dim3(grid), dim3(256), s, kc, vc, vecs,
                   cache->num_blocks, (const int32_t *)nullptr, (int64_t)0, list, base, hk,
                   hv) != cudaSuccess)
      return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

extern "C" pkv_status paged_kv_swap_out(const pkv_cache *cache, const int32_t *block_ids,
                                        int64_t n, int ids_on_host, void *host_k, void *host_v,
                                        void *stream) {
  return swap_blocks<true>(cache, block_ids, n, ids_on_host, host_k, host_v, stream);
}

extern "C" pkv_status paged_kv_swap_in(const pkv_cache *cache, const int32_t *block_ids,
                                       int64_t n, int ids_on_host, const void *host_k,
                                       const void *host_v, void *stream) {
  return swap_blocks<false>(cache, block_ids, n, ids_on_host, host_k, host_v, stream);
}
