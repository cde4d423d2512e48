// attention_noalloc.cu -- decode attention for callers that cannot allocate
// device memory.
//
// paged_attention_decode needs a caller-provided workspace whenever it
// splits long sequences into partitions (the per-partition max, sum and
// partial outputs).  Some callers have no way to obtain one: code that runs
// where cudaMalloc is forbidden or unavailable (inside a custom allocator or
// an allocation callback, under a memory budget that is already fully
// handed out, or in a host runtime with no device allocator of its own).
// For them this file keeps one fixed scratch area in the library's own
// device memory and forwards to paged_attention_decode with it.
//
// The scratch is a file-scope __device__ array of PKV_NOALLOC_SCRATCH_BYTES.
// Its name is only a host-side stand-in in host code, so the device address
// is looked up once per device with cudaGetSymbolAddress (with that device
// current) and cached; the first call on each device does this look-up, so
// make that first call before capturing any stream.  That first look-up is
// also when the CUDA driver loads the module holding the array (with lazy
// module loading, the default, nothing is loaded earlier) and so when the
// 16 MiB are taken from the device: a caller that cannot allocate later
// should make one call at set-up, while memory is still available.  From
// then on the device holds the array until the process exits, and calls
// allocate nothing.  The cached address does not survive cudaDeviceReset:
// do not call this entry point on a device after resetting it.
//
// All calls share the one array and it keeps whatever the last call left
// there.  Nothing in it has to start at zero: a call writes every partial
// result before it reads it.  Calls whose kernels overlap on the GPU (for
// example on two streams without ordering between them) race on the array;
// order them on one stream or with events.
#include <mutex>

#include "pkv_host.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of g_noalloc_scratch on the current device (looked up once
// per device); nullptr on failure.
void *scratch_address() {
  static std::mutex mu;
  static void *addr[kMaxDevices] = {nullptr};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" pkv_status paged_attention_decode_noalloc(
    const void *q, const pkv_cache *cache, const int32_t *block_tables, int32_t max_blocks,
    const int32_t *seq_lens, int32_t batch, int32_t num_heads, float scale, void *out,
    int32_t max_seq_len, int32_t partition_tokens, void *stream) {
  pkv_status st = pkv::validate_cache(cache);
  if (st != PKV_OK) return st;
  if (batch < 0 || num_heads <= 0 || max_seq_len < 0 || partition_tokens < 0 ||
      partition_tokens % 16)
    return PKV_ERR_ARG;
  // Arguments paged_attention_decode rejects as invalid get that answer here
  // too, before the scratch size is looked at: more than 65535 sequences or
  // partitions per sequence (grid limits), or an invalid head count.
  if (num_heads % cache->num_kv_heads) return PKV_ERR_SHAPE;
  if (batch > 65535) return PKV_ERR_ARG;
  const int32_t pt = paged_attention_partition_tokens(batch, num_heads, cache->num_kv_heads,
                                                      max_seq_len, partition_tokens);
  if (pt <= 0 || ((int64_t)max_seq_len + pt - 1) / pt > 65535) return PKV_ERR_ARG;
  const size_t need = paged_attention_workspace_bytes(
      batch, num_heads, cache->num_kv_heads, cache->head_dim, max_seq_len, partition_tokens);
  if (need > PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
  void *ws = nullptr;
  if (need > 0) {
    ws = scratch_address();
    if (!ws) return PKV_ERR_CUDA;
  }
  return paged_attention_decode(q, cache, block_tables, max_blocks, seq_lens, batch, num_heads,
                                scale, out, max_seq_len, partition_tokens, ws,
                                need > 0 ? (size_t)PKV_NOALLOC_SCRATCH_BYTES : 0, stream);
}
