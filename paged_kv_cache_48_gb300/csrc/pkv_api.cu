// pkv_api.cu -- shared host entry points of the paged KV-cache library:
// argument validation, device properties, the error-word check, status
// strings and the version.
#include <atomic>

#include "pkv_host.h"

namespace pkv {

pkv_status validate_cache(const pkv_cache *c) {
  if (!c || !c->key_cache || !c->value_cache) return PKV_ERR_ARG;
  if (c->dtype != PKV_BF16 && c->dtype != PKV_FP8_E4M3) return PKV_ERR_DTYPE;
  if (c->block_size != 16) return PKV_ERR_SHAPE;
  if (c->head_dim != 64 && c->head_dim != 128) return PKV_ERR_SHAPE;
  if (c->num_kv_heads <= 0 || c->num_blocks <= 0) return PKV_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(c->key_cache) |
       reinterpret_cast<uintptr_t>(c->value_cache)) & 15)
    return PKV_ERR_ARG;
  return PKV_OK;
}

int device_sm_count() {
  // one entry per device, written once with the same value by any thread
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
  if (dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
      cudaSuccess)
    return -1;
  if (dev < 64) cached[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_check(void *stream, int64_t *detail) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (detail) *detail = -1;
  cudaError_t e[5] = {cudaSuccess, cudaSuccess, cudaSuccess, cudaSuccess, cudaSuccess};
  const unsigned long long words[5] = {
      read_and_clear_error_write_zero(s, &e[0]), read_and_clear_error_attention(s, &e[1]),
      read_and_clear_error_blocks(s, &e[2]), read_and_clear_error_prep(s, &e[3]),
      read_and_clear_error_prefill(s, &e[4])};
  unsigned long long w = 0ull;
  for (int i = 0; i < 5; ++i) {
    if (e[i] != cudaSuccess) return PKV_ERR_CUDA;
    if (!w) w = words[i];
  }
  if (!w) return PKV_OK;
  if (detail) *detail = (int64_t)(w & 0x00FFFFFFFFFFFFFFull) - 1;
  return static_cast<pkv_status>(w >> 56);
}

extern "C" const char *pkv_status_str(pkv_status status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_ARG: return "invalid argument";
    case PKV_ERR_DTYPE: return "unsupported cache dtype";
    case PKV_ERR_SHAPE: return "unsupported shape (block_size 16, head_dim 64/128, "
                               "num_heads a multiple of num_kv_heads)";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_RANGE: return "slot, block id or sequence length out of range";
    case PKV_ERR_TIMEOUT: return "device wait timed out";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

extern "C" int32_t pkv_version(void) { return 200; }
