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
  constexpr int kUnits = 5;
  const void *sym[kUnits] = {error_word_write_zero(), error_word_attention(),
                             error_word_blocks(), error_word_prep(), error_word_prefill()};
  // one 16-byte record per unit: {code, global-timer stamp}
  unsigned long long rec[kUnits][2] = {};
  for (int i = 0; i < kUnits; ++i)
    if (cudaMemcpyFromSymbolAsync(rec[i], sym[i], sizeof rec[i], 0, cudaMemcpyDeviceToHost, s) !=
        cudaSuccess)
      return PKV_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ERR_CUDA;
  // the earliest record over all units (ties: the lower unit index) wins
  int first = -1;
  for (int i = 0; i < kUnits; ++i)
    if (rec[i][0] && (first < 0 || rec[i][1] < rec[first][1])) first = i;
  if (first < 0) return PKV_OK;
  static const unsigned long long zero[2] = {0ull, 0ull};
  for (int i = 0; i < kUnits; ++i)
    if (rec[i][0] && cudaMemcpyToSymbolAsync(sym[i], zero, sizeof zero, 0, cudaMemcpyHostToDevice,
                                             s) != cudaSuccess)
      return PKV_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ERR_CUDA;
  const unsigned long long w = rec[first][0];
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
