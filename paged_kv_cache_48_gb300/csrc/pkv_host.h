// pkv_host.h -- host-side helpers shared by the translation units of the
// paged KV-cache library: argument validation, device properties and the
// per-unit device error words.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pagedkv.h"

namespace pkv {

// Validates a cache descriptor: non-null 16-byte-aligned buffers, block
// size 16, head_dim 64 or 128, a known dtype, positive counts.
pkv_status validate_cache(const pkv_cache *cache);

// SM count of the current device (cached per device); <= 0 on failure.
int device_sm_count();

// Each translation unit that launches kernels owns a device error word;
// these read it (after synchronising `s`) and clear it when set.
unsigned long long read_and_clear_error_write_zero(cudaStream_t s,
                                                   cudaError_t *err);
unsigned long long read_and_clear_error_attention(cudaStream_t s,
                                                  cudaError_t *err);
unsigned long long read_and_clear_error_blocks(cudaStream_t s, cudaError_t *err);
unsigned long long read_and_clear_error_prep(cudaStream_t s, cudaError_t *err);
unsigned long long read_and_clear_error_prefill(cudaStream_t s, cudaError_t *err);

}  // namespace pkv
