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

// Each translation unit that launches kernels owns a device error word
// (ErrorWord in pkv_device.cuh: a code and the global-timer stamp of the
// moment it was recorded); these return the host-side handle of each unit's
// word for cudaMemcpy{From,To}SymbolAsync.
const void *error_word_write_zero();
const void *error_word_attention();
const void *error_word_blocks();
const void *error_word_prep();
const void *error_word_prefill();

// Shared-prefix pass of cascade decode (attention_prefill.cu): for every
// group, the members' queries against the group's prefix on the tensor
// cores, one (m, l, o / l) partial per prefix partition in merge slots
// 0 .. of each member row.
pkv_status launch_prefix_partials(const void *q, const pkv_cache *cache,
                                  const int32_t *block_tables, int32_t max_blocks,
                                  const int32_t *seq_lens, const int32_t *group_start,
                                  const int32_t *prefix_len, int32_t num_groups,
                                  int32_t max_group_size, int32_t max_prefix_len, int32_t batch,
                                  int32_t num_heads, float scale, float *part_o, float2 *part_ml,
                                  int part_stride, int prefix_part_tokens, cudaStream_t s);

}  // namespace pkv
