// input_prep.cu -- step input preparation on the GPU from a persistent
// request state table (Model Runner V2 summary, papercache.org, Figure 2
// and "GPU原生的输入准备": every active request keeps a stable row; each step
// gathers the scheduled rows, in batch order, into the step's block table,
// seq_lens, query_start_loc, positions, input ids and slot mapping, all on
// the GPU).
//
// Two launches: a single-CTA scan builds query_start_loc and seq_lens; a
// per-entry kernel (programmatic dependent launch) gathers the block-table
// row and writes the per-token outputs.
#include <algorithm>
#include <utility>

#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {

static __device__ ErrorWord g_err_prep = {0ull, 0ull};

struct PrepParams {
  const int32_t *idx_mapping, *num_scheduled;
  const int32_t *state_block_table, *state_num_computed, *state_token_ids;
  int32_t *block_tables, *seq_lens, *query_start_loc, *positions, *input_ids;
  int64_t *slot_mapping;
  int32_t batch, max_blocks, max_model_len, num_rows;
  int64_t total_tokens;
};

constexpr int kScanThreads = 1024;

// query_start_loc[b] = sum of max(num_scheduled, 0) before b (entry `batch`
// = the total); seq_lens[b] = num_computed[row] + n for valid rows.
__global__ void __launch_bounds__(kScanThreads) prep_scan_kernel(const PrepParams p) {
  __shared__ long long warp_sums[kScanThreads / 32];
  __shared__ long long carry;
  grid_dependency_wait();
  allow_dependent_launch();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int b0 = 0; b0 < p.batch; b0 += kScanThreads) {
    const int b = b0 + tid;
    int n = 0;
    if (b < p.batch) {
      n = __ldg(p.num_scheduled + b);
      if (n < 0) {
        record_error(&g_err_prep, PKV_ERR_RANGE, b);
        n = 0;
      }
    }
    long long incl = n;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      long long w = warp_sums[lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, w, off);
        if (lane >= off) w += y;
      }
      warp_sums[lane] = w;  // inclusive prefix of warp totals
    }
    __syncthreads();
    const long long base = carry + (warp ? warp_sums[warp - 1] : 0);
    const long long excl = base + incl - n;
    if (b < p.batch) {
      p.query_start_loc[b] = (int32_t)excl;
      const int r = __ldg(p.idx_mapping + b);
      if (excl + n > p.total_tokens)
        record_error(&g_err_prep, PKV_ERR_RANGE, b);
      else if (r >= 0 && r < p.num_rows)
        p.seq_lens[b] = __ldg(p.state_num_computed + r) + n;
    }
    __syncthreads();
    if (tid == 0) carry += warp_sums[kScanThreads / 32 - 1];
    __syncthreads();
  }
  if (tid == 0) p.query_start_loc[p.batch] = (int32_t)carry;
}

// One CTA per batch entry (grid-strided): the block-table row and the
// entry's tokens.
__global__ void __launch_bounds__(128) prep_gather_kernel(const PrepParams p) {
  grid_dependency_wait();
  allow_dependent_launch();
  for (int b = blockIdx.x; b < p.batch; b += gridDim.x) {
    int n = __ldg(p.num_scheduled + b);
    if (n < 0) n = 0;
    const int64_t t0 = p.query_start_loc[b];
    if (t0 + n > p.total_tokens) continue;
    const int r = __ldg(p.idx_mapping + b);
    if (r < 0 || r >= p.num_rows) {
      if (threadIdx.x == 0) record_error(&g_err_prep, PKV_ERR_RANGE, b);
      for (int i = threadIdx.x; i < n; i += blockDim.x) p.slot_mapping[t0 + i] = -1;
      continue;
    }
    const int32_t *row = p.state_block_table + (size_t)r * p.max_blocks;
    for (int j = threadIdx.x; j < p.max_blocks; j += blockDim.x)
      p.block_tables[(size_t)b * p.max_blocks + j] = __ldg(row + j);
    const int c = __ldg(p.state_num_computed + r);
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const int64_t t = t0 + i;
      const int pos = c + i;
      p.positions[t] = pos;
      if (pos < 0 || pos >= p.max_blocks * 16 || pos >= p.max_model_len) {
        record_error(&g_err_prep, PKV_ERR_RANGE, b);
        p.slot_mapping[t] = -1;
        continue;
      }
      p.input_ids[t] = __ldg(p.state_token_ids + (size_t)r * p.max_model_len + pos);
      p.slot_mapping[t] = (int64_t)__ldg(row + pos / 16) * 16 + pos % 16;
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

const void *error_word_prep() { return &g_err_prep; }

}  // namespace pkv

using namespace pkv;

extern "C" pkv_status paged_prepare_inputs(
    const int32_t *idx_mapping, const int32_t *num_scheduled, int32_t batch,
    const int32_t *state_block_table, int32_t max_blocks, const int32_t *state_num_computed,
    const int32_t *state_token_ids, int32_t max_model_len, int32_t num_rows,
    int64_t total_tokens, int32_t *block_tables, int32_t *seq_lens, int32_t *query_start_loc,
    int32_t *positions, int32_t *input_ids, int64_t *slot_mapping, void *stream) {
  if (batch < 0 || max_blocks <= 0 || max_model_len <= 0 || num_rows < 0 || total_tokens < 0)
    return PKV_ERR_ARG;
  if (!query_start_loc) return PKV_ERR_ARG;
  if (batch > 0 && (!idx_mapping || !num_scheduled || !state_block_table ||
                    !state_num_computed || !state_token_ids || !block_tables || !seq_lens))
    return PKV_ERR_ARG;
  if (total_tokens > 0 && (!positions || !input_ids || !slot_mapping)) return PKV_ERR_ARG;
  if ((int64_t)max_blocks * 16 > INT32_MAX) return PKV_ERR_ARG;
  const int sms = device_sm_count();
  if (sms <= 0) return PKV_ERR_CUDA;
  PrepParams p;
  p.idx_mapping = idx_mapping;
  p.num_scheduled = num_scheduled;
  p.state_block_table = state_block_table;
  p.state_num_computed = state_num_computed;
  p.state_token_ids = state_token_ids;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.query_start_loc = query_start_loc;
  p.positions = positions;
  p.input_ids = input_ids;
  p.slot_mapping = slot_mapping;
  p.batch = batch;
  p.max_blocks = max_blocks;
  p.max_model_len = max_model_len;
  p.num_rows = num_rows;
  p.total_tokens = total_tokens;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_pdl(prep_scan_kernel, dim3(1), dim3(kScanThreads), s, p) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (batch > 0) {
    const int grid = std::min(batch, sms * 16);
    if (launch_pdl(prep_gather_kernel, dim3(grid), dim3(128), s, p) != cudaSuccess)
      return PKV_ERR_CUDA;
  }
  return PKV_OK;
}
