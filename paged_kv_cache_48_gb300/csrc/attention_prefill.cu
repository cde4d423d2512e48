// attention_prefill.cu -- paged prefill / chunked-prefill attention on the
// fifth-generation tensor cores (tcgen05, sm_103a).
//
// What it computes (vLLM concept page, "Continuous Batching" with chunked
// prefill, and the PagedAttention pseudocode of its "技术原理" section):
// sequence b brings n_b = query_start_loc[b+1] - query_start_loc[b] query
// tokens whose K/V already sit in the cache as its last n_b tokens
// (seq_lens[b] = c_b + n_b).  Query token i of the chunk is at position
// c_b + i and attends to key positions 0 .. c_b + i, gathered through the
// sequence's block table, with scores scale * q.k, a softmax and a weighted
// sum of V.
//
// One CTA owns two query tiles of one (kv head, sequence).  A tile's 128
// M-rows are the (token, q head) pairs of TQ = floor(128 / g) consecutive
// chunk tokens times the g q heads of the kv head's group (grouped-query
// attention packed along M); the two tiles cover 2 TQ consecutive tokens
// and share every K/V tile the CTA loads.  Per key tile of 128 positions
// (8 cache blocks) and query tile t:
//   S_t  = Q_t K^T   tcgen05.mma, M 128 x N 128 x K head_dim, fp32 in TMEM
//   P_t  = exp2(S_t * scale * log2 e - m)   four softmax warps per tile,
//                    one TMEM lane (one M-row) per thread; bf16 P written
//                    back over the first 64 columns of S_t
//   O_t += P_t V     tcgen05.mma with A read from TMEM, M 128 x N head_dim
//                    x K 128, fp32 in TMEM
// Warp roles: warp 0 issues the TMA loads (Q once; K and V one 16-token
// block and 64-element head_dim slice per copy, at the block id the table
// names), warp 1 owns TMEM and issues the MMAs from one thread, warps 2-5
// and 6-9 run the online softmax and the epilogue of tiles 0 and 1.  The
// MMA order PV_0(i), S_0(i+1), PV_1(i), S_1(i+1) keeps the tensor core on
// one tile while the other tile's probabilities are formed, and since
// MMAs of one thread run in issue order, S_t(i+1) completing also means
// PV_t(i) has read P_t(i) and finished updating O_t.  O is rescaled in TMEM
// only when a row's running maximum grows by more than 2^8 (probabilities
// stay below 256, exact in fp32 and safe in bf16; the final division by l
// uses the same maximum, so the result is unchanged).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "pkv_device.cuh"
#include "pkv_host.h"
#include "tcgen05.cuh"

namespace pkv {

__device__ ErrorWord g_err_prefill = {0ull, 0ull};

struct PrefillParams {
  const int32_t *block_tables;     // [batch, max_blocks]
  const int32_t *seq_lens;         // [batch]
  const int32_t *query_start_loc;  // [batch + 1]
  __nv_bfloat16 *out;              // [num_tokens, num_heads, head_dim]
  long long num_tokens;
  int batch, num_heads, num_kv_heads, group, tile_tokens;
  int num_blocks, max_blocks;
  float scale_log2;   // scale * log2(e) (* k_scale for an fp8 cache)
  float v_scale;      // 1 for bf16
  unsigned long long timeout_ns;
  // Shared-prefix mode (part_o != nullptr): grid.z runs over groups; the
  // members of group z are rows group_start[z] .. group_start[z+1] - 1 of q
  // ([batch, num_heads, head_dim]), all reading the prefix_len[z] tokens
  // named by the first member's table.  Every member row sees every key of
  // its prefix partition (prefix_part_tokens keys, grid.x / pairs_per_part
  // of them), and the CTA writes the partition's (m, l, o / l) to merge
  // slot `partition` of the row instead of a bf16 output.  Which members
  // use these partials (their table and length checks) is decided by the
  // decode pass.
  float *part_o;       // [batch * num_heads, part_stride, head_dim]
  float2 *part_ml;     // [batch * num_heads, part_stride]
  int part_stride;
  const int32_t *group_start;  // [num_groups + 1]
  const int32_t *prefix_len;   // [num_groups], multiples of 16
  int prefix_part_tokens, pairs_per_part, max_prefix_len, max_group_size;
  int pair_major;  // ordinary prefill: grid order, see the kernel
};

// bf16 cache: K and V tiles arrive by TMA directly in the MMA operand
// layout.  fp8 cache: the MMAs run on f16 operands (every E4M3 value is
// exact in f16; q is converted from bf16 once), and the producer warp
// converts each fp8 tile from a TMA staging ring into f16 operand tiles.
// PREFIX: the shared-prefix pass of cascade decode.  Its groups hold few
// query rows, so one query tile, a 2-stage K ring, a 1-stage V ring and 6
// warps (about 128 KB of shared memory, 256 TMEM columns) let one of its
// CTAs share an SM with a decode CTA.
template <bool FP8, int D, bool PREFIX = false>
struct PrefillCfg {
  static constexpr int SLICES = D / 64;          // 64-element head_dim slices
  static constexpr int SLICE_BYTES = 128 * 128;  // 128 rows x 128 bytes
  static constexpr int TILE_BYTES = SLICES * SLICE_BYTES;
  static constexpr int NQT = PREFIX ? 1 : 2;     // query tiles per CTA
  // K is released as soon as both Q K^T products have read it, V only after
  // both P V products: K runs one tile ahead of V and gets the deeper ring.
  // fp8 cache: V converted a tile ahead (2 stages), K just in time for the
  // next Q K^T (1 stage, refilled once both Q K^T of a tile are done).
  static constexpr int KSTAGES = PREFIX ? 2 : (FP8 ? 1 : 3);
  static constexpr int VSTAGES = PREFIX ? 1 : 2;
  static constexpr int KEYS = 128;               // keys per tile (8 blocks)
  static constexpr int STG_HALF = KEYS * D;      // fp8 K (or V) of one tile
  static constexpr int STG_STAGES = FP8 ? 2 : 0;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + NQT * TILE_BYTES;
  static constexpr int V_OFF = K_OFF + KSTAGES * TILE_BYTES;
  static constexpr int STG_OFF = V_OFF + VSTAGES * TILE_BYTES;
  static constexpr int BAR_OFF = STG_OFF + STG_STAGES * 2 * STG_HALF;
  static constexpr int SMEM_BYTES = BAR_OFF + 256 + 1024;  // + alignment slack
  // TMEM: tile t uses columns 256 t .. 256 t + 127 for S_t (P_t in the
  // first 64) and 256 t + 128 .. for O_t.
  static constexpr uint32_t TMEM_COLS = 256 * NQT;
  // warp 0: TMA producer (and fp8 converter); warp 1: TMEM owner and MMA
  // issuer; warps 2-5 / 6-9: softmax of tiles 0 / 1; fp8 cache with two
  // tiles: warps 10 and 11 convert tiles too (12 warps still fit 168
  // registers a thread).
  static constexpr int CONVERTERS = (FP8 && !PREFIX) ? 3 : 1;
  static constexpr int THREADS = PREFIX ? 192 : (FP8 ? 384 : 320);
  static constexpr int MIN_BLOCKS = 1;
};

struct PrefillBars {
  uint64_t q_full;
  uint64_t q_ready;    // fp8 cache: q converted to f16 in place
  uint64_t k_full[3], k_empty[3];
  uint64_t v_full[2], v_empty[2];
  uint64_t stg_full[2];  // fp8 cache: a tile's K and V bytes staged
  uint64_t stg_empty[2]; // fp8 cache: both halves of a stage converted
  uint64_t v_fix;      // last tile: stale V rows past the keys zeroed
  uint64_t s_full[2];  // S_t(i) in TMEM (and PV_t(i-1) complete)
  uint64_t p_full[2];  // P_t(i) in TMEM, O_t rescaled
  uint64_t o_done[2];  // O_t += P_t(i) V(i) complete
  uint32_t tmem_slot;
  int abort_flag;
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// O_t += P_t V with A = P_t read from TMEM (packed bf16 / f16 pairs, the
// even element in the low half; 16 keys = 8 columns per MMA).
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "setp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Slow path of a wait: mbarrier.try_wait with a suspend-time hint, so that
// the waiting thread sleeps until the phase completes (or the hint runs
// out) instead of polling and taking issue slots from the warps that share
// its SM sub-partition; bounded by `limit_ns` of wall time.  Out of line:
// the callers' hot loops keep only the first, non-suspending test.
constexpr uint32_t kWaitHintNs = 10000;

__device__ __noinline__ bool wait_suspended(uint64_t *bar, uint32_t parity,
                                            unsigned long long limit_ns) {
  const uint64_t start = global_timer_ns();
  while (true) {
    uint32_t done;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kWaitHintNs)
        : "memory");
    if (done) return true;
    if (global_timer_ns() - start > limit_ns) return false;
  }
}

__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity,
                                              const PrefillParams &p, volatile int *abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  if (*abort_flag) return false;
  if (wait_suspended(bar, parity, p.timeout_ns)) return true;
  record_error(&g_err_prefill, PKV_ERR_TIMEOUT, -1);
  *abort_flag = 1;
  return false;
}

// The same for code that the whole warp runs together (TMEM loads and
// stores, warp barriers): every lane gets the same answer, so a timeout
// never splits the warp.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const PrefillParams &p,
                                          volatile int *abort_flag) {
  return __all_sync(0xffffffffu, wait_or_abort(bar, parity, p, abort_flag));
}

// 16 E4M3 bytes -> 16 f16 values (two 16-byte chunks, element order kept).
__device__ __forceinline__ void e4m3x16_to_f16(const uint4 v, uint4 &lo, uint4 &hi) {
  e4m3x4_to_f16x2x2(v.x, lo.x, lo.y);
  e4m3x4_to_f16x2x2(v.y, lo.z, lo.w);
  e4m3x4_to_f16x2x2(v.z, hi.x, hi.y);
  e4m3x4_to_f16x2x2(v.w, hi.z, hi.w);
}

// 8 bf16 -> 8 f16 (exact for values inside the f16 range).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v));
  const __half2 h = __float22half2_rn(f);
  return *reinterpret_cast<const uint32_t *>(&h);
}

// Two-lane fp32 arithmetic (sm_100 family): one instruction for a pair of
// elements, each lane rounded as the scalar fma / add would be.  The
// softmax uses them to halve its FMA-pipe instructions; those instructions
// compete for issue slots with the one thread that issues the MMAs, and
// fewer of them shorten the MMA chain of every tile.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n"
      ".reg .b64 ra, rb, rc, rd;\n"
      "mov.b64 ra, {%2, %3};\n"
      "mov.b64 rb, {%4, %5};\n"
      "mov.b64 rc, {%6, %7};\n"
      "fma.rn.f32x2 rd, ra, rb, rc;\n"
      "mov.b64 {%0, %1}, rd;\n"
      "}\n"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{\n"
      ".reg .b64 ra, rb, rd;\n"
      "mov.b64 ra, {%2, %3};\n"
      "mov.b64 rb, {%4, %5};\n"
      "add.rn.f32x2 rd, ra, rb;\n"
      "mov.b64 {%0, %1}, rd;\n"
      "}\n"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <bool FP8>
__device__ __forceinline__ uint32_t pack_p(float lo, float hi) {
  return FP8 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi);
}

template <bool FP8, int D, bool PREFIX>
__global__ void __launch_bounds__(PrefillCfg<FP8, D, PREFIX>::THREADS,
                                  PrefillCfg<FP8, D, PREFIX>::MIN_BLOCKS)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                         const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
  using C = PrefillCfg<FP8, D, PREFIX>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  PrefillBars &bars = *reinterpret_cast<PrefillBars *>(smem + C::BAR_OFF);
  volatile int *abort_flag = &bars.abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Grid (tile pair, kv head, sequence): a (kv head, sequence) unit's pairs
  // run together, its longest (latest tokens) first.  With pair_major,
  // grid (kv head, sequence, tile pair): every unit's last pair first, then
  // every unit's second-to-last, ..., so that CTAs start in order of
  // decreasing causal work across the grid (whole prompts: the short pairs
  // make the tail).  The shared-prefix pass keeps the first form.
  constexpr bool prefix_mode = PREFIX;
  const bool pair_major = !prefix_mode && p.pair_major;
  const int b = pair_major ? blockIdx.y : blockIdx.z;
  const int kvh = pair_major ? blockIdx.x : blockIdx.y;
  const int order = pair_major ? gridDim.z - 1 - blockIdx.z : gridDim.x - 1 - blockIdx.x;
  const int qp = prefix_mode ? order % p.pairs_per_part : order;
  const int pp = prefix_mode ? order / p.pairs_per_part : 0;  // prefix partition
  const int g = p.group, TQ = p.tile_tokens;

  grid_dependency_wait();
  allow_dependent_launch();

  // Query rows q0 .. q0 + n_b - 1 of the pair's "sequence"; the pair sees
  // keys kv_begin .. kv_len - 1 through block-table row table_row.
  int q0, n_b, c = 0, kv_begin = 0, kv_len = 0, table_row = b;
  bool bad_seq;
  const int j0 = qp * C::NQT * TQ;
  // Ordinary prefill reads table row b from entry 0 on: each thread loads
  // one entry alongside the sequence's extent, so that checking the ids
  // costs no round trip of its own.
  int32_t spec_id = 0;
  const bool spec_ok = !prefix_mode && (int)threadIdx.x < p.max_blocks;
  if (spec_ok) spec_id = __ldg(p.block_tables + (size_t)b * p.max_blocks + threadIdx.x);
  if (prefix_mode) {
    q0 = p.group_start[b];
    n_b = p.group_start[b + 1] - q0;
    const int P = p.prefix_len[b];
    // the same structural test the decode pass applies: a group that fails
    // it is attended in full there, so no partial is needed
    bad_seq = n_b < 1 || q0 < 0 || (long long)q0 + n_b > p.num_tokens || P <= 0 || (P & 15) ||
              P > p.max_blocks * 16 || P > p.max_prefix_len || n_b > p.max_group_size ||
              n_b > p.pairs_per_part * C::NQT * TQ;
    if (bad_seq) return;
    kv_begin = pp * p.prefix_part_tokens;
    kv_len = min(P, kv_begin + p.prefix_part_tokens);
    if (j0 >= n_b || kv_begin >= kv_len) return;
    table_row = q0;
  } else {
    q0 = p.query_start_loc[b];
    n_b = p.query_start_loc[b + 1] - q0;
    const int L = p.seq_lens[b];
    c = L - n_b;  // tokens before this chunk
    if (j0 >= n_b && n_b >= 0) return;  // this pair has no query token
    bad_seq = n_b < 0 || c < 0 || L > p.max_blocks * 16 || q0 < 0 ||
              (long long)q0 + n_b > p.num_tokens;
  }
  const bool has_b = C::NQT == 2 && j0 + TQ < n_b;  // a second tile with a query token
  const int j_last = min(j0 + C::NQT * TQ, n_b) - 1;
  if (!prefix_mode) kv_len = c + j_last + 1;  // keys any row of the pair sees
  const int n_tiles = (kv_len - kv_begin + C::KEYS - 1) / C::KEYS;
  const int blk_begin = kv_begin / 16;          // kv_begin is a multiple of 128
  const int nblk = (kv_len + 15) / 16;          // end of the block range
  const int ntq = has_b ? 2 : 1;                // query tiles in use
  const int32_t *row = p.block_tables + (size_t)table_row * p.max_blocks + blk_begin;

  // ---- barriers, TMEM and (ordinary prefill) the first copies, while the
  // ---- block ids are checked.  A copy at an id outside the pool reads
  // ---- zeros (the tensor map's bounds), so nothing faults before the check.
  if (threadIdx.x == 0) {
    mbar_init(&bars.q_full, 1);
    mbar_init(&bars.q_ready, 4 * ntq);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.stg_full[s], 1);
      mbar_init(&bars.stg_empty[s], C::CONVERTERS);
    }
    for (int s = 0; s < C::KSTAGES; ++s) {
      mbar_init(&bars.k_full[s], C::CONVERTERS);
      mbar_init(&bars.k_empty[s], 1);
    }
    for (int s = 0; s < C::VSTAGES; ++s) {
      mbar_init(&bars.v_full[s], C::CONVERTERS);
      mbar_init(&bars.v_empty[s], 1);
    }
    mbar_init(&bars.v_fix, C::CONVERTERS);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars.s_full[t], 1);
      mbar_init(&bars.p_full[t], 4);
      mbar_init(&bars.o_done[t], 1);
    }
    bars.abort_flag = 0;
    fence_barrier_init();
  }
  const bool early = !prefix_mode && !bad_seq;  // first copies before the check
  const uint64_t pol = l2_policy_evict_normal();
  constexpr uint32_t TB = C::TILE_BYTES;
  // bf16: K(0) and V(0); fp8: the staging of tiles 0 and 1
  auto first_copies = [&]() {
    if constexpr (!FP8) {
      const int nv = min(8, nblk - blk_begin);
      mbar_arrive_expect_tx(&bars.k_full[0], nv * C::SLICES * 2048);
      mbar_arrive_expect_tx(&bars.v_full[0], nv * C::SLICES * 2048);
      for (int j = 0; j < nv; ++j) {
        const int blk = row[j];
        for (int s = 0; s < C::SLICES; ++s) {
          tma_load_5d(smem + C::K_OFF + s * C::SLICE_BYTES + j * 2048, &kmap, &bars.k_full[0], 0,
                      0, kvh, s, blk, pol);
          tma_load_5d(smem + C::V_OFF + s * C::SLICE_BYTES + j * 2048, &vmap, &bars.v_full[0], 0,
                      0, kvh, s, blk, pol);
        }
      }
    } else {
      for (int i = 0; i < min(2, n_tiles); ++i) {
        const int nv = min(8, nblk - blk_begin - 8 * i);
        mbar_arrive_expect_tx(&bars.stg_full[i], 2 * nv * 16 * D);
        uint8_t *dst = smem + C::STG_OFF + i * 2 * C::STG_HALF;
        for (int j = 0; j < nv; ++j) {
          const int blk = row[8 * i + j];
          tma_load_5d(dst + j * 16 * D, &kmap, &bars.stg_full[i], 0, 0, kvh, 0, blk, pol);
          tma_load_5d(dst + C::STG_HALF + j * 16 * D, &vmap, &bars.stg_full[i], 0, 0, kvh, 0, blk,
                      pol);
        }
      }
    }
  };
  if (threadIdx.x == 0 && !bad_seq) {
    prefetch_tensormap(&qmap);
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    mbar_arrive_expect_tx(&bars.q_full, ntq * C::SLICES * 128 * g * TQ);
    for (int t = 0; t < ntq; ++t)
      for (int s = 0; s < C::SLICES; ++s)
        tc::tma_load_4d(smem_u32(smem + C::Q_OFF + t * TB + s * C::SLICE_BYTES), &qmap,
                        smem_u32(&bars.q_full), 0, kvh * g, s, q0 + j0 + t * TQ);
    if (early) first_copies();
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(&bars.tmem_slot), C::TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();

  // every block id the pair reads must be inside the pool
  int bad = bad_seq ? 1 : 0;
  if (!bad) {
    const int32_t *trow = p.block_tables + (size_t)table_row * p.max_blocks;
    for (int j = blk_begin + threadIdx.x; j < nblk; j += blockDim.x) {
      const int32_t id = (spec_ok && j == (int)threadIdx.x) ? spec_id : trow[j];
      if (id < 0 || id >= p.num_blocks) {
        bad = 1;
        record_error(&g_err_prefill, PKV_ERR_RANGE, (long long)table_row * p.max_blocks + j);
      }
    }
  } else if (threadIdx.x == 0) {
    record_error(&g_err_prefill, PKV_ERR_RANGE, b);
  }
  if (__syncthreads_or(bad)) {
    // let the copies already issued land, release TMEM, zero the pair's
    // output rows of a valid token range (in shared-prefix mode: an empty
    // partial, weight zero in the merge), then leave
    if (threadIdx.x == 0 && !bad_seq) {
      mbar_wait_bounded(&bars.q_full, 0, p.timeout_ns);
      if (early) {
        if constexpr (!FP8) {
          mbar_wait_bounded(&bars.k_full[0], 0, p.timeout_ns);
          mbar_wait_bounded(&bars.v_full[0], 0, p.timeout_ns);
        } else {
          for (int i = 0; i < min(2, n_tiles); ++i)
            mbar_wait_bounded(&bars.stg_full[i], 0, p.timeout_ns);
        }
      }
    }
    if (warp == 1) {
      tc::fence_after_sync();
      tc::tmem_dealloc(bars.tmem_slot, C::TMEM_COLS);
    }
    if (!bad_seq) {
      const int rows = (j_last - j0 + 1) * g;
      for (int idx = threadIdx.x; idx < rows * (D / 8); idx += blockDim.x) {
        const int r = idx / (D / 8), ch = idx % (D / 8);
        const long long tok = (long long)q0 + j0 + r / g;
        const size_t orow = (size_t)tok * p.num_heads + kvh * g + r % g;
        if (prefix_mode) {
          float *po = p.part_o + (orow * p.part_stride + pp) * D + ch * 8;
          *reinterpret_cast<float4 *>(po) = make_float4(0.f, 0.f, 0.f, 0.f);
          *reinterpret_cast<float4 *>(po + 4) = make_float4(0.f, 0.f, 0.f, 0.f);
          if (ch == 0) p.part_ml[orow * p.part_stride + pp] = make_float2(-INFINITY, 0.f);
        } else {
          *reinterpret_cast<uint4 *>(p.out + orow * D + ch * 8) = make_uint4(0, 0, 0, 0);
        }
      }
    }
    return;
  }
  tc::fence_after_sync();
  const uint32_t tmem = bars.tmem_slot;

  const uint32_t sQ = smem_u32(smem + C::Q_OFF);
  const uint32_t sK = smem_u32(smem + C::K_OFF);
  const uint32_t sV = smem_u32(smem + C::V_OFF);

  if (warp == 0 || warp >= 10) {
    // ------------------------------------------------------------ producer
    // (the Q tiles, and for ordinary prefill the first copies, went out
    // before the block-id check)
    if (warp == 0 && lane == 0 && !early) first_copies();
    if constexpr (!FP8) {
      if (lane == 0) {
        // K(i + 1) is issued before V(i): Q K^T of the next tile needs its
        // keys while the current tile's probabilities are still formed.
        auto issue = [&](bool is_k, int i) -> bool {
          const int stages = is_k ? C::KSTAGES : C::VSTAGES;
          const int st = i % stages;
          uint64_t *empty = is_k ? &bars.k_empty[st] : &bars.v_empty[st];
          uint64_t *full = is_k ? &bars.k_full[st] : &bars.v_full[st];
          if (i >= stages && !wait_or_abort(empty, ((i / stages) - 1) & 1, p, abort_flag))
            return false;
          const int nv = min(8, nblk - blk_begin - 8 * i);
          mbar_arrive_expect_tx(full, nv * C::SLICES * 2048);
          uint8_t *dst = smem + (is_k ? C::K_OFF : C::V_OFF) + st * TB;
          for (int j = 0; j < nv; ++j) {
            const int blk = row[8 * i + j];
            for (int s = 0; s < C::SLICES; ++s)
              tma_load_5d(dst + s * C::SLICE_BYTES + j * 2048, is_k ? &kmap : &vmap, full, 0, 0,
                          kvh, s, blk, pol);
          }
          return true;
        };
        // K(0) and V(0) are in flight already
        bool go = true;
        for (int i = 0; go && i < n_tiles; ++i) {
          if (i + 1 < n_tiles) go = issue(true, i + 1);
          if (i > 0) go = go && issue(false, i);
        }
      }
      __syncwarp();
      // The last tile's V rows past kv_len hold bytes that are not part of
      // the sequence (stale cache contents or an older stage): zero them so
      // that a zero probability never meets a NaN.
      const int last = n_tiles - 1, st = last % C::VSTAGES;
      if (warp_wait(&bars.v_full[st], (last / C::VSTAGES) & 1, p, abort_flag)) {
        const int first = kv_len - kv_begin - last * C::KEYS;
        uint8_t *vbase = smem + C::V_OFF + st * TB;
        for (int idx = first * 8 + lane; idx < C::KEYS * 8; idx += 32)
          for (int s = 0; s < C::SLICES; ++s)
            *reinterpret_cast<uint4 *>(vbase + s * C::SLICE_BYTES + idx * 16) =
                make_uint4(0, 0, 0, 0);
        tc::fence_proxy_async_smem();
      }
    } else {
      // fp8 cache: TMA stages each tile's K and V bytes (one box of 16 rows
      // per block, rows of head_dim bytes, unswizzled) two tiles ahead; the
      // whole warp converts them into the f16 operand tiles.
      auto stage_load = [&](int i) {
        const int sst = i % 2;
        const int nv = min(8, nblk - blk_begin - 8 * i);
        mbar_arrive_expect_tx(&bars.stg_full[sst], 2 * nv * 16 * D);
        uint8_t *dst = smem + C::STG_OFF + sst * 2 * C::STG_HALF;
        for (int j = 0; j < nv; ++j) {
          const int blk = row[8 * i + j];
          tma_load_5d(dst + j * 16 * D, &kmap, &bars.stg_full[sst], 0, 0, kvh, 0, blk, pol);
          tma_load_5d(dst + C::STG_HALF + j * 16 * D, &vmap, &bars.stg_full[sst], 0, 0, kvh, 0, blk,
                      pol);
        }
      };
      const int ci = warp == 0 ? 0 : warp - 9;  // converter index
      constexpr int STRIDE = 32 * C::CONVERTERS;
      // (tiles 0 and 1 are staged already)
      __syncwarp();
      // Convert tile i's K or V; V rows past the sequence's keys become 0.
      auto convert = [&](bool is_k, int i) -> bool {
        const int sst = i % 2;
        const int stages = is_k ? C::KSTAGES : C::VSTAGES;
        const int st = i % stages;
        uint64_t *empty = is_k ? &bars.k_empty[st] : &bars.v_empty[st];
        if (!warp_wait(&bars.stg_full[sst], (i / 2) & 1, p, abort_flag) ||
            (i >= stages && !warp_wait(empty, ((i / stages) - 1) & 1, p, abort_flag)))
          return false;
        const uint8_t *src = smem + C::STG_OFF + sst * 2 * C::STG_HALF + (is_k ? 0 : C::STG_HALF);
        uint8_t *dst = smem + (is_k ? C::K_OFF : C::V_OFF) + st * TB;
        const int loaded = min(8, nblk - blk_begin - 8 * i) * 16;
        const int rows = is_k ? loaded : min(C::KEYS, kv_len - kv_begin - i * C::KEYS);
        const int last_row = is_k ? loaded : C::KEYS;  // K rows past `loaded` stay stale (masked)
        constexpr int CH = D / 16;                     // 16-byte fp8 chunks per row
        const int total = last_row * CH;
        if (rows >= last_row) {
          // Every row comes from the staging (full tiles, and K): a lane
          // keeps one 16-byte column, so its source and destination
          // columns are fixed and only the row moves (rows row0 + k RSTEP).
          static_assert(STRIDE % CH == 0, "converter lanes keep their column");
          constexpr int RSTEP = STRIDE / CH;
          const int tid = ci * 32 + lane;
          const int cc = tid % CH;
          const int c16 = ((cc * 16) % 64) / 8;  // 16-byte column of the low half
          const uint8_t *s0 = src + cc * 16;
          uint8_t *d0 = dst + ((cc * 16) / 64) * C::SLICE_BYTES;
          auto put = [&](int rr, const uint4 &v) {
            uint4 lo, hi;
            e4m3x16_to_f16(v, lo, hi);
            uint8_t *base = d0 + rr * 128;
            const int sw = rr & 7;
            *reinterpret_cast<uint4 *>(base + ((c16 ^ sw) << 4)) = lo;
            *reinterpret_cast<uint4 *>(base + (((c16 + 1) ^ sw) << 4)) = hi;
          };
          int r = tid / CH;
          // four rows per lane in flight: loads first, then convert + store
          for (; r + 3 * RSTEP < last_row; r += 4 * RSTEP) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
              v[u] = *reinterpret_cast<const uint4 *>(s0 + (r + u * RSTEP) * D);
#pragma unroll
            for (int u = 0; u < 4; ++u) put(r + u * RSTEP, v[u]);
          }
          for (; r < last_row; r += RSTEP) put(r, *reinterpret_cast<const uint4 *>(s0 + r * D));
        } else
        // four chunks per lane in flight: loads first, then convert + store
        for (int q0c = ci * 32; q0c < total; q0c += 4 * STRIDE) {
          uint4 v[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int q = q0c + u * STRIDE + lane, r = q / CH;
            v[u] = (q < total && r < rows)
                       ? *reinterpret_cast<const uint4 *>(src + r * D + (q % CH) * 16)
                       : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int q = q0c + u * STRIDE + lane;
            if (q >= total) break;
            const int r = q / CH, cb = (q % CH) * 16;  // row, first element
            uint4 lo, hi;
            e4m3x16_to_f16(v[u], lo, hi);  // zero bytes give +0
            const int c16 = (cb % 64) / 8;
            uint8_t *base = dst + (cb / 64) * C::SLICE_BYTES + r * 128;
            *reinterpret_cast<uint4 *>(base + ((c16 ^ (r & 7)) * 16)) = lo;
            *reinterpret_cast<uint4 *>(base + (((c16 + 1) ^ (r & 7)) * 16)) = hi;
          }
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(smem_u32(is_k ? &bars.k_full[st] : &bars.v_full[st]));
        return true;
      };
      bool go = convert(true, 0);
      for (int i = 0; go && i < n_tiles; ++i) {
        go = convert(false, i);
        if (go && i + 1 < n_tiles) go = convert(true, i + 1);
        __syncwarp();
        // both halves of stage i % 2 (K(i) in the previous round, V(i) in
        // this one) are converted by every converter: warp 0 refills it
        if (go && lane == 0) tc::mbar_arrive(smem_u32(&bars.stg_empty[i % 2]));
        if (go && warp == 0 && lane == 0 && i + 2 < n_tiles) {
          if (!wait_or_abort(&bars.stg_empty[i % 2], (i / 2) & 1, p, abort_flag))
            go = false;
          else
            stage_load(i + 2);
        }
        go = __all_sync(0xffffffffu, go);
      }
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(smem_u32(&bars.v_fix));
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = FP8 ? tc::idesc_f16_f32(128, C::KEYS, false, false)
                                   : tc::idesc_bf16_f32(128, C::KEYS, false, false);
      constexpr uint32_t idO = FP8 ? tc::idesc_f16_f32(128, D, false, true)
                                   : tc::idesc_bf16_f32(128, D, false, true);
      // Descriptors are built once; stepping K adds the byte offset / 16 to
      // the start-address field (bits 0-13), which never carries out.
      const uint64_t q_desc0 = tc::smem_desc(sQ, 16, 1024, tc::kSwizzle128B);
      const uint64_t k_desc0 = tc::smem_desc(sK, 16, 1024, tc::kSwizzle128B);
      const uint64_t v_desc0 = tc::smem_desc(sV, C::SLICE_BYTES, 1024, tc::kSwizzle128B);
      auto issue_s = [&](int t, int i) {
        const uint64_t qd = q_desc0 + ((t * TB) >> 4);
        const uint64_t kd = k_desc0 + (((i % C::KSTAGES) * TB) >> 4);
        const uint32_t d = tmem + 256 * t;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = ((k / 4) * C::SLICE_BYTES + (k % 4) * 32) >> 4;
          tc::mma_bf16_ss(d, qd + off, kd + off, idS, k > 0);
        }
        tc::mma_commit(smem_u32(&bars.s_full[t]));
        if (t == ntq - 1) tc::mma_commit(smem_u32(&bars.k_empty[i % C::KSTAGES]));
      };
      auto issue_pv = [&](int t, int i) {
        const uint64_t vd = v_desc0 + (((i % C::VSTAGES) * TB) >> 4);
        const uint32_t d = tmem + 256 * t + 128, a = tmem + 256 * t;
#pragma unroll
        for (int k = 0; k < C::KEYS / 16; ++k)
          mma_bf16_ts(d, a + 8 * k, vd + ((k * 2048) >> 4), idO, (i > 0 || k > 0) ? 1u : 0u);
        tc::mma_commit(smem_u32(&bars.o_done[t]));
        if (t == ntq - 1) tc::mma_commit(smem_u32(&bars.v_empty[i % C::VSTAGES]));
      };
      bool ok = wait_or_abort(FP8 ? &bars.q_ready : &bars.q_full, 0, p, abort_flag) &&
                wait_or_abort(&bars.k_full[0], 0, p, abort_flag);
      if (ok) {
        tc::fence_after_sync();
        for (int t = 0; t < ntq; ++t) issue_s(t, 0);
      }
      for (int i = 0; ok && i < n_tiles; ++i) {
        const int vst = i % C::VSTAGES;
        ok = wait_or_abort(&bars.v_full[vst], (i / C::VSTAGES) & 1, p, abort_flag) &&
             (i + 1 < n_tiles || wait_or_abort(&bars.v_fix, 0, p, abort_flag));
        const bool next = i + 1 < n_tiles;
        for (int t = 0; ok && t < ntq; ++t) {
          if (!(ok = wait_or_abort(&bars.p_full[t], i & 1, p, abort_flag))) break;
          tc::fence_after_sync();
          issue_pv(t, i);
          if (next) {
            if (t == 0 && !(ok = wait_or_abort(&bars.k_full[(i + 1) % C::KSTAGES],
                                              ((i + 1) / C::KSTAGES) & 1, p, abort_flag)))
              break;
            tc::fence_after_sync();
            issue_s(t, i + 1);
          }
        }
      }
    }
    __syncwarp();
  } else if (warp < 2 + 4 * C::NQT) {
    // ------------------------------------------------------------ softmax
    const int t = (warp - 2) / 4;  // query tile of this warp
    const int quarter = warp % 4;
    const int r = quarter * 32 + lane;  // M-row = TMEM lane
    const uint32_t lane_addr = tmem + 256 * t + ((uint32_t)(quarter * 32) << 16);
    const uint32_t s_addr = lane_addr, o_addr = lane_addr + 128;
    const int jr = j0 + t * TQ + r / g;
    const bool row_valid = r < TQ * g && jr < n_b;
    // last key this row sees (every prefix key in shared-prefix mode)
    const int lim = row_valid && !prefix_mode ? c + jr : kv_len - 1;
    float m_used = -INFINITY, l = 0.f;
    bool ok = t == 0 || has_b;
    if (FP8 && ok) {
      // q of this tile from bf16 to f16, in place (same swizzled layout)
      if ((ok = warp_wait(&bars.q_full, 0, p, abort_flag))) {
        uint8_t *qt = smem + C::Q_OFF + t * TB;
        for (int idx = quarter * 32 + lane; idx < TB / 16; idx += 128) {
          uint4 v = *reinterpret_cast<uint4 *>(qt + idx * 16);
          v.x = bf16x2_to_f16x2(v.x);
          v.y = bf16x2_to_f16x2(v.y);
          v.z = bf16x2_to_f16x2(v.z);
          v.w = bf16x2_to_f16x2(v.w);
          *reinterpret_cast<uint4 *>(qt + idx * 16) = v;
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(smem_u32(&bars.q_ready));
      }
    }
    for (int i = 0; ok && i < n_tiles; ++i) {
      if (!(ok = warp_wait(&bars.s_full[t], i & 1, p, abort_flag))) break;
      tc::fence_after_sync();
      uint32_t sr[4][32];
#pragma unroll
      for (int q = 0; q < 4; ++q) tc::tmem_ld_32x32b_x32(s_addr + q * 32, sr[q]);
      tc::tmem_wait_ld();

      const int key0 = kv_begin + i * C::KEYS;
      if (key0 + C::KEYS - 1 > lim) {
        // keys past this row's last visible position are excluded by
        // selection (a stale NaN in the cache becomes -inf, never a factor)
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (key0 + q * 32 + e > lim) sr[q][e] = __float_as_uint(-INFINITY);
      }
      // Row maximum of the raw scores in eight independent chains, two new
      // scores per step (the scale is positive, so it commutes with the
      // maximum).
      float mx[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = -INFINITY;
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          mx[(e / 2) % 8] = max3(mx[(e / 2) % 8], __uint_as_float(sr[q][e]),
                                 __uint_as_float(sr[q][e + 1]));
      const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) *
                       p.scale_log2;
      const bool rescale = mt > m_used + 8.f;
      const float m_new = rescale ? mt : m_used;
      const float alpha = rescale ? fast_exp2(m_used - m_new) : 1.f;  // 0 on the first tile
      // Eight partial sums of p kept as four lane pairs: pair j holds the
      // sums of columns 2j and 2j + 1 (mod 8).
      float2 ls[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) ls[k] = make_float2(0.f, 0.f);
      const float2 scale2 = make_float2(p.scale_log2, p.scale_log2);
      const float2 neg_m2 = make_float2(-m_new, -m_new);
      // P as packed bf16 pairs, written in place over the consumed scores
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 x = fma2(
              make_float2(__uint_as_float(sr[q][e]), __uint_as_float(sr[q][e + 1])), scale2,
              neg_m2);
          const float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
          ls[(e / 2) % 4] = add2(ls[(e / 2) % 4], make_float2(p0, p1));
          sr[q][e / 2] = pack_p<FP8>(p0, p1);
        }
      l = l * alpha + (((ls[0].x + ls[0].y) + (ls[1].x + ls[1].y)) +
                       ((ls[2].x + ls[2].y) + (ls[3].x + ls[3].y)));
      m_used = m_new;
      // s_full(i) also means PV_t(i-1) is complete: O_t may be rescaled
      if (i > 0 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
        for (int q = 0; q < D / 32; ++q) {
          uint32_t o[32];
          tc::tmem_ld_32x32b_x32(o_addr + q * 32, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tc::tmem_st_32x32b_x32(o_addr + q * 32, o);
        }
      }
      // P_t over the first 64 columns of S_t
#pragma unroll
      for (int q = 0; q < 4; ++q) tc::tmem_st_32x32b_x16(s_addr + 16 * q, sr[q]);
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(smem_u32(&bars.p_full[t]));
    }
    // epilogue: O_t / l -> bf16 rows of out, or the partition's partial
    if (ok && warp_wait(&bars.o_done[t], (n_tiles - 1) & 1, p, abort_flag)) {
      tc::fence_after_sync();
      const float inv = l > 0.f ? p.v_scale / l : 0.f;
      const size_t orow_i = (size_t)(q0 + jr) * p.num_heads + kvh * g + r % g;
      if (prefix_mode && row_valid) p.part_ml[orow_i * p.part_stride + pp] = make_float2(m_used, l);
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        uint32_t o[32];
        tc::tmem_ld_32x32b_x32(o_addr + q * 32, o);
        tc::tmem_wait_ld();
        if (row_valid && prefix_mode) {
          float *po = p.part_o + (orow_i * p.part_stride + pp) * D + q * 32;
#pragma unroll
          for (int h = 0; h < 8; ++h)
            *reinterpret_cast<float4 *>(po + 4 * h) =
                make_float4(__uint_as_float(o[4 * h + 0]) * inv, __uint_as_float(o[4 * h + 1]) * inv,
                            __uint_as_float(o[4 * h + 2]) * inv, __uint_as_float(o[4 * h + 3]) * inv);
        } else if (row_valid) {
          __nv_bfloat16 *orow = p.out + orow_i * D;
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[8 * h + 0]) * inv, __uint_as_float(o[8 * h + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(o[8 * h + 2]) * inv, __uint_as_float(o[8 * h + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(o[8 * h + 4]) * inv, __uint_as_float(o[8 * h + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(o[8 * h + 6]) * inv, __uint_as_float(o[8 * h + 7]) * inv);
            *reinterpret_cast<uint4 *>(orow + q * 32 + h * 8) = v;
          }
        }
      }
    }
  }

  // Before TMEM is released every MMA this CTA issued must have completed:
  // the softmax warps waited for the last P V of their tile, and the
  // commits behind it track every earlier MMA.  On an abort, wait for the
  // last commit with a bound.
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    if (*abort_flag && lane == 0)
      mbar_wait_bounded(&bars.o_done[has_b ? 1 : 0], (n_tiles - 1) & 1, p.timeout_ns);
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 prefill_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// K or V cache: dims {64, 16 tokens, num_kv_heads, head_dim / 64, num_blocks},
// box {64, 16, 1, 1, 1}: one 64-element head_dim slice of one kv head of
// one block lands as 16 consecutive 128-byte swizzled rows.
// fp8 cache: dims {head_dim, 16 tokens, num_kv_heads, 1, num_blocks}, box
// {head_dim, 16, 1, 1, 1}, unswizzled: a block-head lands as 16 rows of
// head_dim bytes for the conversion into f16 operand tiles.
bool encode_prefill_cache_map(CUtensorMap *map, void *base, const pkv_cache *c) {
  auto fn = prefill_encode_fn();
  if (!fn) return false;
  if (c->dtype == PKV_FP8_E4M3) {
    const cuuint64_t row = (cuuint64_t)c->head_dim;
    cuuint64_t dims[5] = {row, 16, (cuuint64_t)c->num_kv_heads, 1, (cuuint64_t)c->num_blocks};
    cuuint64_t strides[4] = {row * c->num_kv_heads, row, row, row * c->num_kv_heads * 16};
    cuuint32_t box[5] = {(cuuint32_t)row, 16, 1, 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  const cuuint64_t row = (cuuint64_t)c->head_dim * 2;
  cuuint64_t dims[5] = {64, 16, (cuuint64_t)c->num_kv_heads, (cuuint64_t)c->head_dim / 64,
                        (cuuint64_t)c->num_blocks};
  cuuint64_t strides[4] = {row * c->num_kv_heads, row, 128, row * c->num_kv_heads * 16};
  cuuint32_t box[5] = {64, 16, 1, 1, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Queries [num_tokens, num_heads, head_dim]: dims {64, num_heads,
// head_dim / 64, num_tokens}, box {64, g, 1, TQ}: the g heads of one kv
// head's group for TQ consecutive tokens, token-major, one 128-byte row per
// (token, head).  Rows past num_tokens read as zeros.
bool encode_query_map(CUtensorMap *map, const void *q, long long num_tokens, int num_heads,
                      int head_dim, int g, int tq) {
  auto fn = prefill_encode_fn();
  if (!fn) return false;
  const cuuint64_t row = (cuuint64_t)head_dim * 2;
  cuuint64_t dims[4] = {64, (cuuint64_t)num_heads, (cuuint64_t)head_dim / 64,
                        (cuuint64_t)num_tokens};
  cuuint64_t strides[3] = {row, 128, row * num_heads};
  cuuint32_t box[4] = {64, (cuuint32_t)g, 1, (cuuint32_t)tq};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(q), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct PrefillMapEntry {
  void *key_cache, *value_cache;
  int32_t num_blocks, num_kv_heads, head_dim, dtype;
  CUtensorMap k, v;
};

bool get_prefill_maps(const pkv_cache *c, CUtensorMap *k, CUtensorMap *v) {
  static std::mutex mu;
  static PrefillMapEntry entries[8];
  static int n_entries = 0, next = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_entries; ++i) {
    const PrefillMapEntry &e = entries[i];
    if (e.key_cache == c->key_cache && e.value_cache == c->value_cache &&
        e.num_blocks == c->num_blocks && e.num_kv_heads == c->num_kv_heads &&
        e.head_dim == c->head_dim && e.dtype == c->dtype) {
      *k = e.k;
      *v = e.v;
      return true;
    }
  }
  PrefillMapEntry e;
  e.key_cache = c->key_cache;
  e.value_cache = c->value_cache;
  e.num_blocks = c->num_blocks;
  e.num_kv_heads = c->num_kv_heads;
  e.head_dim = c->head_dim;
  e.dtype = c->dtype;
  if (!encode_prefill_cache_map(&e.k, c->key_cache, c) ||
      !encode_prefill_cache_map(&e.v, c->value_cache, c))
    return false;
  entries[next] = e;
  next = (next + 1) % 8;
  if (n_entries < 8) ++n_entries;
  *k = e.k;
  *v = e.v;
  return true;
}

template <bool FP8, int D, bool PREFIX>
pkv_status launch_prefill(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                          const PrefillParams &p, int q_tiles, cudaStream_t s) {
  using C = PrefillCfg<FP8, D, PREFIX>;
  static int configured[64] = {0};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PKV_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!configured[dev]) {
      if (cudaFuncSetAttribute(paged_prefill_kernel<FP8, D, PREFIX>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               C::SMEM_BYTES) != cudaSuccess)
        return PKV_ERR_CUDA;
      configured[dev] = 1;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = p.pair_major ? dim3(p.num_kv_heads, p.batch, q_tiles)
                             : dim3(q_tiles, p.num_kv_heads, p.batch);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, paged_prefill_kernel<FP8, D, PREFIX>, mq, mk, mv, p) !=
      cudaSuccess)
    return PKV_ERR_CUDA;
  return PKV_OK;
}

template <bool PREFIX>
pkv_status dispatch_prefill(const pkv_cache *cache, const CUtensorMap &mq, const CUtensorMap &mk,
                            const CUtensorMap &mv, const PrefillParams &p, int q_tiles,
                            cudaStream_t s) {
  const bool fp8 = cache->dtype == PKV_FP8_E4M3;
  if (cache->head_dim == 128)
    return fp8 ? launch_prefill<true, 128, PREFIX>(mq, mk, mv, p, q_tiles, s)
               : launch_prefill<false, 128, PREFIX>(mq, mk, mv, p, q_tiles, s);
  return fp8 ? launch_prefill<true, 64, PREFIX>(mq, mk, mv, p, q_tiles, s)
             : launch_prefill<false, 64, PREFIX>(mq, mk, mv, p, q_tiles, s);
}

// Score and output scales: fp8 folds k_scale into the score scale and
// v_scale into the output.
void set_scales(PrefillParams *p, const pkv_cache *cache, float scale) {
  const bool fp8 = cache->dtype == PKV_FP8_E4M3;
  p->scale_log2 = scale * 1.4426950408889634f * (fp8 ? cache->k_scale : 1.f);
  p->v_scale = fp8 ? cache->v_scale : 1.f;
}

}  // namespace

pkv_status launch_prefix_partials(const void *q, const pkv_cache *cache,
                                  const int32_t *block_tables, int32_t max_blocks,
                                  const int32_t *seq_lens, const int32_t *group_start,
                                  const int32_t *prefix_len, int32_t num_groups,
                                  int32_t max_group_size, int32_t max_prefix_len, int32_t batch,
                                  int32_t num_heads, float scale, float *part_o, float2 *part_ml,
                                  int part_stride, int prefix_part_tokens, cudaStream_t s) {
  const int g = num_heads / cache->num_kv_heads;
  const int tq = 128 / g;
  const int pairs = std::max(1, (max_group_size + tq - 1) / tq);  // one query tile per CTA
  const int parts = std::max(1, (max_prefix_len + prefix_part_tokens - 1) / prefix_part_tokens);
  if ((int64_t)pairs * parts > INT32_MAX || num_groups > 65535) return PKV_ERR_ARG;
  CUtensorMap mq, mk, mv;
  if (!encode_query_map(&mq, q, batch, num_heads, cache->head_dim, g, tq)) return PKV_ERR_CUDA;
  if (!get_prefill_maps(cache, &mk, &mv)) return PKV_ERR_CUDA;
  PrefillParams p;
  std::memset(&p, 0, sizeof p);
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.num_tokens = batch;
  p.batch = num_groups;
  p.num_heads = num_heads;
  p.num_kv_heads = cache->num_kv_heads;
  p.group = g;
  p.tile_tokens = tq;
  p.num_blocks = cache->num_blocks;
  p.max_blocks = max_blocks;
  set_scales(&p, cache, scale);
  p.timeout_ns = 2000000000ull;
  p.part_o = part_o;
  p.part_ml = part_ml;
  p.part_stride = part_stride;
  p.group_start = group_start;
  p.prefix_len = prefix_len;
  p.prefix_part_tokens = prefix_part_tokens;
  p.pairs_per_part = pairs;
  p.max_prefix_len = max_prefix_len;
  p.max_group_size = max_group_size;
  return dispatch_prefill<true>(cache, mq, mk, mv, p, pairs * parts, s);
}

const void *error_word_prefill() { return &g_err_prefill; }

}  // namespace pkv

using namespace pkv;

extern "C" pkv_status paged_attention_prefill(const void *q, const pkv_cache *cache,
                                              const int32_t *block_tables, int32_t max_blocks,
                                              const int32_t *seq_lens,
                                              const int32_t *query_start_loc, int32_t batch,
                                              int32_t num_heads, int64_t num_tokens, float scale,
                                              void *out, int32_t max_query_len, void *stream) {
  pkv_status st = validate_cache(cache);
  if (st != PKV_OK) return st;
  if (cache->dtype == PKV_FP8_E4M3 && !(cache->k_scale > 0.f && cache->v_scale > 0.f))
    return PKV_ERR_ARG;
  if (batch < 0 || num_heads <= 0 || max_blocks <= 0 || num_tokens < 0 || max_query_len < 0 ||
      !std::isfinite(scale) || !(scale > 0.f))
    return PKV_ERR_ARG;
  if (num_heads % cache->num_kv_heads) return PKV_ERR_SHAPE;
  const int g = num_heads / cache->num_kv_heads;
  if (g > 128) return PKV_ERR_SHAPE;
  if (batch == 0 || num_tokens == 0 || max_query_len == 0) return PKV_OK;
  if (!q || !out || !block_tables || !seq_lens || !query_start_loc) return PKV_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15)
    return PKV_ERR_ARG;
  if (batch > 65535 || cache->num_kv_heads > 65535 || num_tokens > INT32_MAX) return PKV_ERR_ARG;
  const int tq = 128 / g;
  const int64_t q_tiles = ((int64_t)max_query_len + 2 * tq - 1) / (2 * tq);  // tile pairs
  if (q_tiles > INT32_MAX) return PKV_ERR_ARG;

  CUtensorMap mq, mk, mv;
  if (!encode_query_map(&mq, q, num_tokens, num_heads, cache->head_dim, g, tq))
    return PKV_ERR_CUDA;
  if (!get_prefill_maps(cache, &mk, &mv)) return PKV_ERR_CUDA;

  PrefillParams p;
  std::memset(&p, 0, sizeof p);
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.query_start_loc = query_start_loc;
  p.out = static_cast<__nv_bfloat16 *>(out);
  p.num_tokens = num_tokens;
  p.batch = batch;
  p.num_heads = num_heads;
  p.num_kv_heads = cache->num_kv_heads;
  p.group = g;
  p.tile_tokens = tq;
  p.num_blocks = cache->num_blocks;
  p.max_blocks = max_blocks;
  set_scales(&p, cache, scale);
  p.timeout_ns = 2000000000ull;
  // Whole prompts (a table no wider than twice the longest chunk, so little
  // history) are ordered pair-major: their CTAs' work varies with the pair
  // alone, and longest-first across the grid shortens the tail (whole
  // 1024-token prompts 608 -> 657 TFLOP/s).  Chunks after long histories
  // keep each unit's pairs together (pair-major measured 1171 -> 1125 there).
  p.pair_major = (int64_t)max_blocks * 16 <= 2 * (int64_t)max_query_len && q_tiles <= 65535;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return dispatch_prefill<false>(cache, mq, mk, mv, p, (int)q_tiles, s);
}
