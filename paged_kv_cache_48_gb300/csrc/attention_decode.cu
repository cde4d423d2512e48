// attention_decode.cu -- PagedAttention decode for sm_103a.
//
// What it computes (vLLM concept page, compassingai.com, "技术原理"): for
// every sequence b and query head h, gather the KV blocks named by the
// sequence's block table, then softmax(scale * q . K^T) . V over the
// seq_lens[b] cached tokens.  GQA: q head h reads kv head h / group (same
// page: fewer KV heads than Q heads).  The gather happens inside the kernel
// (vLLM internals, naphjohn.github.io, §4.1); positions past seq_len are
// excluded by selection, never multiplied by zero (vLLM v0.17.1 notes,
// admirer.cn, "重点：35219": 0 x NaN = NaN).
//
// Schedule: one CTA per (kv head, query sub-group of <= 8 heads, partition
// of a sequence, sequence); the grid is ordered heads-fastest.  The CTA's 4
// warps take the partition's 16-token blocks round-robin, and each warp
// streams its blocks through a private ring of shared-memory stages: lane 0
// reads the physical block id from the block table and issues one TMA load
// per K and per V tile (5-D tensor map over [num_blocks, 16, num_kv_heads,
// head_dim] laid out so that one box is the 16 token rows of one head,
// 128-byte swizzled); the block-table indirection is simply the block
// coordinate of the load.  Per block: S^T = K . Q^T with mma.sync
// m16n8k16 (16 tokens x 8 query heads x head_dim), an online softmax over
// tokens with warp shuffles, then O^T += V^T . P^T (P^T formed with
// movmatrix).  fp8 E4M3 tiles are decoded to f16 in registers (exact) and
// multiplied with an f16 copy of q; k_scale is folded into the score scale
// and v_scale into the output.  The warps merge through shared memory; a
// sequence split into several partitions writes (max, sum, output)
// partials that a second kernel merges with a log-sum-exp reduce (one warp
// per output row, launched with programmatic dependent launch so that it is
// resident before the decode kernel ends; one CTA per row when a row may
// hold more than 8 partitions).  Every reduction has a fixed order, so
// results are bitwise deterministic and independent of where blocks sit in
// the pool.
//
// Also here: the decode step in one call (each sequence's new token written
// into the cache by the warp that reads its block, before that block's
// copy; vLLM concept page, "15 分钟专家深入" item 2, and the v0.17.1 notes'
// zeroing of a freshly allocated block), and the host side of shared-prefix
// (cascade) decode: the tensor-core prefix pass (attention_prefill.cu), this
// kernel over each sequence's own tokens launched beside it, and the merge.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <atomic>
#include <cstring>
#include <mutex>

#include "e4m3_encode.cuh"
#include "pkv_device.cuh"
#include "pkv_host.h"
#include "../../include/pagedkv_testing.h"

namespace pkv {

static __device__ ErrorWord g_err_attention = {0ull, 0ull};

struct DecodeParams {
  const __nv_bfloat16 *q;      // [B, Hq, D]
  const int32_t *block_tables;  // [B, max_blocks]
  const int32_t *seq_lens;      // [B]
  __nv_bfloat16 *out;           // [B, Hq, D]
  // split sequences: partials [B, Hq, max_parts, D] and [B, Hq, max_parts]
  // (max in log2 units, sum)
  float *part_o;
  float2 *part_ml;
  int32_t batch, num_heads, num_kv_heads, group, q_groups;
  int32_t num_blocks, max_blocks, max_seq_len, max_parts, part_tokens;
  float scale_log2;  // scale * log2(e) (* k_scale for fp8)
  float v_scale;     // 1 for bf16
  unsigned long long timeout_ns;
  int32_t grid_parts;  // partitions per (kv head group, sequence)
  // 0: the CTA's warps share one partition (blocks dealt round-robin) and
  // merge through shared memory.  1: each warp owns one partition (warp w
  // of grid row y takes partition 4y + w, its blocks in order) and writes
  // its own partial, with no cross-warp step: short partitions then cost
  // no CTA-wide merge and a CTA still streams four partitions' worth.
  int32_t warp_parts;
  // Test hook (-1 = off): every warp working on this sequence stops after
  // its first block as if the wait for the next one had timed out.  No wait
  // is shortened; the copies already issued are drained as on a real
  // timeout.  Set only through pkv_testing_fail_decode_sequence().
  int32_t test_fail_seq;
  // Shared-prefix (cascade) decode, when group_start != nullptr: group G is
  // sequences group_start[G] .. group_start[G+1] - 1 sharing the first
  // prefix_len[G] tokens.  A member that passes the checks of
  // cascade_start() starts at token prefix_len[G]: its prefix was reduced
  // into merge slots 0 .. ceil(prefix_len / prefix_part_tokens) - 1 by the
  // tensor-core pass, and its own partitions follow.  The decode kernel
  // records each sequence's start in seq_start[b] for the merge kernel.
  const int32_t *group_start, *prefix_len;
  int32_t num_groups, max_group_size, max_prefix_len, prefix_part_tokens;
  int32_t *seq_start;
  // 1: the launch just before this one in the stream is the shared-prefix
  // pass, whose CTAs all waited for the kernels before it before letting
  // this grid launch.  This grid then skips its own wait at entry (which
  // would wait for the whole prefix pass) and runs beside the prefix pass;
  // its last CTA waits for the prefix pass before it exits, so that the
  // grid does not complete, and the merge after it does not start, before
  // the prefix partials are written.
  int32_t defer_dep_wait;
  // Decode step (k_new != nullptr): sequence b's new tokens, the last n_b
  // of its seq_lens[b] positions, are written into the cache before they
  // are attended: k_new / v_new [num_new, Hkv, D] bf16 rows
  // new_start_loc[b] .. new_start_loc[b+1] - 1 (without new_start_loc, one
  // token per sequence, row b), the cache bases and k_scale for the E4M3
  // encode (v_scale above).  A block whose first position is a new token
  // was allocated for this step: its rows past the sequence are zeroed.
  // Each warp writes its kv head's rows of the blocks it reads.
  const __nv_bfloat16 *k_new, *v_new;
  const int32_t *new_start_loc;
  long long num_new;
  uint8_t *k_cache, *v_cache;
  float k_scale;
};

// First token of sequence b this launch attends to (0, or its group's
// prefix length when the group and the member pass every check); the same
// value in every lane of the calling warp.  Checks: the group lies inside
// the batch and within the host bounds that sized the prefix pass, the
// prefix is a positive multiple of 16 no longer than the sequence, and the
// member's first prefix_len / 16 block ids equal the first member's and lie
// in the pool.  A failed check is recorded (when `report`) and the member
// is attended in full, which is still the right result.
__device__ int cascade_start(const DecodeParams &p, int b, int L, int lane, bool report) {
  if (!p.group_start || p.num_groups <= 0) return 0;
  // Two dependent memory round trips.  First, what does not depend on the
  // group: this sequence's first table entries and the group starts, 32 a
  // time; starts ascend, so a ballot finds the last one at or before b.
  constexpr int PRE = 2;  // table entries per lane loaded ahead (prefixes <= 1024 tokens)
  const int nchk = min(p.max_prefix_len >> 4, p.max_blocks);  // entries a prefix can cover
  const int32_t *mine = p.block_tables + (size_t)b * p.max_blocks;
  int32_t mine_pre[PRE], lead_pre[PRE];
#pragma unroll
  for (int k = 0; k < PRE; ++k) mine_pre[k] = lane + 32 * k < nchk ? __ldg(mine + lane + 32 * k) : 0;
  int G = -1, q0 = 0;
  for (int base = 0; base < p.num_groups; base += 32) {
    const int gi = base + lane;
    const int st = gi < p.num_groups ? __ldg(p.group_start + gi) : INT_MAX;
    const unsigned m = __ballot_sync(0xffffffffu, st <= b);
    if (m) {
      const int last = 31 - __clz(m);
      G = base + last;
      q0 = __shfl_sync(0xffffffffu, st, last);
    }
    if (m != 0xffffffffu) break;
  }
  if (G < 0) return 0;
  // Second: the group's end and prefix length, and the first member's
  // table entries.
  const int q1 = __ldg(p.group_start + G + 1), P = __ldg(p.prefix_len + G);
  const int32_t *lead = p.block_tables + (size_t)max(q0, 0) * p.max_blocks;
  const bool lead_ok = q0 >= 0 && q0 < p.batch;
#pragma unroll
  for (int k = 0; k < PRE; ++k)
    lead_pre[k] = lead_ok && lane + 32 * k < nchk ? __ldg(lead + lane + 32 * k) : 0;
  const int n = q1 - q0;
  if (b >= q0 + n || P == 0) return 0;  // in no group / nothing shared
  if (n < 1 || q0 < 0 || q0 + n > p.batch || P < 0 || (P & 15) || P > p.max_blocks * 16 ||
      P > p.max_prefix_len || n > p.max_group_size || L < P) {
    if (report && lane == 0) record_error(&g_err_attention, PKV_ERR_RANGE, b);
    return 0;
  }
  int bad_j = INT_MAX;
#pragma unroll
  for (int k = 0; k < PRE; ++k) {
    const int j = lane + 32 * k;
    const int32_t id = mine_pre[k];
    if (j < (P >> 4) && (id != lead_pre[k] || id < 0 || id >= p.num_blocks)) bad_j = min(bad_j, j);
  }
  for (int j = lane + 32 * PRE; j < (P >> 4); j += 32) {
    const int32_t id = __ldg(mine + j);
    if (id != __ldg(lead + j) || id < 0 || id >= p.num_blocks) bad_j = min(bad_j, j);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) bad_j = min(bad_j, __shfl_xor_sync(0xffffffffu, bad_j, off));
  if (bad_j != INT_MAX) {
    if (report && lane == 0)
      record_error(&g_err_attention, PKV_ERR_RANGE, (long long)b * p.max_blocks + bad_j);
    return 0;
  }
  return P;
}

__device__ __forceinline__ int prefix_slots(const DecodeParams &p, int start) {
  return start > 0 ? (start + p.prefix_part_tokens - 1) / p.prefix_part_tokens : 0;
}

// NW warps per CTA share RING_KB KiB of stages (3 CTAs/SM at 4 warps, 64).
template <bool FP8, int D, int NW_ = 4, int RING_KB = 64>
struct Cfg {
  static constexpr int ELT = FP8 ? 1 : 2;
  static constexpr int ROW_BYTES = D * ELT;
  static constexpr int BOX_BYTES = ROW_BYTES >= 128 ? 128 : ROW_BYTES;
  static constexpr int NBOX = ROW_BYTES / BOX_BYTES;
  static constexpr int BOX_ELEMS = BOX_BYTES / ELT;
  static constexpr int TILE_BYTES = 16 * ROW_BYTES;    // K (or V) of a block-head
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;   // K + V
  static constexpr int NW = NW_;                       // warps per CTA
  static constexpr int RING_BYTES = RING_KB * 1024;    // all stages of a CTA
  static constexpr int S0 = RING_BYTES / (NW * STAGE_BYTES);
  static constexpr int STAGES = S0 < 2 ? 2 : (S0 > 8 ? 8 : S0);
  static constexpr int MT = D / 16;                    // 16-row tiles of head_dim
  static constexpr int OS_STRIDE = D + 4;              // padded row of o_s
  static constexpr int SMEM_BYTES = NW * STAGES * STAGE_BYTES + 1024;
  static_assert(8 * OS_STRIDE * 4 + 8 * 8 <= STAGES * STAGE_BYTES,
                "combine scratch (outputs, then max/sum pairs) must fit in a warp's ring");
};

__device__ __forceinline__ int clamp_len(int L, int cap) {
  return L < 0 ? 0 : (L > cap ? cap : L);
}

// Row of head_dim held by output fragment element (m-tile mt, upper half
// `hi` of the 16 rows) for lane group g = lane / 4.
template <bool FP8>
__device__ __forceinline__ int o_row(int mt, int hi, int g) {
  return FP8 ? 16 * mt + 2 * g + hi : 16 * mt + 8 * hi + g;
}

template <bool FP8>
__device__ __forceinline__ void mma_kv(float (&d)[4], uint32_t a0, uint32_t a1,
                                       uint32_t a2, uint32_t a3, uint32_t b0,
                                       uint32_t b1) {
  if (FP8)
    mma_f16(d, a0, a1, a2, a3, b0, b1);
  else
    mma_bf16(d, a0, a1, a2, a3, b0, b1);
}

// Online-softmax state of one warp over one piece of an item.  Lane
// (g = lane/4, c = lane%4) holds columns (query heads) 2c and 2c+1: the
// running max and sum (log2 domain) and O^T rows o_row(mt, hi, g).
template <bool FP8, int D>
struct WarpState {
  float o[Cfg<FP8, D>::MT][4];
  float m0, m1, l0, l1;
  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int mt = 0; mt < Cfg<FP8, D>::MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
  }
  // Sum of l over the lanes that share a column.
  __device__ __forceinline__ void reduce_l() {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
  }
};

// B-operand fragments of S^T = K . Q^T for query heads qh0 .. qh0+7 (heads
// at or past `valid` are zero).  fp8 tiles hand each lane 4 consecutive
// head_dim values per row, so the k order of the mma is permuted to match
// (a dot product does not depend on it) and q is loaded in that order.
template <bool FP8, int D>
__device__ __forceinline__ void load_q(uint32_t (&qf)[Cfg<FP8, D>::MT][2],
                                       const __nv_bfloat16 *q_item, int valid, int lane) {
  const int g = lane >> 2, c = lane & 3;
  const __nv_bfloat16 *qrow = q_item + (size_t)g * D;
#pragma unroll
  for (int ks = 0; ks < Cfg<FP8, D>::MT; ++ks) {
    if (g >= valid) {
      qf[ks][0] = qf[ks][1] = 0u;
      continue;
    }
    if (!FP8) {
      qf[ks][0] = __ldg(reinterpret_cast<const unsigned int *>(qrow + 16 * ks + 2 * c));
      qf[ks][1] = __ldg(reinterpret_cast<const unsigned int *>(qrow + 16 * ks + 8 + 2 * c));
    } else {
      const uint2 four = __ldg(reinterpret_cast<const uint2 *>(qrow + 16 * ks + 4 * c));
      const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&four.x));
      const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&four.y));
      qf[ks][0] = pack_f16x2(f0.x, f0.y);
      qf[ks][1] = pack_f16x2(f1.x, f1.y);
    }
  }
}

// S^T[16 tokens x 8 heads] = K . Q^T for one 16-token block; sk is the
// shared address of the K tile.  sc[0], sc[1]: token g, heads 2c, 2c+1;
// sc[2], sc[3]: token g + 8.
template <bool FP8, int D>
__device__ __forceinline__ void block_scores(uint32_t sk,
                                             const uint32_t (&qf)[Cfg<FP8, D>::MT][2],
                                             float (&sc)[4], int lane,
                                             uint32_t box_stride = 16 * Cfg<FP8, D>::BOX_BYTES) {
  using C = Cfg<FP8, D>;
  // ldmatrix source rows/chunks for this lane (fragment layouts of
  // mma.m16n8k16): K uses (row = lane%8 + 8*bit3, chunk = 2x + bit4).
  const int k_row = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int k_chk = lane >> 4;
  // Two accumulators over alternating k-steps halve the dependent mma chain.
  float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
  if (!FP8) {
#pragma unroll
    for (int ks = 0; ks < C::MT; ++ks) {
      uint32_t a0, a1, a2, a3;
      ldmatrix_x4(sk + tile_offset<C::BOX_BYTES>(k_row, 2 * ks + k_chk, box_stride), a0, a1, a2,
                  a3);
      mma_kv<FP8>((ks & 1) ? sb : sa, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
    }
  } else {
#pragma unroll
    for (int kp = 0; kp < C::MT / 2; ++kp) {
      uint32_t r0, r1, r2, r3;
      ldmatrix_x4(sk + tile_offset<C::BOX_BYTES>(k_row, 2 * kp + k_chk, box_stride), r0, r1, r2,
                  r3);
      uint32_t a0l, a0h, a1l, a1h, a2l, a2h, a3l, a3h;
      e4m3x4_to_f16x2x2(r0, a0l, a0h);
      e4m3x4_to_f16x2x2(r1, a1l, a1h);
      e4m3x4_to_f16x2x2(r2, a2l, a2h);
      e4m3x4_to_f16x2x2(r3, a3l, a3h);
      mma_kv<FP8>(sa, a0l, a1l, a0h, a1h, qf[2 * kp][0], qf[2 * kp][1]);
      mma_kv<FP8>(sb, a2l, a3l, a2h, a3h, qf[2 * kp + 1][0], qf[2 * kp + 1][1]);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) sc[i] = sa[i] + sb[i];
}

// Online softmax update with one block's scores and P.V accumulation; sv is
// the shared address of the V tile, nv the block's valid tokens (0..16).
template <bool FP8, int D, bool FULL>
__device__ __forceinline__ void block_update(uint32_t sv, int nv, const float (&sc)[4],
                                             float scale_log2, WarpState<FP8, D> &st, int lane,
                                             uint32_t box_stride = 16 * Cfg<FP8, D>::BOX_BYTES) {
  using C = Cfg<FP8, D>;
  const int g = lane >> 2, c = lane & 3;
  // V^T uses (row = lane%8 + 8*bit4, chunk = 2x + bit3) for bf16 and the K
  // pattern for fp8.
  const int v_row = FP8 ? (lane & 7) + ((lane >> 3) & 1) * 8 : (lane & 7) + (lane >> 4) * 8;
  const int v_chk = FP8 ? lane >> 4 : (lane >> 3) & 1;

  // -- online softmax per query-head column -------------------------------
  // sc[0], sc[1]: token g, heads 2c, 2c+1; sc[2], sc[3]: token g + 8.
  const bool v_lo = FULL || g < nv, v_hi = FULL || g + 8 < nv;
  const float s0 = v_lo ? sc[0] * scale_log2 : -INFINITY;
  const float s1 = v_lo ? sc[1] * scale_log2 : -INFINITY;
  const float s2 = v_hi ? sc[2] * scale_log2 : -INFINITY;
  const float s3 = v_hi ? sc[3] * scale_log2 : -INFINITY;
  float bm0 = fmaxf(s0, s2), bm1 = fmaxf(s1, s3);
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
    bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
  }
  const float mn0 = fmaxf(st.m0, bm0), mn1 = fmaxf(st.m1, bm1);
  const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
  const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
  const float al0 = exp2f(st.m0 - mu0), al1 = exp2f(st.m1 - mu1);
  const float p0 = exp2f(s0 - mu0), p2 = exp2f(s2 - mu0);
  const float p1 = exp2f(s1 - mu1), p3 = exp2f(s3 - mu1);
  st.l0 = st.l0 * al0 + (p0 + p2);
  st.l1 = st.l1 * al1 + (p1 + p3);
  st.m0 = mn0;
  st.m1 = mn1;
  // Once the running maxima settle, alpha is 1 for every column: skip the
  // rescale then (the result is the same, multiplying by 1 is exact).
  if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt) {
      st.o[mt][0] *= al0;
      st.o[mt][1] *= al1;
      st.o[mt][2] *= al0;
      st.o[mt][3] *= al1;
    }
  }

  // -- P^T fragment (B operand of O^T += V^T . P^T) -----------------------
  const uint32_t pb0 = movmatrix_trans(FP8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1));
  const uint32_t pb1 = movmatrix_trans(FP8 ? pack_f16x2(p2, p3) : pack_bf16x2(p2, p3));

  // V rows past the sequence may hold stale NaN/Inf bits: zero them in the
  // A fragment (tokens 2c, 2c+1 in regs 0/1, 8+2c, 9+2c in regs 2/3), so
  // that p = 0 never meets a NaN inside the mma.
  uint32_t vm_lo = 0xffffffffu, vm_hi = 0xffffffffu;
  if (!FULL) {
    vm_lo = (2 * c < nv ? 0x0000ffffu : 0u) | (2 * c + 1 < nv ? 0xffff0000u : 0u);
    vm_hi = (2 * c + 8 < nv ? 0x0000ffffu : 0u) | (2 * c + 9 < nv ? 0xffff0000u : 0u);
  }
  auto mask = [&](uint32_t x, uint32_t m) { return FULL ? x : (x & m); };

  // -- O^T[head_dim x 8] += V^T . P^T -------------------------------------
  if (!FP8) {
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt) {
      uint32_t a0, a1, a2, a3;
      ldmatrix_x4_trans(sv + tile_offset<C::BOX_BYTES>(v_row, 2 * mt + v_chk, box_stride), a0,
                        a1, a2, a3);
      mma_kv<FP8>(st.o[mt], mask(a0, vm_lo), mask(a1, vm_lo), mask(a2, vm_hi), mask(a3, vm_hi),
                  pb0, pb1);
    }
  } else {
#pragma unroll
    for (int qq = 0; qq < C::MT / 2; ++qq) {
      uint32_t r0, r1, r2, r3;
      ldmatrix_x4_trans(sv + tile_offset<C::BOX_BYTES>(v_row, 2 * qq + v_chk, box_stride), r0,
                        r1, r2, r3);
      // r0/r2: tokens 2c, 2c+1 (rows 0-7); r1/r3: tokens 8+2c, 9+2c.  Each
      // holds [t0 dA, t0 dB, t1 dA, t1 dB]; regroup per head_dim row.
      const uint32_t x0 = prmt(r0, 0u, 0x3120u), x1 = prmt(r1, 0u, 0x3120u);
      const uint32_t x2 = prmt(r2, 0u, 0x3120u), x3 = prmt(r3, 0u, 0x3120u);
      uint32_t c0l, c0h, c1l, c1h, c2l, c2h, c3l, c3h;
      e4m3x4_to_f16x2x2(x0, c0l, c0h);
      e4m3x4_to_f16x2x2(x1, c1l, c1h);
      e4m3x4_to_f16x2x2(x2, c2l, c2h);
      e4m3x4_to_f16x2x2(x3, c3l, c3h);
      mma_kv<FP8>(st.o[2 * qq], mask(c0l, vm_lo), mask(c0h, vm_lo), mask(c1l, vm_hi),
                  mask(c1h, vm_hi), pb0, pb1);
      mma_kv<FP8>(st.o[2 * qq + 1], mask(c2l, vm_lo), mask(c2h, vm_lo), mask(c3l, vm_hi),
                  mask(c3h, vm_hi), pb0, pb1);
    }
  }
}

// One 16-token block: scores, online softmax update and P.V accumulation.
template <bool FP8, int D>
__device__ __forceinline__ void attend_block(uint32_t sk, uint32_t sv, int nv,
                                             const uint32_t (&qf)[Cfg<FP8, D>::MT][2],
                                             float scale_log2, WarpState<FP8, D> &st,
                                             int lane) {
  float sc[4];
  block_scores<FP8, D>(sk, qf, sc, lane);
  if (nv == 16)
    block_update<FP8, D, true>(sv, nv, sc, scale_log2, st, lane);
  else
    block_update<FP8, D, false>(sv, nv, sc, scale_log2, st, lane);
}

// fp8 caches: two 16-token blocks per online-softmax step.  Their scores
// come from independent mma chains, one shuffle reduction and one rescale
// serve both, and both P.V products accumulate into O.  The result is the
// same softmax, with the running maximum advanced once per pair.
template <int D, bool FULL>
__device__ __forceinline__ void pair_update(uint32_t sva, int nva, const float (&sa)[4],
                                            uint32_t svb, int nvb, const float (&sb)[4],
                                            float scale_log2, WarpState<true, D> &st, int lane) {
  using C = Cfg<true, D>;
  const int g = lane >> 2, c = lane & 3;
  const int v_row = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int v_chk = lane >> 4;
  const bool a_lo = FULL || g < nva, a_hi = FULL || g + 8 < nva;
  const bool b_lo = FULL || g < nvb, b_hi = FULL || g + 8 < nvb;
  const float s0 = a_lo ? sa[0] * scale_log2 : -INFINITY;
  const float s1 = a_lo ? sa[1] * scale_log2 : -INFINITY;
  const float s2 = a_hi ? sa[2] * scale_log2 : -INFINITY;
  const float s3 = a_hi ? sa[3] * scale_log2 : -INFINITY;
  const float t0 = b_lo ? sb[0] * scale_log2 : -INFINITY;
  const float t1 = b_lo ? sb[1] * scale_log2 : -INFINITY;
  const float t2 = b_hi ? sb[2] * scale_log2 : -INFINITY;
  const float t3 = b_hi ? sb[3] * scale_log2 : -INFINITY;
  float bm0 = fmaxf(fmaxf(s0, s2), fmaxf(t0, t2)), bm1 = fmaxf(fmaxf(s1, s3), fmaxf(t1, t3));
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
    bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
  }
  const float mn0 = fmaxf(st.m0, bm0), mn1 = fmaxf(st.m1, bm1);
  const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
  const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
  const float al0 = exp2f(st.m0 - mu0), al1 = exp2f(st.m1 - mu1);
  const float p0 = exp2f(s0 - mu0), p2 = exp2f(s2 - mu0);
  const float p1 = exp2f(s1 - mu1), p3 = exp2f(s3 - mu1);
  const float q0 = exp2f(t0 - mu0), q2 = exp2f(t2 - mu0);
  const float q1 = exp2f(t1 - mu1), q3 = exp2f(t3 - mu1);
  st.l0 = st.l0 * al0 + ((p0 + p2) + (q0 + q2));
  st.l1 = st.l1 * al1 + ((p1 + p3) + (q1 + q3));
  st.m0 = mn0;
  st.m1 = mn1;
  if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt) {
      st.o[mt][0] *= al0;
      st.o[mt][1] *= al1;
      st.o[mt][2] *= al0;
      st.o[mt][3] *= al1;
    }
  }
  const uint32_t pa0 = movmatrix_trans(pack_f16x2(p0, p1));
  const uint32_t pa1 = movmatrix_trans(pack_f16x2(p2, p3));
  const uint32_t pb0 = movmatrix_trans(pack_f16x2(q0, q1));
  const uint32_t pb1 = movmatrix_trans(pack_f16x2(q2, q3));
  // stale V rows (past the sequence) are zeroed in the A fragments, as in
  // block_update
  uint32_t ma_lo = 0xffffffffu, ma_hi = 0xffffffffu, mb_lo = 0xffffffffu, mb_hi = 0xffffffffu;
  if (!FULL) {
    ma_lo = (2 * c < nva ? 0x0000ffffu : 0u) | (2 * c + 1 < nva ? 0xffff0000u : 0u);
    ma_hi = (2 * c + 8 < nva ? 0x0000ffffu : 0u) | (2 * c + 9 < nva ? 0xffff0000u : 0u);
    mb_lo = (2 * c < nvb ? 0x0000ffffu : 0u) | (2 * c + 1 < nvb ? 0xffff0000u : 0u);
    mb_hi = (2 * c + 8 < nvb ? 0x0000ffffu : 0u) | (2 * c + 9 < nvb ? 0xffff0000u : 0u);
  }
  auto mask = [&](uint32_t x, uint32_t m) { return FULL ? x : (x & m); };
#pragma unroll
  for (int qq = 0; qq < C::MT / 2; ++qq) {
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      const uint32_t sv = blk ? svb : sva;
      const uint32_t m_lo = blk ? mb_lo : ma_lo, m_hi = blk ? mb_hi : ma_hi;
      const uint32_t f0 = blk ? pb0 : pa0, f1 = blk ? pb1 : pa1;
      uint32_t r0, r1, r2, r3;
      ldmatrix_x4_trans(sv + tile_offset<C::BOX_BYTES>(v_row, 2 * qq + v_chk), r0, r1, r2, r3);
      const uint32_t x0 = prmt(r0, 0u, 0x3120u), x1 = prmt(r1, 0u, 0x3120u);
      const uint32_t x2 = prmt(r2, 0u, 0x3120u), x3 = prmt(r3, 0u, 0x3120u);
      uint32_t c0l, c0h, c1l, c1h, c2l, c2h, c3l, c3h;
      e4m3x4_to_f16x2x2(x0, c0l, c0h);
      e4m3x4_to_f16x2x2(x1, c1l, c1h);
      e4m3x4_to_f16x2x2(x2, c2l, c2h);
      e4m3x4_to_f16x2x2(x3, c3l, c3h);
      mma_kv<true>(st.o[2 * qq], mask(c0l, m_lo), mask(c0h, m_lo), mask(c1l, m_hi),
                   mask(c1h, m_hi), f0, f1);
      mma_kv<true>(st.o[2 * qq + 1], mask(c2l, m_lo), mask(c2h, m_lo), mask(c3l, m_hi),
                   mask(c3h, m_hi), f0, f1);
    }
  }
}

template <int D>
__device__ __forceinline__ void attend_pair(uint32_t ska, int nva, uint32_t skb, int nvb,
                                            const uint32_t (&qf)[Cfg<true, D>::MT][2],
                                            float scale_log2, WarpState<true, D> &st,
                                            int lane) {
  using C = Cfg<true, D>;
  float sa[4], sb[4];
  block_scores<true, D>(ska, qf, sa, lane);
  block_scores<true, D>(skb, qf, sb, lane);
  if (nva == 16 && nvb == 16)
    pair_update<D, true>(ska + C::TILE_BYTES, nva, sa, skb + C::TILE_BYTES, nvb, sb, scale_log2,
                         st, lane);
  else
    pair_update<D, false>(ska + C::TILE_BYTES, nva, sa, skb + C::TILE_BYTES, nvb, sb,
                          scale_log2, st, lane);
}

// Lane 0 issues the TMA loads of one block-head (K and V tiles) into a
// stage: one box per tile, [head_dim slice][token][BOX_BYTES].
template <bool FP8, int D>
__device__ __forceinline__ void issue_block(uint8_t *stage, uint64_t *bar,
                                            const CUtensorMap *tk, const CUtensorMap *tv,
                                            int kvh, int phys, uint64_t policy) {
  using C = Cfg<FP8, D>;
  mbar_arrive_expect_tx(bar, C::STAGE_BYTES);
  tma_load_5d(stage, tk, bar, 0, 0, kvh, 0, phys, policy);
  tma_load_5d(stage + C::TILE_BYTES, tv, bar, 0, 0, kvh, 0, phys, policy);
}

// Generic-proxy global stores of this thread ordered before the async
// proxy's (TMA) later accesses to them: each writing lane runs this, then the
// warp synchronises, then lane 0 issues the copy.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Decode step, one new token: the warp writes the token's K and V rows of
// kv head kvh (token row src) to row `off` of block `blk`, and when the
// token opens the block (off == 0) zeroes the block's other 15 rows of the
// head.  The caller fences (fence_proxy_async_global) before the warp's TMA
// copy of the block.
template <bool FP8, int D>
__device__ __forceinline__ void write_one_token(const DecodeParams &p, int blk, int off, int kvh,
                                                long long src, int lane) {
  constexpr int ELT = FP8 ? 1 : 2;
  constexpr int CH = D * ELT / 16;  // 16-byte chunks of one head's row
  const size_t row_bytes = (size_t)p.num_kv_heads * D * ELT;
  const size_t head0 = (size_t)blk * 16 * row_bytes + (size_t)kvh * D * ELT;
  uint8_t *kc = p.k_cache + head0, *vc = p.v_cache + head0;
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  const bool is_v = lane >= D / 8;
  const int vec = is_v ? lane - D / 8 : lane;  // 8 elements
  if (lane < 2 * (D / 8))
    v = __ldg(reinterpret_cast<const uint4 *>((is_v ? p.v_new : p.k_new) +
                                              ((size_t)src * p.num_kv_heads + kvh) * D) +
              vec);
  if (off == 0) {
    for (int idx = lane; idx < 2 * 15 * CH; idx += 32) {
      const int rem = idx % (15 * CH);
      uint8_t *base = idx < 15 * CH ? kc : vc;
      *reinterpret_cast<uint4 *>(base + (size_t)(1 + rem / CH) * row_bytes + (rem % CH) * 16) =
          make_uint4(0u, 0u, 0u, 0u);
    }
  }
  if (lane < 2 * (D / 8)) {
    uint8_t *dst = (is_v ? vc : kc) + (size_t)off * row_bytes;
    if constexpr (FP8) {
      const float scale = is_v ? p.v_scale : p.k_scale;
      *reinterpret_cast<uint2 *>(dst + vec * 8) = quant8_e4m3(v, scale, e4m3_recip(scale));
    } else {
      *reinterpret_cast<uint4 *>(dst + vec * 16) = v;
    }
  }
}

// Decode step: the warp's part of sequence b's new tokens in block j
// (physical id blk) of kv head kvh: the rows of new positions (w0 .. L - 1)
// get the tokens' K and V (position t from token row src0 + t - w0), and a
// block that opens at or after w0 has its rows past L zeroed; rows before
// w0 are left alone.  Loads go out eight 16-byte vectors a lane at a time
// before their stores.  The caller fences (fence_proxy_async_global) before
// the warp's TMA copy of the block.
template <bool FP8, int D>
__device__ __forceinline__ void write_new_rows(const DecodeParams &p, int blk, int j, int w0,
                                               int L, long long src0, int kvh, int lane) {
  constexpr int ELT = FP8 ? 1 : 2;
  constexpr int VPR = D / 8;  // 8-element vectors of one head's row
  constexpr int ITEMS_PER_ROW = 2 * VPR;  // K and V
  constexpr int BATCH = 8;
  const size_t row_bytes = (size_t)p.num_kv_heads * D * ELT;
  uint8_t *kc = p.k_cache + (size_t)blk * 16 * row_bytes + (size_t)kvh * D * ELT;
  uint8_t *vc = p.v_cache + (size_t)blk * 16 * row_bytes + (size_t)kvh * D * ELT;
  const int t0 = 16 * j;
  const int r_lo = max(0, w0 - t0);        // first row written
  const int r_hi = min(16, L - t0);        // one past the last row written
  const int r_end = t0 >= w0 ? 16 : r_hi;  // and then the zeroed rows
  const int items = (r_end - r_lo) * ITEMS_PER_ROW;
  const E4m3Recip kr = e4m3_recip(p.k_scale), vr = e4m3_recip(p.v_scale);
  for (int base = 0; base < items; base += 32 * BATCH) {
    uint4 src[BATCH];
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int idx = base + u * 32 + lane;
      const int r = r_lo + idx / ITEMS_PER_ROW, rem = idx % ITEMS_PER_ROW;
      const bool is_v = rem >= VPR;
      src[u] = make_uint4(0u, 0u, 0u, 0u);
      if (idx < items && r < r_hi) {
        const long long tok = src0 + (t0 + r - w0);
        src[u] = __ldg(reinterpret_cast<const uint4 *>((is_v ? p.v_new : p.k_new) +
                                                       ((size_t)tok * p.num_kv_heads + kvh) * D) +
                       (is_v ? rem - VPR : rem));
      }
    }
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int idx = base + u * 32 + lane;
      if (idx >= items) break;
      const int r = r_lo + idx / ITEMS_PER_ROW, rem = idx % ITEMS_PER_ROW;
      const bool is_v = rem >= VPR;
      uint8_t *dst = (is_v ? vc : kc) + (size_t)r * row_bytes + (is_v ? rem - VPR : rem) * 8 * ELT;
      if constexpr (FP8) {
        *reinterpret_cast<uint2 *>(dst) =
            r < r_hi ? quant8_e4m3(src[u], is_v ? p.v_scale : p.k_scale, is_v ? vr : kr)
                     : make_uint2(0u, 0u);
      } else {
        *reinterpret_cast<uint4 *>(dst) = src[u];  // zero past r_hi
      }
    }
  }
}

// ===========================================================================
// Decode kernel
// ===========================================================================
template <bool FP8, int D, int NW = 4, int RING_KB = 64>
__global__ void __launch_bounds__(NW * 32)
paged_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v,
                    const DecodeParams p) {
  using C = Cfg<FP8, D, NW, RING_KB>;
  extern __shared__ uint8_t smem_dyn[];
  __shared__ uint64_t bars[C::NW][C::STAGES];
  __shared__ int stage_ok[C::NW][C::STAGES];
  __shared__ float m_s[C::NW][8];
  __shared__ float l_s[C::NW][8];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int c = lane & 3;
  const int kvh = blockIdx.x / p.q_groups;
  const int qg = blockIdx.x - kvh * p.q_groups;
  const bool wmode = p.warp_parts != 0;  // uniform over the grid
  // grid (kv head group, partition, sequence); with warp-owned partitions
  // (kv head group, sequence, row of 4 partitions), so that every
  // sequence's first rows launch before any sequence's last
  const int prow = wmode ? blockIdx.z : blockIdx.y;
  const int part = wmode ? prow * C::NW + warp : prow;
  const int b = wmode ? blockIdx.y : blockIdx.z;
  // this warp's blocks of the partition: j0 + i * jstep
  const int j_off = wmode ? 0 : warp, jstep = wmode ? 1 : C::NW;

  const uint32_t base_u32 = smem_u32(smem_dyn);
  uint8_t *rings = smem_dyn + (((base_u32 + 1023u) & ~1023u) - base_u32);
  uint8_t *ring = rings + warp * C::STAGES * C::STAGE_BYTES;
  if (lane == 0) {
    for (int s = 0; s < C::STAGES; ++s) mbar_init(&bars[warp][s], 1);
    fence_barrier_init();
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }
  __syncwarp();
  const bool wait_at_exit = p.defer_dep_wait && blockIdx.x == gridDim.x - 1 &&
                            blockIdx.y == gridDim.y - 1 && blockIdx.z == gridDim.z - 1;
  if (!p.defer_dep_wait) grid_dependency_wait();
  allow_dependent_launch();

  // q does not depend on the sequence's extent: its loads go out first
  const int heads_here = min(8, p.group - qg * 8);
  const size_t row0 = (size_t)b * p.num_heads + (size_t)kvh * p.group + qg * 8;
  uint32_t qf[C::MT][2];
  load_q<FP8, D>(qf, p.q + row0 * D, heads_here, lane);
  // The partition's first block is (start + part * part_tokens) / 16 whatever
  // the length, where start is 0 without shared prefixes: this warp's first
  // 32 block ids go out now too (masked to the partition's blocks once the
  // length is known).  With shared prefixes the start is guessed to be the
  // longest prefix (every member of a group that shares it) and the ids are
  // used only if the guess proves right.
  const int spec_start = p.group_start ? p.max_prefix_len : 0;
  int ids_pre = -1;
  {
    const long long j = (long long)(spec_start >> 4) + (long long)part * (p.part_tokens >> 4) +
                        j_off + (long long)lane * jstep;
    if (j < p.max_blocks) ids_pre = __ldg(p.block_tables + (size_t)b * p.max_blocks + j);
  }

  // ---- sequence extent and this CTA's partition --------------------------
  int L = __ldg(p.seq_lens + b);
  int nsl0 = 0, nsl1 = 0;  // decode step: the sequence's new-token rows
  if (p.k_new != nullptr && p.new_start_loc) {
    nsl0 = __ldg(p.new_start_loc + b);
    nsl1 = __ldg(p.new_start_loc + b + 1);
  }
  bool len_ok = true;  // (a clamped length writes no new token)
  {
    const int cap = min(p.max_blocks * 16, p.max_seq_len);
    if (L < 0 || L > cap) {
      if (part == 0 && blockIdx.x == 0 && threadIdx.x == 0)
        record_error(&g_err_attention, PKV_ERR_RANGE, b);
      L = clamp_len(L, cap);
      len_ok = false;
    }
  }
  const int start =
      cascade_start(p, b, L, lane, blockIdx.x == 0 && part == 0 && warp == 0);
  const int slot_base = prefix_slots(p, start);
  const bool ids_early = start == spec_start;
  if (p.seq_start && blockIdx.x == 0 && part == 0 && threadIdx.x == 0) p.seq_start[b] = start;
  const int Ls = L - start;
  const int nparts = Ls <= p.part_tokens ? 1 : (Ls + p.part_tokens - 1) / p.part_tokens;
  if (part >= nparts) {  // the whole CTA, or (warp-owned) this warp
    if (wait_at_exit) grid_dependency_wait();
    return;
  }
  const int tok0 = start + part * p.part_tokens;  // multiple of 16
  const int tok1 = min(L, tok0 + p.part_tokens);
  const int blk0 = tok0 >> 4;
  const int nblk = (tok1 - tok0 + 15) >> 4;
  const int my_n = wmode ? nblk : (nblk > warp ? (nblk - warp + C::NW - 1) / C::NW : 0);

  // ---- block ids of this warp, 32 at a time in registers -----------------
  const int32_t *table = p.block_tables + (size_t)b * p.max_blocks + blk0 + j_off;
  int ids_reg = -1;
  const uint64_t policy = l2_policy_evict_normal();
  auto issue = [&](int i) {
    if ((i & 31) == 0)
      ids_reg = (i + lane < my_n) ? (i == 0 && ids_early ? ids_pre : __ldg(table + (i + lane) * jstep))
                                  : -1;
    int phys = __shfl_sync(0xffffffffu, ids_reg, i & 31);
    if (lane == 0) {
      const int stage = i % C::STAGES;
      int ok = 1;
      if (phys < 0 || phys >= p.num_blocks) {
        record_error(&g_err_attention, PKV_ERR_RANGE, b);
        phys = 0;
        ok = 0;
      }
      stage_ok[warp][stage] = ok;
      issue_block<FP8, D>(ring + stage * C::STAGE_BYTES, &bars[warp][stage], &tmap_k, &tmap_v,
                          kvh, phys, policy);
    }
  };

  WarpState<FP8, D> st;
  st.reset();
  int issued = 0;
  const int pre = min(C::STAGES, my_n);
  // Decode step: the warp writes the new tokens of the blocks it reads (the
  // sequence's last blocks, so its last ones) first.  Its copies of earlier
  // blocks go out before the write, the copies of those blocks after.
  if (p.k_new != nullptr && len_ok) {
    // without new_start_loc: one new token per non-empty sequence, row b
    const int n_new = p.new_start_loc ? nsl1 - nsl0 : (L > 0 ? 1 : 0);
    const long long src0 = p.new_start_loc ? nsl0 : b;
    const bool ok_new = n_new >= 0 && n_new <= L && nsl0 >= 0 &&
                        (!p.new_start_loc || (long long)nsl1 <= p.num_new);
    if (!ok_new && part == 0 && blockIdx.x == 0 && threadIdx.x == 0)
      record_error(&g_err_attention, PKV_ERR_RANGE, b);
    const int w0 = L - n_new;  // first new position
    // the warp's first block at or after the one holding w0
    const int jw = (w0 >> 4) - blk0 - j_off;
    const int i_w = jw <= 0 ? 0 : (jw + jstep - 1) / jstep;
    if (ok_new && n_new > 0 && my_n > 0 && i_w < my_n) {
      for (; issued < min(pre, i_w); ++issued) issue(issued);
      const int32_t *trow = p.block_tables + (size_t)b * p.max_blocks;
      if (n_new == 1) {  // the usual decode step: the last block only
        const int wblk = __ldg(trow + (w0 >> 4));
        if (wblk >= 0 && wblk < p.num_blocks)  // (else reported when issued)
          write_one_token<FP8, D>(p, wblk, w0 & 15, kvh, src0, lane);
      } else {
        for (int ii = i_w; ii < my_n; ++ii) {
          const int j = blk0 + j_off + ii * jstep;
          const int wblk = __ldg(trow + j);
          if (wblk >= 0 && wblk < p.num_blocks)  // (else reported when issued)
            write_new_rows<FP8, D>(p, wblk, j, w0, L, src0, kvh, lane);
        }
      }
      fence_proxy_async_global();
      __syncwarp();
    }
  }
  for (; issued < pre; ++issued) issue(issued);

  bool failed = false;
  int i = 0;
  const int stop_at = b == p.test_fail_seq ? min(my_n, 1) : my_n;  // test hook
  if constexpr (FP8 && C::STAGES >= 4) {
    // two blocks per step while two more are in flight
    for (; i + 1 < stop_at; i += 2) {
      const int sa = i % C::STAGES, sb = (i + 1) % C::STAGES;
      if (!mbar_wait_bounded(&bars[warp][sa], (i / C::STAGES) & 1, p.timeout_ns) ||
          !mbar_wait_bounded(&bars[warp][sb], ((i + 1) / C::STAGES) & 1, p.timeout_ns)) {
        failed = true;
        break;
      }
      const int ja = blk0 + j_off + i * jstep, jb = ja + jstep;
      const int nva = stage_ok[warp][sa] ? min(16, tok1 - ja * 16) : 0;
      const int nvb = stage_ok[warp][sb] ? min(16, tok1 - jb * 16) : 0;
      attend_pair<D>(smem_u32(ring + sa * C::STAGE_BYTES), nva,
                     smem_u32(ring + sb * C::STAGE_BYTES), nvb, qf, p.scale_log2, st, lane);
      __syncwarp();
      if (issued < my_n) issue(issued++);
      if (issued < my_n) issue(issued++);
    }
  }
  for (; !failed && i < stop_at; ++i) {
    const int stage = i % C::STAGES;
    if (!mbar_wait_bounded(&bars[warp][stage], (i / C::STAGES) & 1, p.timeout_ns)) {
      failed = true;
      break;
    }
    const int j = blk0 + j_off + i * jstep;
    const int nv = stage_ok[warp][stage] ? min(16, tok1 - j * 16) : 0;
    const uint32_t sk = smem_u32(ring + stage * C::STAGE_BYTES);
    attend_block<FP8, D>(sk, sk + C::TILE_BYTES, nv, qf, p.scale_log2, st, lane);
    __syncwarp();
    if (issued < my_n) issue(issued++);
  }
  if (i < my_n) failed = true;  // only under the test hook, or after a timeout

  if (failed) {
    if (lane == 0) record_error(&g_err_attention, PKV_ERR_TIMEOUT, b);
    // let copies still in flight land before the ring is reused or the CTA
    // exits (bounded as well)
    for (int i = 0; i < issued; ++i)
      mbar_wait_bounded(&bars[warp][i % C::STAGES], (i / C::STAGES) & 1, p.timeout_ns);
    st.m0 = st.m1 = -INFINITY;
  }

  // ---- warp-owned partition: this warp's result, staged through its ring --
  st.reduce_l();
  float *o_s = reinterpret_cast<float *>(ring);  // this warp's ring, now idle
  if (wmode) {
    float2 *ml_w = reinterpret_cast<float2 *>(o_s + 8 * C::OS_STRIDE);
    if (!failed) {
#pragma unroll
      for (int mt = 0; mt < C::MT; ++mt) {
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {
          const int d = o_row<FP8>(mt, hi, g);
          o_s[(2 * c) * C::OS_STRIDE + d] = st.o[mt][2 * hi];
          o_s[(2 * c + 1) * C::OS_STRIDE + d] = st.o[mt][2 * hi + 1];
        }
      }
    }
    if (g == 0) {
      ml_w[2 * c] = make_float2(st.m0, st.l0);
      ml_w[2 * c + 1] = make_float2(st.m1, st.l1);
    }
    __syncwarp();
    const bool direct = nparts == 1 && slot_base == 0;
    for (int idx = lane; idx < heads_here * D; idx += 32) {
      const int h = idx / D;
      const int d = idx - h * D;
      const float2 ml = ml_w[h];
      const bool live = !failed && ml.x != -INFINITY && ml.y > 0.f;
      const float res = live ? o_s[h * C::OS_STRIDE + d] / ml.y * p.v_scale : 0.f;
      const size_t r = row0 + h;
      if (direct) {
        p.out[r * D + d] = __float2bfloat16_rn(res);
      } else {
        const size_t slot = r * p.max_parts + slot_base + part;
        p.part_o[slot * D + d] = res;
        if (d == 0) p.part_ml[slot] = live ? ml : make_float2(-INFINITY, 0.f);
      }
    }
    if (wait_at_exit) grid_dependency_wait();
    return;
  }

  // ---- merge the warps' states -------------------------------------------
  if (!failed && my_n > 0) {
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt) {
#pragma unroll
      for (int hi = 0; hi < 2; ++hi) {
        const int d = o_row<FP8>(mt, hi, g);
        o_s[(2 * c) * C::OS_STRIDE + d] = st.o[mt][2 * hi];
        o_s[(2 * c + 1) * C::OS_STRIDE + d] = st.o[mt][2 * hi + 1];
      }
    }
  }
  if (g == 0) {
    m_s[warp][2 * c] = st.m0;
    m_s[warp][2 * c + 1] = st.m1;
    l_s[warp][2 * c] = st.l0;
    l_s[warp][2 * c + 1] = st.l1;
  }
  __syncthreads();

  for (int idx = threadIdx.x; idx < heads_here * D; idx += blockDim.x) {
    const int h = idx / D;
    const int d = idx - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < C::NW; ++w) M = fmaxf(M, m_s[w][h]);
    float lsum = 0.f, acc = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < C::NW; ++w) {
        const float mw = m_s[w][h];
        if (mw == -INFINITY) continue;
        const float e = exp2f(mw - M);
        lsum += e * l_s[w][h];
        acc += e * reinterpret_cast<const float *>(
                       rings + w * C::STAGES * C::STAGE_BYTES)[h * C::OS_STRIDE + d];
      }
    }
    const float res = lsum > 0.f ? acc / lsum * p.v_scale : 0.f;
    const size_t r = row0 + h;
    if (nparts == 1 && slot_base == 0) {
      p.out[r * D + d] = __float2bfloat16_rn(res);
    } else {
      const size_t slot = r * p.max_parts + slot_base + part;
      p.part_o[slot * D + d] = res;
      if (d == 0) p.part_ml[slot] = make_float2(M, lsum);
    }
  }
  if (wait_at_exit) grid_dependency_wait();
}

// Log-sum-exp merge of split sequences: one warp per (sequence, query head)
// row, lane l owning head_dim elements l, l + 32, ...  Partition j carries
// m_j (log2 domain), l_j and its normalised output o_j; the result is
// sum_j 2^(m_j - M) l_j o_j / sum_j 2^(m_j - M) l_j with M = max_j m_j.  The
// (m, l) pairs of up to 32 partitions are loaded at once (one per lane) and
// reduced with shuffles; outputs accumulate partition by partition, in
// partition order.
template <int D>
__global__ void __launch_bounds__(256) paged_decode_merge_kernel(const DecodeParams p) {
  constexpr int KD = D / 32;
  constexpr int PRE = 4;  // partitions loaded before the row's count is known
  grid_dependency_wait();
  allow_dependent_launch();
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= (long long)p.batch * p.num_heads) return;
  const float2 *ml = p.part_ml + (size_t)row * p.max_parts;
  const float *po = p.part_o + (size_t)row * p.max_parts * D + lane;
  // Every slot below max_parts lies inside this row's workspace, so the
  // first partitions' (m, l) and outputs are loaded alongside the sequence
  // length rather than after it: one memory round trip instead of three.
  // Slots past the row's partition count are never used.
  const float2 v0 = lane < p.max_parts ? ml[lane] : make_float2(-INFINITY, 0.f);
  float pre[PRE][KD];
#pragma unroll
  for (int r = 0; r < PRE; ++r)
#pragma unroll
    for (int k = 0; k < KD; ++k) pre[r][k] = r < p.max_parts ? po[(size_t)r * D + 32 * k] : 0.f;
  const int b = (int)(row / p.num_heads);
  const int cap = min(p.max_blocks * 16, p.max_seq_len);
  const int L = clamp_len(__ldg(p.seq_lens + b), cap);
  int start = p.seq_start ? __ldg(p.seq_start + b) : 0;  // decided by the decode kernel
  if (start < 0 || start > L || (start & 15)) start = 0;
  const int slot_base = prefix_slots(p, start);
  const int Ls = L - start;
  const int nparts =
      slot_base + (Ls <= p.part_tokens ? 1 : (Ls + p.part_tokens - 1) / p.part_tokens);
  if (nparts <= 1) return;  // the decode kernel wrote this row
  float wsum = 0.f, acc[KD];
#pragma unroll
  for (int k = 0; k < KD; ++k) acc[k] = 0.f;
  if (nparts <= 32) {
    // common case: lane j holds partition j's (m, l); shuffles reduce them
    const float2 v = lane < nparts ? v0 : make_float2(-INFINITY, 0.f);
    float M = v.x;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float w = v.x == -INFINITY ? 0.f : exp2f(v.x - M) * v.y;
    float t = w;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
    wsum = t;
#pragma unroll
    for (int r = 0; r < PRE; ++r) {
      const float wr = __shfl_sync(0xffffffffu, w, r);
      if (r < nparts) {
#pragma unroll
        for (int k = 0; k < KD; ++k) acc[k] += wr * pre[r][k];
      }
    }
#pragma unroll 4
    for (int r = PRE; r < nparts; ++r) {
      const float wr = __shfl_sync(0xffffffffu, w, r);
      const float *pj = po + (size_t)r * D;
#pragma unroll
      for (int k = 0; k < KD; ++k) acc[k] += wr * pj[32 * k];
    }
  } else {
    float M = -INFINITY;
    for (int j = lane; j < nparts; j += 32) M = fmaxf(M, ml[j].x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    for (int j0 = 0; j0 < nparts; j0 += 32) {
      float w = 0.f;
      if (j0 + lane < nparts) {
        const float2 v = ml[j0 + lane];
        w = v.x == -INFINITY ? 0.f : exp2f(v.x - M) * v.y;
      }
      float t = w;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
      wsum += t;
      const int cnt = min(32, nparts - j0);
#pragma unroll 4
      for (int r = 0; r < cnt; ++r) {
        const float wr = __shfl_sync(0xffffffffu, w, r);
        const float *pj = po + (size_t)(j0 + r) * D;
#pragma unroll
        for (int k = 0; k < KD; ++k) acc[k] += wr * pj[32 * k];
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  __nv_bfloat16 *orow = p.out + (size_t)row * D + lane;
#pragma unroll
  for (int k = 0; k < KD; ++k) orow[32 * k] = __float2bfloat16_rn(acc[k] * inv);
}

// The same merge for sequences split into many partitions: one CTA of 8
// warps per (sequence, query head) row.  The row's maximum M comes from a
// block-wide reduction over its (m, l) pairs; the weights 2^(m_j - M) l_j go
// to shared memory (kMergeChunk at a time); partition j is accumulated by
// slot j mod 8*PPW (a warp covers PPW partitions per step, each lane four
// consecutive head_dim elements with one 16-byte load), and the slots are
// summed in a fixed order at the end, so the result is deterministic.
constexpr int kMergeWideThreads = 256;
constexpr int kMergeChunk = 2048;

template <int D>
__global__ void __launch_bounds__(kMergeWideThreads)
paged_decode_merge_wide_kernel(const DecodeParams p) {
  constexpr int NWM = kMergeWideThreads / 32;
  constexpr int LPP = D / 4;      // lanes per partition (float4 each)
  constexpr int PPW = 32 / LPP;   // partitions per warp step
  constexpr int SLOTS = NWM * PPW;
  __shared__ float w_s[kMergeChunk];
  __shared__ float red_s[NWM];
  __shared__ float4 acc_s[SLOTS][LPP];
  grid_dependency_wait();
  allow_dependent_launch();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long row = blockIdx.x;
  const int b = (int)(row / p.num_heads);
  const int cap = min(p.max_blocks * 16, p.max_seq_len);
  const int L = clamp_len(__ldg(p.seq_lens + b), cap);
  int start = p.seq_start ? __ldg(p.seq_start + b) : 0;  // decided by the decode kernel
  if (start < 0 || start > L || (start & 15)) start = 0;
  const int slot_base = prefix_slots(p, start);
  const int Ls = L - start;
  const int nparts =
      slot_base + (Ls <= p.part_tokens ? 1 : (Ls + p.part_tokens - 1) / p.part_tokens);
  if (nparts <= 1) return;  // the decode kernel wrote this row (uniform over the CTA)
  const float2 *ml = p.part_ml + (size_t)row * p.max_parts;
  // 1. the row maximum
  float M = -INFINITY;
  for (int j = tid; j < nparts; j += kMergeWideThreads) M = fmaxf(M, ml[j].x);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (lane == 0) red_s[warp] = M;
  __syncthreads();
  M = red_s[0];
#pragma unroll
  for (int w = 1; w < NWM; ++w) M = fmaxf(M, red_s[w]);
  // 2. weights and the weighted sum of outputs, a chunk of partitions at a time
  const int sub = lane / LPP, l4 = lane - sub * LPP;
  const int slot = warp * PPW + sub;
  float wsum = 0.f;  // this thread's weights, in j order
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = 0; c0 < nparts; c0 += kMergeChunk) {
    const int cnt = min(kMergeChunk, nparts - c0);
    __syncthreads();  // the previous chunk's weights are consumed (and red_s read)
    for (int j = tid; j < cnt; j += kMergeWideThreads) {
      const float2 v = ml[c0 + j];
      const float w = v.x == -INFINITY ? 0.f : exp2f(v.x - M) * v.y;
      w_s[j] = w;
      wsum += w;
    }
    __syncthreads();
    const float4 *po =
        reinterpret_cast<const float4 *>(p.part_o + ((size_t)row * p.max_parts + c0) * D) + l4;
    // batches of 8 partitions: their loads go out together, then the sums
    // in partition order
    constexpr int BATCH = 8;
    int j = slot;
    for (; j + (BATCH - 1) * SLOTS < cnt; j += BATCH * SLOTS) {
      float4 o[BATCH];
#pragma unroll
      for (int k = 0; k < BATCH; ++k) o[k] = po[(size_t)(j + k * SLOTS) * LPP];
#pragma unroll
      for (int k = 0; k < BATCH; ++k) {
        const float w = w_s[j + k * SLOTS];
        acc.x += w * o[k].x;
        acc.y += w * o[k].y;
        acc.z += w * o[k].z;
        acc.w += w * o[k].w;
      }
    }
    for (; j < cnt; j += SLOTS) {
      const float w = w_s[j];
      const float4 o = po[(size_t)j * LPP];
      acc.x += w * o.x;
      acc.y += w * o.y;
      acc.z += w * o.z;
      acc.w += w * o.w;
    }
  }
  acc_s[slot][l4] = acc;
  // 3. the total weight: fixed-order warp and block sums
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
  __syncthreads();  // acc_s written; everyone is past the reads of red_s
  if (lane == 0) red_s[warp] = wsum;
  __syncthreads();
  if (tid < LPP) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < NWM; ++w) t += red_s[w];
    float4 a = acc_s[0][tid];
#pragma unroll
    for (int k = 1; k < SLOTS; ++k) {
      const float4 v = acc_s[k][tid];
      a.x += v.x;
      a.y += v.y;
      a.z += v.z;
      a.w += v.w;
    }
    const float inv = t > 0.f ? 1.f / t : 0.f;
    __nv_bfloat16 *orow = p.out + (size_t)row * D + 4 * tid;  // out is only 2-byte aligned
    orow[0] = __float2bfloat16_rn(a.x * inv);
    orow[1] = __float2bfloat16_rn(a.y * inv);
    orow[2] = __float2bfloat16_rn(a.z * inv);
    orow[3] = __float2bfloat16_rn(a.w * inv);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 5-D map over one cache: dims (innermost first) {box_elems, 16 tokens,
// num_kv_heads, head_dim slices, num_blocks}.  The token stride is larger
// than the head stride, so a box {box_elems, 16, 1, slices, 1} -- one head
// of one block -- lands in shared memory as [slice][token][box bytes]: the
// 16 tokens are consecutive swizzled rows, conflict-free for ldmatrix, and
// the whole tile is one copy.
bool encode_cache_map(CUtensorMap *map, void *base, const pkv_cache *c) {
  auto fn = encode_fn();
  if (!fn) return false;
  const bool fp8 = c->dtype == PKV_FP8_E4M3;
  const cuuint64_t elt = fp8 ? 1 : 2;
  const cuuint64_t row = (cuuint64_t)c->head_dim * elt;
  const cuuint32_t box_bytes = row >= 128 ? 128 : (cuuint32_t)row;
  const cuuint64_t slices = row / box_bytes;
  cuuint64_t dims[5] = {box_bytes / elt, 16, (cuuint64_t)c->num_kv_heads, slices,
                        (cuuint64_t)c->num_blocks};
  cuuint64_t strides[4] = {row * c->num_kv_heads, row, box_bytes, row * c->num_kv_heads * 16};
  cuuint32_t box[5] = {(cuuint32_t)(box_bytes / elt), 16, 1, (cuuint32_t)slices, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r =
      fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base,
         dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Small cache of encoded maps keyed by the cache geometry.
struct MapEntry {
  void *key_cache, *value_cache;
  int32_t num_blocks, num_kv_heads, head_dim, dtype;
  CUtensorMap k, v;
};

bool get_maps(const pkv_cache *c, CUtensorMap *k, CUtensorMap *v) {
  static std::mutex mu;
  static MapEntry entries[8];
  static int n_entries = 0, next = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_entries; ++i) {
    const MapEntry &e = entries[i];
    if (e.key_cache == c->key_cache && e.value_cache == c->value_cache &&
        e.num_blocks == c->num_blocks && e.num_kv_heads == c->num_kv_heads &&
        e.head_dim == c->head_dim && e.dtype == c->dtype) {
      *k = e.k;
      *v = e.v;
      return true;
    }
  }
  MapEntry e;
  e.key_cache = c->key_cache;
  e.value_cache = c->value_cache;
  e.num_blocks = c->num_blocks;
  e.num_kv_heads = c->num_kv_heads;
  e.head_dim = c->head_dim;
  e.dtype = c->dtype;
  if (!encode_cache_map(&e.k, c->key_cache, c) || !encode_cache_map(&e.v, c->value_cache, c))
    return false;
  entries[next] = e;
  next = (next + 1) % 8;
  if (n_entries < 8) ++n_entries;
  *k = e.k;
  *v = e.v;
  return true;
}

constexpr int kCtasPerSm = 3;  // 64 KiB rings

// Sequence index for DecodeParams::test_fail_seq (-1 = off).
std::atomic<int32_t> g_test_fail_seq{-1};

// Rows of sequences split into more partitions than this are merged by one
// CTA each (paged_decode_merge_wide_kernel), fewer by one warp each.
constexpr int kMergeWarpMaxParts = 8;

// Partitions this short are owned by single warps (DecodeParams::warp_parts).
constexpr int kWarpPartMaxTokens = 512;

// Automatic partition length: the longest of 256 * 2^k tokens that still
// gives about three waves of CTAs for the worst case (every sequence at
// max_seq_len); no split at all when the sequences alone fill them.
int auto_partition_tokens(int64_t batch, int64_t num_heads, int64_t num_kv_heads,
                          int64_t max_seq_len, int sms) {
  const int64_t whole = std::max<int64_t>(16, (max_seq_len + 15) / 16 * 16);
  const int64_t group = num_heads / num_kv_heads;
  const int64_t units = batch * num_kv_heads * ((group + 7) / 8);
  const int64_t target = (int64_t)sms * kCtasPerSm * 3;
  if (units >= target) return (int)std::min<int64_t>(whole, 1 << 30);
  int64_t pt = 256;
  while (pt * 2 < whole && units * ((whole + 2 * pt - 1) / (2 * pt)) >= target) pt *= 2;
  return (int)std::min<int64_t>(pt, whole);
}

struct PartLayout {
  size_t ml_off, bytes;
};

PartLayout part_layout(int64_t batch, int64_t num_heads, int64_t num_kv_heads,
                       int64_t head_dim, int64_t max_parts) {
  (void)num_kv_heads;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t rows = (size_t)batch * num_heads * max_parts;
  PartLayout l;
  l.ml_off = up(rows * head_dim * sizeof(float));
  l.bytes = l.ml_off + up(rows * sizeof(float2));
  return l;
}

// Launch with programmatic stream serialisation (see grid_dependency_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <bool FP8, int D, int NW = 4, int RING_KB = 64>
pkv_status launch_decode(const CUtensorMap &mk, const CUtensorMap &mv, const DecodeParams &p,
                         cudaStream_t s) {
  using C = Cfg<FP8, D, NW, RING_KB>;
  static int configured[64] = {0};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PKV_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!configured[dev]) {
      if (cudaFuncSetAttribute(paged_decode_kernel<FP8, D, NW, RING_KB>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               C::SMEM_BYTES) != cudaSuccess)
        return PKV_ERR_CUDA;
      configured[dev] = 1;
    }
  }
  const int grid_y = p.warp_parts ? (p.grid_parts + C::NW - 1) / C::NW : p.grid_parts;
  // partition-row-major launch order for warp-owned partitions: 512-token
  // partitions on the long-context step 412.6 -> 405.7 us; sequence-major
  // for CTA-shared partitions (Llama-8B step 95.9 vs 97.9 us part-major)
  dim3 grid = p.warp_parts ? dim3(p.num_kv_heads * p.q_groups, p.batch, grid_y)
                           : dim3(p.num_kv_heads * p.q_groups, grid_y, p.batch);
  if (launch_pdl(paged_decode_kernel<FP8, D, NW, RING_KB>, grid, dim3(C::NW * 32), C::SMEM_BYTES, s,
                 mk, mv, p) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (p.max_parts > 1) {
    const long long rows = (long long)p.batch * p.num_heads;
    const cudaError_t e =
        p.max_parts > kMergeWarpMaxParts
            ? launch_pdl(paged_decode_merge_wide_kernel<D>, dim3((unsigned)rows),
                         dim3(kMergeWideThreads), 0, s, p)
            : launch_pdl(paged_decode_merge_kernel<D>, dim3((unsigned)((rows + 7) / 8)),
                         dim3(256), 0, s, p);
    if (e != cudaSuccess) return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

}  // namespace

const void *error_word_attention() { return &g_err_attention; }

}  // namespace pkv

using namespace pkv;

extern "C" void pkv_testing_fail_decode_sequence(int32_t sequence) {
  g_test_fail_seq.store(sequence < 0 ? -1 : sequence, std::memory_order_relaxed);
}

extern "C" int32_t paged_attention_partition_tokens(int32_t batch, int32_t num_heads,
                                                    int32_t num_kv_heads, int32_t max_seq_len,
                                                    int32_t partition_tokens) {
  if (batch < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads ||
      max_seq_len < 0 || partition_tokens < 0 || partition_tokens % 16)
    return -1;
  if (partition_tokens > 0) return partition_tokens;
  const int sms = device_sm_count();
  return auto_partition_tokens(batch, num_heads, num_kv_heads, max_seq_len, sms > 0 ? sms : 148);
}

extern "C" size_t paged_attention_workspace_bytes(int32_t batch, int32_t num_heads,
                                                  int32_t num_kv_heads, int32_t head_dim,
                                                  int32_t max_seq_len,
                                                  int32_t partition_tokens) {
  const int32_t pt = paged_attention_partition_tokens(batch, num_heads, num_kv_heads, max_seq_len,
                                                      partition_tokens);
  if (pt <= 0 || batch <= 0 || head_dim <= 0) return 0;
  const int64_t parts = std::max<int64_t>(1, ((int64_t)max_seq_len + pt - 1) / pt);
  if (parts <= 1 || parts > INT32_MAX / 2) return 0;
  return part_layout(batch, num_heads, num_kv_heads, head_dim, parts).bytes;
}

namespace {

// paged_attention_decode, and with k_new / v_new the decode step (see
// DecodeParams::k_new).
pkv_status decode_entry(const void *q, const void *k_new, const void *v_new,
                        const int32_t *new_start_loc, int64_t num_new,
                        const pkv_cache *cache, const int32_t *block_tables, int32_t max_blocks,
                        const int32_t *seq_lens, int32_t batch, int32_t num_heads, float scale,
                        void *out, int32_t max_seq_len, int32_t partition_tokens,
                        void *workspace, size_t workspace_bytes, void *stream) {
  pkv_status st = validate_cache(cache);
  if (st != PKV_OK) return st;
  if (batch < 0 || num_heads <= 0 || max_blocks <= 0 || max_seq_len < 0 ||
      partition_tokens < 0 || partition_tokens % 16 || !std::isfinite(scale))
    return PKV_ERR_ARG;
  if (num_heads % cache->num_kv_heads) return PKV_ERR_SHAPE;
  if (batch == 0) return PKV_OK;
  if (!q || !out || !block_tables || !seq_lens) return PKV_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(q) & 15) return PKV_ERR_ARG;
  const bool fp8 = cache->dtype == PKV_FP8_E4M3;
  if (fp8 && !(cache->k_scale > 0.f && cache->v_scale > 0.f)) return PKV_ERR_ARG;
  if (batch > 65535) return PKV_ERR_ARG;
  const int group = num_heads / cache->num_kv_heads;
  const int q_groups = (group + 7) / 8;
  if ((int64_t)cache->num_kv_heads * q_groups > INT32_MAX) return PKV_ERR_ARG;
  const int32_t pt = paged_attention_partition_tokens(batch, num_heads, cache->num_kv_heads,
                                                      max_seq_len, partition_tokens);
  if (pt <= 0) return PKV_ERR_ARG;
  const int64_t parts64 = std::max<int64_t>(1, ((int64_t)max_seq_len + pt - 1) / pt);
  if (parts64 > 65535) return PKV_ERR_ARG;  // grid.y or grid.z

  DecodeParams p;
  std::memset(&p, 0, sizeof p);
  p.max_parts = (int)parts64;
  p.grid_parts = (int)parts64;
  p.part_tokens = pt;
  p.warp_parts = parts64 > 1 && pt <= kWarpPartMaxTokens;
  p.test_fail_seq = g_test_fail_seq.load(std::memory_order_relaxed);
  const size_t need = paged_attention_workspace_bytes(batch, num_heads, cache->num_kv_heads,
                                                      cache->head_dim, max_seq_len,
                                                      partition_tokens);
  if (need > 0) {
    if (!workspace || workspace_bytes < need) return PKV_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return PKV_ERR_WORKSPACE;
    const PartLayout l =
        part_layout(batch, num_heads, cache->num_kv_heads, cache->head_dim, p.max_parts);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    p.part_o = reinterpret_cast<float *>(ws);
    p.part_ml = reinterpret_cast<float2 *>(ws + l.ml_off);
  }

  CUtensorMap mk, mv;
  if (!get_maps(cache, &mk, &mv)) return PKV_ERR_CUDA;

  p.q = static_cast<const __nv_bfloat16 *>(q);
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.out = static_cast<__nv_bfloat16 *>(out);
  p.batch = batch;
  p.num_heads = num_heads;
  p.num_kv_heads = cache->num_kv_heads;
  p.group = group;
  p.q_groups = q_groups;
  p.num_blocks = cache->num_blocks;
  p.max_blocks = max_blocks;
  p.max_seq_len = max_seq_len;
  p.scale_log2 = scale * 1.4426950408889634f * (fp8 ? cache->k_scale : 1.f);
  p.v_scale = fp8 ? cache->v_scale : 1.f;
  p.timeout_ns = 2000000000ull;
  if (k_new) {
    p.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    p.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    p.new_start_loc = new_start_loc;
    p.num_new = num_new;
    p.k_cache = static_cast<uint8_t *>(cache->key_cache);
    p.v_cache = static_cast<uint8_t *>(cache->value_cache);
    p.k_scale = fp8 ? cache->k_scale : 1.f;
  }

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (fp8)
    return cache->head_dim == 128 ? launch_decode<true, 128>(mk, mv, p, s)
                                  : launch_decode<true, 64>(mk, mv, p, s);
  return cache->head_dim == 128 ? launch_decode<false, 128>(mk, mv, p, s)
                                : launch_decode<false, 64>(mk, mv, p, s);
}

}  // namespace

extern "C" pkv_status paged_attention_decode(const void *q, const pkv_cache *cache,
                                             const int32_t *block_tables, int32_t max_blocks,
                                             const int32_t *seq_lens, int32_t batch,
                                             int32_t num_heads, float scale, void *out,
                                             int32_t max_seq_len, int32_t partition_tokens,
                                             void *workspace, size_t workspace_bytes,
                                             void *stream) {
  return decode_entry(q, nullptr, nullptr, nullptr, 0, cache, block_tables, max_blocks,
                      seq_lens, batch, num_heads, scale, out, max_seq_len, partition_tokens,
                      workspace, workspace_bytes, stream);
}

extern "C" pkv_status paged_attention_decode_step(
    const void *q, const void *k_new, const void *v_new, const int32_t *new_start_loc,
    int64_t num_new_tokens, const pkv_cache *cache, const int32_t *block_tables,
    int32_t max_blocks, const int32_t *seq_lens, int32_t batch, int32_t num_heads, float scale,
    void *out, int32_t max_seq_len, int32_t partition_tokens, void *workspace,
    size_t workspace_bytes, void *stream) {
  if (num_new_tokens < 0 || (!new_start_loc && num_new_tokens != batch))
    return PKV_ERR_ARG;
  const bool any = batch > 0 && num_new_tokens > 0;
  if (any && (!k_new || !v_new ||
              ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15)))
    return PKV_ERR_ARG;
  return decode_entry(q, any ? k_new : nullptr, v_new, new_start_loc, num_new_tokens, cache,
                      block_tables, max_blocks, seq_lens, batch, num_heads, scale, out,
                      max_seq_len, partition_tokens, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------------------
// Cascade (shared-prefix) decode
// ---------------------------------------------------------------------------
namespace {

// The workspace holds prefix partials of this length (4 key tiles of the
// prefix pass); a launch may use longer ones, never shorter.
constexpr int kCascadePrefixPartTokens = 512;

// Prefix partition length for one call: as few partitions as fill one wave
// of CTAs (one per SM), so that the prefix pass leaves room on the SMs for
// the suffix pass running beside it and the merge has fewer slots to read.
// Shorter partitions (more CTAs than SMs) measured slower on a 16-group x
// 8-kv-head prefix of 1024 tokens: 512-token parts 83.7 us, 1024-token 81.2.
int cascade_prefix_part_tokens(int32_t num_groups, int32_t num_heads, int32_t num_kv_heads,
                               int32_t max_group_size, int32_t max_prefix_len) {
  const int g = num_heads / num_kv_heads;
  const int tq = std::max(1, 128 / g);
  const int64_t pairs = std::max(1, (max_group_size + tq - 1) / tq);
  const int64_t units = pairs * num_groups * num_kv_heads;
  const int64_t parts = std::max<int64_t>(1, device_sm_count() / std::max<int64_t>(1, units));
  const int64_t len = (max_prefix_len + parts - 1) / parts;
  const int64_t tokens = (len + 127) / 128 * 128;
  return (int)std::max<int64_t>(kCascadePrefixPartTokens, std::min<int64_t>(tokens, INT32_MAX / 2));
}

struct CascadeLayout {
  int32_t pt, prefix_parts, suffix_parts, stride;
  size_t ml_off, start_off, bytes;
};

bool cascade_layout(int32_t batch, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                    int32_t max_seq_len, int32_t max_prefix_len, int32_t partition_tokens,
                    CascadeLayout *l) {
  if (batch <= 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_seq_len < 0 ||
      max_prefix_len < 0 || max_prefix_len > max_seq_len)
    return false;
  const int32_t pt = paged_attention_partition_tokens(batch, num_heads, num_kv_heads,
                                                      max_seq_len, partition_tokens);
  if (pt <= 0) return false;
  l->pt = pt;
  l->prefix_parts =
      std::max(1, (max_prefix_len + kCascadePrefixPartTokens - 1) / kCascadePrefixPartTokens);
  l->suffix_parts = std::max<int32_t>(1, (int32_t)(((int64_t)max_seq_len + pt - 1) / pt));
  if ((int64_t)l->prefix_parts + l->suffix_parts > 65535) return false;
  l->stride = l->prefix_parts + l->suffix_parts;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t rows = (size_t)batch * num_heads * l->stride;
  l->ml_off = up(rows * head_dim * sizeof(float));
  l->start_off = l->ml_off + up(rows * sizeof(float2));
  l->bytes = l->start_off + up((size_t)batch * sizeof(int32_t));
  return true;
}

}  // namespace

extern "C" size_t paged_attention_cascade_workspace_bytes(int32_t batch, int32_t num_heads,
                                                          int32_t num_kv_heads, int32_t head_dim,
                                                          int32_t max_seq_len,
                                                          int32_t max_prefix_len,
                                                          int32_t partition_tokens) {
  CascadeLayout l;
  if (!cascade_layout(batch, num_heads, num_kv_heads, head_dim, max_seq_len, max_prefix_len,
                      partition_tokens, &l))
    return 0;
  return l.bytes;
}

extern "C" pkv_status paged_attention_decode_cascade(
    const void *q, const pkv_cache *cache, const int32_t *block_tables, int32_t max_blocks,
    const int32_t *seq_lens, int32_t batch, int32_t num_heads, const int32_t *group_start,
    const int32_t *prefix_len, int32_t num_groups, int32_t max_group_size, int32_t max_prefix_len,
    float scale, void *out, int32_t max_seq_len, int32_t partition_tokens, void *workspace,
    size_t workspace_bytes, void *stream) {
  pkv_status st = validate_cache(cache);
  if (st != PKV_OK) return st;
  const bool fp8 = cache->dtype == PKV_FP8_E4M3;
  if (fp8 && !(cache->k_scale > 0.f && cache->v_scale > 0.f)) return PKV_ERR_ARG;
  if (batch < 0 || num_heads <= 0 || max_blocks <= 0 || max_seq_len < 0 || num_groups < 0 ||
      max_group_size < 0 || max_prefix_len < 0 || (max_prefix_len & 15) ||
      partition_tokens < 0 || (partition_tokens & 15) || !std::isfinite(scale) ||
      !(scale > 0.f))
    return PKV_ERR_ARG;
  if (num_heads % cache->num_kv_heads) return PKV_ERR_SHAPE;
  const int group = num_heads / cache->num_kv_heads;
  if (group > 128) return PKV_ERR_SHAPE;
  if (batch == 0) return PKV_OK;
  if (!q || !out || !block_tables || !seq_lens || (num_groups > 0 && (!group_start || !prefix_len)))
    return PKV_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15) return PKV_ERR_ARG;
  if (batch > 65535 || num_groups > 65535) return PKV_ERR_ARG;
  CascadeLayout l;
  if (!cascade_layout(batch, num_heads, cache->num_kv_heads, cache->head_dim, max_seq_len,
                      max_prefix_len, partition_tokens, &l))
    return PKV_ERR_ARG;
  if (!workspace || workspace_bytes < l.bytes || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return PKV_ERR_WORKSPACE;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  float *part_o = reinterpret_cast<float *>(ws);
  float2 *part_ml = reinterpret_cast<float2 *>(ws + l.ml_off);
  int32_t *seq_start = reinterpret_cast<int32_t *>(ws + l.start_off);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  CUtensorMap mk, mv;
  if (!get_maps(cache, &mk, &mv)) return PKV_ERR_CUDA;
  // 1. each group's prefix, once for all its members (tensor cores).  Its
  //    CTAs (one wave) start first; the decode pass launches programmatically
  //    beside them, since the two passes do not depend on each other
  const bool with_prefix = num_groups > 0 && max_prefix_len > 0;
  const int part_tokens = cascade_prefix_part_tokens(num_groups, num_heads, cache->num_kv_heads,
                                                     max_group_size, max_prefix_len);
  if (with_prefix) {
    st = launch_prefix_partials(q, cache, block_tables, max_blocks, seq_lens, group_start,
                                prefix_len, num_groups, max_group_size, max_prefix_len, batch,
                                num_heads, scale, part_o, part_ml, l.stride, part_tokens, s);
    if (st != PKV_OK) return st;
  }
  // 2. each sequence's own tokens (and its start), then the log-sum-exp
  //    merge of all slots
  DecodeParams p;
  std::memset(&p, 0, sizeof p);
  p.q = static_cast<const __nv_bfloat16 *>(q);
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.out = static_cast<__nv_bfloat16 *>(out);
  p.part_o = part_o;
  p.part_ml = part_ml;
  p.batch = batch;
  p.num_heads = num_heads;
  p.num_kv_heads = cache->num_kv_heads;
  p.group = group;
  p.q_groups = (group + 7) / 8;
  p.num_blocks = cache->num_blocks;
  p.max_blocks = max_blocks;
  p.max_seq_len = max_seq_len;
  p.max_parts = l.stride;
  p.grid_parts = l.suffix_parts;
  p.part_tokens = l.pt;
  p.warp_parts = l.pt <= kWarpPartMaxTokens;
  p.test_fail_seq = g_test_fail_seq.load(std::memory_order_relaxed);
  p.scale_log2 = scale * 1.4426950408889634f * (fp8 ? cache->k_scale : 1.f);
  p.v_scale = fp8 ? cache->v_scale : 1.f;
  p.timeout_ns = 2000000000ull;
  p.group_start = with_prefix ? group_start : nullptr;
  p.prefix_len = prefix_len;
  p.num_groups = num_groups;
  p.max_group_size = max_group_size;
  p.max_prefix_len = max_prefix_len;
  p.prefix_part_tokens = part_tokens;
  p.seq_start = seq_start;
  p.defer_dep_wait = with_prefix;
  return fp8 ? (cache->head_dim == 128 ? launch_decode<true, 128>(mk, mv, p, s)
                                       : launch_decode<true, 64>(mk, mv, p, s))
             : (cache->head_dim == 128 ? launch_decode<false, 128>(mk, mv, p, s)
                                       : launch_decode<false, 64>(mk, mv, p, s));
}
