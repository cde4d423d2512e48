// pkv_device.cuh -- device-side building blocks shared by the kernels of the
// paged KV-cache library: the device error word, bounded mbarrier waits,
// TMA tile loads, ldmatrix / movmatrix / mma.sync wrappers and the shared
// memory swizzle that matches the TMA tensor maps.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pagedkv.h"

namespace pkv {

// ---------------------------------------------------------------------------
// Device error word.  Each translation unit owns one (no relocatable device
// code).  Within a unit the first error since the last pkv_check() wins the
// compare-and-swap on `code` and stamps `when` with the GPU's global
// nanosecond timer; pkv_check() reports the earliest stamp over all units.
// Encoding of `code`: bits 63..56 = pkv_status, bits 55..0 = offending
// index + 1 (0 = none).
// ---------------------------------------------------------------------------
struct ErrorWord {
  unsigned long long code;
  unsigned long long when;
};

__device__ __forceinline__ void record_error(ErrorWord *word, int status, long long index) {
  const unsigned long long v =
      ((unsigned long long)(status & 0xFF) << 56) |
      ((unsigned long long)(index + 1) & 0x00FFFFFFFFFFFFFFull);
  if (atomicCAS(&word->code, 0ull, v) == 0ull) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    word->when = t;
  }
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of the library is launched
// with programmatic stream serialisation; it waits for its predecessor in
// the stream (completion and memory flush) before touching global memory,
// and immediately lets its own successor start launching, so launch latency
// overlaps the predecessor's tail.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Shared memory addressing
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Byte offset of 16-byte chunk `chunk` of token row `t` inside a K or V tile
// that TMA wrote as boxes of 16 rows x BOX_BYTES, consecutive boxes
// (head_dim slices) `box_stride` bytes apart: inside a box the 16-byte chunk
// index is XORed with the row index (128-byte swizzle: 3 bits, 64-byte
// swizzle: 2 bits of the 128-byte line index).  Box bases are multiples of
// the swizzle atom, so the XOR only depends on the offset within the box.
template <int BOX_BYTES>
__device__ __forceinline__ uint32_t tile_offset(int t, int chunk, uint32_t box_stride) {
  constexpr int CHUNKS = BOX_BYTES / 16;
  const int box = chunk / CHUNKS;
  const int c = chunk % CHUNKS;
  uint32_t off = t * BOX_BYTES + c * 16;
  if (BOX_BYTES == 128) {
    off ^= ((off >> 7) & 7u) << 4;
  } else {  // 64-byte rows, 64-byte swizzle
    off ^= ((off >> 7) & 3u) << 4;
  }
  return box * box_stride + off;
}

template <int BOX_BYTES>
__device__ __forceinline__ uint32_t tile_offset(int t, int chunk) {
  return tile_offset<BOX_BYTES>(t, chunk, 16 * BOX_BYTES);
}

// ---------------------------------------------------------------------------
// mbarrier (CTA scope)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar,
                                                      uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of `bar` to complete, giving up after about
// `limit_ns` nanoseconds.  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar,
                                                  uint32_t parity,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t start = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0 && global_timer_ns() - start > limit_ns) return false;
  }
}

// ---------------------------------------------------------------------------
// TMA: 5-D tiled tensor load into shared memory, completion on an mbarrier.
// Coordinates are element indices, innermost first.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_5d(void *dst, const CUtensorMap *map,
                                            uint64_t *bar, int c0, int c1, int c2, int c3,
                                            int c4, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_"
      "tx::bytes.L2::cache_hint [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3), "r"(c4), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;"
               : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;"
               : "=l"(p));
  return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(
                   reinterpret_cast<uint64_t>(map))
               : "memory");
}

// ---------------------------------------------------------------------------
// Warp-level matrix movement and mma.sync (m16n8k16, fp32 accumulate)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0,
                                            uint32_t &r1, uint32_t &r2,
                                            uint32_t &r3) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(addr)
      : "memory");
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t &r0,
                                                  uint32_t &r1, uint32_t &r2,
                                                  uint32_t &r3) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(addr)
      : "memory");
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;"
               : "=r"(d)
               : "r"(a));
  return d;
}

// D = A * B + D with A 16x16 (row), B 16x8 (col), bf16 inputs.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0,
                                         uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Same with f16 inputs (used for fp8 caches, decoded exactly to f16).
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0,
                                        uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two E4M3 bytes (low byte = first element) -> f16x2 (low half = first
// element).  Every E4M3 value, NaN included, is exactly representable.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(two));
  return d;
}

// Four E4M3 bytes of a register -> two f16x2 (bytes 0,1 -> lo; 2,3 -> hi),
// reading the register's 16-bit halves directly.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t four, uint32_t &lo, uint32_t &hi) {
  asm("{\n"
      ".reg .b16 a, b;\n"
      "mov.b32 {a, b}, %2;\n"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n"
      "cvt.rn.f16x2.e4m3x2 %1, b;\n"
      "}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(four));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b,
                                         uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

}  // namespace pkv
