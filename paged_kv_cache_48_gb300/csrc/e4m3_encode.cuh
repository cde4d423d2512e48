// e4m3_encode.cuh -- bf16 / binary32 to E4M3 (OCP FP8, 4 exponent bits,
// 3 mantissa bits, bias 7, no infinities, NaN = S.1111.111), the cache
// encoding of an fp8 paged KV cache: q = E4M3(RN-even, saturating to
// +-448)(x / scale) with x / scale the IEEE binary32 quotient.  Shared by
// the slot-mapped write and the decode step's in-kernel write of the new
// token, so that both store the same bytes.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cstdint>

namespace pkv {

// Reciprocal bounds for the E4M3 encode: lo and hi bracket 1 / scale
// tightly enough that x * lo and x * hi (each rounded once) enclose the
// rounded quotient RN(x / scale) for every finite x whose quotient is a
// normal binary32 number: lo = RN(RN(1/s)(1 - 2^-20)) is below
// (1/s)(1 - 2^-21), so x * lo, rounded, stays below x/s (1 - 2^-21), which
// is below RN(x/s) (relative error at most 2^-24); hi likewise above.  E4M3
// rounding is monotonic, so when both products round to the same E4M3 code
// the quotient does too.  Where they differ (the quotient is near an E4M3
// midpoint) the quotient is computed by IEEE division; tiny quotients, in
// binary32's subnormal range, are far below the smallest E4M3 step and give
// +-0 either way.  ok = 0 (a scale below 1e-38 or above 2^126, where the
// reciprocal or its bounds leave the normal range) sends every value to
// division.
struct E4m3Recip {
  float lo, hi;
  int ok;
};

__device__ __forceinline__ E4m3Recip e4m3_recip(float scale) {
  const float r = __frcp_rn(scale);
  E4m3Recip e;
  e.ok = r >= 1.17549435e-38f && r < 1e38f;
  e.lo = __fmul_rn(r, 1.f - 0x1p-20f);
  e.hi = __fmul_rn(r, 1.f + 0x1p-20f);
  return e;
}

// Two values to two E4M3 bytes (low byte = a): the IEEE binary32 quotient
// x / scale, rounded to nearest even and saturated to +-448.  Both
// bracketing products of the pair come from one two-lane multiply each
// (each lane rounded as the scalar multiply), and each pair of products
// converts in one instruction.
__device__ __forceinline__ uint32_t quant2_e4m3(float a, float b, float scale, E4m3Recip r) {
  uint32_t lo, hi;
  asm("{\n"
      ".reg .b64 x, pl, ph, rl, rh;\n"
      ".reg .f32 l0, l1, h0, h1;\n"
      ".reg .b16 cl, ch;\n"
      "mov.b64 x, {%2, %3};\n"
      "mov.b64 rl, {%4, %4};\n"
      "mov.b64 rh, {%5, %5};\n"
      "mul.rn.f32x2 pl, x, rl;\n"
      "mul.rn.f32x2 ph, x, rh;\n"
      "mov.b64 {l0, l1}, pl;\n"
      "mov.b64 {h0, h1}, ph;\n"
      "cvt.rn.satfinite.e4m3x2.f32 cl, l1, l0;\n"
      "cvt.rn.satfinite.e4m3x2.f32 ch, h1, h0;\n"
      "cvt.u32.u16 %0, cl;\n"
      "cvt.u32.u16 %1, ch;\n"
      "}\n"
      : "=r"(lo), "=r"(hi)
      : "f"(a), "f"(b), "f"(r.lo), "f"(r.hi));
  if (r.ok && lo == hi) return lo;
  return __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(a, scale), __fdiv_rn(b, scale)),
                                  __NV_SATFINITE, __NV_E4M3);
}

// Eight bf16 values to eight E4M3 bytes.
__device__ __forceinline__ uint2 quant8_e4m3(const uint4 &src, float scale, E4m3Recip r) {
  const uint32_t w[4] = {src.x, src.y, src.z, src.w};
  uint32_t q[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)  // bf16 pair -> the binary32 values (exact)
    q[i] = quant2_e4m3(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u), scale, r);
  return make_uint2(__byte_perm(q[0], q[1], 0x5410), __byte_perm(q[2], q[3], 0x5410));
}

}  // namespace pkv
