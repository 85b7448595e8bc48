// nvfp4_device.cuh -- device-side number-format and arithmetic helpers for
// the NVFP4 kernels (sm_103a).  Hardware conversions are issued as inline PTX
// (cvt ... e2m1x2 / e4m3x2); every fp32 operation that decides a code is
// written with an explicit rounding intrinsic so the compiler cannot fuse or
// reorder it (the library is also built with --fmad=false).
//
// Citation keys (page title, part of the page):
//   [SOAR-Q]  "SOAR: Scale Optimization for Accurate Reconstruction in NVFP4
//             Quantization", NVFP4 quantizer equation (alpha, Delta_i,
//             piecewise FP4 rounding; M_FP4 = 6, M_FP8 = 448).
//   [FOS-01]  "SOAR 周冠军笔记 07 | 香草小张：NVFP4 量化改进与推测解码实践",
//             section 01 (the E2M1 value set).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace nvfp4 {

// Two fp32 -> two E4M3FN codes (round to nearest even, saturate at 448):
// `hi` goes to bits 8-15, `lo` to bits 0-7.  [SOAR-Q] Q_E4M3.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t e4m3_code(float v) { return cvt_e4m3x2(0.0f, v) & 0xFFu; }

// E4M3 code -> its value (exact: every E4M3FN value is an fp16 value).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  uint32_t h;
  uint16_t c = static_cast<uint16_t>(code & 0xFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(c));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
}

// Two fp32 -> one byte of two E2M1 codes, round to nearest with ties to the
// even code, saturating at 6: `hi` in bits 4-7, `lo` in bits 0-3.
// [SOAR-Q] piecewise FP4 rounding; [FOS-01] value set.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float hi, float lo) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// One byte of two E2M1 codes -> two floats (.x from bits 0-3, .y from bits 4-7).
__device__ __forceinline__ float2 e2m1x2_to_f32x2(uint32_t byte) {
  uint32_t h;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(h) : "r"(byte));
  return __half22float2(*reinterpret_cast<__half2 *>(&h));
}

// fl(x / s) for s > 0 given r = fl(1/s) (IEEE reciprocal): one Markstein
// correction of the product x*r.  Equals the IEEE quotient whenever the
// remainder x - q*s does not underflow, which holds for every x whose code
// depends on it under the inputs' range precondition (max|W| >= 2^-64).
__device__ __forceinline__ float div_by_scale(float x, float s, float r) {
  float q0 = __fmul_rn(x, r);
  float e = __fmaf_rn(-q0, s, x);
  return __fmaf_rn(e, r, q0);
}

// bf16 pair in a 32-bit word -> floats (element 2k in the low half).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Error of a candidate scale minus the block's common sum x^2:
// s * (s*R - 2P), as fl(s * fma(s, R, -2P)).
__device__ __forceinline__ float cand_err(float s, float P, float R) {
  return __fmul_rn(s, __fmaf_rn(s, R, __fmul_rn(-2.0f, P)));
}

// Eight elements (half of a 16-element block) quantized with dequant scale s
// and its reciprocal r: magnitude codes (nibble k = element k), P = sum |x| q
// and R = sum q^2.  A zero scale gives zero codes and sums.
struct HalfQ {
  uint32_t mags;
  float P, R;
};

__device__ __forceinline__ HalfQ quant_half(const float (&ax)[8], float s, float r) {
  HalfQ o;
  uint32_t mags = 0;
  float P = 0.0f, R = 0.0f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float v0 = div_by_scale(ax[2 * k], s, r);
    float v1 = div_by_scale(ax[2 * k + 1], s, r);
    uint32_t b = cvt_e2m1x2(v1, v0);
    float2 q = e2m1x2_to_f32x2(b);
    P = __fmaf_rn(ax[2 * k], q.x, P);
    P = __fmaf_rn(ax[2 * k + 1], q.y, P);
    R = __fmaf_rn(q.x, q.x, R);
    R = __fmaf_rn(q.y, q.y, R);
    mags |= b << (8 * k);
  }
  const bool live = s > 0.0f;
  o.mags = live ? mags : 0u;
  o.P = live ? P : 0.0f;
  o.R = live ? R : 0.0f;
  return o;
}

// Unpacks 8 bf16 (one uint4) into |x|, the sign nibble bits (bit 4k+3 = sign
// of element k) and the largest |x| as bf16 bits (0..0x7FFF).
__device__ __forceinline__ void unpack8(const uint4 &w, float (&ax)[8], uint32_t &sgn, uint32_t &amax_bits) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  sgn = 0;
  amax_bits = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t a = ws[k] & 0x7FFF7FFFu;
    ax[2 * k] = bf16_lo(a);
    ax[2 * k + 1] = bf16_hi(a);
    amax_bits = max(amax_bits, max(a & 0xFFFFu, a >> 16));
    sgn |= ((ws[k] >> 15) & 1u) << (8 * k + 3);
    sgn |= (ws[k] >> 31) << (8 * k + 7);
  }
}

// Compensated (float, float) accumulator, ~48 significant bits.
struct FF {
  float hi, lo;
};

__device__ __forceinline__ void ff_add(FF &a, float bh, float bl) {
  float s = __fadd_rn(a.hi, bh);
  float bp = __fsub_rn(s, a.hi);
  float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bp)), __fsub_rn(bh, bp));
  float lo = __fadd_rn(a.lo, __fadd_rn(e, bl));
  float t = __fadd_rn(s, lo);
  a.lo = __fsub_rn(lo, __fsub_rn(t, s));
  a.hi = t;
}

// Adds the exact product x*y (two-product via fma).
__device__ __forceinline__ void ff_add_prod(FF &a, float x, float y) {
  float p = __fmul_rn(x, y);
  float pe = __fmaf_rn(x, y, -p);
  ff_add(a, p, pe);
}

}  // namespace nvfp4
