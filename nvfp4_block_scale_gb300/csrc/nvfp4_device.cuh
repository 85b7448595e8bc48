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
#include <cuda_runtime.h>
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

// Error of a candidate scale minus the block's common sum x^2:
// s * (s*R - 2P), as fl(s * fma(s, R, -2P)).
__device__ __forceinline__ float cand_err(float s, float P, float R) {
  return __fmul_rn(s, __fmaf_rn(s, R, __fmul_rn(-2.0f, P)));
}

// 8 code bytes (16 weights) and their scale -> 8 bf16x2 of What: per byte,
// the E2M1 pair -> f16x2 (exact) -> f32 pair, times s (one packed multiply,
// fl(q * s)), -> bf16x2 (RNE).
__device__ __forceinline__ void dequant16_bf16(uint2 cw, float s, uint32_t (&w)[8]) {
#pragma unroll
  for (int k = 0; k < 8; k += 4) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t.reg .b32 h0, h1, h2, h3;\n\t"
        ".reg .f16 l0, u0, l1, u1, l2, u2, l3, u3;\n\t.reg .f32 fl0, fu0, fl1, fu1, fl2, fu2, fl3, fu3;\n\t"
        ".reg .b64 p0, p1, p2, p3, ss;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 h0, b0;\n\tcvt.rn.f16x2.e2m1x2 h1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 h2, b2;\n\tcvt.rn.f16x2.e2m1x2 h3, b3;\n\t"
        "mov.b32 {l0, u0}, h0;\n\tmov.b32 {l1, u1}, h1;\n\tmov.b32 {l2, u2}, h2;\n\tmov.b32 {l3, u3}, h3;\n\t"
        "cvt.f32.f16 fl0, l0;\n\tcvt.f32.f16 fu0, u0;\n\tcvt.f32.f16 fl1, l1;\n\tcvt.f32.f16 fu1, u1;\n\t"
        "cvt.f32.f16 fl2, l2;\n\tcvt.f32.f16 fu2, u2;\n\tcvt.f32.f16 fl3, l3;\n\tcvt.f32.f16 fu3, u3;\n\t"
        "mov.b64 ss, {%5, %5};\n\t"
        "mov.b64 p0, {fl0, fu0};\n\tmov.b64 p1, {fl1, fu1};\n\tmov.b64 p2, {fl2, fu2};\n\tmov.b64 p3, {fl3, fu3};\n\t"
        "mul.rn.f32x2 p0, p0, ss;\n\tmul.rn.f32x2 p1, p1, ss;\n\tmul.rn.f32x2 p2, p2, ss;\n\tmul.rn.f32x2 p3, p3, ss;\n\t"
        "mov.b64 {fl0, fu0}, p0;\n\tmov.b64 {fl1, fu1}, p1;\n\tmov.b64 {fl2, fu2}, p2;\n\tmov.b64 {fl3, fu3}, p3;\n\t"
        "cvt.rn.bf16x2.f32 %0, fu0, fl0;\n\tcvt.rn.bf16x2.f32 %1, fu1, fl1;\n\t"
        "cvt.rn.bf16x2.f32 %2, fu2, fl2;\n\tcvt.rn.bf16x2.f32 %3, fu3, fl3;\n\t}"
        : "=r"(w[k]), "=r"(w[k + 1]), "=r"(w[k + 2]), "=r"(w[k + 3])
        : "r"(k == 0 ? cw.x : cw.y), "f"(s));
  }
}

// ---------------------------------------------------------------------------
// Packed primitives for one 16-element block held by one thread.
// ---------------------------------------------------------------------------

typedef unsigned long long f32x2;  // two fp32 in one 64-bit register: {lo, hi}

__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// -fl(x / s) for both lanes of a signed pair (Markstein step of div_by_scale
// with negated operands, nr = -r): nq = fl(-x*r), e = fl(x + nq*s) (the exact
// remainder), w = fl(e*nr + nq) = -fl(x/s).  Negation commutes with
// round-to-nearest, so w is exactly the negated IEEE quotient, and the signs
// of zeros come out right: w = -(+-0) for x = +-0, and for s = 0 (r = 0)
// w = -(+-0) with the sign of x.  Callers encode w and flip the code signs.
__device__ __forceinline__ f32x2 negdiv2_by_scale(f32x2 x, f32x2 s, f32x2 nr) {
  f32x2 nq = mul2(x, nr);
  f32x2 e = fma2(nq, s, x);
  return fma2(e, nr, nq);
}

// One 16-element block: the signed weights as fp32 pairs; x[k] holds
// elements 2k (lo) and 2k+1 (hi).
struct Block16 {
  f32x2 x[8];
};

// Signed E2M1 codes of 8 quotients (4 pairs) packed into one word (element
// 2k in the low nibble of byte k).
__device__ __forceinline__ uint32_t encode8(f32x2 v0, f32x2 v1, f32x2 v2, f32x2 v3) {
  uint32_t r;
  asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\t.reg .f32 a0, b0, a1, b1, a2, b2, a3, b3;\n\t"
      "mov.b64 {a0, b0}, %1;\n\tmov.b64 {a1, b1}, %2;\n\tmov.b64 {a2, b2}, %3;\n\tmov.b64 {a3, b3}, %4;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t0, b0, a0;\n\tcvt.rn.satfinite.e2m1x2.f32 t1, b1, a1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t2, b2, a2;\n\tcvt.rn.satfinite.e2m1x2.f32 t3, b3, a3;\n\t"
      "mov.b32 %0, {t0, t1, t2, t3};\n\t}"
      : "=r"(r) : "l"(v0), "l"(v1), "l"(v2), "l"(v3));
  return r;
}

// As encode8, and also accumulates the sums of the block: P2 += x * q over
// the 4 pairs (fp32 pairs; products exact, sums exact by the range argument)
// and R2 += q^2 (f16x2, exact for up to 8 terms per lane).  q is decoded
// from the codes just produced (cvt f16x2 <- e2m1x2, then f16 -> f32).
__device__ __forceinline__ uint32_t encode8_sums(f32x2 v0, f32x2 v1, f32x2 v2, f32x2 v3, f32x2 x0, f32x2 x1,
                                                 f32x2 x2, f32x2 x3, f32x2 &P2, uint32_t &R2) {
  uint32_t r, q0, q1, q2, q3;
  asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\t.reg .f32 a0, b0, a1, b1, a2, b2, a3, b3;\n\t"
      "mov.b64 {a0, b0}, %5;\n\tmov.b64 {a1, b1}, %6;\n\tmov.b64 {a2, b2}, %7;\n\tmov.b64 {a3, b3}, %8;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t0, b0, a0;\n\tcvt.rn.satfinite.e2m1x2.f32 t1, b1, a1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t2, b2, a2;\n\tcvt.rn.satfinite.e2m1x2.f32 t3, b3, a3;\n\t"
      "mov.b32 %0, {t0, t1, t2, t3};\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, t0;\n\tcvt.rn.f16x2.e2m1x2 %2, t1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, t2;\n\tcvt.rn.f16x2.e2m1x2 %4, t3;\n\t}"
      : "=r"(r), "=r"(q0), "=r"(q1), "=r"(q2), "=r"(q3)
      : "l"(v0), "l"(v1), "l"(v2), "l"(v3));
  const uint32_t q[4] = {q0, q1, q2, q3};
  const f32x2 x[4] = {x0, x1, x2, x3};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    asm("fma.rn.f16x2 %0, %1, %1, %0;" : "+r"(R2) : "r"(q[k]));
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&q[k]));
    P2 = fma2(x[k], pack2(f.x, f.y), P2);
  }
  return r;
}

// f16x2 -> sum of both halves in fp32 (exact for the small integers/4 of R).
__device__ __forceinline__ float f16x2_sum(uint32_t h) {
  __half2 v = *reinterpret_cast<__half2 *>(&h);
  float2 f = __half22float2(v);
  return __fadd_rn(f.x, f.y);
}

// Loads of one block: 2 x 16 bytes -> Block16 (signed fp32 pairs) and the
// block's max |x| as bf16 bits.
__device__ __forceinline__ uint32_t unpack16(const uint4 &a, const uint4 &b, Block16 &blk) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t m = w[0];
#pragma unroll
  for (int k = 1; k < 8; ++k) asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(w[k]));
  m &= 0x7FFF7FFFu;
  const uint32_t amax_bits = max(m & 0xFFFFu, m >> 16);
#pragma unroll
  for (int k = 0; k < 8; ++k) blk.x[k] = pack2(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xFFFF0000u));
  return amax_bits;
}

// Quantizes a block with dequant scale s (reciprocal r): signed codes of
// elements 0-7 / 8-15 in c0 / c1; with `sums`, P = sum |x| q and R = sum q^2
// (both exact).  A zero scale (r = 0) gives sign-only codes and zero sums.
// The quotients are computed negated (negdiv2_by_scale): encoding -v gives
// the codes with every sign bit flipped and P with its sign flipped; both
// are undone once per word / block.
template <bool SUMS>
__device__ __forceinline__ void quant16(const Block16 &blk, float s, float r, uint32_t &c0, uint32_t &c1,
                                        float &P, float &R) {
  const f32x2 s2 = pack2(s, s), nr2 = pack2(-r, -r);
  f32x2 w[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) w[k] = negdiv2_by_scale(blk.x[k], s2, nr2);
  if (SUMS) {
    f32x2 p2 = 0ull;  // {+0, +0}
    uint32_t r2h = 0u;
    c0 = encode8_sums(w[0], w[1], w[2], w[3], blk.x[0], blk.x[1], blk.x[2], blk.x[3], p2, r2h);
    c1 = encode8_sums(w[4], w[5], w[6], w[7], blk.x[4], blk.x[5], blk.x[6], blk.x[7], p2, r2h);
    float plo, phi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(plo), "=f"(phi) : "l"(p2));
    P = -__fadd_rn(plo, phi);  // sum of x * (-q) -> sum |x| q
    R = f16x2_sum(r2h);
  } else {
    c0 = encode8(w[0], w[1], w[2], w[3]);
    c1 = encode8(w[4], w[5], w[6], w[7]);
  }
  c0 ^= 0x88888888u;
  c1 ^= 0x88888888u;
}

// P and R only (no codes): the candidate evaluation of the decoupled search.
__device__ __forceinline__ void sums8(f32x2 v0, f32x2 v1, f32x2 v2, f32x2 v3, f32x2 x0, f32x2 x1, f32x2 x2,
                                      f32x2 x3, f32x2 &P2, uint32_t &R2) {
  uint32_t q0, q1, q2, q3;
  asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\t.reg .f32 a0, b0, a1, b1, a2, b2, a3, b3;\n\t"
      "mov.b64 {a0, b0}, %4;\n\tmov.b64 {a1, b1}, %5;\n\tmov.b64 {a2, b2}, %6;\n\tmov.b64 {a3, b3}, %7;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t0, b0, a0;\n\tcvt.rn.satfinite.e2m1x2.f32 t1, b1, a1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t2, b2, a2;\n\tcvt.rn.satfinite.e2m1x2.f32 t3, b3, a3;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, t0;\n\tcvt.rn.f16x2.e2m1x2 %1, t1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, t2;\n\tcvt.rn.f16x2.e2m1x2 %3, t3;\n\t}"
      : "=r"(q0), "=r"(q1), "=r"(q2), "=r"(q3)
      : "l"(v0), "l"(v1), "l"(v2), "l"(v3));
  const uint32_t q[4] = {q0, q1, q2, q3};
  const f32x2 x[4] = {x0, x1, x2, x3};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    asm("fma.rn.f16x2 %0, %1, %1, %0;" : "+r"(R2) : "r"(q[k]));
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&q[k]));
    P2 = fma2(x[k], pack2(f.x, f.y), P2);
  }
}

// P = sum |x| q and R = sum q^2 of a block quantized with scale s (no codes).
__device__ __forceinline__ void block_sums(const Block16 &blk, float s, float r, float &P, float &R) {
  const f32x2 s2 = pack2(s, s), nr2 = pack2(-r, -r);
  f32x2 w[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) w[k] = negdiv2_by_scale(blk.x[k], s2, nr2);
  f32x2 p2 = 0ull;
  uint32_t r2h = 0u;
  sums8(w[0], w[1], w[2], w[3], blk.x[0], blk.x[1], blk.x[2], blk.x[3], p2, r2h);
  sums8(w[4], w[5], w[6], w[7], blk.x[4], blk.x[5], blk.x[6], blk.x[7], p2, r2h);
  float plo, phi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(plo), "=f"(phi) : "l"(p2));
  P = -__fadd_rn(plo, phi);
  R = f16x2_sum(r2h);
}

// The weights of a block as f16 pairs scaled by 2^sh, for the mixed
// f16 x f16 -> f32 fma of P.  sh = 4 - floor(log2 amax): |x| * 2^sh < 32 for
// the whole block, and every |x| >= amax / 2^18 -- which includes every
// element whose code is nonzero for any candidate scale -- has an exact f16
// image (8 significant bits, f16 normal range).
struct BlockH16 {
  uint32_t xh[8];
  float m2_unscale;  // 2 * 2^-sh: P = -(scaled sum) * 2^-sh, so -2P = scaled sum * m2_unscale
};

__device__ __forceinline__ void make_h16(const Block16 &blk, uint32_t amax_bits, BlockH16 &bh) {
  const int e = (int)(amax_bits >> 7);            // bf16 exponent field of amax
  const int se = min(max(258 - e, 1), 253);       // biased exponent of 2^sh
  const float sc = __uint_as_float((uint32_t)se << 23);
  bh.m2_unscale = __uint_as_float((uint32_t)(255 - se) << 23);  // 2^(1 - sh)
  const f32x2 sc2 = pack2(sc, sc);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const f32x2 y = mul2(blk.x[k], sc2);
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(y));
    __half2 hh = __floats2half2_rn(lo, hi);
    bh.xh[k] = *reinterpret_cast<uint32_t *>(&hh);
  }
}

// P (scaled, of the negated codes) and R2 of 4 pairs via mixed fma.
__device__ __forceinline__ void sums8_h(f32x2 v0, f32x2 v1, f32x2 v2, f32x2 v3, uint32_t h0, uint32_t h1,
                                        uint32_t h2, uint32_t h3, float &P, uint32_t &R2) {
  asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\t.reg .f32 a0, b0, a1, b1, a2, b2, a3, b3;\n\t"
      ".reg .b32 q0, q1, q2, q3;\n\t.reg .f16 ql, qh, xl, xh;\n\t"
      "mov.b64 {a0, b0}, %2;\n\tmov.b64 {a1, b1}, %3;\n\tmov.b64 {a2, b2}, %4;\n\tmov.b64 {a3, b3}, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t0, b0, a0;\n\tcvt.rn.satfinite.e2m1x2.f32 t1, b1, a1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t2, b2, a2;\n\tcvt.rn.satfinite.e2m1x2.f32 t3, b3, a3;\n\t"
      "cvt.rn.f16x2.e2m1x2 q0, t0;\n\tcvt.rn.f16x2.e2m1x2 q1, t1;\n\t"
      "cvt.rn.f16x2.e2m1x2 q2, t2;\n\tcvt.rn.f16x2.e2m1x2 q3, t3;\n\t"
      "fma.rn.f16x2 %1, q0, q0, %1;\n\tfma.rn.f16x2 %1, q1, q1, %1;\n\t"
      "fma.rn.f16x2 %1, q2, q2, %1;\n\tfma.rn.f16x2 %1, q3, q3, %1;\n\t"
      "mov.b32 {ql, qh}, q0;\n\tmov.b32 {xl, xh}, %6;\n\t"
      "fma.rn.f32.f16 %0, ql, xl, %0;\n\tfma.rn.f32.f16 %0, qh, xh, %0;\n\t"
      "mov.b32 {ql, qh}, q1;\n\tmov.b32 {xl, xh}, %7;\n\t"
      "fma.rn.f32.f16 %0, ql, xl, %0;\n\tfma.rn.f32.f16 %0, qh, xh, %0;\n\t"
      "mov.b32 {ql, qh}, q2;\n\tmov.b32 {xl, xh}, %8;\n\t"
      "fma.rn.f32.f16 %0, ql, xl, %0;\n\tfma.rn.f32.f16 %0, qh, xh, %0;\n\t"
      "mov.b32 {ql, qh}, q3;\n\tmov.b32 {xl, xh}, %9;\n\t"
      "fma.rn.f32.f16 %0, ql, xl, %0;\n\tfma.rn.f32.f16 %0, qh, xh, %0;\n\t}"
      : "+f"(P), "+r"(R2)
      : "l"(v0), "l"(v1), "l"(v2), "l"(v3), "r"(h0), "r"(h1), "r"(h2), "r"(h3));
}

// As block_sums, with P from the block's scaled f16 image; returns -2P (one
// exact power-of-two multiply of the scaled sum) for the error comparisons.
__device__ __forceinline__ void block_sums_h(const Block16 &blk, const BlockH16 &bh, float s, float r,
                                             float &m2P, float &R) {
  const f32x2 s2 = pack2(s, s), nr2 = pack2(-r, -r);
  f32x2 w[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) w[k] = negdiv2_by_scale(blk.x[k], s2, nr2);
  float p = 0.0f;
  uint32_t r2h = 0u;
  sums8_h(w[0], w[1], w[2], w[3], bh.xh[0], bh.xh[1], bh.xh[2], bh.xh[3], p, r2h);
  sums8_h(w[4], w[5], w[6], w[7], bh.xh[4], bh.xh[5], bh.xh[6], bh.xh[7], p, r2h);
  m2P = __fmul_rn(p, bh.m2_unscale);
  R = f16x2_sum(r2h);
}

// cand_err with -2P given: s * (s*R - 2P).
__device__ __forceinline__ float cand_err_m2p(float s, float m2P, float R) {
  return __fmul_rn(s, __fmaf_rn(s, R, m2P));
}

// Programmatic dependent launch: let the next kernel of the stream be
// scheduled now / wait until the previous kernel's writes are visible.  Both
// are no-ops when the launch carries no programmatic dependency.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Checked build (-DNVFP4_CHECKED).  The hot-path kernels test the index of
// each global-memory and table access against its buffer's extent before
// making it: NVFP4_IN(i, n, site) is true for 0 <= i < n; otherwise the access
// is skipped and `site` is recorded (the first failure wins) in a device word
// of the translation unit, which nvfp4_check_take reads and clears.  Without
// the define NVFP4_IN is the constant true and its arguments are not
// evaluated, so the normal build is unchanged.
// ---------------------------------------------------------------------------

// Sites: kernel << 8 | access.
enum : unsigned {
  kCkSelfTest = 0x0001u,
  kCkAmaxW = 0x0101u, kCkAmaxPart = 0x0102u,
  kCkBulkChunk = 0x0111u, kCkBulkStage = 0x0112u, kCkBulkPart = 0x0113u,
  kCkFoldPart = 0x0121u,
  kCkQuantW = 0x0201u, kCkQuantTab = 0x0202u, kCkQuantCodes = 0x0203u, kCkQuantScales = 0x0204u,
  kCkSweepW = 0x0301u, kCkSweepScales = 0x0302u, kCkSweepTab = 0x0303u, kCkSweepCodes = 0x0304u,
  kCkSweepPartIn = 0x0305u, kCkSweepPartOut = 0x0306u, kCkSweepHist = 0x0307u,
  kCkDecW = 0x0401u, kCkDecScales = 0x0402u, kCkDecTab = 0x0403u, kCkDecSlot = 0x0404u, kCkDecList = 0x0405u,
  kCkDecCodes = 0x0406u, kCkDecHist = 0x0407u,
  kCkPlainList = 0x0501u, kCkPlainW = 0x0502u, kCkPlainScales = 0x0503u, kCkPlainTab = 0x0504u,
  kCkPlainCodes = 0x0505u,
  kCkDequantIn = 0x0601u, kCkDequantTab = 0x0602u, kCkDequantOut = 0x0603u,
  kCkGroupTensor = 0x0701u, kCkGroupW = 0x0702u, kCkGroupAmax = 0x0703u, kCkGroupTab = 0x0704u,
  kCkGroupOut = 0x0705u,
};

#ifdef NVFP4_CHECKED
static __device__ unsigned int g_check_site;  // this translation unit's first failed check (0: none)

__device__ __forceinline__ bool ck_in(int64_t i, int64_t n, unsigned site) {
  const bool in = i >= 0 && i < n;
  if (!in) atomicCAS(&g_check_site, 0u, site);
  return in;
}
#define NVFP4_IN(i, n, site) ::nvfp4::ck_in((int64_t)(i), (int64_t)(n), (site))

// Reads and clears this translation unit's word (the device must be idle);
// a nonzero value goes to *site unless *site already holds one.
static inline cudaError_t check_take_here(uint32_t *site) {
  uint32_t v = 0u;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_check_site, sizeof v);
  if (e == cudaSuccess && v != 0u) {
    const uint32_t z = 0u;
    e = cudaMemcpyToSymbol(g_check_site, &z, sizeof z);
    if (*site == 0u) *site = v;
  }
  return e;
}
#else
#define NVFP4_IN(i, n, site) true
#endif

}  // namespace nvfp4
