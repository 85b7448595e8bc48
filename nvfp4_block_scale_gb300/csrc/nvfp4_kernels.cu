// nvfp4_kernels.cu -- sm_103a kernels of the NVFP4 quantization hot path.
//
// Work unit: one 16-element block (32 bytes of bf16, two 16-byte loads) per
// thread; a warp's loads cover 1 KiB of contiguous W.  The amax pass reads W
// as 16-byte units with 16 loads in flight per thread.  Per element the
// quotient |x| / fl(alpha * Delta) is an IEEE fp32 division reproduced by one
// packed Markstein step, and the code is the hardware E2M1 conversion of it.
//
// Citation keys (page title, part of the page):
//   [SOAR-Q]   "SOAR: Scale Optimization for Accurate Reconstruction in NVFP4
//              Quantization": NVFP4 quantizer equation.
//   [SOAR-DQ]  same page: dequantization equation.
//   [SOAR-A]   same page: closed form for the global scale alpha*.
//   [SOAR-D]   same page: closed form for a block scale Delta_i*.
//   [SOAR-SCHED] same page: CJSO schedule (max-rule start, re-quantize after
//              every update).
//   [FOS-02]   "SOAR 周冠军笔记 07 | 香草小张：NVFP4 量化改进与推测解码实践",
//              section 02 (FourOverSix).
#include <cuda_runtime.h>

#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// ---------------------------------------------------------------------------
// Block-wide reductions
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t *red) {
  v = __reduce_max_sync(0xFFFFFFFFu, v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t t = lane < kWarps ? red[lane] : 0u;
    t = __reduce_max_sync(0xFFFFFFFFu, t);
    if (lane == 0) red[0] = t;
  }
  __syncthreads();
  uint32_t r = red[0];
  __syncthreads();
  return r;
}

typedef unsigned __int128 u128;

__device__ __forceinline__ u128 shfl_xor_u128(u128 v, int o) {
  const uint64_t lo = __shfl_xor_sync(0xFFFFFFFFu, (unsigned long long)v, o);
  const uint64_t hi = __shfl_xor_sync(0xFFFFFFFFu, (unsigned long long)(v >> 64), o);
  return ((u128)hi << 64) | lo;
}

// Sums two 128-bit integers over the CTA (exact, so the order is immaterial);
// the result is valid in thread 0.
__device__ __forceinline__ void block_sum2_u128(u128 &a, u128 &b, ulonglong2 *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += shfl_xor_u128(a, o);
    b += shfl_xor_u128(b, o);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    red[2 * warp] = make_ulonglong2((unsigned long long)a, (unsigned long long)(a >> 64));
    red[2 * warp + 1] = make_ulonglong2((unsigned long long)b, (unsigned long long)(b >> 64));
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    u128 x = 0, y = 0;
    for (int w = 0; w < kWarps; ++w) {
      x += ((u128)red[2 * w].y << 64) | red[2 * w].x;
      y += ((u128)red[2 * w + 1].y << 64) | red[2 * w + 1].x;
    }
    a = x;
    b = y;
  }
  __syncthreads();
}

// A nonnegative 128-bit integer -> the nearest double, ties to the even one.
__device__ __forceinline__ double u128_to_double_rne(u128 v) {
  const uint64_t hi = (uint64_t)(v >> 64), lo = (uint64_t)v;
  const int h = hi ? 127 - __clzll((long long)hi) : (lo ? 63 - __clzll((long long)lo) : -1);
  if (h < 53) return (double)lo;  // exact
  const int drop = h - 52;
  uint64_t top = (uint64_t)(v >> drop);  // 53 bits
  const u128 rest = v & (((u128)1 << drop) - 1);
  const u128 half = (u128)1 << (drop - 1);
  if (rest > half || (rest == half && (top & 1u))) top += 1;  // 2^53 at most: still exact
  return ldexp((double)top, drop);
}

// A 128-bit accumulator as two 64-bit words (added with carries by hand:
// cheaper than the compiler's 128-bit arithmetic on the hot path).
struct Acc128 {
  uint64_t lo = 0, hi = 0;
  __device__ __forceinline__ void add(uint64_t l, uint64_t h) {
    lo += l;
    hi += h + (lo < l ? 1u : 0u);
  }
  __device__ __forceinline__ u128 get() const { return ((u128)hi << 64) | lo; }
};

// The exact terms of [SOAR-A]'s sums for one block: Delta^2 R in units of
// 2^-20 (Delta = M 2^-9, R = R4 / 4) and Delta P in units of 2^U, P the exact
// fp32 sum (bits below 2^U, which in-range inputs never have, are dropped).
__device__ __forceinline__ void alpha_terms(uint32_t M, float P, float R, int U, Acc128 &num, Acc128 &den) {
  const uint32_t R4 = __float2uint_rz(__fmul_rn(R, 4.0f));
  den.add((uint64_t)M * M * R4, 0u);  // < 2^48
  const uint32_t pb = __float_as_uint(P);
  if (P > 0.0f && M > 0u) {
    const uint32_t e = pb >> 23;
    const uint64_t mP = e ? (pb & 0x7FFFFFu) | 0x800000u : (pb & 0x7FFFFFu);  // P = mP 2^(max(e,1) - 150)
    const int sh = (int)(e ? e : 1u) - 150 - 9 - U;
    const uint64_t tv = (uint64_t)M * mP;  // < 2^42
    if (sh >= 0 && sh < 64) {              // the usual case
      num.add(tv << sh, sh ? tv >> (64 - sh) : 0u);
    } else {
      const u128 v = sh >= 0 ? (u128)tv << sh : (u128)tv >> (-sh);
      num.add((uint64_t)v, (uint64_t)(v >> 64));
    }
  }
}

// [SOAR-Q] alpha = max|W| / (6*448), from the per-CTA amax partials.
__device__ __forceinline__ float fold_alpha(const uint32_t *__restrict__ part, int n, uint32_t *red) {
  uint32_t m = 0;
  for (int i = threadIdx.x; i < n; i += 4 * kThreads) {  // four loads in flight per thread
    const uint32_t a = NVFP4_IN(i, n, kCkFoldPart) ? part[i] : 0u;
    const uint32_t b = i + kThreads < n ? part[i + kThreads] : 0u;
    const uint32_t c = i + 2 * kThreads < n ? part[i + 2 * kThreads] : 0u;
    const uint32_t d = i + 3 * kThreads < n ? part[i + 3 * kThreads] : 0u;
    m = max(max(m, a), max(b, max(c, d)));
  }
  m = block_max_u32(m, red);
  return __fdiv_rn(__uint_as_float(m << 16), 2688.0f);
}

// Per-CTA tables over all 128 non-negative E4M3 codes: dequant scale
// s = fl(alpha*Delta) and its IEEE reciprocal (0 where s == 0).
__device__ __forceinline__ void build_scale_tables(float alpha, float *s_tab, float *r_tab) {
  if (threadIdx.x < 128) {
    float s = __fmul_rn(alpha, e4m3_value(threadIdx.x));
    s_tab[threadIdx.x] = s;
    r_tab[threadIdx.x] = s > 0.0f ? __frcp_rn(s) : 0.0f;
  }
}

// [SOAR-Q] max rule for one block: Delta = e4m3(fl(amax_i / fl(6 alpha))).
__device__ __forceinline__ uint32_t max_rule_code(uint32_t amax_bits, float six_a, float r6) {
  if (!(six_a > 0.0f)) return 0u;
  return e4m3_code(div_by_scale(__uint_as_float(amax_bits << 16), six_a, r6));
}

__device__ __forceinline__ uint4 load_half(const uint4 *__restrict__ W, int64_t h, bool valid) {
  return valid ? __ldg(W + h) : make_uint4(0u, 0u, 0u, 0u);
}

// ---------------------------------------------------------------------------
// a1: global amax partials
// ---------------------------------------------------------------------------

// Each CTA walks tiles of kThreads * kAmaxUnroll 16-byte units (all loads of
// a tile in flight at once), keeps max |x| as a bf16 pair, and writes one
// partial.  Launched as a programmatic dependent of whatever precedes it on
// the stream, it waits for that grid before touching W, then lets the
// quantize kernel be scheduled at once; that kernel waits for this grid's
// completion before reading the partials.
constexpr int kAmaxUnroll = 8;

__global__ void __launch_bounds__(kThreads) k_amax_partials(const uint4 *__restrict__ W, int64_t n16,
                                                            uint32_t *__restrict__ part) {
  __shared__ uint32_t red[kWarps];
  const int64_t tile = (int64_t)kThreads * kAmaxUnroll;
  pdl_wait();  // W may be written by the previous kernel of the stream
  pdl_launch_dependents();
  uint32_t m = 0u;
  for (int64_t base = (int64_t)blockIdx.x * tile + threadIdx.x; base < n16; base += (int64_t)gridDim.x * tile) {
    uint4 v[kAmaxUnroll];
    if (base + (int64_t)(kAmaxUnroll - 1) * kThreads < n16) {
      // whole tile: every load issued before the first use (volatile keeps the order)
#pragma unroll
      for (int u = 0; u < kAmaxUnroll; ++u) {
        v[u] = make_uint4(0u, 0u, 0u, 0u);
        if (NVFP4_IN(base + (int64_t)u * kThreads, n16, kCkAmaxW))
          asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(v[u].x), "=r"(v[u].y), "=r"(v[u].z), "=r"(v[u].w)
                       : "l"(W + base + (int64_t)u * kThreads));
      }
    } else {
#pragma unroll
      for (int u = 0; u < kAmaxUnroll; ++u) {
        const int64_t i = base + (int64_t)u * kThreads;
        v[u] = i < n16 ? __ldg(W + i) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u) {
      asm volatile("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(v[u].x));
      asm volatile("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(v[u].y));
      asm volatile("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(v[u].z));
      asm volatile("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(v[u].w));
    }
  }
  m &= 0x7FFF7FFFu;
  m = block_max_u32(max(m & 0xFFFFu, m >> 16), red);
  if (threadIdx.x == 0) part[blockIdx.x] = m;
}

// Bulk-copy form of the same pass: each CTA streams chunks c, c + G, ... of
// kAmaxChunk bytes through kAmaxStages shared-memory stages filled by
// cp.async.bulk (one elected thread issues, an mbarrier counts the bytes);
// all threads reduce a stage, then it is refilled.  Every mbarrier wait is
// bounded: on a timeout the CTA waits (bounded, at the normal limit) for its
// copies in flight and writes the partial 0xFFFFFFFF, which makes the
// quantize kernel's alpha NaN.
constexpr int kAmaxStages = 4;
constexpr int kAmaxChunk = 32768;
constexpr size_t kAmaxBulkSmem = (size_t)kAmaxStages * kAmaxChunk;
constexpr long kSpinLimit = 1L << 24;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool mbar_wait_bounded(uint32_t mb, uint32_t parity, long limit = kSpinLimit) {
  uint32_t done = 0;
  for (long it = 0; !done && it < limit; ++it)
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}" : "=r"(done) : "r"(mb), "r"(parity) : "memory");
  return done != 0;
}

__global__ void __launch_bounds__(kThreads) k_amax_bulk(const uint4 *__restrict__ W, int64_t n16,
                                                        uint32_t *__restrict__ part, long first_limit) {
  extern __shared__ __align__(128) uint4 stage[];  // kAmaxStages x kAmaxChunk bytes
  __shared__ __align__(8) uint64_t mbar[kAmaxStages];
  __shared__ uint32_t red[kWarps];
  constexpr int64_t kUnits = kAmaxChunk / 16;
  const int64_t nch = (n16 + kUnits - 1) / kUnits;
  const char *src = reinterpret_cast<const char *>(W);
  if (threadIdx.x == 0) {
    for (int st = 0; st < kAmaxStages; ++st) asm volatile("mbarrier.init.shared.b64 [%0], 1;" ::"r"(smem_addr(&mbar[st])));
    asm volatile("fence.mbarrier_init.release.cluster;");
    asm volatile("fence.proxy.async.shared::cta;");
  }
  __syncthreads();
  pdl_wait();  // W may be written by the previous kernel of the stream
  pdl_launch_dependents();
  auto bytes_of = [&](int64_t ch) { return (uint32_t)(min(kUnits, n16 - ch * kUnits) * 16); };
  auto issue = [&](int64_t ch, int st) {
    const uint32_t mb = smem_addr(&mbar[st]), nb = bytes_of(ch);
    if (!NVFP4_IN(ch * kUnits + nb / 16 - 1, n16, kCkBulkChunk) || !NVFP4_IN(st, kAmaxStages, kCkBulkStage)) return;
    asm volatile("mbarrier.arrive.expect_tx.shared.b64 _, [%0], %1;" ::"r"(mb), "r"(nb) : "memory");
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_addr(stage + (int64_t)st * kUnits)), "l"(src + ch * kAmaxChunk), "r"(nb), "r"(mb)
                 : "memory");
  };
  if (threadIdx.x == 0)
    for (int st = 0; st < kAmaxStages; ++st) {
      const int64_t ch = blockIdx.x + (int64_t)st * gridDim.x;
      if (ch < nch) issue(ch, st);
    }
  uint32_t m = 0u;
  bool ok = true;  // uniform over the CTA
  int j = 0;
  for (int64_t ch = blockIdx.x; ch < nch; ch += gridDim.x, ++j) {
    const int st = j % kAmaxStages;
    // (first_limit < 0: the normal limit; a test hook can make the first wait give up)
    const bool arrived = mbar_wait_bounded(smem_addr(&mbar[st]), (uint32_t)((j / kAmaxStages) & 1),
                                           j == 0 && first_limit >= 0 ? first_limit : kSpinLimit);
    if (!__syncthreads_and(arrived)) {
      ok = false;
      break;
    }
    const uint4 *p = stage + (int64_t)st * kUnits;
    const int units = (int)(bytes_of(ch) / 16);
    for (int i = threadIdx.x; i < units; i += kThreads) {
      const uint4 v = NVFP4_IN((int64_t)st * kUnits + i, (int64_t)kAmaxStages * kUnits, kCkBulkStage)
                          ? p[i] : make_uint4(0u, 0u, 0u, 0u);
      asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(v.x));
      asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(v.y));
      asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(v.z));
      asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(v.w));
    }
    __syncthreads();  // the stage has been read by every thread
    if (threadIdx.x == 0) {
      const int64_t nx = ch + (int64_t)kAmaxStages * gridDim.x;
      if (nx < nch) issue(nx, st);
    }
  }
  if (!ok) {  // a copy did not arrive in time: wait (bounded) for every copy still in flight
    if (threadIdx.x == 0)
      for (int jj = j; jj < j + kAmaxStages; ++jj) {
        if ((int64_t)blockIdx.x + (int64_t)jj * gridDim.x >= nch) break;
        mbar_wait_bounded(smem_addr(&mbar[jj % kAmaxStages]), (uint32_t)((jj / kAmaxStages) & 1));
      }
    if (threadIdx.x == 0) part[blockIdx.x] = 0xFFFFFFFFu;
    return;
  }
  m &= 0x7FFF7FFFu;
  m = block_max_u32(max(m & 0xFFFFu, m >> 16), red);
  if (threadIdx.x == 0) part[blockIdx.x] = m;
}

// ---------------------------------------------------------------------------
// a2-a4, a7: max rule and FourOverSix
// ---------------------------------------------------------------------------

// One 16-element block per thread, the thread's next two blocks in flight
// while one is computed.  Two block orders: `ranged` (W fits in L2, so the
// order does not matter for traffic) gives every CTA a contiguous, equal
// range, so all SMs finish together; otherwise the grid strides from the last
// block down, because the amax pass read the end of W last and that part is
// still in L2.  Launched as a programmatic dependent of k_amax_partials: W was
// final before that kernel read it, so the first blocks are fetched before the
// wait.  It lets the next kernel of the stream be scheduled early; that kernel
// waits for this one to finish.
template <int MODE>
__global__ void __launch_bounds__(kThreads) k_quant_max_fos(const uint4 *__restrict__ W, int64_t B,
                                                            const uint32_t *__restrict__ amax_part, int n_amax,
                                                            uint32_t *__restrict__ codes32,
                                                            uint8_t *__restrict__ scales,
                                                            float *__restrict__ alpha_out, int ranged) {
  __shared__ uint32_t red[kWarps];
  __shared__ float s_tab[128], r_tab[128], ev_tab[128];
  __shared__ uint8_t c4_tab[128];
  constexpr bool FOS = MODE == kModeFourOverSix;
  int64_t b, step, end;
  if (ranged) {  // blocks [B*c/G, B*(c+1)/G) of CTA c, ascending
    b = B * blockIdx.x / gridDim.x + threadIdx.x;
    end = B * (blockIdx.x + 1) / gridDim.x;
    step = kThreads;
  } else {  // grid-stride from the last block down
    b = B - 1 - ((int64_t)blockIdx.x * kThreads + threadIdx.x);
    step = -(int64_t)gridDim.x * kThreads;
    end = -1;
  }
  auto ok = [&](int64_t x) { return ranged ? x < end : x > end; };
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  const bool v0 = ok(b) && NVFP4_IN(2 * b + 1, 2 * B, kCkQuantW);
  uint4 a0 = v0 ? __ldg(W + 2 * b) : z, a1 = v0 ? __ldg(W + 2 * b + 1) : z;
  const int64_t b1 = b + step;
  const bool v1 = ok(b1) && NVFP4_IN(2 * b1 + 1, 2 * B, kCkQuantW);
  uint4 n0 = v1 ? __ldg(W + 2 * b1) : z, n1 = v1 ? __ldg(W + 2 * b1 + 1) : z;
  if (threadIdx.x < 128) {  // alpha-independent part of the tables
    const float ev = e4m3_value(threadIdx.x);
    ev_tab[threadIdx.x] = ev;
    if (FOS) c4_tab[threadIdx.x] = (uint8_t)e4m3_code(__fmul_rn(ev, 1.5f));  // [FOS-02] scale_m4 = fp8(scale_m6 * 1.5)
  }

  pdl_launch_dependents();
  pdl_wait();
  const float alpha = fold_alpha(amax_part, n_amax, red);  // (its barriers also publish ev_tab)
  if (blockIdx.x == 0 && threadIdx.x == 0) *alpha_out = alpha;
  const float six_a = __fmul_rn(alpha, 6.0f);
  const float r6 = six_a > 0.0f ? __frcp_rn(six_a) : 0.0f;
  if (threadIdx.x < 128) {
    const float sv = __fmul_rn(alpha, ev_tab[threadIdx.x]);
    s_tab[threadIdx.x] = sv;
    r_tab[threadIdx.x] = sv > 0.0f ? __frcp_rn(sv) : 0.0f;
  }
  __syncthreads();

  // The walk, unrolled three times: each step issues the loads of the block two steps
  // ahead into the buffer it has just consumed, so the three buffers take turns
  // without register copies.
  auto fetch = [&](int64_t x, uint4 &y0, uint4 &y1) {
    const bool v = ok(x) && NVFP4_IN(2 * x + 1, 2 * B, kCkQuantW);
    y0 = v ? __ldg(W + 2 * x) : z;
    y1 = v ? __ldg(W + 2 * x + 1) : z;
  };
  auto quantize_block = [&](const uint4 &x0, const uint4 &x1) {
    Block16 blk;
    const uint32_t am = unpack16(x0, x1, blk);
    uint32_t d6 = max_rule_code(am, six_a, r6);
    if (!NVFP4_IN(d6, 128, kCkQuantTab)) d6 = 0u;
    uint32_t c0, c1, d = d6;
    float P6, R6;
    quant16<FOS>(blk, s_tab[d6], r_tab[d6], c0, c1, P6, R6);
    if (FOS) {
      // [FOS-02] keep scale_m4 iff its dequant error is strictly lower.
      uint32_t d4 = c4_tab[d6];
      if (!NVFP4_IN(d4, 128, kCkQuantTab)) d4 = 0u;
      uint32_t e0, e1;
      float P4, R4;
      quant16<true>(blk, s_tab[d4], r_tab[d4], e0, e1, P4, R4);
      const bool use4 = cand_err(s_tab[d4], P4, R4) < cand_err(s_tab[d6], P6, R6);
      d = use4 ? d4 : d6;
      c0 = use4 ? e0 : c0;
      c1 = use4 ? e1 : c1;
    }
    if (NVFP4_IN(2 * b + 1, 2 * B, kCkQuantCodes)) {
      codes32[2 * b] = c0;  // two 4-byte stores: codes is only 4-byte aligned
      codes32[2 * b + 1] = c1;
    }
    if (NVFP4_IN(b, B, kCkQuantScales)) scales[b] = (uint8_t)d;
  };
  uint4 m0, m1;
  while (ok(b)) {
    fetch(b + 2 * step, m0, m1);
    quantize_block(a0, a1);
    b += step;
    if (!ok(b)) break;
    fetch(b + 2 * step, a0, a1);
    quantize_block(n0, n1);
    b += step;
    if (!ok(b)) break;
    fetch(b + 2 * step, n0, n1);
    quantize_block(m0, m1);
    b += step;
  }
}

// ---------------------------------------------------------------------------
// a5: CJSO sweeps
// ---------------------------------------------------------------------------

// One sweep over all blocks, one block per thread.  INIT: max rule from the
// amax partials.  Otherwise: alpha from the previous sweep's partial sums
// ([SOAR-A]), sums with the stored Delta, Delta* ([SOAR-D]) rounded to E4M3,
// re-quantize ([SOAR-SCHED]).  Every sweep stores Delta, writes its CTA's
// partial sums sum Delta P and sum Delta^2 R (exact 128-bit integers: Delta P
// in units of 2^U with U = the exponent of the sweep's alpha - 48, Delta^2 R
// in units of 2^-20), and records alpha in alpha_hist[t]; the next sweep adds
// all partials exactly, rounds each sum once to double and takes the quotient
// in double, so alpha does not depend on the order of the blocks.  Sweeps
// chain by programmatic dependent launch: each prefetches its first blocks of
// W (an input, final before the chain began) and then waits for the previous
// sweep before reading the partials and the scales.  `descending` alternates
// between sweeps so that each starts on the part of W the previous one read
// last (still in L2 when W is larger than L2).  A sweep without SUMS (the last
// of a call: no alpha step follows) neither forms nor writes the partial sums.
__device__ __forceinline__ int alpha_unit(float alpha) { return (int)((__float_as_uint(alpha) >> 23) & 0xFFu) - 127 - 48; }

template <bool INIT, bool SUMS>
__global__ void __launch_bounds__(kThreads) k_cjso_sweep(const uint4 *__restrict__ W, int64_t B,
                                                         const uint32_t *__restrict__ amax_part, int n_amax,
                                                         const ulonglong2 *__restrict__ part_in, int n_in,
                                                         ulonglong2 *__restrict__ part_out,
                                                         float *__restrict__ alpha_hist, int t,
                                                         uint8_t *__restrict__ scales,
                                                         uint32_t *__restrict__ codes32, int write_codes,
                                                         float *__restrict__ alpha_out, int write_alpha,
                                                         int descending) {
  __shared__ uint32_t red[kWarps];
  __shared__ ulonglong2 redu[2 * kWarps];
  __shared__ float s_tab[128], r_tab[128], ev_tab[128];
  __shared__ uint32_t m_tab[128];  // E4M3 value * 2^9
  __shared__ float sh_alpha;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  const int64_t i0 = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const int64_t step = descending ? -stride : stride;
  int64_t b = descending ? B - 1 - i0 : i0;
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  auto ok = [&](int64_t x) { return x >= 0 && x < B; };
  const bool v0 = ok(b) && NVFP4_IN(2 * b + 1, 2 * B, kCkSweepW);
  const bool v1 = ok(b + step) && NVFP4_IN(2 * (b + step) + 1, 2 * B, kCkSweepW);
  uint4 a0 = v0 ? __ldg(W + 2 * b) : z, a1 = v0 ? __ldg(W + 2 * b + 1) : z;
  uint4 n0 = v1 ? __ldg(W + 2 * (b + step)) : z, n1 = v1 ? __ldg(W + 2 * (b + step) + 1) : z;
  if (threadIdx.x < 128) {
    const float ev = e4m3_value(threadIdx.x);
    ev_tab[threadIdx.x] = ev;
    m_tab[threadIdx.x] = __float2uint_rz(__fmul_rn(ev, 512.0f));
  }

  pdl_launch_dependents();
  pdl_wait();
  float alpha;
  if (INIT) {
    alpha = fold_alpha(amax_part, n_amax, red);
  } else {
    u128 num = 0, den = 0;
    for (int i = threadIdx.x; i < n_in; i += kThreads) {
      const ulonglong2 pn = part_in[2 * i], pd = part_in[2 * i + 1];
      num += ((u128)pn.y << 64) | pn.x;
      den += ((u128)pd.y << 64) | pd.x;
    }
    block_sum2_u128(num, den, redu);
    if (threadIdx.x == 0) {
      // the alpha the partial sums were formed with
      const float prev = NVFP4_IN(t - 1, kMaxIters + 1, kCkSweepHist) ? alpha_hist[t - 1] : 0.0f;
      if (den == 0) {
        sh_alpha = prev;
      } else {
        const double dn = ldexp(u128_to_double_rne(num), alpha_unit(prev));
        const double dd = ldexp(u128_to_double_rne(den), -20);
        sh_alpha = __double2float_rn(__ddiv_rn(dn, dd));
      }
    }
    __syncthreads();
    alpha = sh_alpha;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (NVFP4_IN(t, kMaxIters + 1, kCkSweepHist)) alpha_hist[t] = alpha;
    if (write_alpha) *alpha_out = alpha;
  }
  const float six_a = __fmul_rn(alpha, 6.0f);
  const float r6 = six_a > 0.0f ? __frcp_rn(six_a) : 0.0f;
  const int U = alpha_unit(alpha);
  build_scale_tables(alpha, s_tab, r_tab);
  uint32_t sa = 0u, sn = 0u;  // stored scales of the current and the next block, fetched ahead
  if (!INIT) {
    sa = ok(b) && NVFP4_IN(b, B, kCkSweepScales) ? scales[b] : 0u;
    sn = ok(b + step) && NVFP4_IN(b + step, B, kCkSweepScales) ? scales[b + step] : 0u;
  }
  __syncthreads();

  Acc128 num_acc, den_acc;
  // The walk, unrolled three times as in k_quant_max_fos: each step issues the loads of the
  // block two steps ahead (W and its stored scale) into the buffer it has just consumed.
  auto fetch = [&](int64_t x, uint4 &y0, uint4 &y1, uint32_t &ys) {
    const bool v = ok(x) && NVFP4_IN(2 * x + 1, 2 * B, kCkSweepW);
    y0 = v ? __ldg(W + 2 * x) : z;
    y1 = v ? __ldg(W + 2 * x + 1) : z;
    ys = (!INIT && ok(x) && NVFP4_IN(x, B, kCkSweepScales)) ? scales[x] : 0u;
  };
  auto sweep_block = [&](const uint4 &x0, const uint4 &x1, uint32_t xs) {
    Block16 blk;
    const uint32_t am = unpack16(x0, x1, blk);
    uint32_t d, d_old = 0xFFu;
    float P, R;
    if (INIT) {
      d = max_rule_code(am, six_a, r6);
    } else {
      d = d_old = NVFP4_IN(xs, 128, kCkSweepTab) ? xs : 0u;
      block_sums(blk, s_tab[d], r_tab[d], P, R);
      if (R > 0.0f) d = e4m3_code(__fdiv_rn(P, __fmul_rn(alpha, R)));
    }
    if (!NVFP4_IN(d, 128, kCkSweepTab)) d = 0u;
    if (write_codes) {
      uint32_t c0, c1;
      quant16<SUMS>(blk, s_tab[d], r_tab[d], c0, c1, P, R);
      if (NVFP4_IN(2 * b + 1, 2 * B, kCkSweepCodes)) {
        codes32[2 * b] = c0;
        codes32[2 * b + 1] = c1;
      }
    } else if (SUMS && d != d_old) {  // an unchanged Delta re-quantizes to the same codes, P and R
      block_sums(blk, s_tab[d], r_tab[d], P, R);
    }
    if (NVFP4_IN(b, B, kCkSweepScales)) scales[b] = (uint8_t)d;
    if (SUMS) alpha_terms(m_tab[d], P, R, U, num_acc, den_acc);
  };
  uint4 m0, m1;
  uint32_t sm;
  while (ok(b)) {
    fetch(b + 2 * step, m0, m1, sm);
    sweep_block(a0, a1, sa);
    b += step;
    if (!ok(b)) break;
    fetch(b + 2 * step, a0, a1, sa);
    sweep_block(n0, n1, sn);
    b += step;
    if (!ok(b)) break;
    fetch(b + 2 * step, n0, n1, sn);
    sweep_block(m0, m1, sm);
    b += step;
  }
  if (SUMS) {
    u128 num = num_acc.get(), den = den_acc.get();
    block_sum2_u128(num, den, redu);
    if (threadIdx.x == 0) {
      part_out[2 * blockIdx.x] = make_ulonglong2((unsigned long long)num, (unsigned long long)(num >> 64));
      part_out[2 * blockIdx.x + 1] = make_ulonglong2((unsigned long long)den, (unsigned long long)(den >> 64));
    }
  }
}

// ---------------------------------------------------------------------------
// a1-a4, a7 over a group of tensors (max rule and FourOverSix)
// ---------------------------------------------------------------------------
//
// The group's tensors lie end to end in a virtual space of tiles of
// kGroupTile blocks; no tile holds blocks of two tensors.  Both kernels give
// CTA c the same tile range [T*c/G, T*(c+1)/G): the amax kernel walks it
// upwards, the quantize kernel downwards, so each CTA re-reads first what it
// read last (still in L2).  Per tensor: max|W| by atomicMax on a zeroed word,
// alpha = max|W| / (6*448) [SOAR-Q], then the same per-block arithmetic as
// k_quant_max_fos.
static_assert(kGroupTile == kThreads, "one block per thread per tile");
constexpr int kGroupAmaxTiles = 8;  // tiles per step of the amax walk: 16 loads in flight per thread

// The tensor owning `tile` (tile < tile_begin[count]); skips empty tensors.
__device__ __forceinline__ int group_find(const GroupArgs &g, int64_t tile) {
  int lo = 0, hi = g.count;  // tile_begin[lo] <= tile < tile_begin[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (g.tile_begin[mid] <= tile) lo = mid; else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kThreads) k_group_amax(const __grid_constant__ GroupArgs g,
                                                         uint32_t *__restrict__ amax) {
  __shared__ uint32_t red[kWarps];
  pdl_wait();  // W and the zeroed words may come from earlier work on the stream
  pdl_launch_dependents();
  const int64_t T = g.tile_begin[g.count];
  int64_t tile = T * blockIdx.x / gridDim.x;
  const int64_t end = T * (blockIdx.x + 1) / gridDim.x;
  if (tile >= end) return;
  int t = group_find(g, tile);
  uint32_t m = 0u;
  while (tile < end) {
    while (tile >= g.tile_begin[t + 1]) ++t;  // (t + 1 <= count: tile < tile_begin[count])
    if (!NVFP4_IN(t, g.count, kCkGroupTensor)) break;  // (uniform over the CTA)
    const int64_t stop = min(end, g.tile_begin[t + 1]);
    const int64_t nt = min((int64_t)kGroupAmaxTiles, stop - tile);
    const uint4 *W = static_cast<const uint4 *>(g.t[t].W);
    const int64_t H = 2 * g.t[t].B;  // 16-byte units of tensor t
    const int64_t u0 = (tile - g.tile_begin[t]) * (2 * kGroupTile);
    uint4 v[2 * kGroupAmaxTiles];
#pragma unroll
    for (int u = 0; u < 2 * kGroupAmaxTiles; ++u) {
      const int64_t i = u0 + (int64_t)u * kThreads + threadIdx.x;
      v[u] = (u < 2 * nt && i < H) ? __ldg(W + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 2 * kGroupAmaxTiles; ++u) {
      asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(v[u].x));
      asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(v[u].y));
      asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(v[u].z));
      asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(v[u].w));
    }
    tile += nt;
    if (tile >= stop) {  // this CTA's part of tensor t is done
      m &= 0x7FFF7FFFu;
      m = block_max_u32(max(m & 0xFFFFu, m >> 16), red);
      if (threadIdx.x == 0 && m != 0u) atomicMax(amax + t, m);
      m = 0u;
    }
  }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads) k_group_quant(const __grid_constant__ GroupArgs g,
                                                          const uint32_t *__restrict__ amax) {
  __shared__ float s_tab[128], r_tab[128], ev_tab[128];
  __shared__ uint8_t c4_tab[128];
  constexpr bool FOS = MODE == kModeFourOverSix;
  const int64_t T = g.tile_begin[g.count];
  const int64_t lo = T * blockIdx.x / gridDim.x;
  int64_t tile = T * (blockIdx.x + 1) / gridDim.x - 1;  // walks down to lo
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  auto load = [&](int64_t tl, int tt, uint4 &x0, uint4 &x1) {
    const bool known = NVFP4_IN(tt, g.count, kCkGroupTensor);
    const int64_t b = (tl - g.tile_begin[known ? tt : 0]) * kGroupTile + threadIdx.x;
    if (known && b < g.t[tt].B) {
      const uint4 *W = static_cast<const uint4 *>(g.t[tt].W);
      x0 = __ldg(W + 2 * b);
      x1 = __ldg(W + 2 * b + 1);
    } else {
      x0 = z;
      x1 = z;
    }
  };
  int t = 0, tn = 0;  // tensors of the current and of the next tile
  uint4 a0 = z, a1 = z, n0 = z, n1 = z;
  if (tile >= lo) {
    t = tn = group_find(g, tile);
    load(tile, t, a0, a1);
    if (tile - 1 >= lo) {
      while (NVFP4_IN(tn, g.count, kCkGroupTensor) && tile - 1 < g.tile_begin[tn]) --tn;
      load(tile - 1, tn, n0, n1);
    }
  }
  if (threadIdx.x < 128) {  // alpha-independent tables
    const float ev = e4m3_value(threadIdx.x);
    ev_tab[threadIdx.x] = ev;
    if (FOS) c4_tab[threadIdx.x] = (uint8_t)e4m3_code(__fmul_rn(ev, 1.5f));  // [FOS-02]
  }
  pdl_launch_dependents();
  pdl_wait();
  if (blockIdx.x == 0)  // an empty tensor's alpha is 0, as in nvfp4_quantize
    for (int i = threadIdx.x; i < g.count; i += kThreads)
      if (g.t[i].B == 0) *g.t[i].alpha = 0.0f;

  int cur = -1;  // tensor whose tables are loaded
  float alpha = 0.0f, six_a = 0.0f, r6 = 0.0f;
  // The walk, unrolled three times as in k_quant_max_fos: each step looks up the tensor of
  // the tile two steps ahead (searching down from its neighbour's) and issues its loads into
  // the buffer it has just consumed.
  auto fetch = [&](int64_t tl, int from, int &tt, uint4 &y0, uint4 &y1) {
    tt = from;
    y0 = z;
    y1 = z;
    if (tl >= lo) {
      while (NVFP4_IN(tt, g.count, kCkGroupTensor) && tl < g.tile_begin[tt]) --tt;
      load(tl, tt, y0, y1);
    }
  };
  auto quant_tile = [&](const uint4 &x0, const uint4 &x1, int tt) {
    if (tt != cur) {  // uniform over the CTA
      alpha = __fdiv_rn(__uint_as_float(amax[tt] << 16), 2688.0f);  // [SOAR-Q] alpha = max|W| / (6*448)
      six_a = __fmul_rn(alpha, 6.0f);
      r6 = six_a > 0.0f ? __frcp_rn(six_a) : 0.0f;
      __syncthreads();  // the previous tensor's tables are no longer read
      if (threadIdx.x < 128) {
        const float sv = __fmul_rn(alpha, ev_tab[threadIdx.x]);
        s_tab[threadIdx.x] = sv;
        r_tab[threadIdx.x] = sv > 0.0f ? __frcp_rn(sv) : 0.0f;
      }
      __syncthreads();
      cur = tt;
    }
    const GroupTensor &gt = g.t[tt];
    if (threadIdx.x == 0 && tile == g.tile_begin[tt]) *gt.alpha = alpha;
    const int64_t b = (tile - g.tile_begin[tt]) * kGroupTile + threadIdx.x;
    if (b < gt.B) {
      Block16 blk;
      const uint32_t am = unpack16(x0, x1, blk);
      uint32_t d6 = max_rule_code(am, six_a, r6);
      if (!NVFP4_IN(d6, 128, kCkGroupTab)) d6 = 0u;
      uint32_t c0, c1, d = d6;
      float P6, R6;
      quant16<FOS>(blk, s_tab[d6], r_tab[d6], c0, c1, P6, R6);
      if (FOS) {  // [FOS-02] keep scale_m4 iff its dequant error is strictly lower
        uint32_t d4 = c4_tab[d6];
        if (!NVFP4_IN(d4, 128, kCkGroupTab)) d4 = 0u;
        uint32_t e0, e1;
        float P4, R4;
        quant16<true>(blk, s_tab[d4], r_tab[d4], e0, e1, P4, R4);
        const bool use4 = cand_err(s_tab[d4], P4, R4) < cand_err(s_tab[d6], P6, R6);
        d = use4 ? d4 : d6;
        c0 = use4 ? e0 : c0;
        c1 = use4 ? e1 : c1;
      }
      uint32_t *codes32 = reinterpret_cast<uint32_t *>(gt.codes);
      codes32[2 * b] = c0;
      codes32[2 * b + 1] = c1;
      gt.scales[b] = (uint8_t)d;
    }
  };
  int tm = 0;
  uint4 m0, m1;
  while (tile >= lo) {  // (t, tn, tm: the tensors of the tiles in a0/a1, n0/n1, m0/m1)
    if (!NVFP4_IN(t, g.count, kCkGroupTensor)) break;  // (uniform over the CTA)
    fetch(tile - 2, tn, tm, m0, m1);
    quant_tile(a0, a1, t);
    if (--tile < lo || !NVFP4_IN(tn, g.count, kCkGroupTensor)) break;
    fetch(tile - 2, tm, t, a0, a1);
    quant_tile(n0, n1, tn);
    if (--tile < lo || !NVFP4_IN(tm, g.count, kCkGroupTensor)) break;
    fetch(tile - 2, t, tn, n0, n1);
    quant_tile(m0, m1, tm);
    --tile;
  }
}

// ---------------------------------------------------------------------------
// a8: dequantize
// ---------------------------------------------------------------------------

constexpr int kDqUnroll = 2;

__global__ void __launch_bounds__(kThreads) k_dequant(const uint32_t *__restrict__ codes32,
                                                      const uint8_t *__restrict__ scales,
                                                      const float *__restrict__ alpha_p, int64_t H,
                                                      uint4 *__restrict__ out) {
  __shared__ float s_tab[256];
  const float alpha = *alpha_p;
  s_tab[threadIdx.x] = __fmul_rn(alpha, e4m3_value(threadIdx.x));  // kThreads == 256
  __syncthreads();
  // kDqUnroll units per thread per trip, a grid stride apart (each unit's accesses coalesced
  // across the warp as in a plain grid-stride loop), all loads issued before the first use
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t h0 = (int64_t)blockIdx.x * kThreads + threadIdx.x; h0 < H; h0 += kDqUnroll * stride) {
    uint32_t cw[kDqUnroll], sc[kDqUnroll];
#pragma unroll
    for (int u = 0; u < kDqUnroll; ++u) {
      const int64_t h = h0 + u * stride;
      const bool in = h < H && NVFP4_IN(h >> 1, H / 2, kCkDequantIn);
      cw[u] = in ? __ldg(codes32 + h) : 0u;
      sc[u] = in ? __ldg(scales + (h >> 1)) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kDqUnroll; ++u) {
      const int64_t h = h0 + u * stride;
      if (h >= H) break;
      const float s = s_tab[sc[u]];
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 q = e2m1x2_to_f32x2((cw[u] >> (8 * k)) & 0xFFu);  // signed codes
        __nv_bfloat162 p = __floats2bfloat162_rn(__fmul_rn(q.x, s), __fmul_rn(q.y, s));
        o[k] = *reinterpret_cast<uint32_t *>(&p);
      }
      out[h] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// ---------------------------------------------------------------------------
// scale layout for block-scaled tensor-core matrix multiplies
// ---------------------------------------------------------------------------
//
// Linear [rows, kb] E4M3 scales -> tiles of 128 x 4 (zero padded), column
// tiles fastest, scale (r, c) of a tile at byte (r % 32) * 16 + (r / 32) * 4
// + c.  A CTA takes 128 rows x 64 scale columns (16 consecutive tiles, one
// contiguous 8 KiB of output): it reads the rows' 64-byte segments
// (consecutive threads, consecutive bytes) into shared memory and writes the
// tiles' words in order.
constexpr int kSwzCols = 64;  // scale columns per CTA = 16 tiles

__global__ void __launch_bounds__(kThreads) k_swizzle_scales(const uint8_t *__restrict__ scales, int64_t rows,
                                                             int64_t kb, uint32_t *__restrict__ out) {
  __shared__ uint32_t tile[128][kSwzCols / 4 + 1];  // +1 word: rows fall in different banks
  const int64_t ct = (kb + 3) / 4;                  // column tiles per row tile
  const int64_t groups = (ct + 15) / 16;            // CTAs per row tile
  const int64_t rt = blockIdx.x / groups, cg = blockIdx.x % groups;
  const int64_t k0 = cg * kSwzCols;
  if (kb % 4 == 0 && k0 + kSwzCols <= kb) {  // whole 4-byte words, each row 4-byte aligned
    const uint32_t *s32 = reinterpret_cast<const uint32_t *>(scales);
    for (int e = threadIdx.x; e < 128 * (kSwzCols / 4); e += kThreads) {
      const int r = e / (kSwzCols / 4), c = e % (kSwzCols / 4);
      const int64_t row = rt * 128 + r;
      tile[r][c] = row < rows ? __ldg(s32 + (row * kb + k0) / 4 + c) : 0u;
    }
  } else {
    uint8_t *t8 = reinterpret_cast<uint8_t *>(&tile[0][0]);
    for (int e = threadIdx.x; e < 128 * kSwzCols; e += kThreads) {
      const int r = e / kSwzCols, c = e % kSwzCols;
      const int64_t row = rt * 128 + r, k = k0 + c;
      t8[r * (kSwzCols + 4) + c] = (row < rows && k < kb) ? __ldg(scales + row * kb + k) : (uint8_t)0;
    }
  }
  __syncthreads();
  const int64_t ntiles = min((int64_t)16, ct - cg * 16);
  uint32_t *dst = out + (rt * ct + cg * 16) * 128;
  for (int o = threadIdx.x; o < ntiles * 128; o += kThreads) {
    const int t = o >> 7, within = o & 127;
    const int r = (within & 3) * 32 + (within >> 2);
    dst[o] = tile[r][t];
  }
}

// ---------------------------------------------------------------------------
// element-wise format conversions (the quantizer's own rounding)
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(kThreads) k_encode_e2m1(const float *__restrict__ v, int64_t n,
                                                          uint8_t *__restrict__ out) {
  for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += (int64_t)gridDim.x * kThreads) {
    const float x = v[i];
    const uint32_t mag = cvt_e2m1x2(0.0f, fabsf(x)) & 7u;
    out[i] = (uint8_t)(mag | ((__float_as_uint(x) >> 31) << 3));
  }
}

__global__ void __launch_bounds__(kThreads) k_encode_e4m3(const float *__restrict__ v, int64_t n,
                                                          uint8_t *__restrict__ out) {
  for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += (int64_t)gridDim.x * kThreads)
    out[i] = (uint8_t)e4m3_code(v[i]);
}

// ---------------------------------------------------------------------------
// launchers (each returns the launch's own status)
// ---------------------------------------------------------------------------

namespace {
cudaLaunchConfig_t make_cfg(int grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  return cfg;
}
}  // namespace

// Checked build: a kernel that makes one checked test of i against [0, n)
// and accesses nothing (the check mechanism's own test).
__global__ void k_check_selftest(int64_t i, int64_t n) {
  if (NVFP4_IN(i, n, kCkSelfTest)) asm volatile("");
}

cudaError_t launch_check_selftest(int64_t i, int64_t n, cudaStream_t st) {
  k_check_selftest<<<1, 1, 0, st>>>(i, n);
  return cudaGetLastError();
}

cudaError_t check_take_kernels(uint32_t *site) {
#ifdef NVFP4_CHECKED
  return check_take_here(site);
#else
  (void)site;
  return cudaSuccess;
#endif
}

cudaError_t launch_amax_partials(const void *W, int64_t n16, uint32_t *part, int grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = make_cfg(grid, st);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_amax_partials, static_cast<const uint4 *>(W), n16, part);
}

cudaError_t launch_amax_bulk(const void *W, int64_t n16, uint32_t *part, int grid, long first_limit,
                             cudaStream_t st) {
  cudaLaunchConfig_t cfg = make_cfg(grid, st);
  cfg.dynamicSmemBytes = kAmaxBulkSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_amax_bulk, static_cast<const uint4 *>(W), n16, part, first_limit);
}

int amax_bulk_chunks(int64_t n16) { return (int)((n16 * 16 + kAmaxChunk - 1) / kAmaxChunk); }

cudaError_t launch_quant_max_fos(int mode, const void *W, int64_t H, const uint32_t *amax_part, int n_amax,
                                 uint8_t *codes, uint8_t *scales, float *alpha, int grid, int ranged,
                                 cudaStream_t st) {
  cudaLaunchConfig_t cfg = make_cfg(grid, st);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const uint4 *w = static_cast<const uint4 *>(W);
  uint32_t *c = reinterpret_cast<uint32_t *>(codes);
  const int64_t B = H / 2;
  if (mode == kModeFourOverSix)
    return cudaLaunchKernelEx(&cfg, k_quant_max_fos<kModeFourOverSix>, w, B, amax_part, n_amax, c, scales, alpha,
                              ranged);
  return cudaLaunchKernelEx(&cfg, k_quant_max_fos<kModeMax>, w, B, amax_part, n_amax, c, scales, alpha, ranged);
}

cudaError_t launch_cjso_sweep(bool init, bool sums, const void *W, int64_t H, const uint32_t *amax_part,
                              int n_amax, const ulonglong2 *part_in, int n_in, ulonglong2 *part_out,
                              float *alpha_hist, int t, uint8_t *scales, uint8_t *codes, int write_codes,
                              float *alpha_out, int write_alpha, int grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = make_cfg(grid, st);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const uint4 *w = static_cast<const uint4 *>(W);
  uint32_t *c = reinterpret_cast<uint32_t *>(codes);
  const int64_t B = H / 2;
  const int descending = (t & 1) == 0;  // amax reads ascending; sweeps alternate from there
  auto kern = init ? (sums ? k_cjso_sweep<true, true> : k_cjso_sweep<true, false>)
                   : (sums ? k_cjso_sweep<false, true> : k_cjso_sweep<false, false>);
  return cudaLaunchKernelEx(&cfg, kern, w, B, amax_part, n_amax, part_in, n_in, part_out, alpha_hist, t, scales, c,
                            write_codes, alpha_out, write_alpha, descending);
}

cudaError_t launch_group_amax(const GroupArgs &g, uint32_t *amax, int grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = make_cfg(grid, st);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_group_amax, g, amax);
}

cudaError_t launch_group_quant(int mode, const GroupArgs &g, const uint32_t *amax, int grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = make_cfg(grid, st);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (mode == kModeFourOverSix) return cudaLaunchKernelEx(&cfg, k_group_quant<kModeFourOverSix>, g, amax);
  return cudaLaunchKernelEx(&cfg, k_group_quant<kModeMax>, g, amax);
}

cudaError_t prepare_quant_kernels() {
  return cudaFuncSetAttribute(k_amax_bulk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAmaxBulkSmem);
}

cudaError_t launch_dequant(const uint8_t *codes, const uint8_t *scales, const float *alpha, int64_t H, void *out,
                           int grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = make_cfg(grid, st);
  return cudaLaunchKernelEx(&cfg, k_dequant, reinterpret_cast<const uint32_t *>(codes), scales, alpha, H,
                            static_cast<uint4 *>(out));
}

cudaError_t launch_swizzle_scales(const uint8_t *scales, int64_t rows, int64_t kb, uint8_t *out,
                                  cudaStream_t st) {
  const int64_t ct = (kb + 3) / 4;
  const int64_t ctas = (rows + 127) / 128 * ((ct + 15) / 16);
  if (ctas > INT32_MAX) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = make_cfg((int)ctas, st);
  return cudaLaunchKernelEx(&cfg, k_swizzle_scales, scales, rows, kb, reinterpret_cast<uint32_t *>(out));
}

cudaError_t launch_encode_e2m1(const float *v, int64_t n, uint8_t *out, int grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = make_cfg(grid, st);
  return cudaLaunchKernelEx(&cfg, k_encode_e2m1, v, n, out);
}

cudaError_t launch_encode_e4m3(const float *v, int64_t n, uint8_t *out, int grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = make_cfg(grid, st);
  return cudaLaunchKernelEx(&cfg, k_encode_e4m3, v, n, out);
}

int max_active_ctas(int which) {
  int n = 0;
  cudaError_t e = cudaSuccess;
  switch (which) {
    case kKernAmax: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_amax_bulk, kThreads, kAmaxBulkSmem); break;
    case kKernQuantMax: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_quant_max_fos<kModeMax>, kThreads, 0); break;
    case kKernQuantFos: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_quant_max_fos<kModeFourOverSix>, kThreads, 0); break;
    case kKernCjso: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_cjso_sweep<false, true>, kThreads, 0); break;
    case kKernAmaxLdg: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_amax_partials, kThreads, 0); break;
    case kKernGroupAmax: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_group_amax, kThreads, 0); break;
    case kKernGroupQuantMax:
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_group_quant<kModeMax>, kThreads, 0);
      break;
    case kKernGroupQuantFos:
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_group_quant<kModeFourOverSix>, kThreads, 0);
      break;
    default: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_dequant, kThreads, 0); break;
  }
  return (e == cudaSuccess && n > 0) ? n : 1;
}

}  // namespace nvfp4
