// nvfp4_decoupled.cu -- the decoupled quantization / dequantization scale
// search of [SOAR-DEC], as an event-driven scan over the 101 candidates.
//
// Citation keys (page title, part of the page):
//   [SOAR-Q]   "SOAR: Scale Optimization for Accurate Reconstruction in NVFP4
//              Quantization": NVFP4 quantizer equation (piecewise FP4
//              rounding of X / (alpha * Delta)).
//   [SOAR-DEC] same page: decoupled objective (Delta^q real, Delta^d FP8)
//              and its search: Delta^q = Delta^d0 * {0.50, 0.51, ..., 1.50},
//              Delta^d limited to the two nearest E4M3 values, the pair of
//              least reconstruction error kept.
//
// What is computed (per 16-element block, alpha and Delta^d0 from CJSO):
// for k = 0..100, sq_k = fl(alpha * fl(Delta^d0 * m_k)) with m_k =
// fl32((50 + k) / 100); the codes Q_k = e2m1(fl(|x| / sq_k)); P_k = sum |x| q,
// R_k = sum q^2 (exact); for the two E4M3 values lo_k <= fl(Delta^d0 m_k) <=
// hi_k, g = fl(sd * fma(sd, R_k, -2 P_k)) with sd = fl(alpha * Delta^d); the
// first strict minimum of g in the order (k ascending, lo before hi) wins.
//
// How: sq_k grows with k, so every element's code only steps down as k grows,
// at most 4 times over the range (the quotient spans a factor of 3, and four
// E2M1 decision points at most fit in a factor of 3).  Element x crosses the
// decision point b between codes i and i+1 at about kappa = 100 |x| / (b
// s50) - 50 (s50 = fl(alpha Delta^d0)); kappa computed in fp32 is within
// 8e-5 of the true crossing (error bound below), so K = ceil(kappa) is the
// first k with the lower code unless kappa lies within 2^-13 of an integer
// (never seen on the benchmark tensors; such a block takes the plain loop
// below).  Each crossing
// adds its exact change of P and R to a per-thread shared-memory slot at K
// (P as an integer multiple of 2^(-E-1), R as quarters, packed in one word);
// a scan then visits only the k where P, R or the E4M3 bracket changes and
// evaluates the two candidates there.  Between visited k, every candidate's
// g equals the previous one bit for bit, and a later equal g never wins
// under the strict comparison, so the winner is that of the full 202-
// candidate loop.
//
// Error bound of kappa: sq_k = alpha Delta^d0 (50+k)/100 (1 + theta), |theta|
// <= 3 u (u = 2^-24: m_k, the product with Delta^d0, the product with
// alpha), s50 carries one more u, and the code changes where fl(|x|/sq_k)
// crosses b, i.e. where |x|/sq_k is within u b of b (half an fp32 spacing
// around each b is below u b); the true crossing k is 100 V / b (1 + lambda)
// - 50 with V = |x| / s50, |lambda| <= 5u, i.e. within 150 * 5u = 4.47e-5.
// kappa = fl(fl(|x| fl(1/s50)) * fl(100/b) - 50) carries at most 3u relative
// on the product (<= 150) and one rounding of a value <= 100: 3.28e-5.
// Total 7.75e-5, against the 2^-13 = 1.22e-4 margin.
//
// Exactness of P: with 2^E chosen so that max|x| 2^E < 2^15, X = |x| 2^E is
// an integer for every element of magnitude >= 2^(7-E); every element whose
// code is nonzero for some candidate has |x| > s50 / 8, so s50 2^E >= 1025
// makes all of them exact, and P = sum X 2q * 2^(-E-1) is exact (sum < 2^23).
// Blocks outside that range (a block maximum far above its scale) take the
// plain per-candidate loop.
//
// SIMT shape: one block per thread; the crossing loops run a fixed 4 steps
// under predicates and the warp reconverges (__syncwarp) after each phase,
// so the 32 lanes of a warp stay together; every lane of a warp runs the
// same number of block iterations (lanes past the last block idle inside).
#include <cuda_runtime.h>

#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {

constexpr int kDecThreads = 512;
constexpr int kPlainThreads = 256;
constexpr int kDecK = 101;
constexpr int kSlotK = 100;  // k = 1..100 (k = 0 is the start state)
constexpr float kAmbig = 0x1p-13f;

// Dynamic shared memory: per-thread event slots and breakpoint masks, then
// the per-CTA tables.
constexpr size_t kOffMask = (size_t)kSlotK * kDecThreads * 4;
constexpr size_t kOffLohi = kOffMask + (size_t)4 * kDecThreads * 4;
constexpr size_t kOffS2 = kOffLohi + 128 * 4 * 4;
constexpr size_t kOffR = kOffS2 + 256 * 8;
constexpr size_t kOffEv = kOffR + 128 * 4;
constexpr size_t kOffM = kOffEv + 128 * 4;
constexpr size_t kOffH = kOffM + 104 * 4;
constexpr size_t kOffStep = kOffH + 8 * 16;
constexpr size_t kOffQ = kOffStep + 8 * 32;
constexpr size_t kOffLo = kOffQ + 8 * 8;
constexpr size_t kDecSmem = kOffLo + 128 * kDecK;
static_assert(kDecSmem <= 232448, "dynamic shared memory of one CTA");

// fl(100 / b_i) for the E2M1 decision points b_i = 0.25, 0.75, 1.25, 1.75,
// 2.5, 3.5, 5 (b_i lies between magnitude codes i and i + 1), and per
// crossing of b_i: 2(q_{i+1} - q_i) = 1,1,1,1,2,2,4 (as a shift) and
// 4(q_{i+1}^2 - q_i^2) = 1,3,5,7,20,28,80.
__constant__ float kHundredOverB[7] = {(float)(100.0 / 0.25), (float)(100.0 / 0.75), (float)(100.0 / 1.25),
                                       (float)(100.0 / 1.75), (float)(100.0 / 2.5),  (float)(100.0 / 3.5),
                                       (float)(100.0 / 5.0)};
__constant__ uint8_t kStepShift[7] = {0, 0, 0, 0, 1, 1, 2};
__constant__ uint8_t kStepR4[7] = {1, 3, 5, 7, 20, 28, 80};

// Byte lookups (prmt on two words holding an 8-byte table).
__device__ __forceinline__ uint32_t lut8(uint32_t lo4, uint32_t hi4, uint32_t idx) {
  return __byte_perm(lo4, hi4, idx & 7u) & 0xFFu;
}
// 2q and 4q^2 of a magnitude code: {0,1,2,3,4,6,8,12}, {0,1,4,9,16,36,64,144}
__device__ __forceinline__ uint32_t two_q(uint32_t c) { return lut8(0x03020100u, 0x0C080604u, c); }
__device__ __forceinline__ uint32_t four_q2(uint32_t c) { return lut8(0x09040100u, 0x90402410u, c); }

// Dequant scales of a bracket byte's two candidates: (fl(alpha * lo),
// fl(alpha * hi)), hi = lo + 1 when bit 7 is set, else lo.
__device__ __forceinline__ float2 scale_pair(uint32_t lb, float alpha, const float *ev_tab) {
  const uint32_t lo = lb & 0x7Fu, hi = (lb >> 7) && lo < 0x7Eu ? lo + 1u : lo;
  return make_float2(__fmul_rn(alpha, ev_tab[lo]), __fmul_rn(alpha, ev_tab[hi]));
}

// E4M3 codes bracketing dq >= 0: lo = largest with value <= dq, hi = smallest
// with value >= dq (448 above 448), packed as lo | (hi != lo) << 7.
__device__ __forceinline__ uint32_t bracket_byte(float dq, const float *ev_tab) {
  const uint32_t n = e4m3_code(dq);  // nearest
  const float vn = ev_tab[n];
  const uint32_t lo = vn > dq ? n - 1u : n;
  const uint32_t hi = vn < dq ? min(n + 1u, 0x7Eu) : n;
  return lo | ((hi != lo ? 1u : 0u) << 7);
}

// The plain search for blocks outside the exact-integer range: every
// candidate's P, R from its own quotients (the block's scaled f16 image for P).
__device__ __noinline__ int search_plain(const uint4 *__restrict__ W, int64_t b, float alpha, float ev0,
                                         uint32_t d0, const float2 *s2_tab, const float *m_tab,
                                         const uint8_t *lo_tab) {
  Block16 blk;
  const uint32_t am = unpack16(__ldg(W + 2 * b), __ldg(W + 2 * b + 1), blk);
  BlockH16 bh;
  make_h16(blk, am, bh);
  float best_g = __int_as_float(0x7F800000);
  int best_i = 0;
  for (int k = 0; k < kDecK; ++k) {
    const float sq = __fmul_rn(alpha, __fmul_rn(ev0, m_tab[k]));
    const float r = sq > 0.0f ? __frcp_rn(sq) : 0.0f;
    float m2P, R;
    block_sums_h(blk, bh, sq, r, m2P, R);
    const uint32_t lb = lo_tab[d0 * kDecK + k];
    const float2 sp = s2_tab[lb & 0x7Fu];
    const float glo = cand_err_m2p(sp.x, m2P, R);
    const float ghi = cand_err_m2p((lb >> 7) ? sp.y : sp.x, m2P, R);
    if (glo < best_g) { best_g = glo; best_i = 2 * k; }
    if (ghi < best_g) { best_g = ghi; best_i = 2 * k + 1; }
  }
  return best_i;
}

// Signed E2M1 codes of 8 elements with dequant scale s (reciprocal r), one
// word (element 2k in the low nibble of byte k); r = 0 gives sign-only codes.
__device__ __forceinline__ uint32_t quant8(const f32x2 (&x)[4], float s, float r) {
  const f32x2 s2 = pack2(s, s), nr2 = pack2(-r, -r);
  const uint32_t c = encode8(negdiv2_by_scale(x[0], s2, nr2), negdiv2_by_scale(x[1], s2, nr2),
                             negdiv2_by_scale(x[2], s2, nr2), negdiv2_by_scale(x[3], s2, nr2));
  return c ^ 0x88888888u;
}

__device__ __forceinline__ float elem(const Block16 &blk, int j) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(blk.x[j >> 1]));
  return (j & 1) ? hi : lo;
}

__global__ void __launch_bounds__(kDecThreads, 1) k_decoupled(const uint4 *__restrict__ W, int64_t B,
                                                              const float *__restrict__ alpha_hist, int t,
                                                              uint8_t *__restrict__ scales,
                                                              uint32_t *__restrict__ codes32,
                                                              uint32_t *__restrict__ defer_count,
                                                              int64_t *__restrict__ defer_list, int defer_cap) {
  extern __shared__ __align__(16) unsigned char dsm[];
  uint32_t *slot = reinterpret_cast<uint32_t *>(dsm);            // [k - 1][thread]
  uint32_t *mask = reinterpret_cast<uint32_t *>(dsm + kOffMask);  // [word][thread]
  uint32_t *lohi = reinterpret_cast<uint32_t *>(dsm + kOffLohi);  // [Delta^d0 code][word]
  float2 *s2_tab = reinterpret_cast<float2 *>(dsm + kOffS2);      // [bracket byte]: fl(alpha * value) of lo, hi
  float *r_tab = reinterpret_cast<float *>(dsm + kOffR);          // IEEE reciprocal of fl(alpha * value)
  float *ev_tab = reinterpret_cast<float *>(dsm + kOffEv);        // E4M3 values
  float *m_tab = reinterpret_cast<float *>(dsm + kOffM);          // m_k
  float4 *h_rows = reinterpret_cast<float4 *>(dsm + kOffH);       // [code c]: fl(100/b) of c-1 .. c-4
  uint4 *step_rows = reinterpret_cast<uint4 *>(dsm + kOffStep);   // [code c][0 | 1]: 2^(11 + shift) | R4 step
  uint2 *q_rows = reinterpret_cast<uint2 *>(dsm + kOffQ);          // [code c]: 2q, 4q^2
  uint8_t *lo_tab = dsm + kOffLo;                                 // [Delta^d0 code][k] bracket byte
  const int tid = threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * kDecThreads;
  const int64_t warp_first = (int64_t)blockIdx.x * kDecThreads + (tid & ~31);
  int64_t b = (int64_t)blockIdx.x * kDecThreads + tid;
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  uint4 a0 = b < B ? __ldg(W + 2 * b) : z, a1 = b < B ? __ldg(W + 2 * b + 1) : z;

  // alpha-independent set-up, overlapping the previous kernel's tail
  for (int e = tid; e < kSlotK * kDecThreads; e += kDecThreads) slot[e] = 0u;
  for (int e = tid; e < 4 * kDecThreads; e += kDecThreads) mask[e] = 0u;
  if (tid < 128) ev_tab[tid] = e4m3_value(tid);
  if (tid < kDecK) m_tab[tid] = __double2float_rn(__ddiv_rn((double)(50 + tid), 100.0));  // m_k
  if (tid < 8) {  // crossing constants of magnitude code c = tid, steps st = 0..3 -> decision point c-1-st
    float hv[4];
    uint32_t mul[4], r4[4];  // a crossing's slot value is X * mul + r4
#pragma unroll
    for (int st = 0; st < 4; ++st) {
      const int i = tid - 1 - st;
      hv[st] = i >= 0 ? kHundredOverB[i] : 0.0f;
      mul[st] = i >= 0 ? 1u << (11 + kStepShift[i]) : 0u;
      r4[st] = i >= 0 ? kStepR4[i] : 0u;
    }
    h_rows[tid] = make_float4(hv[0], hv[1], hv[2], hv[3]);
    step_rows[2 * tid] = make_uint4(mul[0], mul[1], mul[2], mul[3]);
    step_rows[2 * tid + 1] = make_uint4(r4[0], r4[1], r4[2], r4[3]);
    q_rows[tid] = make_uint2(two_q(tid), four_q2(tid));
  }
  __syncthreads();
  for (int e = tid; e < 128 * kDecK; e += kDecThreads) {
    const int c = e / kDecK, k = e - c * kDecK;
    lo_tab[e] = (uint8_t)bracket_byte(__fmul_rn(ev_tab[c], m_tab[k]), ev_tab);
  }
  __syncthreads();
  if (tid < 128) {  // the k where the bracket (lo, hi) of Delta^d0 = code tid changes, and k = 0
    uint32_t m0 = 1u, m1 = 0u, m2 = 0u, m3 = 0u;
    uint32_t prev = lo_tab[tid * kDecK];
    for (int k = 1; k < kDecK; ++k) {
      const uint32_t cur = lo_tab[tid * kDecK + k];
      const uint32_t bit = cur != prev ? 1u << (k & 31) : 0u;
      m0 |= (k >> 5) == 0 ? bit : 0u;
      m1 |= (k >> 5) == 1 ? bit : 0u;
      m2 |= (k >> 5) == 2 ? bit : 0u;
      m3 |= (k >> 5) == 3 ? bit : 0u;
      prev = cur;
    }
    lohi[tid * 4 + 0] = m0;
    lohi[tid * 4 + 1] = m1;
    lohi[tid * 4 + 2] = m2;
    lohi[tid * 4 + 3] = m3;
  }
  pdl_launch_dependents();
  pdl_wait();
  const float alpha = NVFP4_IN(t, kMaxIters + 1, kCkDecHist) ? alpha_hist[t] : 0.0f;
  if (tid < 256) s2_tab[tid] = scale_pair(tid, alpha, ev_tab);
  if (tid < 128) {
    const float s = __fmul_rn(alpha, ev_tab[tid]);
    r_tab[tid] = s > 0.0f ? __frcp_rn(s) : 0.0f;
  }
  __syncthreads();

  uint32_t *my_slot = slot + tid;
  uint32_t *my_mask = mask + tid;
  uint32_t dn = b < B ? scales[b] : 0u;  // Delta^d0 of the block, fetched one iteration ahead
  // warp-uniform trip count: wf is the warp's first block of the iteration
  for (int64_t wf = warp_first; wf < B; wf += stride, b += stride) {
    const bool live = b < B;
    const int64_t nb = b + stride;
    const uint4 n0 = nb < B ? __ldg(W + 2 * nb) : z, n1 = nb < B ? __ldg(W + 2 * nb + 1) : z;
    const uint32_t d0 = live && NVFP4_IN(dn, 128, kCkDecTab) ? dn : 0u;
    dn = nb < B ? scales[nb] : 0u;
    Block16 blk;
    const uint32_t am = unpack16(a0, a1, blk);
    const float s50 = s2_tab[d0].x;
    const float r50 = r_tab[d0];
    const float ev0 = ev_tab[d0];
    const int e_a = (int)(am >> 7);  // biased exponent of the block maximum
    const int e_c = min(max(e_a, 15), 230);
    const float sc = __uint_as_float((uint32_t)(268 - e_c) << 23);  // 2^E, E = 141 - e_a
    // 0: zero scale (sign-only codes); 1: event scan; 2: plain loop
    int path = !(s50 > 0.0f) ? 0 : ((e_a == e_c && __fmul_rn(s50, sc) >= 1025.0f) ? 1 : 2);
    int best_i = 0;
    if (path == 1) {
      const float nsc = -__uint_as_float((uint32_t)(e_c - 14) << 23);  // -2^-E
      // exact magnitude codes at k = 0 (sq_0 = s50 / 2, its reciprocal 2 / s50)
      const float s0 = __fmul_rn(s50, 0.5f), r0 = __fmul_rn(r50, 2.0f);
      const uint32_t qw[2] = {quant8(*reinterpret_cast<const f32x2(*)[4]>(&blk.x[0]), s0, r0) & 0x77777777u,
                              quant8(*reinterpret_cast<const f32x2(*)[4]>(&blk.x[4]), s0, r0) & 0x77777777u};
      int P = 0, R4 = 0;  // P = P_int * 2^(-E-1), R = R4 / 4
      bool amb = false;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float xa = fabsf(elem(blk, j));
        const uint32_t c = (qw[j >> 3] >> (4 * (j & 7))) & 7u;
        // X = xa 2^E (< 2^15) read off the bits of 2^23 + xa 2^E; exact whenever c > 0,
        // the only case where X is used (a code-0 element adds 0 and has no crossing)
        const uint32_t X = __float_as_uint(__fmaf_rn(xa, sc, 8388608.0f)) - 0x4B000000u;
        const uint2 q = q_rows[c];  // 2q, 4q^2
        P += (int)(X * q.x);
        R4 += (int)q.y;
        const float v = __fmul_rn(xa, r50);
        const float4 hr = h_rows[c];
        const uint4 mr = step_rows[2 * c], rr = step_rows[2 * c + 1];
        const float hv[4] = {hr.x, hr.y, hr.z, hr.w};
        const uint32_t mv[4] = {mr.x, mr.y, mr.z, mr.w}, rv[4] = {rr.x, rr.y, rr.z, rr.w};
        bool go = true;
#pragma unroll
        for (int st = 0; st < 4; ++st) {  // the element's crossings, in k order: decision points c-1, c-2, ...
          go = go && (int)c > st;
          const float kap = __fmaf_rn(v, hv[st], -50.0f);
          // K = ceil(kap) from an addition rounded up onto the integers of
          // [2^23, 2^24) (|kap| < 2^22); at least 1, the crossing lies past k = 0
          const int K = max(__float_as_int(__fadd_ru(kap, 12582912.0f)) - 0x4B400000, 1);
          // within kAmbig of an integer (its nearest, by the same addition
          // rounded to nearest) the crossing may be at either neighbour
          const float rn = __fsub_rn(__fadd_rn(kap, 12582912.0f), 12582912.0f);
          amb = amb || (go && fabsf(__fsub_rn(kap, rn)) < kAmbig);
          go = go && K <= kSlotK;
          if (go && NVFP4_IN(K - 1, kSlotK, kCkDecSlot)) {
            atomicAdd(my_slot + (K - 1) * kDecThreads, X * mv[st] + rv[st]);
            atomicOr(my_mask + (K >> 5) * kDecThreads, 1u << (K & 31));
          }
        }
      }
      if (amb) {  // a crossing too close to an integer k: undo the events, take the plain loop
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t bits = my_mask[w * kDecThreads];
          my_mask[w * kDecThreads] = 0u;
          while (bits) {
            const int k = 32 * w + __ffs(bits) - 1;
            bits &= bits - 1u;
            if (NVFP4_IN(k - 1, kSlotK, kCkDecSlot)) my_slot[(k - 1) * kDecThreads] = 0u;
          }
        }
        path = 2;
      } else {
        // scan the breakpoints in k order.  P and R4 are held as the bits of
        // the floats 2^23 + P and 2^23 + R4 (both < 2^23, so adding 0x4B000000
        // to the integer is exact); the scaling subtracts the 2^23 back.
        const float c23 = __fmul_rn(-8388608.0f, nsc);
        const uint32_t *lm = lohi + d0 * 4;
        const uint8_t *lrow = lo_tab + d0 * kDecK;
        int Pb = P + 0x4B000000, Rb = R4 + 0x4B000000;
        // k = 0 (always a breakpoint: the start state)
        float best_g;
        {
          const float m2P = __fmaf_rn(__int_as_float(Pb), nsc, c23);
          const float R = __fmaf_rn(__int_as_float(Rb), 0.25f, -2097152.0f);
          const float2 sp = s2_tab[lrow[0]];
          const float glo = cand_err_m2p(sp.x, m2P, R);
          const float ghi = cand_err_m2p(sp.y, m2P, R);
          best_g = glo;
          best_i = ghi < glo ? 1 : 0;
          best_g = ghi < glo ? ghi : glo;
        }
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t bits = (lm[w] | my_mask[w * kDecThreads]) & (w == 0 ? ~1u : ~0u);
          my_mask[w * kDecThreads] = 0u;
          while (bits) {
            const int k = 32 * w + __ffs(bits) - 1;
            bits &= bits - 1u;
            if (!NVFP4_IN(k, kDecK, kCkDecTab)) continue;
            const uint32_t ev = my_slot[(k - 1) * kDecThreads];
            my_slot[(k - 1) * kDecThreads] = 0u;
            Pb -= (int)(ev >> 11);
            Rb -= (int)(ev & 0x7FFu);
            const float m2P = __fmaf_rn(__int_as_float(Pb), nsc, c23);
            const float R = __fmaf_rn(__int_as_float(Rb), 0.25f, -2097152.0f);
            const float2 sp = s2_tab[lrow[k]];
            const float glo = cand_err_m2p(sp.x, m2P, R);
            const float ghi = cand_err_m2p(sp.y, m2P, R);
            const bool tlo = glo < best_g;
            best_g = tlo ? glo : best_g;
            best_i = tlo ? 2 * k : best_i;
            const bool thi = ghi < best_g;
            best_g = thi ? ghi : best_g;
            best_i = thi ? 2 * k + 1 : best_i;
          }
        }
      }
    }
    // a block for the plain loop goes to the deferred list (k_decoupled_plain
    // searches it after this kernel), or, when the list is full, is searched here
    bool deferred = false;
    if (path == 2) {
      const uint32_t slot_i = atomicAdd(defer_count, 1u);
      if ((int64_t)slot_i < (int64_t)defer_cap) {
        defer_list[slot_i] = b;
        deferred = true;
      }
    }
    __syncwarp();
    if (path == 2 && !deferred) best_i = search_plain(W, b, alpha, ev0, d0, s2_tab + 128, m_tab, lo_tab);
    __syncwarp();
    const int bk = NVFP4_IN(best_i >> 1, kDecK, kCkDecTab) ? best_i >> 1 : 0;
    const uint32_t lb = lo_tab[d0 * kDecK + bk];
    const uint32_t best_d = path == 0 ? d0 : (lb & 0x7Fu) + ((best_i & 1) ? (lb >> 7) : 0u);
    const float sq = path == 0 ? 0.0f : __fmul_rn(alpha, __fmul_rn(ev0, m_tab[bk]));
    const float rq = sq > 0.0f ? __frcp_rn(sq) : 0.0f;  // zero scale: signs only
    const uint32_t c0 = quant8(*reinterpret_cast<const f32x2(*)[4]>(&blk.x[0]), sq, rq);
    const uint32_t c1 = quant8(*reinterpret_cast<const f32x2(*)[4]>(&blk.x[4]), sq, rq);
    if (live && !deferred) {  // a deferred block keeps Delta^d0 in scales[b] for the second kernel
      codes32[2 * b] = c0;
      codes32[2 * b + 1] = c1;
      scales[b] = (uint8_t)best_d;
    }
    a0 = n0;
    a1 = n1;
  }
}

// The deferred blocks of k_decoupled (a crossing too close to an integer k,
// or a block outside the exact-integer range): the plain search, one block
// per thread.  Launched as a programmatic dependent of k_decoupled; waits for
// it before reading the list.
__global__ void __launch_bounds__(kPlainThreads) k_decoupled_plain(const uint4 *__restrict__ W, int64_t B,
                                                                   const float *__restrict__ alpha_hist, int t,
                                                                   uint8_t *__restrict__ scales,
                                                                   uint32_t *__restrict__ codes32,
                                                                   const uint32_t *__restrict__ defer_count,
                                                                   const int64_t *__restrict__ defer_list,
                                                                   int defer_cap) {
  __shared__ float ev_tab[128], m_tab[kDecK];
  __shared__ float2 s2_tab[128];  // [code c]: fl(alpha * value) of c, c + 1
  __shared__ uint8_t lo_tab[128 * kDecK];
  const int tid = threadIdx.x;
  if (tid < 128) ev_tab[tid] = e4m3_value(tid);
  if (tid < kDecK) m_tab[tid] = __double2float_rn(__ddiv_rn((double)(50 + tid), 100.0));
  __syncthreads();
  for (int e = tid; e < 128 * kDecK; e += kPlainThreads) {
    const int c = e / kDecK, k = e - c * kDecK;
    lo_tab[e] = (uint8_t)bracket_byte(__fmul_rn(ev_tab[c], m_tab[k]), ev_tab);
  }
  pdl_launch_dependents();
  pdl_wait();
  const float alpha = NVFP4_IN(t, kMaxIters + 1, kCkDecHist) ? alpha_hist[t] : 0.0f;
  if (tid < 128) s2_tab[tid] = scale_pair(tid | 0x80u, alpha, ev_tab);
  __syncthreads();
  const int64_t n = min((int64_t)*defer_count, (int64_t)defer_cap);
  for (int64_t i = (int64_t)blockIdx.x * kPlainThreads + tid; i < n; i += (int64_t)gridDim.x * kPlainThreads) {
    const int64_t b = defer_list[i];
    if (!NVFP4_IN(b, B, kCkPlainList)) continue;
    const uint32_t d0 = scales[b];
    if (!NVFP4_IN(d0, 128, kCkPlainTab)) continue;
    const float ev0 = ev_tab[d0];
    const int best_i = search_plain(W, b, alpha, ev0, d0, s2_tab, m_tab, lo_tab);
    const int bk = NVFP4_IN(best_i >> 1, kDecK, kCkPlainTab) ? best_i >> 1 : 0;
    const uint32_t lb = lo_tab[d0 * kDecK + bk];
    const uint32_t best_d = (lb & 0x7Fu) + ((best_i & 1) ? (lb >> 7) : 0u);
    const float sq = __fmul_rn(alpha, __fmul_rn(ev0, m_tab[bk]));
    Block16 blk;
    unpack16(__ldg(W + 2 * b), __ldg(W + 2 * b + 1), blk);
    uint32_t c0, c1;
    float P_unused, R_unused;
    quant16<false>(blk, sq, sq > 0.0f ? __frcp_rn(sq) : 0.0f, c0, c1, P_unused, R_unused);
    codes32[2 * b] = c0;
    codes32[2 * b + 1] = c1;
    scales[b] = (uint8_t)best_d;
  }
}

cudaError_t launch_decoupled(const void *W, int64_t B, const float *alpha_hist, int t, uint8_t *scales,
                             uint8_t *codes, uint32_t *defer_count, int64_t *defer_list, int defer_cap, int sms,
                             cudaStream_t st) {
  const int64_t need = (B + kDecThreads - 1) / kDecThreads;
  const int grid = (int)(need < sms ? (need < 1 ? 1 : need) : sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = kDecSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const uint4 *w = static_cast<const uint4 *>(W);
  uint32_t *c = reinterpret_cast<uint32_t *>(codes);
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_decoupled, w, B, alpha_hist, t, scales, c, defer_count, defer_list,
                                     defer_cap);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3((unsigned)sms);
  cfg.blockDim = dim3(kPlainThreads);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, k_decoupled_plain, w, B, static_cast<const float *>(alpha_hist), t, scales, c,
                            static_cast<const uint32_t *>(defer_count), static_cast<const int64_t *>(defer_list),
                            defer_cap);
}

cudaError_t check_take_decoupled(uint32_t *site) {
#ifdef NVFP4_CHECKED
  return check_take_here(site);
#else
  (void)site;
  return cudaSuccess;
#endif
}

cudaError_t prepare_decoupled_kernel() {
  return cudaFuncSetAttribute(k_decoupled, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDecSmem);
}

}  // namespace nvfp4
