// nvfp4_gemm_tc.cu -- the W4A16 product on the tensor cores, for batches of
// activation vectors: Y[b][r] = sum_c What[r][c] * X[b][c], What the
// dequantized bf16 weights exactly as k_dequant writes them ([SOAR-DQ]).
//
// Citation keys (page title, part of the page):
//   [SOAR-DQ]  "SOAR: Scale Optimization for Accurate Reconstruction in NVFP4
//              Quantization": dequantization equation.
//
// The work is a sequence of T = tiles x K steps: a step is 128 rows of W (one
// tile) times 128 columns (K = ceil(cols / 128) steps per tile).  The grid is
// persistent (at most one CTA per SM) and CTA c takes the contiguous range
// [c T / G, (c+1) T / G) of that sequence, so every CTA gets the same number of
// steps whatever the shape; where a range crosses a tile boundary the CTA
// starts a new segment (a new accumulator).  Each segment's 128 x N partial
// sum goes to a workspace slot and k_gemm_tc_reduce adds the slots of a tile
// in CTA order (a fixed order: the result does not depend on timing).
//
// Roles inside a CTA (768 threads), every hand-off through an mbarrier:
//   - warps 0-15 (512 threads, four per row of the tile) dequantize: per step
//     each reads its 16 code bytes and two scales from a ring slot and writes
//     its 32 bf16 weights into the stage's 128 x 128 A tile (K-major, 128-byte
//     swizzle);
//   - warp 19 (one lane) fills the ring by TMA, one slot per step: the tile's
//     128 x 64 code bytes and the 128 x 16 scale bytes holding the step's 8.
//     Where rows of codes or scales are not whole multiples of 16 bytes, the
//     producer threads instead keep their own bytes in flight with cp.async;
//   - warp 18 (one lane) loads the N x 128 tile of X per step with TMA (the
//     tensor map's 128-byte swizzle gives the layout the MMA reads) once the
//     stage's previous MMAs are done;
//   - warps 16 and 17 (one lane each) issue the eight tcgen05.mma (kind::f16,
//     bf16 x bf16 -> fp32, M = 128, K = 16 each) of every other step into
//     their own accumulator of a pair in tensor memory, and commit them to the
//     stage's mbarrier;
//   - warps 20-23 read each finished pair back with tcgen05.ld and add it in
//     a fixed order (pairs are double-buffered for N <= 128, so this overlaps
//     the next segment).
// Every mbarrier wait is bounded; a CTA that gives up waits (bounded) for its
// own copies and MMAs in flight, writes NaN to its workspace slots and frees
// its tensor memory.
#include <algorithm>
#include <cstring>

#include <cuda.h>
#include <cuda_runtime.h>

#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {

constexpr int kTcM = 128;            // rows per tile (tensor-memory lanes)
constexpr int kTcK = 128;            // columns per step = two 64-column (128-byte) swizzle atoms
constexpr int kTcProducers = 512;    // warps 0-15
constexpr int kTcMmaWarp = 16;      // warps 16-17: one issuing thread each
constexpr int kTcXWarp = 18;
constexpr int kTcCodeWarp = 19;
constexpr int kTcEpiWarp0 = 20;      // warps 20-23
constexpr int kTcThreads = 768;
// ring slot: TMA layout [128 rows][64 code bytes] + [128 rows][16 scale bytes];
// per-thread layout [512 threads][16 code bytes] + [256][4 scale bytes]
constexpr uint32_t kTcSlot = 10240;
constexpr int kTcDynBudget = 227 * 1024 - 2048;  // dynamic shared memory (static arrays take the rest)
// A wait suspends the thread (no spinning) for up to kTcSuspendNs per try,
// and gives up after kTcTries tries (about 2 s): far beyond any legitimate
// wait, which lasts a few microseconds.
constexpr uint32_t kTcSuspendNs = 1000000u;
constexpr int kTcTries = 2000;

// S stages, each a dequantized A tile (32 KiB) and the matching N x 128 tile
// of X (N x 256 bytes), then D ring slots of codes (10 KiB each), within
// 227 KiB.  A stage is freed by the completion of its MMAs.
template <int N>
struct TcCfg {
  static constexpr int S = N <= 32 ? 4 : N <= 128 ? 3 : 2;
  static constexpr uint32_t kAtomA = kTcM * 128u;                  // one 64-column atom of A
  static constexpr uint32_t kAtomB = (uint32_t)N * 128u;           // one 64-column atom of X
  static constexpr uint32_t kStage = 2 * kAtomA + 2 * kAtomB;      // A atoms, then X atoms
  static constexpr uint32_t kRing = S * kStage;                    // offset of the ring
  static constexpr int D0 = (int)((kTcDynBudget - 1024 - (int)kRing) / (int)kTcSlot);
  static constexpr int D = D0 > 12 ? 12 : D0;                       // ring depth (steps in flight)
  static constexpr uint32_t kCols = N <= 32 ? 32u : (uint32_t)N;    // tensor-memory columns per accumulator
  static constexpr int NB = N <= 128 ? 2 : 1;                       // accumulator pairs (buffers)
  static constexpr uint32_t kTmem = (uint32_t)NB * 2u * kCols;      // <= 512
  static constexpr size_t kSmem = 1024 + (size_t)kRing + (size_t)D * kTcSlot;
  static_assert(D >= 3, "ring too shallow");
  static_assert(kSmem <= (size_t)kTcDynBudget, "shared memory");
};

__device__ __forceinline__ uint32_t tc_smem(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

// Byte offset of 16-byte chunk `c` (0..7) of row `r` in a K-major tile with
// the 128-byte swizzle: rows of 128 bytes, chunk index XOR (row mod 8).
__device__ __forceinline__ uint32_t sw128(uint32_t r, uint32_t c) { return r * 128u + ((c ^ (r & 7u)) << 4); }

// Shared-memory matrix descriptor of a K-major, 128-byte-swizzled operand:
// start address >> 4 (bits 0-13), leading byte offset 16 (unused by this
// layout), stride byte offset 1024 (8 rows of 128 bytes, bits 32-45),
// descriptor version 1 (bits 46-47), swizzle mode 128 bytes (bits 61-63).
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), A and
// B bf16 (bits 7-9 = 1, bits 10-12 = 1), both K-major, N >> 3 at bits 17-22,
// M >> 4 at bits 24-28.
__device__ __forceinline__ uint32_t tc_idesc(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kTcM >> 4) << 24);
}

__device__ __forceinline__ void mbar_init(uint32_t mb, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(mb), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t mb) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mb) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t mb, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t mb, uint32_t parity) {
  uint32_t done;
  asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}" : "=r"(done) : "r"(mb), "r"(parity), "n"(kTcSuspendNs) : "memory");
  return done != 0;
}

__device__ __forceinline__ bool mbar_test(uint32_t mb, uint32_t parity) {
  uint32_t done;
  asm volatile("{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}" : "=r"(done) : "r"(mb), "r"(parity) : "memory");
  return done != 0;
}

// Bounded wait for the phase of `parity`; gives up early once another role of
// the CTA has raised `fail`, and raises it itself when the limit (about 2 s)
// runs out.  SLEEP_NS = 0: suspending tries, for the waits on the critical
// path; otherwise the warp sleeps that long between tests, which keeps
// waiting warps that are off the critical path from taking issue slots from
// the dequantizing ones.
template <int SLEEP_NS = 0>
__device__ __forceinline__ bool tc_wait(uint32_t mb, uint32_t parity, volatile int *fail) {
  if (mbar_test(mb, parity)) return true;
  constexpr int kTries = SLEEP_NS ? 2000000000 / SLEEP_NS : kTcTries;
  for (int it = 0; it < kTries; ++it) {
    if (SLEEP_NS) {
      __nanosleep(SLEEP_NS);
      if (mbar_test(mb, parity)) return true;
    } else if (mbar_try(mb, parity)) {
      return true;
    }
    if (*fail) return false;
  }
  *fail = 1;
  return false;
}

// The first wait of a CTA's MMA thread under the test hook: gives up after
// `tries` tries (0: at once) and raises `fail`.
__device__ __forceinline__ bool tc_wait_tries(uint32_t mb, uint32_t parity, volatile int *fail, int tries) {
  for (int it = 0; it < tries; ++it)
    if (mbar_try(mb, parity)) return true;
  *fail = 1;
  return false;
}

// The same wait without the early exit: used after a failure to let this
// CTA's own copies and MMAs in flight finish before it leaves.
__device__ __forceinline__ void tc_drain(uint32_t mb, uint32_t parity) {
  for (int it = 0; it < kTcTries && !mbar_try(mb, parity); ++it) {
  }
}

// Tiles of the work sequence: CTA c covers steps [c T / G, (c+1) T / G); the
// CTA holding step g is floor(((g+1) G - 1) / T).
__host__ __device__ __forceinline__ int64_t tc_first_step(int64_t c, int64_t T, int64_t G) { return c * T / G; }
__host__ __device__ __forceinline__ int64_t tc_cta_of(int64_t g, int64_t T, int64_t G) { return ((g + 1) * G - 1) / T; }

// 16 consecutive fp32 columns of tensor memory, one lane per thread (the
// warp's 32 lanes); the caller waits with tcgen05.wait::ld.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
               "%12, %13, %14, %15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                 "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                 "=r"(r[15])
               : "r"(taddr));
}

// Kernel arguments beside the tensor map.
struct TcArgs {
  const uint8_t *codes;
  const uint8_t *scales;
  const float *alpha;
  int64_t rows, cols;
  int batch;
  int64_t K;      // steps per tile
  int64_t T;      // steps in all
  int maxc;       // workspace slots per tile
  float *ws;      // [tiles][maxc][batch][128] partial sums
  int tma;        // codes and scales by TMA (cmap, smap) rather than per-thread copies
  int first_tries;  // < 0: normal; else the MMA thread's first wait gives up after this many tries (test hook)
};

template <int N>
__global__ void __launch_bounds__(kTcThreads, 1) k_gemm_tc(const __grid_constant__ CUtensorMap xmap,
                                                           const __grid_constant__ CUtensorMap cmap,
                                                           const __grid_constant__ CUtensorMap smap,
                                                           const __grid_constant__ TcArgs a) {
  using C = TcCfg<N>;
  constexpr int S = C::S, D = C::D;
  extern __shared__ uint8_t dsm[];
  // full[s]: the stage's A tile written (one arrival per producer warp) and its
  // X tile landed (one arrival with the TMA byte count); empty[s]: its MMAs done
  __shared__ __align__(8) uint64_t full[S], empty[S], acc_full[2], acc_empty[2];
  // ring_full[d]: slot d's codes and scales landed (TMA); ring_empty[d]: read by every producer warp
  __shared__ __align__(8) uint64_t ring_full[D], ring_empty[D];
  __shared__ uint32_t tmem_slot;
  __shared__ int fail;
  __shared__ float s_tab[256];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t raw = tc_smem(dsm);
  const uint32_t base = (raw + 1023u) & ~1023u;  // swizzle atoms need 1024-byte alignment
  uint8_t *gbase = dsm + (base - raw);
  uint8_t *ring = gbase + C::kRing;
  const int64_t G = gridDim.x;
  const int64_t g0 = tc_first_step(blockIdx.x, a.T, G), g1 = tc_first_step(blockIdx.x + 1, a.T, G);
  const int n = (int)(g1 - g0);  // >= 1: the host launches at most T CTAs
  const int64_t t_first = g0 / a.K;
  const int nseg = (int)((g1 - 1) / a.K - t_first + 1);
  volatile int *vfail = &fail;

  if (tid < 256) s_tab[tid] = __fmul_rn(*a.alpha, e4m3_value(tid));
  if (tid == 0) fail = 0;
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tc_smem(&tmem_slot)),
                 "r"(C::kTmem));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == kTcMmaWarp * 32) {
    for (int s = 0; s < S; ++s) {
      mbar_init(tc_smem(&full[s]), kTcProducers / 32 + 1);
      mbar_init(tc_smem(&empty[s]), 1);
    }
    for (int d = 0; d < D; ++d) {
      mbar_init(tc_smem(&ring_full[d]), 1);
      mbar_init(tc_smem(&ring_empty[d]), kTcProducers / 32);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tc_smem(&acc_full[b]), 2);   // one arrival per issuing thread
      mbar_init(tc_smem(&acc_empty[b]), 4);  // one per epilogue warp
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }

  // ---- producers: this thread's row and 32-column quarter of every step
  const int trow = tid >> 2, quar = tid & 3;
  const int64_t cb = a.cols / 16;  // scale bytes per row
  const bool vec = (a.cols % 64) == 0 && (reinterpret_cast<uintptr_t>(a.codes) % 16) == 0 &&
                   (reinterpret_cast<uintptr_t>(a.scales) % 4) == 0;
  // step (tile t, column step ks) for this thread into ring slot `slot`: its
  // two blocks' codes, and for an even quarter the scales of both quarters
  auto fetch = [&](int64_t t, int64_t ks, int slot) {
    uint8_t *sl = ring + (uint32_t)slot * kTcSlot;
    uint8_t *dc = sl + tid * 16, *ds = sl + 8192 + (tid >> 1) * 4;
    const int64_t row = t * kTcM + trow;
    const int64_t col0 = ks * kTcK + 32 * quar;
    if (vec && row < a.rows && col0 < a.cols) {  // whole blocks, 16-byte aligned codes, 4-byte aligned scales
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc_smem(dc)),
                   "l"(a.codes + row * (a.cols / 2) + col0 / 2) : "memory");
      if ((quar & 1) == 0)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(tc_smem(ds)), "l"(a.scales + row * cb + col0 / 16)
                     : "memory");
      return;
    }
    uint32_t w[4] = {0u, 0u, 0u, 0u}, sc = 0u;  // zero codes: zero weights
    if (row < a.rows) {
      const uint2 *crow = reinterpret_cast<const uint2 *>(a.codes) + row * cb;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int64_t col = col0 + 16 * j;
        if (col < a.cols) {
          const uint2 v = __ldg(crow + (col >> 4));
          w[2 * j] = v.x;
          w[2 * j + 1] = v.y;
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t col = col0 + 16 * j;
        if ((quar & 1) == 0 && col < a.cols) sc |= (uint32_t)__ldg(a.scales + row * cb + (col >> 4)) << (8 * j);
      }
    }
    *reinterpret_cast<uint4 *>(dc) = make_uint4(w[0], w[1], w[2], w[3]);
    if ((quar & 1) == 0) *reinterpret_cast<uint32_t *>(ds) = sc;
  };
  int64_t ft = g0 / a.K, fks = g0 % a.K;  // the next step to fetch
  auto fetch_next = [&](int slot) {
    fetch(ft, fks, slot);
    if (++fks == a.K) {
      fks = 0;
      ++ft;
    }
  };
  if (warp < kTcProducers / 32 && !a.tma) {
#pragma unroll 1
    for (int i = 0; i < D; ++i) {  // the ring's first D steps (one commit group each)
      if (i < n) fetch_next(i);
      asm volatile("cp.async.commit_group;" ::: "memory");
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t tmem = tmem_slot;

  if (warp < kTcProducers / 32) {
    // ---- dequantize: step i of this CTA goes to stage i % S and ring slot i % D
    // this thread's four 16-byte chunks in a stage: columns 32*quar .., atom
    // quar / 2, chunks 4 (quar % 2) .. 4 (quar % 2) + 3 of row trow
    uint32_t aoff[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) aoff[j] = (uint32_t)(quar >> 1) * C::kAtomA + sw128((uint32_t)trow, 4u * (uint32_t)(quar & 1) + j);
    int64_t pks = g0 % a.K;  // column step of step i
    int st = 0, slot = 0;
    uint32_t eph = 0, rph = 0;  // parities to wait for: empty[st] (from step S on), ring_full[slot]
#pragma unroll 1
    for (int i = 0; i < n; ++i) {
      // (the decision to leave is taken by the whole warp: __syncwarp below needs every lane)
      const bool free_st = i < S || tc_wait(tc_smem(&empty[st]), eph, vfail);
      if (!__all_sync(0xFFFFFFFFu, free_st)) break;
      const uint8_t *sl = ring + (uint32_t)slot * kTcSlot;
      uint4 c;
      uint32_t sc;
      if (a.tma) {  // slot i % D holds step i's [128][64] codes and [128][16] scales (this step's half)
        if (!__all_sync(0xFFFFFFFFu, tc_wait(tc_smem(&ring_full[slot]), rph, vfail))) break;
        c = *reinterpret_cast<const uint4 *>(sl + trow * 64 + quar * 16);
        sc = (quar & 1) == 0 ? *reinterpret_cast<const uint32_t *>(sl + 8192 + trow * 16 + (pks & 1) * 8 + (quar >> 1) * 4)
                             : 0u;
      } else {
        asm volatile("cp.async.wait_group %0;" ::"n"(D - 1) : "memory");  // step i's codes have landed
        c = *reinterpret_cast<const uint4 *>(sl + tid * 16);
        sc = (quar & 1) == 0 ? *reinterpret_cast<const uint32_t *>(sl + 8192 + (tid >> 1) * 4) : 0u;
      }
      sc = __shfl_sync(0xFFFFFFFFu, sc, lane & ~1) >> (16 * (quar & 1));  // this quarter's two scales
      uint8_t *A = gbase + st * C::kStage;
      uint32_t w[8];
      dequant16_bf16(make_uint2(c.x, c.y), s_tab[sc & 0xFFu], w);
      *reinterpret_cast<uint4 *>(A + aoff[0]) = make_uint4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<uint4 *>(A + aoff[1]) = make_uint4(w[4], w[5], w[6], w[7]);
      dequant16_bf16(make_uint2(c.z, c.w), s_tab[(sc >> 8) & 0xFFu], w);
      *reinterpret_cast<uint4 *>(A + aoff[2]) = make_uint4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<uint4 *>(A + aoff[3]) = make_uint4(w[4], w[5], w[6], w[7]);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> tensor-core reads
      __syncwarp();
      if (lane == 0) mbar_arrive(tc_smem(&full[st]));
      // the slot just read (its values are consumed above) takes step i + D
      if (a.tma) {
        if (lane == 0) mbar_arrive(tc_smem(&ring_empty[slot]));
      } else {
        if (i + D < n) fetch_next(slot);
        asm volatile("cp.async.commit_group;" ::: "memory");
      }
      if (++pks == a.K) pks = 0;
      if (++st == S) {  // a round of stages done: from the second on, the next waits the other parity
        st = 0;
        if (i >= S) eph ^= 1u;
      }
      if (++slot == D) {
        slot = 0;
        rph ^= 1u;
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // no copy outlives the CTA
  } else if (warp == kTcMmaWarp || warp == kTcMmaWarp + 1) {
    // ---- MMAs: the thread of warp 16 + p takes the steps i with i % 2 == p
    // into accumulator p of buffer (segment % NB), so the two issue in
    // parallel; the epilogue adds the pair in a fixed order
    if (lane == 0) {
      const int p = warp - kTcMmaWarp;
      const uint32_t idesc = tc_idesc(N);
      // descriptors of stage 0's A and X atoms; stage s and K-slice kk add
      // (s * kStage + atom offset + 32 kk) >> 4 to the start-address field
      const uint64_t ad0 = tc_desc(base), bd0 = tc_desc(base + 2 * C::kAtomA);
      int last = -1;      // this thread's last committed step
      int seg = -1;
      bool mine = false;  // MMAs issued into this segment's accumulator p
      int64_t ks = g0 % a.K;  // column step of step i
#pragma unroll 1
      for (int i = 0; i < n; ++i, ks = ks + 1 == a.K ? 0 : ks + 1) {
        if (i == 0 || ks == 0) {  // a new segment: its buffer must have been read back
          ++seg;
          mine = false;
          if (seg >= C::NB &&
              !tc_wait(tc_smem(&acc_empty[seg % C::NB]), (uint32_t)(((seg - C::NB) / C::NB) & 1), vfail))
            break;
        }
        if ((i & 1) == p) {
          const int st = i % S;
          const bool ready = i == 0 && a.first_tries >= 0
                                 ? tc_wait_tries(tc_smem(&full[st]), 0u, vfail, a.first_tries)
                                 : tc_wait(tc_smem(&full[st]), (uint32_t)((i / S) & 1), vfail);
          if (!ready) break;
          asm volatile("tcgen05.fence::after_thread_sync;");
          const uint64_t so = (uint64_t)((st * C::kStage) >> 4);
          const uint32_t acc_t = tmem + (uint32_t)((seg % C::NB) * 2 + p) * C::kCols;
#pragma unroll
          for (int kk = 0; kk < kTcK / 16; ++kk) {  // 4 K-slices of 16 in each of the two atoms
            const uint64_t ka = (uint64_t)(((kk >> 2) * C::kAtomA + 32u * (kk & 3)) >> 4);
            const uint64_t kb = (uint64_t)(((kk >> 2) * C::kAtomB + 32u * (kk & 3)) >> 4);
            const uint32_t acc = (mine || kk > 0) ? 1u : 0u;
            asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                         "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                         ::"r"(acc_t), "l"(ad0 + so + ka), "l"(bd0 + so + kb), "r"(idesc), "r"(acc));
          }
          asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                       ::"r"(tc_smem(&empty[st])) : "memory");
          mine = true;
          last = i;
        }
        if (ks == a.K - 1 || i == n - 1) {  // the segment's last step: accumulator p is final
          if (mine)
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                         ::"r"(tc_smem(&acc_full[seg % C::NB])) : "memory");
          else  // no step of this segment was this thread's: nothing to wait for
            mbar_arrive(tc_smem(&acc_full[seg % C::NB]));
        }
      }
      // after a failure: let the MMAs already issued finish before the CTA leaves
      if (*vfail && last >= 0) tc_drain(tc_smem(&empty[last % S]), (uint32_t)((last / S) & 1));
    }
    __syncwarp();
  } else if (warp == kTcXWarp) {
    // ---- X by TMA: step i's N x 128 tile into stage i % S once the MMAs of step i - S are done
    if (lane == 0) {
      const uint64_t tmap = reinterpret_cast<uint64_t>(&xmap);
      int64_t xks = g0 % a.K;
      int x_hi = 0;  // steps whose X has been requested: [0, x_hi)
#pragma unroll 1
      for (int i = 0; i < n; ++i, xks = xks + 1 == a.K ? 0 : xks + 1) {
        const int st = i % S;
        if (i >= S && !tc_wait<200>(tc_smem(&empty[st]), (uint32_t)(((i - S) / S) & 1), vfail)) break;
        const uint32_t mb = tc_smem(&full[st]);
        const uint32_t dst = base + st * C::kStage + 2 * C::kAtomA;
        const int c0 = (int)(xks * kTcK);
        mbar_expect_tx(mb, 2 * C::kAtomB);
#pragma unroll
        for (int h = 0; h < 2; ++h)
          asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                       " [%0], [%1, {%2, %3}], [%4];"
                       ::"r"(dst + h * C::kAtomB), "l"(tmap), "r"(c0 + 64 * h), "r"(0), "r"(mb) : "memory");
        x_hi = i + 1;
      }
      // after a failure: let the loads whose completion nothing has seen yet land
      // (a load of step i was seen once the MMAs of step i were done; the
      // phase of a later one may never complete when producers gave up, and
      // then the bounded wait outlasts the copy)
      if (*vfail)
        for (int i = x_hi - S > 0 ? x_hi - S : 0; i < x_hi; ++i)
          tc_drain(tc_smem(&full[i % S]), (uint32_t)((i / S) & 1));
    }
    __syncwarp();
  } else if (warp == kTcCodeWarp) {
    // ---- codes and scales by TMA: step i's 128 x 64 code bytes and the
    // 16-byte-aligned 128 x 16 scale bytes holding its 8 into slot i % D once
    // every producer warp has read step i - D from it
    if (lane == 0 && a.tma) {
      const uint64_t cm = reinterpret_cast<uint64_t>(&cmap), sm = reinterpret_cast<uint64_t>(&smap);
      int64_t t = g0 / a.K, ks = g0 % a.K;
      int r_hi = 0;  // steps requested: [0, r_hi)
#pragma unroll 1
      for (int i = 0; i < n; ++i) {
        const int slot = i % D;
        if (i >= D && !tc_wait<200>(tc_smem(&ring_empty[slot]), (uint32_t)(((i - D) / D) & 1), vfail)) break;
        const uint32_t mb = tc_smem(&ring_full[slot]);
        const uint32_t dst = tc_smem(ring) + (uint32_t)slot * kTcSlot;
        mbar_expect_tx(mb, 8192u + 2048u);
        asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                     " [%0], [%1, {%2, %3}], [%4];"
                     ::"r"(dst), "l"(cm), "r"((int)(ks * 64)), "r"((int)(t * kTcM)), "r"(mb) : "memory");
        asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                     " [%0], [%1, {%2, %3}], [%4];"
                     ::"r"(dst + 8192u), "l"(sm), "r"((int)((ks * 8) & ~15LL)), "r"((int)(t * kTcM)), "r"(mb)
                     : "memory");
        r_hi = i + 1;
        if (++ks == a.K) {
          ks = 0;
          ++t;
        }
      }
      // after a failure: let the loads not yet seen by a producer land
      if (*vfail)
        for (int i = r_hi - D > 0 ? r_hi - D : 0; i < r_hi; ++i)
          tc_drain(tc_smem(&ring_full[i % D]), (uint32_t)((i / D) & 1));
    }
    __syncwarp();
  } else {
    // ---- read back each segment's accumulator pair: warp w takes lanes 32 (w % 4) ..
    const int q = warp & 3;
    const int64_t c = blockIdx.x;
#pragma unroll 1
    for (int k = 0; k < nseg; ++k) {
      const int b = k % C::NB;
      if (!__all_sync(0xFFFFFFFFu, tc_wait<500>(tc_smem(&acc_full[b]), (uint32_t)((k / C::NB) & 1), vfail))) break;
      asm volatile("tcgen05.fence::after_thread_sync;");
      const int64_t t = t_first + k;
      const int64_t s0 = t * a.K > g0 ? t * a.K : g0, s1 = (t + 1) * a.K < g1 ? (t + 1) * a.K : g1;
      // a one-step segment: only the accumulator of that step's parity holds it
      const int only = s1 - s0 == 1 ? (int)((s0 - g0) & 1) : -1;
      const int64_t j = c - tc_cta_of(t * a.K, a.T, G);
      float *dst = a.ws + ((t * a.maxc + j) * a.batch) * kTcM + q * 32 + lane;
      const uint32_t tb = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * 2) * C::kCols;
#pragma unroll 1
      for (int n0 = 0; n0 < N && n0 < a.batch; n0 += 16) {
        uint32_t r0[16], r1[16];
        tc_ld16(tb + (only == 1 ? C::kCols : 0u) + (uint32_t)n0, r0);
        if (only < 0) tc_ld16(tb + C::kCols + (uint32_t)n0, r1);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const float v = only < 0 ? __fadd_rn(__uint_as_float(r0[u]), __uint_as_float(r1[u])) : __uint_as_float(r0[u]);
          if (n0 + u < a.batch) dst[(int64_t)(n0 + u) * kTcM] = v;
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;");
      __syncwarp();
      if (lane == 0) mbar_arrive(tc_smem(&acc_empty[b]));
    }
  }

  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  if (*vfail && warp >= kTcEpiWarp0) {  // report the failure through every slot of this CTA
    const int q = warp & 3;
    for (int k = 0; k < nseg; ++k) {
      const int64_t t = t_first + k;
      const int64_t j = (int64_t)blockIdx.x - tc_cta_of(t * a.K, a.T, G);
      float *dst = a.ws + ((t * a.maxc + j) * a.batch) * kTcM + q * 32 + lane;
      for (int b = 0; b < a.batch; ++b) dst[(int64_t)b * kTcM] = __int_as_float(0x7FC00000);
    }
  }
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmem));
}

// y[b][r] = the workspace slots of r's tile added in CTA order.  A thread
// takes 4 consecutive rows of one tile and batch column (16-byte loads of
// every slot issued together; the additions keep the slot order).
__global__ void __launch_bounds__(256) k_gemm_tc_reduce(const float *__restrict__ ws, int64_t rows, int batch,
                                                         int64_t K, int64_t T, int64_t G, int maxc,
                                                         float *__restrict__ y) {
  const int64_t tiles = (rows + kTcM - 1) / kTcM;
  const int64_t n = (int64_t)batch * tiles * (kTcM / 4);  // groups of 4 rows
  const int64_t slot = (int64_t)batch * kTcM;
  const bool vec_y = (rows % 4) == 0 && (reinterpret_cast<uintptr_t>(y) % 16) == 0;
  for (int64_t g = (int64_t)blockIdx.x * 256 + threadIdx.x; g < n; g += (int64_t)gridDim.x * 256) {
    const int64_t rg = g % (tiles * (kTcM / 4)), b = g / (tiles * (kTcM / 4));
    const int64_t t = rg / (kTcM / 4), r0 = t * kTcM + (rg % (kTcM / 4)) * 4;
    if (r0 >= rows) continue;
    const int cnt = (int)(tc_cta_of((t + 1) * K - 1, T, G) - tc_cta_of(t * K, T, G)) + 1;
    const float4 *p = reinterpret_cast<const float4 *>(ws + ((t * maxc) * batch + b) * kTcM + (r0 - t * kTcM));
    const int64_t s4 = slot / 4;
    const float4 z = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    const float4 v0 = p[0], v1 = cnt > 1 ? p[s4] : z, v2 = cnt > 2 ? p[2 * s4] : z, v3 = cnt > 3 ? p[3 * s4] : z;
    float4 acc = v0;
    auto add = [](float4 &x, const float4 &u) {
      x.x = __fadd_rn(x.x, u.x);
      x.y = __fadd_rn(x.y, u.y);
      x.z = __fadd_rn(x.z, u.z);
      x.w = __fadd_rn(x.w, u.w);
    };
    if (cnt > 1) add(acc, v1);
    if (cnt > 2) add(acc, v2);
    if (cnt > 3) add(acc, v3);
    for (int j = 4; j < cnt; ++j) add(acc, p[j * s4]);
    float *o = y + b * rows + r0;
    if (vec_y && r0 + 4 <= rows) {
      *reinterpret_cast<float4 *>(o) = acc;
    } else {
      const float w[4] = {acc.x, acc.y, acc.z, acc.w};
      for (int u = 0; u < 4 && r0 + u < rows; ++u) o[u] = w[u];
    }
  }
}

namespace {

// cuTensorMapEncodeTiled, reached through the runtime's driver entry point
// (the library does not link the driver library itself).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

template <int N>
cudaError_t tc_launch(const CUtensorMap &m, const CUtensorMap &cm, const CUtensorMap &sm, const TcArgs &a, int grid,
                      cudaStream_t st) {
  k_gemm_tc<N><<<grid, kTcThreads, TcCfg<N>::kSmem, st>>>(m, cm, sm, a);
  return cudaGetLastError();
}

// A 2-D uint8 tensor map [rows, width] (row stride = width bytes) with
// boxes of box_w bytes x 128 rows, no swizzle, zeros outside.
bool tc_bytes_map(CUtensorMap *m, const void *p, int64_t rows, int64_t width, uint32_t box_w) {
  const cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)width};
  const cuuint32_t box[2] = {box_w, (cuuint32_t)kTcM};
  const cuuint32_t es[2] = {1u, 1u};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(p), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct TcPlan {
  int64_t tiles, K, T, G;
  int maxc;
};

TcPlan tc_plan(int64_t rows, int64_t cols, int sms) {
  TcPlan p;
  p.tiles = (rows + kTcM - 1) / kTcM;
  p.K = (cols + kTcK - 1) / kTcK;
  p.T = p.tiles * p.K;
  p.G = std::min<int64_t>(p.T, sms);
  // K consecutive steps meet at most (K - 1) / (shortest range) + 2 CTA ranges
  const int64_t shortest = std::max<int64_t>(1, p.T / p.G);
  p.maxc = (int)std::min<int64_t>(p.G, (p.K - 1) / shortest + 2);
  return p;
}

}  // namespace

int gemm_tc_tile_n(int batch) { return batch <= 16 ? 16 : batch <= 32 ? 32 : batch <= 64 ? 64 : batch <= 128 ? 128 : 256; }

size_t gemm_tc_workspace_bytes(int64_t rows, int64_t cols, int batch, int sms) {
  const TcPlan p = tc_plan(rows, cols, sms);
  return sizeof(float) * (size_t)(p.tiles * p.maxc) * (size_t)batch * kTcM;
}

cudaError_t launch_gemm_tc(const uint8_t *codes, const uint8_t *scales, const float *alpha, int64_t rows,
                           int64_t cols, const void *x, int batch, int sms, float *ws, float *y, int first_tries,
                           cudaStream_t st) {
  if (!g_encode) return cudaErrorInitializationError;
  const TcPlan p = tc_plan(rows, cols, sms);
  const int n = gemm_tc_tile_n(batch);
  // X [batch, cols] bf16, boxes of 64 columns x n rows (rows past the batch
  // and columns past the end read as zeros), 128-byte swizzle
  CUtensorMap m;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)batch};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64u, (cuuint32_t)n};
  const cuuint32_t es[2] = {1u, 1u};
  if (g_encode(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(x), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // codes [rows, cols/2] and scales [rows, cols/16] by TMA when their rows
  // are whole multiples of 16 bytes (cols % 256 == 0) and they start 16-byte
  // aligned; otherwise each producer thread copies its own bytes
  CUtensorMap cm, sm;
  memset(&cm, 0, sizeof(cm));
  memset(&sm, 0, sizeof(sm));
  const bool tma = cols % 256 == 0 && rows < (int64_t(1) << 31) && reinterpret_cast<uintptr_t>(codes) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(scales) % 16 == 0 && tc_bytes_map(&cm, codes, rows, cols / 2, 64u) &&
                   tc_bytes_map(&sm, scales, rows, cols / 16, 16u);
  const TcArgs a = {codes, scales, alpha, rows, cols, batch, p.K, p.T, p.maxc, ws, tma ? 1 : 0, first_tries};
  const int grid = (int)p.G;
  cudaError_t e;
  switch (n) {
    case 16: e = tc_launch<16>(m, cm, sm, a, grid, st); break;
    case 32: e = tc_launch<32>(m, cm, sm, a, grid, st); break;
    case 64: e = tc_launch<64>(m, cm, sm, a, grid, st); break;
    case 128: e = tc_launch<128>(m, cm, sm, a, grid, st); break;
    default: e = tc_launch<256>(m, cm, sm, a, grid, st); break;
  }
  return e;
}

cudaError_t launch_gemm_tc_reduce(const float *ws, int64_t rows, int64_t cols, int batch, int sms, float *y,
                                  int grid, cudaStream_t st) {
  const TcPlan p = tc_plan(rows, cols, sms);
  k_gemm_tc_reduce<<<grid, 256, 0, st>>>(ws, rows, batch, p.K, p.T, p.G, p.maxc, y);
  return cudaGetLastError();
}

cudaError_t prepare_gemm_tc_kernels() {
  if (!g_encode) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorSymbolNotFound;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  cudaError_t e = cudaFuncSetAttribute(k_gemm_tc<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TcCfg<16>::kSmem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_tc<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TcCfg<32>::kSmem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_tc<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TcCfg<64>::kSmem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_tc<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TcCfg<128>::kSmem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_tc<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TcCfg<256>::kSmem);
  return e;
}

}  // namespace nvfp4
