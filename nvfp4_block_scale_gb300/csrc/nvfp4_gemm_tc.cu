// nvfp4_gemm_tc.cu -- the W4A16 product on the tensor cores, for batches of
// activation vectors: Y[b][r] = sum_c What[r][c] * X[b][c], What the
// dequantized bf16 weights exactly as k_dequant writes them ([SOAR-DQ]).
//
// Citation keys (page title, part of the page):
//   [SOAR-DQ]  "SOAR: Scale Optimization for Accurate Reconstruction in NVFP4
//              Quantization": dequantization equation.
//
// One CTA computes a 128-row x N tile of Y^T (N = the batch rounded up to 16)
// over a range of K (split-K: partial sums go to a workspace and a second
// kernel adds them in a fixed order).  Per K step of 64 columns:
//   - the 128 threads dequantize one row of W each (4 blocks: 32 code bytes,
//     4 scales) into a 128 x 64 bf16 tile and copy the N x 64 bf16 tile of X,
//     both in shared memory in the K-major 128-byte-swizzled layout;
//   - one thread issues four tcgen05.mma (kind::f16, bf16 x bf16 -> fp32,
//     M = 128, K = 16 each) accumulating into tensor memory, and commits them
//     to the stage's mbarrier, so the next step's dequantization overlaps them
//     (two stages).
// The 128 x N fp32 accumulator lives in tensor memory (one lane per row), is
// read back with tcgen05.ld and written to the partial sums.  Every mbarrier
// wait is bounded; a CTA that gives up writes NaN partials.
#include <algorithm>

#include <cuda_runtime.h>

#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {

constexpr int kTcThreads = 256;  // two threads per row of the tile; warps 0-3 read the accumulator back
constexpr int kTcM = 128;
constexpr int kTcK = 128;        // columns per step = two 64-column (128-byte) swizzle atoms
constexpr int kTcMaxN = 256;
// shared-memory stages of the A and X tiles: three while they fit twice per SM
template <int N>
struct TcStages {
  static constexpr int value = N <= 64 ? 3 : 2;
};
constexpr long kTcSpin = 1L << 24;

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

__device__ __forceinline__ bool tc_wait(uint32_t mbar, uint32_t parity) {
  uint32_t done = 0;
  for (long it = 0; !done && it < kTcSpin; ++it)
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}" : "=r"(done) : "r"(mbar), "r"(parity) : "memory");
  return done != 0;
}

struct TcCodes {  // this thread's 4 blocks of W for one step (32 code bytes and 4 scales)
  uint4 c[2];
  uint32_t s;
};

template <int N>
__global__ void __launch_bounds__(kTcThreads, 1) k_gemm_tc(const uint8_t *__restrict__ codes,
                                                           const uint8_t *__restrict__ scales,
                                                           const float *__restrict__ alpha_p, int64_t rows,
                                                           int64_t cols, const uint4 *__restrict__ x, int batch,
                                                           int64_t kspan, float *__restrict__ out) {
  constexpr int S = TcStages<N>::value;
  constexpr uint32_t kAtomA = kTcM * 128u, kAtomB = (uint32_t)N * 128u;  // one 64-column swizzle atom
  constexpr uint32_t kA = 2 * kAtomA, kStage = kA + 2 * kAtomB;
  constexpr uint32_t kCols = N <= 32 ? 32u : N <= 64 ? 64u : N <= 128 ? 128u : 256u;  // TMEM columns
  extern __shared__ uint8_t dsm[];
  __shared__ __align__(8) uint64_t mbar[S];
  __shared__ uint32_t tmem_slot;
  __shared__ float s_tab[256];
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t raw = tc_smem(dsm);
  const uint32_t base = (raw + 1023u) & ~1023u;  // swizzle atoms need 1024-byte alignment
  uint8_t *gbase = dsm + (base - raw);
  const int64_t row0 = (int64_t)blockIdx.x * kTcM;
  const int64_t k0 = (int64_t)blockIdx.y * kspan;
  const int64_t k1 = min(cols, k0 + kspan);
  const int nsteps = (int)((k1 - k0 + kTcK - 1) / kTcK);  // >= 1: the host sizes the splits so
  // adjacent threads take the two 64-column halves (swizzle atoms) of one row
  const int trow = tid >> 1, half = tid & 1;
  const int64_t row = row0 + trow;
  const int64_t bpr = cols / 16;  // blocks per row
  const bool vec = (cols % 64) == 0 && (reinterpret_cast<uintptr_t>(codes) % 16) == 0 &&
                   (reinterpret_cast<uintptr_t>(scales) % 4) == 0;  // 4 blocks = two aligned 16-byte loads
  const uint2 *crow = reinterpret_cast<const uint2 *>(codes) + (row < rows ? row : 0) * bpr;
  const uint8_t *srow = scales + (row < rows ? row : 0) * bpr;
  auto load_codes = [&](int step, TcCodes &t) {
    const int64_t col0 = k0 + (int64_t)step * kTcK + 64 * half;
    const int64_t b0 = col0 >> 4;
    if (vec && step < nsteps && row < rows && col0 + 48 < k1) {  // all 4 blocks inside the range
      t.c[0] = __ldg(reinterpret_cast<const uint4 *>(crow + b0));
      t.c[1] = __ldg(reinterpret_cast<const uint4 *>(crow + b0) + 1);
      t.s = __ldg(reinterpret_cast<const uint32_t *>(srow + b0));
      return;
    }
    uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u}, sc = 0u;  // zero code and scale: zero weights
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t col = col0 + 16 * j;
      if (step < nsteps && row < rows && col < k1) {
        const uint2 v = __ldg(crow + (col >> 4));
        w[2 * j] = v.x;
        w[2 * j + 1] = v.y;
        sc |= (uint32_t)__ldg(srow + (col >> 4)) << (8 * j);
      }
    }
    t.c[0] = make_uint4(w[0], w[1], w[2], w[3]);
    t.c[1] = make_uint4(w[4], w[5], w[6], w[7]);
    t.s = sc;
  };
  // the step's N x 128 tile of X into stage `st` (asynchronous 16-byte copies)
  auto issue_x = [&](int step, int st) {
    const int64_t c0 = k0 + (int64_t)step * kTcK;
    uint8_t *B = gbase + st * kStage + kA;
    for (int u = tid; u < N * 16; u += kTcThreads) {
      const int b = u >> 4, c = u & 15;
      const int64_t col = c0 + 8 * c;
      uint8_t *dst = B + (c >> 3) * kAtomB + sw128((uint32_t)b, (uint32_t)(c & 7));
      if (b < batch && col < k1)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(tc_smem(dst)),
                     "l"(x + ((int64_t)b * cols + col) / 8) : "memory");
      else
        *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  TcCodes cur, nx1, nx2;
  load_codes(0, cur);
  load_codes(1, nx1);
  const float alpha = *alpha_p;
  s_tab[tid] = __fmul_rn(alpha, e4m3_value(tid));  // kTcThreads == 256: every code
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tc_smem(&tmem_slot)),
                 "r"(kCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int st = 0; st < S; ++st) asm volatile("mbarrier.init.shared.b64 [%0], 1;" ::"r"(tc_smem(&mbar[st])));
    asm volatile("fence.mbarrier_init.release.cluster;");
  }
  issue_x(0, 0);
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t tmem = tmem_slot;
  const uint32_t idesc = tc_idesc(N);
  bool ok = true;  // uniform over the CTA
  for (int s = 0; s < nsteps; ++s) {
    const int st = s % S;
    const int sn = (s + 1) % S;
    if (s + 1 >= S) {  // stage sn was last read by the MMAs of step s + 1 - S
      const int prev = s + 1 - S;
      const bool arrived = tc_wait(tc_smem(&mbar[sn]), (uint32_t)((prev / S) & 1));
      if (!__syncthreads_and(arrived)) {
        ok = false;
        break;
      }
    }
    uint8_t *A = gbase + st * kStage + half * kAtomA;  // this thread's atom: columns 64*half ..
    const uint32_t cw[8] = {cur.c[0].x, cur.c[0].y, cur.c[0].z, cur.c[0].w,
                            cur.c[1].x, cur.c[1].y, cur.c[1].z, cur.c[1].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t w[8];
      dequant16_bf16(make_uint2(cw[2 * j], cw[2 * j + 1]), s_tab[(cur.s >> (8 * j)) & 0xFFu], w);
      *reinterpret_cast<uint4 *>(A + sw128((uint32_t)trow, 2u * j)) = make_uint4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<uint4 *>(A + sw128((uint32_t)trow, 2u * j + 1u)) = make_uint4(w[4], w[5], w[6], w[7]);
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");  // this step's X has landed
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> tensor-core reads
    __syncthreads();
    // the next loads are issued after the proxy fence, which would otherwise wait for them
    if (s + 1 < nsteps) issue_x(s + 1, sn);
    load_codes(s + 2, nx2);
    if (tid == 0) {
      asm volatile("tcgen05.fence::after_thread_sync;");
      const uint32_t a0 = base + st * kStage, b0 = a0 + kA;
#pragma unroll
      for (int kk = 0; kk < kTcK / 16; ++kk) {  // 4 K-slices of 16 in each of the two atoms
        const uint32_t atom = (uint32_t)(kk >> 2), ko = 32u * (uint32_t)(kk & 3);
        const uint64_t ad = tc_desc(a0 + atom * kAtomA + ko), bd = tc_desc(b0 + atom * kAtomB + ko);
        const uint32_t acc = (s > 0 || kk > 0) ? 1u : 0u;
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                     "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                     ::"r"(tmem), "l"(ad), "l"(bd), "r"(idesc), "r"(acc));
      }
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                   ::"r"(tc_smem(&mbar[st])) : "memory");
    }
    cur = nx1;
    nx1 = nx2;
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");  // no copy outlives the CTA
  if (ok) {  // the last commit covers every MMA of this CTA
    const int last = nsteps - 1;
    ok = __syncthreads_and(tc_wait(tc_smem(&mbar[last % S]), (uint32_t)((last / S) & 1)));
  } else {   // give the MMAs already issued their time (bounded), then report NaN
    for (int st = 0; st < S; ++st) tc_wait(tc_smem(&mbar[st]), 0u);
  }
  asm volatile("tcgen05.fence::after_thread_sync;");
  float *dst = out + (int64_t)blockIdx.y * batch * rows;
  const int64_t orow = row0 + tid;  // the row whose accumulator lane this thread reads (warps 0-3)
#pragma unroll 1
  for (int n0 = 0; n0 < N && warp < 4; n0 += 16) {  // warp w reads tensor-memory lanes 32w..32w+31
    uint32_t r[16];
    const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)n0;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
                 "%12, %13, %14, %15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    if (orow < rows) {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (n0 + i < batch) dst[(int64_t)(n0 + i) * rows + orow] = ok ? __uint_as_float(r[i]) : __int_as_float(0x7FC00000);
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols));
}

// y = sum over the splits of the partial products, in split order.
__global__ void __launch_bounds__(256) k_gemm_tc_reduce(const float *__restrict__ part, int splits, int64_t n,
                                                         float *__restrict__ y) {
  for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (int64_t)gridDim.x * 256) {
    float acc = part[i];
    for (int sp = 1; sp < splits; ++sp) acc = __fadd_rn(acc, part[(int64_t)sp * n + i]);
    y[i] = acc;
  }
}

namespace {
template <int N>
size_t tc_smem_bytes() { return TcStages<N>::value * 2 * ((size_t)kTcM * 128 + (size_t)N * 128) + 1024; }

template <int N>
cudaError_t tc_launch(dim3 grid, const uint8_t *codes, const uint8_t *scales, const float *alpha, int64_t rows,
                      int64_t cols, const uint4 *x, int batch, int64_t kspan, float *out, cudaStream_t st) {
  k_gemm_tc<N><<<grid, kTcThreads, tc_smem_bytes<N>(), st>>>(codes, scales, alpha, rows, cols, x, batch, kspan, out);
  return cudaGetLastError();
}
}  // namespace

int gemm_tc_tile_n(int batch) { return batch <= 16 ? 16 : batch <= 32 ? 32 : batch <= 64 ? 64 : batch <= 128 ? 128 : 256; }

// Resident CTAs per SM of the tile width serving `batch`: the smallest of the
// shared-memory, tensor-memory (512 columns), register and thread limits.
int gemm_tc_ctas_per_sm(int batch) {
  const int n = gemm_tc_tile_n(batch);
  size_t smem = 0;
  cudaFuncAttributes fa = {};
  cudaError_t e;
  switch (n) {
    case 16: smem = tc_smem_bytes<16>(); e = cudaFuncGetAttributes(&fa, k_gemm_tc<16>); break;
    case 32: smem = tc_smem_bytes<32>(); e = cudaFuncGetAttributes(&fa, k_gemm_tc<32>); break;
    case 64: smem = tc_smem_bytes<64>(); e = cudaFuncGetAttributes(&fa, k_gemm_tc<64>); break;
    case 128: smem = tc_smem_bytes<128>(); e = cudaFuncGetAttributes(&fa, k_gemm_tc<128>); break;
    default: smem = tc_smem_bytes<256>(); e = cudaFuncGetAttributes(&fa, k_gemm_tc<256>); break;
  }
  int dev = 0, sm_smem = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (e != cudaSuccess) return 1;
  const size_t per_cta = smem + fa.sharedSizeBytes + 1024;  // + the per-CTA reservation
  int c = (int)(sm_smem / per_cta);
  c = std::min(c, 512 / (n <= 32 ? 32 : n));
  if (fa.numRegs > 0) c = std::min(c, 65536 / (fa.numRegs * kTcThreads));
  c = std::min(c, 2048 / kTcThreads);
  return c < 1 ? 1 : c;
}

cudaError_t launch_gemm_tc(const uint8_t *codes, const uint8_t *scales, const float *alpha, int64_t rows,
                           int64_t cols, const void *x, int batch, int64_t kspan, int splits, float *out,
                           cudaStream_t st) {
  const dim3 grid((unsigned)((rows + kTcM - 1) / kTcM), (unsigned)splits);
  const uint4 *xv = static_cast<const uint4 *>(x);
  switch (gemm_tc_tile_n(batch)) {
    case 16: return tc_launch<16>(grid, codes, scales, alpha, rows, cols, xv, batch, kspan, out, st);
    case 32: return tc_launch<32>(grid, codes, scales, alpha, rows, cols, xv, batch, kspan, out, st);
    case 64: return tc_launch<64>(grid, codes, scales, alpha, rows, cols, xv, batch, kspan, out, st);
    case 128: return tc_launch<128>(grid, codes, scales, alpha, rows, cols, xv, batch, kspan, out, st);
    default: return tc_launch<256>(grid, codes, scales, alpha, rows, cols, xv, batch, kspan, out, st);
  }
}

cudaError_t launch_gemm_tc_reduce(const float *part, int splits, int64_t n, float *y, int grid, cudaStream_t st) {
  k_gemm_tc_reduce<<<grid, 256, 0, st>>>(part, splits, n, y);
  return cudaGetLastError();
}

cudaError_t prepare_gemm_tc_kernels() {
  cudaError_t e = cudaFuncSetAttribute(k_gemm_tc<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc_smem_bytes<16>());
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_tc<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc_smem_bytes<32>());
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_tc<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc_smem_bytes<64>());
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_tc<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc_smem_bytes<128>());
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_tc<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc_smem_bytes<256>());
  return e;
}

}  // namespace nvfp4
