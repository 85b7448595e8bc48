// nvfp4_gemv.cu -- the W4A16 consumer of the quantized weights: y = What x
// for 1..8 bf16 activation vectors, What the dequantized weights exactly as
// k_dequant writes them, bf16(q * fl(alpha * Delta_i)).  [SOAR-DQ] (one
// dequantization for every scale rule: [FOS-02], the kernel is unchanged).
//
// Citation keys (page title, part of the page):
//   [SOAR-DQ]  "SOAR: Scale Optimization for Accurate Reconstruction in NVFP4
//              Quantization": dequantization equation.
//   [FOS-02]   "SOAR 周冠军笔记 07 | 香草小张：NVFP4 量化改进与推测解码实践",
//              section 02 (FourOverSix): the dequantization kernel is unchanged.
//
// Bound: HBM for one vector (0.5625 B of codes and scales per weight, read
// once); each extra vector adds one fused multiply-add per weight.
//
// Work split: a CTA owns kGemvCtaRows consecutive rows (kGemvRows per warp)
// and walks the columns in chunks of kGemvChunk.  A chunk of every activation
// vector is staged in shared memory (double buffered) and shared by the CTA's
// rows; each lane takes one 16-element block per row and half chunk (8 code
// bytes, one scale byte), the next chunk's codes in flight while the current
// one is computed.  Per weight pair: E2M1 pair -> f16x2 (cvt), -> f32,
// times the block's fp32 scale, -> bf16x2 (cvt, RNE), then one mixed
// bf16 x bf16 + fp32 fused multiply-add per vector (the product is exact, so
// every accumulation rounds once).  Each lane sums its blocks in column
// order; the 32 lanes' sums are combined by a fixed butterfly, so results
// are reproducible run to run.
#include <algorithm>

#include <cuda_runtime.h>

#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {

constexpr int kGemvWarps = 8;
constexpr int kGemvRows = 2;                            // rows per warp
constexpr int kGemvCtaRows = kGemvWarps * kGemvRows;    // rows per CTA
constexpr int kGemvChunk = 1024;                        // columns per step
constexpr int kGemvThreads = kGemvWarps * 32;
constexpr int kGemvHalves = kGemvChunk / 512;           // 32 lanes x 16 columns per half chunk

// Codes of one lane for one chunk: per row and half chunk, 8 code bytes and
// the scale byte.
struct GemvLoad {
  uint2 c[kGemvRows][kGemvHalves];
  uint32_t s[kGemvRows][kGemvHalves];
};

__device__ __forceinline__ void gemv_load(GemvLoad &L, const uint2 *__restrict__ codes,
                                          const uint8_t *__restrict__ scales, int64_t row0, int64_t rows,
                                          int64_t cols, int64_t c0, int lane) {
#pragma unroll
  for (int r = 0; r < kGemvRows; ++r)
#pragma unroll
    for (int h = 0; h < kGemvHalves; ++h) {
      const int64_t col = c0 + h * 512 + lane * 16;
      const int64_t row = row0 + r;
      if (row < rows && col < cols) {
        const int64_t blk = (row * cols + col) >> 4;
        L.c[r][h] = __ldg(codes + blk);
        L.s[r][h] = __ldg(scales + blk);
      } else {
        L.c[r][h] = make_uint2(0u, 0u);
        L.s[r][h] = 0u;
      }
    }
}

// acc += sum over the 8 pairs of w * x (bf16 operands, fp32 accumulation).
__device__ __forceinline__ float gemv_dot16(const uint32_t (&w)[8], const uint4 &xa, const uint4 &xb, float acc) {
  const uint32_t x[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
        "mov.b32 {wl, wh}, %1;\n\tmov.b32 {xl, xh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, wl, xl, %0;\n\tfma.rn.f32.bf16 %0, wh, xh, %0;\n\t}"
        : "+f"(acc) : "r"(w[k]), "r"(x[k]));
  }
  return acc;
}

// Stages columns [c0, c0 + kGemvChunk) of the NB activation vectors (bf16,
// row-major [NB, cols]) into xs; columns past `cols` read as zero.
template <int NB>
__device__ __forceinline__ void gemv_stage_x(uint4 (&reg)[(NB * kGemvChunk / 8 + kGemvThreads - 1) / kGemvThreads],
                                             const uint4 *__restrict__ x, int64_t cols, int64_t c0) {
  constexpr int kUnits = NB * kGemvChunk / 8;  // 16-byte units (8 bf16)
#pragma unroll
  for (int i = 0; i < (kUnits + kGemvThreads - 1) / kGemvThreads; ++i) {
    const int u = i * kGemvThreads + threadIdx.x;
    const int b = u / (kGemvChunk / 8), j = u % (kGemvChunk / 8);
    const int64_t col = c0 + 8 * j;
    reg[i] = (u < kUnits && col < cols) ? __ldg(x + (b * cols + col) / 8) : make_uint4(0u, 0u, 0u, 0u);
  }
}

template <int NB>
__device__ __forceinline__ void gemv_store_x(const uint4 (&reg)[(NB * kGemvChunk / 8 + kGemvThreads - 1) / kGemvThreads],
                                             uint4 *xs) {
  constexpr int kUnits = NB * kGemvChunk / 8;
#pragma unroll
  for (int i = 0; i < (kUnits + kGemvThreads - 1) / kGemvThreads; ++i) {
    const int u = i * kGemvThreads + threadIdx.x;
    if (u < kUnits) xs[u] = reg[i];
  }
}

template <int NB>
__global__ void __launch_bounds__(kGemvThreads) k_gemv(const uint2 *__restrict__ codes,
                                                       const uint8_t *__restrict__ scales,
                                                       const float *__restrict__ alpha_p, int64_t rows, int64_t cols,
                                                       const uint4 *__restrict__ x, float *__restrict__ y) {
  constexpr int kXUnits = NB * kGemvChunk / 8;
  constexpr int kXRegs = (kXUnits + kGemvThreads - 1) / kGemvThreads;
  __shared__ float s_tab[256];
  __shared__ uint4 xs[2][kXUnits];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  s_tab[threadIdx.x] = __fmul_rn(*alpha_p, e4m3_value(threadIdx.x));  // kGemvThreads == 256: every code
  const int64_t groups = (rows + kGemvCtaRows - 1) / kGemvCtaRows;
  const int64_t nchunks = (cols + kGemvChunk - 1) / kGemvChunk;
  for (int64_t g = blockIdx.x; g < groups; g += gridDim.x) {
    const int64_t row0 = g * kGemvCtaRows + warp * kGemvRows;
    float acc[kGemvRows][NB];
#pragma unroll
    for (int r = 0; r < kGemvRows; ++r)
#pragma unroll
      for (int b = 0; b < NB; ++b) acc[r][b] = 0.0f;
    GemvLoad cur, nxt;
    uint4 xr[kXRegs];
    gemv_load(cur, codes, scales, row0, rows, cols, 0, lane);
    gemv_stage_x<NB>(xr, x, cols, 0);
    __syncthreads();  // the previous group's last chunk is no longer read (and s_tab is written)
    gemv_store_x<NB>(xr, xs[0]);
    __syncthreads();
    for (int64_t ch = 0; ch < nchunks; ++ch) {
      const int64_t c0 = ch * kGemvChunk;
      const bool more = ch + 1 < nchunks;
      if (more) {
        gemv_load(nxt, codes, scales, row0, rows, cols, c0 + kGemvChunk, lane);
        gemv_stage_x<NB>(xr, x, cols, c0 + kGemvChunk);
      }
      const uint4 *xb = xs[ch & 1];
#pragma unroll
      for (int h = 0; h < kGemvHalves; ++h) {
        const int j = (h * 512 + lane * 16) / 8;  // this lane's 16 columns = units j, j + 1 of each vector
#pragma unroll
        for (int r = 0; r < kGemvRows; ++r) {
          uint32_t w[8];
          dequant16_bf16(cur.c[r][h], s_tab[cur.s[r][h]], w);
#pragma unroll
          for (int b = 0; b < NB; ++b)
            acc[r][b] = gemv_dot16(w, xb[b * (kGemvChunk / 8) + j], xb[b * (kGemvChunk / 8) + j + 1], acc[r][b]);
        }
      }
      if (more) {
        gemv_store_x<NB>(xr, xs[(ch + 1) & 1]);  // that buffer was last read in chunk ch - 1
        cur = nxt;
      }
      __syncthreads();
    }
#pragma unroll
    for (int r = 0; r < kGemvRows; ++r)
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        float v = acc[r][b];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
        if (lane == 0 && row0 + r < rows) y[b * rows + row0 + r] = v;
      }
  }
}

// Resident form, used when the activations fit in shared memory
// (NB * cols * 2 bytes <= kGemvResidentBytes): every CTA stages all of x
// once, then each warp takes whole rows (row = CTA * 16 + warp, striding by
// the grid) with no barrier between rows; a lane takes blocks lane,
// lane + 32, ..., kGemvUnroll of them in flight at a time.
constexpr int kGemvResWarps = 16;
constexpr int kGemvUnroll = 4;
constexpr int kGemvResidentBytes = 112 * 1024;

template <int NB>
__global__ void __launch_bounds__(kGemvResWarps * 32) k_gemv_resident(const uint2 *__restrict__ codes,
                                                                      const uint8_t *__restrict__ scales,
                                                                      const float *__restrict__ alpha_p, int64_t rows,
                                                                      int64_t cols, const uint4 *__restrict__ x,
                                                                      float *__restrict__ y) {
  extern __shared__ uint4 xs_all[];  // [NB][cols / 8]
  __shared__ float s_tab[256];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t units = cols / 8;
  for (int64_t u = threadIdx.x; u < NB * units; u += kGemvResWarps * 32) xs_all[u] = __ldg(x + u);
  if (threadIdx.x < 256) s_tab[threadIdx.x] = __fmul_rn(*alpha_p, e4m3_value(threadIdx.x));
  __syncthreads();
  const int64_t nblk = cols / 16;
  for (int64_t row = (int64_t)blockIdx.x * kGemvResWarps + warp; row < rows;
       row += (int64_t)gridDim.x * kGemvResWarps) {
    float acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.0f;
    const uint2 *crow = codes + row * nblk;
    const uint8_t *srow = scales + row * nblk;
    for (int64_t j0 = lane; j0 < nblk; j0 += 32 * kGemvUnroll) {
      uint2 c[kGemvUnroll];
      uint32_t sc[kGemvUnroll];
#pragma unroll
      for (int u = 0; u < kGemvUnroll; ++u) {
        const int64_t j = j0 + 32 * u;
        c[u] = j < nblk ? __ldg(crow + j) : make_uint2(0u, 0u);
        sc[u] = j < nblk ? __ldg(srow + j) : 0u;
      }
#pragma unroll
      for (int u = 0; u < kGemvUnroll; ++u) {
        const int64_t j = j0 + 32 * u;
        if (j < nblk) {
          uint32_t w[8];
          dequant16_bf16(c[u], s_tab[sc[u]], w);
#pragma unroll
          for (int b = 0; b < NB; ++b)
            acc[b] = gemv_dot16(w, xs_all[b * units + 2 * j], xs_all[b * units + 2 * j + 1], acc[b]);
        }
      }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      float v = acc[b];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
      if (lane == 0) y[b * rows + row] = v;
    }
  }
}

bool gemv_resident(int batch, int64_t cols) { return (int64_t)batch * cols * 2 <= kGemvResidentBytes; }

cudaError_t launch_gemv(const uint8_t *codes, const uint8_t *scales, const float *alpha, int64_t rows, int64_t cols,
                        const void *x, int batch, float *y, int grid, cudaStream_t st) {
  const uint2 *c = reinterpret_cast<const uint2 *>(codes);
  const uint4 *xv = static_cast<const uint4 *>(x);
  if (gemv_resident(batch, cols)) {
    const dim3 g((unsigned)grid), b(kGemvResWarps * 32);
    const size_t sm = (size_t)batch * cols * 2;
    switch (batch) {
      case 1: k_gemv_resident<1><<<g, b, sm, st>>>(c, scales, alpha, rows, cols, xv, y); break;
      case 2: k_gemv_resident<2><<<g, b, sm, st>>>(c, scales, alpha, rows, cols, xv, y); break;
      case 3: k_gemv_resident<3><<<g, b, sm, st>>>(c, scales, alpha, rows, cols, xv, y); break;
      case 4: k_gemv_resident<4><<<g, b, sm, st>>>(c, scales, alpha, rows, cols, xv, y); break;
      case 5: k_gemv_resident<5><<<g, b, sm, st>>>(c, scales, alpha, rows, cols, xv, y); break;
      case 6: k_gemv_resident<6><<<g, b, sm, st>>>(c, scales, alpha, rows, cols, xv, y); break;
      case 7: k_gemv_resident<7><<<g, b, sm, st>>>(c, scales, alpha, rows, cols, xv, y); break;
      default: k_gemv_resident<8><<<g, b, sm, st>>>(c, scales, alpha, rows, cols, xv, y); break;
    }
    return cudaGetLastError();
  }
  const dim3 g((unsigned)grid), b(kGemvThreads);
  switch (batch) {
    case 1: k_gemv<1><<<g, b, 0, st>>>(c, scales, alpha, rows, cols, xv, y); break;
    case 2: k_gemv<2><<<g, b, 0, st>>>(c, scales, alpha, rows, cols, xv, y); break;
    case 3: k_gemv<3><<<g, b, 0, st>>>(c, scales, alpha, rows, cols, xv, y); break;
    case 4: k_gemv<4><<<g, b, 0, st>>>(c, scales, alpha, rows, cols, xv, y); break;
    case 5: k_gemv<5><<<g, b, 0, st>>>(c, scales, alpha, rows, cols, xv, y); break;
    case 6: k_gemv<6><<<g, b, 0, st>>>(c, scales, alpha, rows, cols, xv, y); break;
    case 7: k_gemv<7><<<g, b, 0, st>>>(c, scales, alpha, rows, cols, xv, y); break;
    default: k_gemv<8><<<g, b, 0, st>>>(c, scales, alpha, rows, cols, xv, y); break;
  }
  return cudaGetLastError();
}

// Grid of a launch: one CTA per kGemvCtaRows rows (chunked form), or one
// wave of resident CTAs (as many as fit, given their shared memory).
int gemv_grid(int sms, int batch, int64_t rows, int64_t cols) {
  if (gemv_resident(batch, cols)) {
    const size_t sm = (size_t)batch * cols * 2;
    int n = 0;
    cudaError_t e;
    switch (batch) {
      case 1: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gemv_resident<1>, kGemvResWarps * 32, sm); break;
      case 2: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gemv_resident<2>, kGemvResWarps * 32, sm); break;
      case 3: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gemv_resident<3>, kGemvResWarps * 32, sm); break;
      case 4: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gemv_resident<4>, kGemvResWarps * 32, sm); break;
      case 5: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gemv_resident<5>, kGemvResWarps * 32, sm); break;
      case 6: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gemv_resident<6>, kGemvResWarps * 32, sm); break;
      case 7: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gemv_resident<7>, kGemvResWarps * 32, sm); break;
      default: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gemv_resident<8>, kGemvResWarps * 32, sm); break;
    }
    if (e != cudaSuccess || n < 1) n = 1;
    const int64_t need = (rows + kGemvResWarps - 1) / kGemvResWarps;
    return (int)std::min<int64_t>(need, (int64_t)sms * n);
  }
  const int64_t groups = (rows + kGemvCtaRows - 1) / kGemvCtaRows;
  return (int)std::min<int64_t>(groups, (int64_t)sms * gemv_max_active_ctas(batch));
}

cudaError_t prepare_gemv_kernels() {
  cudaError_t e = cudaSuccess;
  const int mx = kGemvResidentBytes;
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemv_resident<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemv_resident<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemv_resident<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemv_resident<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemv_resident<5>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemv_resident<6>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemv_resident<7>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemv_resident<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  return e;
}

int gemv_max_active_ctas(int batch) {
  int n = 0;
  cudaError_t e;
  switch (batch) {
    case 1: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gemv<1>, kGemvThreads, 0); break;
    case 2: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gemv<2>, kGemvThreads, 0); break;
    case 3: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gemv<3>, kGemvThreads, 0); break;
    case 4: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gemv<4>, kGemvThreads, 0); break;
    case 5: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gemv<5>, kGemvThreads, 0); break;
    case 6: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gemv<6>, kGemvThreads, 0); break;
    case 7: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gemv<7>, kGemvThreads, 0); break;
    default: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gemv<8>, kGemvThreads, 0); break;
  }
  return (e == cudaSuccess && n > 0) ? n : 1;
}

}  // namespace nvfp4
