// nvfp4_probe.cu -- FP32 fused multiply-add throughput probe.
//
// The decoupled scale search is bound by the fp32 pipe, so its roofline
// needs the fp32 peak of the GPU it runs on, at the clock it runs at.  This
// kernel measures it: every thread runs kChains independent FMA chains (enough
// to hide the pipe latency), either as scalar fma.rn.f32 or as packed
// fma.rn.f32x2, and the host divides 2 flop x FMAs by the kernel's duration.
// Instrumentation only: no step of the quantizer uses it.
#include <cuda_runtime.h>

#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {

constexpr int kProbeThreads = 256;
constexpr int kChains = 8;

template <bool PACKED>
__global__ void __launch_bounds__(kProbeThreads) k_ffma_probe(int64_t rounds, float *__restrict__ sink) {
  const float a = 1.0f + 1e-7f * (float)(threadIdx.x & 7);
  const float b = 1e-8f * (float)(blockIdx.x & 3);
  if (PACKED) {
    f32x2 acc[kChains], m = pack2(a, a), c = pack2(b, -b);
#pragma unroll
    for (int i = 0; i < kChains; ++i) acc[i] = pack2((float)i, -(float)i);
    for (int64_t r = 0; r < rounds; ++r) {
#pragma unroll
      for (int i = 0; i < kChains; ++i) acc[i] = fma2(acc[i], m, c);  // 2 FMAs each
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < kChains; ++i) {
      float lo, hi;
      asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(acc[i]));
      s = __fadd_rn(s, __fadd_rn(lo, hi));
    }
    sink[(int64_t)blockIdx.x * kProbeThreads + threadIdx.x] = s;
  } else {
    float acc[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i) acc[i] = (float)i;
    for (int64_t r = 0; r < rounds; ++r) {
#pragma unroll
      for (int i = 0; i < kChains; ++i) acc[i] = __fmaf_rn(acc[i], a, b);
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s = __fadd_rn(s, acc[i]);
    sink[(int64_t)blockIdx.x * kProbeThreads + threadIdx.x] = s;
  }
}

int64_t ffma_probe_fmas_per_thread(int packed, int64_t rounds) { return rounds * kChains * (packed ? 2 : 1); }

cudaError_t launch_ffma_probe(int packed, int64_t rounds, int grid, float *sink, cudaStream_t st) {
  if (packed) k_ffma_probe<true><<<grid, kProbeThreads, 0, st>>>(rounds, sink);
  else k_ffma_probe<false><<<grid, kProbeThreads, 0, st>>>(rounds, sink);
  return cudaGetLastError();
}

int ffma_probe_threads() { return kProbeThreads; }

int ffma_probe_occupancy(int packed) {
  int n = 0;
  cudaError_t e = packed ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_ffma_probe<true>, kProbeThreads, 0)
                         : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_ffma_probe<false>, kProbeThreads, 0);
  return (e == cudaSuccess && n > 0) ? n : 1;
}

}  // namespace nvfp4
