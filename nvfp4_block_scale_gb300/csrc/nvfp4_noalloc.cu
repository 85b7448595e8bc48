// nvfp4_noalloc.cu -- nvfp4_quantize_noalloc: the max-rule / FourOverSix
// quantizer without any device allocation.
//
// Why it exists: nvfp4_quantize takes its few KB of scratch from a stream-
// ordered memory pool.  Some callers cannot allow any allocation from inside
// the library: serving engines that reserve nearly all device memory up front
// and account for every byte themselves, latency-critical threads that must
// never enter an allocator (which can block or reach the driver), and
// embedders whose own allocator must stay the only one in the process.  This
// entry point runs the same two kernels (per-CTA amax partials, then the
// quantize kernel that folds them) with the partials in a fixed static device
// array instead.
//
// The array lives in every GPU that loads the library, from load until exit:
// NVFP4_NOALLOC_SCRATCH_BYTES = 16 KiB = 4096 four-byte slots, one per amax
// CTA.  The amax pass gets a full wave of CTAs (SMs x resident CTAs), and at
// least one CTA per 65,536 elements, never more than 4096; the size limit
// 4096 * 65,536 = 2^28 elements keeps that within the slots, and larger
// tensors are rejected on the host.  In host code the array's name is only a
// host-side stand-in; the device address is fetched once per device with
// cudaGetSymbolAddress (first call on that device, with that device current)
// and passed to the kernels.
#include <algorithm>
#include <cstdint>
#include <mutex>

#include "../../include/nvfp4.h"
#include "nvfp4_internal.h"

namespace {

using namespace nvfp4;

constexpr int kNoAllocMaxCtas = NVFP4_NOALLOC_SCRATCH_BYTES / 4;
constexpr int64_t kElemsPerAmaxCta = 65536;
static_assert(int64_t(kNoAllocMaxCtas) * kElemsPerAmaxCta == NVFP4_NOALLOC_MAX_ELEMS, "scratch / size limit");
constexpr int kMaxDevices = 64;
constexpr int64_t kMaxElems = int64_t(1) << 40;

// Per-CTA amax partials of the call in flight.  Every slot the quantize
// kernel reads is written by the amax kernel of the same call first, so the
// array never needs clearing; calls that overlap on the GPU share it and race.
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocMaxCtas];

struct NoAllocDev {
  bool ready = false;
  int status = NVFP4_OK;
  int sms = 0;
  int l2 = 0;
  int occ_max = 1, occ_fos = 1, occ_amax = 1;
  uint32_t *scratch = nullptr;  // device address of g_noalloc_scratch
};

std::mutex g_na_mu;
NoAllocDev g_na[kMaxDevices];

int na_map(cudaError_t e) {
  if (e == cudaSuccess) return NVFP4_OK;
  if (e == cudaErrorMemoryAllocation) return NVFP4_ERR_OUT_OF_MEMORY;
  return NVFP4_ERR_CUDA;
}

// One-time set-up of the current device: architecture check, occupancy and
// the device address of the static scratch array.  Allocates nothing.
int na_device(NoAllocDev **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return na_map(e);
  if (dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_na_mu);
  NoAllocDev &d = g_na[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.l2, cudaDevAttrL2CacheSize, dev);
    if (e != cudaSuccess) return na_map(e);
    if (major != 10 || minor != 3) {
      d.status = NVFP4_ERR_UNSUPPORTED_DEVICE;
    } else {
      void *p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || p == nullptr) return na_map(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
      d.scratch = static_cast<uint32_t *>(p);
      d.occ_max = max_active_ctas(kKernQuantMax);
      d.occ_fos = max_active_ctas(kKernQuantFos);
      d.occ_amax = max_active_ctas(kKernAmaxLdg);
      d.status = NVFP4_OK;
    }
    d.ready = true;
  }
  *out = &d;
  return d.status;
}

int na_grid(int sms, int occ, int64_t work_items) {
  int64_t full = int64_t(sms) * occ;
  int64_t need = (work_items + 255) / 256;
  if (need < 1) need = 1;
  return (int)(need < full ? need : full);
}

bool na_aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int nvfp4_quantize_noalloc(const void *W, int64_t rows, int64_t cols, int mode, uint8_t *codes,
                                      uint8_t *scales, float *alpha, cudaStream_t stream) {
  if (rows < 0 || cols < 0 || cols % 16 != 0) return NVFP4_ERR_INVALID_ARG;
  if (rows > 0 && cols > kMaxElems / rows) return NVFP4_ERR_INVALID_ARG;
  if (rows * cols >= kMaxElems) return NVFP4_ERR_INVALID_ARG;
  if (rows * cols > NVFP4_NOALLOC_MAX_ELEMS) return NVFP4_ERR_INVALID_ARG;  // scratch holds 4096 partials
  if ((mode != kModeMax && mode != kModeFourOverSix) || !alpha) return NVFP4_ERR_INVALID_ARG;
  const int64_t n = rows * cols;
  if (n > 0 && (!W || !codes || !scales)) return NVFP4_ERR_INVALID_ARG;
  if (!na_aligned(alpha, 4) || (n > 0 && (!na_aligned(W, 16) || !na_aligned(codes, 4))))
    return NVFP4_ERR_MISALIGNED;
  NoAllocDev *d = nullptr;
  int st = na_device(&d);
  if (st != NVFP4_OK) return st;
  if (n == 0) return na_map(cudaMemsetAsync(alpha, 0, sizeof(float), stream));

  const int64_t H = n / 8;
  // One 4-byte slot per amax CTA: a full wave, at least one CTA per 65,536
  // elements, at most 4096 (the size limit above keeps the second term there).
  const int64_t per_elems = (n + kElemsPerAmaxCta - 1) / kElemsPerAmaxCta;
  const int64_t wave = na_grid(d->sms, d->occ_amax, H / 8 + 1);  // as nvfp4_quantize sizes it (8 loads per thread)
  const int g_amax = (int)std::min<int64_t>(kNoAllocMaxCtas, std::max<int64_t>(per_elems, wave));
  const int g_quant = na_grid(d->sms, mode == kModeFourOverSix ? d->occ_fos : d->occ_max, n / 16);
  cudaError_t e = launch_amax_partials(W, H, d->scratch, g_amax, stream);
  const int ranged = 2 * n <= int64_t(d->l2) / 2;
  if (e == cudaSuccess)
    e = launch_quant_max_fos(mode, W, H, d->scratch, g_amax, codes, scales, alpha, g_quant, ranged, stream);
  return na_map(e);
}
