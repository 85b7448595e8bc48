// nvfp4_api.cu -- the C ABI declared in include/nvfp4.h: argument checks,
// scratch allocation from a stream-ordered pool, and the launch sequence of
// each scale rule.
//
// Launch sequences (all on the caller's stream):
//   max / FourOverSix : amax partials -> quantize (folds the partials itself)
//   CJSO(T)           : amax partials -> init sweep -> T iteration sweeps
//                       (each folds the previous sweep's partial sums)
//   decoupled CJSO(T) : the CJSO(T) sweeps without codes -> decoupled search
//   dequantize        : one kernel
//   grouped max / FourOverSix: per slice of up to kGroupMax tensors, one
//                       amax launch and one quantize launch for all of them
//                       (after one memset of the slices' max|W| words)
// Grid-wide dependencies are kernel boundaries: no kernel waits on another
// CTA, so nothing can spin.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/nvfp4.h"
#include "nvfp4_internal.h"

namespace {

using namespace nvfp4;

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxElems = int64_t(1) << 40;
// grouped max rule / FourOverSix: groups of at least kPipeMinL2 x L2 bytes of
// bf16 run in parts of about kPipePartL2 x L2 on two streams; there each
// quantize pass runs one CTA per SM fewer than fit, which leaves the registers
// of kPipeAmaxCtas amax CTAs (the other stream's) on every SM
constexpr int kPipeMinL2 = 4;
constexpr int kPipePartL2 = 3;
constexpr int kPipeAmaxCtas = 2;

struct DevInfo {
  bool ready = false;
  int status = NVFP4_OK;
  int sms = 0;
  int l2 = 0;  // L2 bytes
  int occ[kKernCount] = {};
  cudaMemPool_t pool = nullptr;
  // second streams (with their fork/join events) of the pipelined grouped
  // quantization: a caller takes one that no other call holds and that is not
  // part of an unfinished stream capture (a captured call's second stream
  // stays in that capture until the caller ends it), creating one if none is
  // free
  struct Side {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    bool busy = false;
  };
  std::mutex side_mu;
  std::vector<Side *> sides;
};

std::mutex g_mu;
DevInfo g_dev[kMaxDevices];

// test hooks (nvfp4_test_*): allocations left to fail, and the first-wait
// limit passed to the kernels with bounded waits (< 0: normal)
std::atomic<int> g_fail_allocs{0};
std::atomic<long> g_first_wait{-1};

// Scratch from the library's pool on `stream` (or a failure the test hook asked for).
cudaError_t pool_alloc(void **p, size_t bytes, cudaMemPool_t pool, cudaStream_t stream) {
  int n = g_fail_allocs.load();
  while (n > 0 && !g_fail_allocs.compare_exchange_weak(n, n - 1)) {
  }
  if (n > 0) return cudaErrorMemoryAllocation;
  return cudaMallocFromPoolAsync(p, bytes, pool, stream);
}

int map_cuda(cudaError_t e) {
  if (e == cudaSuccess) return NVFP4_OK;
  if (e == cudaErrorMemoryAllocation) return NVFP4_ERR_OUT_OF_MEMORY;
  return NVFP4_ERR_CUDA;
}

// Per-device facts, queried once: SM count, occupancy of every kernel and a
// library-owned memory pool that keeps its memory (release threshold = max),
// so steady-state scratch allocations never reach the driver.
int device_info(DevInfo **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return map_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  DevInfo &d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.l2, cudaDevAttrL2CacheSize, dev);
    if (e != cudaSuccess) return map_cuda(e);
    if (major != 10 || minor != 3) {
      d.status = NVFP4_ERR_UNSUPPORTED_DEVICE;
    } else {
      e = prepare_decoupled_kernel();
      if (e == cudaSuccess) e = prepare_quant_kernels();
      if (e != cudaSuccess) return map_cuda(e);
      for (int k = 0; k < kKernCount; ++k) d.occ[k] = max_active_ctas(k);
      e = prepare_gemv_kernels();
      if (e == cudaSuccess) e = prepare_gemm_tc_kernels();
      if (e != cudaSuccess) return map_cuda(e);
      cudaMemPoolProps props = {};
      props.allocType = cudaMemAllocationTypePinned;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      e = cudaMemPoolCreate(&d.pool, &props);
      if (e != cudaSuccess) return map_cuda(e);
      uint64_t keep = UINT64_MAX;
      e = cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep);
      if (e != cudaSuccess) return map_cuda(e);
      d.status = NVFP4_OK;
    }
    d.ready = true;
  }
  *out = &d;
  return d.status;
}

// A second stream for one grouped call (see DevInfo::Side); nullptr with *err
// set if none could be made.
DevInfo::Side *side_acquire(DevInfo &d, cudaError_t *err) {
  std::lock_guard<std::mutex> lock(d.side_mu);
  for (DevInfo::Side *s : d.sides) {
    if (s->busy) continue;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s->stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) continue;
    s->busy = true;
    return s;
  }
  DevInfo::Side *s = new (std::nothrow) DevInfo::Side;
  if (!s) {
    *err = cudaErrorMemoryAllocation;
    return nullptr;
  }
  cudaError_t e = cudaStreamCreateWithFlags(&s->stream, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s->fork, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s->join, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    if (s->join) cudaEventDestroy(s->join);
    if (s->fork) cudaEventDestroy(s->fork);
    if (s->stream) cudaStreamDestroy(s->stream);
    delete s;
    *err = e;
    return nullptr;
  }
  s->busy = true;
  d.sides.push_back(s);
  return s;
}

void side_release(DevInfo &d, DevInfo::Side *s) {
  std::lock_guard<std::mutex> lock(d.side_mu);
  s->busy = false;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_shape(int64_t rows, int64_t cols) {
  if (rows < 0 || cols < 0 || cols % 16 != 0) return NVFP4_ERR_INVALID_ARG;
  if (rows > 0 && cols > kMaxElems / rows) return NVFP4_ERR_INVALID_ARG;
  if (rows * cols >= kMaxElems) return NVFP4_ERR_INVALID_ARG;
  return NVFP4_OK;
}

int grid_for(const DevInfo &d, int kern, int64_t work_items) {
  int64_t full = int64_t(d.sms) * d.occ[kern];
  int64_t need = (work_items + 255) / 256;
  if (need < 1) need = 1;
  return (int)(need < full ? need : full);
}

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------------------
// Kernel tracing: CUDA events around each launch while enabled.
// ---------------------------------------------------------------------------

enum { kTrAmax = 0, kTrQuantMax, kTrQuantFos, kTrCjsoInit, kTrCjsoIter, kTrDecoupled, kTrDequant, kTrEncode,
       kTrGroupAmax, kTrGroupQuantMax, kTrGroupQuantFos, kTrGemv, kTrSwizzle, kTrAmaxLdg, kTrGemmTc,
       kTrGemmTcReduce, kTrKinds };
const char *const kTraceNames[kTrKinds] = {"k_amax_bulk",        "k_quant_max_fos<max>", "k_quant_max_fos<fos>",
                                           "k_cjso_sweep<init>",  "k_cjso_sweep<iter>",   "k_decoupled",
                                           "k_dequant",           "k_encode",             "k_group_amax",
                                           "k_group_quant<max>",  "k_group_quant<fos>",   "k_gemv",
                                           "k_swizzle_scales",   "k_amax_partials",      "k_gemm_tc",
                                           "k_gemm_tc_reduce"};

struct TraceRec {
  int kind;
  cudaEvent_t start, stop;
};

std::mutex g_tr_mu;
bool g_tr_on = false;
std::vector<TraceRec> g_tr_pending;
int64_t g_tr_launches[kTrKinds] = {};
double g_tr_ms[kTrKinds] = {};

// Records the start event (if tracing) before a launch and the stop event after.
struct TraceScope {
  int kind;
  cudaStream_t st;
  cudaEvent_t a = nullptr, b = nullptr;
  TraceScope(int k, cudaStream_t s) : kind(k), st(s) {
    bool on;
    {
      std::lock_guard<std::mutex> lock(g_tr_mu);
      on = g_tr_on;
    }
    if (!on) return;
    if (cudaEventCreate(&a) != cudaSuccess || cudaEventCreate(&b) != cudaSuccess ||
        cudaEventRecord(a, st) != cudaSuccess) {
      if (a) cudaEventDestroy(a);
      if (b) cudaEventDestroy(b);
      a = b = nullptr;
    }
  }
  ~TraceScope() {
    if (!a) return;
    if (cudaEventRecord(b, st) != cudaSuccess) {
      cudaEventDestroy(a);
      cudaEventDestroy(b);
      return;
    }
    std::lock_guard<std::mutex> lock(g_tr_mu);
    g_tr_pending.push_back({kind, a, b});
  }
};

}  // namespace

extern "C" {

const char *nvfp4_status_string(int status) {
  switch (status) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_INVALID_ARG: return "invalid argument";
    case NVFP4_ERR_MISALIGNED: return "misaligned pointer";
    case NVFP4_ERR_CUDA: return "CUDA runtime error";
    case NVFP4_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
    case NVFP4_ERR_OUT_OF_MEMORY: return "out of device memory";
    default: return "unknown status";
  }
}

int nvfp4_quantize(const void *W, int64_t rows, int64_t cols, int mode, int iters, uint8_t *codes,
                   uint8_t *scales, float *alpha, cudaStream_t stream) {
  int st = check_shape(rows, cols);
  if (st != NVFP4_OK) return st;
  if (mode < kModeMax || mode > kModeCjsoDecoupled || !alpha) return NVFP4_ERR_INVALID_ARG;
  const bool cjso = mode == kModeCjso || mode == kModeCjsoDecoupled;
  if (cjso && (iters < 0 || iters > kMaxIters)) return NVFP4_ERR_INVALID_ARG;
  const int64_t n = rows * cols;
  if (n > 0 && (!W || !codes || !scales)) return NVFP4_ERR_INVALID_ARG;
  if (!aligned(alpha, 4) || (n > 0 && (!aligned(W, 16) || !aligned(codes, 4)))) return NVFP4_ERR_MISALIGNED;
  DevInfo *d = nullptr;
  st = device_info(&d);
  if (st != NVFP4_OK) return st;
  if (n == 0) return map_cuda(cudaMemsetAsync(alpha, 0, sizeof(float), stream));

  const int64_t H = n / 8;   // half blocks = 16-byte loads
  const int64_t B = n / 16;  // blocks
  const int T = cjso ? iters : 0;
  // amax pass: bulk copies through shared memory for tensors beyond half of L2
  // (measured faster there), plain 16-byte loads for smaller ones (faster there)
  const bool bulk = 2 * n > int64_t(d->l2) / 2;
  const int g_amax = bulk ? (int)std::min<int64_t>(amax_bulk_chunks(H), int64_t(d->sms) * d->occ[kKernAmax])
                          : grid_for(*d, kKernAmaxLdg, H / 8 + 1);  // 8 loads per thread per tile
  const int ranged = 2 * n <= int64_t(d->l2) / 2;  // W stays in L2 between the two passes
  const int g_quant = grid_for(*d, mode == kModeFourOverSix ? kKernQuantFos : kKernQuantMax, B);
  const int g_cjso = grid_for(*d, kKernCjso, B);
  // scratch: amax partials | 2 x CJSO partial sums (two 128-bit integers per CTA) | alpha history |
  // (decoupled) the count and list of the search's deferred blocks
  const int64_t off_part = round_up(int64_t(g_amax) * 4, 256);
  const int64_t off_hist = off_part + round_up(2 * int64_t(g_cjso) * 32, 256);
  const int64_t off_defer = off_hist + round_up(int64_t(kMaxIters + 1) * 4, 256);
  const int defer_cap = (int)std::min<int64_t>(kDeferCap, B);
  const int64_t ws_bytes = off_defer + (mode == kModeCjsoDecoupled ? 256 + round_up(int64_t(defer_cap) * 8, 256) : 0);
  void *ws = nullptr;
  cudaError_t e = pool_alloc(&ws, (size_t)ws_bytes, d->pool, stream);
  if (e != cudaSuccess) return map_cuda(e);
  char *base = static_cast<char *>(ws);
  uint32_t *amax_part = reinterpret_cast<uint32_t *>(base);
  ulonglong2 *part[2] = {reinterpret_cast<ulonglong2 *>(base + off_part),
                         reinterpret_cast<ulonglong2 *>(base + off_part) + 2 * int64_t(g_cjso)};
  float *hist = reinterpret_cast<float *>(base + off_hist);
  uint32_t *defer_count = reinterpret_cast<uint32_t *>(base + off_defer);
  int64_t *defer_list = reinterpret_cast<int64_t *>(base + off_defer + 256);

  if (mode == kModeCjsoDecoupled) e = cudaMemsetAsync(defer_count, 0, sizeof(uint32_t), stream);
  if (e == cudaSuccess) {
    TraceScope tr(bulk ? kTrAmax : kTrAmaxLdg, stream);
    e = bulk ? launch_amax_bulk(W, H, amax_part, g_amax, g_first_wait.load(), stream)
             : launch_amax_partials(W, H, amax_part, g_amax, stream);
  }
  if (e == cudaSuccess && !cjso) {
    TraceScope tr(mode == kModeFourOverSix ? kTrQuantFos : kTrQuantMax, stream);
    e = launch_quant_max_fos(mode, W, H, amax_part, g_amax, codes, scales, alpha, g_quant, ranged, stream);
  } else if (e == cudaSuccess) {
    const bool plain = mode == kModeCjso;
    {
      TraceScope tr(kTrCjsoInit, stream);
      e = launch_cjso_sweep(true, T > 0, W, H, amax_part, g_amax, nullptr, 0, part[0], hist, 0, scales, codes,
                            plain && T == 0, alpha, T == 0, g_cjso, stream);
    }
    for (int t = 1; t <= T && e == cudaSuccess; ++t) {
      TraceScope tr(kTrCjsoIter, stream);
      e = launch_cjso_sweep(false, t < T, W, H, amax_part, g_amax, part[(t - 1) & 1], g_cjso, part[t & 1], hist,
                            t, scales, codes, plain && t == T, alpha, t == T, g_cjso, stream);
    }
    if (e == cudaSuccess && !plain) {
      TraceScope tr(kTrDecoupled, stream);
      e = launch_decoupled(W, B, hist, T, scales, codes, defer_count, defer_list, defer_cap, d->sms, stream);
    }
  }
  // The scratch goes back to the pool in stream order, after the last kernel.
  cudaError_t ef = cudaFreeAsync(ws, stream);
  return map_cuda(e != cudaSuccess ? e : ef);
}

int nvfp4_quantize_grouped(const nvfp4_tensor *tensors, int count, int mode, int iters, cudaStream_t stream) {
  if (count < 0 || (count > 0 && !tensors)) return NVFP4_ERR_INVALID_ARG;
  if (mode < kModeMax || mode > kModeCjsoDecoupled) return NVFP4_ERR_INVALID_ARG;
  const bool cjso = mode == kModeCjso || mode == kModeCjsoDecoupled;
  if (cjso && (iters < 0 || iters > kMaxIters)) return NVFP4_ERR_INVALID_ARG;
  for (int i = 0; i < count; ++i) {  // every descriptor before anything is enqueued
    const nvfp4_tensor &x = tensors[i];
    int st = check_shape(x.rows, x.cols);
    if (st != NVFP4_OK) return st;
    const int64_t n = x.rows * x.cols;
    if (!x.alpha || (n > 0 && (!x.W || !x.codes || !x.scales))) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(x.alpha, 4) || (n > 0 && (!aligned(x.W, 16) || !aligned(x.codes, 4))))
      return NVFP4_ERR_MISALIGNED;
  }
  DevInfo *d = nullptr;
  int st = device_info(&d);
  if (st != NVFP4_OK) return st;
  if (count == 0) return NVFP4_OK;
  if (cjso) {
    // the single-tensor sequence per tensor, tensors alternating between the
    // caller's stream and the library's second one, so that one tensor's
    // sweeps (HBM-bound) can run beside another's search (ALU-bound)
    cudaError_t e = cudaSuccess;
    DevInfo::Side *sd = count >= 2 ? side_acquire(*d, &e) : nullptr;
    if (sd) {
      e = cudaEventRecord(sd->fork, stream);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(sd->stream, sd->fork, 0);
    }
    for (int i = 0; i < count && e == cudaSuccess && st == NVFP4_OK; ++i) {
      const nvfp4_tensor &x = tensors[i];
      st = nvfp4_quantize(x.W, x.rows, x.cols, mode, iters, x.codes, x.scales, x.alpha,
                          sd && (i & 1) ? sd->stream : stream);
    }
    if (sd) {  // join, also after an error
      cudaError_t ej = cudaEventRecord(sd->join, sd->stream);
      if (ej == cudaSuccess) ej = cudaStreamWaitEvent(stream, sd->join, 0);
      if (e == cudaSuccess) e = ej;
      side_release(*d, sd);
    }
    return st != NVFP4_OK ? st : map_cuda(e);
  }

  // Parts of at most kGroupMax tensors, each an amax pass and a quantize pass
  // over its tiles.  A group of at least kPipeMinL2 x L2 of bf16 is cut into
  // parts of about kPipePartL2 x L2 that alternate between the caller's stream
  // and a second stream, so one part's amax pass (HBM-bound) runs beside
  // another's quantize pass (issue-bound) on the same SMs: the quantize grid
  // then holds one CTA per SM fewer than fit (with both modes' register counts
  // that frees room for two amax CTAs) and the amax grid kPipeAmaxCtas per SM.
  // Smaller groups keep one part per kGroupMax tensors, which lets the
  // quantize pass re-read from L2 what the amax pass read last.
  int64_t total = 0;
  for (int i = 0; i < count; ++i) total += tensors[i].rows * tensors[i].cols;
  const bool pipe = total * 2 >= int64_t(kPipeMinL2) * d->l2 && count >= 2;
  const int parts = pipe ? (int)std::max<int64_t>(2, (total * 2 + int64_t(kPipePartL2) * d->l2 / 2) /
                                                         (int64_t(kPipePartL2) * d->l2))
                         : 1;
  std::vector<int> cut;  // part k covers tensors [cut[k], cut[k + 1])
  cut.push_back(0);
  int64_t acc = 0;
  for (int i = 0; i + 1 < count; ++i) {  // a cut after tensor i where 1/parts of the elements is passed
    acc += tensors[i].rows * tensors[i].cols;
    if ((pipe && acc * parts >= total * (int64_t)cut.size()) || i + 1 - cut.back() == kGroupMax) cut.push_back(i + 1);
  }
  cut.push_back(count);
  const int nparts = (int)cut.size() - 1;
  const size_t slot = (size_t)round_up(int64_t(kGroupMax) * 4, 256);
  void *ws = nullptr;
  cudaError_t e = pool_alloc(&ws, slot * nparts, d->pool, stream);
  if (e != cudaSuccess) return map_cuda(e);
  e = cudaMemsetAsync(ws, 0, slot * nparts, stream);  // every tensor's max|W| word starts at 0
  DevInfo::Side *sd = pipe && e == cudaSuccess ? side_acquire(*d, &e) : nullptr;
  if (sd) {  // fork the second stream off the caller's
    e = cudaEventRecord(sd->fork, stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(sd->stream, sd->fork, 0);
  }
  GroupArgs *g = new (std::nothrow) GroupArgs;
  if (!g && e == cudaSuccess) e = cudaErrorMemoryAllocation;
  const int kq = mode == kModeFourOverSix ? kKernGroupQuantFos : kKernGroupQuantMax;
  const int64_t full = int64_t(d->sms) * std::min(d->occ[kKernGroupAmax], d->occ[kq]);
  for (int k = 0; k < nparts && e == cudaSuccess; ++k) {
    const int s0 = cut[k];
    cudaStream_t ps = sd && (k & 1) ? sd->stream : stream;
    g->count = cut[k + 1] - s0;
    g->tile_begin[0] = 0;
    for (int i = 0; i < g->count; ++i) {
      const nvfp4_tensor &x = tensors[s0 + i];
      GroupTensor &gt = g->t[i];
      gt.W = x.W;
      gt.codes = x.codes;
      gt.scales = x.scales;
      gt.alpha = x.alpha;
      gt.B = x.rows * x.cols / 16;
      g->tile_begin[i + 1] = g->tile_begin[i] + (gt.B + kGroupTile - 1) / kGroupTile;
    }
    const int64_t tiles = g->tile_begin[g->count];
    const int grid = (int)std::max<int64_t>(1, std::min(full, tiles));
    const int grid_a = sd ? (int)std::max<int64_t>(1, std::min<int64_t>(int64_t(d->sms) * kPipeAmaxCtas, tiles)) : grid;
    const int grid_q =
        sd ? (int)std::max<int64_t>(1, std::min<int64_t>(int64_t(d->sms) * std::max(1, d->occ[kq] - 1), tiles)) : grid;
    uint32_t *amax = reinterpret_cast<uint32_t *>(static_cast<char *>(ws) + slot * k);
    {
      TraceScope tr(kTrGroupAmax, ps);
      e = launch_group_amax(*g, amax, grid_a, ps);
    }
    if (e == cudaSuccess) {
      TraceScope tr(mode == kModeFourOverSix ? kTrGroupQuantFos : kTrGroupQuantMax, ps);
      e = launch_group_quant(mode, *g, amax, grid_q, ps);
    }
  }
  delete g;
  if (sd) {  // join: the caller's stream waits for the second stream's parts
    cudaError_t ej = cudaEventRecord(sd->join, sd->stream);
    if (ej == cudaSuccess) ej = cudaStreamWaitEvent(stream, sd->join, 0);
    if (e == cudaSuccess) e = ej;
    side_release(*d, sd);
  }
  cudaError_t ef = cudaFreeAsync(ws, stream);
  return map_cuda(e != cudaSuccess ? e : ef);
}

int nvfp4_dequantize(const uint8_t *codes, const uint8_t *scales, const float *alpha, int64_t rows, int64_t cols,
                     void *out, cudaStream_t stream) {
  int st = check_shape(rows, cols);
  if (st != NVFP4_OK) return st;
  const int64_t n = rows * cols;
  if (!alpha || (n > 0 && (!codes || !scales || !out))) return NVFP4_ERR_INVALID_ARG;
  if (!aligned(alpha, 4) || (n > 0 && (!aligned(codes, 4) || !aligned(out, 16)))) return NVFP4_ERR_MISALIGNED;
  DevInfo *d = nullptr;
  st = device_info(&d);
  if (st != NVFP4_OK) return st;
  if (n == 0) return NVFP4_OK;
  const int64_t H = n / 8;
  TraceScope tr(kTrDequant, stream);
  return map_cuda(launch_dequant(codes, scales, alpha, H, out, grid_for(*d, kKernDequant, H), stream));
}

int nvfp4_gemv(const uint8_t *codes, const uint8_t *scales, const float *alpha, int64_t rows, int64_t cols,
               const void *x, int batch, float *y, cudaStream_t stream) {
  int st = check_shape(rows, cols);
  if (st != NVFP4_OK) return st;
  if (batch < 1 || batch > 8) return NVFP4_ERR_INVALID_ARG;
  const int64_t n = rows * cols;
  if (!alpha || (n > 0 && (!codes || !scales || !x || !y))) return NVFP4_ERR_INVALID_ARG;
  if (!aligned(alpha, 4) || (n > 0 && (!aligned(codes, 8) || !aligned(x, 16) || !aligned(y, 4))))
    return NVFP4_ERR_MISALIGNED;
  DevInfo *d = nullptr;
  st = device_info(&d);
  if (st != NVFP4_OK) return st;
  if (rows == 0) return NVFP4_OK;
  if (cols == 0) return map_cuda(cudaMemsetAsync(y, 0, sizeof(float) * (size_t)(rows * batch), stream));
  TraceScope tr(kTrGemv, stream);
  return map_cuda(launch_gemv(codes, scales, alpha, rows, cols, x, batch, y,
                              gemv_grid(d->sms, batch, rows, cols), stream));
}

int nvfp4_gemm(const uint8_t *codes, const uint8_t *scales, const float *alpha, int64_t rows, int64_t cols,
               const void *x, int batch, float *y, cudaStream_t stream) {
  int st = check_shape(rows, cols);
  if (st != NVFP4_OK) return st;
  if (batch < 1 || batch > 256) return NVFP4_ERR_INVALID_ARG;
  const int64_t n = rows * cols;
  if (!alpha || (n > 0 && (!codes || !scales || !x || !y))) return NVFP4_ERR_INVALID_ARG;
  if (!aligned(alpha, 4) || (n > 0 && (!aligned(codes, 8) || !aligned(x, 16) || !aligned(y, 4))))
    return NVFP4_ERR_MISALIGNED;
  DevInfo *d = nullptr;
  st = device_info(&d);
  if (st != NVFP4_OK) return st;
  if (rows == 0) return NVFP4_OK;
  if (cols == 0) return map_cuda(cudaMemsetAsync(y, 0, sizeof(float) * (size_t)(rows * batch), stream));
  // one persistent CTA per SM over all (tile, 128-column step) pairs; the
  // partial sums of tiles shared by several CTAs meet in a workspace
  const int64_t ny = int64_t(batch) * rows;
  void *ws = nullptr;
  cudaError_t e = pool_alloc(&ws, gemm_tc_workspace_bytes(rows, cols, batch, d->sms), d->pool, stream);
  if (e != cudaSuccess) return map_cuda(e);
  float *part = static_cast<float *>(ws);
  {
    TraceScope tr(kTrGemmTc, stream);
    const long fw = g_first_wait.load();
    e = launch_gemm_tc(codes, scales, alpha, rows, cols, x, batch, d->sms, part, y,
                       fw < 0 ? -1 : (int)std::min<long>(fw, INT32_MAX), stream);
  }
  if (e == cudaSuccess) {
    TraceScope tr(kTrGemmTcReduce, stream);
    e = launch_gemm_tc_reduce(part, rows, cols, batch, d->sms, y, grid_for(*d, kKernDequant, ny), stream);
  }
  cudaError_t ef = cudaFreeAsync(ws, stream);
  return map_cuda(e != cudaSuccess ? e : ef);
}

int64_t nvfp4_swizzled_scales_bytes(int64_t rows, int64_t cols) {
  if (check_shape(rows, cols) != NVFP4_OK) return -1;
  return round_up(rows, 128) * round_up(cols / 16, 4);
}

int nvfp4_swizzle_scales(const uint8_t *scales, int64_t rows, int64_t cols, uint8_t *out, cudaStream_t stream) {
  int st = check_shape(rows, cols);
  if (st != NVFP4_OK) return st;
  const int64_t bytes = round_up(rows, 128) * round_up(cols / 16, 4);
  if (bytes > 0 && (!scales || !out)) return NVFP4_ERR_INVALID_ARG;
  if (bytes > 0 && !aligned(out, 4)) return NVFP4_ERR_MISALIGNED;
  DevInfo *d = nullptr;
  st = device_info(&d);
  if (st != NVFP4_OK) return st;
  if (bytes == 0) return NVFP4_OK;
  TraceScope tr(kTrSwizzle, stream);
  return map_cuda(launch_swizzle_scales(scales, rows, cols / 16, out, stream));
}

int nvfp4_encode_e2m1(const float *v, int64_t n, uint8_t *out, cudaStream_t stream) {
  if (n < 0 || n >= kMaxElems || (n > 0 && (!v || !out))) return NVFP4_ERR_INVALID_ARG;
  if (n > 0 && !aligned(v, 4)) return NVFP4_ERR_MISALIGNED;
  DevInfo *d = nullptr;
  int st = device_info(&d);
  if (st != NVFP4_OK) return st;
  if (n == 0) return NVFP4_OK;
  TraceScope tr(kTrEncode, stream);
  return map_cuda(launch_encode_e2m1(v, n, out, grid_for(*d, kKernDequant, n), stream));
}

int nvfp4_encode_e4m3(const float *v, int64_t n, uint8_t *out, cudaStream_t stream) {
  if (n < 0 || n >= kMaxElems || (n > 0 && (!v || !out))) return NVFP4_ERR_INVALID_ARG;
  if (n > 0 && !aligned(v, 4)) return NVFP4_ERR_MISALIGNED;
  DevInfo *d = nullptr;
  int st = device_info(&d);
  if (st != NVFP4_OK) return st;
  if (n == 0) return NVFP4_OK;
  TraceScope tr(kTrEncode, stream);
  return map_cuda(launch_encode_e4m3(v, n, out, grid_for(*d, kKernDequant, n), stream));
}

int nvfp4_ffma_probe(int packed, int64_t rounds, float *sink, int64_t sink_floats, int64_t *fmas,
                     cudaStream_t stream) {
  if ((packed != 0 && packed != 1) || rounds < 1 || rounds > (int64_t(1) << 32) || !sink || !fmas)
    return NVFP4_ERR_INVALID_ARG;
  if (!aligned(sink, 4)) return NVFP4_ERR_MISALIGNED;
  DevInfo *d = nullptr;
  int st = device_info(&d);
  if (st != NVFP4_OK) return st;
  const int grid = d->sms * ffma_probe_occupancy(packed);
  const int64_t threads = int64_t(grid) * ffma_probe_threads();
  if (sink_floats < threads) return NVFP4_ERR_INVALID_ARG;
  *fmas = threads * ffma_probe_fmas_per_thread(packed, rounds);
  return map_cuda(launch_ffma_probe(packed, rounds, grid, sink, stream));
}

int nvfp4_test_fail_allocations(int count) {
  if (count < 0) return NVFP4_ERR_INVALID_ARG;
  g_fail_allocs.store(count);
  return NVFP4_OK;
}

int nvfp4_test_first_wait_tries(int64_t tries) {
  g_first_wait.store(tries < 0 ? -1L : (long)std::min<int64_t>(tries, int64_t(1) << 30));
  return NVFP4_OK;
}

int nvfp4_checked_build(void) {
#ifdef NVFP4_CHECKED
  return 1;
#else
  return 0;
#endif
}

int nvfp4_check_take(uint32_t *site) {
  if (!site) return NVFP4_ERR_INVALID_ARG;
  *site = 0u;
#ifdef NVFP4_CHECKED
  DevInfo *d = nullptr;
  int st = device_info(&d);
  if (st != NVFP4_OK) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = check_take_kernels(site);
  if (e == cudaSuccess) e = check_take_decoupled(site);
  return map_cuda(e);
#else
  return NVFP4_OK;
#endif
}

int nvfp4_check_selftest(int64_t i, int64_t n, cudaStream_t stream) {
  DevInfo *d = nullptr;
  int st = device_info(&d);
  if (st != NVFP4_OK) return st;
  return map_cuda(launch_check_selftest(i, n, stream));
}

int nvfp4_profiler_enable(int on) {
  std::lock_guard<std::mutex> lock(g_tr_mu);
  g_tr_on = on != 0;
  return NVFP4_OK;
}

int nvfp4_profiler_reset(void) {
  std::lock_guard<std::mutex> lock(g_tr_mu);
  for (auto &r : g_tr_pending) {
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  g_tr_pending.clear();
  for (int k = 0; k < kTrKinds; ++k) {
    g_tr_launches[k] = 0;
    g_tr_ms[k] = 0.0;
  }
  return NVFP4_OK;
}

int nvfp4_profiler_kinds(void) {
  std::lock_guard<std::mutex> lock(g_tr_mu);
  int status = 0;
  for (auto &r : g_tr_pending) {
    float ms = 0.0f;
    cudaError_t e = cudaEventSynchronize(r.stop);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.start, r.stop);
    if (e == cudaSuccess) {
      g_tr_launches[r.kind] += 1;
      g_tr_ms[r.kind] += ms;
    } else {
      status = -NVFP4_ERR_CUDA;
    }
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  g_tr_pending.clear();
  if (status < 0) return status;
  int n = 0;
  for (int k = 0; k < kTrKinds; ++k) n += g_tr_launches[k] > 0;
  return n;
}

int nvfp4_profiler_get(int index, char *name, int name_len, int64_t *launches, double *total_ms) {
  std::lock_guard<std::mutex> lock(g_tr_mu);
  int seen = -1;
  for (int k = 0; k < kTrKinds; ++k) {
    if (g_tr_launches[k] == 0) continue;
    if (++seen != index) continue;
    if (name && name_len > 0) {
      std::strncpy(name, kTraceNames[k], (size_t)name_len - 1);
      name[name_len - 1] = '\0';
    }
    if (launches) *launches = g_tr_launches[k];
    if (total_ms) *total_ms = g_tr_ms[k];
    return NVFP4_OK;
  }
  return NVFP4_ERR_INVALID_ARG;
}

}  // extern "C"
