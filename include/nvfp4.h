/*
 * nvfp4.h -- C ABI of libnvfp4_gb300.so: NVFP4 block quantization of bf16
 * weight tensors on an sm_103 GPU (GB300).
 *
 * NVFP4 here means: 4-bit E2M1 codes, one FP8 E4M3 scale Delta_i per block of
 * 16 consecutive elements of a row, and one fp32 tensor scale alpha, so that an
 * element dequantizes to q * alpha * Delta_i.  Sources of the method:
 *   [SOAR]  "SOAR: Scale Optimization for Accurate Reconstruction in NVFP4
 *           Quantization" (july-h5kf3.github.io notes): the NVFP4 quantizer
 *           equation (alpha = max|W| / (6*448), Delta_i = e4m3(max|W_i| /
 *           (6 alpha)), piecewise FP4 rounding), the dequantization equation,
 *           CJSO (closed forms for alpha* and Delta_i*, schedule) and the
 *           decoupled quantization / dequantization scale search.
 *   [FOS]   "SOAR 周冠军笔记 07 | 香草小张：NVFP4 量化改进与推测解码实践"
 *           (openbmb.cn blog), section 01 (E2M1 value set) and section 02
 *           (FourOverSix: scale_m4 = fp8(scale_m6 * 1.5), keep the lower MSE).
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never frees or keeps them.  Every call is asynchronous on `stream`
 *     (a cudaStream_t; NULL = the legacy default stream); outputs are valid
 *     once the stream has reached the call's end.
 *   - W is bf16, row-major [rows, cols], contiguous.  cols must be a multiple
 *     of 16 (one block = 16 consecutive elements of a row).
 *   - codes: rows*cols/2 bytes, row-major [rows, cols/2]; byte k of a row holds
 *     element 2k in its low nibble and element 2k+1 in its high nibble; bit 3
 *     of a nibble is the sign, bits 0-2 index {0,0.5,1,1.5,2,3,4,6}.
 *   - scales: rows*cols/16 bytes, row-major [rows, cols/16], E4M3FN bit
 *     patterns (linear layout, not swizzled).
 *   - alpha: one fp32 on the device.
 *   - Arguments are checked on the host before anything is enqueued; on an
 *     error nothing is enqueued and a nonzero status is returned.
 *   - Inputs must be finite, and either all zero or with max|W| >= 2^-64; for
 *     other inputs the outputs are unspecified (no memory is touched beyond
 *     the documented buffers either way).
 *   - The first call on a device performs a one-time set-up with that
 *     device current (device queries, kernel attributes, the library's
 *     memory pool); make it before any stream capture (a warm-up call).
 *   - Calls on different streams may run concurrently; the library keeps no
 *     per-call global state.  Scratch memory comes from a library-owned,
 *     stream-ordered memory pool (cudaMallocFromPoolAsync / cudaFreeAsync on
 *     `stream`); it is a few tens of KB per call.
 */
#ifndef NVFP4_GB300_H
#define NVFP4_GB300_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
enum nvfp4_status {
  NVFP4_OK = 0,
  NVFP4_ERR_INVALID_ARG = 1,        /* null pointer, negative size, cols % 16 != 0, bad mode/iters, size overflow */
  NVFP4_ERR_MISALIGNED = 2,         /* W/out not 16-byte aligned, codes or alpha not 4-byte aligned */
  NVFP4_ERR_CUDA = 3,               /* a CUDA runtime call or launch failed */
  NVFP4_ERR_UNSUPPORTED_DEVICE = 4, /* current device is not compute capability 10.3 */
  NVFP4_ERR_OUT_OF_MEMORY = 5       /* the scratch allocation failed */
};

/* Scale rules ([SOAR] quantizer equation; [FOS] section 02; [SOAR] CJSO and
 * decoupled search). */
enum nvfp4_mode {
  NVFP4_MODE_MAX = 0,            /* Delta_i = e4m3(amax_i / (6 alpha)) */
  NVFP4_MODE_FOUR_OVER_SIX = 1,  /* per block: the max-rule scale, or e4m3(1.5 * it) if that
                                    gives a strictly lower dequantization error */
  NVFP4_MODE_CJSO = 2,           /* max rule, then `iters` rounds of: alpha* (closed form),
                                    re-quantize, Delta_i* (closed form, rounded to E4M3),
                                    re-quantize */
  NVFP4_MODE_CJSO_DECOUPLED = 3  /* CJSO(iters), then per block a search over 101 quantization
                                    scales Delta^d0 * {0.50, 0.51, ..., 1.50} and, for each, the
                                    two E4M3 values bracketing it as the stored scale; the pair
                                    with the least reconstruction error is kept */
};

/*
 * nvfp4_quantize -- bf16 W [rows, cols] -> codes, scales, alpha.
 *   [SOAR] quantizer equation (alpha, Delta_i, FP4 rounding); mode-specific
 *   passages as listed for enum nvfp4_mode.
 * Arguments:
 *   W      device, bf16, 16-byte aligned; rows*cols elements.
 *   rows   >= 0.  cols >= 0, cols % 16 == 0.  rows*cols < 2^40.
 *   mode   an nvfp4_mode value.
 *   iters  CJSO iterations, 0..64 (modes 2 and 3); ignored by modes 0 and 1.
 *   codes  device, 4-byte aligned, rows*cols/2 bytes (written).
 *   scales device, rows*cols/16 bytes (written).
 *   alpha  device, 4-byte aligned, 1 float (written; 0 for an empty or all-zero W).
 *   stream cudaStream_t.
 * Returns an nvfp4_status.  rows*cols == 0 is valid: only *alpha = 0 is written
 * (W, codes and scales may then be NULL).  Every wait inside a kernel is
 * bounded: should a device-side copy never complete, the kernel gives up
 * after its limit and *alpha comes out NaN (the status, returned before the
 * kernels run, cannot report it).
 */
int nvfp4_quantize(const void *W, int64_t rows, int64_t cols, int mode, int iters,
                   uint8_t *codes, uint8_t *scales, float *alpha, cudaStream_t stream);

/*
 * nvfp4_quantize_grouped -- quantize a list of tensors, each exactly as
 *   nvfp4_quantize would (its own alpha from its own max|W|, [SOAR] quantizer
 *   equation), with one pair of launches for up to NVFP4_GROUP_MAX tensors of
 *   the max rule or FourOverSix: the first finds every tensor's max|W|, the
 *   second quantizes every block of every tensor.  The pages quantize one
 *   weight tensor at a time; this is a batching of that operation for a whole
 *   model's weights, where per-tensor launches and the latency of small
 *   tensors would otherwise dominate.
 * Arguments:
 *   tensors host array of `count` descriptors (read during the call only);
 *           each descriptor's W, rows, cols, codes, scales and alpha follow
 *           the rules of nvfp4_quantize.  Outputs of different tensors must
 *           not overlap each other or any W.
 *   count   >= 0 (0: nothing is enqueued).  Longer lists are processed in
 *           consecutive slices of NVFP4_GROUP_MAX tensors.  A list holding at
 *           least 4 x L2 bytes of bf16 is cut into parts of about 3 x L2
 *           that alternate between `stream` and a second stream owned by the
 *           library (forked from `stream` and joined back into it by events,
 *           so the call can be captured in a CUDA graph), letting one part's
 *           max|W| pass run on the same SMs as another part's quantize pass
 *           (which then leaves room for it on every SM).  The library
 *           keeps a small pool of such second streams per device: a call
 *           takes one that no other call holds and that is not part of an
 *           unfinished stream capture, so concurrent calls from several host
 *           threads, captured or not, never share one.
 *   mode, iters, stream  as for nvfp4_quantize.  Modes 2 and 3 run the
 *           nvfp4_quantize launch sequence tensor by tensor (their search and
 *           sweeps, not launches, dominate), tensors alternating between
 *           `stream` and the second stream.
 * Every descriptor is checked before anything is enqueued; the first bad one
 * decides the returned status.
 */
#define NVFP4_GROUP_MAX 256
typedef struct nvfp4_tensor {
  const void *W;
  int64_t rows;
  int64_t cols;
  uint8_t *codes;
  uint8_t *scales;
  float *alpha;
} nvfp4_tensor;
int nvfp4_quantize_grouped(const nvfp4_tensor *tensors, int count, int mode, int iters,
                           cudaStream_t stream);

/*
 * nvfp4_dequantize -- codes, scales, alpha -> bf16 out [rows, cols],
 *   out = bf16_rne(q * fl(alpha * Delta_i)).  [SOAR] dequantization equation;
 *   one path for every scale rule ([FOS] section 02: no kernel change).
 * Arguments: codes (device, 4-byte aligned, rows*cols/2 bytes), scales (device,
 *   rows*cols/16 bytes), alpha (device, 1 float), rows/cols as for
 *   nvfp4_quantize, out (device, bf16, 16-byte aligned, rows*cols elements,
 *   written), stream.
 * Returns an nvfp4_status.
 */
int nvfp4_dequantize(const uint8_t *codes, const uint8_t *scales, const float *alpha,
                     int64_t rows, int64_t cols, void *out, cudaStream_t stream);

/*
 * nvfp4_gemv -- the W4A16 product that consumes a quantized tensor:
 *   y[b][r] = sum_c What[r][c] * x[b][c] for b < batch, with What the
 *   dequantized weights exactly as nvfp4_dequantize writes them
 *   (bf16_rne(q * fl(alpha * Delta_i)), [SOAR] dequantization equation) and
 *   fp32 accumulation (each product of two bf16 values is exact; the sum's
 *   order is fixed, so results repeat bit for bit).  One kernel for every
 *   scale rule ([FOS] section 02: the dequantization path is unchanged).
 *   The pages quantize weights for such a decode kernel; the product itself
 *   is the consumer of the path, not a step of it.
 * Arguments:
 *   codes, scales, alpha  a quantized [rows, cols] tensor as nvfp4_quantize
 *          writes it (device; codes 8-byte aligned).
 *   rows, cols  as for nvfp4_quantize.
 *   x      device, bf16, 16-byte aligned, row-major [batch, cols].
 *   batch  1..8 activation vectors.
 *   y      device, fp32, 4-byte aligned, row-major [batch, rows] (written;
 *          zeros when cols == 0).
 *   stream cudaStream_t.
 * Returns an nvfp4_status.
 */
int nvfp4_gemv(const uint8_t *codes, const uint8_t *scales, const float *alpha, int64_t rows,
               int64_t cols, const void *x, int batch, float *y, cudaStream_t stream);

/*
 * nvfp4_gemm -- the same product as nvfp4_gemv for 1..256 activation vectors,
 *   on the tensor cores: the weights are dequantized (exactly as
 *   nvfp4_dequantize writes them) into shared memory and multiplied with
 *   bf16 x bf16 -> fp32 tcgen05 matrix multiplies.  The work (128-row tiles
 *   x 128-column steps) is cut into equal contiguous ranges, one per SM;
 *   the partial sums of a tile shared by several ranges are added in range
 *   order.  The tensor cores' fp32 accumulation order is the hardware's;
 *   results repeat bit for bit for the same shapes on the same GPU model.
 * Arguments as for nvfp4_gemv, with batch in 1..256.  Scratch for the
 *   partial sums comes from the library's pool (at most about
 *   4 * batch * 128 * (2 * rows / 128 + SMs) bytes).  Should an internal wait time out, the
 *   affected outputs are NaN.
 */
int nvfp4_gemm(const uint8_t *codes, const uint8_t *scales, const float *alpha, int64_t rows,
               int64_t cols, const void *x, int batch, float *y, cudaStream_t stream);

/*
 * nvfp4_swizzle_scales -- the E4M3 block scales of a quantized [rows, cols]
 *   tensor, from the linear [rows, cols/16] layout that nvfp4_quantize
 *   writes to the layout block-scaled tensor-core matrix multiplies read
 *   (NVFP4 x NVFP4 GEMM inputs, 16-element blocks, E4M3 scales): the scale
 *   matrix is padded with zeros to a multiple of 128 rows and 4 columns and
 *   cut into 128 x 4 tiles stored one after another, column tiles varying
 *   fastest; inside a tile the scale of row r (0..127) and column c (0..3)
 *   is byte (r % 32) * 16 + (r / 32) * 4 + c.  The pages store the scales as
 *   FP8 but fix no layout; this is the tensor-core one.  The codes need no
 *   change (two per byte, even element in the low nibble, rows contiguous).
 * Arguments: scales (device, rows*cols/16 bytes), rows/cols as for
 *   nvfp4_quantize, out (device, 4-byte aligned,
 *   nvfp4_swizzled_scales_bytes(rows, cols) bytes, written, padding zeroed),
 *   stream.
 * nvfp4_swizzled_scales_bytes returns that size, or -1 for an invalid shape.
 */
int64_t nvfp4_swizzled_scales_bytes(int64_t rows, int64_t cols);
int nvfp4_swizzle_scales(const uint8_t *scales, int64_t rows, int64_t cols, uint8_t *out,
                         cudaStream_t stream);

/*
 * nvfp4_encode_e2m1 -- element-wise fp32 -> E2M1 code (one code per output
 *   byte, sign in bit 3), rounding to nearest with ties to the even code and
 *   saturation at 6, exactly as the quantizer rounds x / (alpha * Delta).
 *   [FOS] section 01 value set; [SOAR] piecewise FP4 rounding.
 * Arguments: v (device, n floats), n >= 0, out (device, n bytes), stream.
 */
int nvfp4_encode_e2m1(const float *v, int64_t n, uint8_t *out, cudaStream_t stream);

/*
 * nvfp4_encode_e4m3 -- element-wise fp32 (>= 0) -> E4M3FN code, round to
 *   nearest even, saturating at 448, exactly as the quantizer rounds block
 *   scales.  [SOAR] quantizer equation (Q_E4M3, M_FP8 = 448).
 * Arguments: v (device, n floats), n >= 0, out (device, n bytes), stream.
 */
int nvfp4_encode_e4m3(const float *v, int64_t n, uint8_t *out, cudaStream_t stream);

/*
 * nvfp4_quantize_noalloc -- the max rule or FourOverSix (mode 0 or 1 only),
 *   with results identical to nvfp4_quantize, for callers that cannot let the
 *   library allocate device memory: serving engines that reserve nearly all
 *   device memory up front and account for every byte themselves,
 *   latency-critical threads that must never enter an allocator (it can
 *   block or reach the driver), and embedders whose own allocator must stay
 *   the only one in the process.  The method's pages have no counterpart:
 *   this is a deployment variant of the same computation.
 * It calls no cudaMalloc/cudaFree or any allocating routine.  Its scratch is a
 *   static device array of NVFP4_NOALLOC_SCRATCH_BYTES (16 KiB) that every GPU
 *   which loads the library holds until the process exits.
 * Limits and sharing:
 *   - rows*cols <= NVFP4_NOALLOC_MAX_ELEMS (2^28): one scratch slot per 65,536
 *     elements; larger tensors return NVFP4_ERR_INVALID_ARG before anything
 *     is enqueued.
 *   - Every call uses the same array.  Each call writes every slot it reads
 *     before reading it, so nothing needs clearing between calls, but calls
 *     that overlap on the GPU (e.g. on two streams) race on it and give wrong
 *     results: serialize them.
 *   - The first call on a device performs a one-time set-up with that device
 *     current (it looks up the array's device address); make that first call
 *     before any stream capture.  Under CUDA's lazy module loading (the
 *     default) that look-up can be what loads the library's device code onto
 *     the GPU, which allocates device memory (the array among it) and can
 *     then fail with NVFP4_ERR_OUT_OF_MEMORY: make the first call at start-up,
 *     before the caller reserves its memory.
 * Arguments, layouts, alignment and the other statuses are those of
 * nvfp4_quantize (without `iters`).
 */
#define NVFP4_NOALLOC_SCRATCH_BYTES 16384
#define NVFP4_NOALLOC_MAX_ELEMS (INT64_C(1) << 28)
int nvfp4_quantize_noalloc(const void *W, int64_t rows, int64_t cols, int mode, uint8_t *codes,
                           uint8_t *scales, float *alpha, cudaStream_t stream);

/*
 * Kernel tracing.  While enabled, every kernel the library launches is
 * bracketed by two CUDA events recorded on the stream it is launched on, so
 * per-kernel device time can be read back without an external profiler.
 * (No counterpart on the method's pages: this is instrumentation.)
 *   nvfp4_profiler_enable(on)  on != 0 starts recording, 0 stops (recorded
 *                              launches are kept).  Returns an nvfp4_status.
 *   nvfp4_profiler_reset()     forgets every record.
 *   nvfp4_profiler_kinds()     waits for the recorded events, folds them into
 *                              per-kernel totals and returns the number of
 *                              distinct kernels seen (< 0 on a CUDA error).
 *   nvfp4_profiler_get(i, name, name_len, launches, total_ms)
 *                              kernel i (0 <= i < kinds): its name (NUL-
 *                              terminated, truncated to name_len), launch
 *                              count and summed device milliseconds.
 * Host cost: about two cudaEventRecord calls per launch while enabled.
 */
int nvfp4_profiler_enable(int on);
int nvfp4_profiler_reset(void);
int nvfp4_profiler_kinds(void);
int nvfp4_profiler_get(int index, char *name, int name_len, int64_t *launches, double *total_ms);

/*
 * nvfp4_ffma_probe -- fp32 fused multiply-add throughput probe: launches one
 *   kernel on `stream` in which every resident thread of every SM runs
 *   independent FMA chains for `rounds` rounds (scalar fma.rn.f32 when
 *   packed == 0, packed fma.rn.f32x2 when packed == 1).  The caller times the
 *   launch (CUDA events on `stream`); 2 x *fmas / seconds is the fp32 peak at
 *   the clock the launch ran at.  (No counterpart on the method's pages: it
 *   gives the fp32-bound scale search its roofline.)
 * Arguments: packed 0 or 1; rounds 1..2^32; sink (device, 4-byte aligned,
 *   sink_floats floats, overwritten; at least 2048 x the SM count is always
 *   enough); fmas (host, written: FMAs the launch performs).
 */
int nvfp4_ffma_probe(int packed, int64_t rounds, float *sink, int64_t sink_floats, int64_t *fmas,
                     cudaStream_t stream);

/*
 * Test hooks.  No counterpart on the method's pages: they let tests drive the
 * library's failure paths without faulting anything.  Process-wide settings
 * that every later call sees; meant for test programs, not for use while other
 * calls are being made.
 *   nvfp4_test_fail_allocations(count): the next `count` scratch allocations
 *     fail as if the device were out of memory; a call that meets one returns
 *     NVFP4_ERR_OUT_OF_MEMORY with nothing enqueued.  count >= 0 (0 clears).
 *   nvfp4_test_first_wait_tries(tries): tries >= 0 makes the first bounded
 *     wait of every CTA of later launches give up after that many polls (0:
 *     at once): in nvfp4_quantize's bulk-copy max|W| pass (tensors larger
 *     than half of L2) the wait for the CTA's first copy, so alpha comes out
 *     NaN; in nvfp4_gemm the first wait of the MMA-issuing thread, so the
 *     outputs come out NaN.  Every copy and MMA already issued still
 *     completes before the CTA exits (those waits keep their normal limits).
 *     tries < 0 restores the normal limits.
 * Both return an nvfp4_status.
 */
int nvfp4_test_fail_allocations(int count);
int nvfp4_test_first_wait_tries(int64_t tries);

/*
 * Checked build.  The library compiled with -DNVFP4_CHECKED
 * (libnvfp4_gb300_checked.so) makes every hot-path kernel (max|W| passes,
 * max-rule / FourOverSix quantize, CJSO sweeps, decoupled search and its
 * deferred-block pass, grouped kernels, dequantize; so every quantize and
 * dequantize entry point, the allocation-free one included) test the index of its
 * global-memory and table accesses against the buffer's extent first: an
 * index outside is not accessed (the output it fed is then unspecified) and
 * the access's site is recorded, the first failure winning.  It is slower and
 * meant for tests; its results are otherwise the normal build's.
 *   nvfp4_checked_build(): 1 in the checked build, 0 in the normal one.
 *   nvfp4_check_take(site): waits for the current device to be idle, then
 *     moves the first recorded site into *site (host; 0: no failed check) and
 *     clears it.  Sites are kernel << 8 | access (0x01xx max|W|, 0x02xx
 *     quantize, 0x03xx CJSO sweep, 0x04xx search, 0x05xx deferred blocks,
 *     0x06xx dequantize, 0x07xx grouped, 0x0001 the self-test).  In the normal
 *     build it sets *site = 0.
 *   nvfp4_check_selftest(i, n, stream): one checked test of i against
 *     [0, n) that accesses nothing, so a test can see the mechanism record
 *     site 0x0001 (a no-op in the normal build).
 * Each returns an nvfp4_status.
 */
int nvfp4_checked_build(void);
int nvfp4_check_take(uint32_t *site);
int nvfp4_check_selftest(int64_t i, int64_t n, cudaStream_t stream);

/* Human-readable text for a status code (static storage, never NULL). */
const char *nvfp4_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_GB300_H */
