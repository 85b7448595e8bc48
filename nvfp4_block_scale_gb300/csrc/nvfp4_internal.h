// nvfp4_internal.h -- launchers shared between the kernels and the C ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime_api.h>
#include <vector_types.h>

namespace nvfp4 {

enum { kModeMax = 0, kModeFourOverSix = 1, kModeCjso = 2, kModeCjsoDecoupled = 3 };
constexpr int kMaxIters = 64;  // CJSO iterations per call at most (the alpha history holds kMaxIters + 1)
enum { kKernAmax = 0, kKernQuantMax, kKernQuantFos, kKernCjso, kKernDequant, kKernGroupAmax,
       kKernGroupQuantMax, kKernGroupQuantFos, kKernAmaxLdg, kKernCount };

// A group of tensors for the grouped max-rule / FourOverSix kernels, passed by
// value as the kernels' parameter.  Tensor t owns the virtual tiles
// [tile_begin[t], tile_begin[t+1]) of kGroupTile blocks each (its last tile
// may be partial; an empty tensor owns none).
constexpr int kGroupMax = 256;
constexpr int kGroupTile = 256;  // blocks per tile = threads per CTA of the quantize kernel
struct GroupTensor {
  const void *W;
  uint8_t *codes;
  uint8_t *scales;
  float *alpha;
  int64_t B;  // 16-element blocks
};
struct GroupArgs {
  int count;
  int64_t tile_begin[kGroupMax + 1];
  GroupTensor t[kGroupMax];
};

cudaError_t launch_amax_partials(const void *W, int64_t n16, uint32_t *part, int grid, cudaStream_t st);
cudaError_t launch_amax_bulk(const void *W, int64_t n16, uint32_t *part, int grid, long first_limit,
                             cudaStream_t st);
int amax_bulk_chunks(int64_t n16);
cudaError_t launch_quant_max_fos(int mode, const void *W, int64_t H, const uint32_t *amax_part, int n_amax,
                                 uint8_t *codes, uint8_t *scales, float *alpha, int grid, int ranged,
                                 cudaStream_t st);
// sums: form and write the partial sums of the next alpha step (false for the last sweep of a call)
cudaError_t launch_cjso_sweep(bool init, bool sums, const void *W, int64_t H, const uint32_t *amax_part,
                              int n_amax, const ulonglong2 *part_in, int n_in, ulonglong2 *part_out,
                              float *alpha_hist, int t, uint8_t *scales, uint8_t *codes, int write_codes,
                              float *alpha_out, int write_alpha, int grid, cudaStream_t st);
cudaError_t launch_decoupled(const void *W, int64_t B, const float *alpha_hist, int t, uint8_t *scales, uint8_t *codes,
                             uint32_t *defer_count, int64_t *defer_list, int defer_cap, int sms, cudaStream_t st);
constexpr int kDeferCap = 1 << 18;  // deferred blocks of one search (beyond it a lane searches inline)
cudaError_t launch_dequant(const uint8_t *codes, const uint8_t *scales, const float *alpha, int64_t H, void *out, int grid,
                    cudaStream_t st);
cudaError_t launch_encode_e2m1(const float *v, int64_t n, uint8_t *out, int grid, cudaStream_t st);
cudaError_t launch_encode_e4m3(const float *v, int64_t n, uint8_t *out, int grid, cudaStream_t st);
cudaError_t launch_group_amax(const GroupArgs &g, uint32_t *amax, int grid, cudaStream_t st);
cudaError_t launch_group_quant(int mode, const GroupArgs &g, const uint32_t *amax, int grid, cudaStream_t st);
cudaError_t launch_gemv(const uint8_t *codes, const uint8_t *scales, const float *alpha, int64_t rows, int64_t cols,
                        const void *x, int batch, float *y, int grid, cudaStream_t st);
int gemv_grid(int sms, int batch, int64_t rows, int64_t cols);
int gemv_max_active_ctas(int batch);
cudaError_t prepare_gemv_kernels();
cudaError_t launch_swizzle_scales(const uint8_t *scales, int64_t rows, int64_t kb, uint8_t *out,
                                  cudaStream_t st);
int gemm_tc_tile_n(int batch);
size_t gemm_tc_workspace_bytes(int64_t rows, int64_t cols, int batch, int sms);
cudaError_t launch_gemm_tc(const uint8_t *codes, const uint8_t *scales, const float *alpha, int64_t rows,
                           int64_t cols, const void *x, int batch, int sms, float *ws, float *y, int first_tries,
                           cudaStream_t st);
cudaError_t launch_gemm_tc_reduce(const float *ws, int64_t rows, int64_t cols, int batch, int sms, float *y,
                                  int grid, cudaStream_t st);
cudaError_t prepare_gemm_tc_kernels();
cudaError_t prepare_decoupled_kernel();
cudaError_t prepare_quant_kernels();
int max_active_ctas(int which);
// checked build (NVFP4_CHECKED): per translation unit, read and clear the
// first failed check's site into *site (if *site is 0); no-ops otherwise
cudaError_t check_take_kernels(uint32_t *site);
cudaError_t check_take_decoupled(uint32_t *site);
cudaError_t launch_check_selftest(int64_t i, int64_t n, cudaStream_t st);
int64_t ffma_probe_fmas_per_thread(int packed, int64_t rounds);
cudaError_t launch_ffma_probe(int packed, int64_t rounds, int grid, float *sink, cudaStream_t st);
int ffma_probe_threads();
int ffma_probe_occupancy(int packed);

}  // namespace nvfp4
