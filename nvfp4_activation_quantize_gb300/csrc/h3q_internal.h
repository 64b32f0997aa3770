// h3q_internal.h -- launchers behind the C ABI (not exported).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace h3q {

// The unique id (cuCtxGetId) of the CUDA context current on the calling thread,
// binding the current device's primary context first when the thread has none.
// Per-context state of the library (launch-size cache, host-call streams) is
// keyed on it: ids are never reused within a process, so state left behind by
// a context the caller destroyed is never taken for the new one's.
cudaError_t current_context_id(unsigned long long* id);

// Blocks to launch for a persistent kernel: every SM filled to the occupancy
// the kernel allows at `threads` threads and `smem_bytes` of dynamic shared
// memory per block, capped at `max_blocks`.  Raises the kernel's dynamic
// shared memory limit when smem_bytes needs it.  Cached per context, kernel
// and launch shape.
cudaError_t persistent_blocks(const void* kernel, int threads, int smem_bytes, int64_t max_blocks,
                              int* blocks);

cudaError_t launch_quantize(const uint16_t* x, int64_t ld, int64_t rows, int64_t cols,
                            const float* gsf, uint8_t* codes, uint8_t* scales, cudaStream_t stream);

cudaError_t launch_adaln(const uint16_t* x, int64_t ld, const uint16_t* gamma,
                         const uint16_t* table, int64_t num_frames, const int32_t* row_frame,
                         int64_t rows_per_frame, float eps, int64_t rows, int64_t cols,
                         const float* gsf, uint8_t* codes, uint8_t* scales, float* row_rstd,
                         cudaStream_t stream);

cudaError_t launch_swiglu(const uint16_t* gate, int64_t ld_gate, const uint16_t* up,
                          int64_t ld_up, int64_t rows, int64_t cols, const float* gsf,
                          uint8_t* codes, uint8_t* scales, cudaStream_t stream);

// Abs-max passes (dynamic and calibrated scales): fold max |y| of the producer's
// bf16 output y into *amax (which must hold a value >= 0) without storing y.
cudaError_t launch_amax_bf16(const uint16_t* x, int64_t ld, int64_t rows, int64_t cols,
                             float* amax, cudaStream_t stream);
cudaError_t launch_adaln_amax(const uint16_t* x, int64_t ld, const uint16_t* gamma,
                              const uint16_t* table, int64_t num_frames, const int32_t* row_frame,
                              int64_t rows_per_frame, float eps, int64_t rows, int64_t cols,
                              float* amax, float* row_rstd, cudaStream_t stream);
// The AdaLN producer with each row's rstd given (an abs-max pass's row_rstd).
cudaError_t launch_adaln_from_rstd(const uint16_t* x, int64_t ld, const uint16_t* gamma, const uint16_t* table,
                                   int64_t num_frames, const int32_t* row_frame, int64_t rows_per_frame,
                                   const float* rstd, int64_t rows, int64_t cols, const float* gsf,
                                   uint8_t* codes, uint8_t* scales, cudaStream_t stream);
cudaError_t launch_swiglu_amax(const uint16_t* gate, int64_t ld_gate, const uint16_t* up,
                               int64_t ld_up, int64_t rows, int64_t cols, float* amax,
                               cudaStream_t stream);
// *gsf = fl(2688 / *amax), 1 for amax = 0, +inf clamped to the largest float.
cudaError_t launch_global_scale(const float* amax, float* gsf, cudaStream_t stream);

// Dynamic quantize without caller scratch: per-CTA partial maxima in a
// file-scope device array of kMaxDynamicPartials floats.  dynamic_scale_partials
// gives the number of CTAs (partials) the abs-max pass launches for a shape;
// launch_dynamic_partials runs that pass (and returns the array's address);
// launch_quantize_after_partials then quantizes with the scale it forms from the
// partial maxima (written to gsf_out too), launched as a programmatic dependent of
// the pass.
constexpr int kMaxDynamicPartials = 4096;
cudaError_t dynamic_scale_partials(int64_t rows, int64_t cols, int* blocks);
cudaError_t launch_dynamic_partials(const uint16_t* x, int64_t ld, int64_t rows, int64_t cols, int blocks,
                                    const float** partials, cudaStream_t stream);
cudaError_t launch_quantize_after_partials(const uint16_t* x, int64_t ld, int64_t rows, int64_t cols,
                                           const float* partials, int n_partials, float* gsf_out,
                                           uint8_t* codes, uint8_t* scales, cudaStream_t stream);

// Residual fold + RMSNorm + AdaLN -> NVFP4 (rows of at most 8,192 columns).
cudaError_t launch_residual_adaln(float* h, int64_t ld_h, const uint16_t* o, int64_t ld_o,
                                  const uint16_t* bias, const uint16_t* gate, const uint16_t* gamma,
                                  const uint16_t* table, int64_t num_frames,
                                  const int32_t* row_frame, int64_t rows_per_frame, float eps,
                                  int64_t rows, int64_t cols, const float* gsf, uint8_t* codes,
                                  uint8_t* scales, float* row_rstd, cudaStream_t stream);

// SwiGLU of a value-first packed projection o [rows, 2f] (value o[:, :f], gate
// o[:, f:]) with its bias [2f] (or NULL) not yet added.
cudaError_t launch_swiglu_packed(const uint16_t* o, int64_t ld_o, const uint16_t* bias, int64_t rows,
                                 int64_t f, const float* gsf, uint8_t* codes, uint8_t* scales,
                                 cudaStream_t stream);

cudaError_t launch_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t rows,
                              int64_t cols, const float* gsf, float* out, cudaStream_t stream);

// QKV epilogue over q, k, v (index 0, 1, 2): bias, per-head RMSNorm and RoPE
// (rotate-half pairs, or interleaved pairs when `interleaved`) on q and k, bias
// on v; head_dim in {64, 128, 256}.
cudaError_t launch_qkv_epilogue(const uint16_t* const x[3], const int64_t ld[3],
                                const uint16_t* const bias[3], uint16_t* const out[3],
                                const uint16_t* cos, const uint16_t* sin, int64_t rot, int interleaved,
                                int64_t rows, int64_t heads, int64_t head_dim, float eps,
                                cudaStream_t stream);

// Block-scaled NVFP4 GEMM acc = A B^T (A [m, k], B [n, k], E2M1 codes and 128x4
// E4M3 scales) on the tensor cores with the SwiGLU + NVFP4 epilogue: column 2j
// of acc is the value and 2j + 1 the gate of output j.  k % 256 == 0,
// n % 256 == 0; y (bf16 [m, n/2]) and acc (fp32 [m, n]) are optional outputs.
cudaError_t launch_gemm_swiglu(const uint8_t* a, const uint8_t* sfa, int64_t m, int64_t k, const uint8_t* b,
                               const uint8_t* sfb, int64_t n, const float* alpha, const float* gsf,
                               uint8_t* codes, uint8_t* scales, uint16_t* y, float* acc, cudaStream_t stream);
// Reads and clears the flag a kernel sets when one of its bounded waits ran out
// (synchronous); the GEMM is the library's kernel with such waits.
cudaError_t gemm_error_flag(int* flag);

// RMSNorm + AdaLN -> NVFP4 on host buffers// RMSNorm + AdaLN -> NVFP4 on host buffers (x in, codes and scales out), the
// copies pipelined with the producer over chunk_rows-row chunks; `workspace`
// holds h3q_host_workspace_bytes(chunk_rows, cols, rows, row_frame == nullptr)
// bytes of device memory (include/h3q.h), 256-byte aligned.
cudaError_t launch_adaln_host(const uint16_t* x_host, int64_t rows, int64_t cols, const uint16_t* gamma,
                              const uint16_t* table, int64_t num_frames, const int32_t* row_frame,
                              int64_t rows_per_frame, float eps, const float* gsf, uint8_t* codes_host,
                              uint8_t* scales_host, uint8_t* workspace, int64_t chunk_rows,
                              cudaStream_t stream);

}  // namespace h3q
