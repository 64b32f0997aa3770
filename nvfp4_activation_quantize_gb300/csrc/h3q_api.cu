// h3q_api.cu -- the exported C ABI (include/h3q.h): host-side validation, then
// one kernel launch on the caller's stream.  No allocation, no synchronisation.
// An argument that breaks the contract returns H3Q_ERR_INVALID_ARGUMENT before
// any CUDA call, so these checks also run on machines without a GPU.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include <cuda.h>  // driver types only; the two driver calls are fetched at run time

#include "../../include/h3q.h"
#include "h3q_internal.h"

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int invalid(const char* fn, const char* what) {
  return fail(H3Q_ERR_INVALID_ARGUMENT, "%s: %s", fn, what);
}

int cuda_failed(const char* fn, cudaError_t err) {
  return fail(H3Q_ERR_CUDA, "%s: CUDA error %d (%s): %s", fn, static_cast<int>(err),
              cudaGetErrorName(err), cudaGetErrorString(err));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

constexpr int64_t kMaxCols = int64_t(1) << 24;
constexpr int64_t kMaxRows = int64_t(1) << 40;

// Byte range [p, p + n) of a buffer, for overlap checks.
struct Span {
  uintptr_t lo, hi;
};
Span span(const void* p, int64_t bytes) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return {lo, lo + static_cast<uintptr_t>(bytes)};
}
bool overlap(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi; }

// Bytes spanned by a bf16 [rows, cols] view with row stride ld.
int64_t view_bytes(int64_t rows, int64_t cols, int64_t ld) { return ((rows - 1) * ld + cols) * 2; }

// Shared shape checks; returns 0 or an error code (message already set).
int check_shape(const char* fn, int64_t rows, int64_t cols) {
  if (rows < 0) return invalid(fn, "rows must be >= 0");
  if (rows > kMaxRows) return invalid(fn, "rows exceeds 2^40");
  if (cols <= 0 || cols % 64 != 0) return invalid(fn, "cols must be a positive multiple of 64");
  if (cols > kMaxCols) return invalid(fn, "cols exceeds 2^24");
  return 0;
}

int check_input(const char* fn, const char* name, const void* p, int64_t ld, int64_t rows,
                int64_t cols) {
  char msg[160];
  if (p == nullptr) return snprintf(msg, sizeof msg, "%s is NULL", name), invalid(fn, msg);
  if (!aligned(p, 32)) return snprintf(msg, sizeof msg, "%s must be 32-byte aligned", name), invalid(fn, msg);
  if (ld < cols || ld % 16 != 0)
    return snprintf(msg, sizeof msg, "ld of %s must be >= cols and a multiple of 16", name), invalid(fn, msg);
  if (ld > (int64_t(1) << 62) / (rows > 0 ? rows : 1))
    return snprintf(msg, sizeof msg, "%s: rows * ld overflows", name), invalid(fn, msg);
  return 0;
}

int check_outputs(const char* fn, const uint8_t* codes, const uint8_t* scales,
                  const float* gsf) {
  if (codes == nullptr || scales == nullptr) return invalid(fn, "codes and scales must not be NULL");
  if (!aligned(codes, 16) || !aligned(scales, 16))
    return invalid(fn, "codes and scales must be 16-byte aligned");
  if (gsf == nullptr || !aligned(gsf, 4)) return invalid(fn, "global_scale must be a 4-byte aligned pointer");
  return 0;
}

// --- per-context, per-kernel launch-size cache ------------------------------

// A kernel whose attributes a runtime call can query: the query loads the
// library's module into the current context, which binds the device's primary
// context to the calling thread when none is current.
__global__ void context_probe_kernel() {}

struct OccupancyEntry {
  const void* kernel;
  unsigned long long context;
  int threads;
  int smem_bytes;
  int blocks_per_sm;
  int sms;
};
constexpr int kOccEntries = 256;
std::mutex g_occ_mutex;
OccupancyEntry g_occ[kOccEntries];
int g_occ_n = 0;
int g_occ_next = 0;

}  // namespace

namespace h3q {

cudaError_t current_context_id(unsigned long long* id) {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static std::once_flag once;
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult found;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &found) ==
            cudaSuccess && found == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &found) ==
            cudaSuccess && found == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
  });
  if (get_current == nullptr || get_id == nullptr) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  if (ctx == nullptr) {  // no context on this thread yet: let the runtime bind the primary one
    cudaFuncAttributes attr;
    cudaError_t err = cudaFuncGetAttributes(&attr, reinterpret_cast<const void*>(&context_probe_kernel));
    if (err != cudaSuccess) return err;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
  }
  return get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}

cudaError_t persistent_blocks(const void* kernel, int threads, int smem_bytes, int64_t max_blocks,
                              int* blocks) {
  int device = 0;
  cudaError_t err = cudaGetDevice(&device);
  if (err != cudaSuccess) return err;
  // Keyed on the context, not the device ordinal: the shared-memory limit set
  // below belongs to the context, and a context the caller re-creates (after
  // cudaDeviceReset, say) starts without it.
  unsigned long long context = 0;
  if ((err = current_context_id(&context)) != cudaSuccess) return err;
  int per_sm = 0, sms = 0;
  {
    std::lock_guard<std::mutex> lock(g_occ_mutex);
    for (int i = 0; i < g_occ_n; ++i)
      if (g_occ[i].kernel == kernel && g_occ[i].context == context && g_occ[i].threads == threads &&
          g_occ[i].smem_bytes == smem_bytes) {
        per_sm = g_occ[i].blocks_per_sm;
        sms = g_occ[i].sms;
      }
  }
  if (per_sm == 0) {
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (err != cudaSuccess) return err;
    if (smem_bytes > 0) {  // the default limit leaves no room beside static shared memory
      err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
      if (err != cudaSuccess) return err;
    }
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem_bytes);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    std::lock_guard<std::mutex> lock(g_occ_mutex);
    if (g_occ_n < kOccEntries) {
      g_occ[g_occ_n++] = {kernel, context, threads, smem_bytes, per_sm, sms};
    } else {  // full (many contexts over the process's life): reuse the slots in turn
      g_occ[g_occ_next] = {kernel, context, threads, smem_bytes, per_sm, sms};
      g_occ_next = (g_occ_next + 1) % kOccEntries;
    }
  }
  int64_t n = static_cast<int64_t>(per_sm) * sms;
  if (max_blocks < n) n = max_blocks;
  *blocks = static_cast<int>(n < 1 ? 1 : n);
  return cudaSuccess;
}

}  // namespace h3q

extern "C" {

const char* h3q_last_error(void) { return g_last_error.c_str(); }

int h3q_abi_version(void) { return H3Q_ABI_VERSION; }

int h3q_quantize_nvfp4(const void* x, int64_t ld_x, int64_t rows, int64_t cols,
                       const float* global_scale, uint8_t* codes, uint8_t* scales,
                       void* stream) {
  static const char* fn = "h3q_quantize_nvfp4";
  g_last_error.clear();
  if (int e = check_shape(fn, rows, cols)) return e;
  if (rows == 0) return H3Q_OK;
  if (int e = check_input(fn, "x", x, ld_x, rows, cols)) return e;
  if (int e = check_outputs(fn, codes, scales, global_scale)) return e;
  const Span in = span(x, view_bytes(rows, cols, ld_x));
  const Span c = span(codes, h3q_code_bytes(rows, cols));
  const Span s = span(scales, h3q_scale_bytes(rows, cols));
  if (overlap(in, c) || overlap(in, s) || overlap(c, s)) return invalid(fn, "outputs overlap an input or each other");
  cudaError_t err = h3q::launch_quantize(static_cast<const uint16_t*>(x), ld_x, rows, cols,
                                         global_scale, codes, scales,
                                         static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? H3Q_OK : cuda_failed(fn, err);
}

int h3q_rmsnorm_adaln_nvfp4(const void* x, int64_t ld_x, const void* gamma, const void* mod_table,
                            int64_t num_frames, const int32_t* row_frame, int64_t rows_per_frame,
                            float eps, int64_t rows, int64_t cols, const float* global_scale,
                            uint8_t* codes, uint8_t* scales, float* row_rstd, void* stream) {
  static const char* fn = "h3q_rmsnorm_adaln_nvfp4";
  g_last_error.clear();
  if (int e = check_shape(fn, rows, cols)) return e;
  if (!std::isfinite(eps) || eps < 0.0f) return invalid(fn, "eps must be finite and >= 0");
  if (num_frames < 1) return invalid(fn, "num_frames must be >= 1");
  if (num_frames > (int64_t(1) << 31)) return invalid(fn, "num_frames exceeds 2^31");
  if (rows == 0) return H3Q_OK;
  if (int e = check_input(fn, "x", x, ld_x, rows, cols)) return e;
  if (int e = check_input(fn, "gamma", gamma, cols, 1, cols)) return e;
  if (int e = check_input(fn, "mod_table", mod_table, cols, 2 * num_frames, cols)) return e;
  if (int e = check_outputs(fn, codes, scales, global_scale)) return e;
  if (row_frame != nullptr) {
    if (!aligned(row_frame, 4)) return invalid(fn, "row_frame must be 4-byte aligned");
  } else {
    if (rows_per_frame < 1) return invalid(fn, "rows_per_frame must be >= 1 when row_frame is NULL");
    if ((rows - 1) / rows_per_frame >= num_frames)
      return invalid(fn, "rows / rows_per_frame reaches past the modulation table");
  }
  if (row_rstd != nullptr && !aligned(row_rstd, 4)) return invalid(fn, "row_rstd must be 4-byte aligned");
  const Span c = span(codes, h3q_code_bytes(rows, cols));
  const Span s = span(scales, h3q_scale_bytes(rows, cols));
  const Span ins[4] = {span(x, view_bytes(rows, cols, ld_x)), span(gamma, cols * 2),
                       span(mod_table, num_frames * 4 * cols),
                       row_frame ? span(row_frame, rows * 4) : Span{0, 0}};
  if (overlap(c, s)) return invalid(fn, "codes and scales overlap");
  for (const Span& in : ins)
    if (overlap(in, c) || overlap(in, s)) return invalid(fn, "an output overlaps an input");
  if (row_rstd != nullptr) {
    const Span r = span(row_rstd, rows * 4);
    if (overlap(r, c) || overlap(r, s)) return invalid(fn, "row_rstd overlaps an output");
    for (const Span& in : ins)
      if (overlap(in, r)) return invalid(fn, "row_rstd overlaps an input");
  }
  cudaError_t err = h3q::launch_adaln(
      static_cast<const uint16_t*>(x), ld_x, static_cast<const uint16_t*>(gamma),
      static_cast<const uint16_t*>(mod_table), num_frames, row_frame, rows_per_frame, eps, rows,
      cols, global_scale, codes, scales, row_rstd, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? H3Q_OK : cuda_failed(fn, err);
}

int h3q_rmsnorm_adaln_nvfp4_from_rstd(const void* x, int64_t ld_x, const void* gamma, const void* mod_table,
                                      int64_t num_frames, const int32_t* row_frame, int64_t rows_per_frame,
                                      const float* row_rstd, int64_t rows, int64_t cols,
                                      const float* global_scale, uint8_t* codes, uint8_t* scales, void* stream) {
  static const char* fn = "h3q_rmsnorm_adaln_nvfp4_from_rstd";
  g_last_error.clear();
  if (int e = check_shape(fn, rows, cols)) return e;
  if (num_frames < 1) return invalid(fn, "num_frames must be >= 1");
  if (num_frames > (int64_t(1) << 31)) return invalid(fn, "num_frames exceeds 2^31");
  if (rows == 0) return H3Q_OK;
  if (int e = check_input(fn, "x", x, ld_x, rows, cols)) return e;
  if (int e = check_input(fn, "gamma", gamma, cols, 1, cols)) return e;
  if (int e = check_input(fn, "mod_table", mod_table, cols, 2 * num_frames, cols)) return e;
  if (int e = check_outputs(fn, codes, scales, global_scale)) return e;
  if (row_frame != nullptr) {
    if (!aligned(row_frame, 4)) return invalid(fn, "row_frame must be 4-byte aligned");
  } else {
    if (rows_per_frame < 1) return invalid(fn, "rows_per_frame must be >= 1 when row_frame is NULL");
    if ((rows - 1) / rows_per_frame >= num_frames)
      return invalid(fn, "rows / rows_per_frame reaches past the modulation table");
  }
  if (row_rstd == nullptr) return invalid(fn, "row_rstd is NULL");
  if (!aligned(row_rstd, 4)) return invalid(fn, "row_rstd must be 4-byte aligned");
  const Span c = span(codes, h3q_code_bytes(rows, cols));
  const Span s = span(scales, h3q_scale_bytes(rows, cols));
  const Span ins[5] = {span(x, view_bytes(rows, cols, ld_x)), span(gamma, cols * 2),
                       span(mod_table, num_frames * 4 * cols),
                       row_frame ? span(row_frame, rows * 4) : Span{0, 0}, span(row_rstd, rows * 4)};
  if (overlap(c, s)) return invalid(fn, "codes and scales overlap");
  for (const Span& in : ins)
    if (overlap(in, c) || overlap(in, s)) return invalid(fn, "an output overlaps an input");
  cudaError_t err = h3q::launch_adaln_from_rstd(
      static_cast<const uint16_t*>(x), ld_x, static_cast<const uint16_t*>(gamma),
      static_cast<const uint16_t*>(mod_table), num_frames, row_frame, rows_per_frame, row_rstd, rows, cols,
      global_scale, codes, scales, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? H3Q_OK : cuda_failed(fn, err);
}

int h3q_swiglu_nvfp4(const void* gate, int64_t ld_gate, const void* up, int64_t ld_up,
                     int64_t rows, int64_t cols, const float* global_scale, uint8_t* codes,
                     uint8_t* scales, void* stream) {
  static const char* fn = "h3q_swiglu_nvfp4";
  g_last_error.clear();
  if (int e = check_shape(fn, rows, cols)) return e;
  if (rows == 0) return H3Q_OK;
  if (int e = check_input(fn, "gate", gate, ld_gate, rows, cols)) return e;
  if (int e = check_input(fn, "up", up, ld_up, rows, cols)) return e;
  if (int e = check_outputs(fn, codes, scales, global_scale)) return e;
  const Span g = span(gate, view_bytes(rows, cols, ld_gate));
  const Span u = span(up, view_bytes(rows, cols, ld_up));
  const Span c = span(codes, h3q_code_bytes(rows, cols));
  const Span s = span(scales, h3q_scale_bytes(rows, cols));
  if (overlap(g, c) || overlap(g, s) || overlap(u, c) || overlap(u, s) || overlap(c, s))
    return invalid(fn, "outputs overlap an input or each other");
  cudaError_t err = h3q::launch_swiglu(static_cast<const uint16_t*>(gate), ld_gate,
                                       static_cast<const uint16_t*>(up), ld_up, rows, cols,
                                       global_scale, codes, scales,
                                       static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? H3Q_OK : cuda_failed(fn, err);
}

int h3q_residual_rmsnorm_adaln_nvfp4(float* h, int64_t ld_h, const void* o, int64_t ld_o,
                                     const void* bias, const void* gate_table, const void* gamma,
                                     const void* mod_table, int64_t num_frames,
                                     const int32_t* row_frame, int64_t rows_per_frame, float eps,
                                     int64_t rows, int64_t cols, const float* global_scale,
                                     uint8_t* codes, uint8_t* scales, float* row_rstd,
                                     void* stream) {
  static const char* fn = "h3q_residual_rmsnorm_adaln_nvfp4";
  g_last_error.clear();
  if (int e = check_shape(fn, rows, cols)) return e;
  if (cols > 8192) return invalid(fn, "cols exceeds 8,192");
  if (!std::isfinite(eps) || eps < 0.0f) return invalid(fn, "eps must be finite and >= 0");
  if (num_frames < 1) return invalid(fn, "num_frames must be >= 1");
  if (num_frames > (int64_t(1) << 31)) return invalid(fn, "num_frames exceeds 2^31");
  if (rows == 0) return H3Q_OK;
  if (h == nullptr || !aligned(h, 32)) return invalid(fn, "h must be a 32-byte aligned pointer");
  if (ld_h < cols || ld_h % 8 != 0) return invalid(fn, "ld of h must be >= cols and a multiple of 8");
  if (ld_h > (int64_t(1) << 61) / rows) return invalid(fn, "h: rows * ld overflows");
  if (int e = check_input(fn, "o", o, ld_o, rows, cols)) return e;
  if (bias != nullptr)
    if (int e = check_input(fn, "bias", bias, cols, 1, cols)) return e;
  if (int e = check_input(fn, "gate_table", gate_table, cols, num_frames, cols)) return e;
  if (int e = check_input(fn, "gamma", gamma, cols, 1, cols)) return e;
  if (int e = check_input(fn, "mod_table", mod_table, cols, 2 * num_frames, cols)) return e;
  if (int e = check_outputs(fn, codes, scales, global_scale)) return e;
  if (row_frame != nullptr) {
    if (!aligned(row_frame, 4)) return invalid(fn, "row_frame must be 4-byte aligned");
  } else {
    if (rows_per_frame < 1) return invalid(fn, "rows_per_frame must be >= 1 when row_frame is NULL");
    if ((rows - 1) / rows_per_frame >= num_frames)
      return invalid(fn, "rows / rows_per_frame reaches past the modulation table");
  }
  if (row_rstd != nullptr && !aligned(row_rstd, 4)) return invalid(fn, "row_rstd must be 4-byte aligned");
  const Span hs = span(h, ((rows - 1) * ld_h + cols) * 4);
  const Span c = span(codes, h3q_code_bytes(rows, cols));
  const Span sc = span(scales, h3q_scale_bytes(rows, cols));
  const Span r = row_rstd ? span(row_rstd, rows * 4) : Span{0, 0};
  const Span ins[7] = {span(o, view_bytes(rows, cols, ld_o)), bias ? span(bias, cols * 2) : Span{0, 0},
                       span(gate_table, num_frames * 2 * cols), span(gamma, cols * 2),
                       span(mod_table, num_frames * 4 * cols),
                       row_frame ? span(row_frame, rows * 4) : Span{0, 0}, span(global_scale, 4)};
  const Span outs[4] = {hs, c, sc, r};
  for (int i = 0; i < 4; ++i) {
    for (const Span& in : ins)
      if (overlap(outs[i], in)) return invalid(fn, "an output (h, codes, scales, row_rstd) overlaps an input");
    for (int k = i + 1; k < 4; ++k)
      if (overlap(outs[i], outs[k])) return invalid(fn, "outputs overlap each other");
  }
  cudaError_t err = h3q::launch_residual_adaln(
      h, ld_h, static_cast<const uint16_t*>(o), ld_o, static_cast<const uint16_t*>(bias),
      static_cast<const uint16_t*>(gate_table), static_cast<const uint16_t*>(gamma),
      static_cast<const uint16_t*>(mod_table), num_frames, row_frame, rows_per_frame, eps, rows,
      cols, global_scale, codes, scales, row_rstd, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? H3Q_OK : cuda_failed(fn, err);
}

// --- dynamic and calibrated scales ------------------------------------------

namespace {
int check_amax(const char* fn, const float* amax) {
  if (amax == nullptr || !aligned(amax, 4)) return invalid(fn, "amax must be a 4-byte aligned pointer");
  return 0;
}
}  // namespace

int h3q_amax_bf16(const void* x, int64_t ld_x, int64_t rows, int64_t cols, float* amax,
                  void* stream) {
  static const char* fn = "h3q_amax_bf16";
  g_last_error.clear();
  if (int e = check_shape(fn, rows, cols)) return e;
  if (rows == 0) return H3Q_OK;
  if (int e = check_input(fn, "x", x, ld_x, rows, cols)) return e;
  if (int e = check_amax(fn, amax)) return e;
  if (overlap(span(x, view_bytes(rows, cols, ld_x)), span(amax, 4))) return invalid(fn, "amax overlaps x");
  cudaError_t err = h3q::launch_amax_bf16(static_cast<const uint16_t*>(x), ld_x, rows, cols, amax,
                                          static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? H3Q_OK : cuda_failed(fn, err);
}

int h3q_rmsnorm_adaln_amax(const void* x, int64_t ld_x, const void* gamma, const void* mod_table,
                           int64_t num_frames, const int32_t* row_frame, int64_t rows_per_frame,
                           float eps, int64_t rows, int64_t cols, float* amax, float* row_rstd,
                           void* stream) {
  static const char* fn = "h3q_rmsnorm_adaln_amax";
  g_last_error.clear();
  if (int e = check_shape(fn, rows, cols)) return e;
  if (!std::isfinite(eps) || eps < 0.0f) return invalid(fn, "eps must be finite and >= 0");
  if (num_frames < 1) return invalid(fn, "num_frames must be >= 1");
  if (num_frames > (int64_t(1) << 31)) return invalid(fn, "num_frames exceeds 2^31");
  if (rows == 0) return H3Q_OK;
  if (int e = check_input(fn, "x", x, ld_x, rows, cols)) return e;
  if (int e = check_input(fn, "gamma", gamma, cols, 1, cols)) return e;
  if (int e = check_input(fn, "mod_table", mod_table, cols, 2 * num_frames, cols)) return e;
  if (int e = check_amax(fn, amax)) return e;
  if (row_frame != nullptr) {
    if (!aligned(row_frame, 4)) return invalid(fn, "row_frame must be 4-byte aligned");
  } else {
    if (rows_per_frame < 1) return invalid(fn, "rows_per_frame must be >= 1 when row_frame is NULL");
    if ((rows - 1) / rows_per_frame >= num_frames)
      return invalid(fn, "rows / rows_per_frame reaches past the modulation table");
  }
  const Span am = span(amax, 4);
  const Span ins[4] = {span(x, view_bytes(rows, cols, ld_x)), span(gamma, cols * 2),
                       span(mod_table, num_frames * 4 * cols),
                       row_frame ? span(row_frame, rows * 4) : Span{0, 0}};
  for (const Span& in : ins)
    if (overlap(am, in)) return invalid(fn, "amax overlaps an input");
  if (row_rstd != nullptr) {
    if (!aligned(row_rstd, 4)) return invalid(fn, "row_rstd must be 4-byte aligned");
    const Span r = span(row_rstd, rows * 4);
    if (overlap(r, am)) return invalid(fn, "row_rstd overlaps amax");
    for (const Span& in : ins)
      if (overlap(r, in)) return invalid(fn, "row_rstd overlaps an input");
  }
  cudaError_t err = h3q::launch_adaln_amax(
      static_cast<const uint16_t*>(x), ld_x, static_cast<const uint16_t*>(gamma),
      static_cast<const uint16_t*>(mod_table), num_frames, row_frame, rows_per_frame, eps, rows,
      cols, amax, row_rstd, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? H3Q_OK : cuda_failed(fn, err);
}

int h3q_swiglu_amax(const void* gate, int64_t ld_gate, const void* up, int64_t ld_up,
                    int64_t rows, int64_t cols, float* amax, void* stream) {
  static const char* fn = "h3q_swiglu_amax";
  g_last_error.clear();
  if (int e = check_shape(fn, rows, cols)) return e;
  if (rows == 0) return H3Q_OK;
  if (int e = check_input(fn, "gate", gate, ld_gate, rows, cols)) return e;
  if (int e = check_input(fn, "up", up, ld_up, rows, cols)) return e;
  if (int e = check_amax(fn, amax)) return e;
  const Span am = span(amax, 4);
  if (overlap(am, span(gate, view_bytes(rows, cols, ld_gate))) ||
      overlap(am, span(up, view_bytes(rows, cols, ld_up))))
    return invalid(fn, "amax overlaps an input");
  cudaError_t err = h3q::launch_swiglu_amax(static_cast<const uint16_t*>(gate), ld_gate,
                                            static_cast<const uint16_t*>(up), ld_up, rows, cols,
                                            amax, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? H3Q_OK : cuda_failed(fn, err);
}

int h3q_global_scale_from_amax(const float* amax, float* global_scale, void* stream) {
  static const char* fn = "h3q_global_scale_from_amax";
  g_last_error.clear();
  if (int e = check_amax(fn, amax)) return e;
  if (global_scale == nullptr || !aligned(global_scale, 4))
    return invalid(fn, "global_scale must be a 4-byte aligned pointer");
  cudaError_t err = h3q::launch_global_scale(amax, global_scale, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? H3Q_OK : cuda_failed(fn, err);
}

int h3q_quantize_nvfp4_dynamic(const void* x, int64_t ld_x, int64_t rows, int64_t cols,
                               float* global_scale, uint8_t* codes, uint8_t* scales,
                               void* stream) {
  static const char* fn = "h3q_quantize_nvfp4_dynamic";
  g_last_error.clear();
  if (int e = check_shape(fn, rows, cols)) return e;
  if (rows == 0) return H3Q_OK;
  if (int e = check_input(fn, "x", x, ld_x, rows, cols)) return e;
  if (int e = check_outputs(fn, codes, scales, global_scale)) return e;
  const Span in = span(x, view_bytes(rows, cols, ld_x));
  const Span c = span(codes, h3q_code_bytes(rows, cols));
  const Span s = span(scales, h3q_scale_bytes(rows, cols));
  const Span g = span(global_scale, 4);
  if (overlap(in, c) || overlap(in, s) || overlap(c, s) || overlap(g, in) || overlap(g, c) ||
      overlap(g, s))
    return invalid(fn, "outputs overlap an input or each other");
  int blocks = 0;
  cudaError_t err = h3q::dynamic_scale_partials(rows, cols, &blocks);
  if (err != cudaSuccess) return cuda_failed(fn, err);
  if (blocks > h3q::kMaxDynamicPartials)
    return fail(H3Q_ERR_INVALID_ARGUMENT, "%s: the abs-max pass needs %d partial maxima, more than "
                "the %d the static scratch holds", fn, blocks, h3q::kMaxDynamicPartials);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float* partials = nullptr;
  err = h3q::launch_dynamic_partials(static_cast<const uint16_t*>(x), ld_x, rows, cols, blocks, &partials, st);
  if (err != cudaSuccess) return cuda_failed(fn, err);
  err = h3q::launch_quantize_after_partials(static_cast<const uint16_t*>(x), ld_x, rows, cols, partials, blocks,
                                            global_scale, codes, scales, st);
  return err == cudaSuccess ? H3Q_OK : cuda_failed(fn, err);
}

int h3q_gemm_swiglu_nvfp4(const uint8_t* a_codes, const uint8_t* a_scales, int64_t m, int64_t k,
                          const uint8_t* b_codes, const uint8_t* b_scales, int64_t n, const float* alpha,
                          const float* global_scale, uint8_t* codes, uint8_t* scales, void* y, float* acc,
                          void* stream) {
  static const char* fn = "h3q_gemm_swiglu_nvfp4";
  g_last_error.clear();
  if (m < 0) return invalid(fn, "m must be >= 0");
  if (m > (int64_t(1) << 31) - 128) return invalid(fn, "m exceeds 2^31 - 128");
  if (k <= 0 || k % 256 != 0 || k > kMaxCols) return invalid(fn, "k must be a positive multiple of 256, at most 2^24");
  if (n <= 0 || n % 256 != 0 || n > kMaxCols) return invalid(fn, "n must be a positive multiple of 256, at most 2^24");
  if (m == 0) return H3Q_OK;
  if (a_codes == nullptr || b_codes == nullptr || a_scales == nullptr || b_scales == nullptr)
    return invalid(fn, "a_codes, a_scales, b_codes and b_scales must not be NULL");
  if (!aligned(a_codes, 16) || !aligned(b_codes, 16) || !aligned(a_scales, 16) || !aligned(b_scales, 16))
    return invalid(fn, "a_codes, a_scales, b_codes and b_scales must be 16-byte aligned");
  if (alpha == nullptr || !aligned(alpha, 4)) return invalid(fn, "alpha must be a 4-byte aligned pointer");
  if (int e = check_outputs(fn, codes, scales, global_scale)) return e;
  if ((y != nullptr && !aligned(y, 16)) || (acc != nullptr && !aligned(acc, 16)))
    return invalid(fn, "y and acc must be 16-byte aligned (or NULL)");
  const int64_t f = n / 2;
  const Span in[] = {span(a_codes, m * (k / 2)), span(a_scales, h3q_scale_bytes(m, k)),
                     span(b_codes, n * (k / 2)), span(b_scales, h3q_scale_bytes(n, k)), span(alpha, 4),
                     span(global_scale, 4)};
  const Span out[] = {span(codes, h3q_code_bytes(m, f)), span(scales, h3q_scale_bytes(m, f)),
                      y ? span(y, m * f * 2) : Span{0, 0}, acc ? span(acc, m * n * 4) : Span{0, 0}};
  for (int i = 0; i < 4; ++i) {
    for (const Span& x : in)
      if (overlap(out[i], x)) return invalid(fn, "outputs overlap an input");
    for (int j = 0; j < i; ++j)
      if (overlap(out[i], out[j])) return invalid(fn, "outputs overlap each other");
  }
  cudaError_t err = h3q::launch_gemm_swiglu(a_codes, a_scales, m, k, b_codes, b_scales, n, alpha, global_scale,
                                            codes, scales, static_cast<uint16_t*>(y), acc,
                                            static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? H3Q_OK : cuda_failed(fn, err);
}

int h3q_kernel_error_flag(int* flag) {
  static const char* fn = "h3q_kernel_error_flag";
  g_last_error.clear();
  if (flag == nullptr) return invalid(fn, "flag must not be NULL");
  cudaError_t err = h3q::gemm_error_flag(flag);
  return err == cudaSuccess ? H3Q_OK : cuda_failed(fn, err);
}

int h3q_swiglu_packed_nvfp4(const void* o, int64_t ld_o, const void* bias, int64_t rows,
                            int64_t f, const float* global_scale, uint8_t* codes, uint8_t* scales,
                            void* stream) {
  static const char* fn = "h3q_swiglu_packed_nvfp4";
  g_last_error.clear();
  if (int e = check_shape(fn, rows, f)) return e;
  if (rows == 0) return H3Q_OK;
  if (int e = check_input(fn, "o", o, ld_o, rows, 2 * f)) return e;
  if (bias != nullptr)
    if (int e = check_input(fn, "bias", bias, 2 * f, 1, 2 * f)) return e;
  if (int e = check_outputs(fn, codes, scales, global_scale)) return e;
  const Span in = span(o, view_bytes(rows, 2 * f, ld_o));
  const Span b = bias ? span(bias, 4 * f) : Span{0, 0};
  const Span c = span(codes, h3q_code_bytes(rows, f));
  const Span s = span(scales, h3q_scale_bytes(rows, f));
  if (overlap(in, c) || overlap(in, s) || overlap(b, c) || overlap(b, s) || overlap(c, s))
    return invalid(fn, "outputs overlap an input or each other");
  cudaError_t err = h3q::launch_swiglu_packed(static_cast<const uint16_t*>(o), ld_o,
                                              static_cast<const uint16_t*>(bias), rows, f,
                                              global_scale, codes, scales,
                                              static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? H3Q_OK : cuda_failed(fn, err);
}

int h3q_dequantize_nvfp4(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t cols,
                         const float* global_scale, float* out, void* stream) {
  static const char* fn = "h3q_dequantize_nvfp4";
  g_last_error.clear();
  if (int e = check_shape(fn, rows, cols)) return e;
  if (rows == 0) return H3Q_OK;
  if (codes == nullptr || scales == nullptr || out == nullptr)
    return invalid(fn, "codes, scales and out must not be NULL");
  if (!aligned(codes, 16) || !aligned(scales, 16)) return invalid(fn, "codes and scales must be 16-byte aligned");
  if (!aligned(out, 32)) return invalid(fn, "out must be 32-byte aligned");
  if (global_scale == nullptr || !aligned(global_scale, 4))
    return invalid(fn, "global_scale must be a 4-byte aligned pointer");
  const Span o = span(out, rows * cols * 4);
  if (overlap(o, span(codes, h3q_code_bytes(rows, cols))) ||
      overlap(o, span(scales, h3q_scale_bytes(rows, cols))))
    return invalid(fn, "out overlaps an input");
  cudaError_t err = h3q::launch_dequantize(codes, scales, rows, cols, global_scale, out,
                                           static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? H3Q_OK : cuda_failed(fn, err);
}

int h3q_qkv_epilogue(const void* q, int64_t ld_q, const void* k, int64_t ld_k, const void* v,
                     int64_t ld_v, const void* bias_q, const void* bias_k, const void* bias_v,
                     const void* cos, const void* sin, int64_t rot, int interleaved, int64_t rows,
                     int64_t heads, int64_t head_dim, float eps, void* q_out, void* k_out,
                     void* v_out, void* stream) {
  static const char* fn = "h3q_qkv_epilogue";
  g_last_error.clear();
  if (rows < 0) return invalid(fn, "rows must be >= 0");
  if (rows > kMaxRows) return invalid(fn, "rows exceeds 2^40");
  if (heads < 1) return invalid(fn, "heads must be >= 1");
  if (head_dim != 64 && head_dim != 128 && head_dim != 256)
    return invalid(fn, "head_dim must be 64, 128 or 256");
  if (heads > kMaxCols / head_dim) return invalid(fn, "heads * head_dim exceeds 2^24");
  if (rot < 0 || rot > head_dim || rot % 16 != 0)
    return invalid(fn, "rot must be a multiple of 16 in [0, head_dim]");
  if (interleaved != 0 && interleaved != 1) return invalid(fn, "interleaved must be 0 or 1");
  if (!std::isfinite(eps) || eps < 0.0f) return invalid(fn, "eps must be finite and >= 0");
  if (rows == 0) return H3Q_OK;
  const int64_t d = heads * head_dim;
  const void* xs[3] = {q, k, v};
  const int64_t lds[3] = {ld_q, ld_k, ld_v};
  const void* bs[3] = {bias_q, bias_k, bias_v};
  void* outs[3] = {q_out, k_out, v_out};
  static const char* xn[3] = {"q", "k", "v"};
  static const char* bn[3] = {"bias_q", "bias_k", "bias_v"};
  for (int i = 0; i < 3; ++i) {
    if (int e = check_input(fn, xn[i], xs[i], lds[i], rows, d)) return e;
    if (int e = check_input(fn, bn[i], bs[i], d, 1, d)) return e;
    if (outs[i] == nullptr || !aligned(outs[i], 16))
      return invalid(fn, "q_out, k_out and v_out must be 16-byte aligned and not NULL");
  }
  if (rot > 0) {
    if (cos == nullptr || sin == nullptr) return invalid(fn, "cos and sin must not be NULL when rot > 0");
    if (!aligned(cos, 16) || !aligned(sin, 16)) return invalid(fn, "cos and sin must be 16-byte aligned");
  }
  Span ins[8];
  int n_in = 0;
  for (int i = 0; i < 3; ++i) {
    ins[n_in++] = span(xs[i], view_bytes(rows, d, lds[i]));
    ins[n_in++] = span(bs[i], d * 2);
  }
  if (rot > 0) {
    ins[n_in++] = span(cos, rows * rot * 2);
    ins[n_in++] = span(sin, rows * rot * 2);
  }
  Span os[3];
  for (int i = 0; i < 3; ++i) os[i] = span(outs[i], rows * d * 2);
  for (int i = 0; i < 3; ++i) {
    for (int j = 0; j < n_in; ++j)
      if (overlap(os[i], ins[j])) return invalid(fn, "outputs overlap an input or each other");
    for (int j = i + 1; j < 3; ++j)
      if (overlap(os[i], os[j])) return invalid(fn, "outputs overlap an input or each other");
  }
  const uint16_t* x16[3];
  const uint16_t* b16[3];
  uint16_t* o16[3];
  for (int i = 0; i < 3; ++i) {
    x16[i] = static_cast<const uint16_t*>(xs[i]);
    b16[i] = static_cast<const uint16_t*>(bs[i]);
    o16[i] = static_cast<uint16_t*>(outs[i]);
  }
  cudaError_t err = h3q::launch_qkv_epilogue(
      x16, lds, b16, o16, static_cast<const uint16_t*>(cos), static_cast<const uint16_t*>(sin), rot,
      interleaved, rows, heads, head_dim, eps, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? H3Q_OK : cuda_failed(fn, err);
}

int h3q_rmsnorm_adaln_nvfp4_host(const void* x_host, int64_t rows, int64_t cols, const void* gamma,
                                 const void* mod_table, int64_t num_frames, const int32_t* row_frame,
                                 int64_t rows_per_frame, float eps, const float* global_scale,
                                 uint8_t* codes_host, uint8_t* scales_host, void* workspace,
                                 int64_t workspace_bytes, int64_t chunk_rows, void* stream) {
  static const char* fn = "h3q_rmsnorm_adaln_nvfp4_host";
  g_last_error.clear();
  if (int e = check_shape(fn, rows, cols)) return e;
  if (!std::isfinite(eps) || eps < 0.0f) return invalid(fn, "eps must be finite and >= 0");
  if (num_frames < 1) return invalid(fn, "num_frames must be >= 1");
  if (num_frames > (int64_t(1) << 31)) return invalid(fn, "num_frames exceeds 2^31");
  if (chunk_rows <= 0 || chunk_rows % 128 != 0) return invalid(fn, "chunk_rows must be a positive multiple of 128");
  if (chunk_rows > (int64_t(1) << 40) / cols) return invalid(fn, "chunk_rows * cols is too large");
  if (rows == 0) return H3Q_OK;
  if (x_host == nullptr || codes_host == nullptr || scales_host == nullptr)
    return invalid(fn, "x_host, codes_host and scales_host must not be NULL");
  if (int e = check_input(fn, "gamma", gamma, cols, 1, cols)) return e;
  if (int e = check_input(fn, "mod_table", mod_table, cols, 2 * num_frames, cols)) return e;
  if (global_scale == nullptr || !aligned(global_scale, 4))
    return invalid(fn, "global_scale must be a 4-byte aligned pointer");
  if (row_frame != nullptr) {
    if (!aligned(row_frame, 4)) return invalid(fn, "row_frame must be 4-byte aligned");
  } else {
    if (rows_per_frame < 1) return invalid(fn, "rows_per_frame must be >= 1 when row_frame is NULL");
    if ((rows - 1) / rows_per_frame >= num_frames)
      return invalid(fn, "rows / rows_per_frame reaches past the modulation table");
  }
  if (workspace == nullptr || !aligned(workspace, 256)) return invalid(fn, "workspace must be 256-byte aligned");
  if (workspace_bytes < h3q_host_workspace_bytes(chunk_rows, cols, rows, row_frame == nullptr))
    return invalid(fn, "workspace_bytes is below h3q_host_workspace_bytes");
  const Span xs = span(x_host, rows * cols * 2);
  const Span c = span(codes_host, h3q_code_bytes(rows, cols));
  const Span s = span(scales_host, h3q_scale_bytes(rows, cols));
  if (overlap(xs, c) || overlap(xs, s) || overlap(c, s))
    return invalid(fn, "host outputs overlap the input or each other");
  const Span ws = span(workspace, workspace_bytes);
  const Span dev_ins[4] = {span(gamma, cols * 2), span(mod_table, num_frames * 4 * cols),
                           span(global_scale, 4), row_frame ? span(row_frame, rows * 4) : Span{0, 0}};
  for (const Span& in : dev_ins)
    if (overlap(in, ws)) return invalid(fn, "workspace overlaps a device input");
  cudaError_t err = h3q::launch_adaln_host(
      static_cast<const uint16_t*>(x_host), rows, cols, static_cast<const uint16_t*>(gamma),
      static_cast<const uint16_t*>(mod_table), num_frames, row_frame, rows_per_frame, eps, global_scale,
      codes_host, scales_host, static_cast<uint8_t*>(workspace), chunk_rows,
      static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? H3Q_OK : cuda_failed(fn, err);
}

}  // extern "C"
