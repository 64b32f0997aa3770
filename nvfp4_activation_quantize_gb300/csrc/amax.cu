// amax.cu -- dynamic and calibrated global scales.
//
// (FastVideo API page, NVFP4DecoderLinear: a dynamic layer scales each call by
// the abs-max of its input, and calibration folds each call's abs-max into a
// running maximum; FlashRT PR #142, commit "...amax pipeline": the abs-max is
// taken on the device in a pass of its own, read by the quantize pass with no
// host synchronisation.)
//
// amax_bf16_kernel folds max |x| over a bf16 [rows, cols] tensor into *amax;
// the producers' own abs-max passes live beside them (adaln.cu, swiglu.cu).
// global_scale_kernel turns an abs-max into the global scale fl(2688 / amax),
// with 0 -> 1 and +inf clamped to the largest finite binary32 first.
#include <cfloat>

#include "h3q_device.cuh"
#include "h3q_internal.h"

namespace h3q {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;

// Warp per 512-column segment, lane per 16-element block, as in the quantize.
__global__ void __launch_bounds__(kThreads)
amax_bf16_kernel(const uint16_t* __restrict__ x, int64_t ld, int64_t rows, int64_t cols,
                 float* __restrict__ amax) {
  __shared__ float scratch[32];
  const int lane = threadIdx.x & 31;
  const int64_t groups = cols >> 4;
  const int64_t segs = (groups + 31) >> 5;
  const int64_t total = rows * segs;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
  float m = 0.0f;
  for (int64_t s0 = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); s0 < total;
       s0 += nwarps * kUnroll) {
    Block16 in[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t s = s0 + u * nwarps;
      const int64_t row = s / segs;
      const int64_t g = (s - row * segs) * 32 + lane;
      if (s < total && g < groups) {
        load_stream(x + row * ld + g * kBlock, in[u]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) in[u].w[i] = 0;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) m = fmaxf(m, block_amax(in[u]));
  }
  commit_amax(m, amax, scratch);
}

__global__ void global_scale_kernel(const float* __restrict__ amax, float* __restrict__ gsf) {
  float a = *amax;
  if (a > FLT_MAX) a = FLT_MAX;
  *gsf = a == 0.0f ? 1.0f : __fdiv_rn(2688.0f, a);
}

// --- dynamic quantize without caller scratch -----------------------------------

// Per-CTA partial maxima of h3q_quantize_nvfp4_dynamic: a file-scope device
// array, so the call needs no scratch from the caller and allocates nothing.
// One array per context (the module's copy); calls that overlap on the device share it.
__device__ __align__(256) float g_partial_amax[kMaxDynamicPartials];

// Each CTA writes its own max |x| to partial[blockIdx.x] (no atomics, nothing to
// zero beforehand).
__global__ void __launch_bounds__(kThreads)
amax_partials_kernel(const uint16_t* __restrict__ x, int64_t ld, int64_t rows, int64_t cols,
                     float* __restrict__ partial) {
  // the quantize launched after this pass (programmatic dependent launch) may start
  // as this grid's CTAs finish; it waits for the grid's completion before it
  // reads the partial maxima
  asm volatile("griddepcontrol.launch_dependents;");
  __shared__ float scratch[32];
  const int lane = threadIdx.x & 31;
  const int64_t groups = cols >> 4;
  const int64_t segs = (groups + 31) >> 5;
  const int64_t total = rows * segs;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
  float m = 0.0f;
  for (int64_t s0 = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); s0 < total;
       s0 += nwarps * kUnroll) {
    Block16 in[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t s = s0 + u * nwarps;
      const int64_t row = s / segs;
      const int64_t g = (s - row * segs) * 32 + lane;
      if (s < total && g < groups) {
        load_stream(x + row * ld + g * kBlock, in[u]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) in[u].w[i] = 0;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) m = fmaxf(m, block_amax(in[u]));
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) scratch[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float v = 0.0f;
    for (int w = 0; w < kWarps; ++w) v = fmaxf(v, scratch[w]);
    partial[blockIdx.x] = v;
  }
}

}  // namespace

cudaError_t dynamic_scale_partials(int64_t rows, int64_t cols, int* blocks) {
  const int64_t segs = (cols / 16 + 31) / 32;
  return persistent_blocks(reinterpret_cast<const void*>(&amax_partials_kernel), kThreads, 0,
                           (rows * segs + kWarps - 1) / kWarps, blocks);
}

cudaError_t launch_dynamic_partials(const uint16_t* x, int64_t ld, int64_t rows, int64_t cols, int blocks,
                                    const float** partials, cudaStream_t stream) {
  // The device address of the scratch array in the current context.  It is
  // looked up on every call (a lookup, no allocation): a cached address would
  // point into a context the caller may since have destroyed, or into another
  // context's copy of the module.
  void* address = nullptr;
  cudaError_t err = cudaGetSymbolAddress(&address, g_partial_amax);
  if (err != cudaSuccess) return err;
  float* partial = static_cast<float*>(address);
  amax_partials_kernel<<<blocks, kThreads, 0, stream>>>(x, ld, rows, cols, partial);
  *partials = partial;
  return cudaGetLastError();
}

cudaError_t launch_amax_bf16(const uint16_t* x, int64_t ld, int64_t rows, int64_t cols,
                             float* amax, cudaStream_t stream) {
  const int64_t segs = (cols / 16 + 31) / 32;
  int blocks = 0;
  cudaError_t err = persistent_blocks(reinterpret_cast<const void*>(&amax_bf16_kernel), kThreads, 0,
                                      (rows * segs + kWarps - 1) / kWarps, &blocks);
  if (err != cudaSuccess) return err;
  amax_bf16_kernel<<<blocks, kThreads, 0, stream>>>(x, ld, rows, cols, amax);
  return cudaGetLastError();
}

cudaError_t launch_global_scale(const float* amax, float* gsf, cudaStream_t stream) {
  global_scale_kernel<<<1, 1, 0, stream>>>(amax, gsf);
  return cudaGetLastError();
}

}  // namespace h3q
