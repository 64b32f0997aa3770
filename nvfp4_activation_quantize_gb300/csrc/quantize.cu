// quantize.cu -- standalone NVFP4 quantize of a bf16 [rows, cols] tensor,
// e.g. the attention output viewed as [tokens, heads*head_dim].
//
// (TensorRT-LLM PR #21483, commit "...quantize it with a bandwidth-bound
// kernel": the stock quantize reads one row per block with one 16-byte load per
// thread and reaches a fifth of HBM bandwidth.)  Here the work is split into
// 512-column segments of a row: one warp, one segment, one 16-element block
// per lane, one 256-bit load per lane (1 KiB contiguous per warp).  Persistent
// warps walk the segments in an interleaved order so that neighbouring warps
// read neighbouring kilobytes.  The loop is software-pipelined: a warp issues
// the loads of its next kUnroll segments before it converts the kUnroll it
// holds, so 2 * kUnroll segments (4 KiB per warp) are in flight while it
// computes and HBM never waits for a warp's conversions (with the loads issued
// only after the previous step's stores the 65,280 x 7,168 launch took 0.186
// ms, 96% of the copy peak; pipelined it takes 0.177 ms).  The first step's
// loads go out before the prologue (the global scale and the inverse-scale
// table), so they are in flight while it runs.  A warp steps its
// (row, segment) positions incrementally, so no division runs per segment.
// Segments of the padding rows (rows..pad128(rows)-1) write zero scale words
// and read nothing.
#include <cfloat>

#include "h3q_device.cuh"
#include "h3q_internal.h"

namespace h3q {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 2;  // segments per step (a step's loads, then the previous step's conversions)

// The quantize of x, persistent over (row, 512-column segment) units.  DYN: the
// dynamic form.  The global scale is not read but formed here from the
// n_partials per-CTA maxima of the abs-max pass launched just before, whose
// completion this waits for (programmatic dependent launch: the CTAs start as the
// pass's CTAs finish and issue their first loads of x, which the pass does not
// write, before the wait); the first CTA also writes the scale to gsf_out.  The
// scale is the one h3q_global_scale_from_amax forms: fl(2688 / max), 1 for 0,
// +inf clamped to the largest finite binary32 first.  Each form has a kernel of
// its own, so the static one keeps its parameters and registers (63: four CTAs
// of 256 threads per SM; the dynamic one takes 64).
template <bool DYN>
__device__ __forceinline__ void quantize_rows(const uint16_t* __restrict__ x, int64_t ld, int64_t rows,
                                              int64_t cols, const float* __restrict__ gsf_ptr,
                                              uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                              const float* __restrict__ partials, int n_partials,
                                              float* __restrict__ gsf_out) {
  __shared__ float inv_table[128];

  const int lane = threadIdx.x & 31;
  const int64_t groups = cols >> 4;
  const int64_t quads = cols >> 6;
  const int64_t segs = (groups + 31) >> 5;
  const int64_t prows = (rows + 127) >> 7 << 7;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);

  // (row, segment) of the kUnroll segments this warp handles per step, and the
  // advance of one step (nwarps * kUnroll segments) in rows and segments.
  int64_t row[kUnroll], seg[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int64_t s = first + u * nwarps;
    row[u] = s / segs;
    seg[u] = s - row[u] * segs;
  }
  const int64_t adv_rows = nwarps * kUnroll / segs;
  const int64_t adv_segs = nwarps * kUnroll - adv_rows * segs;

  Block16 in[kUnroll];
  auto load_step = [&](Block16 (&dst)[kUnroll], const int64_t (&r)[kUnroll], const int64_t (&sg)[kUnroll]) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t g = sg[u] * 32 + lane;
      if (r[u] < rows && g < groups) {
        load_stream(x + r[u] * ld + g * kBlock, dst[u]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[u].w[i] = 0;
      }
    }
  };
  load_step(in, row, seg);  // the first loads are in flight during the prologue
  const float gsf = [&]() -> float {
    if constexpr (DYN) {
      asm volatile("griddepcontrol.wait;" ::: "memory");  // the abs-max pass has completed
      __shared__ float scratch[kWarps];
      float m = 0.0f;
      for (int i = threadIdx.x; i < n_partials; i += kThreads) m = fmaxf(m, partials[i]);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) scratch[threadIdx.x >> 5] = m;
      __syncthreads();
      float a = 0.0f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) a = fmaxf(a, scratch[w]);
      if (a > FLT_MAX) a = FLT_MAX;
      const float g = a == 0.0f ? 1.0f : __fdiv_rn(2688.0f, a);
      if (blockIdx.x == 0 && threadIdx.x == 0) *gsf_out = g;
      return g;
    } else {
      return *gsf_ptr;
    }
  }();
  fill_inverse_scales(inv_table, gsf);
  __syncthreads();
  while (row[0] < prows) {
    int64_t nrow[kUnroll], nseg[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      nrow[u] = row[u] + adv_rows;
      nseg[u] = seg[u] + adv_segs;
      if (nseg[u] >= segs) {
        nseg[u] -= segs;
        nrow[u] += 1;
      }
    }
    Block16 nxt[kUnroll];
    if (nrow[0] < prows) load_step(nxt, nrow, nseg);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (row[u] >= prows) break;  // warp-uniform
      const int64_t g = seg[u] * 32 + lane;
      const bool in_row = row[u] < rows;
      const bool in_cols = g < groups;
      Quantized q = quantize_block(in[u], gsf, inv_table);
      if (!in_row) q.sf = 0;
      if (in_row && in_cols)
        store_codes(codes + row[u] * (cols >> 1) + g * 8, q.codes_lo, q.codes_hi);
      store_scale_quad(scales, row[u], g, quads, q.sf, in_cols);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      row[u] = nrow[u];
      seg[u] = nseg[u];
      in[u] = nxt[u];
    }
  }
}


__global__ void __launch_bounds__(kThreads)
quantize_kernel(const uint16_t* __restrict__ x, int64_t ld, int64_t rows, int64_t cols,
                const float* __restrict__ gsf_ptr, uint8_t* __restrict__ codes,
                uint8_t* __restrict__ scales) {
  quantize_rows<false>(x, ld, rows, cols, gsf_ptr, codes, scales, nullptr, 0, nullptr);
}

__global__ void __launch_bounds__(kThreads)
quantize_dynamic_kernel(const uint16_t* __restrict__ x, int64_t ld, int64_t rows, int64_t cols,
                        const float* __restrict__ partials, int n_partials, float* __restrict__ gsf_out,
                        uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  quantize_rows<true>(x, ld, rows, cols, nullptr, codes, scales, partials, n_partials, gsf_out);
}

}  // namespace

cudaError_t launch_quantize(const uint16_t* x, int64_t ld, int64_t rows, int64_t cols,
                            const float* gsf, uint8_t* codes, uint8_t* scales,
                            cudaStream_t stream) {
  const int64_t segs = (cols / 16 + 31) / 32;
  const int64_t work = (rows + 127) / 128 * 128 * segs;
  int blocks = 0;
  cudaError_t err = persistent_blocks(reinterpret_cast<const void*>(&quantize_kernel), kThreads, 0,
                                      (work + kWarps - 1) / kWarps, &blocks);
  if (err != cudaSuccess) return err;
  quantize_kernel<<<blocks, kThreads, 0, stream>>>(x, ld, rows, cols, gsf, codes, scales);
  return cudaGetLastError();
}

cudaError_t launch_quantize_after_partials(const uint16_t* x, int64_t ld, int64_t rows, int64_t cols,
                                           const float* partials, int n_partials, float* gsf_out,
                                           uint8_t* codes, uint8_t* scales, cudaStream_t stream) {
  const int64_t segs = (cols / 16 + 31) / 32;
  const int64_t work = (rows + 127) / 128 * 128 * segs;
  int blocks = 0;
  cudaError_t err = persistent_blocks(reinterpret_cast<const void*>(&quantize_dynamic_kernel), kThreads, 0,
                                      (work + kWarps - 1) / kWarps, &blocks);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, quantize_dynamic_kernel, x, ld, rows, cols, partials, n_partials, gsf_out, codes,
                            scales);
}

}  // namespace h3q
