// quantize.cu -- (c) standalone NVFP4 quantize of a bf16 [rows, cols] tensor,
// e.g. the attention output viewed as [tokens, heads*head_dim].
//
// (TensorRT-LLM PR #21483, commit "...quantize it with a bandwidth-bound
// kernel": the stock quantize reads one row per block with one 16-byte load per
// thread and reaches a fifth of HBM bandwidth.)  Here the work is split into
// 512-column segments of a row: one warp, one segment, one 16-element block
// per lane, one 256-bit load per lane (1 KiB contiguous per warp).  Persistent
// warps walk the segments in an interleaved order so that neighbouring warps
// read neighbouring kilobytes, and each warp keeps kUnroll segments' loads in
// flight before it converts any of them.  Segments of the padding rows
// (rows..pad128(rows)-1) write zero scale words and read nothing.
#include "h3q_device.cuh"
#include "h3q_internal.h"

namespace h3q {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kThreads)
quantize_kernel(const uint16_t* __restrict__ x, int64_t ld, int64_t rows, int64_t cols,
                const float* __restrict__ gsf_ptr, uint8_t* __restrict__ codes,
                uint8_t* __restrict__ scales) {
  const float gsf = *gsf_ptr;
  const int lane = threadIdx.x & 31;
  const int64_t groups = cols >> 4;
  const int64_t quads = cols >> 6;
  const int64_t segs = (groups + 31) >> 5;
  const int64_t total = ((rows + 127) >> 7 << 7) * segs;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;

  for (int64_t s = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); s < total;
       s += nwarps * kUnroll) {
    Block16 in[kUnroll];
    int64_t row[kUnroll], grp[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t su = s + u * nwarps;
      row[u] = su / segs;
      grp[u] = (su - row[u] * segs) * 32 + lane;
      if (su < total && row[u] < rows && grp[u] < groups) {
        load_stream(x + row[u] * ld + grp[u] * kBlock, in[u]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) in[u].w[i] = 0;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (s + u * nwarps >= total) break;  // warp-uniform
      const bool in_row = row[u] < rows;
      const bool in_cols = grp[u] < groups;
      Quantized q = quantize_block(in[u], gsf);
      if (!in_row) q.sf = 0;
      if (in_row && in_cols)
        store_codes(codes + row[u] * (cols >> 1) + grp[u] * 8, q.codes_lo, q.codes_hi);
      store_scale_quad(scales, row[u], grp[u], quads, q.sf, in_cols);
    }
  }
}

}  // namespace

cudaError_t launch_quantize(const uint16_t* x, int64_t ld, int64_t rows, int64_t cols,
                            const float* gsf, uint8_t* codes, uint8_t* scales,
                            cudaStream_t stream) {
  const int64_t segs = (cols / 16 + 31) / 32;
  const int64_t work = (rows + 127) / 128 * 128 * segs;
  int blocks = 0;
  cudaError_t err = persistent_blocks(reinterpret_cast<const void*>(&quantize_kernel), kThreads,
                                      (work + kWarps - 1) / kWarps, &blocks);
  if (err != cudaSuccess) return err;
  quantize_kernel<<<blocks, kThreads, 0, stream>>>(x, ld, rows, cols, gsf, codes, scales);
  return cudaGetLastError();
}

}  // namespace h3q
