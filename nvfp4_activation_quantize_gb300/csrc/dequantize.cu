// dequantize.cu -- checking path: codes + swizzled E4M3 scales -> fp32.
//
// out = fl((E2M1value(c) * E4M3value(sf)) / gsf): the value a block-scaled
// NVFP4 GEMM with alpha = 1/gsf sees for the element.  The product is exact
// (2 x 4 significant bits), so there is one rounding, a correctly rounded
// division.  The value depends only on the code and the scale byte, so each
// CTA first tabulates it for all 16 codes x 128 scale values (8 KB of shared
// memory, one division per entry) and an element is then a table load.  One
// lane per 16-element block: an 8-byte code load, the scale byte from its
// swizzled position, two 256-bit stores of fp32.
#include "h3q_device.cuh"
#include "h3q_internal.h"

namespace h3q {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// E2M1 code (sign bit 3, magnitude index 0..7) -> binary32 value.
__device__ __forceinline__ float e2m1_value(uint32_t c) {
  const uint32_t m = c & 7u;
  uint32_t bits = m >= 2 ? (((m >> 1) + 126u) << 23) | ((m & 1u) << 22)
                         : (m == 1 ? 0x3f000000u : 0u);
  bits |= (c & 8u) << 28;
  return __uint_as_float(bits);
}

__global__ void __launch_bounds__(kThreads)
dequantize_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                  int64_t rows, int64_t cols, const float* __restrict__ gsf_ptr,
                  float* __restrict__ out) {
  // tab[sf * 16 + c] = fl((E2M1value(c) * E4M3value(sf)) / gsf); the decode
  // reads the scale byte's low seven bits (bit 7 is not part of the code)
  __shared__ float tab[128 * 16];
  const float gsf = *gsf_ptr;
  for (int i = threadIdx.x; i < 128 * 16; i += blockDim.x)
    tab[i] = __fdiv_rn(__fmul_rn(e2m1_value(static_cast<uint32_t>(i & 15)),
                                 e4m3_value(static_cast<uint32_t>(i >> 4))), gsf);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t groups = cols >> 4;
  const int64_t quads = cols >> 6;
  const int64_t segs = (groups + 31) >> 5;
  const int64_t total = rows * segs;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
  for (int64_t s = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); s < total;
       s += nwarps) {
    const int64_t row = s / segs;
    const int64_t g = (s - row * segs) * 32 + lane;
    if (g >= groups) continue;
    uint32_t lo, hi;
    asm volatile("ld.global.nc.v2.b32 {%0,%1}, [%2];"
                 : "=r"(lo), "=r"(hi)
                 : "l"(codes + row * (cols >> 1) + g * 8));
    const uint32_t sf = scales[scale_word_offset(row, g >> 2, quads) + (g & 3)];
    const float* row_tab = tab + (sf & 0x7fu) * 16;
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = row_tab[((i < 8 ? lo : hi) >> (4 * (i & 7))) & 15u];
    float* o = out + row * cols + g * kBlock;
    asm volatile("st.global.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(o), "f"(v[0]),
                 "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
                 : "memory");
    asm volatile("st.global.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(o + 8), "f"(v[8]),
                 "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]),
                 "f"(v[15])
                 : "memory");
  }
}

}  // namespace

cudaError_t launch_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t rows,
                              int64_t cols, const float* gsf, float* out, cudaStream_t stream) {
  const int64_t segs = (cols / 16 + 31) / 32;
  int blocks = 0;
  cudaError_t err = persistent_blocks(reinterpret_cast<const void*>(&dequantize_kernel), kThreads, 0,
                                      (rows * segs + kWarps - 1) / kWarps, &blocks);
  if (err != cudaSuccess) return err;
  dequantize_kernel<<<blocks, kThreads, 0, stream>>>(codes, scales, rows, cols, gsf, out);
  return cudaGetLastError();
}

}  // namespace h3q
