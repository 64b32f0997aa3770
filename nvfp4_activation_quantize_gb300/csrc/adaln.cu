// adaln.cu -- (a) RMSNorm with fp32 statistics + AdaLN modulation + NVFP4.
//
// (TensorRT-LLM PR #21483, summary and commit "...SwiGLU producers": the AdaLN
// RMSNorm + modulation kernel writes packed E2M1 codes and swizzled E4M3 block
// scales directly, so the bf16 activation is never written and re-read.
// FastVideo API page, introduction: fp32 statistics with sequential FMAs per
// thread, no contraction of products that eager rounds.)
//
// One warp owns one row.  Lane l owns the row's 16-element blocks l, l+32, ...
// (the canonical reduction order of the library is defined on exactly this
// assignment).  The lane loads all of its blocks with 256-bit streaming loads
// into registers (a 7,168-wide row is 14 blocks = 112 registers per lane), so
// the row is read from HBM once:
//   pass 1  eight fp32 partials per lane, fused multiply-adds element by
//           element (paired f32x2), then ((p0+p1)+(p2+p3))+((p4+p5)+(p6+p7))
//           and a butterfly over xor-distances 16, 8, 4, 2, 1;
//           rstd = fl(1 / fl(sqrt(fl(fl(ss / cols) + eps))))
//   pass 2  per block: y = bf16(fl(fl(fl(fl(x*rstd)*gamma)*fl(1+scale)) + shift))
//           from the registers, then the block quantize.
// gamma and the frame's modulation rows are read with L1-allocating loads: all
// rows of a frame share them, so they come from L1/L2, not HBM.
// Rows wider than the register budget take the same order in chunks of
// NB*32 blocks, re-reading x (from L2) in pass 2.
// Persistent warps take rows round-robin; warps on the padding rows
// rows..pad128(rows)-1 write their zero scale words.
#include "h3q_device.cuh"
#include "h3q_internal.h"

namespace h3q {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;

struct AdalnArgs {
  const uint16_t* x;
  int64_t ld;
  const uint16_t* gamma;
  const uint16_t* table;
  int64_t num_frames;
  const int32_t* row_frame;
  int64_t rows_per_frame;
  float eps;
  int64_t rows;
  int64_t cols;
  const float* gsf;
  uint8_t* codes;
  uint8_t* scales;
  float* row_rstd;
};

template <int NB>
__device__ __forceinline__ void load_blocks(const uint16_t* xr, int64_t first, int64_t groups,
                                            Block16 (&xb)[NB]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const int64_t g = first + b * 32 + lane;
    if (g < groups) {
      load_stream(xr + g * kBlock, xb[b]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) xb[b].w[i] = 0;
    }
  }
}

// Partials: acc[j] holds (p_2j, p_2j+1); element e of a block goes to p_(e%8).
template <int NB>
__device__ __forceinline__ void accumulate(const Block16 (&xb)[NB], float2 (&acc)[4]) {
#pragma unroll
  for (int b = 0; b < NB; ++b) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 v = bf16x2_to_float2(xb[b].w[4 * half + j]);
        acc[j] = __ffma2_rn(v, v, acc[j]);
      }
    }
  }
}

// Modulate and quantize NB blocks starting at block index `first` of the row.
template <int NB>
__device__ __forceinline__ void emit(const AdalnArgs& a, int64_t row, int64_t first,
                                     const Block16 (&xb)[NB], float rstd, const uint16_t* shift,
                                     const uint16_t* scale, float gsf) {
  const int lane = threadIdx.x & 31;
  const int64_t groups = a.cols >> 4;
  const int64_t quads = a.cols >> 6;
  const float2 rstd2 = make_float2(rstd, rstd);
  const float2 one2 = make_float2(1.0f, 1.0f);
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const int64_t g0 = first + b * 32;
    if (g0 >= groups) break;  // warp-uniform
    const int64_t g = g0 + lane;
    const bool active = g < groups;
    Block16 gm, sc, sh;
    if (active) {
      load_reused(a.gamma + g * kBlock, gm);
      load_reused(scale + g * kBlock, sc);
      load_reused(shift + g * kBlock, sh);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) gm.w[i] = sc.w[i] = sh.w[i] = 0;
    }
    Block16 y;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float2 n = __fmul2_rn(bf16x2_to_float2(xb[b].w[i]), rstd2);
      const float2 h = __fmul2_rn(n, bf16x2_to_float2(gm.w[i]));
      const float2 f = __fadd2_rn(one2, bf16x2_to_float2(sc.w[i]));
      const float2 m = __fmul2_rn(h, f);
      const float2 o = __fadd2_rn(m, bf16x2_to_float2(sh.w[i]));
      y.w[i] = float2_to_bf16x2(o);
    }
    const Quantized q = quantize_block(y, gsf);
    if (active) store_codes(a.codes + row * (a.cols >> 1) + g * 8, q.codes_lo, q.codes_hi);
    store_scale_quad(a.scales, row, g, quads, q.sf, active);
  }
}

template <int NB>
__global__ void __launch_bounds__(kThreads) adaln_kernel(const AdalnArgs a) {
  const float gsf = *a.gsf;
  const int lane = threadIdx.x & 31;
  const int64_t groups = a.cols >> 4;
  const int64_t quads = a.cols >> 6;
  const int64_t chunk = NB * 32;
  const int64_t prows = (a.rows + 127) >> 7 << 7;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;

  for (int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); row < prows;
       row += nwarps) {
    if (row >= a.rows) {
      for (int64_t g0 = 0; g0 < groups; g0 += 32)
        store_scale_quad(a.scales, row, g0 + lane, quads, 0u, g0 + lane < groups);
      continue;
    }
    int64_t t = a.row_frame ? static_cast<int64_t>(a.row_frame[row]) : row / a.rows_per_frame;
    t = t < 0 ? 0 : (t >= a.num_frames ? a.num_frames - 1 : t);  // memory safety only
    const uint16_t* shift = a.table + t * 2 * a.cols;
    const uint16_t* scale = shift + a.cols;
    const uint16_t* xr = a.x + row * a.ld;

    Block16 xb[NB];
    float2 acc[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j] = make_float2(0.0f, 0.0f);
    const bool resident = groups <= chunk;
    for (int64_t first = 0; first < groups; first += chunk) {
      load_blocks<NB>(xr, first, groups, xb);
      accumulate<NB>(xb, acc);
    }
    float ss = __fadd_rn(__fadd_rn(__fadd_rn(acc[0].x, acc[0].y), __fadd_rn(acc[1].x, acc[1].y)),
                         __fadd_rn(__fadd_rn(acc[2].x, acc[2].y), __fadd_rn(acc[3].x, acc[3].y)));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    const float mean = __fdiv_rn(ss, static_cast<float>(a.cols));
    const float rstd = __frcp_rn(__fsqrt_rn(__fadd_rn(mean, a.eps)));
    if (a.row_rstd && lane == 0) a.row_rstd[row] = rstd;

    if (resident) {
      emit<NB>(a, row, 0, xb, rstd, shift, scale, gsf);
    } else {
      for (int64_t first = 0; first < groups; first += chunk) {
        load_blocks<NB>(xr, first, groups, xb);
        emit<NB>(a, row, first, xb, rstd, shift, scale, gsf);
      }
    }
  }
}

template <int NB>
cudaError_t launch_nb(const AdalnArgs& a, cudaStream_t stream) {
  const int64_t prows = (a.rows + 127) / 128 * 128;
  int blocks = 0;
  cudaError_t err = persistent_blocks(reinterpret_cast<const void*>(&adaln_kernel<NB>), kThreads,
                                      (prows + kWarps - 1) / kWarps, &blocks);
  if (err != cudaSuccess) return err;
  adaln_kernel<NB><<<blocks, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_adaln(const uint16_t* x, int64_t ld, const uint16_t* gamma,
                         const uint16_t* table, int64_t num_frames, const int32_t* row_frame,
                         int64_t rows_per_frame, float eps, int64_t rows, int64_t cols,
                         const float* gsf, uint8_t* codes, uint8_t* scales, float* row_rstd,
                         cudaStream_t stream) {
  const AdalnArgs a{x,    ld,   gamma, table, num_frames, row_frame, rows_per_frame,
                    eps,  rows, cols,  gsf,   codes,      scales,    row_rstd};
  const int64_t per_lane = (cols / 16 + 31) / 32;  // blocks each lane owns
  if (per_lane <= 4) return launch_nb<4>(a, stream);
  if (per_lane <= 8) return launch_nb<8>(a, stream);
  if (per_lane <= 14) return launch_nb<14>(a, stream);
  return launch_nb<16>(a, stream);
}

}  // namespace h3q
