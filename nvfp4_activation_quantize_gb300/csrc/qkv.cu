// qkv.cu -- QKV epilogue: bias + per-head RMSNorm + partial rotate-half RoPE.
//
// (FastVideo API page, qkv_epilogue: projected q/k/v [M, H*HD] bf16 with the
// bias not yet added -> roped q, k and biased v, each [M, H, HD]; cos/sin are
// bf16 [M, ROT], the eager path's cos.to(query.dtype).  FastVideo commit log:
// the q/k norm + partial RoPE kernel, with int64 indexing.)
//
//   x' = bf16(fl(x + b))                                   q, k and v (v stops here)
//   per head of q and k: ss over the head's HD = 128 values of x' in the
//   canonical order (chunk c of the head on lane c, eight fmaf partials, the
//   lane total, a butterfly over the 16 lanes), rstd = fl(1/fl(sqrt(fl(fl(ss/128)
//   + eps)))), n = bf16(fl(x' * rstd));
//   out_i = bf16(fl(bf16(fl(n_i cos_i)) + bf16(fl(r_i sin_i)))) for i < ROT with
//   r_i = -n_{i+ROT/2} (i < ROT/2), n_{i-ROT/2} (otherwise); out_i = n_i beyond.
//
// A warp covers 32 / (HD/8) heads at a time (two heads of 128: lanes 0-15 the
// first, 16-31 the second), one 8-element chunk per lane; the head's reduction
// is a butterfly inside its lanes, and the rotate-half partner of chunk c is
// chunk c +- ROT/16 of the same head, one shuffle away.  Persistent warps take
// one (row, tensor) unit at a time and walk its heads in batches whose loads
// are all in flight together.  Every element is read once and written once
// (6 + 6 bytes per element of the three tensors), so the kernel is bound by HBM
// bandwidth.
#include "h3q_device.cuh"
#include "h3q_internal.h"

namespace h3q {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct QkvArgs {
  const uint16_t* x[3];  // q, k, v
  int64_t ld[3];
  const uint16_t* bias[3];
  uint16_t* out[3];
  const uint16_t* cos;  // [rows, rot]
  const uint16_t* sin;
  int64_t rot;
  int interleaved;  // RoPE pairs (2j, 2j+1) instead of (i, i + ROT/2)
  int64_t rows;
  int64_t heads;
  float eps;
};

// bf16 pair w with its sign bits flipped: the exact negation of both values.
__device__ __forceinline__ uint32_t neg_bf16x2(uint32_t w) { return w ^ 0x80008000u; }

// The interleaved rotation partner of a bf16 pair (n_2j, n_2j+1): (-n_2j+1, n_2j).
__device__ __forceinline__ uint32_t rot_pair_bf16x2(uint32_t w) {
  return __byte_perm(w, 0, 0x1032) ^ 0x00008000u;
}

// x' = bf16(fl(x + b)) for the eight values of a chunk (one bf16x2 add per
// pair: the same bits, see add_bf16x2).
__device__ __forceinline__ void biased(const uint4& xw, const uint4& bw, uint32_t* xb) {
  xb[0] = add_bf16x2(xw.x, bw.x);
  xb[1] = add_bf16x2(xw.y, bw.y);
  xb[2] = add_bf16x2(xw.z, bw.z);
  xb[3] = add_bf16x2(xw.w, bw.w);
}

// One (row, tensor) unit: the row's heads of q, k or v, `kHeadsPerWarp` at a
// time, U head groups per batch with all their x loads issued before any use.
// ILV: interleaved RoPE pairs (2j, 2j+1), whose partner is the other half of the
// same bf16 pair; otherwise rotate-half pairs (i, i + ROT/2), one shuffle away.
// The bias is loaded where it is used: it is re-read by every row and stays in
// L1, and keeping U bias chunks live would cost the registers (and so the
// resident warps) that hold the loads of x in flight.
// NORM: q or k (norm and rotation); otherwise v (the bias only).
template <int LPH, int U, bool NORM, bool ILV>
__device__ __forceinline__ void qkv_unit(const uint16_t* __restrict__ xrow,
                                         const uint16_t* __restrict__ bias, uint16_t* __restrict__ orow,
                                         int heads, int lane, int c, int src, int half, int rot_chunks,
                                         const uint4& cw, const uint4& sw, float eps) {
  constexpr int kHd = 8 * LPH;
  constexpr int kHeadsPerWarp = 32 / LPH;
  const int groups = (heads + kHeadsPerWarp - 1) / kHeadsPerWarp;
  const int col0 = (lane / LPH) * kHd + c * 8;
  const float hd_f = static_cast<float>(kHd);
  for (int g0 = 0; g0 < groups; g0 += U) {
    uint4 xw[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int head = (g0 + j) * kHeadsPerWarp + lane / LPH;
      xw[j] = make_uint4(0u, 0u, 0u, 0u);
      if (head < heads) {
        const int col = (g0 + j) * (kHeadsPerWarp * kHd) + col0;
        xw[j] = load16_stream(xrow + col);
      }
    }
#pragma unroll
    for (int j = 0; j < U; ++j) {
      if (g0 + j >= groups) break;  // warp-uniform
      const int head = (g0 + j) * kHeadsPerWarp + lane / LPH;
      const int col = (g0 + j) * (kHeadsPerWarp * kHd) + col0;
      uint4 bw = make_uint4(0u, 0u, 0u, 0u);
      if (head < heads) bw = load16_reused(bias + col);
      uint32_t xb[4];
      biased(xw[j], bw, xb);
      if constexpr (!NORM) {
        if (head < heads) store16(orow + col, make_uint4(xb[0], xb[1], xb[2], xb[3]));
      } else {
        // the head's sum of squares: eight fmaf partials, the chunk total, a
        // butterfly over the head's lanes
        float2 acc[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = bf16x2_to_float2(xb[i]);
          acc[i] = fma2(f, f, make_float2(0.0f, 0.0f));
        }
        float ss = __fadd_rn(__fadd_rn(__fadd_rn(acc[0].x, acc[0].y), __fadd_rn(acc[1].x, acc[1].y)),
                             __fadd_rn(__fadd_rn(acc[2].x, acc[2].y), __fadd_rn(acc[3].x, acc[3].y)));
#pragma unroll
        for (int o = LPH / 2; o >= 1; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
        const float rstd = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(ss, hd_f), eps)));
        const float2 rstd2 = make_float2(rstd, rstd);
        uint32_t nw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) nw[i] = float2_to_bf16x2(mul2(bf16x2_to_float2(xb[i]), rstd2));
        // RoPE on the head's first ROT values: r, the rotation partner of each value
        uint32_t rw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if constexpr (ILV) {
            rw[i] = rot_pair_bf16x2(nw[i]);
          } else {
            const uint32_t pw = __shfl_sync(0xffffffffu, nw[i], src);
            rw[i] = c < half ? neg_bf16x2(pw) : pw;
          }
        }
        uint4 res = make_uint4(nw[0], nw[1], nw[2], nw[3]);
        if (c < rot_chunks) {
          const uint32_t cs[4] = {cw.x, cw.y, cw.z, cw.w};
          const uint32_t sn[4] = {sw.x, sw.y, sw.z, sw.w};
          uint32_t o[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t p1 = float2_to_bf16x2(mul2(bf16x2_to_float2(nw[i]), bf16x2_to_float2(cs[i])));
            const uint32_t p2 = float2_to_bf16x2(mul2(bf16x2_to_float2(rw[i]), bf16x2_to_float2(sn[i])));
            o[i] = add_bf16x2(p1, p2);  // bf16(fl(p1 + p2)) of two bf16 values
          }
          res = make_uint4(o[0], o[1], o[2], o[3]);
        }
        if (head < heads) store16(orow + col, res);
      }
    }
  }
}

// HD = 8 * LPH: LPH lanes per head, 32 / LPH heads per warp.  Persistent warps
// walk the (row, tensor) units with the row outermost, so the three units of a
// row (which share its cos/sin) run on neighbouring warps.
template <int LPH, int U, bool ILV>
__global__ void __launch_bounds__(kThreads, 4) qkv_epilogue_kernel(const QkvArgs a) {
  const int lane = threadIdx.x & 31;
  const int c = lane % LPH;  // chunk of the head
  const int heads = static_cast<int>(a.heads);
  const int64_t units = 3 * a.rows;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
  const int rot_chunks = static_cast<int>(a.rot >> 3);  // ROT / 8
  const int half = rot_chunks >> 1;                      // ROT / 16: chunks in each half
  // the rotate-half partner chunk: c + ROT/2 in the first half, c - ROT/2 in the second
  const int src = (lane - c) + (c < half ? c + half : (c < rot_chunks ? c - half : c));
  const int64_t out_ld = a.heads * (8 * LPH);

  for (int64_t u = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); u < units;
       u += nwarps) {
    const int64_t row = u / 3;
    const int tensor = static_cast<int>(u - row * 3);  // warp-uniform
    const uint16_t* xrow = a.x[tensor] + row * a.ld[tensor];
    uint16_t* orow = a.out[tensor] + row * out_ld;
    if (tensor == 2) {
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      qkv_unit<LPH, U, false, ILV>(xrow, a.bias[2], orow, heads, lane, c, src, half, rot_chunks, z, z, a.eps);
    } else {
      uint4 cw = make_uint4(0u, 0u, 0u, 0u), sw = make_uint4(0u, 0u, 0u, 0u);
      if (c < rot_chunks) {
        cw = load16_reused(a.cos + row * a.rot + c * 8);
        sw = load16_reused(a.sin + row * a.rot + c * 8);
      }
      qkv_unit<LPH, U, true, ILV>(xrow, a.bias[tensor], orow, heads, lane, c, src, half, rot_chunks, cw,
                                  sw, a.eps);
    }
  }
}

// Head groups per batch: 2 KB of x in flight per warp (64 registers, four
// 256-thread blocks per SM).
constexpr int kUnroll = 4;

template <int LPH, bool ILV>
cudaError_t launch_lph(const QkvArgs& a, cudaStream_t stream) {
  int blocks = 0;
  cudaError_t err = persistent_blocks(reinterpret_cast<const void*>(&qkv_epilogue_kernel<LPH, kUnroll, ILV>),
                                      kThreads, 0, (3 * a.rows + kWarps - 1) / kWarps, &blocks);
  if (err != cudaSuccess) return err;
  qkv_epilogue_kernel<LPH, kUnroll, ILV><<<blocks, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

template <bool ILV>
cudaError_t launch_ilv(const QkvArgs& a, int64_t head_dim, cudaStream_t stream) {
  switch (head_dim) {
    case 64: return launch_lph<8, ILV>(a, stream);
    case 128: return launch_lph<16, ILV>(a, stream);
    case 256: return launch_lph<32, ILV>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_qkv_epilogue(const uint16_t* const x[3], const int64_t ld[3],
                                const uint16_t* const bias[3], uint16_t* const out[3],
                                const uint16_t* cos, const uint16_t* sin, int64_t rot, int interleaved,
                                int64_t rows, int64_t heads, int64_t head_dim, float eps,
                                cudaStream_t stream) {
  QkvArgs a;
  for (int i = 0; i < 3; ++i) {
    a.x[i] = x[i];
    a.ld[i] = ld[i];
    a.bias[i] = bias[i];
    a.out[i] = out[i];
  }
  a.cos = cos;
  a.sin = sin;
  a.rot = rot;
  a.interleaved = interleaved;
  a.rows = rows;
  a.heads = heads;
  a.eps = eps;
  if (rows == 0) return cudaSuccess;
  return interleaved ? launch_ilv<true>(a, head_dim, stream) : launch_ilv<false>(a, head_dim, stream);
}

}  // namespace h3q
