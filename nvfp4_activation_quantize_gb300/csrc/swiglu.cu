// swiglu.cu -- SwiGLU producer: y = silu(gate) * up rounded to bf16, then NVFP4.
//
// (FastVideo compare "fasth3-spark-exact-perf", minimax_h3_swiglu_quant.cuh,
// swiglu_bf16: value * silu(gate), one bf16 rounding; TensorRT-LLM PR #21483,
// the SiLU-and-mul producer that writes NVFP4 directly.)
//
// Per element, in binary32 with one rounding per operation:
//   E = exp_c(-g), sigma = fl(1 / fl(1 + E)), s = fl(g * sigma), y = bf16(fl(s * u))
// exp_c is this library's fixed exponential: Cody-Waite additive reduction
// (W. J. Cody and W. Waite, "Software Manual for the Elementary Functions",
// 1980) by a two-part ln 2 applied with FMAs, and the degree-7 Taylor
// polynomial of e^r in Horner form:
//   z > 89 -> +inf, z < -104 -> +0, otherwise
//   t = fl(z * L2E), k = rint(t), r = fma(-k, C1, z), r = fma(-k, C2, r),
//   p = P7, p = fma(p, r, Pn) for n = 6..2, p = fma(p, r, 1), p = fma(p, r, 1),
//   result = p * 2^k rounded once.
//   L2E = fl(1/ln 2), C1 = fl(ln 2), C2 = fl(ln 2 - C1), Pn = fl(1/n!).
// rint uses the 1.5 * 2^23 addition: for |t| <= 2^22 the sum lands where the
// binary32 spacing is 1, so the addition itself rounds t half-to-even, and
// subtracting the constant again is exact.
//
// s = fl(g * sigma) depends on the bf16 gate alone, so -- as the pages' fused
// SwiGLU producer does with its SiLU table (FastVideo API page,
// swiglu_quantize) -- each CTA first tabulates s for every bf16 gate with
// 2^-25 <= |g| <= 127.5 (8,192 values, 32 KB of shared memory), computed with
// the arithmetic below.  A warp whose gates all lie in that range looks s up and
// only forms y = bf16(fl(s * u)); other warps compute s directly.  Both give
// the same bits.
//
// Work layout as in the standalone quantize: one warp per 512-column segment,
// one 16-element block per lane.  The plain producer stages gate and up through
// a per-warp cp.async ring (swiglu_ring_kernel: one 768-thread CTA per SM, two
// segments' copies in flight per warp while it computes a third); the abs-max
// pass and the packed projection with its bias load them with 256-bit loads
// into registers (swiglu_kernel).  In the direct
// computation, when every gate of the warp's segment has |g| <= 87, 2^k is a
// normal number for every element and the scaling is a single multiply by a
// power of two built from k's bits; otherwise the warp scales with ldexpf,
// which gives identical results wherever both apply.
#include "h3q_device.cuh"
#include "h3q_internal.h"
#include "h3q_silu.cuh"

namespace h3q {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
// Segments in flight per warp in swiglu_kernel: two for the abs-max pass; one
// for the packed projection with its bias, whose extra bias loads and adds would
// otherwise cost the registers of a fourth CTA per SM (52 registers, not 64).
constexpr int kUnrollPlain = 2;

// x = bf16(fl(x + b)) for the 16 bf16 values of a block and their biases b
// (one bf16x2 add per pair: the same bits, see add_bf16x2).
__device__ __forceinline__ void add_bias(Block16& x, const Block16& b) {
#pragma unroll
  for (int i = 0; i < 8; ++i) x.w[i] = add_bf16x2(x.w[i], b.w[i]);
}

// AMAX: the abs-max pass -- y is formed the same way, its max |y| folded into
// *amax, and nothing is quantized or stored.  BIAS: gate and up get their
// per-column biases (bias_gate, bias_up) added and are rounded to bf16 first
// (the value-first packed projection with its bias not yet added).
template <bool AMAX, bool BIAS>
__global__ void __launch_bounds__(kThreads)
swiglu_kernel(const uint16_t* __restrict__ gate, int64_t ld_gate, const uint16_t* __restrict__ up,
              int64_t ld_up, int64_t rows, int64_t cols, const float* __restrict__ gsf_ptr,
              uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, float* __restrict__ amax,
              const uint16_t* __restrict__ bias_gate, const uint16_t* __restrict__ bias_up) {
  constexpr int kUnroll = BIAS ? 1 : kUnrollPlain;
  __shared__ float inv_table[128];
  __shared__ __align__(16) float silu_table[2 * kTabHalf];
  const float gsf = AMAX ? 0.0f : *gsf_ptr;
  if (!AMAX) fill_inverse_scales(inv_table, gsf);
  float run_max = 0.0f;
  fill_silu_table(silu_table);
  __syncthreads();
  const char* table = reinterpret_cast<const char*>(silu_table);

  const int lane = threadIdx.x & 31;
  const int64_t groups = cols >> 4;
  const int64_t quads = cols >> 6;
  const int64_t segs = (groups + 31) >> 5;
  const int64_t prows = AMAX ? rows : (rows + 127) >> 7 << 7;  // the abs-max pass has no padding to write
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);

  int64_t row[kUnroll], seg[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int64_t s = first + u * nwarps;
    row[u] = s / segs;
    seg[u] = s - row[u] * segs;
  }
  const int64_t adv_rows = nwarps * kUnroll / segs;
  const int64_t adv_segs = nwarps * kUnroll - adv_rows * segs;

  while (row[0] < prows) {
    Block16 gb[kUnroll], ub[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t g = seg[u] * 32 + lane;
      if (row[u] < rows && g < groups) {
        load_stream(gate + row[u] * ld_gate + g * kBlock, gb[u]);
        load_stream(up + row[u] * ld_up + g * kBlock, ub[u]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) gb[u].w[i] = ub[u].w[i] = 0;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (row[u] >= prows) break;  // warp-uniform
      const int64_t g = seg[u] * 32 + lane;
      const bool in_row = row[u] < rows;
      const bool in_cols = g < groups;
      if (BIAS && in_row && in_cols) {
        // the biases are loaded here rather than with x: they are re-read by
        // every row and stay in L1, and holding them across the batch would
        // cost the registers (and so the resident warps) that keep x in flight
        Block16 b;
        load_reused(bias_gate + g * kBlock, b);
        add_bias(gb[u], b);
        load_reused(bias_up + g * kBlock, b);
        add_bias(ub[u], b);
      }
      Block16 y;
      uint32_t dw[8];
      if (__all_sync(0xffffffffu, table_words(gb[u], dw))) {
        swiglu_block_table(dw, ub[u], y, table);
      } else if (__all_sync(0xffffffffu, block_amax(gb[u]) <= kFastLimit)) {
        swiglu_block<true>(gb[u], ub[u], y);
      } else {
        swiglu_block<false>(gb[u], ub[u], y);
      }
      if (AMAX) {
        if (in_row && in_cols) run_max = fmaxf(run_max, block_amax(y));
        continue;
      }
      Quantized q = quantize_block<true>(y, gsf, inv_table);
      if (!in_row) q.sf = 0;
      if (in_row && in_cols)
        store_codes(codes + row[u] * (cols >> 1) + g * 8, q.codes_lo, q.codes_hi);
      store_scale_quad(scales, row[u], g, quads, q.sf, in_cols);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      row[u] += adv_rows;
      seg[u] += adv_segs;
      if (seg[u] >= segs) {
        seg[u] -= segs;
        row[u] += 1;
      }
    }
  }
  if (AMAX) commit_amax(run_max, amax, inv_table);  // inv_table is unused in this mode
}

// The plain producer with its loads staged through a per-warp cp.async ring:
// one CTA of 768 threads per SM sharing one SiLU table, each warp one segment
// per step with the next kRingStages - 1 segments' copies in flight.  Each lane
// copies and later reads only its own 32 bytes of gate and of up, so only its
// own cp.async.wait_group orders them; its two 16-byte halves sit swapped in
// lanes 4-7 of every 8 (slot c ^ ((lane >> 2) & 1)), which keeps the 16-byte
// shared loads of a quarter-warp on distinct banks.
constexpr int kRingThreads = 768;
constexpr int kRingWarps = kRingThreads / 32;
constexpr int kRingStages = 3;
constexpr int kRingWarpBytes = kRingStages * 2 * 1024;

__device__ __forceinline__ void ring_cp16(uint32_t smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem), "l"(gmem) : "memory");
}
__device__ __forceinline__ void ring_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void ring_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ring_ld16(uint32_t smem, uint32_t* w) {
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
               : "r"(smem)
               : "memory");
}

__global__ void __launch_bounds__(kRingThreads, 1)
swiglu_ring_kernel(const uint16_t* __restrict__ gate, int64_t ld_gate, const uint16_t* __restrict__ up,
                   int64_t ld_up, int64_t rows, int64_t cols, const float* __restrict__ gsf_ptr,
                   uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  __shared__ float inv_table[128];
  __shared__ __align__(16) float silu_table[2 * kTabHalf];
  extern __shared__ __align__(16) uint8_t ring[];  // [warp][stage][gate, up][lane][32 bytes]
  const float gsf = *gsf_ptr;
  fill_inverse_scales(inv_table, gsf);
  fill_silu_table(silu_table);
  __syncthreads();
  const char* table = reinterpret_cast<const char*>(silu_table);

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t groups = cols >> 4;
  const int64_t quads = cols >> 6;
  const int64_t segs = (groups + 31) >> 5;
  const int64_t prows = (rows + 127) >> 7 << 7;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kRingWarps;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kRingWarps + warp;
  const int64_t adv_rows = nwarps / segs;
  const int64_t adv_segs = nwarps - adv_rows * segs;
  const uint32_t sw = ((lane >> 2) & 1) * 16;
  const uint32_t mine = static_cast<uint32_t>(__cvta_generic_to_shared(ring)) + warp * kRingWarpBytes + lane * 32;

  int64_t crow = first / segs, cseg = first - crow * segs;  // the segment computed
  int64_t irow = crow, iseg = cseg;                          // the next segment copied
  auto issue = [&](int stage) {
    const int64_t g = iseg * 32 + lane;
    if (irow < rows && g < groups) {
      const uint32_t d = mine + stage * 2048;
      const uint16_t* gp = gate + irow * ld_gate + g * kBlock;
      const uint16_t* upp = up + irow * ld_up + g * kBlock;
      ring_cp16(d + sw, gp);
      ring_cp16(d + (sw ^ 16), gp + 8);
      ring_cp16(d + 1024 + sw, upp);
      ring_cp16(d + 1024 + (sw ^ 16), upp + 8);
    }
    ring_commit();
    iseg += adv_segs;
    irow += adv_rows;
    if (iseg >= segs) {
      iseg -= segs;
      irow += 1;
    }
  };
#pragma unroll
  for (int s = 0; s < kRingStages - 1; ++s) issue(s);
  int stage = 0;
  while (crow < prows) {
    ring_wait<kRingStages - 2>();  // this step's copies (this lane's) landed
    const int64_t g = cseg * 32 + lane;
    const bool in_row = crow < rows;
    const bool in_cols = g < groups;
    Block16 gb, ub;
    if (in_row && in_cols) {
      const uint32_t d = mine + stage * 2048;
      ring_ld16(d + sw, gb.w);
      ring_ld16(d + (sw ^ 16), gb.w + 4);
      ring_ld16(d + 1024 + sw, ub.w);
      ring_ld16(d + 1024 + (sw ^ 16), ub.w + 4);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) gb.w[i] = ub.w[i] = 0;
    }
    // the stage read in the previous step (its loads long consumed) takes the
    // step kRingStages - 1 ahead
    issue(stage == 0 ? kRingStages - 1 : stage - 1);
    Block16 y;
    uint32_t dw[8];
    if (__all_sync(0xffffffffu, table_words(gb, dw))) {
      swiglu_block_table(dw, ub, y, table);
    } else if (__all_sync(0xffffffffu, block_amax(gb) <= kFastLimit)) {
      swiglu_block<true>(gb, ub, y);
    } else {
      swiglu_block<false>(gb, ub, y);
    }
    Quantized q = quantize_block<true>(y, gsf, inv_table);
    if (!in_row) q.sf = 0;
    if (in_row && in_cols) store_codes(codes + crow * (cols >> 1) + g * 8, q.codes_lo, q.codes_hi);
    store_scale_quad(scales, crow, g, quads, q.sf, in_cols);
    stage = stage + 1 == kRingStages ? 0 : stage + 1;
    cseg += adv_segs;
    crow += adv_rows;
    if (cseg >= segs) {
      cseg -= segs;
      crow += 1;
    }
  }
  ring_wait<0>();
}

// The producer with its loads staged through the per-warp cp.async ring (the
// plain producer above), for the value-first packed projection with its
// biases: gate and up get their per-column biases added (bf16(fl(x + b)), one
// bf16x2 add per pair) after the ring.  Each warp keeps one 512-column segment
// for all its rows -- warp w of the `active` = (warps / segs) * segs warps owns
// segment w % segs and every (active / segs)-th row from w / segs -- so each
// lane loads its 32 bytes of gate bias and of up bias once and holds them in
// registers (re-reading them per row from L1 costs more than the ring gains:
// the ring's shared memory leaves L1 too small for 2 x 2F bytes of bias).
__global__ void __launch_bounds__(kRingThreads, 1)
swiglu_ring_bias_kernel(const uint16_t* __restrict__ gate, const uint16_t* __restrict__ up, int64_t ld,
                        int64_t rows, int64_t cols, const float* __restrict__ gsf_ptr,
                        uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                        const uint16_t* __restrict__ bias_gate, const uint16_t* __restrict__ bias_up) {
  __shared__ float inv_table[128];
  __shared__ __align__(16) float silu_table[2 * kTabHalf];
  extern __shared__ __align__(16) uint8_t ring[];  // [warp][stage][gate, up][lane][32 bytes]
  const float gsf = *gsf_ptr;
  fill_inverse_scales(inv_table, gsf);
  fill_silu_table(silu_table);
  __syncthreads();
  const char* table = reinterpret_cast<const char*>(silu_table);

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t groups = cols >> 4;
  const int64_t quads = cols >> 6;
  const int64_t segs = (groups + 31) >> 5;
  const int64_t prows = (rows + 127) >> 7 << 7;
  const int64_t active = static_cast<int64_t>(gridDim.x) * kRingWarps / segs * segs;
  const int64_t w = static_cast<int64_t>(blockIdx.x) * kRingWarps + warp;
  if (w >= active) return;  // warp-uniform; no barrier follows
  const int64_t seg = w % segs;
  const int64_t row_step = active / segs;
  const int64_t g = seg * 32 + lane;
  const bool in_cols = g < groups;
  const uint32_t sw = ((lane >> 2) & 1) * 16;
  const uint32_t mine = static_cast<uint32_t>(__cvta_generic_to_shared(ring)) + warp * kRingWarpBytes + lane * 32;
  Block16 bg, bu;
  if (in_cols) {
    load_reused(bias_gate + g * kBlock, bg);
    load_reused(bias_up + g * kBlock, bu);
  }
  const uint16_t* gp = gate + g * kBlock;
  const uint16_t* upp = up + g * kBlock;

  int64_t crow = w / segs;  // the row computed
  int64_t irow = crow;      // the next row copied
  auto issue = [&](int stage) {
    if (irow < rows && in_cols) {
      const uint32_t d = mine + stage * 2048;
      ring_cp16(d + sw, gp + irow * ld);
      ring_cp16(d + (sw ^ 16), gp + irow * ld + 8);
      ring_cp16(d + 1024 + sw, upp + irow * ld);
      ring_cp16(d + 1024 + (sw ^ 16), upp + irow * ld + 8);
    }
    ring_commit();
    irow += row_step;
  };
#pragma unroll
  for (int s = 0; s < kRingStages - 1; ++s) issue(s);
  int stage = 0;
  while (crow < prows) {
    ring_wait<kRingStages - 2>();  // this step's copies (this lane's) landed
    const bool in_row = crow < rows;
    Block16 gb, ub;
    if (in_row && in_cols) {
      const uint32_t d = mine + stage * 2048;
      ring_ld16(d + sw, gb.w);
      ring_ld16(d + (sw ^ 16), gb.w + 4);
      ring_ld16(d + 1024 + sw, ub.w);
      ring_ld16(d + 1024 + (sw ^ 16), ub.w + 4);
      add_bias(gb, bg);
      add_bias(ub, bu);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) gb.w[i] = ub.w[i] = 0;
    }
    issue(stage == 0 ? kRingStages - 1 : stage - 1);
    Block16 y;
    uint32_t dw[8];
    if (__all_sync(0xffffffffu, table_words(gb, dw))) {
      swiglu_block_table(dw, ub, y, table);
    } else if (__all_sync(0xffffffffu, block_amax(gb) <= kFastLimit)) {
      swiglu_block<true>(gb, ub, y);
    } else {
      swiglu_block<false>(gb, ub, y);
    }
    Quantized q = quantize_block<true>(y, gsf, inv_table);
    if (!in_row) q.sf = 0;
    if (in_row && in_cols) store_codes(codes + crow * (cols >> 1) + g * 8, q.codes_lo, q.codes_hi);
    store_scale_quad(scales, crow, g, quads, q.sf, in_cols);
    stage = stage + 1 == kRingStages ? 0 : stage + 1;
    crow += row_step;
  }
  ring_wait<0>();
}

}  // namespace

cudaError_t launch_swiglu(const uint16_t* gate, int64_t ld_gate, const uint16_t* up,
                          int64_t ld_up, int64_t rows, int64_t cols, const float* gsf,
                          uint8_t* codes, uint8_t* scales, cudaStream_t stream) {
  const int64_t segs = (cols / 16 + 31) / 32;
  const int64_t work = (rows + 127) / 128 * 128 * segs;
  int blocks = 0;
  const int smem = kRingWarps * kRingWarpBytes;
  cudaError_t err = persistent_blocks(reinterpret_cast<const void*>(&swiglu_ring_kernel), kRingThreads, smem,
                                      (work + kRingWarps - 1) / kRingWarps, &blocks);
  if (err != cudaSuccess) return err;
  swiglu_ring_kernel<<<blocks, kRingThreads, smem, stream>>>(gate, ld_gate, up, ld_up, rows, cols, gsf,
                                                             codes, scales);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_packed(const uint16_t* o, int64_t ld_o, const uint16_t* bias, int64_t rows,
                                 int64_t f, const float* gsf, uint8_t* codes, uint8_t* scales,
                                 cudaStream_t stream) {
  if (bias == nullptr) return launch_swiglu(o + f, ld_o, o, ld_o, rows, f, gsf, codes, scales, stream);
  const int64_t segs = (f / 16 + 31) / 32;
  const int64_t work = (rows + 127) / 128 * 128 * segs;
  int blocks = 0;
  const int smem = kRingWarps * kRingWarpBytes;
  cudaError_t err = persistent_blocks(reinterpret_cast<const void*>(&swiglu_ring_bias_kernel), kRingThreads,
                                      smem, (work + kRingWarps - 1) / kRingWarps, &blocks);
  if (err != cudaSuccess) return err;
  if (int64_t{blocks} * kRingWarps >= segs) {
    // value first: up = o[:, :f] with bias[:f], gate = o[:, f:] with bias[f:]
    swiglu_ring_bias_kernel<<<blocks, kRingThreads, smem, stream>>>(o + f, o, ld_o, rows, f, gsf, codes, scales,
                                                                    bias + f, bias);
    return cudaGetLastError();
  }
  // rows wider than one segment per warp of the grid: warps cycle over segments
  err = persistent_blocks(reinterpret_cast<const void*>(&swiglu_kernel<false, true>), kThreads, 0,
                          (work + kWarps - 1) / kWarps, &blocks);
  if (err != cudaSuccess) return err;
  swiglu_kernel<false, true><<<blocks, kThreads, 0, stream>>>(o + f, ld_o, o, ld_o, rows, f, gsf, codes, scales,
                                                              nullptr, bias + f, bias);
  return cudaGetLastError();
}

}  // namespace h3q

namespace h3q {

cudaError_t launch_swiglu_amax(const uint16_t* gate, int64_t ld_gate, const uint16_t* up,
                               int64_t ld_up, int64_t rows, int64_t cols, float* amax,
                               cudaStream_t stream) {
  const int64_t segs = (cols / 16 + 31) / 32;
  const int64_t work = rows * segs;  // no padding rows to visit
  int blocks = 0;
  cudaError_t err = persistent_blocks(reinterpret_cast<const void*>(&swiglu_kernel<true, false>),
                                      kThreads, 0, (work + kWarps - 1) / kWarps, &blocks);
  if (err != cudaSuccess) return err;
  swiglu_kernel<true, false><<<blocks, kThreads, 0, stream>>>(gate, ld_gate, up, ld_up, rows, cols,
                                                              nullptr, nullptr, nullptr, amax, nullptr,
                                                              nullptr);
  return cudaGetLastError();
}

}  // namespace h3q
