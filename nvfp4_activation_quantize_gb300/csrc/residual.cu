// residual.cu -- residual fold + RMSNorm (fp32 statistics) + AdaLN + NVFP4.
//
// (TensorRT-LLM PR #21483, commit "...norm1 ... from a second table": a block
// folds its MLP residual into the next block's norm1 kernel, reading the gate
// from its own AdaLN table while the scale and shift come from the next
// block's.  FastVideo API page, residual_norm_quantize: in place
// h += bf16(o + bias) * scale on a contiguous fp32 residual h, then NVFP4 of
// the normed h.)
//
// Per row, with t the row's frame:
//   u  = bf16(fl(o + bias))        (u = o without a bias)
//   h' = fl(h + fl(u * gate[t]))   written back to h
//   rstd of h' in the canonical order (chunk c on lane c % 128, eight fmaf
//   partials per lane, the lane total, a butterfly per warp, (T0+T1)+(T2+T3)),
//   y  = bf16(fl(fl(fl(fl(h' * rstd) * gamma) * fl(1 + scale[t])) + shift[t]))
//   and the NVFP4 quantize of y.
//
// One CTA of 128 threads owns one row at a time (two CTAs per SM, persistent
// over a contiguous range of rows); thread t owns the row's chunks t, t+128,
// ... in both passes.  It holds the row's h (fp32) and o (bf16) in registers
// and issues the loads of the next row before working on this one, so a row's
// loads are in flight while the previous row is computed.  The per-column
// tables live in shared memory: bias and gamma for the whole launch, the gate,
// fl(1 + scale) and shift of the current frame, reloaded (between two
// barriers) when the frame changes.  The kernel moves 4 + 2 + 4 + 0.5 + 1/16
// bytes per element (h read and written, o read, codes and scales written), so
// it is bound by HBM bandwidth, not by its arithmetic.
#include "h3q_device.cuh"
#include "h3q_internal.h"

namespace h3q {
namespace {

constexpr int kThreads = 128;  // the lanes of the canonical order

struct ResidualArgs {
  float* h;
  int64_t ld_h;
  const uint16_t* o;
  int64_t ld_o;
  const uint16_t* bias;  // may be null
  const uint16_t* gate;  // [num_frames, cols]
  const uint16_t* gamma;
  const uint16_t* table;  // [num_frames, 2, cols]: [t, 0] shift, [t, 1] scale
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

__device__ __forceinline__ int64_t frame_of(const ResidualArgs& a, int64_t row) {
  const int64_t t = a.row_frame ? static_cast<int64_t>(a.row_frame[row]) : row / a.rows_per_frame;
  return t < 0 ? 0 : (t >= a.num_frames ? a.num_frames - 1 : t);  // memory safety only
}

// Eight fp32 of h: a 256-bit load (h is read once, written back by this kernel).
__device__ __forceinline__ void ld_h8(const float* p, float (&v)[8]) {
  asm volatile("ld.global.L1::no_allocate.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]),
                 "=f"(v[6]), "=f"(v[7])
               : "l"(p));
}

__device__ __forceinline__ void st_h8(float* p, const float (&v)[8]) {
  asm volatile("st.global.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(v[0]), "f"(v[1]),
               "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
               : "memory");
}

// Shared-memory tables, one 16-byte entry per 8-column chunk c (lane-consecutive,
// conflict-free): bias and gamma (bf16) for the launch; gate and shift (bf16)
// and fl(1 + scale) (fp32, two planes) for the current frame.
struct Tables {
  uint4* bias;
  uint4* gamma;
  uint4* gate;
  uint4* shift;
  float4* fc_lo;
  float4* fc_hi;
};

__device__ __forceinline__ Tables carve(uint4* smem, int chunk_slots) {
  Tables tb;
  tb.bias = smem;
  tb.gamma = smem + chunk_slots;
  tb.gate = smem + 2 * chunk_slots;
  tb.shift = smem + 3 * chunk_slots;
  tb.fc_lo = reinterpret_cast<float4*>(smem + 4 * chunk_slots);
  tb.fc_hi = reinterpret_cast<float4*>(smem + 5 * chunk_slots);
  return tb;
}

__device__ __forceinline__ void load_frame_tables(const ResidualArgs& a, const Tables& tb,
                                                  int64_t f, int64_t chunks) {
  for (int64_t c = threadIdx.x; c < chunks; c += blockDim.x) {
    tb.gate[c] = load16_stream(a.gate + f * a.cols + c * 8);
    const uint16_t* shift = a.table + f * 2 * a.cols + c * 8;
    tb.shift[c] = load16_stream(shift);
    const uint4 sc = load16_stream(shift + a.cols);
    const float2 s0 = add2(make_float2(1.0f, 1.0f), bf16x2_to_float2(sc.x));
    const float2 s1 = add2(make_float2(1.0f, 1.0f), bf16x2_to_float2(sc.y));
    const float2 s2 = add2(make_float2(1.0f, 1.0f), bf16x2_to_float2(sc.z));
    const float2 s3 = add2(make_float2(1.0f, 1.0f), bf16x2_to_float2(sc.w));
    tb.fc_lo[c] = make_float4(s0.x, s0.y, s1.x, s1.y);
    tb.fc_hi[c] = make_float4(s2.x, s2.y, s3.x, s3.y);
  }
}

// Modulate one chunk (the folded residual hp[0..7] of chunk c) and quantize this
// thread's half of its 16-element block: the two threads of a block (lanes 2k,
// 2k+1, chunks c and c+1) exchange their half maxima with one shuffle; the even
// one writes the scale byte.  All 32 lanes call this; `valid` masks the stores.
__device__ __forceinline__ void emit_chunk(const float (&hp)[8], float rstd, const Tables& tb,
                                           int64_t c, bool valid, uint8_t* codes_at,
                                           uint8_t* scale_at, float gsf, const float* inv_table) {
  const uint4 g4 = tb.gamma[c];
  const uint4 h4 = tb.shift[c];
  const float4 f0 = tb.fc_lo[c], f1 = tb.fc_hi[c];
  const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w};
  const uint32_t sw[4] = {h4.x, h4.y, h4.z, h4.w};
  const float2 fc[4] = {make_float2(f0.x, f0.y), make_float2(f0.z, f0.w), make_float2(f1.x, f1.y),
                        make_float2(f1.z, f1.w)};
  const float2 rstd2 = make_float2(rstd, rstd);
  uint32_t y[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 n = mul2(make_float2(hp[2 * i], hp[2 * i + 1]), rstd2);
    const float2 hh = mul2(n, bf16x2_to_float2(gw[i]));
    const float2 m = mul2(hh, fc[i]);
    y[i] = float2_to_bf16x2(add_bf16x2_f32(sw[i], m));
  }
  float amax = halves_amax(absmax_bf16x2(absmax_bf16x2(y[0], y[1]), absmax_bf16x2(y[2], y[3])));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  const uint32_t sf = block_scale(amax, gsf);
  const uint32_t codes = codes8(y, inv_table[sf]);
  if (valid) store_word(codes_at, codes);
  if (valid && !(threadIdx.x & 1)) store_byte(scale_at, sf);
}

// Fold chunk c of a row: hp = fl(h + fl(bf16(fl(o + bias)) * gate)).
__device__ __forceinline__ void fold_chunk(float (&hv)[8], const uint4& ov, const Tables& tb,
                                           int64_t c, bool has_bias) {
  const uint4 g4 = tb.gate[c];
  const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w};
  const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w};
  uint32_t bw[4] = {0u, 0u, 0u, 0u};
  if (has_bias) {
    const uint4 b4 = tb.bias[c];
    bw[0] = b4.x; bw[1] = b4.y; bw[2] = b4.z; bw[3] = b4.w;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    // u as a bf16 pair: o itself, or bf16(fl(o + bias)) by one bf16x2 add (the
    // same bits, see add_bf16x2)
    const uint32_t u = has_bias ? add_bf16x2(ow[i], bw[i]) : ow[i];
    const float2 t = mul2(bf16x2_to_float2(u), bf16x2_to_float2(gw[i]));
    // scalar adds: a paired add of a paired product would be contracted
    hv[2 * i] = __fadd_rn(hv[2 * i], t.x);
    hv[2 * i + 1] = __fadd_rn(hv[2 * i + 1], t.y);
  }
}

// Rows of up to 1,024 * C1 columns (FULL: exactly); dynamic shared memory holds
// the six tables of 128 * C1 chunk entries.
template <int C1, bool FULL>
__global__ void __launch_bounds__(kThreads, 2) residual_adaln_kernel(const ResidualArgs a) {
  constexpr int kSlots = kThreads * C1;
  extern __shared__ uint4 smem[];
  __shared__ float inv_table[128];
  __shared__ float totals[2][4];
  const Tables tb = carve(smem, kSlots);
  const float gsf = *a.gsf;
  fill_inverse_scales(inv_table, gsf);

  const int t = threadIdx.x;
  const int64_t chunks = a.cols >> 3;
  const int64_t quads = a.cols >> 6;
  const float cols_f = static_cast<float>(a.cols);  // exact: cols <= 2^24
  const bool has_bias = a.bias != nullptr;
  for (int64_t c = t; c < chunks; c += kThreads) {  // the launch-wide tables
    tb.gamma[c] = load16_stream(a.gamma + c * 8);
    if (has_bias) tb.bias[c] = load16_stream(a.bias + c * 8);
  }
  const int64_t r_begin = a.rows * blockIdx.x / gridDim.x;
  const int64_t r_end = a.rows * (blockIdx.x + 1) / gridDim.x;
  int64_t frame = -1;

  auto load = [&](int64_t r, float (&h)[C1][8], uint4 (&o)[C1]) {
    if (r >= r_end) return;  // CTA-uniform
    const float* hr = a.h + r * a.ld_h + t * 8;
    const uint16_t* orow = a.o + r * a.ld_o + t * 8;
#pragma unroll
    for (int j = 0; j < C1; ++j) {
      if (FULL || t + j * kThreads < chunks) {
        ld_h8(hr + j * (kThreads * 8), h[j]);
        o[j] = load16_stream(orow + j * (kThreads * 8));
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) h[j][e] = 0.0f;
        o[j] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  };

  auto process = [&](int64_t r, float (&h)[C1][8], const uint4 (&o)[C1], int slot) {
    const int64_t f = frame_of(a, r);  // CTA-uniform
    if (f != frame) {
      __syncthreads();  // nobody reads the previous frame's tables any more
      load_frame_tables(a, tb, f, chunks);
      __syncthreads();
      frame = f;
    }
    // fold, write back, squares in the canonical order (partial e of each chunk)
    float* hr = a.h + r * a.ld_h + t * 8;
    float2 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int j = 0; j < C1; ++j) {
      const int64_t c = t + j * kThreads;
      if (FULL || c < chunks) {
        fold_chunk(h[j], o[j], tb, c, has_bias);
        st_h8(hr + j * (kThreads * 8), h[j]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 v = make_float2(h[j][2 * i], h[j][2 * i + 1]);
          acc[i] = fma2(v, v, acc[i]);
        }
      }
    }
    float tot = __fadd_rn(__fadd_rn(__fadd_rn(acc[0].x, acc[0].y), __fadd_rn(acc[1].x, acc[1].y)),
                          __fadd_rn(__fadd_rn(acc[2].x, acc[2].y), __fadd_rn(acc[3].x, acc[3].y)));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) tot = __fadd_rn(tot, __shfl_xor_sync(0xffffffffu, tot, off));
    if ((t & 31) == 0) totals[slot][t >> 5] = tot;
    __syncthreads();
    const float* T = totals[slot];
    const float ss = __fadd_rn(__fadd_rn(T[0], T[1]), __fadd_rn(T[2], T[3]));
    const float rstd = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(ss, cols_f), a.eps)));
    if (a.row_rstd != nullptr && t == 0) a.row_rstd[r] = rstd;
    uint8_t* const codes_at = a.codes + r * (a.cols >> 1) + t * 4;
    uint8_t* const scale_at = a.scales + scale_row_offset(r, quads) + (t >> 3) * 512 + ((t >> 1) & 3);
#pragma unroll
    for (int j = 0; j < C1; ++j) {
      const int64_t c = t + j * kThreads;
      emit_chunk(h[j], rstd, tb, c, FULL || c < chunks, codes_at + j * (kThreads * 4),
                 scale_at + j * (kThreads / 8 * 512), gsf, inv_table);
    }
  };

  // Two register sets: the next row's loads are in flight while a row is worked on.
  float hA[C1][8], hB[C1][8];
  uint4 oA[C1], oB[C1];
  load(r_begin, hA, oA);
  for (int64_t r = r_begin; r < r_end; r += 2) {
    load(r + 1, hB, oB);
    process(r, hA, oA, 0);
    if (r + 1 < r_end) {  // CTA-uniform
      load(r + 2, hA, oA);
      process(r + 1, hB, oB, 1);
    }
  }

  // zero the scale words of the padding rows rows..pad128(rows)-1
  const int64_t prows = (a.rows + 127) >> 7 << 7;
  for (int64_t p = a.rows + blockIdx.x; p < prows; p += gridDim.x)
    for (int64_t q = t; q < quads; q += kThreads)
      store_word(a.scales + scale_word_offset(p, q, quads), 0u);
}

template <int C1>
cudaError_t launch_c1(const ResidualArgs& a, cudaStream_t stream) {
  const int smem = 6 * kThreads * C1 * 16;
  const bool full = a.cols == int64_t(1024) * C1;
  const void* kernel = full ? reinterpret_cast<const void*>(&residual_adaln_kernel<C1, true>)
                            : reinterpret_cast<const void*>(&residual_adaln_kernel<C1, false>);
  int blocks = 0;
  cudaError_t err = persistent_blocks(kernel, kThreads, smem, a.rows > 0 ? a.rows : 1, &blocks);
  if (err != cudaSuccess) return err;
  if (full)
    residual_adaln_kernel<C1, true><<<blocks, kThreads, smem, stream>>>(a);
  else
    residual_adaln_kernel<C1, false><<<blocks, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_residual_adaln(float* h, int64_t ld_h, const uint16_t* o, int64_t ld_o,
                                  const uint16_t* bias, const uint16_t* gate, const uint16_t* gamma,
                                  const uint16_t* table, int64_t num_frames,
                                  const int32_t* row_frame, int64_t rows_per_frame, float eps,
                                  int64_t rows, int64_t cols, const float* gsf, uint8_t* codes,
                                  uint8_t* scales, float* row_rstd, cudaStream_t stream) {
  const ResidualArgs a{h,    ld_h, o,    ld_o, bias, gate,  gamma,  table,   num_frames, row_frame,
                       rows_per_frame, eps, rows, cols, gsf, codes, scales, row_rstd};
  const int64_t per_lane = (cols / 8 + kThreads - 1) / kThreads;
  if (per_lane <= 1) return launch_c1<1>(a, stream);
  if (per_lane <= 2) return launch_c1<2>(a, stream);
  if (per_lane <= 4) return launch_c1<4>(a, stream);
  if (per_lane <= 7) return launch_c1<7>(a, stream);
  if (per_lane <= 8) return launch_c1<8>(a, stream);
  return cudaErrorInvalidValue;  // the API rejects rows wider than 8,192 first
}

}  // namespace h3q
