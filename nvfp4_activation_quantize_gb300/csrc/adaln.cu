// adaln.cu -- (a) RMSNorm with fp32 statistics + AdaLN modulation + NVFP4.
//
// (TensorRT-LLM PR #21483, summary and commit "...SwiGLU producers": the AdaLN
// RMSNorm + modulation kernel writes packed E2M1 codes and swizzled E4M3 block
// scales directly, so the bf16 activation is never written and re-read.
// FastVideo API page, introduction: fp32 statistics with sequential FMAs per
// thread, no contraction of products that eager rounds.)
//
// One CTA of 128 threads owns one row at a time; thread t owns the row's
// 8-element chunks t, t+128, t+256, ... -- exactly the lanes of the library's
// canonical reduction order.  Per row:
//   pass 1  eight fp32 partials per thread (paired f32x2 FMAs, element by
//           element), ((p0+p1)+(p2+p3))+((p4+p5)+(p6+p7)), a butterfly inside
//           each warp, and (T0+T1)+(T2+T3) over the four warps through shared
//           memory (one barrier per row);
//           rstd = fl(1 / fl(sqrt(fl(fl(ss / cols) + eps))))
//   pass 2  y = bf16(fl(fl(fl(fl(x*rstd)*gamma)*fl(1+scale)) + shift)) and the
//           NVFP4 quantize; the two threads holding the halves of a 16-element
//           block exchange their half maxima with one shuffle.
// The rows of a CTA are a contiguous range, so the frame changes rarely: each
// thread keeps gamma, 1+scale and shift of its own chunks in registers as fp32
// and reloads them only when the frame changes.  Neither the modulation table
// nor gamma is re-read per row.
// x streams through a ring of kStages rows in shared memory filled with
// cp.async: each thread copies exactly the chunks it will read, so the data
// needs no barrier, only the thread's own cp.async.wait_group; kStages-1 rows
// per CTA are in flight while one is computed.
// Rows wider than 8,192 take a generic kernel with the same chunk-to-thread
// mapping and order that reads x twice and the tables per row.
#include "h3q_device.cuh"
#include "h3q_internal.h"

namespace h3q {
namespace {

constexpr int kThreads = 128;  // the lanes of the canonical order
constexpr int kStages = 4;     // rows of x per CTA in the cp.async ring

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

__device__ __forceinline__ void cp_async16(uint32_t smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 load16_reused(const uint16_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 load16_stream(const uint16_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ int64_t frame_of(const AdalnArgs& a, int64_t row) {
  int64_t t = a.row_frame ? static_cast<int64_t>(a.row_frame[row]) : row / a.rows_per_frame;
  return t < 0 ? 0 : (t >= a.num_frames ? a.num_frames - 1 : t);  // memory safety only
}

// fp32 gamma, 1 + scale and shift of chunk c of frame t.
__device__ __forceinline__ void load_tables(const AdalnArgs& a, int64_t t, int64_t c, float* gm,
                                            float* fc, float* sh) {
  const uint16_t* shift = a.table + t * 2 * a.cols + c * 8;
  const uint4 g4 = load16_reused(a.gamma + c * 8);
  const uint4 s4 = load16_reused(shift + a.cols);
  const uint4 h4 = load16_reused(shift);
  const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w};
  const uint32_t sw[4] = {s4.x, s4.y, s4.z, s4.w};
  const uint32_t hw[4] = {h4.x, h4.y, h4.z, h4.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 g = bf16x2_to_float2(gw[i]);
    const float2 f = __fadd2_rn(make_float2(1.0f, 1.0f), bf16x2_to_float2(sw[i]));
    const float2 h = bf16x2_to_float2(hw[i]);
    gm[2 * i] = g.x, gm[2 * i + 1] = g.y;
    fc[2 * i] = f.x, fc[2 * i + 1] = f.y;
    sh[2 * i] = h.x, sh[2 * i + 1] = h.y;
  }
}

// Partials (p_2i, p_2i+1) in acc[i]; element e of the chunk goes to p_e.
__device__ __forceinline__ void accumulate(const uint4& v, float2 (&acc)[4]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = bf16x2_to_float2(w[i]);
    acc[i] = __ffma2_rn(f, f, acc[i]);
  }
}

// ss of the row from this thread's partials: lane total, warp butterfly, then
// (T0+T1)+(T2+T3) over the four warps.  `slot` alternates between rows so one
// barrier per row suffices.
__device__ __forceinline__ float row_sum_of_squares(const float2 (&acc)[4], float (*totals)[4],
                                                    int slot) {
  float tot = __fadd_rn(__fadd_rn(__fadd_rn(acc[0].x, acc[0].y), __fadd_rn(acc[1].x, acc[1].y)),
                        __fadd_rn(__fadd_rn(acc[2].x, acc[2].y), __fadd_rn(acc[3].x, acc[3].y)));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) tot = __fadd_rn(tot, __shfl_xor_sync(0xffffffffu, tot, o));
  if ((threadIdx.x & 31) == 0) totals[slot][threadIdx.x >> 5] = tot;
  __syncthreads();
  const float* T = totals[slot];
  return __fadd_rn(__fadd_rn(T[0], T[1]), __fadd_rn(T[2], T[3]));
}

__device__ __forceinline__ float rstd_of(float ss, int64_t cols, float eps) {
  const float mean = __fdiv_rn(ss, static_cast<float>(cols));
  return __frcp_rn(__fsqrt_rn(__fadd_rn(mean, eps)));
}

// Modulate chunk c (x words v) of row `row`, quantize this thread's half
// block, store its four code bytes and, from the first lane of each group of
// eight, the scale word of the four blocks of the group.  All 32 lanes of the
// warp call this (it shuffles); `valid` masks the stores.
__device__ __forceinline__ void emit_chunk(const AdalnArgs& a, int64_t row, int64_t c, bool valid,
                                           const uint4& v, float rstd, const float* gm,
                                           const float* fc, const float* sh, float gsf,
                                           const float* inv_table) {
  const uint32_t xw[4] = {v.x, v.y, v.z, v.w};
  const float2 rstd2 = make_float2(rstd, rstd);
  uint32_t y[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 n = __fmul2_rn(bf16x2_to_float2(xw[i]), rstd2);
    const float2 h = __fmul2_rn(n, make_float2(gm[2 * i], gm[2 * i + 1]));
    const float2 m = __fmul2_rn(h, make_float2(fc[2 * i], fc[2 * i + 1]));
    const float2 o = __fadd2_rn(m, make_float2(sh[2 * i], sh[2 * i + 1]));
    y[i] = float2_to_bf16x2(o);
  }
  const int lane = threadIdx.x & 31;
  const float half_amax = halves_amax(absmax_bf16x2(absmax_bf16x2(y[0], y[1]),
                                                    absmax_bf16x2(y[2], y[3])));
  const float amax = fmaxf(half_amax, __shfl_xor_sync(0xffffffffu, half_amax, 1));
  const uint32_t sf = block_scale(amax, gsf);
  const uint32_t codes = codes8(y, inv_table[sf]);
  if (valid) store_word(a.codes + row * (a.cols >> 1) + c * 4, codes);
  uint32_t word = (lane & 1) ? 0u : sf << (8 * ((lane >> 1) & 3));
  word |= __shfl_xor_sync(0xffffffffu, word, 2);
  word |= __shfl_xor_sync(0xffffffffu, word, 4);
  if (valid && (lane & 7) == 0)
    store_word(a.scales + scale_word_offset(row, c >> 3, a.cols >> 6), word);
}

// Zero scale words of the padding rows rows..pad128(rows)-1, spread over CTAs.
__device__ __forceinline__ void zero_padding_rows(const AdalnArgs& a) {
  const int64_t prows = (a.rows + 127) >> 7 << 7;
  const int64_t quads = a.cols >> 6;
  for (int64_t p = a.rows + blockIdx.x; p < prows; p += gridDim.x)
    for (int64_t q = threadIdx.x; q < quads; q += kThreads)
      store_word(a.scales + scale_word_offset(p, q, quads), 0u);
}

// Rows up to 128 * CPL chunks (CPL * 1,024 columns): tables resident in
// registers, x through the cp.async ring in dynamic shared memory laid out as
// [kStages][CPL][128] 16-byte chunks (each warp's 32 chunks are contiguous).
template <int CPL>
__global__ void __launch_bounds__(kThreads, 2) adaln_kernel(const AdalnArgs a) {
  extern __shared__ uint4 ring[];
  __shared__ float inv_table[128];
  __shared__ float totals[2][4];
  const float gsf = *a.gsf;
  fill_inverse_scales(inv_table, gsf);

  const int t = threadIdx.x;
  const int64_t chunks = a.cols >> 3;
  const int64_t r_begin = a.rows * blockIdx.x / gridDim.x;
  const int64_t r_end = a.rows * (blockIdx.x + 1) / gridDim.x;
  const uint32_t ring_base = static_cast<uint32_t>(__cvta_generic_to_shared(ring));

  // Copy this thread's chunks of row r into ring stage s; always commit a
  // group (empty past the range) so that group counting stays uniform.
  auto issue = [&](int64_t r, int s) {
    if (r < r_end) {
      const uint16_t* xr = a.x + r * a.ld;
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        const int64_t c = t + j * kThreads;
        if (c < chunks) cp_async16(ring_base + ((s * CPL + j) * kThreads + t) * 16, xr + c * 8);
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) issue(r_begin + s, s);

  float gm[CPL][8], fc[CPL][8], sh[CPL][8];
  int64_t frame = -1;
  __syncthreads();  // inv_table

  int stage = 0;
  for (int64_t r = r_begin; r < r_end; ++r) {
    issue(r + kStages - 1, stage == 0 ? kStages - 1 : stage - 1);
    cp_async_wait<kStages - 1>();

    const int64_t f = frame_of(a, r);  // the same for the whole CTA
    if (f != frame) {
      frame = f;
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        const int64_t c = t + j * kThreads;
        if (c < chunks) load_tables(a, f, c, gm[j], fc[j], sh[j]);
      }
    }

    const uint4* buf = ring + stage * CPL * kThreads + t;
    float2 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int j = 0; j < CPL; ++j)
      if (t + j * kThreads < chunks) accumulate(buf[j * kThreads], acc);
    const float rstd = rstd_of(row_sum_of_squares(acc, totals, static_cast<int>(r & 1)), a.cols, a.eps);
    if (a.row_rstd != nullptr && t == 0) a.row_rstd[r] = rstd;

#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      const int64_t c = t + j * kThreads;
      if (j * kThreads >= chunks) break;  // CTA-uniform
      emit_chunk(a, r, c, c < chunks, buf[j * kThreads], rstd, gm[j], fc[j], sh[j], gsf, inv_table);
    }
    stage = stage == kStages - 1 ? 0 : stage + 1;
  }
  cp_async_wait<0>();
  zero_padding_rows(a);
}


// Any width: the same chunk-to-thread mapping and order, x read from global
// memory in both passes (the second read mostly hits L2) and the tables read
// per chunk and row.
__global__ void __launch_bounds__(kThreads) adaln_generic_kernel(const AdalnArgs a) {
  __shared__ float inv_table[128];
  __shared__ float totals[2][4];
  const float gsf = *a.gsf;
  fill_inverse_scales(inv_table, gsf);
  __syncthreads();

  const int t = threadIdx.x;
  const int64_t chunks = a.cols >> 3;
  const int64_t r_begin = a.rows * blockIdx.x / gridDim.x;
  const int64_t r_end = a.rows * (blockIdx.x + 1) / gridDim.x;
  for (int64_t r = r_begin; r < r_end; ++r) {
    const int64_t f = frame_of(a, r);
    const uint16_t* xr = a.x + r * a.ld;
    float2 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.0f, 0.0f);
    for (int64_t c = t; c < chunks; c += kThreads) accumulate(load16_stream(xr + c * 8), acc);
    const float rstd = rstd_of(row_sum_of_squares(acc, totals, static_cast<int>(r & 1)), a.cols, a.eps);
    if (a.row_rstd != nullptr && t == 0) a.row_rstd[r] = rstd;
    for (int64_t c0 = 0; c0 < chunks; c0 += kThreads) {  // CTA-uniform trip count
      const int64_t c = c0 + t;
      const bool valid = c < chunks;
      float gm[8], fc[8], sh[8];
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (valid) {
        v = load16_reused(xr + c * 8);
        load_tables(a, f, c, gm, fc, sh);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) gm[i] = fc[i] = sh[i] = 0.0f;
      }
      emit_chunk(a, r, c, valid, v, rstd, gm, fc, sh, gsf, inv_table);
    }
  }
  zero_padding_rows(a);
}

template <int CPL>
cudaError_t launch_resident(const AdalnArgs& a, cudaStream_t stream) {
  const int smem = kStages * CPL * kThreads * 16;
  int blocks = 0;
  cudaError_t err = persistent_blocks(reinterpret_cast<const void*>(&adaln_kernel<CPL>), kThreads,
                                      smem, a.rows > 0 ? a.rows : 1, &blocks);
  if (err != cudaSuccess) return err;
  adaln_kernel<CPL><<<blocks, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_generic(const AdalnArgs& a, cudaStream_t stream) {
  int blocks = 0;
  cudaError_t err = persistent_blocks(reinterpret_cast<const void*>(&adaln_generic_kernel),
                                      kThreads, 0, a.rows > 0 ? a.rows : 1, &blocks);
  if (err != cudaSuccess) return err;
  adaln_generic_kernel<<<blocks, kThreads, 0, stream>>>(a);
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
  const int64_t per_thread = (cols / 8 + kThreads - 1) / kThreads;  // chunks per thread
  if (per_thread <= 1) return launch_resident<1>(a, stream);
  if (per_thread <= 2) return launch_resident<2>(a, stream);
  if (per_thread <= 4) return launch_resident<4>(a, stream);
  if (per_thread <= 7) return launch_resident<7>(a, stream);
  if (per_thread <= 8) return launch_resident<8>(a, stream);
  return launch_generic(a, stream);
}

}  // namespace h3q
