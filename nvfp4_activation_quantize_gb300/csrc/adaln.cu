// adaln.cu -- RMSNorm with fp32 statistics + AdaLN modulation + NVFP4.
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
// x streams through a ring of row pairs in shared memory filled with cp.async:
// each thread copies exactly the chunks it will read, so the data needs no
// barrier, only the thread's own cp.async.wait_group.  With four pairs in the
// ring, three are in flight or waiting while one is computed, so a pair's
// copy is issued two iterations before its pass 1.  Rows are processed in pairs,
// which shares one barrier and the table registers between two independent
// rows' arithmetic.
// Rows of exactly 7,168 columns take a block-per-thread kernel (one CTA of
// 448 threads per SM, described above it) with the same pass-1 order; rows
// wider than 8,192 take a generic kernel with the same chunk-to-thread
// mapping and order that reads x twice and the tables per row.
#include "h3q_device.cuh"
#include "h3q_internal.h"

namespace h3q {
namespace {

constexpr int kThreads = 128;   // CTA size of the generic kernel
constexpr int kLanes128 = 128;  // the lanes of the canonical order
constexpr int kBlockStages = 5;  // ring stages of the 7,168-column kernel (215 KB of shared memory)

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
  float* amax;  // abs-max pass: fold max |y| into *amax instead of quantizing (codes, scales unused)
  const float* rstd_in;  // each row's rstd given (from an abs-max pass): the statistics are not formed
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

__device__ __forceinline__ int64_t clamp_frame(const AdalnArgs& a, int64_t t) {
  return t < 0 ? 0 : (t >= a.num_frames ? a.num_frames - 1 : t);  // memory safety only
}

__device__ __forceinline__ int64_t frame_of(const AdalnArgs& a, int64_t row) {
  return clamp_frame(a, a.row_frame ? static_cast<int64_t>(a.row_frame[row]) : row / a.rows_per_frame);
}

// Frame of increasing rows without a division per row: with rows_per_frame the
// cursor keeps the first row of the next frame and steps across boundaries.
struct FrameCursor {
  int64_t frame, next;
  __device__ __forceinline__ FrameCursor(const AdalnArgs& a, int64_t row) {
    frame = a.row_frame ? 0 : row / a.rows_per_frame;
    next = a.row_frame ? 0 : (frame + 1) * a.rows_per_frame;
  }
  __device__ __forceinline__ int64_t at(const AdalnArgs& a, int64_t row) {
    if (a.row_frame) return clamp_frame(a, a.row_frame[row]);
    while (row >= next) {
      ++frame;
      next += a.rows_per_frame;
    }
    return clamp_frame(a, frame);
  }
  // the same for decreasing rows: next - rows_per_frame is the frame's first row
  __device__ __forceinline__ int64_t at_down(const AdalnArgs& a, int64_t row) {
    if (a.row_frame) return clamp_frame(a, a.row_frame[row]);
    while (row < next - a.rows_per_frame) {
      --frame;
      next -= a.rows_per_frame;
    }
    return clamp_frame(a, frame);
  }
};

// gamma and 1 + scale of chunk c of frame t as fp32 pairs (elements 2i, 2i+1)
// for the paired multiplies, and the shift as the bf16 pairs it is stored in
// (the final add takes bf16 operands directly).
struct ChunkTables {
  float2 gm[4], fc[4];
  uint32_t sh[4];
};

__device__ __forceinline__ void load_tables(const AdalnArgs& a, int64_t t, int64_t c,
                                            ChunkTables& tb) {
  const uint16_t* shift = a.table + t * 2 * a.cols + c * 8;
  const uint4 g4 = load16_reused(a.gamma + c * 8);
  const uint4 s4 = load16_reused(shift + a.cols);
  const uint4 h4 = load16_reused(shift);
  const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w};
  const uint32_t sw[4] = {s4.x, s4.y, s4.z, s4.w};
  const uint32_t hw[4] = {h4.x, h4.y, h4.z, h4.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    tb.gm[i] = bf16x2_to_float2(gw[i]);
    tb.fc[i] = add2(make_float2(1.0f, 1.0f), bf16x2_to_float2(sw[i]));
    tb.sh[i] = hw[i];
  }
}

// Partials (p_2i, p_2i+1) in acc[i]; element e of the chunk goes to p_e.
// The squares come from the bf16 halves directly (fma.rn.f32.bf16: exact
// product of two bf16 values, one rounding with the fp32 partial).
__device__ __forceinline__ void accumulate(const uint4& v, float2 (&acc)[4]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "fma.rn.f32.bf16 %0, l, l, %0;\n\tfma.rn.f32.bf16 %1, h, h, %1;\n\t}"
        : "+f"(acc[i].x), "+f"(acc[i].y)
        : "r"(w[i]));
  }
}

// Row sums of squares of R rows from this thread's partials, in two halves
// around a CTA barrier: post_totals forms the lane totals, runs the warp
// butterfly and leaves each warp's total in totals[slot]; after a barrier,
// gather_totals combines the four warp totals as (T0+T1)+(T2+T3).
template <int R>
__device__ __forceinline__ void post_totals(const float2 (&acc)[R][4], float (*totals)[R][4],
                                            int slot) {
  float tot[R];
#pragma unroll
  for (int k = 0; k < R; ++k) {
    tot[k] = __fadd_rn(
        __fadd_rn(__fadd_rn(acc[k][0].x, acc[k][0].y), __fadd_rn(acc[k][1].x, acc[k][1].y)),
        __fadd_rn(__fadd_rn(acc[k][2].x, acc[k][2].y), __fadd_rn(acc[k][3].x, acc[k][3].y)));
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
    for (int k = 0; k < R; ++k) tot[k] = __fadd_rn(tot[k], __shfl_xor_sync(0xffffffffu, tot[k], o));
  if ((threadIdx.x & 31) == 0)  // warp index within the 128-lane group
#pragma unroll
    for (int k = 0; k < R; ++k) totals[slot][k][(threadIdx.x >> 5) & 3] = tot[k];
}

template <int R>
__device__ __forceinline__ void gather_totals(float (*totals)[R][4], int slot, float (&ss)[R]) {
#pragma unroll
  for (int k = 0; k < R; ++k) {
    const float* T = totals[slot][k];
    ss[k] = __fadd_rn(__fadd_rn(T[0], T[1]), __fadd_rn(T[2], T[3]));
  }
}

template <int R>
__device__ __forceinline__ void row_sums(const float2 (&acc)[R][4], float (*totals)[R][4],
                                         int slot, float (&ss)[R]) {
  post_totals<R>(acc, totals, slot);
  __syncthreads();
  gather_totals<R>(totals, slot, ss);
}

__device__ __forceinline__ float rstd_of(float ss, float cols, float eps) {
  const float mean = __fdiv_rn(ss, cols);
  return __frcp_rn(__fsqrt_rn(__fadd_rn(mean, eps)));
}

// Modulate one chunk of R rows (x words v[k], statistics rstd[k]) with the
// chunk's tables, quantize this thread's half block of each row, store its four
// code bytes at codes_at[k] and, from the even thread of the pair, the block's
// scale byte at scale_at[k].  All 32 lanes of the warp call this (it
// shuffles); `valid` masks the stores.  With AMAX the chunk's max |y| is
// folded into run_max instead (for valid chunks) and nothing is stored.
template <int R, bool AMAX>
__device__ __forceinline__ void emit_chunk(const uint4 (&v)[R], const float (&rstd)[R],
                                           const ChunkTables& tb, bool valid,
                                           uint8_t* const (&codes_at)[R],
                                           uint8_t* const (&scale_at)[R], float gsf,
                                           const float* inv_table, float& run_max) {
  const int lane = threadIdx.x & 31;
  // Stages run across all R rows before the next stage, so that the rows'
  // independent work sits side by side for the scheduler.
  uint32_t y[R][4];
#pragma unroll
  for (int k = 0; k < R; ++k) {
    const uint32_t xw[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
    const float2 rstd2 = make_float2(rstd[k], rstd[k]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 n = mul2(bf16x2_to_float2(xw[i]), rstd2);
      const float2 h = mul2(n, tb.gm[i]);
      const float2 m = mul2(h, tb.fc[i]);
      y[k][i] = float2_to_bf16x2(add_bf16x2_f32(tb.sh[i], m));
    }
  }
  float amax[R];
#pragma unroll
  for (int k = 0; k < R; ++k)
    amax[k] = halves_amax(absmax_bf16x2(absmax_bf16x2(y[k][0], y[k][1]),
                                        absmax_bf16x2(y[k][2], y[k][3])));
  if constexpr (AMAX) {
#pragma unroll
    for (int k = 0; k < R; ++k)
      if (valid) run_max = fmaxf(run_max, amax[k]);
  } else {
#pragma unroll
    for (int k = 0; k < R; ++k) amax[k] = fmaxf(amax[k], __shfl_xor_sync(0xffffffffu, amax[k], 1));
#pragma unroll
    for (int k = 0; k < R; ++k) {
      const uint32_t sf = block_scale(amax[k], gsf);
      const uint32_t codes = codes8(y[k], inv_table[sf]);
      if (valid) store_word(codes_at[k], codes);
      // the even thread of the pair writes the block's scale byte
      if (valid && !(lane & 1)) store_byte(scale_at[k], sf);
    }
  }
}

// Zero scale words of the padding rows rows..pad128(rows)-1, spread over CTAs.
__device__ __forceinline__ void zero_padding_rows(const AdalnArgs& a) {
  const int64_t prows = (a.rows + 127) >> 7 << 7;
  const int64_t quads = a.cols >> 6;
  for (int64_t p = a.rows + blockIdx.x; p < prows; p += gridDim.x)
    for (int64_t q = threadIdx.x; q < quads; q += blockDim.x)
      store_word(a.scales + scale_word_offset(p, q, quads), 0u);
}

// Rows up to 128 * C1 chunks (C1 * 1,024 columns), with NT threads per CTA and
// S row pairs in the ring (S - 1 pairs in flight ahead of the one computed).
// Pass 1 runs on threads 0..127, the lanes of the canonical order, C1 chunks
// each (chunk c on lane c % 128).  Pass 2 is element-wise, so it spreads the
// row over all NT threads, J chunks each (chunk c on thread c % NT); a thread
// keeps the tables of its J chunks in registers (gamma and 1 + scale as fp32
// pairs, the shift as bf16 pairs), so more threads mean fewer registers each.
// x streams through a cp.async ring in dynamic shared memory,
// [S][2 rows][128 * C1 chunks] of 16 bytes, copied by the pass-1
// lanes chunk by chunk as they will read it.  Rows go in consecutive pairs
// with a skewed pipeline: the iteration for pair p forms the partial sums of
// pair p+1 and modulates and quantizes pair p, then one barrier publishes
// pair p+1's warp totals.  Pass 2 of pair p reads chunks copied by other
// threads; every thread's wait for pair p came before the previous barrier.
template <int NT, int J, int C1, int S, bool FULL, bool AMAX>
__global__ void __launch_bounds__(NT, 2) adaln_kernel(const AdalnArgs a) {
  constexpr int kRow = kLanes128 * C1;  // chunk slots per row in the ring
  extern __shared__ uint4 ring[];
  __shared__ float inv_table[128];
  __shared__ float totals[2][2][4];
  const float gsf = AMAX ? 0.0f : *a.gsf;
  if (!AMAX) fill_inverse_scales(inv_table, gsf);
  float run_max = 0.0f;

  const int t = threadIdx.x;
  const bool lane1 = t < kLanes128;  // a pass-1 lane (warp-uniform)
  const int64_t chunks = a.cols >> 3;
  const int64_t quads = a.cols >> 6;
  const float cols_f = static_cast<float>(a.cols);  // exact: cols <= 2^24
  const int64_t r_begin = a.rows * blockIdx.x / gridDim.x;
  const int64_t r_end = a.rows * (blockIdx.x + 1) / gridDim.x;
  const int64_t pairs = (r_end - r_begin + 1) >> 1;
  const uint32_t ring_base = static_cast<uint32_t>(__cvta_generic_to_shared(ring));

  // The pass-1 lanes copy their chunks of pair p into ring stage s; every
  // thread commits a group (empty for the others and past the range).
  const uint16_t* x_t = a.x + t * 8;
  const uint32_t ring_t = ring_base + t * 16;
  auto issue = [&](int64_t p, int s) {
    if (lane1) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int64_t r = r_begin + 2 * p + k;
        if (r < r_end) {
          const uint16_t* xr = x_t + r * a.ld;
          const uint32_t dst = ring_t + (s * 2 + k) * (kRow * 16);
#pragma unroll
          for (int j = 0; j < C1; ++j)
            if (FULL || t + j * kLanes128 < chunks)
              cp_async16(dst + j * (kLanes128 * 16), xr + j * (kLanes128 * 8));
        }
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int s = 0; s < S - 1; ++s) issue(s, s);

  ChunkTables tb[J];
  int64_t frame = -1;
  FrameCursor cursor(a, r_begin);
  auto use_frame = [&](int64_t f) {  // CTA-uniform
    if (f == frame) return;
    frame = f;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int64_t c = t + j * NT;
      if (FULL || c < chunks) load_tables(a, f, c, tb[j]);
    }
  };

  auto partial_sums = [&](int64_t p, int s) {  // pass 1 of pair p from stage s (lanes only)
    if (!lane1) return;
    const int64_t r0 = r_begin + 2 * p;
    const bool has1 = r0 + 1 < r_end;
    const uint4* buf = ring + s * 2 * kRow + t;
    float2 acc[2][4];
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[k][i] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int j = 0; j < C1; ++j) {
      if (FULL || t + j * kLanes128 < chunks) {
        accumulate(buf[j * kLanes128], acc[0]);
        if (has1) accumulate(buf[kRow + j * kLanes128], acc[1]);
      }
    }
    post_totals<2>(acc, totals, static_cast<int>(p & 1));
  };
  auto statistics = [&](int64_t p, float (&rstd)[2]) {  // after the barrier
    float ss[2];
    gather_totals<2>(totals, static_cast<int>(p & 1), ss);
    rstd[0] = rstd_of(ss[0], cols_f, a.eps);
    rstd[1] = rstd_of(ss[1], cols_f, a.eps);
    if (a.rstd_in != nullptr) {  // the rows' rstd given
      const int64_t r = r_begin + 2 * p;
      rstd[0] = a.rstd_in[r];
      rstd[1] = r + 1 < r_end ? a.rstd_in[r + 1] : 0.0f;
    }
  };

  float rstd[2] = {0.0f, 0.0f};
  if (pairs > 0) {
    cp_async_wait<S - 2>();  // pair 0 landed (this thread's copies)
    partial_sums(0, 0);
  }
  __syncthreads();  // inv_table, pair 0's totals, every thread's pair-0 copies
  if (pairs > 0) statistics(0, rstd);

  int stage = 0;
  for (int64_t p = 0; p < pairs; ++p) {
    const int next = stage == S - 1 ? 0 : stage + 1;
    issue(p + S - 1, stage == 0 ? S - 1 : stage - 1);
    cp_async_wait<S - 2>();  // pair p+1 landed (this thread's copies)
    const bool more = p + 1 < pairs;   // CTA-uniform
    if (more) partial_sums(p + 1, next);

    const int64_t r0 = r_begin + 2 * p;
    const bool has1 = r0 + 1 < r_end;  // CTA-uniform
    const uint4* buf = ring + stage * 2 * kRow + t;
    if (a.row_rstd != nullptr && t == 0) {
      a.row_rstd[r0] = rstd[0];
      if (has1) a.row_rstd[r0 + 1] = rstd[1];
    }
    uint8_t* code_base[2];
    uint8_t* scale_base[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      code_base[k] = a.codes + (r0 + k) * (a.cols >> 1) + t * 4;
      scale_base[k] = a.scales + scale_row_offset(r0 + k, quads) + (t >> 3) * 512 + ((t >> 1) & 3);
    }
    const int64_t f0 = cursor.at(a, r0);
    const int64_t f1 = has1 ? cursor.at(a, r0 + 1) : f0;
    if (has1 && f0 == f1) {
      use_frame(f0);
#pragma unroll
      for (int j = 0; j < J; ++j) {
        if (!FULL && j * NT >= chunks) break;  // CTA-uniform
        const uint4 v[2] = {buf[j * NT], buf[kRow + j * NT]};
        uint8_t* const ca[2] = {code_base[0] + j * (NT * 4), code_base[1] + j * (NT * 4)};
        uint8_t* const sa[2] = {scale_base[0] + j * (NT / 8 * 512), scale_base[1] + j * (NT / 8 * 512)};
        emit_chunk<2, AMAX>(v, rstd, tb[j], FULL || t + j * NT < chunks, ca, sa, gsf, inv_table, run_max);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        if (k == 1 && !has1) break;
        use_frame(k == 0 ? f0 : f1);
#pragma unroll
        for (int j = 0; j < J; ++j) {
          if (!FULL && j * NT >= chunks) break;
          const uint4 v[1] = {buf[k * kRow + j * NT]};
          const float rs[1] = {rstd[k]};
          uint8_t* const ca[1] = {code_base[k] + j * (NT * 4)};
          uint8_t* const sa[1] = {scale_base[k] + j * (NT / 8 * 512)};
          emit_chunk<1, AMAX>(v, rs, tb[j], FULL || t + j * NT < chunks, ca, sa, gsf, inv_table, run_max);
        }
      }
    }
    __syncthreads();  // pair p+1's totals and every thread's pair-(p+1) copies
    if (more) statistics(p + 1, rstd);
    stage = next;
  }
  cp_async_wait<0>();
  if (AMAX)
    commit_amax(run_max, a.amax, inv_table);  // inv_table is unused in this mode
  else
    zero_padding_rows(a);
}

// Any width: the same chunk-to-thread mapping and order, x read from global
// memory in both passes (the second read mostly hits L2) and the tables read
// per chunk and row.
template <bool AMAX>
__global__ void __launch_bounds__(kThreads) adaln_generic_kernel(const AdalnArgs a) {
  __shared__ float inv_table[128];
  __shared__ float totals[2][1][4];
  const float gsf = AMAX ? 0.0f : *a.gsf;
  if (!AMAX) fill_inverse_scales(inv_table, gsf);
  float run_max = 0.0f;
  __syncthreads();

  const int t = threadIdx.x;
  const int64_t chunks = a.cols >> 3;
  const int64_t quads = a.cols >> 6;
  const int64_t r_begin = a.rows * blockIdx.x / gridDim.x;
  const int64_t r_end = a.rows * (blockIdx.x + 1) / gridDim.x;
  for (int64_t r = r_begin; r < r_end; ++r) {
    const int64_t f = frame_of(a, r);
    const uint16_t* xr = a.x + r * a.ld;
    float2 acc[1][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[0][i] = make_float2(0.0f, 0.0f);
    for (int64_t c = t; c < chunks; c += kThreads) accumulate(load16_stream(xr + c * 8), acc[0]);
    float ss[1];
    row_sums<1>(acc, totals, static_cast<int>(r & 1), ss);
    const float rstd[1] = {a.rstd_in != nullptr ? a.rstd_in[r] : rstd_of(ss[0], static_cast<float>(a.cols), a.eps)};
    if (a.row_rstd != nullptr && t == 0) a.row_rstd[r] = rstd[0];
    for (int64_t c0 = 0; c0 < chunks; c0 += kThreads) {  // CTA-uniform trip count
      const int64_t c = c0 + t;
      const bool valid = c < chunks;
      ChunkTables tb;
      uint4 v[1] = {make_uint4(0u, 0u, 0u, 0u)};
      if (valid) {
        v[0] = load16_reused(xr + c * 8);
        load_tables(a, f, c, tb);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          tb.gm[i] = tb.fc[i] = make_float2(0.0f, 0.0f);
          tb.sh[i] = 0u;
        }
      }
      uint8_t* const ca[1] = {a.codes + r * (a.cols >> 1) + c * 4};
      uint8_t* const sa[1] = {a.scales + scale_row_offset(r, quads) + (c >> 3) * 512 + ((c >> 1) & 3)};
      emit_chunk<1, AMAX>(v, rstd, tb, valid, ca, sa, gsf, inv_table, run_max);
    }
  }
  if (AMAX)
    commit_amax(run_max, a.amax, inv_table);
  else
    zero_padding_rows(a);
}

__device__ __forceinline__ void named_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// bf16(v) as the fp32 value it stands for: cvt.rn.bf16x2 puts bf16(v) in the
// upper half and bf16(0) = 0 in the lower, which is that value's fp32 pattern.
__device__ __forceinline__ float bf16_round(float v) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(v), "f"(0.0f));
  return __uint_as_float(r);
}

// Modulate and quantize one full 16-element block (x words v[k][0..7], chunks
// 2b and 2b+1) of R rows, and store its 8 code bytes and scale byte per row
// (with AMAX: fold the block's max |y| into run_max instead).
template <int R, bool AMAX>
__device__ __forceinline__ void emit_block(const uint32_t (&v)[R][8], const float (&rstd)[R],
                                           const ChunkTables (&tb)[2],
                                           uint8_t* const (&codes_at)[R],
                                           uint8_t* const (&scale_at)[R], float gsf,
                                           const float* inv_table, float& run_max) {
  if constexpr (AMAX) {
    // bf16 rounding is monotone in the magnitude, so max |bf16(o)| = bf16(max |o|):
    // the unrounded values' maximum is rounded once per block
#pragma unroll
    for (int k = 0; k < R; ++k) {
      const float2 rstd2 = make_float2(rstd[k], rstd[k]);
      float am = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const ChunkTables& t = tb[i >> 2];
        const float2 n = mul2(bf16x2_to_float2(v[k][i]), rstd2);
        const float2 h = mul2(n, t.gm[i & 3]);
        const float2 m = mul2(h, t.fc[i & 3]);
        const float2 o = add_bf16x2_f32(t.sh[i & 3], m);
        am = fmaxf(am, fmaxf(fabsf(o.x), fabsf(o.y)));
      }
      run_max = fmaxf(run_max, fabsf(bf16_round(am)));
    }
  } else {
    float2 y[R][8];
#pragma unroll
    for (int k = 0; k < R; ++k) {
      const float2 rstd2 = make_float2(rstd[k], rstd[k]);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const ChunkTables& t = tb[i >> 2];
        const float2 n = mul2(bf16x2_to_float2(v[k][i]), rstd2);
        const float2 h = mul2(n, t.gm[i & 3]);
        const float2 m = mul2(h, t.fc[i & 3]);
        const float2 o = add_bf16x2_f32(t.sh[i & 3], m);
        y[k][i] = make_float2(bf16_round(o.x), bf16_round(o.y));
      }
    }
#pragma unroll
    for (int k = 0; k < R; ++k) {
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fmaxf(fabsf(y[k][i].x), fabsf(y[k][i].y)));
      const uint32_t sf = block_scale(amax, gsf);
      const float inv = inv_table[sf];
      const float2 inv2 = make_float2(inv, inv);
      const uint32_t lo = e2m1x8(mul2(y[k][0], inv2), mul2(y[k][1], inv2), mul2(y[k][2], inv2), mul2(y[k][3], inv2));
      const uint32_t hi = e2m1x8(mul2(y[k][4], inv2), mul2(y[k][5], inv2), mul2(y[k][6], inv2), mul2(y[k][7], inv2));
      store_codes(codes_at[k], lo, hi);
      store_byte(scale_at[k], sf);
    }
  }
}

// Rows of exactly 16 * NB columns with NB = 448 (7,168, the attention width):
// one CTA of NB threads per SM, thread t owning 16-element block t of every row
// in pass 2, so a thread quantizes whole blocks (one scale computation per
// block, no exchange between threads) and keeps the tables of only 16 columns
// (40 registers).  Pass 1 keeps the canonical order: R = NB / 128 = 3 groups of
// 128 lanes (four warps each), group g summing row g of each 3-row step (chunk c
// on lane c % 128).  x streams through a ring of kStages steps of R rows, each
// pass-1 lane copying its own chunks; chunk c sits at slot c ^ ((c >> 3) & 1),
// which keeps both the pass-1 reads (lane l, chunk l + 128 j) and the pass-2
// reads (thread t, chunks 2t and 2t + 1) free of bank conflicts.
// One warp, the stats warp, does no pass 1: per row of a step it publishes the
// rstd (from the warp totals, one lane per row), the frame and the row's scale
// offset in shared memory, so the per-row bookkeeping is done once per row, not
// once per thread.  The warps are not held in step
// with one another.  Each of the other 13 warps waits on a named barrier of its
// own (count 64) on which the stats warp arrives once the step's rows are
// published; a warp that is ahead goes on without waiting for the slowest.
// After passing its own barrier of step q, each of them arrives on one shared
// barrier that only the stats warp waits on before it publishes step q + 1 (and
// only then emits step q itself, so its own pass 2 is off the others' path).
// That arrival says the warp has posted its pass-1 totals of step q + 1 and
// finished pass 2 of step q - 1, so neither the published rows nor the totals
// are overwritten while still to be read, and no warp arrives twice in one phase
// of any barrier.  A warp past its barrier of step q thus knows that every warp
// has finished pass 2 of step q - 2, and refills that stage; with five stages a
// step's copies are issued two steps before its pass 1.  The stats warp is warp
// 2: warps go to the SM's four sub-partitions by warp index mod 4, and
// sub-partition 2 holds three of the 14 warps, not four.  Pass 1 runs on 12 of
// the other 13 warps (three rows of four 32-lane groups).

// Per-row values published by the stats warp for one step.
struct RowInfo {
  float rstd;
  int32_t frame;
  int64_t scale_off;  // byte offset of the row's part of a scale word (scale_row_offset)
};

template <int NB, int C1, bool AMAX, bool GIVEN = false>
__global__ void __launch_bounds__(NB, 1) adaln_block_kernel(const AdalnArgs a) {
  constexpr int R = NB / kLanes128;
  constexpr int kStages = kBlockStages;
  constexpr int kAhead = kStages - 2;  // steps in flight ahead of the step being emitted
  constexpr int kChunks = kLanes128 * C1;
  constexpr int64_t kCodeRow = 8 * NB;  // code bytes per row (cols / 2)
  static_assert(kChunks == 2 * NB, "one thread per 16-element block");
  constexpr int kStatsWarp = 2;
  // The warp with neither pass 1 nor the statistics: on sub-partition 1 for the
  // quantizing instance; on sub-partition 2, beside the stats warp, for the
  // abs-max pass, whose lighter pass 2 leaves pass 1 a larger share of the work.
  constexpr int kPass2Only = AMAX ? 6 : NB / 32 - 1;
  static_assert(NB / 32 == R * 4 + 2 && NB / 32 - 1 <= 13 && kPass2Only != kStatsWarp,
                "one stats warp, one pass-2-only warp, a named barrier (3..15) per warp but the stats warp");
  extern __shared__ uint4 ring[];  // [kStages][R][kChunks]
  __shared__ float inv_table[128];
  __shared__ float totals[2][R][4];
  __shared__ RowInfo rows_s[2][R];
  const float gsf = AMAX ? 0.0f : *a.gsf;
  if (!AMAX) fill_inverse_scales(inv_table, gsf);
  float run_max = 0.0f;

  const int t = threadIdx.x;
  const int warp = t >> 5;
  const int lane = t & 31;
  const int pi = warp < kStatsWarp ? warp : warp - 1;  // index among the warps but the stats warp
  constexpr bool kLastPass2Only = kPass2Only == NB / 32 - 1;
  const int ppi = kLastPass2Only ? pi : pi - (warp > kPass2Only ? 1 : 0);  // index among the pass-1 warps
  const bool p1 = warp != kStatsWarp && (kLastPass2Only ? pi < R * 4 : warp != kPass2Only);  // warp-uniform
  const int grp = ppi >> 2;
  const int l = (ppi & 3) * 32 + lane;
  const int64_t quads = a.cols >> 6;
  const float cols_f = static_cast<float>(a.cols);
  const int64_t r_begin = a.rows * blockIdx.x / gridDim.x;
  const int64_t r_end = a.rows * (blockIdx.x + 1) / gridDim.x;
  // steps of this CTA: rows / (blocks * R) + 1 < 2^31 for any x that fits a device
  const int steps = static_cast<int>((r_end - r_begin + R - 1) / R);
  const uint32_t ring_base = static_cast<uint32_t>(__cvta_generic_to_shared(ring));

  // The abs-max pass takes the rows of its range from the end to the start (row
  // r_end - 1 - i where the producer takes r_begin + i): the producer that
  // follows starts each range at its first rows, the last ones this pass read,
  // part of them still in L2 (a maximum and a row's rstd do not depend on the
  // order).
  constexpr bool kReverse = AMAX;

  // pass-1 lanes: the next row to copy and its ring slot
  const uint16_t* x_next = kReverse ? a.x + (r_end - 1 - grp) * a.ld + l * 8 : a.x + (r_begin + grp) * a.ld + l * 8;
  const int64_t x_step = kReverse ? -R * a.ld : R * a.ld;
  const int l_slot = l ^ ((l >> 3) & 1);  // chunk c at slot c ^ ((c >> 3) & 1): conflict-free in both passes
  const uint32_t ring_l = ring_base + static_cast<uint32_t>(grp * kChunks + l_slot) * 16;
  // a step's ring stage is its index mod kStages, kept by a wrapping counter
  auto stage_after = [](int s, int k) { return s + k >= kStages ? s + k - kStages : s + k; };
  int issued = 0;  // steps issued so far
  auto issue = [&](int stage) {  // the next step, into this stage
    if (p1 && issued < steps && r_begin + R * int64_t{issued} + grp < r_end) {
      const uint32_t dst = ring_l + static_cast<uint32_t>(stage * R * kChunks) * 16;
#pragma unroll
      for (int j = 0; j < C1; ++j) cp_async16(dst + j * (kLanes128 * 16), x_next + j * (kLanes128 * 8));
    }
    cp_async_commit();
    x_next += x_step;
    ++issued;
  };
  auto pass1 = [&](int q, int stage) {
    if (GIVEN || q >= steps || !p1) return;  // GIVEN: the rows' rstd are given, no sums
    float2 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.0f, 0.0f);
    if (r_begin + R * int64_t{q} + grp < r_end) {
      const uint4* buf = ring + (stage * R + grp) * kChunks + l_slot;
#pragma unroll
      for (int j = 0; j < C1; ++j) accumulate(buf[j * kLanes128], acc);
    }
    float tot = __fadd_rn(__fadd_rn(__fadd_rn(acc[0].x, acc[0].y), __fadd_rn(acc[1].x, acc[1].y)),
                          __fadd_rn(__fadd_rn(acc[2].x, acc[2].y), __fadd_rn(acc[3].x, acc[3].y)));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) tot = __fadd_rn(tot, __shfl_xor_sync(0xffffffffu, tot, o));
    if (lane == 0) totals[q & 1][grp][ppi & 3] = tot;
  };
  // the stats warp: lane k < R publishes row k of step q.  GIVEN: the rstd is read
  // a step ahead of its publication, so the load is off the publishing chain.
  FrameCursor lane_cursor(a, kReverse ? (r_end > r_begin ? r_end - 1 : r_begin) : r_begin + (lane < R ? lane : 0));
  float given = 0.0f;
  auto fetch_given = [&](int q) {
    const int64_t r = r_begin + R * int64_t{q} + lane;
    if (GIVEN && q < steps && lane < R && r < r_end) given = a.rstd_in[r];
  };
  fetch_given(0);
  auto stats = [&](int q) {
    if (q >= steps || lane >= R) return;
    const int64_t r = kReverse ? r_end - 1 - (R * int64_t{q} + lane) : r_begin + R * int64_t{q} + lane;
    const bool valid = kReverse ? r >= r_begin : r < r_end;
    const float* T = totals[q & 1][lane];
    RowInfo info;
    if (GIVEN) {
      info.rstd = given;
      fetch_given(q + 1);
    } else {
      info.rstd = rstd_of(__fadd_rn(__fadd_rn(T[0], T[1]), __fadd_rn(T[2], T[3])), cols_f, a.eps);
    }
    info.frame = valid ? static_cast<int32_t>(kReverse ? lane_cursor.at_down(a, r) : lane_cursor.at(a, r)) : -1;
    info.scale_off = scale_row_offset(r, quads);
    rows_s[q & 1][lane] = info;
    if (a.row_rstd != nullptr && valid) a.row_rstd[r] = info.rstd;
  };

  ChunkTables tb[2];
  int32_t frame = -1;
  auto use_frame = [&](int32_t f) {  // CTA-uniform
    if (f == frame) return;
    frame = f;
    load_tables(a, f, 2 * t, tb[0]);
    load_tables(a, f, 2 * t + 1, tb[1]);
  };

#pragma unroll
  for (int q = 0; q < kAhead; ++q) issue(q);
  cp_async_wait<kAhead - 1>();  // step 0 landed (this thread's copies)
  pass1(0, 0);
  __syncthreads();  // inv_table, step 0's totals and copies
  if (warp == kStatsWarp && steps > 0) {
    stats(0);
    __syncwarp();
#pragma unroll 1
    for (int c = 0; c < NB / 32 - 1; ++c) named_arrive(3 + c, 64);  // rows of step 0 published
  }

  uint8_t* code_step = a.codes + r_begin * kCodeRow + t * 8;
  uint8_t* const scale_t = a.scales + (t >> 2) * 512 + (t & 3);
  int stage = 0;  // of step q
  for (int q = 0; q < steps; ++q, stage = stage_after(stage, 1)) {
    if (warp == kStatsWarp) {
      if (q + 1 < steps) {
        named_sync(2, NB);  // step q+1's totals posted; every warp past its barrier of step q
        stats(q + 1);
        __syncwarp();
#pragma unroll 1
        for (int c = 0; c < NB / 32 - 1; ++c) named_arrive(3 + c, 64);  // rows of step q+1 published
      }
      cp_async_commit();  // keep the group count in step with the copying warps
    } else {
      cp_async_wait<kAhead - 2>();  // step q+1 landed (this thread's copies)
      pass1(q + 1, stage_after(stage, 1));
      named_sync(3 + pi, 64);  // rows of step q published; every warp done with step q-2
      if (q + 1 < steps) named_arrive(2, NB);  // step q+1's totals posted; done with step q-1
      issue(stage_after(stage, kAhead));  // step q+3 into step q-2's stage
    }

    const int n = static_cast<int>(r_end - r_begin - R * int64_t{q} < R ? r_end - r_begin - R * int64_t{q} : R);
    const uint4* buf = ring + stage * R * kChunks + 2 * t;
    const int sw = (t >> 2) & 1;
    RowInfo info[R];
    bool one_frame = n == R;  // all R rows present and in one frame (frames need not be monotone)
#pragma unroll
    for (int k = 0; k < R; ++k) {
      info[k] = rows_s[q & 1][k];
      one_frame = one_frame && info[k].frame == info[0].frame;
    }
    if (one_frame) {
      use_frame(info[0].frame);
      uint32_t v[R][8];
      float rs[R];
      uint8_t* ca[R];
      uint8_t* sa[R];
#pragma unroll
      for (int k = 0; k < R; ++k) {
        const uint4 lo = buf[k * kChunks + sw], hi = buf[k * kChunks + 1 - sw];
        v[k][0] = lo.x; v[k][1] = lo.y; v[k][2] = lo.z; v[k][3] = lo.w;
        v[k][4] = hi.x; v[k][5] = hi.y; v[k][6] = hi.z; v[k][7] = hi.w;
        rs[k] = info[k].rstd;
        ca[k] = code_step + k * kCodeRow;
        sa[k] = scale_t + info[k].scale_off;
      }
      emit_block<R, AMAX>(v, rs, tb, ca, sa, gsf, inv_table, run_max);
    } else {
#pragma unroll
      for (int k = 0; k < R; ++k) {
        if (k >= n) break;  // CTA-uniform
        use_frame(info[k].frame);
        uint32_t v[1][8];
        const uint4 lo = buf[k * kChunks + sw], hi = buf[k * kChunks + 1 - sw];
        v[0][0] = lo.x; v[0][1] = lo.y; v[0][2] = lo.z; v[0][3] = lo.w;
        v[0][4] = hi.x; v[0][5] = hi.y; v[0][6] = hi.z; v[0][7] = hi.w;
        const float rs[1] = {info[k].rstd};
        uint8_t* const ca[1] = {code_step + k * kCodeRow};
        uint8_t* const sa[1] = {scale_t + info[k].scale_off};
        emit_block<1, AMAX>(v, rs, tb, ca, sa, gsf, inv_table, run_max);
      }
    }
    code_step += R * kCodeRow;
  }
  cp_async_wait<0>();
  if (AMAX)
    commit_amax(run_max, a.amax, inv_table);  // inv_table is unused in this mode
  else
    zero_padding_rows(a);
}

template <bool AMAX, bool GIVEN>
cudaError_t launch_block7168(const AdalnArgs& a, cudaStream_t stream) {
  constexpr int NB = 448, C1 = 7, R = NB / kLanes128;
  const int smem = kBlockStages * R * kLanes128 * C1 * 16;
  int blocks = 0;
  cudaError_t err = persistent_blocks(reinterpret_cast<const void*>(&adaln_block_kernel<NB, C1, AMAX, GIVEN>),
                                      NB, smem, a.rows > 0 ? (a.rows + R - 1) / R : 1, &blocks);
  if (err != cudaSuccess) return err;
  adaln_block_kernel<NB, C1, AMAX, GIVEN><<<blocks, NB, smem, stream>>>(a);
  return cudaGetLastError();
}

template <int NT, int J, int C1, int S, bool AMAX>
cudaError_t launch_resident(const AdalnArgs& a, cudaStream_t stream) {
  const int smem = S * 2 * kLanes128 * C1 * 16;
  const bool full = a.cols / 8 == int64_t(NT) * J && a.cols / 8 == int64_t(kLanes128) * C1;
  const void* kernel = full ? reinterpret_cast<const void*>(&adaln_kernel<NT, J, C1, S, true, AMAX>)
                            : reinterpret_cast<const void*>(&adaln_kernel<NT, J, C1, S, false, AMAX>);
  int blocks = 0;
  cudaError_t err = persistent_blocks(kernel, NT, smem, a.rows > 0 ? a.rows : 1, &blocks);
  if (err != cudaSuccess) return err;
  if (full)
    adaln_kernel<NT, J, C1, S, true, AMAX><<<blocks, NT, smem, stream>>>(a);
  else
    adaln_kernel<NT, J, C1, S, false, AMAX><<<blocks, NT, smem, stream>>>(a);
  return cudaGetLastError();
}

template <bool AMAX>
cudaError_t launch_generic(const AdalnArgs& a, cudaStream_t stream) {
  int blocks = 0;
  cudaError_t err = persistent_blocks(reinterpret_cast<const void*>(&adaln_generic_kernel<AMAX>),
                                      kThreads, 0, a.rows > 0 ? a.rows : 1, &blocks);
  if (err != cudaSuccess) return err;
  adaln_generic_kernel<AMAX><<<blocks, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

template <bool AMAX>
cudaError_t dispatch(const AdalnArgs& a, cudaStream_t stream) {
  const int64_t chunks = a.cols / 8;
  const int64_t per_lane = (chunks + kLanes128 - 1) / kLanes128;
  // Four pairs in the ring (two in flight ahead of pass 1) while two CTAs still
  // fit an SM's shared memory; three for the widest rows.
  if (per_lane <= 1) return launch_resident<128, 1, 1, 4, AMAX>(a, stream);
  if (per_lane <= 2) return launch_resident<128, 2, 2, 4, AMAX>(a, stream);
  if (per_lane <= 4) return launch_resident<128, 4, 4, 4, AMAX>(a, stream);
  if (chunks == 2 * 448)  // 7,168 columns
    return a.rstd_in != nullptr && !AMAX ? launch_block7168<false, true>(a, stream)
                                         : launch_block7168<AMAX, false>(a, stream);
  if (per_lane <= 7) return launch_resident<128, 7, 7, 4, AMAX>(a, stream);
  if (per_lane <= 8) return launch_resident<128, 8, 8, 3, AMAX>(a, stream);
  return launch_generic<AMAX>(a, stream);
}

}  // namespace

cudaError_t launch_adaln(const uint16_t* x, int64_t ld, const uint16_t* gamma,
                         const uint16_t* table, int64_t num_frames, const int32_t* row_frame,
                         int64_t rows_per_frame, float eps, int64_t rows, int64_t cols,
                         const float* gsf, uint8_t* codes, uint8_t* scales, float* row_rstd,
                         cudaStream_t stream) {
  const AdalnArgs a{x,    ld,   gamma, table,  num_frames, row_frame, rows_per_frame, eps,
                    rows, cols, gsf,   codes,  scales,     row_rstd,  nullptr, nullptr};
  return dispatch<false>(a, stream);
}

cudaError_t launch_adaln_from_rstd(const uint16_t* x, int64_t ld, const uint16_t* gamma, const uint16_t* table,
                                   int64_t num_frames, const int32_t* row_frame, int64_t rows_per_frame,
                                   const float* rstd, int64_t rows, int64_t cols, const float* gsf,
                                   uint8_t* codes, uint8_t* scales, cudaStream_t stream) {
  const AdalnArgs a{x,    ld,   gamma, table,  num_frames, row_frame, rows_per_frame, 0.0f,
                    rows, cols, gsf,   codes,  scales,     nullptr,   nullptr,        rstd};
  return dispatch<false>(a, stream);
}

cudaError_t launch_adaln_amax(const uint16_t* x, int64_t ld, const uint16_t* gamma,
                              const uint16_t* table, int64_t num_frames, const int32_t* row_frame,
                              int64_t rows_per_frame, float eps, int64_t rows, int64_t cols,
                              float* amax, float* row_rstd, cudaStream_t stream) {
  const AdalnArgs a{x,    ld,   gamma,   table,   num_frames, row_frame, rows_per_frame, eps,
                    rows, cols, nullptr, nullptr, nullptr,    row_rstd,  amax,           nullptr};
  return dispatch<true>(a, stream);
}

}  // namespace h3q
