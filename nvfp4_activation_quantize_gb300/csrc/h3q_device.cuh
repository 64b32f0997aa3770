// h3q_device.cuh -- device building blocks of the NVFP4 producers (sm_103a).
//
// One lane owns one 16-element block: it loads the block's 32 bytes of bf16 with
// a single 256-bit load, computes the block's E4M3 scale and its eight bytes of
// packed E2M1 codes in registers, and stores the codes as one 8-byte write.
// Four neighbouring lanes own the four scale columns of one 128x4 swizzle atom
// row, so their scale bytes leave as one 4-byte word.
//
// Arithmetic is binary32 with one rounding per operation: explicit _rn
// intrinsics (never contracted into FMAs), paired f32x2 operations where two
// independent elements take the same step, and correctly rounded division,
// reciprocal and square root.  The library is built with -fmad=false and
// without fast-math, so no expression is fused behind these calls' back.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace h3q {

constexpr int kBlock = 16;          // elements per NVFP4 block
constexpr int kLanes = 32;

// ---------------------------------------------------------------------------
// Memory
// ---------------------------------------------------------------------------

// 32 bytes = 16 bf16 = one NVFP4 block.
struct Block16 {
  uint32_t w[8];
};

// Streaming read of data touched once (activations): bypasses L1 allocation.
__device__ __forceinline__ void load_stream(const void* p, Block16& b) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(b.w[0]), "=r"(b.w[1]), "=r"(b.w[2]), "=r"(b.w[3]), "=r"(b.w[4]),
                 "=r"(b.w[5]), "=r"(b.w[6]), "=r"(b.w[7])
               : "l"(p));
}

// Read of data reused by many rows (gamma, modulation table): cached in L1.
__device__ __forceinline__ void load_reused(const void* p, Block16& b) {
  asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(b.w[0]), "=r"(b.w[1]), "=r"(b.w[2]), "=r"(b.w[3]), "=r"(b.w[4]),
                 "=r"(b.w[5]), "=r"(b.w[6]), "=r"(b.w[7])
               : "l"(p));
}

__device__ __forceinline__ void store_codes(uint8_t* p, uint32_t lo, uint32_t hi) {
  asm volatile("st.global.v2.b32 [%0], {%1,%2};" ::"l"(p), "r"(lo), "r"(hi) : "memory");
}

__device__ __forceinline__ void store_word(uint8_t* p, uint32_t v) {
  asm volatile("st.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// Number formats
// ---------------------------------------------------------------------------

// bf16 pair (low half = element 2i, high half = element 2i+1) -> two fp32.
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Two fp32 -> bf16 pair, round to nearest even.
__device__ __forceinline__ uint32_t float2_to_bf16x2(float2 v) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(v.y), "f"(v.x));
  return r;
}

// E4M3 encode: round to nearest even, saturating at 448 (0x7E).
__device__ __forceinline__ uint32_t e4m3_encode(float s) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(r) : "f"(s));
  return r & 0xffu;
}

// E4M3 decode of a non-negative finite code: exponent bias 7, three mantissa
// bits, subnormals m * 2^-9 (exact construction of the binary32 value).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  const uint32_t e = (code >> 3) & 15u;
  const uint32_t m = code & 7u;
  return e == 0 ? __fmul_rn(static_cast<float>(m), 0x1p-9f)
                : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// Eight fp32 values -> four bytes of E2M1 codes (round to nearest even,
// saturating at 6, sign kept).  Element 2i goes to the low nibble of byte i.
__device__ __forceinline__ uint32_t e2m1x8(float2 a, float2 b, float2 c, float2 d) {
  uint32_t r;
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
      : "=r"(r)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y), "f"(d.x), "f"(d.y));
  return r;
}

// ---------------------------------------------------------------------------
// Block quantize
// ---------------------------------------------------------------------------

// Largest |y| of a block of 16 bf16 values, exact: the magnitude bit patterns
// of non-NaN bf16 values order like the values.
__device__ __forceinline__ float block_amax(const Block16& y) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t a = y.w[i] & 0x7fff7fffu;
    asm("max.u16x2 %0, %0, %1;" : "+r"(m) : "r"(a));
  }
  const uint32_t hi = m >> 16, lo = m & 0xffffu;
  return __uint_as_float((hi > lo ? hi : lo) << 16);
}

struct Quantized {
  uint32_t sf;        // E4M3 scale byte
  uint32_t codes_lo;  // codes of elements 0..7
  uint32_t codes_hi;  // codes of elements 8..15
};

// NVFP4 of one block of bf16 values y under the global scale gsf:
//   sf = E4M3(fl(gsf * fl(amax / 6))), dec = fl(E4M3value(sf) / gsf),
//   inv = dec != 0 ? fl(1 / dec) : 0, code_i = E2M1(fl(y_i * inv)).
__device__ __forceinline__ Quantized quantize_block(const Block16& y, float gsf) {
  const float amax = block_amax(y);
  const float s = __fmul_rn(gsf, __fdiv_rn(amax, 6.0f));
  Quantized q;
  q.sf = e4m3_encode(s);
  const float dec = __fdiv_rn(e4m3_value(q.sf), gsf);
  const float inv = dec != 0.0f ? __frcp_rn(dec) : 0.0f;
  const float2 inv2 = make_float2(inv, inv);
  float2 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __fmul2_rn(bf16x2_to_float2(y.w[i]), inv2);
  q.codes_lo = e2m1x8(v[0], v[1], v[2], v[3]);
  q.codes_hi = e2m1x8(v[4], v[5], v[6], v[7]);
  return q;
}

// ---------------------------------------------------------------------------
// 128x4 scale layout
// ---------------------------------------------------------------------------

// Byte offset, inside the scale matrix, of the 4-byte word that holds scale
// columns 4*quad .. 4*quad+3 of row `row`: atoms of 128 rows x 4 columns (512 B)
// laid out row-tile major; inside an atom, row r sits at (r%32)*16 + ((r/32)%4)*4.
__device__ __forceinline__ int64_t scale_word_offset(int64_t row, int64_t quad,
                                                     int64_t quads_per_row) {
  const int64_t atom = (row >> 7) * quads_per_row + quad;
  return atom * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4;
}

// Lanes 4a..4a+3 of a warp hold the scale bytes of four consecutive scale
// columns starting at a multiple of 4; lane 4a stores them as one word.
// All 32 lanes must call this (it shuffles); `active` masks the store.
__device__ __forceinline__ void store_scale_quad(uint8_t* scales, int64_t row, int64_t group,
                                                 int64_t quads_per_row, uint32_t sf, bool active) {
  const int lane = threadIdx.x & 31;
  uint32_t word = sf << (8 * (lane & 3));
  word |= __shfl_xor_sync(0xffffffffu, word, 1);
  word |= __shfl_xor_sync(0xffffffffu, word, 2);
  if (active && (lane & 3) == 0)
    store_word(scales + scale_word_offset(row, group >> 2, quads_per_row), word);
}

}  // namespace h3q
